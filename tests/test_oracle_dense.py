"""Pins of the oracle's dense NVFP4 projection (the small-M QPN2 projection of
"[SM70][Draft] Extend Qwen3.8 DFlash2 concurrency paths", section "Purpose"):
a hand-worked case, torch.matmul on FP64-dequantised weights, row
independence (eight-row tiles equal one call), and agreement with the layer
oracle's own second GEMM."""
import os

import numpy as np
import torch

import oracle
from helpers import dequant_np, parse_golden
from nvfp4_weight_mixture_gb300 import synth


def _golden(golden_dir):
    rows = parse_golden(os.path.join(golden_dir, "dense_worked_case.txt"))
    q = np.array([[int(b, 16) for b in r[2:]] for r in rows if r[0] == "q"], np.uint8)
    s = np.array([[int(r[2], 16)] for r in rows if r[0] == "s"], np.uint8)
    g = [float(r[1]) for r in rows if r[0] == "g"][0]
    x = np.array([[float(v) for v in r[2:]] for r in rows if r[0] == "x"], np.float16)
    y = np.array([[float(v) for v in r[2:]] for r in rows if r[0] == "y"], np.float64)
    return q, s, g, x, y


def test_dense_worked_case(golden_dir):
    q, s, g, x, y = _golden(golden_dir)
    got = oracle.dense(x, q, s, g)
    np.testing.assert_array_equal(got.astype(np.float64), y)


def _random_case(M, N, K, seed):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    q, s, g, st = oracle.quantize(w[None])
    x = rng.standard_normal((M, K)).astype(np.float16)
    return x, q[0], s[0], g[0]


def test_dense_matches_torch_matmul_fp64():
    x, q, s, g = _random_case(16, 96, 512, 5)
    got = oracle.dense(x, q, s, g)
    W = torch.from_numpy(dequant_np(q, s)) * float(g)
    ref = torch.matmul(torch.from_numpy(x.astype(np.float64)), W.T).numpy()
    same = got.view(np.uint16) == ref.astype(np.float16).view(np.uint16)
    assert same.mean() > 0.999
    np.testing.assert_allclose(got.astype(np.float64), ref, rtol=2 ** -10, atol=2 ** -24)


def test_dense_rows_are_independent():
    # eight-row tiles, single rows and the whole batch give the same bits
    x, q, s, g = _random_case(16, 64, 256, 7)
    y = oracle.dense(x, q, s, g).view(np.uint16)
    y8 = np.concatenate([oracle.dense(x[:8], q, s, g), oracle.dense(x[8:], q, s, g)])
    np.testing.assert_array_equal(y8.view(np.uint16), y)
    np.testing.assert_array_equal(oracle.dense(x[5:6], q, s, g).view(np.uint16), y[5:6])
    # a transposed operand would mix rows: permuting the rows permutes y
    perm = np.random.default_rng(1).permutation(16)
    np.testing.assert_array_equal(oracle.dense(x[perm], q, s, g).view(np.uint16), y[perm])


def test_dense_is_the_layers_second_gemm():
    # one expert, weight 1: the layer's output is the dense projection of its
    # FP16 h by W2, bit for bit (same FP64 sum, one rounding)
    wl = synth.custom("d", 6, 128, 1, 1, 64)
    x = synth.activations(wl)
    a = oracle.quantize(synth.expert_w13(wl, 0)[None])
    b = oracle.quantize(synth.expert_w2(wl, 0)[None])
    w13 = (a[0], a[1], a[2])
    w2 = (b[0], b[1], b[2])
    ids = np.zeros((6, 1), np.int32)
    y, st, h = oracle.forward(x, ids, np.ones((6, 1), np.float32), w13, w2, want_h=True)
    h16 = h[:, 0, :].astype(np.float16)
    np.testing.assert_array_equal(h16.astype(np.float64), h[:, 0, :])
    yd = oracle.dense(h16, b[0][0], b[1][0], b[2][0])
    np.testing.assert_array_equal(yd.view(np.uint16), y.view(np.uint16))
