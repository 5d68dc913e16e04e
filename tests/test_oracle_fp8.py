"""Pins of the oracle's channel-FP8 (QPN8) quantiser and projection and of its
prepared-scale expansion: a hand-worked case, torch's float8_e4m3fn
conversions (library routines) and torch.matmul in FP64.

Pages: "[SM70][Draft] Extend Qwen3.8 DFlash2 concurrency paths", section
"Follow-up: exact channel-FP8 QPN8 concurrency paths" (FP8 weights with one
scale per output channel, few-row projections); "[Kernel][SM70] Improve
Qwen3.8 no-MTP concurrency", sections "Scope and related PRs" and "Test
Result" (prepared effective decode scales beside raw E4M3 storage).
"""
import os

import numpy as np
import torch

import oracle
from helpers import parse_golden


def _golden(golden_dir):
    rows = parse_golden(os.path.join(golden_dir, "fp8_channel_worked_case.txt"))
    out = {}
    for r in rows:
        kind, i = r[0], int(r[1])
        if kind == "q":
            vals = [int(t, 16) for t in r[2:]]
        else:
            vals = [float(t) for t in r[2:]]
        out.setdefault(kind, {})[i] = vals
    return out


def test_fp8_quantize_worked_case(golden_dir):
    g = _golden(golden_dir)
    w = np.array([g["w"][i] for i in range(3)], np.float32)
    q, cs, st = oracle.fp8_quantize(w)
    assert st == 0
    np.testing.assert_array_equal(q, np.array([g["q"][i] for i in range(3)], np.uint8))
    np.testing.assert_array_equal(cs, np.array([g["cs"][i][0] for i in range(3)], np.float32))


def test_fp8_dense_worked_case(golden_dir):
    g = _golden(golden_dir)
    w = np.array([g["w"][i] for i in range(3)], np.float32)
    q, cs, _ = oracle.fp8_quantize(w)
    x = np.array([g["x"][0]], np.float16)
    y = oracle.fp8_dense(x, q, cs)
    np.testing.assert_array_equal(y.astype(np.float64), np.array([g["y"][0]]))


def _torch_e4m3(a):
    """FP32 -> E4M3 codes by torch's float8_e4m3fn conversion (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_fp8_quantize_vs_torch_float8():
    rng = np.random.default_rng(21)
    w = (rng.standard_normal((96, 256)) * 0.02).astype(np.float32)
    w[3] = 0.0
    w[5, :7] *= 1e4                     # one row with a wide range (subnormal codes)
    q, cs, st = oracle.fp8_quantize(w)
    assert st == 0
    amax = np.abs(w).max(axis=1)
    cs_ref = np.where(amax == 0, np.float32(1.0), (amax / np.float32(448.0)).astype(np.float32))
    np.testing.assert_array_equal(cs, cs_ref)
    ref = _torch_e4m3(w / cs_ref[:, None])
    np.testing.assert_array_equal(q, ref)
    # the largest magnitude of each nonzero row maps to +-448
    i = np.abs(w).argmax(axis=1)
    top = q[np.arange(96), i] & 0x7F
    assert np.all(top[amax > 0] == 0x7E)


def test_fp8_quantize_flags_nonfinite():
    w = np.ones((2, 64), np.float32)
    w[1, 5] = np.nan
    q, cs, st = oracle.fp8_quantize(w)
    assert st & oracle.ST_NONFINITE
    assert q[1, 5] == 0 and cs[1] == np.float32(1.0 / 448.0)


def test_fp8_dense_vs_torch_matmul():
    rng = np.random.default_rng(22)
    M, N, K = 5, 48, 320
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    q, cs, _ = oracle.fp8_quantize(w)
    x = rng.standard_normal((M, K)).astype(np.float16)
    y = oracle.fp8_dense(x, q, cs).astype(np.float64)
    wd = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64)
    ref = (torch.from_numpy(x.astype(np.float64)) @ wd.T) * torch.from_numpy(cs.astype(np.float64))
    ref16 = ref.numpy().astype(np.float16).astype(np.float64)
    # FP64 sums in different orders round to the same FP16 except at rare ties
    assert np.mean(y == ref16) > 0.99
    np.testing.assert_allclose(y, ref.numpy(), rtol=2 ** -10, atol=1e-6)


def test_fp8_dense_rows_independent():
    rng = np.random.default_rng(23)
    w = (rng.standard_normal((32, 128)) * 0.02).astype(np.float32)
    q, cs, _ = oracle.fp8_quantize(w)
    x = rng.standard_normal((9, 128)).astype(np.float16)
    full = oracle.fp8_dense(x, q, cs)
    parts = np.concatenate([oracle.fp8_dense(x[:8], q, cs), oracle.fp8_dense(x[8:], q, cs)])
    np.testing.assert_array_equal(full.view(np.uint16), parts.view(np.uint16))


def test_prepare_scales_vs_torch():
    """Every finite E4M3 code widens to the FP16 value torch gives it (exact);
    the two NaN codes give FP16 NaN and the status bit."""
    codes = np.arange(256, dtype=np.uint8)
    out, st = oracle.prepare_scales(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float16) \
        .view(torch.int16).numpy().view(np.uint16)
    finite = np.array([c not in (0x7F, 0xFF) for c in range(256)])
    np.testing.assert_array_equal(out[finite], ref[finite])
    assert np.all(out[~finite] == 0x7E00) and st & oracle.ST_NONFINITE
    out2, st2 = oracle.prepare_scales(codes[finite].reshape(2, -1))
    assert st2 == 0 and out2.shape == (2, 127)
