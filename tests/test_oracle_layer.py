"""Pins of the oracle's quantiser, router, plan and layer forward.

Each test checks the oracle against something other than itself: a
hand-worked case, a library routine (numpy stable argsort, torch float8
conversion, torch.matmul), brute force over all experts in FP64, or an
invariant that a dropped term, wrong sign or transposed operand would break.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from helpers import dequant_np, e4m3_table_torch, num, parse_golden, rel_l2
from nvfp4_weight_mixture_gb300 import synth

TINY = synth.WORKLOADS["tiny_m8"]


# ---- quantiser ------------------------------------------------------------------

def test_quantize_worked_case(golden_dir):
    rows = parse_golden(os.path.join(golden_dir, "quantize_worked_case.txt"))
    x = np.zeros((4, 16), np.float32)
    q_exp = np.zeros((4, 16), np.int64)
    s_exp = np.zeros(4, np.int64)
    g_exp = None
    for r in rows:
        if r[0] == "x":
            x[int(r[1])] = [float(v) for v in r[2:]]
        elif r[0] == "q":
            q_exp[int(r[1])] = [int(v, 16) for v in r[2:]]
        elif r[0] == "s":
            s_exp[int(r[1])] = int(r[2], 16)
        elif r[0] == "g":
            g_exp = float(r[1])
    q, s, g, st = oracle.quantize(x[None])
    assert st == 0
    assert g[0] == g_exp
    codes = np.stack([q[0] & 15, q[0] >> 4], -1).reshape(4, 16)
    np.testing.assert_array_equal(codes, q_exp)
    np.testing.assert_array_equal(s[0, :, 0], s_exp)


def test_quantize_invariants_random():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((3, 64, 256)) * 0.02).astype(np.float32)
    w[1, 5, 17] = -0.0
    w[2, :, :16] = 0.0                     # an all-zero block in every row
    w[2, 3, 32:48] *= 1e-6                 # tiny block -> subnormal / zero scale
    q, s, g, st = oracle.quantize(w)
    assert st == 0
    tab = e4m3_table_torch()
    for m in range(3):
        amax = np.abs(w[m]).max()
        assert g[m] == np.float32(amax) / np.float32(2688.0)
        # block scales: torch's float8 conversion of (amax_b / g) / 6, all in FP32
        bmax = np.abs(w[m].reshape(64, 16, 16)).max(-1).astype(np.float32)
        sb = (bmax / g[m]).astype(np.float32) / np.float32(6.0)
        ref_s = torch.from_numpy(sb.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        np.testing.assert_array_equal(s[m], ref_s)
        # reconstruction error within half an E2M1 step of the block scale
        deq = dequant_np(q[m], s[m]) * np.float64(g[m])
        d = np.repeat(tab[s[m]] * np.float64(g[m]), 16, axis=-1)
        err = np.abs(deq - w[m].astype(np.float64))
        sat = np.abs(w[m]) > 6 * d
        # the widest E2M1 gap is 2 (between 4 and 6) -> half-gap 1 * d
        assert np.all((err <= 1.0 * d + 1e-30) | sat)
        small = np.abs(w[m]) <= 2 * d       # spacing 0.5 below 2: half-gap 0.25 d
        assert np.all((err <= 0.25 * d + 1e-30) | ~small | sat)
        # signs are kept, including on zero
        codes = np.stack([q[m] & 15, q[m] >> 4], -1).reshape(64, 256)
        assert np.all((codes >= 8) == np.signbit(w[m]))
    # the tensor maximum: its block scale is 448 (0x7E) and its code is 6
    m = 0
    r, c = np.unravel_index(np.argmax(np.abs(w[m])), w[m].shape)
    assert s[m, r, c // 16] == 0x7E
    code = (q[m, r, c // 2] >> (4 * (c % 2))) & 7
    assert code == 7
    # NaN codes are never emitted
    assert not np.any(s == 0x7F) and not np.any(s == 0xFF)


def test_quantize_zero_tensor_and_nonfinite():
    q, s, g, st = oracle.quantize(np.zeros((1, 16, 32), np.float32))
    assert st == 0 and g[0] == 1.0 and not q.any() and not s.any()
    w = np.ones((1, 16, 32), np.float32)
    w[0, 3, 4] = np.inf
    *_, st = oracle.quantize(w)
    assert st & oracle.ST_NONFINITE
    w[0, 3, 4] = np.nan
    *_, st = oracle.quantize(w)
    assert st & oracle.ST_NONFINITE


# ---- router ----------------------------------------------------------------------

def _router_np(x, wr, bias, k):
    l = x.astype(np.float64) @ wr.astype(np.float64)
    if bias is not None:
        l = l + bias.astype(np.float64)
    return l


@pytest.mark.parametrize("bias_kind", ["none", "normal"])
def test_router_against_fp64(bias_kind):
    wl = synth.custom("r", 64, 512, 96, 6, 64, bias=bias_kind)
    x = synth.activations(wl)
    wr = synth.router_weight(wl)
    b = synth.router_bias(wl)
    logits, ids, w = oracle.router(x, wr, b, wl.k)
    ref = _router_np(x, wr, b, wl.k)
    assert np.max(np.abs(logits - ref)) < 1e-5
    for t in range(wl.M):
        order = np.argsort(-ref[t], kind="stable")
        lk = np.sort(ref[t])[::-1]
        gap = lk[wl.k - 1] - lk[wl.k]
        if gap > 1e-5:
            assert set(ids[t]) == set(order[: wl.k])
        # weights: softmax over the selected logits (FP64 reference)
        sel = ref[t, ids[t]]
        p = np.exp(sel - sel.max())
        p /= p.sum()
        assert np.max(np.abs(w[t] - p)) < 1e-6
        assert abs(w[t].sum() - 1.0) < 1e-6
        assert np.all(np.diff(logits[t, ids[t]]) <= 0)          # descending
        assert len(set(ids[t])) == wl.k


def test_router_ties_and_k1():
    wl = synth.custom("r", 4, 64, 8, 3, 32)
    x = synth.activations(wl)
    wr = synth.router_weight(wl)
    wr[:, 5] = wr[:, 2]          # experts 2 and 5 always tie
    wr[:, 6] = wr[:, 2]
    bias = np.zeros(8, np.float32)
    bias[[2, 5, 6]] = 50.0       # ... and are always the top three
    logits, ids, w = oracle.router(x, wr, bias, 3)
    assert np.all(ids == np.array([2, 5, 6]))
    np.testing.assert_allclose(w, 1.0 / 3.0, rtol=1e-6)
    _, ids1, w1 = oracle.router(x, wr, None, 1)
    assert np.all(w1 == 1.0)
    ref = _router_np(x, wr, None, 1)
    assert np.all(ids1[:, 0] == np.argmax(ref, axis=1))


def test_shared_gate():
    wl = synth.custom("g", 5, 128, 4, 1, 32, shared=True)
    x = synth.activations(wl)
    wg = synth.gate_weight(wl)
    gm = oracle.shared_gate(x, wg)
    z = x.astype(np.float64) @ wg.astype(np.float64)
    np.testing.assert_allclose(gm, 1 / (1 + np.exp(-z)), rtol=1e-6)
    assert np.all(oracle.shared_gate(x, np.zeros_like(wg)) == 0.5)


# ---- plan ------------------------------------------------------------------------

def _check_plan(ids, E, bn):
    p = oracle.plan(ids, E, bn)
    flat = ids.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    assert (p["status"] & oracle.ST_INVALID_ID) == (0 if valid.all() else oracle.ST_INVALID_ID)
    np.testing.assert_array_equal(p["counts"], np.bincount(flat[valid], minlength=E))
    np.testing.assert_array_equal(p["offsets"], np.concatenate([[0], np.cumsum(p["counts"])]))
    vidx = np.nonzero(valid)[0]
    ref_perm = vidx[np.argsort(flat[valid], kind="stable")]
    np.testing.assert_array_equal(p["perm"], ref_perm)
    inv = p["inv"]
    assert np.all(inv[~valid] == -1)
    np.testing.assert_array_equal(p["perm"][inv[valid]], vidx)
    assert p["counts"].sum() == valid.sum()
    # tiles cover each segment in order, each at most bn rows
    tiles = p["tiles"]
    cover = np.zeros(E, np.int64)
    for e, r0, rows in tiles:
        assert 0 < rows <= bn and r0 == cover[e]
        cover[e] += rows
    np.testing.assert_array_equal(cover, p["counts"])
    assert list(tiles[:, 0]) == sorted(tiles[:, 0])
    return p


def test_plan_random_and_edge_cases():
    wl = synth.custom("p", 300, 64, 37, 5, 32)
    _check_plan(synth.random_ids(wl), 37, 16)
    _check_plan(synth.random_ids(wl), 37, 128)
    # all tokens to one expert (k = 1)
    _check_plan(np.full((300, 1), 7, np.int32), 37, 64)
    # all-singleton: every expert exactly once
    _check_plan(np.arange(37, dtype=np.int32).reshape(37, 1), 37, 16)
    # invalid ids are dropped and flagged
    ids = synth.random_ids(wl)
    ids[3, 1] = -1
    ids[10, 4] = 37
    ids[11, 0] = 1 << 30
    _check_plan(ids, 37, 16)
    # empty
    p = oracle.plan(np.zeros((0, 4), np.int32), 8, 16)
    assert p["counts"].sum() == 0 and len(p["tiles"]) == 0


# ---- layer forward -----------------------------------------------------------------

def _quant_all(wl, shared=False):
    w13 = oracle.quantize(synth.all_w13(wl))[:3]
    w2 = oracle.quantize(synth.all_w2(wl))[:3]
    sh = None
    if shared:
        a = oracle.quantize(synth.shared_w13(wl)[None])[:3]
        b = oracle.quantize(synth.shared_w2(wl)[None])[:3]
        sh = ((a[0][0], a[1][0], a[2][0]), (b[0][0], b[1][0], b[2][0]))
    return w13, w2, sh


def _dense_moe_fp64(x, wr, bias, k, w13, w2, sh=None, wg=None):
    """Brute force: every expert on every token in FP64, then keep the top-k."""
    E = w13[0].shape[0]
    I = w13[0].shape[1] // 2
    xd = x.astype(np.float64)
    l = xd @ wr.astype(np.float64)
    if bias is not None:
        l = l + bias
    W13 = dequant_np(w13[0], w13[1]) * w13[2][:, None, None].astype(np.float64)
    W2 = dequant_np(w2[0], w2[1]) * w2[2][:, None, None].astype(np.float64)
    outs = []
    for e in range(E):
        G = xd @ W13[e, :I].T
        U = xd @ W13[e, I:].T
        h = (G / (1 + np.exp(-G)) * U).astype(np.float16).astype(np.float64)
        outs.append(h @ W2[e].T)
    outs = np.stack(outs, 1)  # [M, E, H]
    y = np.zeros((x.shape[0], x.shape[1]))
    ids = np.zeros((x.shape[0], k), np.int64)
    for t in range(x.shape[0]):
        sel = np.argsort(-l[t], kind="stable")[:k]
        ids[t] = sel
        p = np.exp(l[t, sel] - l[t, sel].max())
        p /= p.sum()
        y[t] = (p[:, None] * outs[t, sel]).sum(0)
    if sh is not None:
        (a, b) = sh
        S13 = dequant_np(a[0], a[1]) * np.float64(a[2])
        S2 = dequant_np(b[0], b[1]) * np.float64(b[2])
        G = xd @ S13[:I].T
        U = xd @ S13[I:].T
        h = (G / (1 + np.exp(-G)) * U).astype(np.float16).astype(np.float64)
        gm = 1 / (1 + np.exp(-(xd @ wg.astype(np.float64))))
        y = y + gm[:, None] * (h @ S2.T)
    return y, ids


@pytest.mark.parametrize("shared", [False, True])
def test_forward_against_dense_brute_force(shared):
    wl = TINY if not shared else synth.custom("t", 8, 256, 16, 2, 128, bias="zipf", shared=True)
    x = synth.activations(wl)
    wr = synth.router_weight(wl)
    b = synth.router_bias(wl)
    wg = synth.gate_weight(wl)
    w13, w2, sh = _quant_all(wl, shared)
    _, ids, w = oracle.router(x, wr, b, wl.k)
    gm = oracle.shared_gate(x, wg) if shared else None
    y, st = oracle.forward(x, ids, w, w13, w2, shared=sh, gamma=gm)
    assert st == 0
    yref, ids_ref = _dense_moe_fp64(x, wr, b, wl.k, w13, w2, sh, wg)
    np.testing.assert_array_equal(np.sort(ids, 1), np.sort(ids_ref, 1))
    # same FP64 math in another order: y must be yref rounded to FP16, except
    # (rarely) one unit in the last place where yref sits on a rounding edge
    same = y.view(np.uint16) == yref.astype(np.float16).view(np.uint16)
    assert same.mean() > 0.999
    np.testing.assert_allclose(y.astype(np.float64), yref, rtol=2 ** -10, atol=2 ** -24)
    assert rel_l2(y, yref) < 4e-4


def test_forward_single_expert_is_dense_swiglu():
    wl = synth.custom("d", 6, 128, 1, 1, 64)
    x = synth.activations(wl)
    w13, w2, _ = _quant_all(wl)
    ids = np.zeros((6, 1), np.int32)
    y, st = oracle.forward(x, ids, np.ones((6, 1), np.float32), w13, w2)
    W13 = torch.from_numpy(dequant_np(w13[0][0], w13[1][0]) * float(w13[2][0]))
    W2 = torch.from_numpy(dequant_np(w2[0][0], w2[1][0]) * float(w2[2][0]))
    xt = torch.from_numpy(x.astype(np.float64))
    gu = torch.matmul(xt, W13.T)
    h = torch.nn.functional.silu(gu[:, :64]) * gu[:, 64:]
    h = h.to(torch.float16).to(torch.float64)
    ref = torch.matmul(h, W2.T).numpy()
    np.testing.assert_allclose(y.astype(np.float64), ref, rtol=2 ** -10, atol=2 ** -24)


def test_forward_token_permutation_and_subsets():
    wl = TINY
    x = synth.activations(wl)
    w13, w2, _ = _quant_all(wl)
    _, ids, w = oracle.router(x, synth.router_weight(wl), None, wl.k)
    y, _ = oracle.forward(x, ids, w, w13, w2)
    perm = np.array([3, 1, 7, 0, 2, 6, 5, 4])
    yp, _ = oracle.forward(x[perm], ids[perm], w[perm], w13, w2)
    np.testing.assert_array_equal(yp.view(np.uint16), y[perm].view(np.uint16))
    ys, _ = oracle.forward(x, ids, w, w13, w2, tokens=[6, 2])
    np.testing.assert_array_equal(ys.view(np.uint16), y[[6, 2]].view(np.uint16))
    # the slot weights enter linearly; swapping two slots changes nothing
    y2, _ = oracle.forward(x, ids[:, ::-1], w[:, ::-1], w13, w2)
    np.testing.assert_allclose(y2.astype(np.float64), y.astype(np.float64), rtol=2 ** -10, atol=1e-7)


def test_forward_invalid_ids_contribute_zero():
    wl = TINY
    x = synth.activations(wl)
    w13, w2, _ = _quant_all(wl)
    _, ids, w = oracle.router(x, synth.router_weight(wl), None, wl.k)
    bad = ids.copy()
    bad[:, 1] = -3
    y, st = oracle.forward(x, bad, w, w13, w2)
    assert st & oracle.ST_INVALID_ID
    w1 = w.copy()
    w1[:, 1] = 0.0
    yref, st2 = oracle.forward(x, ids, w1, w13, w2)
    assert st2 == 0
    np.testing.assert_array_equal(y.view(np.uint16) & 0x7FFF, yref.view(np.uint16) & 0x7FFF)


def test_forward_h_is_fp16_rounded_swiglu():
    wl = TINY
    x = synth.activations(wl)
    w13, w2, _ = _quant_all(wl)
    _, ids, w = oracle.router(x, synth.router_weight(wl), None, wl.k)
    y, st, h = oracle.forward(x, ids, w, w13, w2, want_h=True)
    t, j = 5, 1
    e = ids[t, j]
    W13 = dequant_np(w13[0][e], w13[1][e]) * np.float64(w13[2][e])
    gu = W13 @ x[t].astype(np.float64)
    ref = gu[:128] / (1 + np.exp(-gu[:128])) * gu[128:]
    np.testing.assert_array_equal(h[t, j], ref.astype(np.float16).astype(np.float64))


def test_forward_h_exact_reading():
    """The other reading of the h hand-off (no FP16 rounding between the
    GEMMs): h equals the FP64 SwiGLU itself, the single-expert layer equals
    the dense MLP with unrounded h (torch.matmul), and on the tiny workload the
    two readings' outputs sit well inside the acceptance bar of each other,
    so that bar does not depend on which reading is taken."""
    wl = TINY
    x = synth.activations(wl)
    w13, w2, _ = _quant_all(wl)
    _, ids, w = oracle.router(x, synth.router_weight(wl), None, wl.k)
    yx, st, h = oracle.forward(x, ids, w, w13, w2, want_h=True, h_exact=True)
    assert st == 0
    t, j = 2, 0
    e = ids[t, j]
    W13 = dequant_np(w13[0][e], w13[1][e]) * np.float64(w13[2][e])
    gu = W13 @ x[t].astype(np.float64)
    ref = gu[:128] / (1 + np.exp(-gu[:128])) * gu[128:]
    np.testing.assert_allclose(h[t, j], ref, rtol=1e-12, atol=1e-15)
    assert np.any(h[t, j] != ref.astype(np.float16).astype(np.float64))
    y16, _ = oracle.forward(x, ids, w, w13, w2)
    r = rel_l2(yx, y16)
    assert 0 < r < 5e-4  # ~3.3e-4: the FP16 rounding of h, averaged over I terms
    assert np.max(np.abs(yx.astype(np.float64) - y16.astype(np.float64))) < 1e-2

    d = synth.custom("d", 6, 128, 1, 1, 64)
    xd = synth.activations(d)
    a13, a2, _ = _quant_all(d)
    y1, _ = oracle.forward(xd, np.zeros((6, 1), np.int32), np.ones((6, 1), np.float32), a13, a2,
                           h_exact=True)
    W13 = torch.from_numpy(dequant_np(a13[0][0], a13[1][0]) * float(a13[2][0]))
    W2 = torch.from_numpy(dequant_np(a2[0][0], a2[1][0]) * float(a2[2][0]))
    gu = torch.matmul(torch.from_numpy(xd.astype(np.float64)), W13.T)
    hh = torch.nn.functional.silu(gu[:, :64]) * gu[:, 64:]
    np.testing.assert_allclose(y1.astype(np.float64), torch.matmul(hh, W2.T).numpy(),
                               rtol=2 ** -10, atol=2 ** -24)
