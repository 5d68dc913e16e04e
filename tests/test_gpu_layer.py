"""GPU router, plan and layer forward vs the CPU oracle.

Acceptance (the layer's stated parity bar):
  * plan: bit-exact given the same expert ids;
  * router: top-k id sets agree except where the oracle's gap between the
    k-th and (k+1)-th logit is below 1e-5; weights within 1e-5;
  * layer output: rel-L2 <= 1e-3 and max-abs <= 2e-2 against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from harness import (DECODE_MAX_TOKENS, MAX_ABS_TOL, REL_L2_TOL, ROUTER_GAP, ROUTER_W_TOL,
                     TILE_ROWS, Case, compare, expected_tile_pos, expected_work_table)
from nvfp4_weight_mixture_gb300 import moe, synth

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny_m8"]
DEC1 = synth.WORKLOADS["decode_m1"]
DEC16 = synth.WORKLOADS["decode_m16_bias"]
PRE = synth.WORKLOADS["prefill_m8192"]
PRE_Z = synth.WORKLOADS["prefill_m8192_zipf_shared"]


def _check_router(case, tokens=None):
    ids_g, w_g = case.gpu_route()
    tok = np.arange(case.wl.M) if tokens is None else np.asarray(tokens)
    logits, ids_o, w_o, _ = case.oracle_route(tok)
    k = case.wl.k
    mismatched = 0
    for i, t in enumerate(tok):
        srt = np.sort(logits[i])[::-1]
        gap = srt[k - 1] - srt[k] if k < len(srt) else np.inf
        if set(ids_g[t]) != set(ids_o[i]):
            assert gap < ROUTER_GAP, (t, ids_g[t], ids_o[i], gap)
            mismatched += 1
            continue
        # same set: same order unless logits tie within the gap tolerance
        if not np.array_equal(ids_g[t], ids_o[i]):
            assert np.min(np.abs(np.diff(logits[i][ids_o[i]]))) < ROUTER_GAP
            continue
        assert np.max(np.abs(w_g[t] - w_o[i])) <= ROUTER_W_TOL, t
        assert abs(float(w_g[t].sum()) - 1.0) < 1e-5
    assert mismatched <= max(1, len(tok) // 1000)
    return ids_g, w_g


def _check_plan(case, ids):
    """GPU plan of `ids` vs the oracle plan of the same ids: bit-exact."""
    wl = case.wl
    k_eff = wl.k + int(wl.shared)
    e_eff = wl.E + int(wl.shared)
    ids_eff = np.asarray(ids, np.int32)
    if wl.shared:
        ids_eff = np.concatenate([ids_eff, np.full((wl.M, 1), wl.E, np.int32)], 1)
    ref = oracle.plan(ids_eff, e_eff, TILE_ROWS)
    got = case.plan_arrays()
    np.testing.assert_array_equal(got["ids"], ids_eff.reshape(-1))
    np.testing.assert_array_equal(got["counts"], ref["counts"])
    np.testing.assert_array_equal(got["offsets"], ref["offsets"])
    np.testing.assert_array_equal(got["perm"], ref["perm"])
    np.testing.assert_array_equal(got["inv"], ref["inv"])
    np.testing.assert_array_equal(got["tiles"], ref["tiles"])
    np.testing.assert_array_equal(got["tile_pos"], expected_tile_pos(ref))
    np.testing.assert_array_equal(got["active"], np.nonzero(ref["counts"])[0])
    assert int(got["hdr"][0]) == wl.M and int(got["hdr"][1]) == k_eff
    if wl.M <= DECODE_MAX_TOKENS:
        # the decode work table the oracle plan implies
        exp_tab = expected_work_table(ref, wl.M, k_eff, e_eff)
        np.testing.assert_array_equal(got["dtab"][:len(exp_tab)], exp_tab)
    return ref


# ---- router ---------------------------------------------------------------------------

@pytest.mark.parametrize("wl,M", [(TINY, 8), (TINY, 1), (TINY, 77), (DEC1, 1), (DEC16, 16),
                                  (DEC16, 9), (PRE, 300)])
def test_router_vs_oracle(wl, M):
    case = Case(synth.with_tokens(wl, M))
    _check_router(case)
    assert int(case.layer.status.item()) == 0


def test_router_full_prefill_sampled():
    case = Case(PRE_Z)
    rng = np.random.default_rng(3)
    tok = np.sort(rng.choice(PRE_Z.M, 256, replace=False))
    _check_router(case, tok)


class _RouteCase:
    """Router-only case: seeded x, W_r, bias; no expert weights (route() needs none)."""

    def __init__(self, wl):
        self.wl = wl
        self.x = synth.activations(wl)
        self.wr = synth.router_weight(wl)
        self.bias = synth.router_bias(wl)
        dev = torch.device("cuda")
        self.x_t = torch.from_numpy(self.x).to(dev)
        self.layer = moe.MoELayer(
            wl.H, wl.E, wl.k, wl.I, torch.from_numpy(self.wr).to(dev), None, None,
            bias=None if self.bias is None else torch.from_numpy(self.bias).to(dev),
            max_tokens=max(wl.M, 1))

    def gpu_route(self):
        ids, w = self.layer.route(self.x_t)
        return ids.cpu().numpy(), w.cpu().numpy()

    def oracle_route(self, tokens=None):
        x = self.x if tokens is None else self.x[np.asarray(tokens)]
        logits, ids, w = oracle.router(x, self.wr, self.bias, self.wl.k)
        return logits, ids, w, None


@pytest.mark.parametrize("M,H,E,k", [(300, 2048, 256, 8), (300, 1024, 384, 10),
                                     (128, 512, 256, 4), (8300, 2048, 512, 10)])
def test_router_tensor_core_shapes(M, H, E, k):
    """The tcgen05 router (M >= 128, E >= 256): a partial last expert slice
    (E 384), M exactly one token tile, and M above one 8192-token logits chunk
    (sampled tokens from both chunks)."""
    case = _RouteCase(synth.custom("rt", M, H, E, k, 128))
    tok = None
    if M > 1000:
        rng = np.random.default_rng(11)
        tok = np.sort(np.concatenate([rng.choice(8192, 128, replace=False),
                                      8192 + rng.choice(M - 8192, 64, replace=False)]))
    _check_router(case, tok)
    assert int(case.layer.status.item()) == 0


def test_router_tensor_core_ties():
    """Exact ties in the tcgen05 router's top-k (M >= 128).  Experts 2j and
    2j + 1 share their router column, so every logit appears twice and the
    lower id must come first (candidates gathered one per lane).  Tokens
    0..63 are zero rows: all 512 logits tie, the top-k is experts 0..k-1
    with equal weights (more than 32 candidates: the general rounds)."""
    wl = synth.custom("rt_ties", 256, 512, 512, 10, 128)
    case = _RouteCase(wl)
    case.x = case.x.copy()
    case.x[:64] = 0
    case.wr = case.wr.copy()
    case.wr[:, 1::2] = case.wr[:, 0::2]
    dev = torch.device("cuda")
    case.x_t = torch.from_numpy(case.x).to(dev)
    case.layer = moe.MoELayer(wl.H, wl.E, wl.k, wl.I, torch.from_numpy(case.wr).to(dev), None,
                              None, max_tokens=wl.M)
    ids_g, w_g = _check_router(case)
    np.testing.assert_array_equal(ids_g[:64], np.tile(np.arange(wl.k, dtype=np.int32), (64, 1)))
    assert np.max(np.abs(w_g[:64] - 1.0 / wl.k)) <= 1e-6
    for t in range(64, wl.M):
        sel = [int(e) for e in ids_g[t]]
        for pos, e in enumerate(sel):
            twin = e ^ 1
            if e & 1:  # an odd expert is taken only after its even twin
                assert twin in sel[:pos], (t, sel)
    assert int(case.layer.status.item()) == 0


@pytest.mark.parametrize("M,H,E,k", [(40, 256, 32, 32), (200, 4096, 136, 10), (100, 512, 512, 3)])
def test_router_mma_shapes(M, H, E, k):
    """The mma.sync router (16 < M with E < 256, or M < 128): k = E = 32, the
    largest hidden size with E not a multiple of 64 (136), and E = 512 below
    the tensor-core router's 128-token minimum."""
    case = _RouteCase(synth.custom("rm", M, H, E, k, 128))
    _check_router(case)
    assert int(case.layer.status.item()) == 0


@pytest.mark.parametrize("M,H,E,k", [(3, 256, 24, 2), (16, 4096, 512, 10), (1, 1024, 512, 32),
                                     (7, 768, 64, 6), (16, 2048, 512, 10)])
def test_router_cluster_shapes(M, H, E, k):
    """The small-M cluster router: a partial last expert slice (E 24), the
    largest hidden size with 16 tokens (one ring stage), k = 32, K rows per
    warp that are not a power of two (H 768)."""
    case = _RouteCase(synth.custom("rc", M, H, E, k, 128))
    _check_router(case)
    assert int(case.layer.status.item()) == 0


# ---- plan ------------------------------------------------------------------------------

@pytest.mark.parametrize("wl,M", [(TINY, 8), (TINY, 16), (TINY, 500), (DEC16, 16),
                                  (PRE, 9000)])
def test_plan_bit_exact_given_ids(wl, M):
    case = Case(synth.with_tokens(wl, M))
    ids = synth.random_ids(case.wl, variant=1)
    w = np.full(ids.shape, 1.0 / wl.k, np.float32)
    case.layer.route(case.x_t, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    _check_plan(case, ids)
    assert int(case.layer.status.item()) == 0


@pytest.mark.parametrize("M", [5, 3000])
def test_plan_edge_cases(M):
    wl = synth.custom("edge", M, 256, 64, 4, 128)
    case = Case(wl)
    # all tokens on the same four experts (one hot expert per slot)
    ids = np.tile(np.array([[3, 9, 40, 63]], np.int32), (M, 1))
    w = np.full(ids.shape, 0.25, np.float32)
    case.layer.route(case.x_t, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    _check_plan(case, ids)
    # invalid ids: dropped, flagged
    bad = ids.copy()
    bad[0, 1] = -1
    bad[M - 1, 3] = 64
    case.layer.status.zero_()
    case.layer.route(case.x_t, torch.from_numpy(bad).cuda(), torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    _check_plan(case, bad)
    assert int(case.layer.status.item()) & moe.ST_INVALID_ID


@pytest.mark.parametrize("dup", [False, True])
def test_plan_decode_bucket_repeats_and_invalid(dup):
    """64 pairs in the decode bucket (M 16, k 4) with invalid ids: distinct
    experts per token (the per-expert token-set plan) and an expert repeated
    inside some tokens (the step-by-step plan), bit-exact against the oracle
    plan, work table included."""
    wl = synth.custom("dq", 16, 256, 64, 4, 128)
    case = Case(wl)
    ids = synth.random_ids(wl, variant=4)
    if dup:
        ids[::3, 2] = ids[::3, 0]
    ids[1, 3] = -1
    ids[14, 0] = 64
    w = np.full(ids.shape, 0.25, np.float32)
    case.layer.status.zero_()
    case.layer.route(case.x_t, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    _check_plan(case, ids)
    assert int(case.layer.status.item()) & moe.ST_INVALID_ID


@pytest.mark.parametrize("M", [8, 12, 600])
def test_plan_with_shared_expert(M):
    wl = synth.custom("sh", M, 256, 16, 2, 128, bias="zipf", shared=True)
    case = Case(wl)
    ids = synth.random_ids(wl, variant=2)
    w = np.full(ids.shape, 0.5, np.float32)
    case.layer.route(case.x_t, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    _check_plan(case, ids)


# ---- layer forward -----------------------------------------------------------------------

def _forward_check(case, tokens=None, ids_from_oracle=True):
    if ids_from_oracle:
        y = case.gpu_forward(ids_from_oracle=True)
        ref = case.oracle_forward()
        rel, mx = compare(y, ref)
    else:
        y = case.gpu_forward()
        ref = case.oracle_forward(tokens=tokens)
        rel, mx = compare(y[np.asarray(tokens)], ref)
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, (rel, mx)
    assert int(case.layer.status.item()) == 0
    return y


@pytest.mark.parametrize("M", [1, 3, 8, 16])
def test_forward_tiny_decode(M):
    _forward_check(Case(synth.with_tokens(TINY, M)))


@pytest.mark.parametrize("M", [17, 40, 300, 777])
def test_forward_tiny_prefill(M):
    _forward_check(Case(synth.with_tokens(TINY, M)))


def test_forward_tiny_shared_expert():
    wl = synth.custom("sh", 8, 256, 16, 2, 128, bias="zipf", shared=True)
    _forward_check(Case(wl))
    wl = synth.custom("sh", 200, 256, 16, 2, 128, bias="zipf", shared=True)
    _forward_check(Case(wl))


@pytest.mark.parametrize("M,H,E,k,I", [(4, 512, 16, 2, 1024), (16, 4096, 8, 2, 256),
                                       (40, 512, 16, 2, 1024), (40, 4096, 8, 2, 256)])
def test_forward_other_shapes(M, H, E, k, I):
    """Shapes away from the benchmark: K = I of 16 segments in W2, H = 4096
    (the largest hidden size), decode and prefill buckets."""
    _forward_check(Case(synth.custom("shape", M, H, E, k, I)))


@pytest.fixture(scope="module")
def largest_case():
    """The largest hidden and intermediate sizes the ABI accepts together
    (H = I = 4096: W13 of 8192 x 4096 and W2 of 4096 x 4096 per expert), 8
    experts, top-2, 40 tokens."""
    return Case(synth.custom("max", 40, 4096, 8, 2, 4096))


def _forward_prefix(case, M):
    """Plan + forward of the case's first M tokens with the oracle router's ids."""
    tok = np.arange(M)
    _, ids, w, _ = case.oracle_route(tok)
    xs = case.x_t[:M]
    case.layer.route(xs, torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda(),
                     torch.from_numpy(np.ascontiguousarray(w, np.float32)).cuda())
    y = case.layer.forward_planned(xs)
    torch.cuda.synchronize()
    rel, mx = compare(y.cpu().numpy(), case.oracle_forward(tokens=tok))
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, (rel, mx)
    assert int(case.layer.status.item()) == 0


@pytest.mark.parametrize("M", [16, 40])
def test_forward_largest_sizes(largest_case, M):
    """H = I = 4096 in the decode bucket (the first 16 tokens: 64 K segments
    of W2 per tensor-map copy) and in the grouped GEMMs (32 W2 K steps)."""
    _forward_prefix(largest_case, M)


@pytest.mark.parametrize("M", [16, 40])
def test_forward_top32_every_expert(M):
    """k = 32 = E, the largest top-k: every token uses every expert, so each
    expert holds all M rows (16 per expert in the decode bucket)."""
    _forward_check(Case(synth.custom("k32", M, 256, 32, 32, 512)))


@pytest.mark.parametrize("wl,M", [(TINY, 40), (PRE, 300), (DEC16, 16)])
def test_forward_within_bar_of_both_h_readings(wl, M):
    """The pages leave open whether h is rounded to FP16 between the two
    GEMMs; the kernels round it (kind::f16 operands).  The output also meets
    the acceptance bar against the oracle that keeps h unrounded."""
    case = Case(synth.with_tokens(wl, M))
    y = case.gpu_forward(ids_from_oracle=True)
    _, ids, w, _ = case.oracle_route()
    o13, o2, _ = case.oracle_weights(set(int(e) for e in ids.ravel()))
    ref, st = oracle.forward(case.x, ids, w, o13, o2, h_exact=True)
    rel, mx = compare(y, ref)
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, (rel, mx)
    assert st == 0 and int(case.layer.status.item()) == 0


def test_forward_decode_m1_full():
    _forward_check(Case(DEC1))


def test_forward_decode_m16_full():
    _forward_check(Case(DEC16))


def test_forward_prefill_midsize():
    _forward_check(Case(synth.with_tokens(PRE, 300)))


@pytest.mark.parametrize("wl", [PRE, PRE_Z])
def test_forward_full_prefill_sampled(wl):
    case = Case(wl)
    rng = np.random.default_rng(5)
    tok = np.sort(rng.choice(wl.M, 24, replace=False))
    _forward_check(case, tokens=tok, ids_from_oracle=False)


def test_forward_zero_tokens():
    case = Case(synth.with_tokens(TINY, 8))
    x0 = case.x_t[:0]
    ids, w = case.layer.route(x0)
    y = case.layer.forward_planned(x0)
    assert y.shape == (0, TINY.H)


def test_forward_repeat_bitwise_and_graph_replay():
    case = Case(synth.with_tokens(TINY, 40))
    y1 = case.gpu_forward()
    y2 = case.gpu_forward()
    np.testing.assert_array_equal(y1.view(np.uint16), y2.view(np.uint16))
    # CUDA graph with changing inputs: capture once, replay on new x
    layer = case.layer
    x_static = case.x_t.clone()
    y_static = torch.empty_like(x_static)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer(x_static, y_static)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer(x_static, y_static)
    for variant in (1, 2):
        x_new = torch.from_numpy(synth.activations(case.wl, variant)).cuda()
        x_static.copy_(x_new)
        y_static.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        y_eager = layer(x_new)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(y_static.cpu().numpy().view(np.uint16),
                                      y_eager.cpu().numpy().view(np.uint16))


def test_decode_batch_invariance():
    """Inside the decode bucket a token's output does not depend on its batch:
    M=16 equals two M=8 calls bitwise, through the plan + forward kernels and
    through the fused single-kernel layer call alike."""
    case = Case(synth.with_tokens(DEC16, 16))
    y16 = case.gpu_forward()
    parts = []
    for sl in (slice(0, 8), slice(8, 16)):
        xs = case.x_t[sl].contiguous()
        case.layer.route(xs)
        parts.append(case.layer.forward_planned(xs).cpu().numpy())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y16.view(np.uint16), np.concatenate(parts).view(np.uint16))
    f16 = case.layer(case.x_t).cpu().numpy()
    fparts = [case.layer(case.x_t[sl].contiguous()).cpu().numpy()
              for sl in (slice(0, 8), slice(8, 16))]
    np.testing.assert_array_equal(f16.view(np.uint16), np.concatenate(fparts).view(np.uint16))


@pytest.mark.parametrize("M", [16, 40])
def test_forward_given_repeated_ids(M):
    """Given ids that repeat an expert inside a token (more than 16 rows of one
    expert even in the decode bucket) against the oracle on the same ids."""
    wl = synth.custom("rep", M, 256, 16, 2, 128)
    case = Case(wl)
    ids = np.zeros((M, 2), np.int32)
    ids[:, 0] = 3
    ids[:, 1] = 3
    ids[::3, 1] = 7
    w = np.full(ids.shape, 0.5, np.float32)
    y = case.gpu_forward(ids=ids, w=w)
    ref = case.oracle_forward(ids=ids, w=w)
    rel, mx = compare(y, ref)
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, (rel, mx)


def test_forward_repeated_ids_across_a_tile_boundary():
    """A token whose two pairs of one expert fall on both sides of a 192-row
    plan tile boundary (two W13 / W2 units) against the oracle: token 0
    routes once to expert 3, every other token twice, so expert 3's rows 191
    and 192 belong to token 96."""
    M = 120
    wl = synth.custom("rep_straddle", M, 256, 16, 2, 128)
    case = Case(wl)
    ids = np.full((M, 2), 3, np.int32)
    ids[0, 1] = 7
    w = np.full(ids.shape, 0.5, np.float32)
    y = case.gpu_forward(ids=ids, w=w)
    ref = case.oracle_forward(ids=ids, w=w)
    rel, mx = compare(y, ref)
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, (rel, mx)
    assert int(case.layer.status.item()) == 0


def test_grouped_batch_invariance():
    """On the grouped path a token's output does not depend on the other
    tokens of its call (its pairs are summed in slot order whatever the
    batch, and an MMA column does not depend on the tile's other columns):
    the first 40 tokens of an 80-token call equal the 40-token call bitwise
    (same ids)."""
    case = Case(synth.with_tokens(TINY, 80))
    _, ids, w, _ = case.oracle_route()
    y80 = case.gpu_forward(ids=ids, w=w)
    xs = case.x_t[:40].contiguous()
    case.layer.route(xs, torch.from_numpy(np.ascontiguousarray(ids[:40])).cuda(),
                     torch.from_numpy(np.ascontiguousarray(w[:40])).cuda())
    y40 = case.layer.forward_planned(xs).cpu().numpy()
    np.testing.assert_array_equal(y80[:40].view(np.uint16), y40.view(np.uint16))


@pytest.mark.parametrize("M", [1, 8, 16])
def test_forward_grouped_bucket_at_small_m(M):
    """Below the crossover the grouped tensor-core path also meets the bar
    (the M bucket only picks the faster path): the decode bucket lowered to
    0 sends M <= 16 through the grouped GEMMs on the small-M plan."""
    case = Case(synth.with_tokens(DEC16, M))
    moe.set_decode_max_tokens(0)
    try:
        y = case.gpu_forward(ids_from_oracle=True)
    finally:
        moe.set_decode_max_tokens(16)
    rel, mx = compare(y, case.oracle_forward())
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, (rel, mx)
    assert int(case.layer.status.item()) == 0


def test_query_plan_bytes_cover_every_smaller_m():
    """The plan size the query returns for max_tokens covers every M up to it:
    the split router's partial logits make the per-M layout non-monotonic
    (M = 127 needs more than M = 128, where the tensor-core router runs)."""
    for E in (512, 136):
        cfg = moe.make_config(2048, E, 10, 512)
        top = {n: moe.query(cfg, n)[0] for n in (128, 784, 8192)}
        for M in (1, 16, 17, 64, 65, 100, 127, 128, 300, 784):
            pb = moe.query(cfg, M)[0]
            for n, v in top.items():
                if M <= n:
                    assert pb <= v, (E, M, n, pb, v)


def test_layer_repeated_calls_match_the_checked_call():
    """MoELayer's repeated calls (the call's fixed C arguments built once,
    after a fully checked call) give the bits of moe.layer with every check,
    for other token counts too, and rebuild their arguments when the layer's
    buffers or weights are replaced."""
    case = Case(synth.with_tokens(TINY, 24))
    L = case.layer
    x = case.x_t

    def checked(xx):
        M = xx.shape[0]
        y = torch.empty_like(xx)
        ids = torch.empty((M, L.k), dtype=torch.int32, device="cuda")
        tw = torch.empty((M, L.k), dtype=torch.float32, device="cuda")
        moe.layer(L.cfg, xx, L.w_router, L.bias, L.w_gate, ids, tw, L.plan_buf, L.w13, L.w2,
                  L.shared13, L.shared2, y, L.ws, L.status)
        torch.cuda.synchronize()
        return y.cpu().numpy(), ids.cpu().numpy()

    def same(a, b):
        np.testing.assert_array_equal(a.view(np.uint16), b.view(np.uint16))

    ref, ref_ids = checked(x)
    for _ in range(3):  # the first call is checked in full, the others take the short path
        y = L(x)
        torch.cuda.synchronize()
        same(y.cpu().numpy(), ref)
        np.testing.assert_array_equal(L.last_ids.cpu().numpy(), ref_ids)
    assert L._fast is not None
    x8 = x[:8].contiguous()
    ref8, _ = checked(x8)
    same(L(x8).cpu().numpy(), ref8)
    # larger buffers, then another copy of the weights: the arguments follow
    L.reserve(256)
    same(L(x).cpu().numpy(), ref)
    L.w13 = tuple(t.clone() for t in L.w13)
    L.w2 = tuple(t.clone() for t in L.w2)
    same(L(x).cpu().numpy(), ref)
    assert L._fast[0][0] is L.w13
    assert int(L.status.item()) == 0
