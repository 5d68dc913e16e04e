"""The decode call exactly as a serving step (and the bench) makes it: the
router and plan on the GPU (no given ids), then the decode forward.

For M <= 16 the plan call runs the small-M router, which also writes the
plan and the decode work table: a thread-block cluster where the device can
co-schedule one, else the 128-block router with arrival tickets (forced here
through the diagnostic switch).  Both are compared with the oracle on the
same seeded inputs, and nothing the GPU computes is fed to the oracle:

  * ids: top-k sets agree except where the oracle's k / k+1 gap is < 1e-5
    (the seeds below have no such token, so the id arrays must be equal);
  * the plan (counts, offsets, perm, inv, tiles, active list) is bit-exact
    against the oracle plan of the oracle's ids, and the decode work table
    equals the one that oracle plan implies;
  * y (GPU-routed) is within rel-L2 1e-3 / max-abs 2e-2 of the oracle's
    own routed layer.

Pages: "[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency", sections "Scope
and related PRs" (one integer plan shared by W13 and W2) and "Test Result"
(M1-M16 changing-route graph replay).
"""
import numpy as np
import pytest
import torch

import oracle
from harness import (MAX_ABS_TOL, REL_L2_TOL, ROUTER_GAP, ROUTER_W_TOL, TILE_ROWS, Case,
                     compare, expected_tile_pos, expected_work_table)
from nvfp4_weight_mixture_gb300 import moe, synth

pytestmark = pytest.mark.gpu

DEC1 = synth.WORKLOADS["decode_m1"]
DEC16 = synth.WORKLOADS["decode_m16_bias"]
TINY = synth.WORKLOADS["tiny_m8"]

CASES = [
    ("decode_m1", DEC1),
    ("decode_m16_bias_m9", synth.with_tokens(DEC16, 9)),
    ("decode_m16_bias", DEC16),
    ("tiny_m8", TINY),
    ("tiny_shared_m12", synth.custom("sh", 12, 256, 16, 2, 128, bias="zipf", shared=True)),
]


@pytest.fixture(params=["cluster", "ticket"])
def router_mode(request):
    moe.set_small_router(request.param == "ticket")
    yield request.param
    moe.set_small_router(False)


_cases = {}


def _case(name, wl):
    if name not in _cases:
        _cases[name] = Case(wl)
    return _cases[name]


def _oracle_ids_eff(wl, ids):
    if wl.shared:
        return np.concatenate([ids, np.full((wl.M, 1), wl.E, np.int32)], 1)
    return ids


@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_gpu_routed_decode_vs_oracle(router_mode, name, wl):
    case = _case(name, wl)
    layer = case.layer
    layer.status.zero_()
    ids_g, w_g = case.gpu_route()
    logits, ids_o, w_o, gamma_o = case.oracle_route()
    k = wl.k
    # ---- router: the seeds leave no near-tie, so the ids are equal ----
    for t in range(wl.M):
        srt = np.sort(logits[t])[::-1]
        assert srt[k - 1] - srt[k] >= ROUTER_GAP, (t, "seed has a near-tie; pick another")
    np.testing.assert_array_equal(ids_g, ids_o)
    assert np.max(np.abs(w_g - w_o)) <= ROUTER_W_TOL
    # ---- plan and decode work table: bit-exact against the oracle plan ----
    k_eff, e_eff = k + int(wl.shared), wl.E + int(wl.shared)
    ids_eff = _oracle_ids_eff(wl, ids_o)
    ref = oracle.plan(ids_eff, e_eff, TILE_ROWS)
    got = case.plan_arrays()
    np.testing.assert_array_equal(got["ids"], ids_eff.reshape(-1))
    for key in ("counts", "offsets", "perm", "inv", "tiles"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    np.testing.assert_array_equal(got["tile_pos"], expected_tile_pos(ref))
    np.testing.assert_array_equal(got["active"], np.nonzero(ref["counts"])[0])
    assert int(got["hdr"][0]) == wl.M and int(got["hdr"][1]) == k_eff
    assert int(got["hdr"][3]) == len(np.nonzero(ref["counts"])[0])
    assert int(got["hdr"][4]) == len(ref["tiles"])
    exp_tab = expected_work_table(ref, wl.M, k_eff, e_eff)
    np.testing.assert_array_equal(got["dtab"][:len(exp_tab)], exp_tab)
    if wl.shared:
        # the shared slot's weight is the gate gamma = sigmoid(x . w_g)
        g_gpu = got["w"].reshape(wl.M, k_eff)[:, k]
        assert np.max(np.abs(g_gpu - gamma_o)) <= ROUTER_W_TOL
    # ---- the layer output of the GPU-routed call vs the oracle's routed layer ----
    y = layer.forward_planned(case.x_t)
    torch.cuda.synchronize()
    rel, mx = compare(y.cpu().numpy(), case.oracle_forward())
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, (rel, mx)
    assert int(layer.status.item()) == 0


@pytest.mark.parametrize("M", [1, 5, 16])
def test_ticket_router_matches_cluster_router(M):
    """The two small-M routers sum the logits in different orders, so their
    weights may differ in the last bits (within 1e-5), but on these seeds
    (no near-tie) their ids, plans and work tables are identical."""
    wl = synth.with_tokens(DEC16, M)
    case = _case(f"dec16_m{M}", wl)
    out = {}
    for mode in (False, True):
        moe.set_small_router(mode)
        try:
            ids, w = case.gpu_route()
            out[mode] = (ids, w, case.plan_arrays())
        finally:
            moe.set_small_router(False)
    np.testing.assert_array_equal(out[False][0], out[True][0])
    assert np.max(np.abs(out[False][1] - out[True][1])) <= ROUTER_W_TOL
    for key in ("counts", "offsets", "perm", "inv", "tiles", "tile_pos", "active", "dtab"):
        np.testing.assert_array_equal(out[False][2][key], out[True][2][key], err_msg=key)


def test_gpu_routed_decode_graph_replay_changing_routes():
    """One CUDA graph of plan + forward (GPU routing), replayed on new token
    batches: each replay's output equals the oracle's routed layer for that
    batch (the routes change from batch to batch)."""
    wl = DEC16
    case = _case("decode_m16_bias", wl)
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
    for variant in (3, 4):
        xv = synth.activations(wl, variant)
        x_static.copy_(torch.from_numpy(xv).cuda())
        y_static.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        logits, ids, w = oracle.router(xv, case.wr, case.bias, wl.k)
        srt = -np.sort(-logits, axis=1)
        clear = srt[:, wl.k - 1] - srt[:, wl.k] >= ROUTER_GAP  # tokens without a near-tie
        assert clear.sum() >= wl.M - 1
        used = set(int(e) for e in ids.ravel())
        o13, o2, _ = case.oracle_weights(used)
        ref, st = oracle.forward(xv, ids, w, o13, o2)
        rel, mx = compare(y_static.cpu().numpy()[clear], ref[clear])
        assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, (variant, rel, mx)
    assert int(layer.status.item()) == 0
