"""Failure paths and buffer hygiene on the GPU, without faulting it.

  * a bounded wait that runs out: the grouped W13 kernel's raw-weight producer
    is held back (test switch), its consumers give up after a short limit,
    set MOE_ST_TIMEOUT, drain, free tensor memory and return; the next call on
    the same context is correct again;
  * poisoned buffers: the plan buffer (past its counters) and the workspace
    filled with NaN bytes before a call change nothing (every location a call
    reads is written first in that call);
  * canaries: bytes past y, past the workspace and past the plan buffer are
    left untouched.

Pages: "[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency", section "Test
Result" (poisoned outputs and tail canaries in the native gate; an unsafe
launch falls back safely; poisoned buffers in the grouped-MoE tests).
"""
import numpy as np
import pytest
import torch

from harness import MAX_ABS_TOL, REL_L2_TOL, Case, compare
from nvfp4_weight_mixture_gb300 import moe, synth

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny_m8"]
DEC1 = synth.WORKLOADS["decode_m1"]
PRE = synth.WORKLOADS["prefill_m8192"]
PLAN_COUNTERS = 512   # plan header and arrival counters: zero between calls


def test_grouped_wait_timeout_sets_status_and_recovers():
    case = Case(synth.with_tokens(TINY, 40))
    layer = case.layer
    ref = case.oracle_forward()
    layer.route(case.x_t)
    torch.cuda.synchronize()
    layer.status.zero_()
    moe.set_wait_test(True, 2_000_000)          # ~1 ms instead of ~200 ms
    try:
        layer.forward_planned(case.x_t)
        torch.cuda.synchronize()
    finally:
        moe.set_wait_test(False, 0)
    assert int(layer.status.item()) & moe.ST_TIMEOUT
    # the context is still usable: the same call is correct again
    layer.status.zero_()
    y = layer(case.x_t)
    torch.cuda.synchronize()
    rel, mx = compare(y.cpu().numpy(), ref)
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, (rel, mx)
    assert int(layer.status.item()) == 0


@pytest.mark.parametrize("wl", [DEC1, synth.with_tokens(TINY, 40), synth.with_tokens(PRE, 300),
                                synth.custom("sh", 12, 256, 16, 2, 128, bias="zipf",
                                             shared=True)],
                         ids=["decode_m1", "tiny_m40", "prefill_m300", "shared_m12"])
def test_poisoned_buffers_and_canaries(wl):
    case = Case(wl)
    layer = case.layer
    M, H = wl.M, wl.H
    ref = case.oracle_forward()
    pb, wb = moe.query(layer.cfg, M)
    canary = 0xA5
    # plan buffer and workspace with canary tails; their own bytes NaN-poisoned
    plan_big = torch.full((pb + 4096,), canary, dtype=torch.uint8, device="cuda")
    plan_big[:PLAN_COUNTERS] = 0
    plan_big[PLAN_COUNTERS:pb] = 0xFF
    ws_big = torch.full((wb + 4096,), canary, dtype=torch.uint8, device="cuda")
    ws_big[:wb] = 0xFF
    y_big = torch.full(((M + 2) * H,), float("nan"), dtype=torch.float16, device="cuda")
    y_big[M * H:] = 1234.0
    plan_v, ws_v, y_v = plan_big[:pb], ws_big[:wb], y_big[:M * H].view(M, H)
    ids = torch.empty((M, wl.k), dtype=torch.int32, device="cuda")
    tw = torch.empty((M, wl.k), dtype=torch.float32, device="cuda")
    layer.status.zero_()
    moe.layer(layer.cfg, case.x_t, layer.w_router, layer.bias, layer.w_gate, ids, tw, plan_v,
              layer.w13, layer.w2, layer.shared13, layer.shared2, y_v, ws_v, layer.status)
    torch.cuda.synchronize()
    rel, mx = compare(y_v.cpu().numpy(), ref)
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, (rel, mx)
    assert int(layer.status.item()) == 0
    assert bool((plan_big[pb:] == canary).all())
    assert bool((ws_big[wb:] == canary).all())
    assert bool((y_big[M * H:] == 1234.0).all())
    # the arrival counters are left at zero for the next call
    assert bool((plan_big[256:PLAN_COUNTERS] == 0).all())
