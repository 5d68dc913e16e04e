"""Prepared-scale storage on the layer forward: the same layer with its E4M3
block scales widened once, at load time, to FP16 (moe_nvfp4_prepare_scales,
MOE_SCALES_PREPARED) gives bitwise the raw-scale output, through the decode
kernels (M = 1..16) and the grouped tcgen05 GEMMs (M = 784 and others), on the
same plan ("[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency", section "Test
Result": raw and prepared outputs bitwise equal at M1-M16 and M784)."""
import numpy as np
import pytest
import torch

from harness import MAX_ABS_TOL, REL_L2_TOL, Case, compare
from nvfp4_weight_mixture_gb300 import moe, synth

pytestmark = pytest.mark.gpu

DEC16 = synth.WORKLOADS["decode_m16_bias"]
PRE = synth.WORKLOADS["prefill_m8192"]
TINY = synth.WORKLOADS["tiny_m8"]


def _prepared(w):
    if w is None:
        return None
    q, s, g = w
    return (q, moe.prepare_scales(s), g)


def _both(case, x):
    """Routes x on the GPU once, then runs the forward with raw and with
    prepared scales on that plan."""
    layer = case.layer
    layer.route(x)
    y_raw = layer.forward_planned(x)
    y_prep = torch.empty_like(y_raw)
    moe.forward(layer.cfg, x, layer.plan_buf, _prepared(layer.w13), _prepared(layer.w2),
                _prepared(layer.shared13), _prepared(layer.shared2), y_prep, layer.ws,
                layer.status)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    return y_raw.cpu().numpy(), y_prep.cpu().numpy()


def test_prepared_bitwise_equal_raw_m1_to_m16():
    case = Case(DEC16)
    for M in range(1, 17):
        xs = case.x_t[:M].contiguous()
        a, b = _both(case, xs)
        np.testing.assert_array_equal(a.view(np.uint16), b.view(np.uint16), err_msg=str(M))


@pytest.mark.parametrize("wl,M", [(PRE, 784), (TINY, 300), (TINY, 17)])
def test_prepared_bitwise_equal_raw_grouped(wl, M):
    case = Case(synth.with_tokens(wl, M))
    a, b = _both(case, case.x_t)
    np.testing.assert_array_equal(a.view(np.uint16), b.view(np.uint16))


@pytest.mark.parametrize("M", [12, 200])
def test_prepared_with_shared_expert_vs_oracle(M):
    wl = synth.custom("sh", M, 256, 16, 2, 128, bias="zipf", shared=True)
    case = Case(wl)
    a, b = _both(case, case.x_t)
    np.testing.assert_array_equal(a.view(np.uint16), b.view(np.uint16))
    rel, mx = compare(b, case.oracle_forward())
    assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, (rel, mx)


def test_mixed_scale_storage_is_refused():
    case = Case(synth.with_tokens(TINY, 4))
    layer = case.layer
    layer.route(case.x_t)
    y = torch.empty((4, TINY.H), dtype=torch.float16, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        moe.forward(layer.cfg, case.x_t, layer.plan_buf, _prepared(layer.w13), layer.w2, None,
                    None, y, layer.ws, layer.status)
    assert ei.value.code == -7
