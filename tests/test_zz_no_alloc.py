"""moe_nvfp4_forward_noalloc: the forward for callers that cannot allocate.

Those callers (a host runtime that owns every device allocation, a phase in
which allocation is forbidden, a fixed C signature without a workspace) get
an entry point whose workspace is a static array inside the library.  These
tests call it through the C ABI and check it against moe_nvfp4_forward, the
entry point with a caller-provided workspace, on two calls in a row.  This
file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from harness import MAX_ABS_TOL, REL_L2_TOL, Case, compare
from nvfp4_weight_mixture_gb300 import moe, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl", [synth.with_tokens(synth.WORKLOADS["tiny_m8"], 8),
                                synth.WORKLOADS["decode_m1"],
                                synth.WORKLOADS["decode_m16_bias"],
                                synth.custom("sh", 12, 256, 16, 2, 128, bias="zipf", shared=True)])
def test_noalloc_matches_forward_twice(wl):
    case = Case(wl)
    layer = case.layer
    for variant in (0, 1):            # two calls in a row, different inputs
        x = torch.from_numpy(synth.activations(wl, variant)).cuda()
        layer.route(x)
        y_ref = layer.forward_planned(x)
        y = torch.full_like(y_ref, float("nan"))
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        moe.forward_noalloc(layer.cfg, x, layer.plan_buf, layer.w13, layer.w2, layer.shared13,
                            layer.shared2, y, st)
        torch.cuda.synchronize()
        a, b = y.cpu().numpy(), y_ref.cpu().numpy()
        rel, mx = compare(a, b)
        assert rel <= REL_L2_TOL and mx <= MAX_ABS_TOL, (variant, rel, mx)
        assert int(st.item()) == 0


def test_noalloc_rejects_oversize_and_launches_nothing():
    wl = synth.with_tokens(synth.WORKLOADS["prefill_m8192"], 512)
    cfg = moe.make_config(wl.H, wl.E, wl.k, wl.I)
    lib = moe.load_library()
    a = ctypes.c_void_p(0x10000)
    w13 = moe.WeightsC(0x10000, 0x10000, 0x10000, moe.LAYOUT_FRAGMENT_W13, 0)
    w2 = moe.WeightsC(0x10000, 0x10000, 0x10000, moe.LAYOUT_FRAGMENT, 0)
    R = ctypes.byref
    # 512 tokens x top-10 needs far more than the static workspace
    rc = lib.moe_nvfp4_forward_noalloc(R(cfg), 512, a, a, R(w13), R(w2), None, None, a, None,
                                       None)
    assert rc == -4
    assert lib.moe_nvfp4_forward_noalloc(R(cfg), 0, None, None, None, None, None, None, None,
                                         None, None) == 0
