"""moe_nvfp4_forward_noalloc: the forward for callers that cannot allocate.

Some callers have no way to hand the layer a device workspace: code running
inside a host runtime or plugin that owns every device allocation and gives
its extensions no allocator, code that runs while a framework forbids new
allocations, or C code behind a fixed signature with no workspace argument.
For them the library keeps a fixed 4 MiB workspace of its own.  These tests
call that entry point through the C ABI and check it against
moe_nvfp4_forward (the caller-workspace entry point) on two calls in a row.
Both run the same kernels on the same plan, so the outputs must be equal bit
for bit (a looser tolerance could hide a workspace-aliasing fault that
perturbs a few rows).  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from harness import Case
from nvfp4_weight_mixture_gb300 import moe, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl", [synth.with_tokens(synth.WORKLOADS["tiny_m8"], 8),
                                synth.WORKLOADS["decode_m1"],
                                synth.WORKLOADS["decode_m16_bias"],
                                synth.custom("sh", 12, 256, 16, 2, 128, bias="zipf", shared=True),
                                # small layers reach the grouped (prefill) kernels too
                                synth.with_tokens(synth.WORKLOADS["tiny_m8"], 64),
                                synth.custom("sh", 256, 256, 16, 2, 128, bias="zipf",
                                             shared=True)],
                         ids=["tiny_m8", "decode_m1", "decode_m16", "shared_m12",
                              "tiny_m64_grouped", "shared_m256_grouped"])
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
        np.testing.assert_array_equal(y.cpu().numpy().view(np.uint16),
                                      y_ref.cpu().numpy().view(np.uint16))
        assert int(st.item()) == 0 and int(layer.status.item()) == 0


def test_noalloc_rejects_oversize_and_launches_nothing():
    """A call beyond the fixed workspace returns MOE_ERR_WORKSPACE.  Every
    buffer argument is NULL, so even if the size gate ever let the call
    through, the host-side argument checks would refuse it (MOE_ERR_INVALID_ARG)
    instead of launching kernels on made-up addresses."""
    wl = synth.with_tokens(synth.WORKLOADS["prefill_m8192"], 512)
    cfg = moe.make_config(wl.H, wl.E, wl.k, wl.I)
    lib = moe.load_library()
    R = ctypes.byref
    # 512 tokens x top-10 needs far more than the static workspace
    rc = lib.moe_nvfp4_forward_noalloc(R(cfg), 512, None, None, None, None, None, None, None,
                                       None, None)
    assert rc == -4
    assert lib.moe_nvfp4_forward_noalloc(R(cfg), 0, None, None, None, None, None, None, None,
                                         None, None) == 0
    # within the size limit, NULL buffers are refused before any launch
    rc = lib.moe_nvfp4_forward_noalloc(R(cfg), 1, None, None, None, None, None, None, None,
                                       None, None)
    assert rc == -1
