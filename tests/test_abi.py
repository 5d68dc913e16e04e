"""The C-ABI library: loads, exports every declared entry point, and fails
closed on bad arguments before touching a GPU (no compute call needs one)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_nvfp4.h")


@pytest.fixture(scope="module")
def lib():
    from nvfp4_weight_mixture_gb300 import build, moe
    build.build()
    return moe.load_library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(moe_\w+)\(", text, re.M)))


def test_exports_every_declared_symbol(lib):
    syms = declared_symbols()
    assert len(syms) >= 7, syms
    for s in syms:
        assert hasattr(lib, s), s
    from nvfp4_weight_mixture_gb300 import moe
    assert set(moe.EXPORTS) <= set(syms)


def test_abi_version_and_status_strings(lib):
    from nvfp4_weight_mixture_gb300 import moe
    assert lib.moe_nvfp4_abi_version() == moe.ABI_VERSION == 1
    for code in list(moe.ERR) + [0, 1, 2, 4]:
        s = moe.status_string(code)
        assert s and s != "unknown code"
    assert moe.status_string(12345) == "unknown code"
    # no call on this thread has failed in CUDA: the error name is empty
    assert lib.moe_nvfp4_last_cuda_error() == b""


def _cfg(H=2048, E=512, k=10, I=512, flags=0):
    from nvfp4_weight_mixture_gb300 import moe
    c = moe.make_config(H, E, k, I)
    c.flags = flags
    return c


def test_query_validates_config_without_device(lib):
    q = lambda c, m=16: lib.moe_nvfp4_query(ctypes.byref(c), m, None, None)
    assert q(_cfg()) == 0
    assert q(_cfg(H=100)) == -2
    assert q(_cfg(H=8192)) == -2
    assert q(_cfg(E=12)) == -2
    assert q(_cfg(E=1024)) == -2
    assert q(_cfg(k=0)) == -2
    assert q(_cfg(k=33)) == -2
    assert q(_cfg(I=96)) == -2
    assert q(_cfg(flags=0x80)) == -1
    c = _cfg()
    c.reserved[1] = 3
    assert q(c) == -1
    assert q(_cfg(), -1) == -2
    assert lib.moe_nvfp4_query(None, 1, None, None) == -1


def test_plan_and_forward_fail_closed(lib):
    from nvfp4_weight_mixture_gb300 import moe
    P = ctypes.c_void_p
    a = P(0x10000)        # aligned dummy pointers: never dereferenced on these paths
    odd = P(0x10004)
    c = _cfg()
    plan = lib.moe_nvfp4_plan
    # M = 0 with valid arguments: OK, nothing launched, no device needed
    assert plan(ctypes.byref(c), 0, a, a, None, None, a, a, a, 1 << 20, None, None) == 0
    assert plan(ctypes.byref(c), 0, None, None, None, None, None, None, None, 0, None, None) == 0
    assert plan(ctypes.byref(c), 1, None, a, None, None, a, a, a, 1 << 20, None, None) == -1
    assert plan(ctypes.byref(c), 1, odd, a, None, None, a, a, a, 1 << 20, None, None) == -3
    assert plan(ctypes.byref(c), 1, a, a, None, None, a, a, a, 16, None, None) == -4
    assert plan(ctypes.byref(c), -1, a, a, None, None, a, a, a, 1 << 20, None, None) == -2
    cs = _cfg(flags=moe.FLAG_SHARED)
    assert plan(ctypes.byref(cs), 1, a, a, None, None, a, a, a, 1 << 20, None, None) == -1
    fwd = lib.moe_nvfp4_forward
    w13 = moe.WeightsC(0x10000, 0x10000, 0x10000, moe.LAYOUT_FRAGMENT_W13, 0)
    w2 = moe.WeightsC(0x10000, 0x10000, 0x10000, moe.LAYOUT_FRAGMENT, 0)
    bad = moe.WeightsC(0x10000, 0x10000, 0x10000, moe.LAYOUT_CANONICAL, 0)
    R = ctypes.byref
    assert fwd(R(c), 0, a, a, R(w13), R(w2), None, None, a, a, 1 << 30, None, None) == 0
    assert fwd(R(c), 4, a, a, R(bad), R(w2), None, None, a, a, 1 << 30, None, None) == -7
    assert fwd(R(c), 4, a, a, R(w13), R(w13), None, None, a, a, 1 << 30, None, None) == -7
    assert fwd(R(c), 4, a, a, R(w13), R(w2), None, None, a, a, 64, None, None) == -4
    assert fwd(R(cs), 4, a, a, R(w13), R(w2), None, None, a, a, 1 << 30, None, None) == -1
    assert fwd(R(c), 4, a, a, None, R(w2), None, None, a, a, 1 << 30, None, None) == -1


def test_quantize_fail_closed(lib):
    P = ctypes.c_void_p
    a = P(0x10000)
    qz = lib.moe_nvfp4_quantize
    assert qz(a, 1, 16, 60, 0, a, a, a, None, None) == -2     # k % 64
    assert qz(a, 1, 8, 64, 0, a, a, a, None, None) == -2      # rows % 16
    assert qz(a, 1, 16, 64, 2, a, a, a, None, None) == -2     # W13 layout needs rows % 32
    assert qz(a, 1, 16, 64, 5, a, a, a, None, None) == -7
    assert qz(None, 1, 16, 64, 0, a, a, a, None, None) == -1
    assert qz(P(0x10008), 1, 16, 64, 0, a, a, a, None, None) == -3


def test_binding_checks_sizes_the_abi_cannot_see():
    """The C ABI takes plain pointers, so the binding checks every tensor's
    dtype and element count against the configuration before a call (CPU
    tensors stand in: only metadata is read)."""
    import torch
    from nvfp4_weight_mixture_gb300 import moe
    H, E, k, I, M = 256, 16, 2, 128, 5
    c = moe.make_config(H, E, k, I)
    f16, f32, i32, u8 = torch.float16, torch.float32, torch.int32, torch.uint8
    x = torch.zeros(M, H, dtype=f16)
    ok = dict(x=x, w_router=torch.zeros(H, E, dtype=f16), bias=torch.zeros(E, dtype=f32),
              w_gate=torch.zeros(H, dtype=f16), ids=torch.zeros(M, k, dtype=i32),
              topk_w=torch.zeros(M, k, dtype=f32), status=torch.zeros(1, dtype=i32))
    assert moe.plan_arg_errors(c, **ok) == []
    assert moe.plan_arg_errors(c, **dict(ok, w_router=None, bias=None, w_gate=None)) == []
    assert moe.plan_arg_errors(c, **dict(ok, x=x[:0], ids=ok["ids"][:0],
                                          topk_w=ok["topk_w"][:0])) == []
    for name, bad in (("ids", torch.zeros(M, k + 1, dtype=i32)),
                      ("ids", torch.zeros(M, k, dtype=torch.int64)),
                      ("topk_w", torch.zeros(M - 1, k, dtype=f32)),
                      ("w_router", torch.zeros(E, H - 8, dtype=f16)),
                      ("bias", torch.zeros(E, dtype=f16)),
                      ("w_gate", torch.zeros(H + 1, dtype=f16)),
                      ("x", torch.zeros(M, H // 2, dtype=f16)),
                      ("status", torch.zeros(1, dtype=f32))):
        errs = moe.plan_arg_errors(c, **dict(ok, **{name: bad}))
        assert errs and errs[0].startswith(name), (name, errs)

    def weights(rows, kk, n):
        return (torch.zeros(n, rows * kk // 2, dtype=u8), torch.zeros(n, rows * kk // 16, dtype=u8),
                torch.zeros(n, dtype=f32))
    w13, w2 = weights(2 * I, H, E), weights(H, I, E)
    fok = dict(x=x, w13=w13, w2=w2, shared13=None, shared2=None, y=torch.zeros(M, H, dtype=f16))
    assert moe.forward_arg_errors(c, **fok) == []
    assert moe.forward_arg_errors(c, **dict(fok, shared13=weights(2 * I, H, 1),
                                            shared2=weights(H, I, 1))) == []
    for name, bad, prefix in (("y", torch.zeros(M - 1, H, dtype=f16), "y"),
                              ("y", torch.zeros(M, H, dtype=f32), "y"),
                              ("w13", weights(2 * I, H, E - 1), "w13.q"),
                              ("w2", weights(2 * I, H, E), "w2.q"),
                              ("w2", (w2[0], w2[1], torch.zeros(E, dtype=f16)), "w2.g"),
                              ("shared2", weights(H, I, 2), "shared2.q")):
        errs = moe.forward_arg_errors(c, **dict(fok, **{name: bad}))
        assert errs and errs[0].startswith(prefix), (name, errs)
    # dequantise: codes and scales of n_mats x rows x k
    q, s = torch.zeros(2 * 256 * 64 // 2, dtype=u8), torch.zeros(2 * 256 * 64 // 16, dtype=u8)
    assert moe.dequantize_arg_errors(q, s, 2, 256, 64) == []
    assert moe.dequantize_arg_errors(q[:-1], s, 2, 256, 64)[0].startswith("q")
    assert moe.dequantize_arg_errors(q, s, 2, 256, 128)[0].startswith("q")


def test_small_router_switch_validates_mode(lib):
    """The diagnostic router switch accepts modes 0 and 1 only (host-only)."""
    assert lib.moe_nvfp4_set_small_router(2) == -1
    assert lib.moe_nvfp4_set_small_router(-1) == -1
    assert lib.moe_nvfp4_set_small_router(1) == 0
    assert lib.moe_nvfp4_set_small_router(0) == 0


def test_dense_query_shapes_without_device(lib):
    """The dense query is host-only arithmetic: shape gates and the workspace
    size, which is 0 for every shape (each block owns whole output tiles over
    all of K, so nothing is added up between blocks)."""
    wb = ctypes.c_size_t(7)
    R = ctypes.byref
    assert lib.moe_nvfp4_dense_query(16, 8704, 5120, R(wb)) == 0 and wb.value == 0
    wb.value = 7
    assert lib.moe_nvfp4_dense_query(32, 65536, 65536, R(wb)) == 0 and wb.value == 0
    assert lib.moe_nvfp4_dense_query(0, 8704, 5120, R(wb)) == 0 and wb.value == 0
    assert lib.moe_nvfp4_dense_query(33, 8704, 5120, R(wb)) == -2   # M above the path
    assert lib.moe_nvfp4_dense_query(8, 8704 + 16, 5120, R(wb)) == -2
    assert lib.moe_nvfp4_dense_query(8, 8704, 5120 + 32, R(wb)) == -2
    assert lib.moe_nvfp4_dense_query(8, 8704, 5120, None) == -1


def test_dense_entry_points_fail_closed_without_device(lib):
    """Argument checks come before any device use: NULL buffers, bad layouts
    and M = 0 are answered on the host."""
    from nvfp4_weight_mixture_gb300 import moe
    R = ctypes.byref
    w = moe.WeightsC(None, None, None, moe.LAYOUT_FRAGMENT, 0)
    assert lib.moe_nvfp4_dense(0, 256, 64, None, R(w), None, None, 0, None, None) == 0
    assert lib.moe_nvfp4_dense(4, 256, 64, None, R(w), None, None, 0, None, None) == -1
    w.layout = moe.LAYOUT_FRAGMENT_W13
    assert lib.moe_nvfp4_dense(4, 256, 64, None, R(w), None, None, 0, None, None) == -7
    assert lib.moe_fp8_dense(4, 256, 64, None, None, None, None, None, 0, None, None) == -1
    assert lib.moe_fp8_quantize(None, 256, 64, 3, None, None, None, None) == -1
    assert lib.moe_nvfp4_prepare_scales(None, 0, None, None, None) == 0
    assert lib.moe_nvfp4_prepare_scales(None, 16, None, None, None) == -1


def test_decode_bucket_switch_validates(lib):
    """The diagnostic decode-bucket switch accepts 0..16 only (host-only)."""
    assert lib.moe_nvfp4_set_decode_max_tokens(17) == -1
    assert lib.moe_nvfp4_set_decode_max_tokens(-1) == -1
    assert lib.moe_nvfp4_set_decode_max_tokens(0) == 0
    assert lib.moe_nvfp4_set_decode_max_tokens(16) == 0

