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
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(moe_nvfp4_\w+)\(", text, re.M)))


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
