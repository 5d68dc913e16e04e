"""CPU oracle of the NVFP4-weight MoE layer (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the bench's ``cpu_baseline``
leg use this package.  The product path (the CUDA library and its Python
binding) never imports it.  The arithmetic lives in ``oracle.c``, a plain C
restatement of the method, built here with gcc (``-O2 -fopenmp
-ffp-contract=off``, no fast-math, no ``-march``); this module only marshals
numpy arrays into it.

Citations are to the pages by title and section:
"[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency", section "Scope and
related PRs" (the layer and its steps) and section "Test Plan" (the codec
edge cases).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ST_INVALID_ID = 0x1
ST_NONFINITE = 0x2


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` beside it (if stale)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_double.restype = ctypes.c_double
        lib.oracle_f16_from_double.argtypes = [ctypes.c_double]
        lib.oracle_f16_from_double.restype = ctypes.c_uint16
        lib.oracle_e2m1_value.argtypes = [ctypes.c_int]
        lib.oracle_e2m1_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_int]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
        lib.oracle_e2m1_encode.restype = ctypes.c_int
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_int
        lib.oracle_dequant_f16.argtypes = [ctypes.c_int, ctypes.c_int]
        lib.oracle_dequant_f16.restype = ctypes.c_uint16
        lib.oracle_quantize.argtypes = [P, I64, I64, I64, P, P, P]
        lib.oracle_quantize.restype = ctypes.c_uint32
        lib.oracle_dequant.argtypes = [P, P, I64, I64, P]
        lib.oracle_dequant.restype = None
        lib.oracle_router.argtypes = [P, P, P, I64, I64, I64, I64, P, P, P]
        lib.oracle_router.restype = None
        lib.oracle_shared_gate.argtypes = [P, P, I64, I64, P]
        lib.oracle_shared_gate.restype = None
        lib.oracle_plan.argtypes = [P, I64, I64, I64, P, P, P, P, P, I64,
                                    ctypes.POINTER(ctypes.c_int64)]
        lib.oracle_plan.restype = ctypes.c_uint32
        lib.oracle_forward.argtypes = [I64] * 5 + [P] * 15 + [P, P, I64, ctypes.c_int, P, P]
        lib.oracle_forward.restype = ctypes.c_uint32
        lib.oracle_dense.argtypes = [I64, I64, I64, P, P, P, ctypes.c_float, P]
        lib.oracle_dense.restype = None
        lib.oracle_prepare_scales.argtypes = [P, I64, P]
        lib.oracle_prepare_scales.restype = ctypes.c_uint32
        lib.oracle_fp8_quantize.argtypes = [P, I64, I64, P, P]
        lib.oracle_fp8_quantize.restype = ctypes.c_uint32
        lib.oracle_fp8_dense.argtypes = [I64, I64, I64, P, P, P, P]
        lib.oracle_fp8_dense.restype = None
        _lib = lib
        return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _f16bits(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype == np.uint16:
        return a
    raise TypeError("expected float16 or uint16 bit patterns")


# ---- codecs -----------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(int(code))


def e2m1_encode(x: float) -> int:
    return _load().oracle_e2m1_encode(float(np.float32(x)))


def e4m3_encode(x: float) -> int:
    return _load().oracle_e4m3_encode(float(np.float32(x)))


def f16_from_double(v: float) -> int:
    return _load().oracle_f16_from_double(float(v))


def f16_to_double(b: int) -> float:
    return _load().oracle_f16_to_double(int(b))


def dequant_f16(q: int, s: int) -> int:
    return _load().oracle_dequant_f16(int(q), int(s))


# ---- quantiser ----------------------------------------------------------------

def quantize(w):
    """FP32 [n_mats, rows, k] -> (q [n,rows,k/2] u8, s [n,rows,k/16] u8, g [n] f32, status)."""
    w = _c(w, np.float32)
    if w.ndim == 2:
        w = w[None]
    n, rows, k = w.shape
    assert k % 16 == 0 and k % 2 == 0
    q = np.empty((n, rows, k // 2), np.uint8)
    s = np.empty((n, rows, k // 16), np.uint8)
    g = np.empty((n,), np.float32)
    st = _load().oracle_quantize(_p(w), n, rows, k, _p(q), _p(s), _p(g))
    return q, s, g, int(st)


def dequant(q, s):
    """Canonical NVFP4 rows -> FP16 values (exact), as np.float16 [rows, k]."""
    q = _c(q, np.uint8)
    s = _c(s, np.uint8)
    rows = q.shape[-2] if q.ndim >= 2 else 1
    k = q.shape[-1] * 2
    lead = q.shape[:-1]
    rows = int(np.prod(lead))
    out = np.empty((rows, k), np.uint16)
    _load().oracle_dequant(_p(q), _p(s), rows, k, _p(out))
    return out.view(np.float16).reshape(*lead, k)


# ---- router / plan / forward ------------------------------------------------------

def router(x, wr, bias, k):
    """Returns (logits [M,E] f32, ids [M,k] i32, w [M,k] f32)."""
    x = _f16bits(x)
    wr = _f16bits(wr)
    M, H = x.shape
    E = wr.shape[1]
    b = None if bias is None else _c(bias, np.float32)
    logits = np.empty((M, E), np.float32)
    ids = np.empty((M, k), np.int32)
    w = np.empty((M, k), np.float32)
    _load().oracle_router(_p(x), _p(wr), _p(b), M, H, E, k, _p(logits), _p(ids), _p(w))
    return logits, ids, w


def shared_gate(x, wg):
    x = _f16bits(x)
    wg = _f16bits(wg)
    M, H = x.shape
    gamma = np.empty((M,), np.float32)
    _load().oracle_shared_gate(_p(x), _p(wg), M, H, _p(gamma))
    return gamma


def plan(ids, n_exp, bn):
    """Returns dict(counts, offsets, perm, inv, tiles, status)."""
    ids = _c(ids, np.int32).reshape(-1)
    P = ids.shape[0]
    counts = np.empty((n_exp,), np.int32)
    offsets = np.empty((n_exp + 1,), np.int32)
    perm = np.empty((max(P, 1),), np.int32)
    inv = np.empty((max(P, 1),), np.int32)
    max_tiles = n_exp + (P + bn - 1) // bn + 1
    tiles = np.empty((max_tiles, 3), np.int32)
    nt = ctypes.c_int64(0)
    st = _load().oracle_plan(_p(ids), P, n_exp, bn, _p(counts), _p(offsets), _p(perm),
                             _p(inv), _p(tiles), max_tiles, ctypes.byref(nt))
    n_valid = int(offsets[-1])
    return dict(counts=counts, offsets=offsets, perm=perm[:n_valid].copy(),
                inv=inv[:P].copy(), tiles=tiles[:nt.value].copy(), status=int(st))


def forward(x, ids, w, w13, w2, shared=None, gamma=None, tokens=None, want_h=False,
            h_exact=False):
    """Layer output for the given tokens.  h is rounded to FP16 between the
    GEMMs (the reading the acceptance bar is stated against); with h_exact it
    is not (the other reading of the same passage).

    w13 = (q [E,2I,H/2], s [E,2I,H/16], g [E]); w2 = (q [E,H,I/2], s [E,H,I/16], g [E]);
    shared = None or ((q13, s13, g13), (q2, s2, g2)) without the expert axis.
    Returns (y float16 [n_tok, H], status[, h float64 [n_tok, k, I]]).
    """
    x = _f16bits(x)
    M, H = x.shape
    ids = _c(ids, np.int32)
    k = ids.shape[1]
    w = _c(w, np.float32)
    q13, s13, g13 = (_c(w13[0], np.uint8), _c(w13[1], np.uint8), _c(w13[2], np.float32))
    q2, s2, g2 = (_c(w2[0], np.uint8), _c(w2[1], np.uint8), _c(w2[2], np.float32))
    E = q13.shape[0]
    I = q13.shape[1] // 2
    if shared is not None:
        (sq13, ss13, sg13), (sq2, ss2, sg2) = shared
        sq13, ss13 = _c(sq13, np.uint8), _c(ss13, np.uint8)
        sq2, ss2 = _c(sq2, np.uint8), _c(ss2, np.uint8)
        sg13 = _c(np.atleast_1d(sg13), np.float32)
        sg2 = _c(np.atleast_1d(sg2), np.float32)
    else:
        sq13 = ss13 = sg13 = sq2 = ss2 = sg2 = None
    gm = None if gamma is None else _c(gamma, np.float32)
    if tokens is None:
        tok = None
        n_tok = M
    else:
        tok = _c(tokens, np.int64)
        n_tok = tok.shape[0]
    y = np.empty((n_tok, H), np.uint16)
    h = np.empty((n_tok, k, I), np.float64) if want_h else None
    st = _load().oracle_forward(M, H, E, k, I, _p(x), _p(ids), _p(w), _p(q13), _p(s13),
                                _p(g13), _p(q2), _p(s2), _p(g2), _p(sq13), _p(ss13),
                                _p(sg13), _p(sq2), _p(ss2), _p(sg2), _p(gm), _p(tok),
                                n_tok, int(bool(h_exact)), _p(y), _p(h))
    y = y.view(np.float16)
    if want_h:
        return y, int(st), h
    return y, int(st)


def dense(x, q, s, g):
    """Dense NVFP4 projection y = fp16(g * x . w16^T) of FP16 rows x [M, K]
    with canonical NVFP4 weights q [N, K/2], s [N, K/16] and global scale g."""
    x = _f16bits(x)
    M, K = x.shape
    q = _c(q, np.uint8)
    s = _c(s, np.uint8)
    N = q.shape[0]
    if q.shape != (N, K // 2) or s.shape != (N, K // 16):
        raise ValueError("dense: q must be [N, K/2] and s [N, K/16]")
    y = np.empty((M, N), np.uint16)
    _load().oracle_dense(M, N, K, _p(x), _p(q), _p(s), float(g), _p(y))
    return y.view(np.float16)


def prepare_scales(s):
    """E4M3 scale bytes -> FP16 bit patterns of their values, same shape
    (the prepared-scale storage); returns (uint16 array, status)."""
    s = _c(s, np.uint8)
    out = np.empty(s.shape, np.uint16)
    st = _load().oracle_prepare_scales(_p(s), s.size, _p(out))
    return out, int(st)


def fp8_quantize(w):
    """FP32 [rows, k] -> (q [rows, k] E4M3 codes, cs [rows] FP32, status):
    channel-FP8 (QPN8) weights."""
    w = _c(w, np.float32)
    rows, k = w.shape
    q = np.empty((rows, k), np.uint8)
    cs = np.empty((rows,), np.float32)
    st = _load().oracle_fp8_quantize(_p(w), rows, k, _p(q), _p(cs))
    return q, cs, int(st)


def fp8_dense(x, q, cs):
    """Dense channel-FP8 projection y = fp16(cs * x . E4M3(q)^T) of FP16 rows
    x [M, K] with q [N, K] E4M3 codes and channel scales cs [N]."""
    x = _f16bits(x)
    M, K = x.shape
    q = _c(q, np.uint8)
    cs = _c(cs, np.float32)
    N = q.shape[0]
    if q.shape != (N, K) or cs.shape != (N,):
        raise ValueError("fp8_dense: q must be [N, K] and cs [N]")
    y = np.empty((M, N), np.uint16)
    _load().oracle_fp8_dense(M, N, K, _p(x), _p(q), _p(cs), _p(y))
    return y.view(np.float16)
