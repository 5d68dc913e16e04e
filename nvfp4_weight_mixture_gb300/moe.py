"""Python binding of ``libmoe_nvfp4.so`` (C ABI in ``include/moe_nvfp4.h``).

Argument marshalling only: torch supplies device memory and the current CUDA
stream; every step of the layer runs in the library's CUDA kernels.  There is
no CPU or PyTorch fallback: if the library is missing or its ABI version
differs, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_nvfp4.so")
ABI_VERSION = 1

OK = 0
ERR_CUDA = -6
ERR = {
    -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_SHAPE", -3: "MOE_ERR_ALIGNMENT",
    -4: "MOE_ERR_WORKSPACE", -5: "MOE_ERR_UNSUPPORTED_DEVICE", -6: "MOE_ERR_CUDA",
    -7: "MOE_ERR_LAYOUT",
}
ST_INVALID_ID = 0x1
ST_NONFINITE = 0x2
ST_TIMEOUT = 0x4
FLAG_IDS_GIVEN = 0x1
FLAG_SHARED = 0x2
LAYOUT_CANONICAL = 0
LAYOUT_FRAGMENT = 1
LAYOUT_FRAGMENT_W13 = 2
LAYOUT_FP8_FRAGMENT = 3
SCALES_PREPARED = 0x100
DENSE_MAX_TOKENS = 32
DECODE_MAX_TOKENS = 16

EXPORTS = ["moe_nvfp4_abi_version", "moe_nvfp4_status_string", "moe_nvfp4_query",
           "moe_nvfp4_quantize", "moe_nvfp4_plan", "moe_nvfp4_forward", "moe_nvfp4_dequantize",
           "moe_nvfp4_set_trace_events", "moe_nvfp4_forward_noalloc",
           "moe_nvfp4_last_cuda_error", "moe_nvfp4_set_small_router",
           "moe_nvfp4_dense_query", "moe_nvfp4_dense", "moe_fp8_quantize", "moe_fp8_dense",
           "moe_nvfp4_prepare_scales", "moe_nvfp4_layer", "moe_nvfp4_set_decode_max_tokens",
           "moe_nvfp4_set_wait_test"]
TRACE_STEPS = ("plan", "w13", "w2", "combine")


class Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("reserved", ctypes.c_int32 * 3)]


class WeightsC(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p), ("g", ctypes.c_void_p),
                ("layout", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class MoEError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        msg = f"{fn} failed: {ERR.get(code, code)} ({status_string(code)})"
        if code == ERR_CUDA:
            msg += f" [{load_library().moe_nvfp4_last_cuda_error().decode()}]"
        super().__init__(msg)


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Opens the CUDA library (once) and checks its ABI version."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing: run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        lib.moe_nvfp4_abi_version.argtypes = []
        lib.moe_nvfp4_abi_version.restype = I32
        lib.moe_nvfp4_status_string.argtypes = [I32]
        lib.moe_nvfp4_status_string.restype = ctypes.c_char_p
        lib.moe_nvfp4_last_cuda_error.argtypes = []
        lib.moe_nvfp4_last_cuda_error.restype = ctypes.c_char_p
        lib.moe_nvfp4_query.argtypes = [P, I64, ctypes.POINTER(SZ), ctypes.POINTER(SZ)]
        lib.moe_nvfp4_query.restype = I32
        lib.moe_nvfp4_quantize.argtypes = [P, I64, I64, I64, I32, P, P, P, P, P]
        lib.moe_nvfp4_quantize.restype = I32
        lib.moe_nvfp4_dequantize.argtypes = [P, P, I64, I64, I64, I32, P, P]
        lib.moe_nvfp4_dequantize.restype = I32
        lib.moe_nvfp4_plan.argtypes = [P, I64, P, P, P, P, P, P, P, SZ, P, P]
        lib.moe_nvfp4_plan.restype = I32
        lib.moe_nvfp4_forward.argtypes = [P, I64, P, P, P, P, P, P, P, P, SZ, P, P]
        lib.moe_nvfp4_forward.restype = I32
        lib.moe_nvfp4_layer.argtypes = [P, I64, P, P, P, P, P, P, P, SZ, P, P, P, P, P, P, SZ,
                                        P, P]
        lib.moe_nvfp4_layer.restype = I32
        lib.moe_nvfp4_forward_noalloc.argtypes = [P, I64, P, P, P, P, P, P, P, P, P]
        lib.moe_nvfp4_forward_noalloc.restype = I32
        lib.moe_nvfp4_set_trace_events.argtypes = [P, I32]
        lib.moe_nvfp4_set_trace_events.restype = I32
        lib.moe_nvfp4_set_wait_test.argtypes = [I32, I64, P]
        lib.moe_nvfp4_set_wait_test.restype = I32
        lib.moe_nvfp4_set_decode_max_tokens.argtypes = [I32]
        lib.moe_nvfp4_set_decode_max_tokens.restype = I32
        lib.moe_nvfp4_set_small_router.argtypes = [I32]
        lib.moe_nvfp4_set_small_router.restype = I32
        lib.moe_nvfp4_dense_query.argtypes = [I64, I64, I64, ctypes.POINTER(SZ)]
        lib.moe_nvfp4_dense_query.restype = I32
        lib.moe_nvfp4_dense.argtypes = [I64, I64, I64, P, P, P, P, SZ, P, P]
        lib.moe_nvfp4_dense.restype = I32
        lib.moe_fp8_quantize.argtypes = [P, I64, I64, I32, P, P, P, P]
        lib.moe_fp8_quantize.restype = I32
        lib.moe_fp8_dense.argtypes = [I64, I64, I64, P, P, P, P, P, SZ, P, P]
        lib.moe_fp8_dense.restype = I32
        lib.moe_nvfp4_prepare_scales.argtypes = [P, I64, P, P, P]
        lib.moe_nvfp4_prepare_scales.restype = I32
        v = lib.moe_nvfp4_abi_version()
        if v != ABI_VERSION:
            raise RuntimeError(f"libmoe_nvfp4 ABI version {v}, binding expects {ABI_VERSION}")
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load_library().moe_nvfp4_status_string(int(code)).decode()


def _check(fn, rc):
    if rc != OK:
        raise MoEError(fn, rc)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


_raw_stream_fn = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _raw_stream(dev_index):
    """The current stream of a device as an integer handle (the cheap query
    where this torch build has it)."""
    if _raw_stream_fn is not None:
        return _raw_stream_fn(dev_index)
    return torch.cuda.current_stream(dev_index).cuda_stream


def _need(t, dtype, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t


def _on_current_device(named):
    """Every given tensor lives on the current CUDA device (the one whose
    stream the library enqueues on)."""
    dev = torch.cuda.current_device()
    for name, t in named:
        if t is not None and t.device.index != dev:
            raise ValueError(f"{name}: on {t.device}, but the current device is cuda:{dev}")


def _expect(errors, name, t, dtype, n):
    if t is None:
        return
    if t.dtype != dtype:
        errors.append(f"{name}: expected {dtype}, got {t.dtype}")
    elif t.numel() != n:
        errors.append(f"{name}: expected {n} elements, got {t.numel()}")


def _expect_weights(errors, name, w, rows, k, n_mats):
    """Codes, scales (raw E4M3 bytes as uint8, or prepared FP16 scales as
    int16) and global scales of n_mats matrices of rows x k."""
    if w is None:
        return
    q, s, g = w
    _expect(errors, name + ".q", q, torch.uint8, n_mats * rows * k // 2)
    _expect(errors, name + ".s", s, torch.int16 if s.dtype == torch.int16 else torch.uint8,
            n_mats * rows * k // 16)
    _expect(errors, name + ".g", g, torch.float32, n_mats)


def _expect_status(errors, status):
    if status is not None and (status.dtype != torch.int32 or status.numel() < 1):
        errors.append("status: expected at least one int32 element")


def plan_arg_errors(cfg, x, w_router, bias, w_gate, ids, topk_w, status=None):
    """Sizes and dtypes the plan call reads and writes through plain pointers
    (the C ABI cannot see them): x [M][H] FP16, W_r [H][E] FP16, bias [E] FP32,
    w_g [H] FP16, ids [M][k] int32, weights [M][k] FP32.  Returns the list of
    mismatches (empty when the arguments fit)."""
    H, E, k = cfg.hidden, cfg.n_experts, cfg.top_k
    M = x.shape[0] if x.dim() > 0 else 0
    e = []
    _expect(e, "x", x, torch.float16, M * H)
    _expect(e, "w_router", w_router, torch.float16, H * E)
    _expect(e, "bias", bias, torch.float32, E)
    _expect(e, "w_gate", w_gate, torch.float16, H)
    _expect(e, "ids", ids, torch.int32, M * k)
    _expect(e, "topk_w", topk_w, torch.float32, M * k)
    _expect_status(e, status)
    return e


def forward_arg_errors(cfg, x, w13, w2, shared13, shared2, y, status=None):
    """As plan_arg_errors for the forward: x and y [M][H] FP16; W13 codes,
    scales and global scales of E matrices of 2I x H, W2 of E matrices of
    H x I (the shared expert's: one matrix each)."""
    H, E, I = cfg.hidden, cfg.n_experts, cfg.intermediate
    M = x.shape[0] if x.dim() > 0 else 0
    e = []
    _expect(e, "x", x, torch.float16, M * H)
    _expect(e, "y", y, torch.float16, M * H)
    _expect_weights(e, "w13", w13, 2 * I, H, E)
    _expect_weights(e, "w2", w2, H, I, E)
    _expect_weights(e, "shared13", shared13, 2 * I, H, 1)
    _expect_weights(e, "shared2", shared2, H, I, 1)
    _expect_status(e, status)
    return e


def _raise_if(fn, errors):
    if errors:
        raise ValueError(f"{fn}: " + "; ".join(errors))


def make_config(hidden, n_experts, top_k, intermediate, shared=False, ids_given=False):
    c = Config()
    c.hidden, c.n_experts, c.top_k, c.intermediate = hidden, n_experts, top_k, intermediate
    c.flags = (FLAG_SHARED if shared else 0) | (FLAG_IDS_GIVEN if ids_given else 0)
    return c


def query(cfg: Config, max_tokens: int):
    pb, wb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check("moe_nvfp4_query", load_library().moe_nvfp4_query(
        ctypes.byref(cfg), int(max_tokens), ctypes.byref(pb), ctypes.byref(wb)))
    return pb.value, wb.value


_trace_keep = None


def set_trace_events(events):
    """Per-step CUDA event records inside plan/forward (diagnostic).

    events: list of 2 * n torch.cuda.Event(enable_timing=True) for the first n
    of TRACE_STEPS, or None to stop tracing."""
    global _trace_keep
    lib = load_library()
    if events is None:
        _check("moe_nvfp4_set_trace_events", lib.moe_nvfp4_set_trace_events(None, 0))
        _trace_keep = None
        return
    for e in events:      # torch creates the CUDA event on its first record
        e.record()
    torch.cuda.synchronize()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _trace_keep = (arr, events)
    _check("moe_nvfp4_set_trace_events", lib.moe_nvfp4_set_trace_events(arr, len(events) // 2))


def set_wait_test(hold_raw_producer: bool, wait_limit_cycles: int = 0):
    """Failure-path test switch of the grouped GEMMs (see the header)."""
    _check("moe_nvfp4_set_wait_test", load_library().moe_nvfp4_set_wait_test(
        1 if hold_raw_producer else 0, int(wait_limit_cycles), _stream()))


def set_decode_max_tokens(m: int):
    """Diagnostic: the forward's largest M on the decode kernels (0..16)."""
    _check("moe_nvfp4_set_decode_max_tokens", load_library().moe_nvfp4_set_decode_max_tokens(int(m)))


def set_small_router(force_ticket_router: bool):
    """Diagnostic: route M <= 16 through the 128-block ticket router (True) or
    choose automatically (False; the thread-block cluster where it fits)."""
    _check("moe_nvfp4_set_small_router",
           load_library().moe_nvfp4_set_small_router(1 if force_ticket_router else 0))


# ---- quantise / dequantise ---------------------------------------------------------

def quantize(w: torch.Tensor, layout: int, status: torch.Tensor | None = None, q=None, s=None,
             g=None):
    """FP32 CUDA [n_mats, rows, k] -> (q uint8, s uint8, g float32 [n_mats]).

    q, s, g may be given (contiguous CUDA tensors of the right sizes) to write
    into, e.g. a slice of a larger per-layer buffer."""
    if w.dim() == 2:
        w = w.unsqueeze(0)
    _need(w, torch.float32, "w")
    n, rows, k = w.shape
    if q is None:
        q = torch.empty((n, rows * k // 2), dtype=torch.uint8, device=w.device)
    if s is None:
        s = torch.empty((n, rows * k // 16), dtype=torch.uint8, device=w.device)
    if g is None:
        g = torch.empty((n,), dtype=torch.float32, device=w.device)
    _need(q, torch.uint8, "q")
    _need(s, torch.uint8, "s")
    _need(g, torch.float32, "g")
    if q.numel() != n * rows * k // 2 or s.numel() != n * rows * k // 16 or g.numel() != n:
        raise ValueError("quantize: output sizes do not match the input")
    if status is not None:
        _need(status, torch.int32, "status")
    _check("moe_nvfp4_quantize", load_library().moe_nvfp4_quantize(
        _ptr(w), n, rows, k, int(layout), _ptr(q), _ptr(s), _ptr(g), _ptr(status), _stream()))
    return q, s, g


def dequantize_arg_errors(q, s, n_mats, rows, k):
    """q and s must hold the codes and scales of n_mats matrices of rows x k."""
    e = []
    _expect(e, "q", q, torch.uint8, n_mats * rows * k // 2)
    _expect(e, "s", s, torch.uint8, n_mats * rows * k // 16)
    return e


def dequantize(q, s, n_mats, rows, k, layout):
    _need(q, torch.uint8, "q")
    _need(s, torch.uint8, "s")
    _raise_if("dequantize", dequantize_arg_errors(q, s, n_mats, rows, k))
    _on_current_device([("q", q), ("s", s)])
    out = torch.empty((n_mats, rows, k), dtype=torch.float16, device=q.device)
    _check("moe_nvfp4_dequantize", load_library().moe_nvfp4_dequantize(
        _ptr(q), _ptr(s), n_mats, rows, k, int(layout), _ptr(out), _stream()))
    return out


# ---- plan / forward ---------------------------------------------------------------------

def _weights_c(w, layout):
    """The C weight set; int16 scales are prepared FP16 scales."""
    if w is None:
        return None
    q, s, g = w
    wc = WeightsC()
    wc.q = q.data_ptr()
    wc.s = s.data_ptr()
    wc.g = g.data_ptr()
    wc.layout = layout | (SCALES_PREPARED if s.dtype == torch.int16 else 0)
    wc.reserved = 0
    return wc


def plan(cfg: Config, x, w_router, bias, w_gate, ids, topk_w, plan_buf, status=None):
    M = x.shape[0]
    _need(x, torch.float16, "x")
    _need(ids, torch.int32, "ids")
    _need(topk_w, torch.float32, "topk_w")
    _need(plan_buf, torch.uint8, "plan")
    for name, t in (("w_router", w_router), ("bias", bias), ("w_gate", w_gate),
                    ("status", status)):
        if t is not None:
            _need(t, t.dtype, name)
    _raise_if("plan", plan_arg_errors(cfg, x, w_router, bias, w_gate, ids, topk_w, status))
    _on_current_device([("x", x), ("w_router", w_router), ("bias", bias), ("w_gate", w_gate),
                        ("ids", ids), ("topk_w", topk_w), ("plan", plan_buf), ("status", status)])
    _check("moe_nvfp4_plan", load_library().moe_nvfp4_plan(
        ctypes.byref(cfg), M, _ptr(x), _ptr(w_router), _ptr(bias), _ptr(w_gate), _ptr(ids),
        _ptr(topk_w), _ptr(plan_buf), plan_buf.numel(), _ptr(status), _stream()))


def _check_forward_args(fn, cfg, x, plan_buf, w13, w2, shared13, shared2, y, status, ws=None):
    _need(x, torch.float16, "x")
    _need(y, torch.float16, "y")
    _need(plan_buf, torch.uint8, "plan")
    if ws is not None:
        _need(ws, torch.uint8, "ws")
    named = [("x", x), ("y", y), ("plan", plan_buf), ("ws", ws), ("status", status)]
    for wn, w in (("w13", w13), ("w2", w2), ("shared13", shared13), ("shared2", shared2)):
        if w is not None:
            for part, t in zip("qsg", w):
                _need(t, t.dtype, f"{wn}.{part}")
                named.append((f"{wn}.{part}", t))
    if status is not None:
        _need(status, torch.int32, "status")
    _raise_if(fn, forward_arg_errors(cfg, x, w13, w2, shared13, shared2, y, status))
    _on_current_device(named)


def forward(cfg: Config, x, plan_buf, w13, w2, shared13, shared2, y, ws, status=None):
    M = x.shape[0]
    _check_forward_args("forward", cfg, x, plan_buf, w13, w2, shared13, shared2, y, status, ws)
    a = _weights_c(w13, LAYOUT_FRAGMENT_W13)
    b = _weights_c(w2, LAYOUT_FRAGMENT)
    c = _weights_c(shared13, LAYOUT_FRAGMENT_W13)
    d = _weights_c(shared2, LAYOUT_FRAGMENT)
    _check("moe_nvfp4_forward", load_library().moe_nvfp4_forward(
        ctypes.byref(cfg), M, _ptr(x), _ptr(plan_buf), ctypes.byref(a), ctypes.byref(b),
        ctypes.byref(c) if c is not None else None, ctypes.byref(d) if d is not None else None,
        _ptr(y), _ptr(ws), ws.numel(), _ptr(status), _stream()))


def layer(cfg: Config, x, w_router, bias, w_gate, ids, topk_w, plan_buf, w13, w2, shared13,
          shared2, y, ws, status=None):
    """moe_nvfp4_layer: router, plan and forward in one call."""
    M = x.shape[0]
    _need(ids, torch.int32, "ids")
    _need(topk_w, torch.float32, "topk_w")
    for name, t in (("w_router", w_router), ("bias", bias), ("w_gate", w_gate)):
        if t is not None:
            _need(t, t.dtype, name)
    _raise_if("layer", plan_arg_errors(cfg, x, w_router, bias, w_gate, ids, topk_w, status))
    _check_forward_args("layer", cfg, x, plan_buf, w13, w2, shared13, shared2, y, status, ws)
    _on_current_device([("w_router", w_router), ("bias", bias), ("w_gate", w_gate),
                        ("ids", ids), ("topk_w", topk_w)])
    a = _weights_c(w13, LAYOUT_FRAGMENT_W13)
    b = _weights_c(w2, LAYOUT_FRAGMENT)
    c = _weights_c(shared13, LAYOUT_FRAGMENT_W13)
    d = _weights_c(shared2, LAYOUT_FRAGMENT)
    _check("moe_nvfp4_layer", load_library().moe_nvfp4_layer(
        ctypes.byref(cfg), M, _ptr(x), _ptr(w_router), _ptr(bias), _ptr(w_gate), _ptr(ids),
        _ptr(topk_w), _ptr(plan_buf), plan_buf.numel(), ctypes.byref(a), ctypes.byref(b),
        ctypes.byref(c) if c is not None else None, ctypes.byref(d) if d is not None else None,
        _ptr(y), _ptr(ws), ws.numel(), _ptr(status), _stream()))


def forward_noalloc(cfg: Config, x, plan_buf, w13, w2, shared13, shared2, y, status=None):
    """moe_nvfp4_forward_noalloc: the forward with the library's own static
    workspace (for callers that cannot allocate; see the header)."""
    M = x.shape[0]
    _check_forward_args("forward_noalloc", cfg, x, plan_buf, w13, w2, shared13, shared2, y,
                        status)
    a = _weights_c(w13, LAYOUT_FRAGMENT_W13)
    b = _weights_c(w2, LAYOUT_FRAGMENT)
    c = _weights_c(shared13, LAYOUT_FRAGMENT_W13)
    d = _weights_c(shared2, LAYOUT_FRAGMENT)
    _check("moe_nvfp4_forward_noalloc", load_library().moe_nvfp4_forward_noalloc(
        ctypes.byref(cfg), M, _ptr(x), _ptr(plan_buf), ctypes.byref(a), ctypes.byref(b),
        ctypes.byref(c) if c is not None else None, ctypes.byref(d) if d is not None else None,
        _ptr(y), _ptr(status), _stream()))


class MoELayer:
    """Owns the quantised weights and the plan / workspace buffers of one layer.

    w13 / w2: (q, s, g) CUDA tensors in the fragment layouts (W13 interleaved).
    """

    def __init__(self, hidden, n_experts, top_k, intermediate, w_router, w13, w2,
                 shared13=None, shared2=None, w_gate=None, bias=None, max_tokens=1,
                 device="cuda"):
        self.shared = shared13 is not None
        self.cfg = make_config(hidden, n_experts, top_k, intermediate, shared=self.shared)
        self.cfg_given = make_config(hidden, n_experts, top_k, intermediate, shared=self.shared,
                                     ids_given=True)
        self.H, self.E, self.k, self.I = hidden, n_experts, top_k, intermediate
        self.w_router, self.w13, self.w2 = w_router, w13, w2
        self.shared13, self.shared2, self.w_gate, self.bias = shared13, shared2, w_gate, bias
        self.max_tokens = 0
        self.device = torch.device(device)
        self._dev_index = self.device.index if self.device.index is not None else \
            torch.cuda.current_device()
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self._fast = None    # the call's fixed C arguments, once the full checks have passed
        self._routes = {}    # M -> (ids, topk_w) reused by calls that pass none
        self.reserve(max_tokens)

    def reserve(self, max_tokens):
        if max_tokens <= self.max_tokens:
            return
        pb, wb = query(self.cfg, max_tokens)
        self.plan_buf = torch.zeros(pb, dtype=torch.uint8, device=self.device)
        self.ws = torch.empty(max(wb, 16), dtype=torch.uint8, device=self.device)
        self.max_tokens = max_tokens

    def route(self, x, ids=None, topk_w=None, out_ids=None, out_w=None):
        """Router + plan; with ids/topk_w given, plans those instead."""
        M = x.shape[0]
        self.reserve(M)
        if ids is not None:
            plan(self.cfg_given, x, None, None, self.w_gate, ids, topk_w, self.plan_buf,
                 self.status)
            return ids, topk_w
        ids = out_ids if out_ids is not None else torch.empty((M, self.k), dtype=torch.int32,
                                                              device=self.device)
        tw = out_w if out_w is not None else torch.empty((M, self.k), dtype=torch.float32,
                                                         device=self.device)
        plan(self.cfg, x, self.w_router, self.bias, self.w_gate, ids, tw, self.plan_buf,
             self.status)
        return ids, tw

    def forward_planned(self, x, y=None):
        M = x.shape[0]
        y = y if y is not None else torch.empty((M, self.H), dtype=torch.float16, device=self.device)
        forward(self.cfg, x, self.plan_buf, self.w13, self.w2, self.shared13, self.shared2, y,
                self.ws, self.status)
        return y

    def _fast_key(self):
        return (self.w13, self.w2, self.shared13, self.shared2, self.w_router, self.bias,
                self.w_gate, self.plan_buf, self.ws, self.status)

    def _build_fast(self):
        """The fixed C arguments of moe_nvfp4_layer (config, weights, buffers),
        built after a call whose arguments passed every check."""
        wc = (_weights_c(self.w13, LAYOUT_FRAGMENT_W13), _weights_c(self.w2, LAYOUT_FRAGMENT),
              _weights_c(self.shared13, LAYOUT_FRAGMENT_W13),
              _weights_c(self.shared2, LAYOUT_FRAGMENT))
        refs = tuple(None if w is None else ctypes.byref(w) for w in wc)
        ptr = lambda t: None if t is None else t.data_ptr()
        fixed = (ctypes.byref(self.cfg), ptr(self.w_router), ptr(self.bias), ptr(self.w_gate),
                 self.plan_buf.data_ptr(), self.plan_buf.numel(), refs, self.ws.data_ptr(),
                 self.ws.numel(), self.status.data_ptr())
        self._fast = (self._fast_key(), fixed, wc)

    def _fast_ready(self, t, M):
        return (isinstance(t, torch.Tensor) and t.dtype is torch.float16 and t.dim() == 2
                and t.shape[0] == M and t.shape[1] == self.H and t.is_contiguous()
                and t.get_device() == self._dev_index)

    def __call__(self, x, y=None, ids=None, topk_w=None):
        """The whole layer through moe_nvfp4_layer (router, plan, forward).
        Returns y; the routes land in ids / topk_w (when not given, in buffers
        of the layer reused by the next call with as many tokens) and the plan
        in the plan buffer.

        After a first call with full argument checks, calls that pass no
        routes and the same weights and buffers go straight to the library
        with the checks that can change between calls (x and y: FP16, [M, H],
        contiguous, on the layer's device); the library validates the rest."""
        M = x.shape[0]
        self.reserve(M)
        f = self._fast
        if (ids is None and topk_w is None and f is not None and self._fast_ready(x, M)
                and (y is None or self._fast_ready(y, M))):
            key = self._fast_key()
            if all(a is b for a, b in zip(f[0], key)):
                if y is None:
                    y = torch.empty((M, self.H), dtype=torch.float16, device=self.device)
                r = self._routes.get(M)
                if r is None:
                    r = (torch.empty((M, self.k), dtype=torch.int32, device=self.device),
                         torch.empty((M, self.k), dtype=torch.float32, device=self.device))
                    self._routes[M] = r
                cfg_ref, wr, bias, wg, plan_p, plan_n, refs, ws_p, ws_n, st_p = f[1]
                _check("moe_nvfp4_layer", load_library().moe_nvfp4_layer(
                    cfg_ref, M, x.data_ptr(), wr, bias, wg, r[0].data_ptr(), r[1].data_ptr(),
                    plan_p, plan_n, refs[0], refs[1], refs[2], refs[3], y.data_ptr(), ws_p, ws_n,
                    st_p, _raw_stream(self._dev_index)))
                self.last_ids, self.last_topk_w = r
                return y
        y = y if y is not None else torch.empty((M, self.H), dtype=torch.float16, device=self.device)
        ids = ids if ids is not None else torch.empty((M, self.k), dtype=torch.int32,
                                                      device=self.device)
        topk_w = topk_w if topk_w is not None else torch.empty((M, self.k), dtype=torch.float32,
                                                               device=self.device)
        layer(self.cfg, x, self.w_router, self.bias, self.w_gate, ids, topk_w, self.plan_buf,
              self.w13, self.w2, self.shared13, self.shared2, y, self.ws, self.status)
        self.last_ids, self.last_topk_w = ids, topk_w
        if self._fast is None or not all(a is b for a, b in zip(self._fast[0], self._fast_key())):
            self._build_fast()
        return y


# ---- dense few-row projections, channel-FP8 weights, prepared scales ---------------

def dense_query(M, N, K):
    wb = ctypes.c_size_t(0)
    _check("moe_nvfp4_dense_query",
           load_library().moe_nvfp4_dense_query(int(M), int(N), int(K), ctypes.byref(wb)))
    return wb.value


def _dense_ws(M, N, K, ws, device):
    need = dense_query(M, N, K)
    if ws is None and need > 0:
        ws = torch.zeros(need, dtype=torch.uint8, device=device)   # counters start at zero
    if ws is not None:
        _need(ws, ws.dtype, "ws")
    return ws, (ws.numel() * ws.element_size() if ws is not None else 0)


def dense(x, w, N, prepared=False, y=None, ws=None, status=None):
    """NVFP4 dense projection (QPN2): y [M, N] = fp16(g * x . w16^T).

    w = (q, s, g) of one N x K matrix in the fragment layout; with prepared
    the scales are FP16 (moe_nvfp4_prepare_scales)."""
    _need(x, torch.float16, "x")
    M, K = x.shape
    q, s, g = w
    for n_, t in (("q", q), ("s", s), ("g", g)):
        _need(t, t.dtype, n_)
    errs = []
    _expect(errs, "q", q, torch.uint8, N * K // 2)
    if s.numel() * s.element_size() != N * K // 16 * (2 if prepared else 1):
        errs.append("s: wrong byte count for the scale format")
    _expect(errs, "g", g, torch.float32, 1)
    _expect_status(errs, status)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _need(y, torch.float16, "y")
    _expect(errs, "y", y, torch.float16, M * N)
    _raise_if("dense", errs)
    ws, wsb = _dense_ws(M, N, K, ws, x.device)
    _on_current_device([("x", x), ("q", q), ("s", s), ("g", g), ("y", y), ("ws", ws),
                        ("status", status)])
    wc = _weights_c(w, LAYOUT_FRAGMENT | (SCALES_PREPARED if prepared else 0))
    _check("moe_nvfp4_dense", load_library().moe_nvfp4_dense(
        M, N, K, _ptr(x), ctypes.byref(wc), _ptr(y), _ptr(ws), wsb, _ptr(status), _stream()))
    return y


def fp8_quantize(w: torch.Tensor, layout: int = LAYOUT_FP8_FRAGMENT, status=None):
    """FP32 CUDA [rows, k] -> (q uint8 [rows * k], channel scales float32 [rows])."""
    _need(w, torch.float32, "w")
    rows, k = w.shape
    q = torch.empty((rows * k,), dtype=torch.uint8, device=w.device)
    cs = torch.empty((rows,), dtype=torch.float32, device=w.device)
    if status is not None:
        _need(status, torch.int32, "status")
    _check("moe_fp8_quantize", load_library().moe_fp8_quantize(
        _ptr(w), rows, k, int(layout), _ptr(q), _ptr(cs), _ptr(status), _stream()))
    return q, cs


def fp8_dense(x, q, cs, y=None, ws=None, status=None):
    """Channel-FP8 dense projection (QPN8): y [M, N] = fp16(cs * x . E4M3(q)^T),
    q in the FP8 fragment layout."""
    _need(x, torch.float16, "x")
    _need(q, torch.uint8, "q")
    _need(cs, torch.float32, "cs")
    M, K = x.shape
    N = cs.numel()
    errs = []
    _expect(errs, "q", q, torch.uint8, N * K)
    _expect_status(errs, status)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _need(y, torch.float16, "y")
    _expect(errs, "y", y, torch.float16, M * N)
    _raise_if("fp8_dense", errs)
    ws, wsb = _dense_ws(M, N, K, ws, x.device)
    _on_current_device([("x", x), ("q", q), ("cs", cs), ("y", y), ("ws", ws), ("status", status)])
    _check("moe_fp8_dense", load_library().moe_fp8_dense(
        M, N, K, _ptr(x), _ptr(q), _ptr(cs), _ptr(y), _ptr(ws), wsb, _ptr(status), _stream()))
    return y


def prepare_scales(s: torch.Tensor, status=None):
    """E4M3 scale bytes -> prepared FP16 scales (as int16, same element order)."""
    _need(s, torch.uint8, "s")
    out = torch.empty(s.shape, dtype=torch.int16, device=s.device)
    if status is not None:
        _need(status, torch.int32, "status")
    _check("moe_nvfp4_prepare_scales", load_library().moe_nvfp4_prepare_scales(
        _ptr(s), s.numel(), _ptr(out), _ptr(status), _stream()))
    return out
