"""Python binding of libtb, the C-ABI library of the TokenButler decode-time hot path.

Argument marshalling only: every step runs in the CUDA kernels of
``libtb.so`` (built in-tree for sm_103a by ``build.py``). There is no CPU or
PyTorch fallback; if the library is missing the first call raises.

Functions keep the C names (``tb_score``, ``tb_topk``, ...) and take torch
tensors on the current CUDA device; streams default to the current torch
stream. bf16 tensors are passed as raw pointers to their 16-bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtb.so")

TB_OK = 0
TB_ERR_INVALID_ARG = 1
TB_ERR_UNSUPPORTED = 2
TB_ERR_WORKSPACE = 3
TB_ERR_CUDA = 4
TB_ERR_TIMEOUT = 5
TB_ERR_NONFINITE = 6

TB_AGG_MEAN = 0
TB_AGG_MAX = 1

TB_STEP_UNFUSED = 1
TB_STEP_BUDGET_NEIGHBOURS = 2
TB_STEP_PIPELINE = 4

EXPORTED = (
    "tb_status_string", "tb_version", "tb_workspace_size", "tb_workspace_init", "tb_project_append",
    "tb_score", "tb_topk", "tb_expand", "tb_sparse_decode_attn", "tb_decode_step", "tb_topk_noalloc",
    "tb_decode_step_buffered", "tb_predict_queries", "tb_decode_step_ragged", "tb_decode_layers",
)

TB_TOPK_NOALLOC_MAX_ROWS = 64


class TBError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class _Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("D", ctypes.c_int32), ("dp", ctypes.c_int32), ("cap", ctypes.c_int64)]


class _StepParams(ctypes.Structure):
    _fields_ = [("k", ctypes.c_int32), ("T", ctypes.c_int32), ("r", ctypes.c_int32),
                ("agg", ctypes.c_int32), ("scale", ctypes.c_float), ("flags", ctypes.c_int32)]


class _BufferParams(ctypes.Structure):
    _fields_ = [("sink", ctypes.c_int32), ("window", ctypes.c_int32)]


class _LayerBuffers(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("q_imp", ctypes.c_void_p), ("K_new", ctypes.c_void_p),
                ("V_new", ctypes.c_void_p), ("Wk", ctypes.c_void_p), ("K", ctypes.c_void_p), ("V", ctypes.c_void_p),
                ("Kp", ctypes.c_void_p), ("idx_state", ctypes.c_void_p), ("sel", ctypes.c_void_p),
                ("counts", ctypes.c_void_p), ("out", ctypes.c_void_p), ("ws", ctypes.c_void_p),
                ("ws_bytes", ctypes.c_size_t)]


@dataclass(frozen=True)
class Shape:
    B: int
    Hq: int
    Hkv: int
    D: int
    dp: int
    cap: int

    def c(self) -> _Shape:
        return _Shape(self.B, self.Hq, self.Hkv, self.D, self.dp, self.cap)


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load libtb.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               f"`python -m predicted_token_importance_tb_b300.build`")
        lib = ctypes.CDLL(path)
        P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        SP = ctypes.POINTER(_Shape)
        lib.tb_status_string.argtypes = [ctypes.c_int]
        lib.tb_status_string.restype = ctypes.c_char_p
        lib.tb_version.restype = i32
        lib.tb_workspace_size.argtypes = [SP, i64, i32, i32, ctypes.POINTER(sz)]
        lib.tb_workspace_init.argtypes = [P, sz, P]
        lib.tb_project_append.argtypes = [SP, P, i64, P, P, i64, i64, P, sz, P, P]
        lib.tb_score.argtypes = [SP, P, P, i64, i32, P, P, P]
        lib.tb_topk.argtypes = [SP, P, i64, i32, P, P, sz, P, P]
        lib.tb_topk_noalloc.argtypes = [SP, P, i64, i32, P, P, P]
        lib.tb_expand.argtypes = [SP, P, i32, i32, i64, i64, P, i32, P, P, P]
        lib.tb_sparse_decode_attn.argtypes = [SP, P, P, P, P, P, i32, f32, P, P, sz, P, P]
        lib.tb_decode_step.argtypes = [SP, ctypes.POINTER(_StepParams), i64, i64, P, P, P, P, P, P, P, P, P,
                                       ctypes.POINTER(i64), P, i32, P, P, P, sz, P, P]
        lib.tb_predict_queries.argtypes = [P, P, P, i32, i32, i32, i32, P, P, sz, P, P]
        # shape, params, t, n_host, n_dev, q, q_imp, K_new, V_new, Wk, K, V, Kp, idx_state, n_pred, sel,
        # sel_stride, counts, out, ws, ws_bytes, dev_status, stream
        lib.tb_decode_step_ragged.argtypes = [SP, ctypes.POINTER(_StepParams), i64, P, P, P, P, P, P, P, P, P, P, P,
                                              P, P, i32, P, P, P, sz, P, P]
        # shape, params, n, L, layers, sel_stride, dev_status, stream, select_stream
        lib.tb_decode_layers.argtypes = [SP, ctypes.POINTER(_StepParams), i64, i32, ctypes.POINTER(_LayerBuffers), i32,
                                         P, P, P]
        lib.tb_decode_step_buffered.argtypes = [SP, ctypes.POINTER(_StepParams), ctypes.POINTER(_BufferParams), i64,
                                                i64, P, P, P, P, P, P, P, P, P, ctypes.POINTER(i64),
                                                ctypes.POINTER(i64), P, i32, P, P, P, sz, P, P]
        for name in EXPORTED:
            if name != "tb_status_string" and name != "tb_version":
                getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(st: int) -> str:
    try:
        return load_library().tb_status_string(int(st)).decode()
    except Exception:  # library not loadable: still give a readable message
        return f"status {st}"


def tb_status_string(st: int) -> str:
    """The library's text for a status code."""
    return load_library().tb_status_string(int(st)).decode()


def tb_version() -> int:
    """The C ABI's version."""
    return int(load_library().tb_version())


def _check(st: int, what: str):
    if st != TB_OK:
        raise TBError(st, what)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if t.device.index != torch.cuda.current_device():
        # the library launches on the current device (and picks its static arrays there)
        raise ValueError(f"tensor is on cuda:{t.device.index} but the current device is "
                         f"cuda:{torch.cuda.current_device()}: make its device current first")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _bf16(t, name):
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    return _ptr(t)


def _kv(t, name):
    """K / V: a CUDA tensor, or a pinned host tensor (the offloaded cache: the device reads it through
    unified addressing, only the selected rows cross the host link)."""
    if isinstance(t, torch.Tensor) and not t.is_cuda and t.is_pinned():
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return ctypes.c_void_p(t.data_ptr())
    return _bf16(t, name)


def _i32(t, name):
    if t is not None and t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32, got {t.dtype}")
    return _ptr(t)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _status_ptr(dev_status):
    return _i32(dev_status, "dev_status") if dev_status is not None else None


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _need(t, elems: int, name: str):
    """The library reads or writes `elems` elements of `t`: refuse a smaller tensor before any launch."""
    if t is not None and t.numel() < elems:
        raise ValueError(f"{name} holds {t.numel()} elements; the call needs {elems}")


def _need_step(shape: "Shape", q, q_imp, K_new, V_new, Wk, K, V, Kp, out):
    B, Hq, Hkv, D, dp, cap = shape.B, shape.Hq, shape.Hkv, shape.D, shape.dp, shape.cap
    for t, n, name in ((q, B * Hq * D, "q"), (q_imp, B * Hq * dp, "q_imp"), (K_new, B * Hkv * D, "K_new"),
                       (V_new, B * Hkv * D, "V_new"), (Wk, Hkv * D * dp, "Wk"), (K, B * Hkv * cap * D, "K"),
                       (V, B * Hkv * cap * D, "V"), (Kp, B * Hkv * cap * dp, "Kp"), (out, B * Hq * D, "out")):
        _need(t, n, name)


def _need_state(shape: "Shape", kc: int, sel_stride: int, idx_state, sel, counts):
    rows = shape.B * shape.Hkv
    _need(idx_state, rows * kc, "idx_state")
    _need(sel, rows * sel_stride, "sel")
    _need(counts, rows, "counts")


def _centres(k: int, r: int, flags: int) -> int:
    return max(1, k // (2 * r + 1)) if flags & TB_STEP_BUDGET_NEIGHBOURS else k


# ------------------------------------------------------------------ workspace

def tb_workspace_size(shape: Shape, n_max: int, k_max: int, sel_stride_max: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().tb_workspace_size(ctypes.byref(shape.c()), n_max, k_max, sel_stride_max,
                                            ctypes.byref(out)), "tb_workspace_size")
    return int(out.value)


def tb_workspace_init(ws: torch.Tensor, stream=None):
    _check(load_library().tb_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "tb_workspace_init")


def workspace(shape: Shape, n_max: int, k_max: int, sel_stride_max: int, device=None) -> torch.Tensor:
    """A zero-filled workspace (uint8 tensor) large enough for every call at these sizes."""
    nbytes = tb_workspace_size(shape, n_max, k_max, sel_stride_max)
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def dev_status(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def check_dev_status(st: torch.Tensor, what: str = "device"):
    v = int(st.item())
    if v != TB_OK:
        raise TBError(v, what)


# ------------------------------------------------------------------ calls

def tb_project_append(shape: Shape, K_src, src_stride: int, Wk, Kp, pos0: int, n_new: int, ws=None,
                      dev_status=None, stream=None, K_src_offset_rows: int = 0):
    """Kp[:, :, pos0:pos0+n_new] = RNE(K_src rows . Wk). K_src is [B,Hkv,src_stride,D] (rows from K_src_offset_rows)."""
    lib = load_library()
    if K_src.dtype != torch.bfloat16:
        raise TypeError("K_src must be bfloat16")
    if n_new > 0:
        rows = (shape.B * shape.Hkv - 1) * src_stride + n_new
        _need(K_src, (K_src_offset_rows + rows) * shape.D, "K_src")
    _need(Wk, shape.Hkv * shape.D * shape.dp, "Wk")
    _need(Kp, shape.B * shape.Hkv * shape.cap * shape.dp, "Kp")
    base = _ptr(K_src).value + K_src_offset_rows * shape.D * 2
    wsp = _ptr(ws) if ws is not None else None
    wsb = _nbytes(ws) if ws is not None else 0
    _check(lib.tb_project_append(ctypes.byref(shape.c()), ctypes.c_void_p(base), src_stride, _bf16(Wk, "Wk"),
                                 _bf16(Kp, "Kp"), pos0, n_new, wsp, wsb, _status_ptr(dev_status),
                                 _stream(stream)), "tb_project_append")


def tb_score(shape: Shape, q_imp, Kp, n: int, s, agg: int = TB_AGG_MEAN, dev_status=None, stream=None):
    if s.dtype != torch.float32:
        raise TypeError("s must be float32")
    rows = shape.B * shape.Hkv
    _need(q_imp, shape.B * shape.Hq * shape.dp, "q_imp")
    if n > 0:
        _need(Kp, ((rows - 1) * shape.cap + n) * shape.dp, "Kp")
    _need(s, rows * n, "s")
    _check(load_library().tb_score(ctypes.byref(shape.c()), _bf16(q_imp, "q_imp"), _bf16(Kp, "Kp"), n, agg,
                                   _ptr(s), _status_ptr(dev_status), _stream(stream)), "tb_score")


def tb_topk(shape: Shape, s, n: int, k: int, idx, ws, dev_status=None, stream=None):
    if s.dtype != torch.float32:
        raise TypeError("s must be float32")
    _need(s, shape.B * shape.Hkv * n, "s")
    _need(idx, shape.B * shape.Hkv * max(k, 0), "idx")
    _check(load_library().tb_topk(ctypes.byref(shape.c()), _ptr(s), n, k, _i32(idx, "idx"), _ptr(ws), _nbytes(ws),
                                  _status_ptr(dev_status), _stream(stream)), "tb_topk")


def tb_topk_noalloc(shape: Shape, s, n: int, k: int, idx, dev_status=None, stream=None):
    """tb_topk for callers that cannot allocate: its scratch is a static array inside libtb."""
    if s.dtype != torch.float32:
        raise TypeError("s must be float32")
    _need(s, shape.B * shape.Hkv * n, "s")
    _need(idx, shape.B * shape.Hkv * max(k, 0), "idx")
    _check(load_library().tb_topk_noalloc(ctypes.byref(shape.c()), _ptr(s), n, k, _i32(idx, "idx"),
                                          _status_ptr(dev_status), _stream(stream)), "tb_topk_noalloc")


def tb_expand(shape: Shape, idx, k: int, r: int, n_pred: int, n_t: int, sel, sel_stride: int, counts,
              dev_status=None, stream=None):
    rows = shape.B * shape.Hkv
    _need(idx, rows * max(k, 0), "idx")
    _need(sel, rows * max(sel_stride, 0), "sel")
    _need(counts, rows, "counts")
    _check(load_library().tb_expand(ctypes.byref(shape.c()), _i32(idx, "idx"), k, r, n_pred, n_t,
                                    _i32(sel, "sel"), sel_stride, _i32(counts, "counts"),
                                    _status_ptr(dev_status), _stream(stream)), "tb_expand")


def tb_sparse_decode_attn(shape: Shape, q, K, V, sel, counts, sel_stride: int, scale: float, out, ws,
                          dev_status=None, stream=None):
    rows = shape.B * shape.Hkv
    _need(q, shape.B * shape.Hq * shape.D, "q")
    _need(K, rows * shape.cap * shape.D, "K")
    _need(V, rows * shape.cap * shape.D, "V")
    _need(sel, rows * max(sel_stride, 0), "sel")
    _need(counts, rows, "counts")
    _need(out, shape.B * shape.Hq * shape.D, "out")
    _check(load_library().tb_sparse_decode_attn(
        ctypes.byref(shape.c()), _bf16(q, "q"), _kv(K, "K"), _kv(V, "V"), _i32(sel, "sel"),
        _i32(counts, "counts"), sel_stride, scale, _bf16(out, "out"), _ptr(ws), _nbytes(ws),
        _status_ptr(dev_status), _stream(stream)), "tb_sparse_decode_attn")


def tb_decode_step(shape: Shape, k: int, T: int, r: int, agg: int, scale: float, t: int, n: int, *, q, q_imp,
                   K_new, V_new, Wk, K, V, Kp, idx_state, n_pred: "ctypes.c_int64", sel, sel_stride: int, counts,
                   out, ws, dev_status=None, stream=None, flags: int = 0):
    """One decode step of one layer (see include/tb.h). n_pred is a ctypes.c_int64 carried across steps."""
    params = _StepParams(k, T, r, agg, scale, flags)
    _need_step(shape, q, q_imp, K_new, V_new, Wk, K, V, Kp, out)
    _need_state(shape, _centres(k, r, flags), sel_stride, idx_state, sel, counts)
    _check(load_library().tb_decode_step(
        ctypes.byref(shape.c()), ctypes.byref(params), t, n, _bf16(q, "q"), _bf16(q_imp, "q_imp"),
        _bf16(K_new, "K_new"), _bf16(V_new, "V_new"), _bf16(Wk, "Wk"), _kv(K, "K"), _kv(V, "V"),
        _bf16(Kp, "Kp"), _i32(idx_state, "idx_state"), ctypes.byref(n_pred), _i32(sel, "sel"), sel_stride,
        _i32(counts, "counts"), _bf16(out, "out"), _ptr(ws), _nbytes(ws), _status_ptr(dev_status),
        _stream(stream)), "tb_decode_step")


def tb_decode_step_buffered(shape: Shape, k: int, T: int, r: int, agg: int, scale: float, sink: int, window: int,
                            t: int, n: int, *, q, q_imp, K_new, V_new, Wk, K, V, Kp, idx_state,
                            n_pred: "ctypes.c_int64", proj_end: "ctypes.c_int64", sel, sel_stride: int, counts, out,
                            ws, dev_status=None, stream=None, flags: int = 0):
    """One decode step with sink and local-window buffers (see include/tb.h). n_pred and proj_end are
    ctypes.c_int64 carried across steps."""
    params = _StepParams(k, T, r, agg, scale, flags)
    bufs = _BufferParams(sink, window)
    _need_step(shape, q, q_imp, K_new, V_new, Wk, K, V, Kp, out)
    _need_state(shape, _centres(k, r, flags), sel_stride, idx_state, sel, counts)
    _check(load_library().tb_decode_step_buffered(
        ctypes.byref(shape.c()), ctypes.byref(params), ctypes.byref(bufs), t, n, _bf16(q, "q"), _bf16(q_imp, "q_imp"),
        _bf16(K_new, "K_new"), _bf16(V_new, "V_new"), _bf16(Wk, "Wk"), _kv(K, "K"), _kv(V, "V"),
        _bf16(Kp, "Kp"), _i32(idx_state, "idx_state"), ctypes.byref(n_pred), ctypes.byref(proj_end),
        _i32(sel, "sel"), sel_stride, _i32(counts, "counts"), _bf16(out, "out"), _ptr(ws), _nbytes(ws),
        _status_ptr(dev_status), _stream(stream)), "tb_decode_step_buffered")


def tb_decode_step_ragged(shape: Shape, k: int, T: int, r: int, agg: int, scale: float, t: int, n_host, n_dev, *,
                          q, q_imp, K_new, V_new, Wk, K, V, Kp, idx_state, n_pred, sel, sel_stride: int, counts,
                          out, ws, dev_status=None, stream=None, flags: int = 0):
    """One decode step for a batch of sequences of different lengths (see include/tb.h). n_host and n_pred
    are ctypes int64 arrays of B entries on the host (n_pred carried across steps); n_dev is an int64
    device tensor [B] holding the values of n_host."""
    for arr, name in ((n_host, "n_host"), (n_pred, "n_pred")):
        # the C side reads B int64 values from each: anything else would be read past its end or misread
        if not isinstance(arr, ctypes.Array) or arr._type_ is not ctypes.c_int64:
            raise TypeError(f"{name} must be a ctypes array (ctypes.c_int64 * {shape.B}), got {type(arr).__name__}")
        if len(arr) != shape.B:
            raise ValueError(f"n_host and n_pred need {shape.B} entries")
    if n_dev.dtype != torch.int64:
        raise TypeError(f"n_dev must be int64, got {n_dev.dtype}")
    _need(n_dev, shape.B, "n_dev")
    _need_step(shape, q, q_imp, K_new, V_new, Wk, K, V, Kp, out)
    _need_state(shape, _centres(k, r, flags), sel_stride, idx_state, sel, counts)
    params = _StepParams(k, T, r, agg, scale, flags)
    _check(load_library().tb_decode_step_ragged(
        ctypes.byref(shape.c()), ctypes.byref(params), t, ctypes.cast(n_host, ctypes.c_void_p), _ptr(n_dev),
        _bf16(q, "q"), _bf16(q_imp, "q_imp"), _bf16(K_new, "K_new"), _bf16(V_new, "V_new"), _bf16(Wk, "Wk"),
        _kv(K, "K"), _kv(V, "V"), _bf16(Kp, "Kp"), _i32(idx_state, "idx_state"), ctypes.cast(n_pred, ctypes.c_void_p),
        _i32(sel, "sel"), sel_stride, _i32(counts, "counts"), _bf16(out, "out"), _ptr(ws), _nbytes(ws),
        _status_ptr(dev_status), _stream(stream)), "tb_decode_step_ragged")


def tb_predict_queries(x, W1, W2, q_imp, ws=None, dev_status=None, stream=None):
    """q_imp [B, O] = RNE(SiLU(x W1^T) W2^T): x [B, E], W1 [F, E], W2 [O, F] bf16 (see include/tb.h).
    ws: a device buffer of at least B F 4 bytes (allocated here if None)."""
    B, E = x.shape[0], x.shape[-1]
    F, O = W1.shape[0], W2.shape[0]
    if W1.shape[-1] != E or W2.shape[-1] != F or q_imp.numel() != B * O:
        raise ValueError("shapes: x [B, E], W1 [F, E], W2 [O, F], q_imp [B, O]")
    if ws is None:
        ws = torch.empty(B * F * 4, dtype=torch.uint8, device=x.device)
    _check(load_library().tb_predict_queries(_bf16(x, "x"), _bf16(W1, "W1"), _bf16(W2, "W2"), B, E, F, O,
                                             _bf16(q_imp, "q_imp"), _ptr(ws), ws.numel() * ws.element_size(),
                                             _status_ptr(dev_status), _stream(stream)), "tb_predict_queries")
    return q_imp


def sel_stride_for(k: int, T: int, r: int, n_max: int) -> int:
    """Selection row length that every step of an interval fits in."""
    return min(n_max + 1, k * (2 * r + 1)) + T - 1


class DecodeLayer:
    """Per-layer decode state on the device: the selection reused across a prediction interval.

    fused=False runs every step as separate kernels; pipeline=True runs a step with T = 1 and r = 0 as the
    three-kernel form instead of the single cooperative kernel (both give the results of tb_decode_step)."""

    def __init__(self, shape: Shape, k: int, T: int = 1, r: int = 0, agg: int = TB_AGG_MEAN,
                 scale: float | None = None, n_max: int | None = None, device=None, fused: bool = True,
                 budget_neighbours: bool = False, pipeline: bool = False):
        self.shape, self.k, self.T, self.r, self.agg = shape, k, T, r, agg
        self.flags = ((0 if fused else TB_STEP_UNFUSED) | (TB_STEP_BUDGET_NEIGHBOURS if budget_neighbours else 0)
                      | (TB_STEP_PIPELINE if pipeline else 0))
        # centres kept per prediction (idx_state row length)
        self.kc = max(1, k // (2 * r + 1)) if budget_neighbours else k
        self.scale = scale if scale is not None else shape.D ** -0.5
        n_max = shape.cap - 1 if n_max is None else n_max
        dev = device or "cuda"
        rows = (shape.B, shape.Hkv)
        self.sel_stride = sel_stride_for(self.kc, T, r, n_max)
        self.idx_state = torch.zeros(rows + (self.kc,), dtype=torch.int32, device=dev)
        self.sel = torch.zeros(rows + (self.sel_stride,), dtype=torch.int32, device=dev)
        self.counts = torch.zeros(rows, dtype=torch.int32, device=dev)
        self.n_pred = ctypes.c_int64(0)
        self.ws = workspace(shape, n_max, max(k, self.kc), self.sel_stride, device=dev)
        self.status = dev_status(dev)
        # marshalled once: the structs, the layer's own buffers, and the caller's tensors per identity
        self._lib = load_library()
        self._shape_c = shape.c()
        self._params = _StepParams(k, T, r, agg, self.scale, self.flags)
        self._own = (_i32(self.idx_state, "idx_state"), _i32(self.sel, "sel"), _i32(self.counts, "counts"),
                     _ptr(self.ws), _nbytes(self.ws), _status_ptr(self.status))
        self._seen = {}

    def _args(self, tensors):
        key = tuple((id(x), x.data_ptr(), x.dtype) for x in tensors)   # (a new tensor misses: checked again)
        got = self._seen.get(key)
        if got is None:
            q, q_imp, K_new, V_new, Wk, K, V, Kp, out = tensors
            _need_step(self.shape, q, q_imp, K_new, V_new, Wk, K, V, Kp, out)
            got = (_bf16(q, "q"), _bf16(q_imp, "q_imp"), _bf16(K_new, "K_new"), _bf16(V_new, "V_new"),
                   _bf16(Wk, "Wk"), _kv(K, "K"), _kv(V, "V"), _bf16(Kp, "Kp"), _bf16(out, "out"))
            if len(self._seen) > 256:
                self._seen.clear()
            self._seen[key] = got
        return got

    def step(self, t: int, n: int, *, q, q_imp, K_new, V_new, Wk, K, V, Kp, out, stream=None):
        pq, pqi, pkn, pvn, pwk, pk, pv, pkp, pout = self._args((q, q_imp, K_new, V_new, Wk, K, V, Kp, out))
        idx, sel, cnt, ws, wsb, st = self._own
        _check(self._lib.tb_decode_step(ctypes.byref(self._shape_c), ctypes.byref(self._params), t, n, pq, pqi, pkn,
                                        pvn, pwk, pk, pv, pkp, idx, ctypes.byref(self.n_pred), sel, self.sel_stride,
                                        cnt, pout, ws, wsb, st, _stream(stream)), "tb_decode_step")
        return out


def tb_decode_layers(shape: Shape, k: int, agg: int, scale: float, n: int, layers, sel_stride: int,
                     dev_status=None, stream=None, select_stream=None):
    """One decode step of len(layers) consumer layers (see include/tb.h): layer l's selection runs on
    select_stream while earlier layers attend on stream. layers: one dict per layer with the tensors of
    tb_decode_step (q, q_imp, K_new, V_new, Wk, K, V, Kp, idx_state, sel, counts, out) and its own zero-filled
    workspace ws."""
    if select_stream is None:
        raise ValueError("tb_decode_layers needs a select_stream distinct from stream")
    arr = (_LayerBuffers * len(layers))()
    for i, y in enumerate(layers):
        _need_step(shape, y["q"], y["q_imp"], y["K_new"], y["V_new"], y["Wk"], y["K"], y["V"], y["Kp"], y["out"])
        _need_state(shape, k, sel_stride, y["idx_state"], y["sel"], y["counts"])
        arr[i] = _LayerBuffers(
            _bf16(y["q"], "q"), _bf16(y["q_imp"], "q_imp"), _bf16(y["K_new"], "K_new"), _bf16(y["V_new"], "V_new"),
            _bf16(y["Wk"], "Wk"), _bf16(y["K"], "K"), _bf16(y["V"], "V"), _bf16(y["Kp"], "Kp"),
            _i32(y["idx_state"], "idx_state"), _i32(y["sel"], "sel"), _i32(y["counts"], "counts"),
            _bf16(y["out"], "out"), _ptr(y["ws"]), _nbytes(y["ws"]))
    params = _StepParams(k, 1, 0, agg, scale, 0)
    _check(load_library().tb_decode_layers(ctypes.byref(shape.c()), ctypes.byref(params), n, len(layers), arr,
                                           sel_stride, _status_ptr(dev_status), _stream(stream),
                                           _stream(select_stream)), "tb_decode_layers")


class DecodeStack:
    """Decode state of L consumer layers stepped together by tb_decode_layers (T = 1, r = 0): per layer its
    selection, counts and own workspace. step() takes per-layer lists of the step's tensors."""

    def __init__(self, shape: Shape, L: int, k: int, agg: int = TB_AGG_MEAN, scale: float | None = None,
                 n_max: int | None = None, device=None):
        self.shape, self.L, self.k, self.agg = shape, L, k, agg
        self.scale = scale if scale is not None else shape.D ** -0.5
        n_max = shape.cap - 1 if n_max is None else n_max
        dev = device or "cuda"
        rows = (shape.B, shape.Hkv)
        self.sel_stride = k
        self.idx_state = [torch.zeros(rows + (k,), dtype=torch.int32, device=dev) for _ in range(L)]
        self.sel = [torch.zeros(rows + (k,), dtype=torch.int32, device=dev) for _ in range(L)]
        self.counts = [torch.zeros(rows, dtype=torch.int32, device=dev) for _ in range(L)]
        self.ws = [workspace(shape, n_max, k, k, device=dev) for _ in range(L)]
        self.status = dev_status(dev)
        self.select_stream = torch.cuda.Stream(device=dev)
        self._lib = load_library()
        self._shape_c = shape.c()
        self._params = _StepParams(k, 1, 0, agg, self.scale, 0)
        self._seen = {}

    def _arr(self, per_layer):
        key = tuple((id(x), x.data_ptr()) for y in per_layer for x in y)
        got = self._seen.get(key)
        if got is None:
            arr = (_LayerBuffers * self.L)()
            for l, (q, q_imp, K_new, V_new, Wk, K, V, Kp, out) in enumerate(per_layer):
                _need_step(self.shape, q, q_imp, K_new, V_new, Wk, K, V, Kp, out)
                arr[l] = _LayerBuffers(
                    _bf16(q, "q"), _bf16(q_imp, "q_imp"), _bf16(K_new, "K_new"), _bf16(V_new, "V_new"),
                    _bf16(Wk, "Wk"), _bf16(K, "K"), _bf16(V, "V"), _bf16(Kp, "Kp"),
                    _i32(self.idx_state[l], "idx_state"), _i32(self.sel[l], "sel"), _i32(self.counts[l], "counts"),
                    _bf16(out, "out"), _ptr(self.ws[l]), _nbytes(self.ws[l]))
            if len(self._seen) > 64:
                self._seen.clear()
            self._seen[key] = got = arr
        return got

    def step(self, n: int, *, q, q_imp, K_new, V_new, Wk, K, V, Kp, out, stream=None):
        """Each argument is a list of L tensors (layer order). n: tokens per layer before this step's append."""
        per_layer = list(zip(q, q_imp, K_new, V_new, Wk, K, V, Kp, out))
        if len(per_layer) != self.L:
            raise ValueError(f"expected {self.L} layers, got {len(per_layer)}")
        arr = self._arr(per_layer)
        _check(self._lib.tb_decode_layers(ctypes.byref(self._shape_c), ctypes.byref(self._params), n, self.L, arr,
                                          self.sel_stride, _status_ptr(self.status), _stream(stream),
                                          _stream(self.select_stream)), "tb_decode_layers")
        return out


class BufferedDecodeLayer:
    """Per-layer decode state with sink and local-window buffers: Kp grows in batches of `window` rows
    (proj_end counts them; pass the rows projected at prefill), the predictor picks the important tokens
    among [sink, proj_end)."""

    def __init__(self, shape: Shape, k: int, sink: int, window: int, proj_end: int, T: int = 1, r: int = 0,
                 agg: int = TB_AGG_MEAN, scale: float | None = None, n_max: int | None = None, device=None,
                 budget_neighbours: bool = False):
        self.shape, self.k, self.T, self.r, self.agg = shape, k, T, r, agg
        self.sink, self.window = sink, window
        self.flags = TB_STEP_BUDGET_NEIGHBOURS if budget_neighbours else 0
        self.kc = max(1, k // (2 * r + 1)) if budget_neighbours else k
        self.scale = scale if scale is not None else shape.D ** -0.5
        n_max = shape.cap - 1 if n_max is None else n_max
        dev = device or "cuda"
        rows = (shape.B, shape.Hkv)
        # sink + widened centres + window (up to 2W - 1 at a prediction) + the interval's steps
        self.sel_stride = min(n_max + 1, sink + min(n_max + 1, self.kc * (2 * r + 1)) + 2 * window + T)
        self.idx_state = torch.zeros(rows + (self.kc,), dtype=torch.int32, device=dev)
        self.sel = torch.zeros(rows + (self.sel_stride,), dtype=torch.int32, device=dev)
        self.counts = torch.zeros(rows, dtype=torch.int32, device=dev)
        self.n_pred = ctypes.c_int64(0)
        self.proj_end = ctypes.c_int64(proj_end)
        self.ws = workspace(shape, n_max, max(k, self.kc), self.sel_stride, device=dev)
        self.status = dev_status(dev)

    def step(self, t: int, n: int, *, q, q_imp, K_new, V_new, Wk, K, V, Kp, out, stream=None):
        tb_decode_step_buffered(self.shape, self.k, self.T, self.r, self.agg, self.scale, self.sink, self.window,
                                t, n, q=q, q_imp=q_imp, K_new=K_new, V_new=V_new, Wk=Wk, K=K, V=V, Kp=Kp,
                                idx_state=self.idx_state, n_pred=self.n_pred, proj_end=self.proj_end, sel=self.sel,
                                sel_stride=self.sel_stride, counts=self.counts, out=out, ws=self.ws,
                                dev_status=self.status, stream=stream, flags=self.flags)
        return out


class RaggedDecodeLayer:
    """Per-layer decode state for a batch whose sequences have different lengths (see
    tb_decode_step_ragged in include/tb.h): n_pred is kept per sequence."""

    def __init__(self, shape: Shape, k: int, T: int = 1, r: int = 0, agg: int = TB_AGG_MEAN,
                 scale: float | None = None, n_max: int | None = None, device=None, budget_neighbours: bool = False):
        self.shape, self.k, self.T, self.r, self.agg = shape, k, T, r, agg
        self.flags = TB_STEP_BUDGET_NEIGHBOURS if budget_neighbours else 0
        self.kc = max(1, k // (2 * r + 1)) if budget_neighbours else k
        self.scale = scale if scale is not None else shape.D ** -0.5
        n_max = shape.cap - 1 if n_max is None else n_max
        dev = device or "cuda"
        rows = (shape.B, shape.Hkv)
        self.sel_stride = sel_stride_for(self.kc, T, r, n_max)
        self.idx_state = torch.zeros(rows + (self.kc,), dtype=torch.int32, device=dev)
        self.sel = torch.zeros(rows + (self.sel_stride,), dtype=torch.int32, device=dev)
        self.counts = torch.zeros(rows, dtype=torch.int32, device=dev)
        self.n_pred = (ctypes.c_int64 * shape.B)()
        self.n_host = (ctypes.c_int64 * shape.B)()
        self.n_dev = torch.zeros(shape.B, dtype=torch.int64, device=dev)
        self.ws = workspace(shape, n_max, max(k, self.kc), self.sel_stride, device=dev)
        self.status = dev_status(dev)

    def step(self, t: int, ns, *, q, q_imp, K_new, V_new, Wk, K, V, Kp, out, stream=None):
        """ns: tokens per sequence before this step's append (B ints)."""
        ns = [int(v) for v in ns]
        if len(ns) != self.shape.B:
            raise ValueError(f"ns holds {len(ns)} lengths; the batch has {self.shape.B} sequences")
        _need_step(self.shape, q, q_imp, K_new, V_new, Wk, K, V, Kp, out)
        if ns != list(self.n_host):   # (unchanged lengths need no copy, so repeated steps can be captured)
            for b, v in enumerate(ns):
                self.n_host[b] = v
            self.n_dev.copy_(torch.tensor(ns, dtype=torch.int64), non_blocking=False)
        params = _StepParams(self.k, self.T, self.r, self.agg, self.scale, self.flags)
        _check(load_library().tb_decode_step_ragged(
            ctypes.byref(self.shape.c()), ctypes.byref(params), t, ctypes.cast(self.n_host, ctypes.c_void_p),
            _ptr(self.n_dev), _bf16(q, "q"), _bf16(q_imp, "q_imp"), _bf16(K_new, "K_new"), _bf16(V_new, "V_new"),
            _bf16(Wk, "Wk"), _kv(K, "K"), _kv(V, "V"), _bf16(Kp, "Kp"), _i32(self.idx_state, "idx_state"),
            ctypes.cast(self.n_pred, ctypes.c_void_p), _i32(self.sel, "sel"), self.sel_stride,
            _i32(self.counts, "counts"), _bf16(out, "out"), _ptr(self.ws), _nbytes(self.ws), _status_ptr(self.status),
            _stream(stream)), "tb_decode_step_ragged")
        return out
