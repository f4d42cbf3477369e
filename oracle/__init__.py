"""CPU oracle for the TokenButler decode-time hot path (fp64).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product library
never calls it, and it never calls the product library.

The arithmetic lives in ``tb_oracle.c`` (plain C, fp64, OpenMP over
independent (batch, KV head) rows); this module compiles it with gcc when the
shared object is missing or stale and marshals numpy arrays in and out. The
only logic written here in Python is the step orchestration of the prediction
interval and of the buffers (``decode_step``, ``decode_step_buffered``,
``decode_step_ragged``), which is host-side control flow, and the predictor
MLP (``predict_queries``: two numpy matmuls and SiLU in fp64).

Sources: "TokenButler: Token Importance is Predictable" -- the arXiv abstract
(searcharxiv.com / fugumt.com pages) and the gist.science technical summary,
sections "Core Architecture", "Inference Strategy" and "Optimizations".

Parity status per function:
  bf16_round, project, score, topk, expand, attn   pinned by tests/test_oracle_pins.py
  decode_step (interval reuse + neighbour fetching + tail)
      the reading of when to predict and what the tail is comes from no page
      (the pages give no schedule detail); its invariants (T=1 equals
      per-step selection, superset, bounds) are pinned, the schedule itself
      is "parity unpinned" by the pages.
  centres (budget-preserving neighbours), decode_step_buffered /
  buffered_select (sink, local window, batched projection)
      readings of the pages' Inference Strategy and Batching; pinned by
      brute-force rank counts and the structure of every selection, the
      rules themselves "parity unpinned" by the pages.
  decode_step_ragged   pinned by its equality with the batched step at equal
      lengths and, at unequal lengths, by torch SDPA in fp64 (full budget),
      a brute-force rank count and independence between sequences.
  silu, predict_queries   pinned against torch's SiLU and matmul in fp64 and
      SiLU's odd-part identity; the MLP's shape is "parity unpinned" by the
      pages.
tests/test_oracle_mutants.py plants plausible mistakes in private copies of
this package and checks that a pin fails for each.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tb_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_STAMP = _LIB + ".buildhash"
_lock = threading.Lock()
_lib = None

AGG_MEAN = 0
AGG_MAX = 1


def _src_hash() -> str:
    with open(_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def build(force: bool = False) -> str:
    """Compile tb_oracle.c into liboracle.so (gcc, -O2, OpenMP, no fp contraction)."""
    h = _src_hash()
    if not force and os.path.exists(_LIB) and os.path.exists(_STAMP):
        with open(_STAMP) as f:
            if f.read().strip() == h:
                return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    with open(_STAMP, "w") as f:
        f.write(h)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.tbo_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.tbo_bf16_to_double.restype = dbl
        lib.tbo_bf16_from_double.argtypes = [dbl]
        lib.tbo_bf16_from_double.restype = ctypes.c_uint16
        lib.tbo_num_threads.restype = i32
        lib.tbo_set_num_threads.argtypes = [i32]
        lib.tbo_project.argtypes = [i32, i32, i64, i32, i32, P, P, P, P]
        lib.tbo_score.argtypes = [i32, i32, i32, i64, i32, P, P, i32, P, P]
        lib.tbo_topk.argtypes = [i64, i64, i64, P, P]
        lib.tbo_topk.restype = i32
        lib.tbo_expand.argtypes = [i64, i64, P, i32, i64, i64, P, i64, P]
        lib.tbo_expand.restype = i32
        lib.tbo_attn.argtypes = [i32, i32, i32, i32, i64, P, P, P, P, P, i64, dbl, P, P]
        lib.tbo_attn.restype = i32
        _lib = lib
        return lib


# ---------------------------------------------------------------- helpers

def as_u16(x) -> np.ndarray:
    """bf16 data as a contiguous uint16 numpy array (accepts a CPU torch bf16 tensor)."""
    if hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch  # only for the view; the oracle does no torch arithmetic
        x = x.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns (uint16), got {x.dtype}")
    return x


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().tbo_num_threads())


def set_num_threads(n: int) -> None:
    _load().tbo_set_num_threads(int(n))


def bf16_to_double(bits: int) -> float:
    return float(_load().tbo_bf16_to_double(int(bits)))


def bf16_round(x) -> np.ndarray:
    """RNE of fp64 values to bf16, returned as uint16 bit patterns (one rounding step)."""
    lib = _load()
    a = np.asarray(x, dtype=np.float64)
    flat = a.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    for i, v in enumerate(flat):
        out[i] = lib.tbo_bf16_from_double(float(v))
    return out.reshape(a.shape)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64 (bits << 16 is an fp32 pattern)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- steps

def project(K, Wk):
    """Key projection. K [B,Hkv,n,D] bf16, Wk [Hkv,D,dp] bf16 -> (Kp bf16 bits, Kp fp64)."""
    K = as_u16(K)
    Wk = as_u16(Wk)
    B, Hkv, n, D = K.shape
    Hw, Dw, dp = Wk.shape
    assert Hw == Hkv and Dw == D
    Kp = np.empty((B, Hkv, n, dp), dtype=np.uint16)
    Kp64 = np.empty((B, Hkv, n, dp), dtype=np.float64)
    _load().tbo_project(B, Hkv, n, D, dp, _ptr(K), _ptr(Wk), _ptr(Kp), _ptr(Kp64))
    return Kp, Kp64


def score(q_imp, Kp, agg: int = AGG_MEAN):
    """Importance scores. q_imp [B,Hq,dp], Kp [B,Hkv,n,dp] -> (s fp64 [B,Hkv,n], l1 bound scale)."""
    q_imp = as_u16(q_imp)
    Kp = as_u16(Kp)
    B, Hq, dp = q_imp.shape
    Bk, Hkv, n, dpk = Kp.shape
    assert Bk == B and dpk == dp and Hq % Hkv == 0
    s = np.empty((B, Hkv, n), dtype=np.float64)
    l1 = np.empty((B, Hkv, n), dtype=np.float64)
    _load().tbo_score(B, Hq, Hkv, n, dp, _ptr(q_imp), _ptr(Kp), int(agg), _ptr(s), _ptr(l1))
    return s, l1


def topk(s, k: int) -> np.ndarray:
    """Sort-based top-k per row. s [..., n] (any float dtype; widened exactly) -> idx int32 [..., k] ascending."""
    s = np.ascontiguousarray(np.asarray(s, dtype=np.float64))
    n = s.shape[-1]
    rows = int(np.prod(s.shape[:-1])) if s.ndim > 1 else 1
    idx = np.empty(s.shape[:-1] + (k,), dtype=np.int32)
    rc = _load().tbo_topk(rows, n, k, _ptr(s), _ptr(idx))
    if rc != 0:
        raise ValueError("oracle top-k: NaN score or k outside [0, n]")
    return idx


def expand(idx, r: int, n_pred: int, n_t: int, sel_stride: int | None = None):
    """Neighbour fetching + tail. idx [..., k] ascending -> (sel [..., sel_stride], counts [...])."""
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int32))
    k = idx.shape[-1]
    rows = int(np.prod(idx.shape[:-1])) if idx.ndim > 1 else 1
    if sel_stride is None:
        sel_stride = min(n_pred, k * (2 * r + 1)) + max(0, n_t - n_pred)
    sel_stride = max(int(sel_stride), 1)
    sel = np.full(idx.shape[:-1] + (sel_stride,), -1, dtype=np.int32)
    counts = np.empty(idx.shape[:-1], dtype=np.int32)
    rc = _load().tbo_expand(rows, k, _ptr(idx), int(r), int(n_pred), int(n_t),
                            _ptr(sel), sel_stride, _ptr(counts))
    if rc != 0:
        raise ValueError("oracle expand: index out of range or sel_stride too small")
    return sel, counts


def attn(q, K, V, sel, counts, scale: float, with_wsum: bool = False):
    """Attention over selected rows. q [B,Hq,D], K/V [B,Hkv,n_cache,D], sel [B,Hkv,S], counts [B,Hkv]."""
    q = as_u16(q)
    K = as_u16(K)
    V = as_u16(V)
    B, Hq, D = q.shape
    Bk, Hkv, n_cache, Dk = K.shape
    assert Bk == B and Dk == D and V.shape == K.shape
    sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int32))
    counts = np.ascontiguousarray(np.asarray(counts, dtype=np.int32))
    assert sel.shape[:2] == (B, Hkv) and counts.shape == (B, Hkv)
    out = np.empty((B, Hq, D), dtype=np.float64)
    wsum = np.empty((B, Hq), dtype=np.float64)
    rc = _load().tbo_attn(B, Hq, Hkv, D, n_cache, _ptr(q), _ptr(K), _ptr(V), _ptr(sel),
                          _ptr(counts), sel.shape[2], float(scale), _ptr(out), _ptr(wsum))
    if rc != 0:
        raise ValueError("oracle attention: index out of range or empty selection")
    return (out, wsum) if with_wsum else out


def dense_attn(q, K, V, n: int, scale: float):
    """Dense attention over the first n cache rows (the selection [0, n))."""
    K = as_u16(K)
    B, Hkv = K.shape[:2]
    sel = np.broadcast_to(np.arange(n, dtype=np.int32), (B, Hkv, n)).copy()
    counts = np.full((B, Hkv), n, dtype=np.int32)
    return attn(q, K, V, sel, counts, scale)


class DecodeState:
    """Host-side state of the prediction interval for one layer."""

    def __init__(self):
        self.idx = None      # [B, Hkv, k] selection made at the last prediction step
        self.n_pred = 0      # tokens present when it was made


def centres(k: int, r: int, budget_neighbours: bool) -> int:
    """Tokens a prediction keeps before widening: k, or with budget-preserving
    neighbour fetching k // (2r + 1) (at least one), so that the widened
    selection stays within k. Reading of the summary's Neighbor Fetching
    (Optimizations): it names no budget rule; this variant is the plainest
    one that keeps |E| <= k (parity unpinned by the pages)."""
    return max(1, k // (2 * r + 1)) if budget_neighbours else k


def decode_step(state: DecodeState, t: int, n: int, *, q, q_imp, K_new, V_new, Wk,
                K, V, Kp, k: int, T: int, r: int, agg: int, scale: float, budget_neighbours: bool = False):
    """One decode step of one layer, on CPU copies of the caches (updated in place).

    [summary] Optimizations: the predictor runs once every T steps, its
    selection is reused in between and widened by +-r neighbours. Reading:
    step t predicts when t % T == 0, after appending its own token, so the
    prediction sees n+1 tokens; the tokens appended after a prediction (the
    tail) are attended as well.

    q [B,Hq,D], q_imp [B,Hq,dp], K_new/V_new [B,Hkv,D] bf16 (uint16 bits).
    K, V [B,Hkv,cap,D], Kp [B,Hkv,cap,dp] uint16 numpy arrays (mutated).
    Returns (out fp64 [B,Hq,D], sel, counts).
    """
    K_new = as_u16(K_new)
    V_new = as_u16(V_new)
    K[:, :, n, :] = K_new
    V[:, :, n, :] = V_new
    kp_new, _ = project(K_new[:, :, None, :], Wk)
    Kp[:, :, n, :] = kp_new[:, :, 0, :]
    n_t = n + 1
    if t % T == 0:
        s, _ = score(q_imp, np.ascontiguousarray(Kp[:, :, :n_t, :]), agg)
        state.idx = topk(s, centres(k, r, budget_neighbours))
        state.n_pred = n_t
    sel, counts = expand(state.idx, r, state.n_pred, n_t)
    out = attn(q, K, V, sel, counts, scale)
    return out, sel, counts


def buffered_select(idx, r: int, sink: int, proj_end: int, n_t: int) -> list:
    """Selection rows of the buffered step: the sink [0, min(S, n_t)), the
    windows [S+i-r, S+i+r] of the centres idx (relative to S) clipped to
    [S, proj_end), then the local window [max(proj_end, min(S, n_t)), n_t).
    idx [B, Hkv, kc] -> list of B*Hkv ascending lists."""
    idx = np.asarray(idx)
    S, P = int(sink), int(proj_end)
    pre = min(S, n_t)
    tail0 = max(P, pre)
    rows = []
    for b in range(idx.shape[0]):
        for h in range(idx.shape[1]):
            body = set()
            for i in idx[b, h].tolist():
                body.update(j for j in range(S + i - r, S + i + r + 1) if S <= j < P)
            rows.append(list(range(pre)) + sorted(body) + list(range(tail0, n_t)))
    return rows


class BufferedState(DecodeState):
    """Host-side state of the buffered step: also the number of rows Kp holds."""

    def __init__(self, proj_end: int):
        super().__init__()
        self.proj_end = int(proj_end)


def decode_step_buffered(state: BufferedState, t: int, n: int, *, q, q_imp, K_new, V_new, Wk, K, V, Kp,
                         k: int, T: int, r: int, agg: int, scale: float, sink: int, window: int,
                         budget_neighbours: bool = False):
    """One decode step with sink and local-window buffers.

    [summary] Inference Strategy: the first S tokens (sink) and a window of
    the newest tokens are always kept, the important buffer is filled from
    the predicted scores; Optimizations, Batching: keys are projected in
    batches of W tokens instead of at every step. Readings: the window is the
    tokens not yet projected; at a prediction step every whole batch of W
    tokens older than the newest W is projected first, so the window then
    holds W to 2W - 1 tokens; the important tokens are chosen among
    [S, proj_end) and widened by +-r inside that range; between predictions
    the new tokens join the selection (they are the window's newest).
    Returns (out fp64 [B,Hq,D], sel, counts).
    """
    K_new = as_u16(K_new)
    V_new = as_u16(V_new)
    K[:, :, n, :] = K_new
    V[:, :, n, :] = V_new
    n_t = n + 1
    S, W = int(sink), int(window)
    if t % T == 0:
        P = state.proj_end
        while n_t - W - P >= W:
            Kp[:, :, P:P + W, :], _ = project(np.ascontiguousarray(K[:, :, P:P + W, :]), Wk)
            P += W
        state.proj_end = P
        nc = max(0, P - S)
        kc = min(centres(k, r, budget_neighbours), nc)
        if kc > 0:
            s, _ = score(q_imp, np.ascontiguousarray(Kp[:, :, S:P, :]), agg)
            idx = topk(s, kc)                                   # relative to S
        else:
            idx = np.zeros(K.shape[:2] + (0,), dtype=np.int32)
        state.idx = idx
        state.n_pred = n_t
        state.sel_rows = buffered_select(idx, r, S, P, n_t)
    else:
        state.sel_rows = [row + [n] for row in state.sel_rows]
    B, Hkv = K.shape[:2]
    width = max(len(x) for x in state.sel_rows)
    sel = np.full((B, Hkv, width), -1, dtype=np.int32)
    counts = np.empty((B, Hkv), dtype=np.int32)
    for x, row in enumerate(state.sel_rows):
        sel[x // Hkv, x % Hkv, :len(row)] = row
        counts[x // Hkv, x % Hkv] = len(row)
    out = attn(q, K, V, sel, counts, scale)
    return out, sel, counts


def silu(v):
    """SiLU(v) = v / (1 + exp(-v)) in fp64."""
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


def predict_queries(x, W1, W2):
    """The importance-query predictor for B tokens.

    [summary] Core Architecture, Query Prediction: a small multi-layer
    perceptron turns the producer layer's hidden state into G low-dimensional
    importance queries for each KV head. Reading (the pages give no depth, width, activation or bias): two
    bias-free layers with SiLU between them, h = SiLU(x W1^T), q_imp =
    RNE_bf16(h W2^T), exact products and fp64 sums here.
    x [B, E], W1 [F, E], W2 [O, F] bf16 bits -> (q_imp bits [B, O], fp64 [B, O], h fp64 [B, F]).
    """
    xf = bf16_bits_to_f64(as_u16(x))
    w1 = bf16_bits_to_f64(as_u16(W1))
    w2 = bf16_bits_to_f64(as_u16(W2))
    h = silu(xf @ w1.T)
    y = h @ w2.T
    return bf16_round(y), y, h


def decode_step_ragged(states: list, t: int, ns, *, q, q_imp, K_new, V_new, Wk, K, V, Kp, k: int, T: int,
                       r: int, agg: int, scale: float, budget_neighbours: bool = False):
    """A decode step for a batch of sequences of different lengths: sequence b
    (n[b] tokens before the append) is exactly decode_step on its own slice
    of every tensor. states: one DecodeState per sequence. K, V, Kp mutated.
    Returns (out [B,Hq,D], sel [B,Hkv,width] padded with -1, counts [B,Hkv])."""
    q, q_imp = as_u16(q), as_u16(q_imp)
    K_new, V_new = as_u16(K_new), as_u16(V_new)
    outs, sels, cnts = [], [], []
    for b, nb in enumerate(ns):
        Kb, Vb, Kpb = K[b:b + 1], V[b:b + 1], Kp[b:b + 1]
        o, sl, c = decode_step(states[b], t, int(nb), q=q[b:b + 1], q_imp=q_imp[b:b + 1], K_new=K_new[b:b + 1],
                               V_new=V_new[b:b + 1], Wk=Wk, K=Kb, V=Vb, Kp=Kpb, k=k, T=T, r=r, agg=agg,
                               scale=scale, budget_neighbours=budget_neighbours)
        outs.append(o)
        sels.append(sl)
        cnts.append(c)
    width = max(x.shape[-1] for x in sels)
    sel = np.full((len(ns), sels[0].shape[1], width), -1, dtype=np.int32)
    for b, x in enumerate(sels):
        sel[b, :, :x.shape[-1]] = x[0]
    return np.concatenate(outs, axis=0), sel, np.concatenate(cnts, axis=0)
