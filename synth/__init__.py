"""Seeded synthetic inputs for the TokenButler decode-time hot path.

This module is shared by the tests, the benchmark and the smoke check. It
draws random tensors and places them; it holds none of the method's
arithmetic (no projection, scoring, selection or attention).

TokenButler's evaluations use RULER, LongBench, AIME24 and their own co-reference task
(gist.science summary, "Experimental Results"); none of that data is used.
These seeded tensors stand in for them at those evaluations' context-length scale
(16K-128K tokens) and at a Llama-3-8B-shaped attention layer.

Recipe (all draws in fp32 from a CPU ``torch.Generator``, then rounded to bf16
by torch's round-to-nearest-even):
  per layer, generator seeded with ``layer_seed(seed, layer)``, drawn in order
    1. Wk    [Hkv, D, dp]    ~ N(0, 1/D)
    2. K     [B, Hkv, N, D]  ~ N(0, 1)
    3. V     [B, Hkv, N, D]  ~ N(0, 1)
    4. q     [B, Hq, D]      ~ N(0, 1)
    5. q_imp [B, Hq, dp]     ~ N(0, 1)
    6. outlier key channels: the first ``outliers`` entries of randperm(D);
       those channels of K are multiplied by ``outlier_scale`` (all heads and
       tokens)
    7. heavy hitters: per (b, h) the first ``planted`` entries of randperm(N);
       those key rows become c*normalize(Wk[h] @ u) + (their drawn row), with
       u = normalize(mean over the group's q_imp rows) and c = 3*sqrt(D)
  per decode step, generator seeded with ``step_seed(seed, layer, step)``:
    q [B,Hq,D], q_imp [B,Hq,dp], K_new [B,Hkv,D], V_new [B,Hkv,D] ~ N(0, 1),
    K_new with the layer's outlier channels scaled the same way.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    dp: int
    N: int                      # cached tokens (before decoding starts)
    k: int                      # budget per (batch, KV head)
    T: int = 1                  # prediction interval
    r: int = 0                  # neighbour radius
    layers: int = 1
    steps: int = 1
    outliers: int = 0
    outlier_scale: float = 8.0
    planted: int = 0
    seed: int = 0
    budgets: tuple = field(default_factory=tuple)   # extra budgets (fractions of N) to sweep

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


def budget(p: float, n: int) -> int:
    """Budget for a fraction p of n tokens, rounded up (10% of 32768 -> 3277)."""
    return min(n, max(1, math.ceil(p * n - 1e-9)))


WORKLOADS = [
    # 0: small parity case
    Workload("small-N2048-k128", B=1, Hq=8, Hkv=8, D=64, dp=16, N=2048, k=128, seed=0),
    # 1: Llama-3-8B-shaped layer, one decode step at N=32K, 10% budget
    Workload("llama3-8b-layer-N32768-k10pct", B=1, Hq=32, Hkv=8, D=128, dp=32, N=32768,
             k=budget(0.10, 32768), outliers=4, seed=1),
    # 2: 32-layer stack, B=8, interval reuse T=16 with +-1 neighbours, 64 steps
    Workload("llama3-8b-32layer-B8-N16384-k1024-T16-r1", B=8, Hq=32, Hkv=8, D=128, dp=32,
             N=16384, k=1024, T=16, r=1, layers=32, steps=64, outliers=4, seed=2),
    # 3: long context with planted heavy hitters
    Workload("long-B4-N131072-k2048-planted64", B=4, Hq=32, Hkv=8, D=128, dp=32, N=131072,
             k=2048, outliers=4, planted=64, seed=3),
    # 4: prefill projection + budget sweep
    Workload("prefill-B2-N65536-sweep", B=2, Hq=32, Hkv=8, D=128, dp=32, N=65536,
             k=budget(0.10, 65536), outliers=4, seed=4,
             budgets=(0.01, 0.05, 0.10, 0.25, 1.00)),
]


def layer_seed(seed: int, layer: int) -> int:
    return seed * 1_000_003 + layer


def step_seed(seed: int, layer: int, step: int) -> int:
    return (seed * 1_000_003 + layer) * 100_003 + step + 1


def _randn(gen, shape, std=1.0):
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def make_layer(w: Workload, layer: int = 0, cap: int | None = None, n: int | None = None):
    """One layer's tensors on the CPU (bf16). K/V/ have ``cap`` rows (>= n), rows >= n are zero.

    Returns dict(Wk, K, V, q, q_imp, outlier_ch, planted_pos).
    """
    n = w.N if n is None else n
    cap = n if cap is None else cap
    assert cap >= n
    gen = torch.Generator().manual_seed(layer_seed(w.seed, layer))
    Wk = _randn(gen, (w.Hkv, w.D, w.dp), std=1.0 / math.sqrt(w.D))
    K = _randn(gen, (w.B, w.Hkv, n, w.D))
    V = _randn(gen, (w.B, w.Hkv, n, w.D))
    q = _randn(gen, (w.B, w.Hq, w.D))
    q_imp = _randn(gen, (w.B, w.Hq, w.dp))
    outlier_ch = torch.randperm(w.D, generator=gen)[: w.outliers]
    if w.outliers:
        K[..., outlier_ch] *= w.outlier_scale
    planted_pos = None
    if w.planted:
        Wk_b = Wk.to(torch.bfloat16).float()
        qi_b = q_imp.to(torch.bfloat16).float()
        planted_pos = torch.empty((w.B, w.Hkv, w.planted), dtype=torch.int64)
        c = 3.0 * math.sqrt(w.D)
        for b in range(w.B):
            for h in range(w.Hkv):
                pos = torch.randperm(n, generator=gen)[: w.planted]
                planted_pos[b, h] = pos
                u = qi_b[b, h * w.G:(h + 1) * w.G].mean(0)
                u = u / u.norm()
                dvec = Wk_b[h] @ u
                dvec = dvec / dvec.norm()
                K[b, h, pos] += c * dvec
    out = dict(
        Wk=Wk.to(torch.bfloat16),
        K=_pad_rows(K.to(torch.bfloat16), cap),
        V=_pad_rows(V.to(torch.bfloat16), cap),
        q=q.to(torch.bfloat16),
        q_imp=q_imp.to(torch.bfloat16),
        outlier_ch=outlier_ch,
        planted_pos=planted_pos,
    )
    return out


def _pad_rows(x: torch.Tensor, cap: int) -> torch.Tensor:
    n = x.shape[2]
    if cap == n:
        return x.contiguous()
    y = torch.zeros(x.shape[:2] + (cap,) + x.shape[3:], dtype=x.dtype)
    y[:, :, :n] = x
    return y


def make_step(w: Workload, layer: int, step: int, outlier_ch=None):
    """Per-step draws (bf16, CPU): q, q_imp, K_new, V_new."""
    gen = torch.Generator().manual_seed(step_seed(w.seed, layer, step))
    q = _randn(gen, (w.B, w.Hq, w.D))
    q_imp = _randn(gen, (w.B, w.Hq, w.dp))
    K_new = _randn(gen, (w.B, w.Hkv, w.D))
    V_new = _randn(gen, (w.B, w.Hkv, w.D))
    if outlier_ch is not None and len(outlier_ch):
        K_new[..., outlier_ch] *= w.outlier_scale
    return dict(q=q.to(torch.bfloat16), q_imp=q_imp.to(torch.bfloat16),
                K_new=K_new.to(torch.bfloat16), V_new=V_new.to(torch.bfloat16))


def small(B=1, Hq=4, Hkv=2, D=16, dp=8, N=64, k=8, T=1, r=0, seed=123, **kw) -> Workload:
    """A tiny ad-hoc workload for unit tests."""
    return Workload(f"adhoc-B{B}-Hq{Hq}-Hkv{Hkv}-D{D}-dp{dp}-N{N}-k{k}", B=B, Hq=Hq, Hkv=Hkv,
                    D=D, dp=dp, N=N, k=k, T=T, r=r, seed=seed, **kw)


def integer_valued(shape, lo=-4, hi=4, seed=0) -> torch.Tensor:
    """Integer-valued bf16 tensor (exact in bf16 and in every sum the tests form)."""
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=gen, dtype=torch.int32).to(torch.bfloat16)
