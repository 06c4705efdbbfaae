"""Seeded synthetic inputs for MoE dispatch / combine.

This module draws inputs only: token activations, top-k routing, routing
weights, masks and stand-in expert outputs.  It performs none of the
dispatch / combine / layout arithmetic, so both the CPU oracle and the CUDA
path can consume the very same bytes.

Workload shapes follow the pages:
  * MORI PR #614 "perf(ep): InterNodeV1LL low-token latency on MI300X + CX7":
    the test_low_latency.py defaults (128 tokens, hidden 7168, top-k 8,
    288 experts) and the serving shape (4/8/16 tokens, hidden 6144, fp8
    dispatch, bf16 combine, top-k 8).
  * DeepEP PR #693 "Pipeline direct NVLink dispatch with triple-buffered
    prefetch", Validation: the "rank unbalanced ratio 1.5" run.

Every array is numpy; bf16 tensors are carried as their uint16 bit patterns.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BF16 = 0
FP8_E4M3 = 1


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of float32 data, rounded to nearest even (torch's cast)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


@dataclass
class Case:
    """One synthetic workload: shapes, routing and activations."""

    name: str
    T: int
    H: int
    K: int
    E: int
    R: int
    cap: int
    dtype: int                      # dispatch output type: BF16 or FP8_E4M3
    x: np.ndarray                   # uint16 [T, H]  (bf16 bits)
    topk_idx: np.ndarray            # int32  [T, K]  (-1 = masked)
    topk_weights: np.ndarray        # float32 [T, K]
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.H // 128


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.float32)
    z = z - z.max(axis=1, keepdims=True)
    e = np.exp(z, dtype=np.float32)
    return (e / e.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)


def _uniform_topk(rng: np.random.Generator, T: int, E: int, K: int) -> np.ndarray:
    # K distinct experts per token, in the random order argsort leaves them
    return np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int32)


def _required_cap(topk_idx: np.ndarray, E: int) -> int:
    """Largest number of unmasked entries any expert receives (buffer sizing)."""
    v = topk_idx[(topk_idx >= 0) & (topk_idx < E)]
    if v.size == 0:
        return 1
    return int(np.bincount(v, minlength=E).max())


def _skewed_topk(rng: np.random.Generator, T: int, E: int, R: int, K: int,
                 zipf_s: float, mask_p: float, target: float) -> tuple[np.ndarray, float, float]:
    """Rank-skewed, Zipf-within-rank routing with K distinct experts per token.

    p_e is proportional to a_rank(e) * (j + 1) ** -zipf_s, with j the expert's
    index inside its rank.  a_r = 1 except a_0, which is bisected (with the
    Gumbel noise and the mask held fixed) until rank 0's unmasked pair load is
    `target` times the mean rank load.  K distinct experts are drawn per token
    by Gumbel-top-k on log p_e.
    """
    epr = E // R
    j = np.arange(E) % epr
    base = -zipf_s * np.log(j + 1.0)
    gumbel = -np.log(-np.log(rng.random((T, E))))
    mask = rng.random((T, K)) < mask_p

    def draw(log_a0: float) -> tuple[np.ndarray, float]:
        logits = base + np.where(np.arange(E) < epr, log_a0, 0.0)
        idx = np.argsort(-(logits[None, :] + gumbel), axis=1)[:, :K].astype(np.int32)
        live = idx[~mask]
        load = np.bincount(live // epr, minlength=R).astype(np.float64)
        return idx, float(load[0] / load.mean())

    lo, hi = 0.0, math.log(50.0)
    for _ in range(60):
        mid = 0.5 * (lo + hi)
        _, ratio = draw(mid)
        if ratio < target:
            lo = mid
        else:
            hi = mid
    idx, ratio = draw(hi)
    idx = idx.copy()
    idx[mask] = -1
    return idx, ratio, math.exp(hi)


CONFIG_NAMES = ("tiny", "low4", "low8", "low16", "default_ll", "throughput", "imbalanced")


def make_case(name: str, seed: int = 0, T: int | None = None) -> Case:
    """Build one of the named workloads.

    tiny        T=64, H=2048, K=4 of E=32, R=4, bf16 dispatch, cap=T, 5% masked
    low4/8/16   T=4/8/16, H=6144, K=8 of E=128, R=16, fp8 dispatch, cap=T
    default_ll  T=128, H=7168, K=8 of E=288, R=8, fp8 dispatch, cap=T,
                1% of rows scaled x100 before the bf16 cast
    throughput  T=4096, H=7168, K=8 of E=256, R=8, fp8 dispatch, cap=max count
    imbalanced  T=4096, H=7168, K=8 of E=256, R=8, bf16 dispatch, cap=max count,
                rank 0 loaded 1.5x the mean, Zipf(1.2) inside each rank, 10% masked
    `T` overrides the token count (the routing recipe stays the same).
    """
    rng = np.random.default_rng(seed)
    extra: dict = {}
    if name == "tiny":
        T = T or 64
        H, K, E, R, dtype = 2048, 4, 32, 4, BF16
        x = rng.standard_normal((T, H), dtype=np.float32)
        idx = _uniform_topk(rng, T, E, K)
        w = _softmax_rows(rng.standard_normal((T, K), dtype=np.float32))
        idx[rng.random((T, K)) < 0.05] = -1
        cap = T
    elif name in ("low4", "low8", "low16"):
        T = T or int(name[3:])
        H, K, E, R, dtype = 6144, 8, 128, 16, FP8_E4M3
        x = rng.standard_normal((T, H), dtype=np.float32)
        idx = _uniform_topk(rng, T, E, K)
        w = _softmax_rows(rng.standard_normal((T, K), dtype=np.float32))
        cap = T
    elif name == "default_ll":
        T = T or 128
        H, K, E, R, dtype = 7168, 8, 288, 8, FP8_E4M3
        x = rng.standard_normal((T, H), dtype=np.float32)
        idx = _uniform_topk(rng, T, E, K)
        w = _softmax_rows(rng.standard_normal((T, K), dtype=np.float32))
        rows = rng.choice(T, math.ceil(0.01 * T), replace=False)
        x[rows] *= 100.0
        extra["outlier_rows"] = np.sort(rows)
        cap = T
    elif name == "throughput":
        T = T or 4096
        H, K, E, R, dtype = 7168, 8, 256, 8, FP8_E4M3
        x = rng.standard_normal((T, H), dtype=np.float32)
        idx = _uniform_topk(rng, T, E, K)
        w = _softmax_rows(rng.standard_normal((T, K), dtype=np.float32))
        cap = _required_cap(idx, E)
    elif name == "imbalanced":
        T = T or 4096
        H, K, E, R, dtype = 7168, 8, 256, 8, BF16
        x = rng.standard_normal((T, H), dtype=np.float32)
        idx, ratio, a0 = _skewed_topk(rng, T, E, R, K, 1.2, 0.10, 1.5)
        w = _softmax_rows(rng.standard_normal((T, K), dtype=np.float32))
        extra["rank0_load_ratio"] = ratio
        extra["a0"] = a0
        cap = _required_cap(idx, E)
    else:
        raise ValueError(f"unknown workload {name!r}; expected one of {CONFIG_NAMES}")
    return Case(name=name, T=T, H=H, K=K, E=E, R=R, cap=cap, dtype=dtype,
                x=f32_to_bf16_bits(x), topk_idx=np.ascontiguousarray(idx, dtype=np.int32),
                topk_weights=np.ascontiguousarray(w, dtype=np.float32), seed=seed, extra=extra)


def make_random_case(seed: int, T: int, H: int, K: int, E: int, R: int, cap: int | None,
                     dtype: int, mask_p: float = 0.0, distinct: bool = True,
                     scale: float = 1.0) -> Case:
    """A free-form uniform workload for edge and fuzz cases.

    distinct=False draws every entry independently, so one token may pick the
    same expert more than once.  cap=None sizes the buffers to the largest
    expert count.
    """
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H), dtype=np.float32) * np.float32(scale)
    if distinct:
        idx = _uniform_topk(rng, T, E, K) if T > 0 else np.zeros((0, K), np.int32)
    else:
        idx = rng.integers(0, E, size=(T, K), dtype=np.int32)
    w = _softmax_rows(rng.standard_normal((T, K), dtype=np.float32)) if T > 0 else \
        np.zeros((0, K), np.float32)
    if mask_p > 0:
        idx[rng.random((T, K)) < mask_p] = -1
    if cap is None:
        cap = max(1, _required_cap(idx, E))
    return Case(name=f"random{seed}", T=T, H=H, K=K, E=E, R=R, cap=cap, dtype=dtype,
                x=f32_to_bf16_bits(x), topk_idx=np.ascontiguousarray(idx, dtype=np.int32),
                topk_weights=np.ascontiguousarray(w, dtype=np.float32), seed=seed)


def make_expert_out(case: Case, seed: int, rows: str = "valid") -> np.ndarray:
    """Stand-in expert outputs, bf16 bits [E, cap, H].

    rows="valid" fills only rows s < (number of entries routed to e), leaving
    the rest zero (combine never reads them); rows="all" fills every row.
    The values are bf16(N(0, 1)).
    """
    rng = np.random.default_rng(seed + 1_000_003)
    E, cap, H = case.E, case.cap, case.H
    out = np.zeros((E, cap, H), dtype=np.uint16)
    if rows == "all":
        out[:] = f32_to_bf16_bits(rng.standard_normal((E, cap, H), dtype=np.float32))
        return out
    v = case.topk_idx[(case.topk_idx >= 0) & (case.topk_idx < E)]
    fill = np.minimum(np.bincount(v, minlength=E), cap) if v.size else np.zeros(E, np.int64)
    for e in range(E):
        n = int(fill[e])
        if n:
            out[e, :n] = f32_to_bf16_bits(rng.standard_normal((n, H), dtype=np.float32))
    return out
