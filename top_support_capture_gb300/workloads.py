"""Seeded synthetic decode-step inputs for the sample · filter · capture step.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no softmax, no filtering, no sampling). Both the CUDA
path (through ``bench.py``) and the float64 oracle (through ``tests/``) take
their inputs from here, so the two sides see identical bytes.

The five workloads follow the configurations the method is benchmarked on:
a Zipf-ranked logit profile (a fixed per-row permutation assigns each token a
rank, offset = -s * ln(rank)) plus Gaussian noise that is re-drawn every
decode step. Vocabulary sizes match real tokenizers (32000, 151936, 129280,
262144). No public dataset is involved.

Every random draw is keyed on (base seed, workload id, row, step, salt[row]),
so any single row can be regenerated with a different ``salt`` without
touching the others; the parity tests use that to resample rows whose
decisions sit within rounding distance of a threshold.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

DT_BF16 = 0
DT_F32 = 1

_PARAMS_STREAM = 0x5EED_0001
_PERM_STREAM = 0x5EED_0002
_NOISE_STREAM = 0x5EED_0003


@dataclasses.dataclass
class Workload:
    """One decode step's inputs, host-resident, in the library's layouts.

    ``logits`` is ``uint16`` (bf16 bit patterns) when ``dtype == DT_BF16`` and
    ``float32`` when ``dtype == DT_F32``; shape ``[B, V]``, row-major.
    """

    name: str
    dtype: int
    logits: np.ndarray
    temperature: np.ndarray  # float32 [B]
    top_k: np.ndarray  # int32 [B]
    top_p: np.ndarray  # float32 [B]
    min_p: np.ndarray  # float32 [B]
    capture: np.ndarray  # uint8 [B]
    packed_width: int
    seed: int
    step: int

    @property
    def B(self) -> int:
        return int(self.logits.shape[0])

    @property
    def V(self) -> int:
        return int(self.logits.shape[1])

    def logits_f32(self) -> np.ndarray:
        """The logits as float32 (exact: every bf16 value is an f32 value)."""
        if self.dtype == DT_BF16:
            return bf16_bits_to_f32(self.logits)
        return self.logits

    def logits_bytes(self) -> int:
        return int(self.logits.nbytes)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even).

    Inputs are finite synthetic values; returns the 16-bit patterns.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(*words: int) -> np.random.Generator:
    return np.random.default_rng([int(w) & 0xFFFFFFFF for w in words])


def _salt(salt: Optional[Sequence[int]], B: int) -> np.ndarray:
    if salt is None:
        return np.zeros(B, dtype=np.int64)
    s = np.asarray(salt, dtype=np.int64)
    assert s.shape == (B,)
    return s


def _zipf_rows(wid: int, seed: int, B: int, V: int, slope: float, span: Optional[float],
               sigma: float, step: int, salt: np.ndarray, out_dtype: int,
               quantum: Optional[float] = None) -> np.ndarray:
    """Per row: offset[perm[j]] = -slope * ln(j + 1), plus N(0, sigma^2) noise.

    With ``span`` set, the offset is instead rescaled linearly so that it covers
    exactly ``span`` logits (the slope then cancels out). With ``quantum`` set,
    each value is rounded to a multiple of it before the final cast. Rows are
    built one at a time into the final array (bf16 bit patterns or float32).
    """
    ln_rank = np.log(np.arange(1, V + 1, dtype=np.float64))
    if span is not None:
        prof = -ln_rank * (span / ln_rank[-1])
    else:
        prof = -slope * ln_rank
    out = np.empty((B, V), dtype=np.uint16 if out_dtype == DT_BF16 else np.float32)
    row = np.empty(V, dtype=np.float64)
    for r in range(B):
        perm = _rng(seed, wid, _PERM_STREAM, r).permutation(V)
        row[perm] = prof
        row += sigma * _rng(seed, wid, _NOISE_STREAM, r, step, int(salt[r])).standard_normal(V)
        if quantum is not None:
            np.round(row / quantum, out=row)
            row *= quantum
        v32 = row.astype(np.float32)
        out[r] = f32_to_bf16_bits(v32) if out_dtype == DT_BF16 else v32
    return out


def config1(seed: int = 1, step: int = 0, salt=None) -> Workload:
    """B=4, V=1024, fp32 logits ~ N(0, 2^2); T=1, k=20, top_p=0.9, min_p=0; all rows capture."""
    B, V = 4, 1024
    s = _salt(salt, B)
    logits = np.empty((B, V), dtype=np.float32)
    for r in range(B):
        logits[r] = (2.0 * _rng(seed, 1, _NOISE_STREAM, r, step, int(s[r])).standard_normal(V)).astype(np.float32)
    return Workload("c1_B4_V1024_f32", DT_F32, logits,
                    np.ones(B, np.float32), np.full(B, 20, np.int32), np.full(B, 0.9, np.float32),
                    np.zeros(B, np.float32), np.ones(B, np.uint8), 1024, seed, step)


def config1_tiny(V: int, seed: int = 1, step: int = 0, salt=None, B: int = 64) -> Workload:
    """B=64 rows of V in {5, 8, 16} tokens drawn from the grid {-2, -1.5, ..., 2}, so ties are common.

    Per row: k uniform in [1, V], top_p in {0.3, 0.45, 0.9, 1}, min_p in {0, 0.2}; T=1; all rows capture.
    """
    s = _salt(salt, B)
    grid = np.arange(-2.0, 2.0001, 0.5, dtype=np.float32)
    logits = np.empty((B, V), dtype=np.float32)
    for r in range(B):
        logits[r] = _rng(seed, 100 + V, _NOISE_STREAM, r, step, int(s[r])).choice(grid, size=V)
    pr = _rng(seed, 100 + V, _PARAMS_STREAM)
    top_k = pr.integers(1, V + 1, size=B).astype(np.int32)
    top_p = pr.choice(np.array([0.3, 0.45, 0.9, 1.0], np.float32), size=B)
    min_p = pr.choice(np.array([0.0, 0.2], np.float32), size=B)
    return Workload(f"c1tiny_B{B}_V{V}_f32", DT_F32, logits, np.ones(B, np.float32), top_k,
                    top_p.astype(np.float32), min_p.astype(np.float32), np.ones(B, np.uint8), V, seed, step)


def config2(seed: int = 2, step: int = 0, salt=None) -> Workload:
    """B=64, V=32000, bf16 logits = N(0,1) + Zipf rank offset rescaled to a 12-logit range.

    Per row: T ~ U[0.5,1.5], top_k ~ U{1..1024}, top_p ~ U[0.5,1.0], min_p in {0, 0.05};
    half the rows (seeded Bernoulli) capture; packed_width 1024.
    """
    B, V = 64, 32000
    s = _salt(salt, B)
    l = _zipf_rows(2, seed, B, V, 1.1, 12.0, 1.0, step, s, DT_BF16)
    pr = _rng(seed, 2, _PARAMS_STREAM)
    T = pr.uniform(0.5, 1.5, size=B).astype(np.float32)
    k = pr.integers(1, 1025, size=B).astype(np.int32)
    tp = pr.uniform(0.5, 1.0, size=B).astype(np.float32)
    mp = np.where(pr.random(B) < 0.5, 0.0, 0.05).astype(np.float32)
    cap = (pr.random(B) < 0.5).astype(np.uint8)
    return Workload("c2_B64_V32000_bf16", DT_BF16, l, T, k, tp, mp, cap, 1024, seed, step)


def config3(seed: int = 3, step: int = 0, salt=None, B: int = 256) -> Workload:
    """B=256, V=151936, bf16; the config-2 profile quantised to 1/16-logit steps so ties form at every cut.

    top_k cycles {20, 50, 1024} by row; top_p=0.95; min_p=0; T=1; all rows capture; packed_width 1024.
    """
    V = 151936
    s = _salt(salt, B)
    l = _zipf_rows(3, seed, B, V, 1.1, 12.0, 1.0, step, s, DT_BF16, quantum=1.0 / 16.0)
    k = np.array([(20, 50, 1024)[r % 3] for r in range(B)], dtype=np.int32)
    return Workload(f"c3_B{B}_V151936_bf16", DT_BF16, l, np.ones(B, np.float32), k,
                    np.full(B, 0.95, np.float32), np.zeros(B, np.float32), np.ones(B, np.uint8),
                    1024, seed, step)


def config4(seed: int = 4, step: int = 0, salt=None, B: int = 256) -> Workload:
    """B=256, V=129280, fp32 logits = -ln(rank) + N(0,1); top_k=8192, top_p alternating {0.95, 1.0}.

    min_p=0; T=1; a seeded quarter of the rows (scattered) capture; packed_width 8192.
    """
    V = 129280
    s = _salt(salt, B)
    l = _zipf_rows(4, seed, B, V, 1.0, None, 1.0, step, s, DT_F32)
    tp = np.array([0.95 if r % 2 == 0 else 1.0 for r in range(B)], dtype=np.float32)
    cap = np.zeros(B, np.uint8)
    cap[_rng(seed, 4, _PARAMS_STREAM).permutation(B)[: B // 4]] = 1
    return Workload(f"c4_B{B}_V129280_f32", DT_F32, l, np.ones(B, np.float32), np.full(B, 8192, np.int32),
                    tp, np.zeros(B, np.float32), cap, 8192, seed, step)


def config5(B: int = 512, seed: int = 5, step: int = 0, salt=None) -> Workload:
    """B in {1,32,128,512}, V=262144, bf16 logits = -1.2 ln(rank) + N(0, 1.5^2).

    top_k=50, top_p=0.95, min_p=0.05, T ~ U[0.7,1.3]; all rows capture; packed_width 1024.
    """
    V = 262144
    s = _salt(salt, B)
    l = _zipf_rows(5, seed, B, V, 1.2, None, 1.5, step, s, DT_BF16)
    T = _rng(seed, 5, _PARAMS_STREAM).uniform(0.7, 1.3, size=B).astype(np.float32)
    return Workload(f"c5_B{B}_V262144_bf16", DT_BF16, l, T, np.full(B, 50, np.int32),
                    np.full(B, 0.95, np.float32), np.full(B, 0.05, np.float32), np.ones(B, np.uint8),
                    1024, seed, step)


CONFIGS = {
    1: config1,
    2: config2,
    3: config3,
    4: config4,
    5: config5,
}


def make(config: int, **kw) -> Workload:
    return CONFIGS[config](**kw)
