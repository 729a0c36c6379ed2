"""Brute-force pins for the oracle on tiny rows (V <= 16), in plain Python, sharing no code with it.

Two restatements of the joint-threshold support, neither of which sorts:
  (i)  pairwise predicates: i in K iff fewer than k logits are strictly larger; i in P iff the
       probability mass strictly above l_i is <= top_p; i in M iff z_i - z_max >= ln(min_p);
  (ii) threshold scan: S is the largest upper set {l >= v} (v ranging over the row's values) whose
       cut value v passes all three tests.
Plus the exponential race's distribution: over many independent steps the token frequencies must match
p_i / sum_S p (a chi-square test), which pins the race's sign and form.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import sample_row
from top_support_capture_gb300 import workloads as wl


def _softmax_py(l, T):
    F = [i for i, x in enumerate(l) if x != -math.inf]
    zmax = max(l[i] / T for i in F)
    w = {i: math.exp(l[i] / T - zmax) for i in F}
    tot = math.fsum(w.values())
    return {i: w[i] / tot for i in F}, zmax, F


def support_pairwise(l, T, k, top_p, min_p):
    p, zmax, F = _softmax_py(l, T)
    out = []
    for i in F:
        bigger = [j for j in F if l[j] > l[i]]
        inK = not (1 <= k < len(F)) or len(bigger) < k
        inP = top_p >= 1.0 or math.fsum(p[j] for j in bigger) <= top_p
        inM = min_p <= 0.0 or (l[i] / T - zmax) >= math.log(min_p)
        if inK and inP and inM:
            out.append(i)
    return set(out)


def support_threshold_scan(l, T, k, top_p, min_p):
    p, zmax, F = _softmax_py(l, T)
    best = None
    for v in sorted(set(l[i] for i in F)):
        above = [j for j in F if l[j] > v]
        ok_k = not (1 <= k < len(F)) or len(above) < k
        ok_p = top_p >= 1.0 or math.fsum(p[j] for j in above) <= top_p
        ok_m = min_p <= 0.0 or (v / T - zmax) >= math.log(min_p)
        if ok_k and ok_p and ok_m:
            best = v
            break  # values ascend: the first passing v gives the largest upper set
    return set(j for j in F if l[j] >= best)


def _margin_ok(res):
    return res.margin_top_p > 1e-9 and res.margin_min_p > 1e-9


@pytest.mark.parametrize("V", [5, 8, 16])
def test_tiny_rows_match_brute_force(V):
    w = wl.config1_tiny(V)
    L = w.logits_f32().astype(np.float64)
    checked = 0
    for r in range(w.B):
        args = (float(w.temperature[r]), int(w.top_k[r]), float(w.top_p[r]), float(w.min_p[r]))
        res = sample_row(L[r], *args[:1], args[1], args[2], args[3], seed=w.seed, step=w.step, row=r)
        if not _margin_ok(res):
            continue
        l = [float(x) for x in L[r]]
        S = set(res.support.tolist())
        assert S == support_pairwise(l, *args), r
        assert S == support_threshold_scan(l, *args), r
        checked += 1
    assert checked >= w.B * 3 // 4


def test_random_tiny_rows_match_brute_force():
    rng = np.random.default_rng(123)
    grid = np.arange(-2.0, 2.01, 0.5)
    checked = 0
    for t in range(600):
        V = int(rng.integers(1, 13))
        l = rng.choice(grid, size=V)
        if rng.random() < 0.2 and V > 1:
            l[rng.integers(0, V)] = -np.inf
        if not np.isfinite(l).any():
            continue
        T = float(rng.choice([0.5, 1.0, 1.7]))
        k = int(rng.integers(-1, V + 2))
        top_p = float(rng.choice([0.0, 0.1, 0.3, 0.45, 0.6, 0.9, 1.0]))
        min_p = float(rng.choice([0.0, 0.05, 0.3, 1.0]))
        res = sample_row(l, T, k, top_p, min_p, seed=5, step=t, row=0)
        if not _margin_ok(res):
            continue
        ll = [float(x) for x in l]
        assert set(res.support.tolist()) == support_pairwise(ll, T, k, top_p, min_p)
        assert set(res.support.tolist()) == support_threshold_scan(ll, T, k, top_p, min_p)
        # canonical order: logit descending, id ascending
        keys = [(-ll[i], i) for i in res.support.tolist()]
        assert keys == sorted(keys)
        checked += 1
    assert checked > 400


def test_race_distribution_matches_renormalised_support():
    """Token frequencies over 20000 decode steps follow p_i / sum_S p (chi-square, 6 dof)."""
    l = np.array([1.0, 0.8, 0.8, 0.3, -0.2, -1.0, -3.0, 0.1])
    T, k, top_p = 0.9, 7, 0.97
    res0 = sample_row(l, T, k, top_p, 0.0, seed=42, step=0, row=0)
    S = res0.support
    expect = np.exp(res0.support_logprobs)
    n = 20000
    counts = dict.fromkeys(S.tolist(), 0)
    for step in range(n):
        counts[sample_row(l, T, k, top_p, 0.0, seed=42, step=step, row=3).token] += 1
    obs = np.array([counts[i] for i in S.tolist()], dtype=np.float64)
    chi2 = float(((obs - n * expect) ** 2 / (n * expect)).sum())
    dof = len(S) - 1
    # 99.9th percentile of chi-square with <= 7 dof is below 24.4
    assert chi2 < 24.4, (chi2, dof, obs, n * expect)
