"""The pins must catch plausible mistakes: each mutant is the oracle's source with one planted error.

Every mutant below is a copy of ``oracle/sfc_oracle.py`` with one textual change, executed as a throwaway
module on the CPU. The pin battery (worked tie example, closed forms, brute force on tiny rows, race
distribution) must pass on the real oracle and fail on each mutant.
"""
import math
import os
import sys
import types

import numpy as np
import pytest

import oracle
from top_support_capture_gb300 import workloads as wl
from test_oracle_bruteforce import support_pairwise

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "sfc_oracle.py")).read()

MUTANTS = {
    # a positional top-k cut drops tie members at the k-th logit
    "positional_top_k": [("else (ls >= ls[k - 1])", "else (np.arange(n) < k)")],
    "kcut_off_by_one": [("else (ls >= ls[k - 1])", "else (ls >= ls[min(k, n - 1)])")],
    # a positional top-p cut breaks a tie group at the cut
    "positional_top_p": [("mass_above = mass_before[group_start]", "mass_above = mass_before")],
    "inclusive_top_p": [("mass_before = np.cumsum(ps) - ps", "mass_before = np.cumsum(ps)")],
    "strict_top_p": [("else (mass_above <= tp)", "else (mass_above < tp)")],
    # sequential semantics: top-p measured on the top-k-renormalised distribution instead of the full one
    "renormalised_top_p": [("mass_before = np.cumsum(ps) - ps",
                            "ps = np.where(in_K, ps, 0.0) / np.where(in_K, ps, 0.0).sum()\n"
                            "    mass_before = np.cumsum(ps) - ps")],
    "race_sign": [("score = zs[:n_S] - np.log(E)", "score = zs[:n_S] + np.log(E)")],
    "race_without_temperature": [("score = zs[:n_S] - np.log(E)", "score = zs[:n_S] * T - np.log(E)")],
    "first_logprob_only": [("lpS = zs[:n_S] - log_ZS", "lpS = np.full(n_S, zs[0] - log_ZS)")],
    "logprob_over_full_vocab": [("log_ZS = np.log(wS.sum())", "log_ZS = np.log(w[F].sum())")],
    "min_p_in_logit_units": [("in_M = zs >= np.log(mp)", "in_M = zs * T >= np.log(mp)")],
    "no_temperature_in_softmax": [("z[F] = l[F] / T", "z[F] = l[F]")],
    # positional mode: ties kept at the k-th position, top-p judged per tie group, inclusive mass
    "positional_mode_keeps_k_ties": [("(np.arange(n) < k) if positional", "(ls >= ls[k - 1]) if positional")],
    "positional_mode_group_top_p": [("(mass_before <= tp) if positional", "(mass_above <= tp) if positional")],
    "positional_mode_inclusive_top_p": [("(mass_before <= tp) if positional",
                                         "(mass_before + ps <= tp) if positional")],
    # min-p-first order: top-p on the full distribution, or on M's masses left unnormalised
    "min_p_first_ignored": [("if min_p_first and mp > 0.0:", "if False:")],
    "min_p_first_unnormalised": [("        ps = ps / ps.sum()\n", "")],
}


def build(name):
    src = SRC
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    mod = types.ModuleType(f"oracle._mutant_{name}")
    mod.__package__ = "oracle"
    sys.modules[mod.__name__] = mod  # dataclasses look their module up by name
    exec(compile(src, f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


def _ln_f32(vals):
    return np.log(np.asarray(vals, np.float64)).astype(np.float32).astype(np.float64)


def pins_pass(m) -> bool:
    """A compact copy of the pin battery, written against a given oracle module."""
    try:
        # worked tie example with closed-form logprobs
        l = _ln_f32([0.4, 0.2, 0.2, 0.1, 0.1])
        res = m.sample_row(l, 1.0, 2, 0.45, 0.0, seed=1, step=0, row=0)
        if res.support.tolist() != [0, 1, 2]:
            return False
        if not np.allclose(res.support_logprobs, [math.log(.5), math.log(.25), math.log(.25)], atol=1e-6):
            return False
        # geometric row, closed-form top-p
        V = 10
        lg = -np.arange(V) * math.log(2.0)
        p = 2.0 ** -np.arange(V)
        p /= p.sum()
        above = np.concatenate([[0.0], np.cumsum(p)[:-1]])
        for tp in [0.3, 0.5, 0.9]:
            if m.sample_row(lg, 1.0, 0, tp, 0.0, seed=1, step=0, row=0).support.tolist() != \
                    [i for i in range(V) if above[i] <= tp]:
                return False
        # the same row at T = 2: p_i ∝ 2^(-i/2)
        p2 = 2.0 ** (-np.arange(V) / 2.0)
        p2 /= p2.sum()
        above2 = np.concatenate([[0.0], np.cumsum(p2)[:-1]])
        for tp in [0.4, 0.8]:
            if m.sample_row(lg, 2.0, 0, tp, 0.0, seed=1, step=0, row=0).support.tolist() != \
                    [i for i in range(V) if above2[i] <= tp]:
                return False
        # top_p = 0: the mass above the maximum group is exactly 0, and 0 <= 0 keeps that group
        if m.sample_row(np.array([3.0, 1.0, 3.0]), 1.0, 0, 0.0, 0.0, seed=1, step=0, row=0).support.tolist() != [0, 2]:
            return False
        # min-p closed form with T = 2
        lm = np.array([0.0, -1.0, -2.0, -3.0, -4.0, -5.0])
        if m.sample_row(lm, 2.0, 0, 1.0, 0.2, seed=1, step=0, row=0).support.tolist() != [0, 1, 2, 3]:
            return False
        # brute force on the tiny workloads
        for V in (5, 8, 16):
            w = wl.config1_tiny(V)
            L = w.logits_f32().astype(np.float64)
            for r in range(w.B):
                a = (float(w.temperature[r]), int(w.top_k[r]), float(w.top_p[r]), float(w.min_p[r]))
                res = m.sample_row(L[r], a[0], a[1], a[2], a[3], seed=1, step=0, row=r)
                if set(res.support.tolist()) != support_pairwise([float(x) for x in L[r]], *a):
                    return False
                if abs(np.exp(res.support_logprobs).sum() - 1.0) > 1e-9:
                    return False
        # positional mode: the worked tie example keeps the first two positions; uniform closed forms
        lw = _ln_f32([0.4, 0.2, 0.2, 0.1, 0.1])
        for k, tp in ((2, 1.0), (0, 0.45)):
            if m.sample_row(lw, 1.0, k, tp, 0.0, seed=1, step=0, row=0, positional=True).support.tolist() != [0, 1]:
                return False
        for k in (1, 7):
            if m.sample_row(np.zeros(40), 1.0, k, 1.0, 0.0, seed=1, step=0, row=0,
                            positional=True).support.size != k:
                return False
        for tp in (0.13, 0.51):
            if m.sample_row(np.zeros(40), 1.0, 0, tp, 0.0, seed=1, step=0, row=0,
                            positional=True).support.size != int(np.floor(tp * 40)) + 1:
                return False
        # min-p-first order: geometric row, M = {0..4}, top-p on masses renormalised over M
        lg2 = -np.arange(10) * math.log(2.0)
        for tp, want in ((0.5, [0]), (0.9, [0, 1, 2]), (0.95, [0, 1, 2, 3])):
            if m.sample_row(lg2, 1.0, 0, tp, 0.05, seed=1, step=0, row=0,
                            min_p_first=True).support.tolist() != want:
                return False
        # race distribution (chi-square, 2000 draws at T = 0.5 so the temperature matters)
        lr = np.array([1.0, 0.6, 0.2, -0.5])
        r0 = m.sample_row(lr, 0.5, 0, 1.0, 0.0, seed=3, step=0, row=0)
        exp_p = dict(zip(r0.support.tolist(), np.exp(r0.support_logprobs).tolist()))
        n = 2000
        cnt = dict.fromkeys(exp_p, 0)
        for s in range(n):
            cnt[m.sample_row(lr, 0.5, 0, 1.0, 0.0, seed=3, step=s, row=1).token] += 1
        chi2 = sum((cnt[i] - n * q) ** 2 / (n * q) for i, q in exp_p.items())
        return chi2 < 16.3  # 99.9th percentile, 3 dof
    except (AssertionError, IndexError, ValueError, ZeroDivisionError, FloatingPointError):
        return False


def test_real_oracle_passes_the_battery():
    assert pins_pass(oracle.sfc_oracle)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    assert not pins_pass(build(name)), f"planted mistake '{name}' slipped through the pins"
