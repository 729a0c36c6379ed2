"""Pins for the parts of the oracle that every parity claim rests on but the method's own examples do not
reach: the exact widening of bf16 logits, and the three decision margins that decide which rows the
bit-exact comparison accepts (a row whose top-p mass, min-p value or race score sits within rounding
distance of its threshold is regenerated instead).

  * bf16 -> float64: hand-decoded codes (sign, exponent, mantissa of the IEEE-style 1-8-7 layout) and
    torch's own bfloat16 type on all 65,536 codes;
  * top-p margin: closed forms on geometric rows, min over the tie groups of K ∩ M (not the maximum
    group) of |mass strictly above the group - top_p|;
  * min-p margin: planted gaps, min over the members of K ∩ P (not the maximum group) of
    |z - z_max - ln(min_p)|;
  * race margin: the gap between the two best race scores z - z_max - ln(-ln u), with u taken from
    cuRAND's host Philox4x32-10 generator rather than the oracle's.
Each pin is chosen so that a plausible mistake (the tie-group mask dropped, K or P ignored, the margin
taken on z instead of the race score, a wrong bf16 shift) fails it; the planted mistakes below check that.
"""
import ctypes
import ctypes.util
import math
import sys
import types
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import sample_row, widen_logits

LN2 = math.log(2.0)


# ---------------------------------------------------------------------------------------------
# bf16 -> float64
# ---------------------------------------------------------------------------------------------

def _bf16_by_hand(code: int) -> float:
    """bfloat16 = sign(1) | exponent(8, bias 127) | mantissa(7): the float32 layout cut to 16 bits."""
    sign = -1.0 if code >> 15 else 1.0
    e = (code >> 7) & 0xFF
    f = code & 0x7F
    if e == 0xFF:
        return sign * math.inf if f == 0 else math.nan
    if e == 0:
        return sign * f * 2.0 ** (-126 - 7)  # subnormal: 0.f x 2^-126
    return sign * (1.0 + f / 128.0) * 2.0 ** (e - 127)


@pytest.mark.parametrize("code,value", [(0x3F80, 1.0), (0xC000, -2.0), (0x4049, 3.140625), (0x3DCD, 0.10009765625),
                                        (0x0001, 2.0 ** -133), (0x0080, 2.0 ** -126), (0x7F7F, 3.3895313892515355e38),
                                        (0x8000, -0.0), (0x7F80, math.inf), (0xFF80, -math.inf)])
def test_bf16_codes_decoded_by_hand(code, value):
    got = widen_logits(np.array([code], np.uint16), oracle.DT_BF16)[0]
    assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value)
    assert _bf16_by_hand(code) == value


def test_bf16_nan_codes():
    got = widen_logits(np.array([0x7FC0, 0xFFC1, 0x7F81], np.uint16), oracle.DT_BF16)
    assert np.isnan(got).all()


def test_bf16_all_codes_match_torch_and_the_layout():
    torch = pytest.importorskip("torch")
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = widen_logits(codes, oracle.DT_BF16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))  # -0.0 stays -0.0
    hand = np.array([_bf16_by_hand(int(c)) for c in range(0, 65536, 97)])
    sub = got[::97]
    assert np.array_equal(np.isnan(hand), np.isnan(sub))
    assert np.array_equal(hand[~np.isnan(hand)], sub[~np.isnan(sub)])


def test_f32_widening_is_exact():
    x = np.array([1.1, -3.3e-39, 7e37, -0.0], np.float32)
    got = widen_logits(x, oracle.DT_F32)
    assert [Fraction(float(a)) for a in got] == [Fraction(float(a)) for a in x.astype(np.float64)]


# ---------------------------------------------------------------------------------------------
# The top-p margin
# ---------------------------------------------------------------------------------------------

def _geometric_above(n_groups, size, V_groups=None):
    """Mass strictly above group j of a row whose group j holds `size` tokens of weight 2^-j: exact."""
    G = n_groups if V_groups is None else V_groups
    total = size * sum(Fraction(1, 2 ** i) for i in range(G))
    return [size * sum(Fraction(1, 2 ** i) for i in range(j)) / total for j in range(G)]


def test_top_p_margin_geometric_row():
    """p_i ∝ 2^-i, no ties: the margin is min over i >= 1 of |(1 - 2^-i)/(1 - 2^-V) - top_p|."""
    V = 12
    l = -np.arange(V) * LN2
    above = _geometric_above(V, 1)
    for tp in (0.3, 0.7, 0.97):
        want = min(abs(float(above[i]) - tp) for i in range(1, V))
        got = sample_row(l, 1.0, 0, tp, 0.0, seed=1, step=0, row=0).margin_top_p
        assert abs(got - want) < 1e-12, (tp, got, want)


def test_top_p_margin_counts_tie_groups_not_positions():
    """Each value twice: only a group's first member decides. top_p sits 1e-4 above the mass before the
    second member of group 2, so a margin over positions would be 1e-4; over groups it is much larger."""
    G = 6
    l = np.repeat(-np.arange(G) * LN2, 2)
    above = _geometric_above(G, 2)
    p2 = Fraction(1, 2 ** 2) / (2 * sum(Fraction(1, 2 ** i) for i in range(G)))  # one member of group 2
    tp = float(above[2] + p2) + 1e-4
    want = min(abs(float(above[j]) - tp) for j in range(1, G))
    got = sample_row(l, 1.0, 0, tp, 0.0, seed=1, step=0, row=0).margin_top_p
    assert abs(got - want) < 1e-12
    assert got > 0.01


def test_top_p_margin_only_inside_k_and_m():
    """Groups outside K (top_k = 3) or M (min_p keeps z - z_max >= -3.5 ln 2, i.e. i <= 3) never decide:
    top_p is put 1e-4 from the mass above token 5."""
    V = 12
    l = -np.arange(V) * LN2
    above = _geometric_above(V, 1)
    tp = float(above[5]) + 1e-4
    got_k = sample_row(l, 1.0, 3, tp, 0.0, seed=1, step=0, row=0).margin_top_p
    assert abs(got_k - min(abs(float(above[i]) - tp) for i in (1, 2))) < 1e-12
    got_m = sample_row(l, 1.0, 0, tp, 2.0 ** -3.5, seed=1, step=0, row=0).margin_top_p
    assert abs(got_m - min(abs(float(above[i]) - tp) for i in (1, 2, 3))) < 1e-12
    got_all = sample_row(l, 1.0, 0, tp, 0.0, seed=1, step=0, row=0).margin_top_p
    assert abs(got_all - 1e-4) < 1e-12


def test_top_p_margin_is_infinite_when_top_p_is_off():
    l = -np.arange(8) * LN2
    assert sample_row(l, 1.0, 0, 1.0, 0.0, seed=1, step=0, row=0).margin_top_p == math.inf


# ---------------------------------------------------------------------------------------------
# The min-p margin
# ---------------------------------------------------------------------------------------------

def test_min_p_margin_planted_gaps():
    """z - z_max = 0, -1, -2.5, -4, -6 against ln(min_p) = -2.4: the closest member is 0.1 away."""
    l = np.array([0.0, -1.0, -2.5, -4.0, -6.0])
    mp = math.exp(-2.4)
    assert abs(sample_row(l, 1.0, 0, 1.0, mp, seed=1, step=0, row=0).margin_min_p - 0.1) < 1e-12
    # top_k = 2: only token 1 (z - z_max = -1) is in K besides the maximum
    assert abs(sample_row(l, 1.0, 2, 1.0, mp, seed=1, step=0, row=0).margin_min_p - 1.4) < 1e-12
    # T = 2 halves every z: 0, -0.5, -1.25, -2, -3 -> 0.4 (at -2)
    assert abs(sample_row(l, 2.0, 0, 1.0, mp, seed=1, step=0, row=0).margin_min_p - 0.4) < 1e-12
    # top_p = 0.9: P = {0, 1} (mass above token 2 is 0.93), so only token 1 decides
    assert abs(sample_row(l, 1.0, 0, 0.9, mp, seed=1, step=0, row=0).margin_min_p - 1.4) < 1e-12
    # min-p before top-p: every min-p decision moves top-p's renormaliser, so all members count
    got = sample_row(l, 1.0, 2, 0.9, mp, seed=1, step=0, row=0, min_p_first=True).margin_min_p
    assert abs(got - 0.1) < 1e-12
    assert sample_row(l, 1.0, 0, 1.0, 0.0, seed=1, step=0, row=0).margin_min_p == math.inf


# ---------------------------------------------------------------------------------------------
# The race margin, with u from cuRAND's host Philox4x32-10
# ---------------------------------------------------------------------------------------------

def _curand_word0(seed, step, row, token):
    """Word 0 of Philox4x32-10 at counter (token, row, step, 0) under key = seed, from cuRAND's host
    generator: its output block j is the counter (j >> 16 over words 0-1, j & 0xFFFF in word 2, 0), so
    block j = ((row << 32 | token) << 16) | step (step < 2^16, row < 2^14)."""
    lib = None
    for name in ("libcurand.so", "libcurand.so.10", ctypes.util.find_library("curand"),
                 "/usr/local/cuda/lib64/libcurand.so"):
        if name:
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                pass
    if lib is None:
        pytest.skip("libcurand not found")
    gen = ctypes.c_void_p()
    if lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) != 0:  # CURAND_RNG_PSEUDO_PHILOX4_32_10
        pytest.skip("cuRAND host generator unavailable")
    try:
        block = (((row << 32) | token) << 16) | step
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(4 * block)) == 0
        out = np.zeros(4, np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(4)) == 0
        return int(out[0])
    finally:
        lib.curandDestroyGenerator(gen)


@pytest.mark.parametrize("T", [1.0, 0.5])
def test_race_margin_from_curand_words(T):
    seed, step, row = 0xABCDEF1234, 7, 5
    l = np.array([0.0, -0.3, -0.45, -2.0])
    res = sample_row(l, T, 0, 1.0, 0.0, seed=seed, step=step, row=row)
    assert res.support.tolist() == [0, 1, 2, 3]
    scores = []
    for i, li in enumerate(l):
        u = (2 * (_curand_word0(seed, step, row, i) >> 9) + 1) * 2.0 ** -24
        scores.append((li - l.max()) / T - math.log(-math.log(u)))
    best, second = sorted(scores)[-1], sorted(scores)[-2]
    assert res.token == int(np.argmax(scores))
    assert abs(res.margin_race - (best - second)) < 1e-12
    # one member: no race, no margin
    assert sample_row(l, T, 1, 1.0, 0.0, seed=seed, step=step, row=row).margin_race == math.inf


# ---------------------------------------------------------------------------------------------
# Planted mistakes that the pins above must catch
# ---------------------------------------------------------------------------------------------

MUTANTS = {
    # each position's own mass before it instead of its tie group's mass above
    "margin_over_positions": [("sel = in_K & in_M & not_top & new_group\n        m_tp = float(np.abs(mass_above[sel]",
                               "sel = in_K & in_M & not_top\n        m_tp = float(np.abs(mass_before[sel]")],
    "margin_ignores_K": [("sel = in_K & in_M & not_top & new_group", "sel = in_M & not_top & new_group")],
    "margin_min_p_ignores_K_and_P": [("else (in_K & in_P & not_top)", "else not_top")],
    "margin_race_on_z": [("top2 = np.partition(score, n_S - 2)[n_S - 2:]",
                          "top2 = np.partition(zs[:n_S], n_S - 2)[n_S - 2:]")],
    "margin_min_p_in_logit_units": [("m_mp = float(np.abs(zs[sel] - np.log(mp)).min())",
                                     "m_mp = float(np.abs(zs[sel] * T - np.log(mp)).min())")],
    "bf16_wrong_shift": [("(bits.astype(np.uint32) << 16)", "(bits.astype(np.uint32) << 15)")],
    "bf16_low_half": [("(bits.astype(np.uint32) << 16)", "(bits.astype(np.uint32))")],
}


def _build(name):
    import os

    src = open(os.path.join(os.path.dirname(oracle.__file__), "sfc_oracle.py")).read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    mod = types.ModuleType(f"oracle._margin_mutant_{name}")
    mod.__package__ = "oracle"
    sys.modules[mod.__name__] = mod
    exec(compile(src, f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


def _battery(m) -> bool:
    """The pins of this file, run against a given oracle module."""
    global sample_row, widen_logits
    saved = sample_row, widen_logits
    sample_row, widen_logits = m.sample_row, m.widen_logits
    try:
        for code, value in ((0x3F80, 1.0), (0xC000, -2.0), (0x0001, 2.0 ** -133)):
            test_bf16_codes_decoded_by_hand(code, value)
        test_top_p_margin_geometric_row()
        test_top_p_margin_counts_tie_groups_not_positions()
        test_top_p_margin_only_inside_k_and_m()
        test_min_p_margin_planted_gaps()
        for T in (1.0, 0.5):
            test_race_margin_from_curand_words(T)
        return True
    except AssertionError:
        return False
    finally:
        sample_row, widen_logits = saved


def test_real_oracle_passes_the_margin_battery():
    assert _battery(oracle.sfc_oracle)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_margin_mutant_is_caught(name):
    assert not _battery(_build(name)), f"planted mistake '{name}' slipped through the margin pins"
