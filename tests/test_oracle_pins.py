"""Pins for the float64 oracle: facts fixed by the sources and by mathematics, not by the oracle itself.

Each test checks the oracle against something other than its own code:
  * the worked tie example printed on the SGLang PR #36630 summary page;
  * closed forms (uniform rows, k = 1, min_p = 1, top_p = 0);
  * invariants that must hold for any input (token in S, logprobs sum to 1, ties at a cut all kept,
    selected logprob equals the support entry);
  * cuRAND's host Philox4x32-10 generator, a library routine independent of the oracle's Philox.
"""
import ctypes
import ctypes.util
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import philox4x32_10, sample_row, sample_filter_capture
from top_support_capture_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ln_f32(vals):
    return np.log(np.asarray(vals, np.float64)).astype(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------------------------
# The worked example (SGLang PR #36630 summary, 关键源码片段: the joint-cutoff tie test)
# ---------------------------------------------------------------------------------------------

def test_worked_example_ties_kept():
    g = json.load(open(os.path.join(GOLDEN, "worked_example_ties.json")))
    l = _ln_f32(g["probs"])
    assert l[1] == l[2]  # the two 0.2 tokens are bitwise tied after rounding to f32
    for row in range(g["batch_size"]):
        res = sample_row(l, 1.0, g["top_k"], g["top_p"], 0.0, seed=1234, step=0, row=row)
        assert res.status == oracle.ROW_OK
        assert sorted(res.support.tolist()) == g["expected_support"]
        assert len(res.support) > g["top_k"]
        assert res.token in g["expected_support"]
        # closed form: logprobs over S = ln(0.5), ln(0.25), ln(0.25) up to the f32 rounding of ln p
        lp = dict(zip(res.support.tolist(), res.support_logprobs.tolist()))
        assert abs(lp[0] - math.log(0.5)) < 1e-6
        assert abs(lp[1] - math.log(0.25)) < 1e-6
        assert abs(lp[2] - math.log(0.25)) < 1e-6
    # canonical order: logit descending, id ascending
    assert res.support.tolist() == [0, 1, 2]


def test_worked_example_every_token_drawn():
    """Over the 256 rows (independent noise per row) every member of S is drawn at least once."""
    g = json.load(open(os.path.join(GOLDEN, "worked_example_ties.json")))
    l = _ln_f32(g["probs"])
    B = g["batch_size"]
    L = np.tile(l.astype(np.float32), (B, 1))
    out = sample_filter_capture(L, oracle.DT_F32, np.ones(B), np.full(B, g["top_k"]), np.full(B, g["top_p"]),
                                np.zeros(B), seed=7, step=3, capture_rows=np.ones(B, np.uint8), packed_width=5)
    assert set(out.tokens.tolist()) == set(g["expected_support"])
    assert (out.lengths == 3).all()


# ---------------------------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("k", [0, 1, 3, 8, 100])
def test_uniform_row_keeps_everything_tied(k):
    """All logits equal: every token is tied at any cut, so S = F and each logprob is -ln V."""
    V = 8
    l = np.full(V, 0.75)
    res = sample_row(l, 1.0, k, 0.5, 0.0, seed=1, step=0, row=0)
    # top_p = 0.5: the mass strictly above the single group is 0 <= 0.5, so the group stays.
    assert res.support.tolist() == list(range(V))
    np.testing.assert_allclose(res.support_logprobs, -math.log(V), atol=1e-15)


def test_k1_unique_max():
    rng = np.random.default_rng(0)
    l = rng.standard_normal(50)
    res = sample_row(l, 0.7, 1, 1.0, 0.0, seed=1, step=0, row=0)
    assert res.support.tolist() == [int(np.argmax(l))]
    assert res.token == int(np.argmax(l))
    assert res.support_logprobs[0] == 0.0


def test_k1_tied_max_keeps_the_group():
    l = np.array([0.0, 2.0, -1.0, 2.0, 2.0])
    res = sample_row(l, 1.0, 1, 1.0, 0.0, seed=1, step=0, row=0)
    assert res.support.tolist() == [1, 3, 4]


def test_min_p_one_keeps_max_group():
    l = np.array([1.0, 3.0, 3.0, 2.999, -5.0])
    res = sample_row(l, 1.3, 0, 1.0, 1.0, seed=1, step=0, row=0)
    assert res.support.tolist() == [1, 2]


def test_top_p_zero_keeps_max_group():
    l = np.array([1.0, 3.0, 0.5, 3.0, 2.9])
    res = sample_row(l, 1.0, 0, 0.0, 0.0, seed=1, step=0, row=0)
    assert res.support.tolist() == [1, 3]


def test_min_p_closed_form():
    """min_p keeps p_i >= min_p * p_max, i.e. z_i - z_max >= ln(min_p)."""
    T = 2.0
    l = np.array([0.0, -1.0, -2.0, -3.0, -4.0, -5.0])
    min_p = 0.2  # ln 0.2 = -1.609: with T=2, keep (l - 0)/2 >= -1.609 -> l >= -3.2189
    res = sample_row(l, T, 0, 1.0, min_p, seed=1, step=0, row=0)
    assert res.support.tolist() == [0, 1, 2, 3]


def test_top_p_closed_form():
    """Geometric row p ∝ 2^-i: the mass above token i is 1 - 2^-i (normalised); keep while <= top_p."""
    V = 10
    l = -np.arange(V) * math.log(2.0)
    p = 2.0 ** -np.arange(V)
    p /= p.sum()
    above = np.concatenate([[0.0], np.cumsum(p)[:-1]])
    for top_p in [0.3, 0.5, 0.7, 0.9, 0.99]:
        res = sample_row(l, 1.0, 0, top_p, 0.0, seed=1, step=0, row=0)
        assert res.support.tolist() == [i for i in range(V) if above[i] <= top_p]


@pytest.mark.parametrize("T", [0.5, 2.0])
def test_top_p_closed_form_with_temperature(T):
    """Geometric logits l_i = -i ln 2 at temperature T: p_i ∝ 2^(-i/T); keep while the mass above is <= top_p."""
    V = 12
    l = -np.arange(V) * math.log(2.0)
    p = 2.0 ** (-np.arange(V) / T)
    p /= p.sum()
    above = np.concatenate([[0.0], np.cumsum(p)[:-1]])
    for top_p in [0.4, 0.8, 0.95]:
        res = sample_row(l, T, 0, top_p, 0.0, seed=1, step=0, row=0)
        assert res.support.tolist() == [i for i in range(V) if above[i] <= top_p]


def test_identical_rows_share_support_not_noise():
    rng = np.random.default_rng(5)
    row = rng.standard_normal(200).astype(np.float32)
    B = 64
    L = np.tile(row, (B, 1))
    out = sample_filter_capture(L, oracle.DT_F32, np.ones(B), np.full(B, 40), np.full(B, 0.9), np.zeros(B),
                                seed=11, step=0, capture_rows=np.ones(B, np.uint8), packed_width=64)
    assert (out.support_ids == out.support_ids[0]).all()
    assert len(set(out.tokens.tolist())) > 1


def test_neg_inf_never_in_support():
    l = np.array([-np.inf, 1.0, -np.inf, 0.5, 0.25])
    res = sample_row(l, 1.0, 0, 1.0, 0.0, seed=1, step=0, row=0)
    assert res.support.tolist() == [1, 3, 4]
    res = sample_row(l, 1.0, 4, 1.0, 0.0, seed=1, step=0, row=0)  # k >= |F|: K = F
    assert res.support.tolist() == [1, 3, 4]


@pytest.mark.parametrize("bad", [
    dict(T=0.0), dict(T=-1.0), dict(T=float("nan")), dict(T=float("inf")),
    dict(top_p=-0.1), dict(top_p=float("nan")),
    dict(min_p=-0.01), dict(min_p=1.5), dict(min_p=float("nan")),
])
def test_bad_parameters(bad):
    l = np.array([0.0, 1.0, 2.0])
    kw = dict(T=1.0, top_p=0.9, min_p=0.0)
    kw.update(bad)
    res = sample_row(l, kw["T"], 2, kw["top_p"], kw["min_p"], seed=1, step=0, row=0)
    assert res.status == oracle.ROW_BADPARAM and res.token == -1


@pytest.mark.parametrize("vals", [[0.0, float("nan"), 1.0], [0.0, float("inf"), 1.0], [-np.inf, -np.inf]])
def test_bad_logits(vals):
    res = sample_row(np.array(vals), 1.0, 1, 1.0, 0.0, seed=1, step=0, row=0)
    assert res.status == oracle.ROW_BADPARAM


def test_top_p_above_one_disables():
    l = np.array([0.0, 1.0, 2.0])
    res = sample_row(l, 1.0, 0, 1.7, 0.0, seed=1, step=0, row=0)
    assert res.support.tolist() == [2, 1, 0]


# ---------------------------------------------------------------------------------------------
# Invariants on the synthetic workloads
# ---------------------------------------------------------------------------------------------

def _check_invariants(w, out, rows):
    L = w.logits_f32().astype(np.float64)
    for r in rows:
        assert out.row_status[r] in (oracle.ROW_OK, oracle.ROW_OVERFLOW)
        nS = int(out.support_size[r])
        res = sample_row(L[r], w.temperature[r], int(w.top_k[r]), w.top_p[r], w.min_p[r], w.seed, w.step, r)
        S = res.support
        assert res.token in set(S.tolist())
        assert abs(np.exp(res.support_logprobs).sum() - 1.0) < 1e-9
        # every token whose logit equals the smallest kept logit is kept (threshold ties)
        tau = L[r, S].min()
        assert set(np.flatnonzero(L[r] >= tau).tolist()) == set(S.tolist())
        k = int(w.top_k[r])
        F = int(np.isfinite(L[r]).sum())
        if float(w.top_p[r]) >= 1.0 and float(w.min_p[r]) == 0.0:
            assert nS >= min(k if 1 <= k < w.V else w.V, F)
        if 1 <= k < F:
            assert nS <= np.sum(L[r] >= np.sort(L[r])[::-1][k - 1])
        if w.capture[r]:
            pos = int(np.flatnonzero(S == res.token)[0])
            assert out.selected_logprob[r] == res.support_logprobs[pos]
            n_out = min(nS, w.packed_width)
            assert out.support_ids[r, :n_out].tolist() == S[:n_out].tolist()
            assert out.lengths[r] == nS
            assert out.row_status[r] == (oracle.ROW_OVERFLOW if nS > w.packed_width else oracle.ROW_OK)
        else:
            assert out.lengths[r] == 0 and (out.support_ids[r] == -1).all()


def test_invariants_config1():
    w = wl.config1()
    out = sample_filter_capture(w.logits, w.dtype, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, w.step,
                                w.capture, w.packed_width)
    _check_invariants(w, out, range(w.B))
    assert (out.lengths >= 20).all()


@pytest.mark.parametrize("V", [5, 8, 16])
def test_invariants_tiny(V):
    w = wl.config1_tiny(V)
    out = sample_filter_capture(w.logits, w.dtype, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, w.step,
                                w.capture, w.packed_width)
    _check_invariants(w, out, range(w.B))


def test_invariants_config2_sampled_rows():
    w = wl.config2()
    rows = list(range(0, w.B, 8))
    out = sample_filter_capture(w.logits, w.dtype, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, w.step,
                                w.capture, w.packed_width, rows=rows)
    _check_invariants(w, out, rows)


# ---------------------------------------------------------------------------------------------
# Philox4x32-10 against cuRAND's host generator (a library routine run on the CPU)
# ---------------------------------------------------------------------------------------------

def _curand():
    for name in ("libcurand.so", "libcurand.so.10", ctypes.util.find_library("curand"),
                 "/usr/local/cuda/lib64/libcurand.so"):
        if not name:
            continue
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    return None


def _curand_block(lib, seed, offset, n=4):
    gen = ctypes.c_void_p()
    CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161
    if lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) != 0:
        pytest.skip("cuRAND host generator unavailable")
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        out = np.zeros(n, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
        return out
    finally:
        lib.curandDestroyGenerator(gen)


@pytest.mark.parametrize("seed", [0, 1, 0xDEADBEEFCAFE, 0x0123456789ABCDEF, 0xFFFFFFFFFFFFFFFF])
@pytest.mark.parametrize("block", [0, 1, 7, 0xFFFF, 0x10000, 0x3_0005, (1 << 48) + (3 << 16) + 5])
def test_philox_matches_curand_host(seed, block):
    """cuRAND's host Philox4_32_10 (default ordering) emits, for output block j, the Philox4x32-10 words at
    counter (j >> 16 as a 64-bit value split over words 0-1, j & 0xFFFF in word 2, 0) under key = seed.
    The layout was read off the generator's outputs, not its code; agreement on these counters pins the
    round function, the multipliers, the Weyl key schedule and the word order of the oracle's Philox."""
    lib = _curand()
    if lib is None:
        pytest.skip("libcurand not found")
    ref = _curand_block(lib, seed, 4 * block)
    hi = block >> 16
    mine = philox4x32_10(hi & 0xFFFFFFFF, hi >> 32, block & 0xFFFF, 0, seed & 0xFFFFFFFF, seed >> 32)
    assert [int(x) for x in mine] == [int(x) for x in ref]


def test_race_uniform_range_and_moments():
    u = oracle.race_uniform(99, 5, 3, np.arange(200000))
    assert (u > 0).all() and (u < 1).all()
    E = -np.log(u)
    assert abs(E.mean() - 1.0) < 0.01 and abs(E.var() - 1.0) < 0.02
    # exact in float32: an odd 24-bit numerator times 2^-24
    assert (u.astype(np.float32).astype(np.float64) == u).all()


# ------------------------------------------------------------------------------------------------
# The support bitmask of overflowing rows
# ------------------------------------------------------------------------------------------------

def test_support_mask_of_the_worked_example():
    """The worked tie example with W = 2 < |S| = 3: the row overflows and its mask holds {0, 1, 2}."""
    g = json.load(open(os.path.join(GOLDEN, "worked_example_ties.json")))
    l = np.log(np.asarray(g["probs"], np.float32)).astype(np.float32)[None, :]
    res = oracle.sample_filter_capture(l, oracle.DT_F32, [1.0], [g["top_k"]], [g["top_p"]], [0.0], 5, 0, [1], 2,
                                       want_mask=True)
    assert res.row_status[0] == oracle.ROW_OVERFLOW
    assert res.support_mask[0, 0] == 0b111


def test_support_mask_is_the_upper_set_of_values():
    """S is closed upwards in value (every filter keeps whole tie groups from the top): the mask is
    exactly {i : l_i >= the smallest logit in S}, its population is |S|, and it holds the packed ids."""
    w = wl.config3(B=6)
    res = oracle.sample_filter_capture(w.logits, w.dtype, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, w.step,
                                       w.capture, w.packed_width, want_mask=True)
    L = oracle.widen_logits(w.logits, w.dtype)
    V = L.shape[1]
    n_over = 0
    for r in range(w.B):
        bits = np.unpackbits(res.support_mask[r].view(np.uint8), bitorder="little")[:V].astype(bool)
        if res.row_status[r] != oracle.ROW_OVERFLOW:
            assert not bits.any()
            continue
        n_over += 1
        assert bits.sum() == res.lengths[r]
        assert bits[res.support_ids[r]].all()
        v_cut = L[r][bits].min()
        np.testing.assert_array_equal(bits, L[r] >= v_cut)
    assert n_over >= 2  # the k = 1024 rows overflow W = 1024


# ------------------------------------------------------------------------------------------------
# Greedy rows (temperature 0 under the greedy flag)
# ------------------------------------------------------------------------------------------------

def test_greedy_rows_closed_form():
    l = np.array([[0.5, 3.0, -1.0, 3.0, 2.0],      # tie at the maximum: the lower id
                  [-np.inf, -2.0, -np.inf, -3.0, -2.5],
                  [1.0, 1.0, 1.0, 1.0, 1.0]], np.float32)
    B = l.shape[0]
    res = oracle.sample_filter_capture(l, oracle.DT_F32, [0.0] * B, [2] * B, [0.5] * B, [0.0] * B, 1, 0, [1] * B, 4,
                                       greedy_t0=True)
    assert list(res.tokens) == [1, 1, 0]
    assert list(res.lengths) == [1, 1, 1] and (res.row_status == oracle.ROW_OK).all()
    assert (res.support_ids[:, 0] == res.tokens).all() and (res.support_ids[:, 1:] == -1).all()
    assert (res.selected_logprob == 0.0).all() and (res.support_logprobs[:, 0] == 0.0).all()


def test_greedy_flag_leaves_sampled_rows_and_bad_rows_alone():
    w = wl.config2()
    T = w.temperature.copy()
    T[::4] = 0.0  # every fourth row greedy
    T[1] = -1.0   # still a bad row
    a = oracle.sample_filter_capture(w.logits, w.dtype, T, w.top_k, w.top_p, w.min_p, w.seed, w.step, w.capture,
                                     w.packed_width, greedy_t0=True)
    b = oracle.sample_filter_capture(w.logits, w.dtype, T, w.top_k, w.top_p, w.min_p, w.seed, w.step, w.capture,
                                     w.packed_width)
    L = oracle.widen_logits(w.logits, w.dtype)
    for r in range(w.B):
        if T[r] == 0.0:
            assert b.row_status[r] == oracle.ROW_BADPARAM  # without the flag T = 0 is out of domain
            assert a.tokens[r] == np.flatnonzero(L[r] == L[r].max()).min()
        else:
            assert a.tokens[r] == b.tokens[r] and a.row_status[r] == b.row_status[r]
    assert a.row_status[1] == oracle.ROW_BADPARAM


# ------------------------------------------------------------------------------------------------
# Positional top-k / top-p (the PyTorch producer's truncation by position)
# ------------------------------------------------------------------------------------------------

def test_positional_worked_example():
    """The worked tie example truncated by position: K = ids {0, 1} (the first two of the canonical
    order), P keeps the positions whose own mass before is <= 0.45 (0, 0.4; not 0.6): S = {0, 1}."""
    g = json.load(open(os.path.join(GOLDEN, "worked_example_ties.json")))
    l = np.log(np.asarray(g["probs"], np.float32)).astype(np.float32)
    for k, tp in ((g["top_k"], 1.0), (0, g["top_p"]), (g["top_k"], g["top_p"])):
        res = sample_row(l.astype(np.float64), 1.0, k, tp, 0.0, 5, 0, 0, positional=True)
        assert list(res.support) == [0, 1], (k, tp)
        np.testing.assert_allclose(res.support_logprobs, [math.log(0.4 / 0.6), math.log(0.2 / 0.6)], atol=1e-6)


def test_positional_uniform_closed_forms():
    n = 40
    l = np.zeros(n)
    for k in (1, 7, 39):
        res = sample_row(l, 1.0, k, 1.0, 0.0, 1, 0, 0, positional=True)
        assert list(res.support) == list(range(k))
    for tp in (0.0, 0.13, 0.51, 0.77):  # away from the knife edges i / n = tp
        res = sample_row(l, 1.0, 0, tp, 0.0, 1, 0, 0, positional=True)
        assert res.support.size == int(np.floor(tp * n + 1e-9)) + 1  # positions i with i / n <= tp


def test_positional_is_the_joint_support_truncated():
    """Positional S is a prefix of the joint S (joint keeps whole tie groups); on tie-free rows the two agree."""
    rng = np.random.default_rng(12)
    for trial in range(30):
        V = int(rng.integers(5, 400))
        grid = rng.integers(0, 2) == 0
        l = (np.round(rng.standard_normal(V) * 4) / 4) if grid else rng.standard_normal(V) * 2
        k = int(rng.integers(0, V + 1))
        tp = float(rng.choice([0.3, 0.7, 0.95, 1.0]))
        mp = float(rng.choice([0.0, 0.05]))
        a = sample_row(l, 1.0, k, tp, mp, 3, 0, trial, positional=True)
        b = sample_row(l, 1.0, k, tp, mp, 3, 0, trial)
        assert a.support.size <= b.support.size
        assert list(a.support) == list(b.support[:a.support.size])
        if np.unique(l).size == V:
            assert list(a.support) == list(b.support)


# ------------------------------------------------------------------------------------------------
# Min-p-first order (the vLLM sampler's: min-p writes -inf, then top-k/top-p on what is left)
# ------------------------------------------------------------------------------------------------

def test_min_p_first_geometric_closed_form():
    """p_i ∝ 2^-i (V = 10), min_p = 0.05 keeps M = {0..4}; renormalised over M the mass strictly above i
    is (2 - 2^(1-i)) * 16/31, so top_p = 0.9 keeps {0, 1, 2} where the joint rule (full-vocabulary
    masses, (2 - 2^(1-i)) / (2 - 2^-9)) keeps {0, 1, 2, 3}."""
    V = 10
    lg = -np.arange(V) * math.log(2.0)
    for tp, want in ((0.5, [0]), (0.9, [0, 1, 2]), (0.95, [0, 1, 2, 3]), (1.0, [0, 1, 2, 3, 4])):
        res = sample_row(lg, 1.0, 0, tp, 0.05, 1, 0, 0, min_p_first=True)
        assert list(res.support) == want, tp
        assert list(res.support) == [i for i in range(5) if (2 - 2.0 ** (1 - i)) * 16 / 31 <= tp]
    assert list(sample_row(lg, 1.0, 0, 0.9, 0.05, 1, 0, 0).support) == [0, 1, 2, 3]


def test_min_p_first_is_the_masked_row_filtered():
    """The page's procedure written out: set every token that min-p drops to -inf, then run the joint
    top-k/top-p filter (no min-p) on what is left. Same support, token and logprobs on random rows."""
    rng = np.random.default_rng(31)
    checked = 0
    for trial in range(60):
        V = int(rng.integers(5, 300))
        l = np.round(rng.standard_normal(V) * 3, 1) if trial % 2 else rng.standard_normal(V) * 2
        T = float(rng.choice([0.7, 1.0, 1.6]))
        k = int(rng.integers(0, V + 1))
        tp = float(rng.choice([0.5, 0.8, 0.95]))
        mp = float(rng.choice([0.02, 0.1, 0.3]))
        a = sample_row(l, T, k, tp, mp, 4, 0, trial, min_p_first=True)
        if a.margin_top_p < 1e-9 or a.margin_min_p < 1e-9:
            continue
        z = l / T
        lm = np.where(z - z.max() >= math.log(mp), l, -np.inf)
        b = sample_row(lm, T, k, tp, 0.0, 4, 0, trial)
        assert list(a.support) == list(b.support), trial
        assert a.token == b.token
        np.testing.assert_allclose(a.support_logprobs, b.support_logprobs, atol=1e-12)
        j = sample_row(l, T, k, tp, mp, 4, 0, trial)
        assert set(a.support) <= set(j.support)
        checked += 1
    assert checked >= 45


def test_min_p_first_brute_force_tiny():
    """Pairwise restatement: i is kept iff it passes min-p, fewer than k logits are larger, and the M-mass
    strictly above it is <= top_p times M's total mass."""
    rng = np.random.default_rng(8)
    grid = np.arange(-2.0, 2.01, 0.5)
    for trial in range(200):
        V = int(rng.integers(2, 12))
        l = [float(x) for x in rng.choice(grid, V)]
        k = int(rng.integers(0, V + 1))
        tp = float(rng.choice([0.3, 0.6, 0.9, 1.0]))
        mp = float(rng.choice([0.0, 0.1, 0.4]))
        res = sample_row(np.array(l), 1.0, k, tp, mp, 1, 0, trial, min_p_first=True)
        if res.margin_top_p < 1e-9 or res.margin_min_p < 1e-9:
            continue
        zmax = max(l)
        w = [math.exp(x - zmax) for x in l]
        M = [i for i in range(V) if mp <= 0.0 or l[i] - zmax >= math.log(mp)]
        ZM = math.fsum(w[i] for i in M)
        want = set()
        for i in M:
            bigger = [j for j in range(V) if l[j] > l[i]]
            inK = not (1 <= k < V) or len(bigger) < k
            inP = tp >= 1.0 or math.fsum(w[j] for j in bigger if j in M) <= tp * ZM
            if inK and inP:
                want.add(i)
        assert set(res.support.tolist()) == want, (trial, l, k, tp, mp)
