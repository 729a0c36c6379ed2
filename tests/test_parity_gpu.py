"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle, element by element.

Every configuration is compared on every row, the full-size ones in the launch configuration the
benchmark times and at several decode steps (the oracle's rows run in a process pool), plus edge cases: ragged and unaligned rows, strides, -inf / NaN / +inf
logits, bad parameters, top-k disabled (the multi-pass path), tie groups larger than the on-chip buffer,
overflowing packed widths, selected vs support mode, capture subsets and determinism.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from top_support_capture_gb300 import workloads as wl
from sfc_parity import clear_margins, compare, gpu_run, oracle_run, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_support_capture_gb300 as sfc

    sfc.load_library()


def _full_check(make, B, rows=None, **kw):
    rows = list(range(B)) if rows is None else rows
    w, ref, left = clear_margins(make, B, rows)
    assert not left, f"rows {left} kept failing the margins"
    got = gpu_run(w, **kw)
    return compare(w, ref, got, rows, support_logprobs=kw.get("support_logprobs", True))


# ------------------------------------------------------------------------------------------------
# The five workloads
# ------------------------------------------------------------------------------------------------

def test_config1_all_rows():
    assert _full_check(lambda salt: wl.config1(salt=salt), 4) == 4


@pytest.mark.parametrize("V", [5, 8, 16])
def test_config1_tiny_all_rows(V):
    assert _full_check(lambda salt: wl.config1_tiny(V, salt=salt), 64) == 64


@pytest.mark.parametrize("step", [0, 1, 37, 99])
def test_config2_all_rows(step):
    """B=64 x V=32000 bf16, the first, second, a middle and the last of the 100 decode steps."""
    assert _full_check(lambda salt: wl.config2(step=step, salt=salt), 64) == 64


@pytest.mark.parametrize("step", [0, 1, 97])
def test_config3_full_size_every_row(step):
    """B=256 x V=151936 bf16, the batch the benchmark times, in the launch configuration it times: every
    row compared at three decode steps."""
    assert _full_check(lambda salt: wl.config3(step=step, salt=salt), 256) == 256


@pytest.mark.parametrize("step", [0, 1, 97])
def test_config4_full_size_every_row(step):
    """B=256 x V=129280 f32, W = 8192, a quarter of the rows capturing: every row compared."""
    assert _full_check(lambda salt: wl.config4(step=step, salt=salt), 256) == 256


@pytest.mark.parametrize("B", [1, 32, 128])
def test_config5_sweep_batches(B):
    """V=262144 bf16 at the sweep's short batches (the library splits these rows into slices)."""
    assert _full_check(lambda salt: wl.config5(B=B, salt=salt), B) == B


@pytest.mark.parametrize("step", [0, 199])
def test_config5_full_size_every_row(step):
    """B=512 x V=262144 bf16, the first and the last of the 200 decode steps: every row compared."""
    assert _full_check(lambda salt: wl.config5(B=512, step=step, salt=salt), 512) == 512


# ------------------------------------------------------------------------------------------------
# The worked example and the modes
# ------------------------------------------------------------------------------------------------

def test_worked_tie_example_on_gpu():
    g = json.load(open(os.path.join(GOLDEN, "worked_example_ties.json")))
    B = g["batch_size"]
    l = np.log(np.asarray(g["probs"], np.float64)).astype(np.float32)
    w = wl.Workload("ties", wl.DT_F32, np.tile(l, (B, 1)), np.ones(B, np.float32), np.full(B, g["top_k"], np.int32),
                    np.full(B, g["top_p"], np.float32), np.zeros(B, np.float32), np.ones(B, np.uint8), 5, 7, 0)
    got = gpu_run(w)
    assert (got["lengths"] == 3).all()
    assert (got["support_ids"][:, :3] == np.array(g["expected_support"])).all()
    assert set(got["tokens"].tolist()) == set(g["expected_support"])
    np.testing.assert_allclose(got["support_logprobs"][:, :3], np.log([0.5, 0.25, 0.25]) + 0 * got["support_logprobs"][:, :3],
                               atol=2e-5)
    ref = oracle_run(w)
    compare(w, ref, got, range(B))


def test_selected_mode_equals_support_mode():
    w = wl.config2(step=3)
    a = gpu_run(w, support_logprobs=True)
    b = gpu_run(w, support_logprobs=False)
    for k in ("tokens", "support_ids", "lengths", "selected_logprob", "row_status"):
        cap = w.capture.astype(bool)
        if k in ("support_ids",):
            for r in np.flatnonzero(cap):
                n = min(int(a["lengths"][r]), w.packed_width)
                assert np.array_equal(a[k][r, :n], b[k][r, :n])
        elif k == "selected_logprob":
            assert np.array_equal(a[k][cap].view(np.uint32), b[k][cap].view(np.uint32))
        else:
            assert np.array_equal(a[k], b[k]), k


def test_no_capture_rows():
    w = wl.config2(step=5)
    ref = oracle_run(w)
    got = gpu_run(w, capture=False)
    assert np.array_equal(got["tokens"], ref.tokens)
    assert (got["lengths"] == 0).all() and (got["row_status"] == 0).all()


def test_capture_subset_matches_all_rows():
    """Capture rows opt in independently: a row's outputs do not depend on which other rows capture."""
    w = wl.config3(B=24)
    w_all = wl.Workload(**{**w.__dict__, "capture": np.ones(w.B, np.uint8)})
    w_some = wl.Workload(**{**w.__dict__, "capture": (np.arange(w.B) % 3 == 1).astype(np.uint8)})
    a, b = gpu_run(w_all), gpu_run(w_some)
    assert np.array_equal(a["tokens"], b["tokens"])
    for r in np.flatnonzero(w_some.capture):
        n = min(int(a["lengths"][r]), w.packed_width)
        assert a["lengths"][r] == b["lengths"][r]
        assert np.array_equal(a["support_ids"][r, :n], b["support_ids"][r, :n])
        assert np.array_equal(a["support_logprobs"][r, :n].view(np.uint32), b["support_logprobs"][r, :n].view(np.uint32))
    assert (b["lengths"][w_some.capture == 0] == 0).all()


def test_deterministic_repeat():
    w = wl.config4(B=24)
    d = to_device(w)
    a, b = gpu_run(w, dev=d), gpu_run(w, dev=d)
    for k in a:
        if a[k] is not None:
            assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k


# ------------------------------------------------------------------------------------------------
# Edge cases
# ------------------------------------------------------------------------------------------------

def _wl(logits, dtype=wl.DT_F32, T=1.0, k=50, tp=0.9, mp=0.0, cap=1, W=64, seed=9, step=0):
    B = logits.shape[0]
    arr = lambda v, dt: np.broadcast_to(np.asarray(v, dt), (B,)).copy()
    return wl.Workload("edge", dtype, logits, arr(T, np.float32), arr(k, np.int32), arr(tp, np.float32),
                       arr(mp, np.float32), arr(cap, np.uint8), W, seed, step)


def _check(w, rows=None):
    rows = list(range(w.B)) if rows is None else rows
    ref = oracle_run(w, rows)
    from sfc_parity import margin_fail
    ok = [r for r in rows if r not in set(margin_fail(ref, rows))]
    got = gpu_run(w)
    return compare(w, ref, got, ok)


@pytest.mark.parametrize("V", [1, 2, 7, 9, 1000, 4099, 50021])
@pytest.mark.parametrize("dtype", [wl.DT_BF16, wl.DT_F32])
def test_ragged_vocab(V, dtype):
    rng = np.random.default_rng(V)
    l = (rng.standard_normal((6, V)) * 2).astype(np.float32)
    logits = wl.f32_to_bf16_bits(l) if dtype == wl.DT_BF16 else l
    k = np.array([1, 3, 50, 0, V, 2000], np.int32)
    w = _wl(logits, dtype, k=k, tp=np.array([0.9, 1.0, 0.5, 0.8, 1.0, 0.95], np.float32),
            mp=np.array([0, 0, 0.05, 0, 0.1, 0], np.float32), W=128)
    assert _check(w) >= 1


@pytest.mark.parametrize("dtype", [wl.DT_BF16, wl.DT_F32])
def test_unaligned_rows_and_stride(dtype):
    """Row starts that are not 16-byte aligned (odd stride), and a stride wider than V."""
    rng = np.random.default_rng(3)
    B, V, stride = 5, 3001, 3007
    base = (rng.standard_normal((B, stride)) * 1.5).astype(np.float32)
    full = wl.f32_to_bf16_bits(base) if dtype == wl.DT_BF16 else base
    w = _wl(np.ascontiguousarray(full[:, :V]), dtype, k=40, tp=0.9, W=64)
    ref = oracle_run(w)
    d = to_device(w)
    if dtype == wl.DT_BF16:
        big = torch.from_numpy(full.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        big = torch.from_numpy(full).cuda()
    d["logits"] = big[:, :V]  # strided view: row_stride = 3007 elements
    got = gpu_run(w, dev=d)
    compare(w, ref, got, range(B))


def test_neg_inf_and_bad_rows():
    rng = np.random.default_rng(4)
    V = 3000
    l = rng.standard_normal((8, V)).astype(np.float32)
    l[0, ::2] = -np.inf              # half the vocabulary masked
    l[1, :] = -np.inf                # no finite logit -> BADPARAM
    l[1, 17] = -np.inf
    l[2, 5] = np.nan                 # NaN -> BADPARAM
    l[3, 2999] = np.inf              # +inf -> BADPARAM
    l[4, :-3] = -np.inf              # three finite tokens, k=50 >= |F|
    T = np.array([1, 1, 1, 1, 1, 0.0, -1, 1], np.float32)      # row 5, 6: bad temperature
    tp = np.array([0.9, 0.9, 0.9, 0.9, 0.9, 0.9, 0.9, np.nan], np.float32)  # row 7: NaN top_p
    w = _wl(l, wl.DT_F32, T=T, k=50, tp=tp, W=64)
    ref = oracle_run(w)
    assert list(ref.row_status) == [0, -1, -1, -1, 0, -1, -1, -1]
    got = gpu_run(w)
    compare(w, ref, got, range(8))


def test_bad_min_p_rows():
    l = np.random.default_rng(5).standard_normal((3, 500)).astype(np.float32)
    w = _wl(l, mp=np.array([-0.1, 1.5, np.nan], np.float32))
    got = gpu_run(w)
    assert (got["row_status"] == -1).all() and (got["tokens"] == -1).all()


@pytest.mark.parametrize("dtype", [wl.DT_BF16, wl.DT_F32])
def test_top_k_disabled_long_rows(dtype):
    """top_k off with top-p / min-p binding on long rows: candidates cannot be bounded on chip, so these
    rows take the multi-pass path (radix descent on counts and fixed-point masses)."""
    B, V = 6, 70000
    w0 = wl.config5(B=B)
    l = wl.bf16_bits_to_f32(w0.logits[:, :V])
    logits = wl.f32_to_bf16_bits(l) if dtype == wl.DT_BF16 else np.ascontiguousarray(l)
    w = _wl(logits, dtype, T=np.array([1, 0.8, 1.2, 1, 1, 2], np.float32), k=np.array([0, -1, V, 0, 0, 0], np.int32),
            tp=np.array([0.9, 0.5, 0.97, 1.0, 0.6, 1.0], np.float32), mp=np.array([0, 0, 0, 0.02, 0.001, 0], np.float32),
            W=1024)
    assert _check(w) >= 4


def test_huge_tie_group():
    """Every logit equal: the tie group at the k-th logit is the whole row, far larger than the buffer."""
    B, V = 3, 60000
    l = np.zeros((B, V), np.float32)
    l[1, 12345] = 1.0  # one larger token; the rest tie
    w = _wl(wl.f32_to_bf16_bits(l), wl.DT_BF16, k=np.array([5, 2, 1], np.int32), tp=1.0, W=2048)
    ref = oracle_run(w)
    got = gpu_run(w)
    compare(w, ref, got, range(B))
    assert got["lengths"][0] == V and got["row_status"][0] == 1  # overflow: |S| = V > W


def test_large_support_wide_output():
    """W = 16384 (the widest class) with a top-k of 12000 on fp32 logits."""
    B, V = 4, 129280
    w0 = wl.config4(B=B)
    w = wl.Workload(**{**w0.__dict__, "top_k": np.full(B, 12000, np.int32), "packed_width": 16384,
                       "capture": np.ones(B, np.uint8)})
    assert _check(w) >= 3


@pytest.mark.parametrize("W", [1, 7, 20])
def test_overflow_narrow_packed_width(W):
    w0 = wl.config3(B=9)
    w = wl.Workload(**{**w0.__dict__, "packed_width": W})
    got = gpu_run(w)
    ref = oracle_run(w)
    compare(w, ref, got, range(w.B))
    assert (got["row_status"] == (ref.support_size > W)).all()


def test_min_p_one_and_top_p_zero():
    l = np.random.default_rng(6).standard_normal((4, 5000)).astype(np.float32)
    l[:, 10] = 9.0
    l[:, 20] = 9.0
    w = _wl(l, k=np.array([0, 100, 0, 100], np.int32), tp=np.array([0.0, 0.0, 1.0, 1.0], np.float32),
            mp=np.array([0, 0, 1.0, 1.0], np.float32))
    got = gpu_run(w)
    assert (got["lengths"] == 2).all()
    assert (got["support_ids"][:, :2] == [10, 20]).all()


# ------------------------------------------------------------------------------------------------
# The value-bins finish (bf16) on skewed pools and its fallbacks: many candidates per marked vector in
# one part of the pool, a sample threshold above the k-th largest logit, and more distinct candidate
# values than the bins hold.
# ------------------------------------------------------------------------------------------------

V_LONG = 151936


def test_dense_tie_block_in_one_pool_part():
    """640 tied tokens fill the first 80 vectors (eight candidates each, one per vector elsewhere). Row 0's
    top-k cut lands inside the tie group, row 1's below the second group (an overflowing row)."""
    l = np.full((2, V_LONG), -10.0, np.float32)
    l[:, :640] = 5.0
    ids = 8 * (32 * np.arange(560) + 100)
    l[:, ids] = 4.0
    w = _wl(wl.f32_to_bf16_bits(l), wl.DT_BF16, k=np.array([200, 700], np.int32), tp=1.0, W=1024)
    ref = oracle_run(w)
    got = gpu_run(w)
    compare(w, ref, got, range(2))
    assert got["lengths"][0] == 640 and got["lengths"][1] == 1200 and got["row_status"][1] == 1


def test_sample_threshold_above_kth_falls_back():
    """All of the row's large logits sit in the first sampled chunk: the sample threshold overshoots the
    k-th largest logit, the bins finish gives up and the multi-pass path answers."""
    rng = np.random.default_rng(11)
    l = (rng.standard_normal((2, V_LONG)) - 10.0).astype(np.float32)
    l[:, 8 * 16 * np.arange(64)] = 5.0
    w = _wl(wl.f32_to_bf16_bits(l), wl.DT_BF16, k=np.array([100, 100], np.int32), tp=np.array([1.0, 0.97], np.float32),
            W=256)
    assert _check(w) >= 1


def test_more_distinct_values_than_bins():
    """2000 distinct bf16 codes spread over the row (the rest far below): more distinct candidates than
    value bins, so a sorting finish answers."""
    codes = np.full((2, V_LONG), wl.f32_to_bf16_bits(np.array([-100.0], np.float32))[0], np.uint16)
    planted = (0x3F80 - np.arange(2000)).astype(np.uint16)
    codes[:, 75 * np.arange(2000) + 3] = planted
    codes[1, 75 * np.arange(2000) + 3] = planted[::-1]  # the same values at mirrored ids
    w = _wl(codes, wl.DT_BF16, k=np.array([1200, 900], np.int32), tp=1.0, W=2048)
    assert _check(w) == 2
