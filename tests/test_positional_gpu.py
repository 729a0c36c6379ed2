"""GPU parity of positional truncation (SFC_FLAG_POSITIONAL): top-k keeps the first k positions of the
canonical order and top-p the positions whose own exclusive cumulative probability is <= top_p, so the
last tie group of the joint support is cut to its lowest ids (prhub summary of SGLang PR #36630,
实现拆解 item 5). Every finish is covered: value bins (bf16), the sorting finishes (fp32 and more
distinct values than bins), the multi-pass path (tie groups far larger than the chip holds) and rows
split over a cluster."""
import numpy as np
import pytest

from top_support_capture_gb300 import workloads as wl
from sfc_parity import clear_margins, compare, gpu_run, margin_fail, oracle_run

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

POS = dict(positional=True)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_support_capture_gb300 as sfc

    sfc.load_library()


def _wl(logits, dtype=wl.DT_F32, T=1.0, k=50, tp=1.0, mp=0.0, cap=1, W=1024, seed=9, step=0):
    B = logits.shape[0]
    arr = lambda v, dt: np.broadcast_to(np.asarray(v, dt), (B,)).copy()
    return wl.Workload("positional", dtype, logits, arr(T, np.float32), arr(k, np.int32), arr(tp, np.float32),
                       arr(mp, np.float32), arr(cap, np.uint8), W, seed, step)


def _check(w, rows=None, min_rows=None, **call_kw):
    rows = list(range(w.B)) if rows is None else list(rows)
    ref = oracle_run(w, rows, **POS)
    ok = [r for r in rows if r not in set(margin_fail(ref, rows))]
    assert len(ok) >= (len(rows) if min_rows is None else min_rows), (len(ok), len(rows))
    got = gpu_run(w, positional=True, **call_kw)
    compare(w, ref, got, ok)
    return ref, got


def _enc(l, dtype):
    return wl.f32_to_bf16_bits(l) if dtype == wl.DT_BF16 else np.ascontiguousarray(l, np.float32)


@pytest.mark.parametrize("step", [0, 5])
def test_config2_all_rows(step):
    w, ref, left = clear_margins(lambda salt: wl.config2(step=step, salt=salt), 64, list(range(64)), **POS)
    assert not left
    compare(w, ref, gpu_run(w, positional=True), range(64))


def test_config1_tiny_ties_everywhere():
    """Logits on a 9-value grid: almost every cut lands inside a tie group."""
    for V in (5, 8, 16):
        w, ref, left = clear_margins(lambda salt: wl.config1_tiny(V, salt=salt), 64, list(range(64)), **POS)
        assert not left
        compare(w, ref, gpu_run(w, positional=True), range(64))


def test_config3_sampled_rows_and_nesting():
    """Full-size bf16 rows quantised to 1/16-logit steps (ties at every cut); the positional support is
    a prefix of the joint one."""
    B = 256
    rows = sorted(set(list(range(0, 12)) + list(range(120, 129)) + list(range(B - 12, B))))
    w, ref, left = clear_margins(lambda salt: wl.config3(salt=salt), B, rows, **POS)
    assert not left
    got = gpu_run(w, positional=True)
    compare(w, ref, got, rows)
    joint = gpu_run(w)
    assert (got["lengths"] <= joint["lengths"]).all()
    assert (got["lengths"] <= w.top_k).all()
    for r in range(B):
        n = min(int(got["lengths"][r]), w.packed_width)
        assert np.array_equal(got["support_ids"][r, :n], joint["support_ids"][r, :n]), r


def test_config4_sampled_rows():
    B = 256
    w0 = wl.config4()
    rows = sorted(np.flatnonzero(w0.capture)[:8].tolist() + np.flatnonzero(w0.capture == 0)[:6].tolist())
    w, ref, left = clear_margins(lambda salt: wl.config4(salt=salt), B, rows, **POS)
    assert not left
    compare(w, ref, gpu_run(w, positional=True), rows)


@pytest.mark.parametrize("B", [1, 32])
def test_config5_split_rows(B):
    """Short batches of the long vocabulary with the top-k hint: rows split over a cluster."""
    w, ref, left = clear_margins(lambda salt: wl.config5(B=B, salt=salt), B, list(range(B)), **POS)
    assert not left
    compare(w, ref, gpu_run(w, positional=True, max_top_k=50), range(B))


@pytest.mark.parametrize("dtype", [wl.DT_BF16, wl.DT_F32])
def test_cuts_inside_tie_groups(dtype):
    """Row 0: top-k inside a 300-token tie group. Row 1: top-p inside it (the cut falls mid-way between
    two members' masses). Row 2: min-p below the group (positional and joint agree). Row 3: top-k and
    top-p both inactive. Row 4: top-k inside the group with top-p binding later. Row 5: V below k."""
    V = 50000
    rng = np.random.default_rng(21)
    base = (rng.standard_normal(V) * 0.3 - 12.0).astype(np.float32)
    tied = rng.choice(np.arange(3, V), 300, replace=False)
    l = np.tile(base, (6, 1))
    l[:, [0, 1, 2]] = [3.0, 2.5, 2.0]
    l[:, tied] = 1.0
    # member weight e^1 over Z ~ e^3 + e^2.5 + e^2 + 300 e^1: a top-p cut half-way between members
    w_all = np.exp(l[1].astype(np.float64) - 3.0)
    Z = w_all.sum()
    above = (w_all[:3]).sum() / Z
    wm = w_all[tied[0]] / Z
    tp1 = above + 120.5 * wm
    w = _wl(_enc(l, dtype), dtype, k=np.array([50, 0, 0, 0, 140, 10], np.int32),
            tp=np.array([1.0, tp1, 1.0, 1.0, above + 200.5 * wm, 1.0], np.float32),
            mp=np.array([0, 0, 0.001, 0, 0, 0], np.float32), W=512)
    ref, got = _check(w)
    assert got["lengths"][0] == 50
    assert got["lengths"][1] == 3 + 121
    assert got["lengths"][4] == 140
    assert list(got["support_ids"][0, 3:50]) == sorted(tied)[:47]


def test_dense_tie_block_bins_finish():
    """640 tied tokens in the first vectors of a long bf16 row: k = 200 keeps their 200 lowest ids; k = 700
    keeps all 640 and the 60 lowest ids of the next group."""
    V = 151936
    l = np.full((2, V), -10.0, np.float32)
    l[:, :640] = 5.0
    ids = 8 * (32 * np.arange(560) + 100)
    l[:, ids] = 4.0
    w = _wl(wl.f32_to_bf16_bits(l), wl.DT_BF16, k=np.array([200, 700], np.int32), tp=1.0, W=1024)
    ref, got = _check(w)
    assert list(got["lengths"]) == [200, 700]
    assert (got["support_ids"][0, :200] == np.arange(200)).all()
    assert (got["support_ids"][1, 640:700] == np.sort(ids)[:60]).all()


def test_more_distinct_values_than_bins():
    codes = np.full((2, 151936), wl.f32_to_bf16_bits(np.array([-100.0], np.float32))[0], np.uint16)
    planted = (0x3F80 - np.arange(2000)).astype(np.uint16)
    codes[:, 75 * np.arange(2000) + 3] = planted
    codes[1, 75 * np.arange(2000) + 3] = planted[::-1]
    w = _wl(codes, wl.DT_BF16, k=np.array([1200, 900], np.int32), tp=np.array([1.0, 0.9], np.float32), W=2048)
    _check(w)


@pytest.mark.parametrize("dtype", [wl.DT_BF16, wl.DT_F32])
def test_huge_tie_groups_multi_pass(dtype):
    """Tie groups far larger than the chip holds (the multi-pass path): row 0 every logit equal with k = 5;
    row 1 a 20000-token group holding the mass, top-p cut half-way between two members (6001 kept);
    row 2 one larger token then the whole row tied, k = 3000 (an overflowing support)."""
    V = 60000
    l = np.zeros((3, V), np.float32)
    l[1] = -30.0
    l[1, np.arange(0, V, 3)] = 0.0
    l[2, 12345] = 1.0
    w = _wl(_enc(l, dtype), dtype, k=np.array([5, 0, 3000], np.int32),
            tp=np.array([1.0, 0.300025, 1.0], np.float32), W=2048)
    ref, got = _check(w)
    assert list(got["lengths"]) == [5, 6001, 3000]
    assert (got["support_ids"][0, :5] == np.arange(5)).all()
    assert (got["support_ids"][1, :6001 if 6001 <= 2048 else 2048] == np.arange(0, 3 * 2048, 3)).all()
    assert got["support_ids"][2, 0] == 12345 and (got["support_ids"][2, 1:2048] == np.arange(2047)).all()
    assert list(got["row_status"]) == [0, 1, 1]


def test_support_mask_of_a_cut_group():
    """The overflow bitmask carries the positional support (a cut tie group) bit for bit."""
    import oracle

    V = 60000
    l = np.zeros((2, V), np.float32)
    l[1, 777] = 2.0
    w = _wl(wl.f32_to_bf16_bits(l), wl.DT_BF16, k=np.array([3000, 2500], np.int32), tp=1.0, W=1000)
    ref = oracle_run(w, **POS, want_mask=True)
    got = gpu_run(w, positional=True, support_mask=True)
    compare(w, ref, got, range(2))
    mask = got["support_mask"].view(np.uint32)
    for r in range(2):
        assert np.array_equal(mask[r], ref.support_mask[r]), r
        assert np.array_equal(mask[r], oracle.support_bits(np.arange(2500 if r else 3000), V)), r


def test_positional_with_greedy_rows():
    w0 = wl.config2()
    T = w0.temperature.copy()
    T[::4] = 0.0
    w = wl.Workload(**{**w0.__dict__, "temperature": T, "capture": np.ones(w0.B, np.uint8)})
    ref = oracle_run(w, greedy_t0=True, positional=True)
    rows = [r for r in range(w.B) if r not in set(margin_fail(ref, range(w.B)))]
    assert len(rows) >= 48
    got = gpu_run(w, greedy_t0=True, positional=True)
    compare(w, ref, got, rows)
    assert (got["lengths"][::4] == 1).all()
