"""GPU parity of rows split over a thread-block cluster (short batches with a small top-k hint): each
row is streamed by 2, 4 or 8 CTAs whose candidates meet in the first CTA's shared memory."""
import numpy as np
import pytest

import oracle
from top_support_capture_gb300 import workloads as wl
from sfc_parity import clear_margins, compare, margin_fail, oracle_run, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_support_capture_gb300 as sfc

    sfc.load_library()


def _run(w, max_top_k, logits_dev=None, **kw):
    import top_support_capture_gb300 as sfc

    d = to_device(w)
    L = d["logits"] if logits_dev is None else logits_dev
    out = sfc.sample_filter_capture(L, d["temperature"], d["top_k"], d["top_p"], d["min_p"], w.seed, w.step,
                                    d["capture_rows"], w.packed_width, max_top_k=max_top_k, **kw)
    torch.cuda.synchronize()
    got = {k: (None if v is None else v.cpu().numpy()) for k, v in out._asdict().items()}
    if got.get("support_mask") is not None:
        got["support_mask"] = got["support_mask"].view(np.uint32)
    return got


def _check(w, max_top_k, rows=None, **kw):
    rows = list(range(w.B)) if rows is None else rows
    ref = oracle_run(w, rows)
    ok = [r for r in rows if r not in set(margin_fail(ref, rows))]
    return compare(w, ref, _run(w, max_top_k, **kw), ok)


@pytest.mark.parametrize("B", [1, 8, 32, 128])
def test_short_batches_of_the_long_vocabulary(B):
    """V = 262144, top_k 50: B = 1, 8, 32 split 8 ways, B = 128 split 2 ways."""
    w, ref, left = clear_margins(lambda salt: wl.config5(B=B, salt=salt), B, list(range(B)))
    assert not left
    assert compare(w, ref, _run(w, 50), range(B)) == B


def test_hint_on_rows_too_short_to_split():
    """V = 32000: slices would be shorter than two ring stages, so the hint leaves one CTA per row."""
    w0 = wl.config2()
    w = wl.Workload(**{**w0.__dict__, "top_k": np.minimum(w0.top_k, 200).astype(np.int32)})
    assert _check(w, 256) >= 56


@pytest.mark.parametrize("dtype", [wl.DT_BF16, wl.DT_F32])
def test_split_ragged_unaligned_rows(dtype):
    """Rows that start off a 16-byte boundary (an odd stride) with a ragged end: the first slice reads the
    head scalars, the last the tail."""
    rng = np.random.default_rng(31 + dtype)
    B, V = 4, 50021
    l = (rng.standard_normal((B, V)) * 2).astype(np.float32)
    logits = wl.f32_to_bf16_bits(l) if dtype == wl.DT_BF16 else l
    w = wl.Workload("split_ragged", dtype, logits, np.ones(B, np.float32), np.array([5, 50, 1, 100], np.int32),
                    np.array([0.9, 0.5, 1.0, 0.95], np.float32), np.zeros(B, np.float32), np.ones(B, np.uint8), 64, 4, 0)
    padded = np.zeros((B, V + 1), logits.dtype)
    padded[:, :V] = logits
    if dtype == wl.DT_BF16:
        dev = torch.from_numpy(padded.view(np.int16)).cuda().view(torch.bfloat16)[:, :V]
    else:
        dev = torch.from_numpy(padded).cuda()[:, :V]
    ref = oracle_run(w)
    ok = [r for r in range(B) if r not in set(margin_fail(ref, range(B)))]
    assert compare(w, ref, _run(w, 100, logits_dev=dev), ok) >= 3


def test_split_rows_beyond_the_hint_bad_rows_and_greedy():
    """Rows whose top-k breaks the hint (off, 2000) stay exact; a NaN in the last slice and +inf in a
    middle slice make bad rows; temperature-0 rows are greedy under the flag."""
    w0 = wl.config5(B=8)
    l = w0.logits.copy()
    l[2, -5] = 0x7FC0  # bf16 NaN in the last slice
    l[3, 100000] = 0x7F80  # bf16 +inf in a middle slice
    k = np.array([50, 0, 50, 50, 2000, 50, 50, 50], np.int32)
    T = w0.temperature.copy()
    T[5] = 0.0
    w = wl.Workload(**{**w0.__dict__, "logits": l, "top_k": k, "temperature": T})
    ref = oracle.sample_filter_capture(w.logits, w.dtype, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, w.step,
                                       w.capture, w.packed_width, greedy_t0=True)
    ok = [r for r in range(w.B) if r not in set(margin_fail(ref, range(w.B)))]
    got = _run(w, 50, greedy_t0=True)
    compare(w, ref, got, ok)
    assert got["row_status"][2] == -1 and got["row_status"][3] == -1
    assert got["lengths"][5] == 1


def test_split_overflow_mask_and_determinism():
    w0 = wl.config5(B=4)
    w = wl.Workload(**{**w0.__dict__, "packed_width": 8})
    ref = oracle.sample_filter_capture(w.logits, w.dtype, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, w.step,
                                       w.capture, w.packed_width, want_mask=True)
    ok = [r for r in range(w.B) if r not in set(margin_fail(ref, range(w.B)))]
    a = _run(w, 50, support_mask=True)
    b = _run(w, 50, support_mask=True)
    compare(w, ref, a, ok)
    for r in ok:
        if ref.row_status[r] == oracle.ROW_OVERFLOW:
            np.testing.assert_array_equal(a["support_mask"][r], ref.support_mask[r])
    for k_ in a:
        if a[k_] is not None:
            assert np.array_equal(a[k_], b[k_], equal_nan=True), k_
