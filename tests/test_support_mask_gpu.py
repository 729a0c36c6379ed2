"""GPU parity of the support bitmask written for overflowing capturing rows, on every finish path:
value bins (bf16), the sorting finish (f32) and the multi-pass path (top-k off), aligned and not."""
import numpy as np
import pytest

import oracle
from top_support_capture_gb300 import workloads as wl
from sfc_parity import compare, oracle_run, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SENTINEL = 0x5A5A5A5A


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_support_capture_gb300 as sfc

    sfc.load_library()


def _run_with_mask(w, logits_dev=None):
    import top_support_capture_gb300 as sfc

    d = to_device(w)
    L = d["logits"] if logits_dev is None else logits_dev
    V = w.logits.shape[1]
    out = sfc.allocate_outputs(w.B, w.packed_width, "cuda", True, True, V)
    out.support_mask.fill_(SENTINEL)
    sfc.sample_filter_capture_into(out, L, d["temperature"], d["top_k"], d["top_p"], d["min_p"], w.seed, w.step,
                                   d["capture_rows"], w.packed_width)
    torch.cuda.synchronize()
    got = {k: (None if v is None else v.cpu().numpy()) for k, v in out._asdict().items()}
    got["support_mask"] = got["support_mask"].view(np.uint32)
    return got


def _check_masks(w, got, rows):
    ref = oracle.sample_filter_capture(w.logits, w.dtype, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, w.step,
                                       w.capture, w.packed_width, rows=rows, want_mask=True)
    compare(w, ref, got, rows)
    n_over = 0
    for r in rows:
        if ref.row_status[r] == oracle.ROW_OVERFLOW:
            n_over += 1
            np.testing.assert_array_equal(got["support_mask"][r], ref.support_mask[r])
        else:
            assert (got["support_mask"][r] == SENTINEL).all(), r  # untouched
    return n_over


def test_mask_bins_finish_bf16():
    w = wl.config3(B=12)  # k = 1024 rows overflow W = 1024
    from sfc_parity import margin_fail

    ref = oracle_run(w)
    rows = [r for r in range(w.B) if r not in set(margin_fail(ref, range(w.B)))]
    assert _check_masks(w, _run_with_mask(w), rows) >= 2


def test_mask_sorting_finish_f32():
    w0 = wl.config4(B=6)
    w = wl.Workload(**{**w0.__dict__, "packed_width": 300, "capture": np.ones(6, np.uint8)})
    from sfc_parity import margin_fail

    ref = oracle_run(w)
    rows = [r for r in range(w.B) if r not in set(margin_fail(ref, range(w.B)))]
    assert _check_masks(w, _run_with_mask(w), rows) >= 3


@pytest.mark.parametrize("dtype", [wl.DT_BF16, wl.DT_F32])
def test_mask_multipass_top_k_off(dtype):
    rng = np.random.default_rng(21 + dtype)
    B, V = 4, 70001
    l = (np.round(rng.standard_normal((B, V)) * 8) / 4).astype(np.float32)  # quarter-logit steps: wide margins
    logits = wl.f32_to_bf16_bits(l) if dtype == wl.DT_BF16 else l
    w = wl.Workload("mask_topk_off", dtype, logits, np.ones(B, np.float32), np.zeros(B, np.int32),
                    np.array([0.9, 0.5, 0.97, 0.8], np.float32), np.zeros(B, np.float32), np.ones(B, np.uint8),
                    16, 3, 0)
    from sfc_parity import margin_fail

    ref = oracle_run(w)
    rows = [r for r in range(w.B) if r not in set(margin_fail(ref, range(w.B)))]
    assert _check_masks(w, _run_with_mask(w), rows) >= 3


def test_mask_unaligned_rows():
    """Rows that start off a 16-byte boundary (an odd row stride) take the element-load mask path."""
    w0 = wl.config3(B=6)
    V = w0.logits.shape[1]
    padded = np.zeros((w0.B, V + 1), np.uint16)
    padded[:, :V] = w0.logits
    dev = torch.from_numpy(padded.view(np.int16)).cuda().view(torch.bfloat16)[:, :V]
    from sfc_parity import margin_fail

    ref = oracle_run(w0)
    rows = [r for r in range(w0.B) if r not in set(margin_fail(ref, range(w0.B)))]
    assert _check_masks(w0, _run_with_mask(w0, logits_dev=dev), rows) >= 1
