"""GPU test of the failure path: a bounded wait of the kernel that runs out.

Every wait of the kernel for its own bulk copies has a limit, after which the row reports SFC_ROW_TIMEOUT
instead of hanging the GPU. With SFC_FLAG_TEST_STALL the copy of each CTA's first ring stage is never
issued (a completion that nothing will signal), and the pass gives up after a few polls. Every row that
streams must then report the timeout (token -1, length 0), rows rejected by their parameters stay BADPARAM,
the copies that were issued are awaited before the kernel ends, and the next normal call on the same
stream must give exactly what a call on a fresh stream gives. Covered: one CTA per row, rows split into
slices (workspace) and into a thread-block cluster, the wide class, and float rows. Nothing here faults,
traps or hangs a GPU: the failure is a missing completion that the kernel's own limits turn into a status.
"""
import numpy as np
import pytest

from top_support_capture_gb300 import workloads as wl
from sfc_parity import clear_margins, compare, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROW_TIMEOUT = -2


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_support_capture_gb300 as sfc

    sfc.load_library()


def _call(w, d, stream, **kw):
    import top_support_capture_gb300 as sfc

    out = sfc.allocate_outputs(w.B, w.packed_width, "cuda")
    with torch.cuda.stream(stream):
        sfc.sample_filter_capture_into(out, d["logits"], d["temperature"], d["top_k"], d["top_p"], d["min_p"], w.seed,
                                       w.step, d["capture_rows"], w.packed_width, stream=stream, **kw)
    stream.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in out._asdict().items()}


CASES = {
    "one_cta_per_row": (lambda salt: wl.config3(B=12, salt=salt), dict(slices=1)),
    "slices": (lambda salt: wl.config3(B=12, salt=salt), dict(slices=4)),
    "cluster": (lambda salt: wl.config5(B=4, salt=salt), dict(max_top_k=50)),
    "wide_class": (lambda salt: wl.config4(B=4, salt=salt), dict()),
    "float_rows": (lambda salt: wl.config1(salt=salt), dict()),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_stalled_copy_reports_timeout_then_the_next_call_is_clean(case):
    make, kw = CASES[case]
    B = make(None).B
    w, ref, left = clear_margins(make, B, list(range(B)))
    assert not left
    d = to_device(w)
    s = torch.cuda.Stream()
    stalled = _call(w, d, s, test_stall=True, **kw)
    assert (stalled["row_status"] == ROW_TIMEOUT).all(), stalled["row_status"]
    assert (stalled["tokens"] == -1).all()
    assert (stalled["lengths"] == 0).all()
    after = _call(w, d, s, **kw)  # the same stream, right after the failed call
    fresh = _call(w, d, torch.cuda.Stream(), **kw)
    for k in ("tokens", "lengths", "row_status", "selected_logprob"):
        assert np.array_equal(after[k].view(np.uint8), fresh[k].view(np.uint8)), k
    for r in range(B):
        n = min(int(fresh["lengths"][r]), w.packed_width)
        assert np.array_equal(after["support_ids"][r, :n], fresh["support_ids"][r, :n]), r
        assert np.array_equal(after["support_logprobs"][r, :n].view(np.uint32),
                              fresh["support_logprobs"][r, :n].view(np.uint32)), r
    assert compare(w, ref, after, range(B)) == B


def test_stall_leaves_rows_with_bad_parameters_bad():
    w = wl.config3(B=6)
    T = w.temperature.copy()
    T[[1, 4]] = -1.0
    w = wl.Workload(**{**w.__dict__, "temperature": T})
    got = _call(w, to_device(w), torch.cuda.Stream(), test_stall=True)
    assert list(got["row_status"]) == [ROW_TIMEOUT, -1, ROW_TIMEOUT, ROW_TIMEOUT, -1, ROW_TIMEOUT]
    assert (got["tokens"] == -1).all()
