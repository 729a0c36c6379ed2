"""GPU parity of greedy rows (temperature 0 under SFC_FLAG_GREEDY_T0) on every finish path."""
import numpy as np
import pytest

import oracle
from top_support_capture_gb300 import workloads as wl
from sfc_parity import compare, margin_fail, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_support_capture_gb300 as sfc

    sfc.load_library()


def _run(w, greedy=True):
    import top_support_capture_gb300 as sfc

    d = to_device(w)
    out = sfc.sample_filter_capture(d["logits"], d["temperature"], d["top_k"], d["top_p"], d["min_p"], w.seed, w.step,
                                    d["capture_rows"], w.packed_width, greedy_t0=greedy)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in out._asdict().items()}


def _ref(w, greedy=True):
    return oracle.sample_filter_capture(w.logits, w.dtype, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, w.step,
                                        w.capture, w.packed_width, greedy_t0=greedy)


@pytest.mark.parametrize("make", [lambda: wl.config2(), lambda: wl.config3(B=12), lambda: wl.config4(B=8)])
def test_greedy_rows_among_sampled_rows(make):
    w0 = make()
    T = w0.temperature.copy()
    T[::3] = 0.0
    w = wl.Workload(**{**w0.__dict__, "temperature": T, "capture": np.ones(w0.B, np.uint8)})
    ref = _ref(w)
    rows = [r for r in range(w.B) if r not in set(margin_fail(ref, range(w.B)))]
    got = _run(w)
    compare(w, ref, got, rows)
    g = np.flatnonzero(T == 0.0)
    assert (got["lengths"][g] == 1).all() and (got["selected_logprob"][g] == 0.0).all()
    # without the flag those rows are bad rows
    plain = _run(w, greedy=False)
    assert (plain["row_status"][g] == -1).all()


def test_greedy_ties_and_huge_tie_group():
    """Ties at the maximum go to the lowest id; a row whose maximum is shared by every token (far more
    than the on-chip pool holds) takes the multi-pass path."""
    B, V = 4, 60000
    l = np.zeros((B, V), np.float32)
    l[1, [40000, 7, 59999]] = 2.0
    l[2, 12345] = -1.0  # all others tie at 0
    l[3] = np.random.default_rng(2).standard_normal(V).astype(np.float32)
    for dtype in (wl.DT_BF16, wl.DT_F32):
        logits = wl.f32_to_bf16_bits(l) if dtype == wl.DT_BF16 else l
        w = wl.Workload("greedy_ties", dtype, logits, np.zeros(B, np.float32), np.full(B, 50, np.int32),
                        np.full(B, 0.9, np.float32), np.zeros(B, np.float32), np.ones(B, np.uint8), 64, 1, 0)
        ref = _ref(w)
        got = _run(w)
        compare(w, ref, got, range(B))
        assert list(got["tokens"][:3]) == [0, 7, 0]
