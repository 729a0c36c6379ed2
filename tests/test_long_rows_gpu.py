"""GPU parity on rows longer than the on-chip candidate bitmap covers (one bit per 16-byte vector:
2^17 vectors in the narrow class, 2^18 in the wide one). Such rows cannot mark their candidates on
chip and take the multi-pass path; a short batch of them split over a cluster gives each CTA a slice
the bitmap does cover."""
import numpy as np
import pytest

from top_support_capture_gb300 import workloads as wl
from sfc_parity import compare, gpu_run, margin_fail, oracle_run

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_support_capture_gb300 as sfc

    sfc.load_library()


def _rows(B, V, seed):
    rng = np.random.default_rng(seed)
    l = np.empty((B, V), np.float32)
    for r in range(B):
        l[r] = (-1.1 * np.log1p(rng.permutation(V)) + rng.normal(0, 1.2, V)).astype(np.float32)
    return l


def _wl(logits, dtype, k, tp, mp, W):
    B = logits.shape[0]
    arr = lambda v, dt: np.broadcast_to(np.asarray(v, dt), (B,)).copy()
    return wl.Workload("long_rows", dtype, logits, arr(1.0, np.float32), arr(k, np.int32), arr(tp, np.float32),
                       arr(mp, np.float32), arr(1, np.uint8), W, 17, 3)


@pytest.mark.parametrize("dtype,V,W", [(wl.DT_BF16, 1_200_000, 1024), (wl.DT_F32, 600_000, 1024),
                                       (wl.DT_BF16, 2_200_000, 4096)])
def test_rows_beyond_the_bitmap(dtype, V, W):
    l = _rows(3, V, V)
    logits = wl.f32_to_bf16_bits(l) if dtype == wl.DT_BF16 else l
    w = _wl(logits, dtype, k=np.array([50, 1000, 0], np.int32), tp=np.array([0.9, 0.95, 0.5], np.float32),
            mp=np.array([0.0, 0.01, 0.0], np.float32), W=W)
    ref = oracle_run(w)
    rows = [r for r in range(w.B) if r not in set(margin_fail(ref, range(w.B)))]
    assert len(rows) >= 2
    compare(w, ref, gpu_run(w), rows)


def test_long_row_split_over_a_cluster():
    """One 1.2M-token bf16 row with the top-k bound: eight slices of 150k tokens, each covered."""
    l = _rows(1, 1_200_000, 5)
    w = _wl(wl.f32_to_bf16_bits(l), wl.DT_BF16, k=50, tp=0.95, mp=0.02, W=1024)
    ref = oracle_run(w)
    assert not margin_fail(ref, [0])
    compare(w, ref, gpu_run(w, max_top_k=50), [0])
