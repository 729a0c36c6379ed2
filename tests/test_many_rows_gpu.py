"""GPU parity on a batch of many short rows (far more rows than CTA slots: the grid runs in waves),
with per-row parameters drawn at random, compared with the oracle on sampled rows; on every row the
drawn token lies in the captured support."""
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


@pytest.mark.parametrize("dtype", [wl.DT_BF16, wl.DT_F32])
def test_three_thousand_rows(dtype):
    B, V = 3000, 5003
    rng = np.random.default_rng(99 + dtype)
    l = (rng.standard_normal((B, V)) * rng.uniform(0.5, 3.0, (B, 1))).astype(np.float32)
    logits = wl.f32_to_bf16_bits(l) if dtype == wl.DT_BF16 else l
    w = wl.Workload("many_rows", dtype, logits, rng.uniform(0.5, 1.5, B).astype(np.float32),
                    rng.integers(0, 2000, B).astype(np.int32), rng.uniform(0.3, 1.0, B).astype(np.float32),
                    rng.choice([0.0, 0.02, 0.1], B).astype(np.float32), (rng.random(B) < 0.7).astype(np.uint8),
                    512, 4, 11)
    got = gpu_run(w)
    sample = sorted(set(rng.choice(B, 48, replace=False).tolist() + [0, B - 1]))
    ref = oracle_run(w, sample)
    rows = [r for r in sample if r not in set(margin_fail(ref, sample))]
    assert len(rows) >= 40
    compare(w, ref, got, rows)
    assert (got["row_status"] >= 0).all()
    for r in np.flatnonzero(w.capture):
        n = min(int(got["lengths"][r]), w.packed_width)
        assert got["lengths"][r] > w.packed_width or got["tokens"][r] in got["support_ids"][r, :n], r
