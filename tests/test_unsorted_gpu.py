"""The bucket finish's route for rows that do not capture: S found as three tests on a candidate's key
(the k-th largest key, the top-p cut's tie group located by fixed-point bin masses, min-p), the race run
over the candidate pool as it lies, no sort of K. Float rows take it whenever they do not capture; the
same rows captured take the sorted route. Both must draw the oracle's tokens (rows clear of the
oracle's margins), and therefore the same tokens.
"""
import numpy as np
import pytest
import torch

from sfc_parity import clear_margins, compare, gpu_run, oracle_run
from top_support_capture_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_support_capture_gb300 as sfc

    sfc.load_library()


def _both_routes(make, B):
    w, ref, left = clear_margins(make, B, range(B))
    assert not left, f"rows {left} kept failing the margins"
    w_cap = wl.Workload(**{**w.__dict__, "capture": np.ones(B, np.uint8)})
    sorted_route = gpu_run(w_cap)
    unsorted_route = gpu_run(w, capture=False)
    assert compare(w, ref, unsorted_route, range(B), capture=False) == B
    assert compare(w_cap, oracle_run(w_cap), sorted_route, range(B)) == B
    np.testing.assert_array_equal(unsorted_route["tokens"], sorted_route["tokens"])
    return w, ref


@pytest.mark.parametrize("step", [0, 3])
def test_wide_float_rows_without_capture(step):
    """The wide class (V=129280 f32, top_k 8192, top_p alternating 0.95 / 1.0), 64 rows."""
    _both_routes(lambda salt: wl.config4(step=step, salt=salt, B=64), 64)


def _grid_rows(salt, B=96, V=3000, step=0):
    """Float rows on a coarse grid (long tie groups at every cut), narrow class: top_k in [1, 700] or
    disabled (every token a candidate: V fits the candidate pool), top_p in {0.3, 0.7, 0.95, 1}, min_p in
    {0, 0.02}, T in {0.7, 1, 1.4}."""
    s = np.zeros(B, np.int64) if salt is None else np.asarray(salt, np.int64)
    l = np.empty((B, V), np.float32)
    T = np.empty(B, np.float32)
    k = np.empty(B, np.int32)
    tp = np.empty(B, np.float32)
    mp = np.empty(B, np.float32)
    for r in range(B):
        g = np.random.default_rng([91, r, step, int(s[r])])
        l[r] = (np.round(g.normal(0.0, 2.0, V) * 4.0) / 4.0).astype(np.float32)  # 1/4-logit grid
        T[r] = (0.7, 1.0, 1.4)[r % 3]
        k[r] = 0 if r % 7 == 0 else int(g.integers(1, 701))
        tp[r] = (0.3, 0.7, 0.95, 1.0)[(r // 3) % 4]
        mp[r] = 0.02 if r % 5 == 0 else 0.0
    return wl.Workload("grid_f32", wl.DT_F32, l, T, k, tp, mp, np.zeros(B, np.uint8), 2048, 17, step)


@pytest.mark.parametrize("step", [0, 1])
def test_tied_float_rows_without_capture(step):
    _both_routes(lambda salt: _grid_rows(salt, step=step), 96)


def _wide_rows(salt, capture, B=200, V=5000):
    """Wide-class rows (packed width 4096), more rows than the GPU has CTA slots for that class (two
    waves, capturing and other rows mixed in both); float logits on a coarse grid, top_k in [1, 3000]."""
    s = np.zeros(B, np.int64) if salt is None else np.asarray(salt, np.int64)
    l = np.empty((B, V), np.float32)
    k = np.empty(B, np.int32)
    for r in range(B):
        g = np.random.default_rng([93, r, int(s[r])])
        l[r] = (np.round(g.normal(0.0, 2.0, V) * 8.0) / 8.0).astype(np.float32)
        k[r] = int(g.integers(1, 3001))
    tp = np.array([(0.8, 0.95, 1.0)[r % 3] for r in range(B)], np.float32)
    return wl.Workload("wide_f32", wl.DT_F32, l, np.ones(B, np.float32), k, tp, np.zeros(B, np.float32),
                       capture.astype(np.uint8), 4096, 29, 0)


@pytest.mark.parametrize("pattern", ["none", "all", "alternate", "last_rows", "random"])
def test_wide_rows_in_two_waves(pattern):
    B = 200
    idx = np.arange(B)
    capture = {"none": idx < 0, "all": idx >= 0, "alternate": idx % 2 == 1, "last_rows": idx >= B - 37,
               "random": np.random.default_rng(7).random(B) < 0.3}[pattern]
    w, ref, left = clear_margins(lambda salt: _wide_rows(salt, capture), B, range(B))
    assert not left, f"rows {left} kept failing the margins"
    got = gpu_run(w)
    assert compare(w, ref, got, range(B)) == B
