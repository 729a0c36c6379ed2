"""GPU parity of the min-p-first order (SFC_FLAG_MIN_P_FIRST): min-p drops its tokens first, then top-k
and top-p run as one joint step on the survivors M, so top-p measures masses renormalised over M ("vLLM
Sampling Mask（Distribution Replay）深入解析", 工作原理 Step 1). Rows whose M lies inside the on-chip
pool take the on-chip finishes (M's mass from the pool); the others take the multi-pass path."""
import numpy as np
import pytest

from top_support_capture_gb300 import workloads as wl
from sfc_parity import clear_margins, compare, gpu_run, margin_fail, oracle_run

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MPF = dict(min_p_first=True)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_support_capture_gb300 as sfc

    sfc.load_library()


def _wl(logits, dtype=wl.DT_F32, T=1.0, k=50, tp=0.9, mp=0.05, cap=1, W=1024, seed=13, step=0):
    B = logits.shape[0]
    arr = lambda v, dt: np.broadcast_to(np.asarray(v, dt), (B,)).copy()
    return wl.Workload("min_p_first", dtype, logits, arr(T, np.float32), arr(k, np.int32), arr(tp, np.float32),
                       arr(mp, np.float32), arr(cap, np.uint8), W, seed, step)


def _check(w, mode=MPF, min_frac=0.75, **call_kw):
    rows = list(range(w.B))
    ref = oracle_run(w, rows, **mode)
    ok = [r for r in rows if r not in set(margin_fail(ref, rows))]
    assert len(ok) >= min_frac * len(rows), (len(ok), len(rows))
    got = gpu_run(w, **mode, **call_kw)
    compare(w, ref, got, ok)
    return ref, got, ok


def _differs_from_joint(w, ref, rows):
    joint = oracle_run(w, rows)
    return sum(int(ref.support_size[r] != joint.support_size[r]) for r in rows)


@pytest.mark.parametrize("step", [0, 3])
def test_config2_all_rows(step):
    """V = 32000 bf16, top_k up to 1024, top_p in [0.5, 1], min_p in {0, 0.05}."""
    w, ref, left = clear_margins(lambda salt: wl.config2(step=step, salt=salt), 64, list(range(64)), **MPF)
    assert not left
    compare(w, ref, gpu_run(w, **MPF), range(64))
    assert _differs_from_joint(w, ref, range(64)) >= 1


@pytest.mark.parametrize("B", [8, 64])
def test_config5_rows(B):
    """The long vocabulary (V = 262144) with top_k 50, top_p 0.95, min_p 0.05 on every row."""
    w, ref, left = clear_margins(lambda salt: wl.config5(B=B, salt=salt), B, list(range(B)), **MPF)
    assert not left
    compare(w, ref, gpu_run(w, **MPF), range(B))


@pytest.mark.parametrize("B", [1, 32])
def test_config5_split_rows(B):
    w, ref, left = clear_margins(lambda salt: wl.config5(B=B, salt=salt), B, list(range(B)), **MPF)
    assert not left
    compare(w, ref, gpu_run(w, max_top_k=50, **MPF), range(B))


def test_config1_tiny_ties():
    for V in (5, 8, 16):
        w, ref, left = clear_margins(lambda salt: wl.config1_tiny(V, salt=salt), 64, list(range(64)), **MPF)
        assert not left
        compare(w, ref, gpu_run(w, **MPF), range(64))


@pytest.mark.parametrize("dtype", [wl.DT_BF16, wl.DT_F32])
def test_inside_and_beyond_the_pool(dtype):
    """Zipf-like rows of 151936 tokens. Rows 0-3: large top_k with a tight min-p (M inside the on-chip
    pool); rows 4-7: small top_k with a loose min-p (M reaches far below the pool: multi-pass path);
    rows 8-9: top-k off."""
    V = 151936
    rng = np.random.default_rng(77)
    l = np.empty((10, V), np.float32)
    for r in range(10):
        l[r] = (-1.0 * np.log1p(rng.permutation(V)) + rng.standard_normal(V) * 0.8).astype(np.float32)
    k = np.array([1024, 700, 2000, 1024, 20, 50, 8, 30, 0, 0], np.int32)
    mp = np.array([0.2, 0.1, 0.3, 0.05, 1e-3, 5e-4, 2e-3, 1e-4, 0.05, 0.01], np.float32)
    tp = np.array([0.6, 0.8, 0.5, 0.9, 0.95, 0.7, 0.99, 0.9, 0.8, 0.9], np.float32)
    logits = wl.f32_to_bf16_bits(l) if dtype == wl.DT_BF16 else l
    w = _wl(logits, dtype, T=np.linspace(0.7, 1.3, 10).astype(np.float32), k=k, tp=tp, mp=mp, W=2048)
    ref, got, ok = _check(w, min_frac=0.7)
    assert _differs_from_joint(w, ref, ok) >= 3


def test_with_positional_and_greedy():
    """All three flags together on the small bf16 workload (a third of the rows greedy)."""
    w0 = wl.config2()
    T = w0.temperature.copy()
    T[::3] = 0.0
    w = wl.Workload(**{**w0.__dict__, "temperature": T, "capture": np.ones(w0.B, np.uint8)})
    _check(w, mode=dict(min_p_first=True, positional=True, greedy_t0=True))


def test_equals_the_masked_row_on_the_gpu():
    """The page's own route on the same GPU: setting min-p's drops to -inf (on the host) and running the
    default joint filter gives the same supports, tokens and lengths."""
    w, ref, left = clear_margins(lambda salt: wl.config2(step=1, salt=salt), 64, list(range(64)), **MPF)
    assert not left
    l = wl.bf16_bits_to_f32(w.logits).astype(np.float64)
    z = l / w.temperature[:, None].astype(np.float64)
    keep = (z - z.max(axis=1, keepdims=True)) >= np.log(np.maximum(w.min_p, 1e-30))[:, None].astype(np.float64)
    keep |= (w.min_p == 0)[:, None]
    masked = np.where(keep, l, -np.inf).astype(np.float32)
    wm = wl.Workload(**{**w.__dict__, "logits": wl.f32_to_bf16_bits(masked),
                        "min_p": np.zeros(w.B, np.float32)})
    a = gpu_run(w, **MPF)
    b = gpu_run(wm)
    jm = oracle_run(wm)
    rows = [r for r in range(w.B) if r not in set(margin_fail(jm, range(w.B)))]
    assert len(rows) >= 56
    for r in rows:
        assert a["tokens"][r] == b["tokens"][r] and a["lengths"][r] == b["lengths"][r], r
        n = min(int(a["lengths"][r]), w.packed_width)
        assert np.array_equal(a["support_ids"][r, :n], b["support_ids"][r, :n]), r
