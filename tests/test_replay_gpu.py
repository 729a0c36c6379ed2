"""GPU parity of the training-side replay (through the C ABI) against the float64 replay oracle."""
import numpy as np
import pytest

import oracle
from top_support_capture_gb300 import workloads as wl
from sfc_parity import gpu_run, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-5


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_support_capture_gb300 as sfc

    sfc.load_library()


def _dev_logits(logits, dtype):
    if dtype == wl.DT_BF16:
        return torch.from_numpy(np.ascontiguousarray(logits).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(logits)).cuda()


def _replay(logits, dtype, T, ids, lengths, tokens, support_logprobs=True):
    import top_support_capture_gb300 as sfc

    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dt)).cuda()
    out = sfc.replay_logprob(_dev_logits(logits, dtype), t(T, np.float32), t(ids, np.int32), t(lengths, np.int32),
                             t(tokens, np.int32), support_logprobs=support_logprobs)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in out._asdict().items()}


def _compare(ref, got, ids, lengths):
    np.testing.assert_array_equal(got["row_status"], ref.row_status)
    for r in range(ref.row_status.size):
        st = ref.row_status[r]
        if st in (oracle.ROW_OK, oracle.ROW_OUTSIDE):
            if st == oracle.ROW_OK:
                assert abs(got["token_logprob"][r] - ref.token_logprob[r]) <= TOL, r
            else:
                assert got["token_logprob"][r] == -np.inf, r
            n = int(lengths[r])
            if got["support_logprobs"] is not None:
                np.testing.assert_allclose(got["support_logprobs"][r, :n], ref.support_logprobs[r, :n], atol=TOL,
                                           rtol=0)
        else:
            assert np.isnan(got["token_logprob"][r]), r


@pytest.mark.parametrize("make", [lambda: wl.config2(), lambda: wl.config3(B=24)])
def test_replay_of_the_gpu_capture(make):
    """The capture's own supports and tokens, replayed under the same logits and under perturbed ones."""
    w = make()
    got = gpu_run(w, capture=True)
    ids, lens, toks = got["support_ids"], got["lengths"], got["tokens"]
    cap = w.capture.astype(bool) & (got["row_status"] >= 0)
    ids = np.where(cap[:, None], ids, -1).astype(np.int32)
    ids[~cap, 0] = np.maximum(toks[~cap], 0)  # other rows: a one-token support
    lens = np.where(cap, lens, 1).astype(np.int32)
    ref = oracle.replay_logprob(w.logits, w.dtype, w.temperature, ids, lens, w.packed_width, toks)
    rep = _replay(w.logits, w.dtype, w.temperature, ids, lens, toks)
    _compare(ref, rep, ids, lens)
    ok = cap & (got["row_status"] == 0)
    assert ok.sum() >= 4
    # the same logits give back the capture's selected log-probability
    assert np.max(np.abs(rep["token_logprob"][ok] - got["selected_logprob"][ok])) <= TOL
    # another policy's logits on the same supports
    rng = np.random.default_rng(5)
    L = oracle.widen_logits(w.logits, w.dtype).astype(np.float32) + rng.standard_normal(w.logits.shape).astype(np.float32)
    L = wl.f32_to_bf16_bits(L) if w.dtype == wl.DT_BF16 else L
    ref2 = oracle.replay_logprob(L, w.dtype, w.temperature, ids, lens, w.packed_width, toks)
    _compare(ref2, _replay(L, w.dtype, w.temperature, ids, lens, toks), ids, lens)


@pytest.mark.parametrize("dtype", [wl.DT_BF16, wl.DT_F32])
@pytest.mark.parametrize("W", [1, 33, 1024, 16384])
def test_random_supports(dtype, W):
    rng = np.random.default_rng(W + 7 * dtype)
    B, V = 12, 50021
    l = (rng.standard_normal((B, V)) * 3).astype(np.float32)
    logits = wl.f32_to_bf16_bits(l) if dtype == wl.DT_BF16 else l
    ids = np.full((B, W), -1, np.int32)
    lens = rng.integers(1, W + 1, size=B).astype(np.int32)
    toks = np.zeros(B, np.int32)
    for r in range(B):
        ids[r, :lens[r]] = rng.choice(V, lens[r], replace=False)
        toks[r] = ids[r, rng.integers(lens[r])]
    T = rng.uniform(0.5, 1.5, size=B).astype(np.float32)
    ref = oracle.replay_logprob(logits, dtype, T, ids, lens, W, toks)
    _compare(ref, _replay(logits, dtype, T, ids, lens, toks), ids, lens)
    # selected-only mode gives the same token log-probabilities
    sel = _replay(logits, dtype, T, ids, lens, toks, support_logprobs=False)
    assert sel["support_logprobs"] is None
    np.testing.assert_array_equal(sel["row_status"], ref.row_status)


def test_statuses():
    V, W = 100, 8
    l = np.zeros((8, V), np.float32)
    l[:, :5] = [3.0, 2.0, 1.0, 0.0, -1.0]
    ids = np.tile(np.array([0, 1, 2, 3, -1, -1, -1, -1], np.int32), (8, 1))
    lens = np.array([4, 4, 9, 0, 4, 4, 4, 4], np.int32)
    toks = np.array([2, 50, 0, 0, 0, 0, 0, 1], np.int32)
    T = np.array([1, 1, 1, 1, 0, np.inf, 1, 1], np.float32)
    ids[6, 3] = V  # an id outside the vocabulary
    l[7, 1] = np.nan  # a NaN logit in the support
    ref = oracle.replay_logprob(l, wl.DT_F32, T, ids, lens, W, toks)
    assert list(ref.row_status) == [0, 2, 1, -1, -1, -1, -1, -1]
    _compare(ref, _replay(l, wl.DT_F32, T, ids, lens, toks), ids, lens)
    ninf = np.full((1, V), -np.inf, np.float32)  # no finite logit in the support
    ref = oracle.replay_logprob(ninf, wl.DT_F32, [1.0], ids[:1], [3], W, [0])
    _compare(ref, _replay(ninf, wl.DT_F32, [1.0], ids[:1], [3], [0]), ids[:1], [3])
