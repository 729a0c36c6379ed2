"""Pins of the replay oracle (CPU): closed forms, the worked tie example, invariances, the page's own
masked log-softmax written over the whole vocabulary, and agreement with the capture oracle."""
import json
import math
import os

import numpy as np

import oracle
from top_support_capture_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _masked_log_softmax(l, T, ids, token):
    """The page's procedure ("RL 训练侧使用"): every token outside the support set to -inf, then
    log-softmax over the whole vocabulary, read at the sampled token."""
    z = np.asarray(l, np.float64) / T
    masked = np.full(z.shape, -np.inf)
    masked[ids] = z[ids]
    m = masked.max()
    return masked[token] - (m + math.log(np.exp(masked - m).sum()))


def test_worked_tie_example():
    g = json.load(open(os.path.join(GOLDEN, "worked_example_ties.json")))
    l = np.repeat(np.log(np.asarray(g["probs"], np.float32)).astype(np.float32)[None, :], 3, axis=0)
    S = np.asarray(g["expected_support"], np.int32)
    ids = np.full((3, 4), -1, np.int32)
    ids[:, :3] = S
    res = oracle.replay_logprob(l, oracle.DT_F32, [1.0] * 3, ids, [3, 3, 3], 4, S)
    np.testing.assert_allclose(res.token_logprob, [math.log(0.5), math.log(0.25), math.log(0.25)], atol=1e-12)
    assert (res.row_status == oracle.ROW_OK).all()


def test_uniform_support_closed_form():
    for n in (1, 2, 7, 100):
        l = np.full((1, 500), 0.75, np.float32)
        ids = np.full((1, 128), -1, np.int32)
        ids[0, :n] = np.arange(0, 3 * n, 3)
        res = oracle.replay_logprob(l, oracle.DT_F32, [1.3], ids, [n], 128, [3 * (n - 1)])
        assert math.isclose(res.token_logprob[0], -math.log(n), abs_tol=1e-12)
        np.testing.assert_allclose(res.support_logprobs[0, :n], -math.log(n), atol=1e-12)


def test_shift_and_temperature_invariance():
    rng = np.random.default_rng(3)
    l = rng.standard_normal((1, 2000)).astype(np.float32)
    ids = np.full((1, 64), -1, np.int32)
    ids[0, :50] = rng.choice(2000, 50, replace=False)
    tok = [int(ids[0, 17])]
    a = oracle.replay_logprob(l, oracle.DT_F32, [2.0], ids, [50], 64, tok)
    b = oracle.replay_logprob((l + np.float32(5.0)).astype(np.float32), oracle.DT_F32, [2.0], ids, [50], 64, tok)
    c = oracle.replay_logprob((l / np.float32(2.0)).astype(np.float32), oracle.DT_F32, [1.0], ids, [50], 64, tok)
    assert abs(a.token_logprob[0] - b.token_logprob[0]) < 1e-6  # f32 rounding of l + 5
    assert abs(a.token_logprob[0] - c.token_logprob[0]) < 1e-12  # l / 2 is exact in f32


def test_matches_the_masked_log_softmax_over_the_vocabulary():
    rng = np.random.default_rng(4)
    for trial in range(40):
        V = int(rng.integers(1, 300))
        n = int(rng.integers(1, V + 1))
        l = (rng.standard_normal(V) * 3).astype(np.float32)
        T = float(np.float32(rng.uniform(0.3, 2.0)))  # the oracle takes temperatures as float32
        S = rng.choice(V, n, replace=False)
        tok = int(S[rng.integers(n)])
        ids = np.full((1, V), -1, np.int32)
        ids[0, :n] = S
        res = oracle.replay_logprob(l[None], oracle.DT_F32, [T], ids, [n], V, [tok])
        assert abs(res.token_logprob[0] - _masked_log_softmax(l, T, S, tok)) < 1e-12
        for j in range(n):
            assert abs(res.support_logprobs[0, j] - _masked_log_softmax(l, T, S, int(S[j]))) < 1e-12


def test_replay_of_the_capture_reproduces_its_logprobs():
    """Replaying the capture's own support with the rollout's logits gives back the capture's
    selected and support log-probabilities (the capture sorts the full row; the replay only gathers)."""
    w = wl.config2()
    cap = oracle.sample_filter_capture(w.logits, w.dtype, w.temperature, w.top_k, w.top_p, w.min_p, w.seed,
                                       w.step, np.ones(w.B, np.uint8), w.packed_width)
    rep = oracle.replay_logprob(w.logits, w.dtype, w.temperature, cap.support_ids, cap.lengths,
                                w.packed_width, cap.tokens)
    for r in range(w.B):
        n = int(cap.lengths[r])
        if n > w.packed_width:
            assert rep.row_status[r] == oracle.ROW_OVERFLOW
            continue
        assert rep.row_status[r] == oracle.ROW_OK
        assert abs(rep.token_logprob[r] - cap.selected_logprob[r]) < 1e-12
        np.testing.assert_allclose(rep.support_logprobs[r, :n], cap.support_logprobs[r, :n], atol=1e-12)


def test_statuses():
    l = np.zeros((6, 10), np.float32)
    l[4, 2] = np.nan
    ids = np.array([[0, 1, 2, -1]] * 6, np.int32)
    ids[3] = [0, 1, 1, -1]  # a repeated id
    ids[5] = [0, 1, 10, -1]  # an id outside the vocabulary
    res = oracle.replay_logprob(l, oracle.DT_F32, [1.0, 0.0, 1.0, 1.0, 1.0, 1.0], ids, [3, 3, 5, 3, 3, 3], 4,
                                [7, 0, 0, 0, 0, 0])
    assert res.row_status[0] == oracle.ROW_OUTSIDE and res.token_logprob[0] == -np.inf
    np.testing.assert_allclose(res.support_logprobs[0, :3], -math.log(3), atol=1e-12)
    assert res.row_status[1] == oracle.ROW_BADPARAM  # T = 0
    assert res.row_status[2] == oracle.ROW_OVERFLOW  # length 5 > W = 4
    assert res.row_status[3] == oracle.ROW_BADPARAM
    assert res.row_status[4] == oracle.ROW_BADPARAM  # a NaN logit in the support
    assert res.row_status[5] == oracle.ROW_BADPARAM
