"""Float64 CPU oracle of the training-side replay: the sampled token's log-probability under a
policy's logits renormalised over a captured support S.

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
leg may import, call or execute anything in this package. The product path never does.

Sources (web pages; cited by title and section):
  [vLLM-mask]  "vLLM Sampling Mask（Distribution Replay）深入解析" — section RL 训练侧使用: the
               current policy's log-probability on the rollout's support is the log-softmax of its
               logits with every token outside the returned support set to -inf, read at the
               sampled token; both policies are then normalised over the same token set.
  [SGL-40986]  "[Sampling] Stream sampling masks as per-request arrays" — section Contract (a
               row's support travels as its ids and its length) and Checks removed item 1 (rows
               whose support exceeds the packed width are marked OVERFLOW).

Readings taken where the pages are silent:
  * The logits are processed like the capture's: z = l / T (T = 1 is the page's raw-logit form).
  * A row whose length exceeds the packed width W carries only the first W ids of its support:
    status OVERFLOW, no log-probabilities (NaN).
  * BADPARAM: T not finite or <= 0; length < 1; an id outside [0, V); a support logit that is NaN
    or +inf; no finite logit in the support. The ids of a support are distinct (a capture writes
    them so); repeated ids are outside the contract, and the oracle rejects them as BADPARAM so that
    no test can pass them by mistake.
  * A sampled token outside the support gets the masked log-softmax's own value, -inf, and the
    status OUTSIDE; the support's log-probabilities are still written.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from .sfc_oracle import ROW_BADPARAM, ROW_OK, ROW_OVERFLOW, widen_logits

ROW_OUTSIDE = 2


@dataclasses.dataclass
class ReplayResult:
    token_logprob: np.ndarray  # float64 [B]; NaN on OVERFLOW / BADPARAM rows, -inf on OUTSIDE rows
    support_logprobs: np.ndarray  # float64 [B, W]; entries j < length on OK / OUTSIDE rows, NaN elsewhere
    row_status: np.ndarray  # int32 [B]


def replay_row(l: np.ndarray, T: float, ids: np.ndarray, n: int, W: int, token: int):
    """One row: (status, token log-probability, log-probabilities of ids[:n] or None)."""
    V = l.shape[0]
    T = float(T)
    if not (np.isfinite(T) and T > 0.0) or n < 1:
        return ROW_BADPARAM, np.nan, None
    if n > W:
        return ROW_OVERFLOW, np.nan, None
    ids = np.asarray(ids[:n], np.int64)
    if ids.min() < 0 or ids.max() >= V or np.unique(ids).size != n:
        return ROW_BADPARAM, np.nan, None
    z = l[ids] / T
    if np.isnan(z).any() or np.isposinf(z).any() or not np.isfinite(z).any():
        return ROW_BADPARAM, np.nan, None
    m = z.max()
    lse = m + np.log(np.exp(z - m).sum())  # exp(-inf) = 0: -inf members carry no mass
    lp = z - lse
    hit = np.flatnonzero(ids == int(token))
    if hit.size == 0:
        return ROW_OUTSIDE, -np.inf, lp
    return ROW_OK, float(lp[hit[0]]), lp


def replay_logprob(logits: np.ndarray, dtype: int, temperature, support_ids: np.ndarray, lengths,
                   packed_width: int, tokens) -> ReplayResult:
    L = widen_logits(logits, dtype)
    B = L.shape[0]
    W = int(packed_width)
    out = ReplayResult(np.full(B, np.nan), np.full((B, W), np.nan), np.zeros(B, np.int32))
    T = np.asarray(temperature, np.float32)
    for r in range(B):
        st, lpt, lp = replay_row(L[r], T[r], np.asarray(support_ids[r]), int(lengths[r]), W, int(tokens[r]))
        out.row_status[r] = st
        out.token_logprob[r] = lpt
        if lp is not None:
            out.support_logprobs[r, :lp.size] = lp
    return out
