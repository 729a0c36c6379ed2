"""Float64 CPU oracle of one decode step of sample · filter · support capture.

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline / reference leg may import, call or execute anything in this
package. The product path (package ``top_support_capture_gb300``) never does:
it runs on the GPU or fails loudly.

The oracle is written for a reader to check against the sources by eye: one
full-row sort per row, every quantity in float64, no blocking, no fusion.

Sources (web pages; cited by title and section):
  [SGL-36630]  prhub summary of SGLang PR #36630, "sampler 原生捕获支持集，修复
               sampling mask 语义偏差" — section 实现拆解 items 2-4 (the support is
               the positive-weight set, top-k and top-p keep-sets are each taken
               on the un-renormalised distribution and intersected, ties at a
               threshold are all kept, min-p applied after), section 关键源码片段
               (test_flashinfer_joint_cutoff_ties_match_capture: the threshold
               derivation kcut = sorted[k-1], mass_before = cumsum - p,
               pcut = sorted[mass_before <= top_p][-1], keep p >= both cuts).
  [SGL-40986]  "[Sampling] Stream sampling masks as per-request arrays" —
               sections Motivation and Contract (selected vs support mode; the
               support's ids, their logprobs and the length per row), Checks
               removed item 1 (packed per-row arrays, OK/OVERFLOW status against
               the packed width), Correctness (each selected logprob equals the
               sampled token's support logprob).
  [vLLM-mask]  "vLLM Sampling Mask（Distribution Replay）深入解析" — sections
               前置要求与参数约束 (temperature must be > 0) and 工作原理 Step 1/2
               (temperature, then min-p, then top-k/top-p; survivors are the
               finite processed logits).
  [Gaudi]      "topk-subset-sampler" — section The fix (draw with the stock
               exponential race, probs / Exp(1), argmax).

Readings taken where the pages are silent:
  * Ties are equal input logit values (after exact widening to f64).
  * The top-p rule keeps a tie group when the mass strictly above it is
    <= top_p (the tie test's own comparison), measured on the full softmax.
  * min-p keeps z - z_max >= ln(min_p); it is an intersection, so its place in
    the order does not matter.
  * top_k <= 0 or >= V disables top-k; top_p >= 1 disables top-p; min_p = 0
    disables min-p. T must be finite and > 0; top_p must not be NaN or < 0;
    min_p must lie in [0, 1]; logits must not be NaN or +inf; a row needs at
    least one finite logit. A row that breaks any of these is BADPARAM.
  * Race noise: Philox4x32-10 keyed on the seed, counter (token, row, step);
    E = -ln u; token = argmax over S of z - ln E, ties to the lowest id.
  * Canonical support order is (logit descending, id ascending); ``lengths``
    is the true |S|; status OVERFLOW when |S| > packed_width.
"""
from __future__ import annotations

import dataclasses
from typing import Iterable, Optional

import numpy as np

from .philox import race_uniform

DT_BF16 = 0
DT_F32 = 1

ROW_OK = 0
ROW_OVERFLOW = 1
ROW_BADPARAM = -1


def widen_logits(logits: np.ndarray, dtype: int) -> np.ndarray:
    """Exact float64 values of the input logits (bf16 bit patterns or float32)."""
    if dtype == DT_BF16:
        bits = np.asarray(logits, dtype=np.uint16)
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == DT_F32:
        return np.asarray(logits, dtype=np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype}")


@dataclasses.dataclass
class RowResult:
    status: int
    token: int
    support: np.ndarray  # int64 ids of S in canonical order (all of S, not truncated)
    support_logprobs: np.ndarray  # float64, aligned with ``support``
    selected_logprob: float
    margin_top_p: float
    margin_min_p: float
    margin_race: float


def _bad_row() -> RowResult:
    return RowResult(ROW_BADPARAM, -1, np.zeros(0, np.int64), np.zeros(0), float("nan"),
                     float("inf"), float("inf"), float("inf"))


def row_params_ok(T: float, top_p: float, min_p: float) -> bool:
    """Per-row parameter domain ([vLLM-mask] 前置要求与参数约束: temperature > 0)."""
    T, top_p, min_p = float(T), float(top_p), float(min_p)
    if not (np.isfinite(T) and T > 0.0):
        return False
    if np.isnan(top_p) or top_p < 0.0:
        return False
    if np.isnan(min_p) or min_p < 0.0 or min_p > 1.0:
        return False
    return True


def greedy_row(l: np.ndarray) -> RowResult:
    """A greedy row ("[Sampling] Stream sampling masks as per-request arrays", Checks removed item 1: the
    greedy producer's packed ids have width 1 and length 1): the token is the largest logit's lowest id,
    the support is that token alone, its log-probability over the support is 0."""
    if np.any(np.isnan(l)) or np.any(l == np.inf):
        return _bad_row()
    F = np.flatnonzero(np.isfinite(l))
    if F.size == 0:
        return _bad_row()
    token = int(F[l[F] == l[F].max()].min())
    return RowResult(ROW_OK, token, np.array([token], np.int64), np.zeros(1), 0.0,
                     float("inf"), float("inf"), float("inf"))


def sample_row(l: np.ndarray, T: float, top_k: int, top_p: float, min_p: float,
               seed: int, step: int, row: int, greedy_t0: bool = False, positional: bool = False,
               min_p_first: bool = False) -> RowResult:
    """The whole method for one row of float64 logits ``l`` (length V). With ``greedy_t0``, a row whose
    temperature is exactly 0 is a greedy row (see greedy_row) instead of a bad one. With ``positional``,
    top-k and top-p truncate the canonical order by position, as the PyTorch producer of the SGLang
    summary does (prhub summary of SGLang PR #36630, 实现拆解 item 5: the PyTorch path is rebuilt by
    positional truncation): K = the first k positions, P = the positions whose own exclusive
    cumulative mass is <= top_p, so a tie group can be cut; min-p stays a threshold on the value.
    With ``min_p_first``, the filters run in the order of the vLLM sampler ("vLLM Sampling Mask
    (Distribution Replay) 深入解析", 工作原理 Step 1: temperature, then min-p, then top-k/top-p, each
    writing -inf over what it drops): top-p measures its masses on the distribution renormalised over
    the min-p survivors M; top-k and top-p stay one joint step (the page treats them as one filter)."""
    V = l.shape[0]
    if greedy_t0 and float(T) == 0.0:
        return greedy_row(l)
    if not row_params_ok(T, top_p, min_p):
        return _bad_row()
    if np.any(np.isnan(l)) or np.any(l == np.inf):
        return _bad_row()
    # F: tokens with a finite logit; -inf never survives ([vLLM-mask] Step 2: keep = finite).
    F = np.flatnonzero(np.isfinite(l))
    if F.size == 0:
        return _bad_row()
    T = float(T)

    # Temperature, then the full-vocabulary softmax ([SGL-36630] 实现拆解 3: both
    # keep-sets are measured on the un-renormalised probabilities).
    z = np.full(V, -np.inf)
    z[F] = l[F] / T
    z_max = z[F].max()
    w = np.zeros(V)
    w[F] = np.exp(z[F] - z_max)
    p = w / w[F].sum()

    # One full-row sort: logit descending, id ascending.
    order = F[np.lexsort((F, -l[F]))]
    ls = l[order]
    ps = p[order]
    n = order.size

    # Start of each element's tie group in the sorted order.
    new_group = np.ones(n, dtype=bool)
    new_group[1:] = ls[1:] != ls[:-1]
    group_start = np.maximum.accumulate(np.where(new_group, np.arange(n), 0))

    # K: every token whose logit is >= the k-th largest logit, so ties at the
    # cut are all kept and |K| may exceed k ([SGL-36630] tie test: kcut = sorted[k-1]).
    k = int(top_k)
    if 1 <= k < n:
        in_K = (np.arange(n) < k) if positional else (ls >= ls[k - 1])
    else:
        in_K = np.ones(n, dtype=bool)

    # M: min-p keeps z - z_max >= ln(min_p) ([vLLM-mask] Step 1 order; an intersection).
    zs = ls / T - z_max
    mp = float(min_p)
    if mp > 0.0:
        in_M = zs >= np.log(mp)
    else:
        in_M = np.ones(n, dtype=bool)

    # P: a token is kept when the mass strictly above its logit is <= top_p
    # ([SGL-36630] tie test: mass_before = cumsum - p at the group's first member). In the min-p-first
    # order the masses are those of the min-p-processed logits' softmax: p renormalised over M.
    if min_p_first and mp > 0.0:
        ps = np.where(in_M, ps, 0.0)
        ps = ps / ps.sum()
    mass_before = np.cumsum(ps) - ps
    mass_above = mass_before[group_start]
    tp = float(top_p)
    if tp < 1.0:
        in_P = (mass_before <= tp) if positional else (mass_above <= tp)
    else:
        in_P = np.ones(n, dtype=bool)

    in_S = in_K & in_P & in_M
    # Each predicate holds on a prefix of the sorted order (upward-closed in the logit and
    # constant on a tie group, or, positionally, a prefix by construction), so S is a prefix.
    n_S = int(in_S.sum())
    assert n_S >= 1 and bool(in_S[:n_S].all()), "support must be a non-empty sorted prefix"
    S = order[:n_S]

    # Logprobs renormalised over S ([SGL-36630] 实现拆解 2: log(w[y] / sum(w))).
    wS = np.exp(zs[:n_S])
    log_ZS = np.log(wS.sum())
    lpS = zs[:n_S] - log_ZS

    # Exponential race over S ([Gaudi] The fix): argmax_i p_i / E_i = argmax_i z_i - ln E_i.
    u = race_uniform(seed, step, row, S)
    E = -np.log(u)
    score = zs[:n_S] - np.log(E)
    best = score.max()
    winners = S[score == best]
    token = int(winners.min())
    pos = int(np.flatnonzero(S == token)[0])

    # Margins: distance of each floating-point decision from its threshold. The
    # maximum group's decisions are exact in any arithmetic (mass above it is 0,
    # its z - z_max is 0), so it is left out.
    not_top = group_start > 0
    if tp < 1.0 and positional:
        sel = in_K & in_M & (np.arange(n) > 0)  # every position's own mass decides
        m_tp = float(np.abs(mass_before[sel] - tp).min()) if sel.any() else float("inf")
    elif tp < 1.0:
        sel = in_K & in_M & not_top & new_group
        m_tp = float(np.abs(mass_above[sel] - tp).min()) if sel.any() else float("inf")
    else:
        m_tp = float("inf")
    if mp > 0.0:
        # in the min-p-first order every min-p decision also moves top-p's renormaliser
        sel = not_top if (min_p_first and tp < 1.0) else (in_K & in_P & not_top)
        m_mp = float(np.abs(zs[sel] - np.log(mp)).min()) if sel.any() else float("inf")
    else:
        m_mp = float("inf")
    if n_S > 1:
        top2 = np.partition(score, n_S - 2)[n_S - 2:]
        m_race = float(top2.max() - top2.min())
    else:
        m_race = float("inf")

    return RowResult(ROW_OK, token, S.astype(np.int64), lpS, float(lpS[pos]), m_tp, m_mp, m_race)


@dataclasses.dataclass
class BatchResult:
    """Oracle outputs in the library's packed layout, plus what tests need to judge parity."""

    tokens: np.ndarray  # int32 [B]
    support_ids: np.ndarray  # int32 [B, W]; -1 beyond min(|S|, W) and on rows that do not capture
    support_logprobs: np.ndarray  # float64 [B, W]; NaN where support_ids is -1
    lengths: np.ndarray  # int32 [B]; |S| on capturing rows, 0 elsewhere
    selected_logprob: np.ndarray  # float64 [B]; NaN on rows that do not capture
    row_status: np.ndarray  # int32 [B]
    support_size: np.ndarray  # int64 [B]; |S| on every good row
    margins: np.ndarray  # float64 [B, 3]: top-p mass, min-p (z units), race score
    rows: np.ndarray  # the rows that were computed
    support_mask: Optional[np.ndarray] = None  # uint32 [B, ceil(V/32)]: S's bits on capturing OVERFLOW rows


def support_bits(support: np.ndarray, V: int) -> np.ndarray:
    """S as V bits packed into ceil(V/32) little-endian uint32 words (bit i % 32 of word i // 32)."""
    bits = np.zeros(((V + 31) // 32) * 32, np.uint8)
    bits[np.asarray(support, np.int64)] = 1
    return np.packbits(bits, bitorder="little").view(np.uint32)


def pack_results(B: int, V: int, packed_width: int, capture_rows, results: dict,
                 want_mask: bool = False) -> BatchResult:
    """Lay per-row results ({row: RowResult}) out as the library's packed outputs: the first
    min(|S|, W) members of S for capturing rows, |S| in lengths, OVERFLOW when |S| > W; rows not in
    ``results`` stay at the fill values."""
    W = int(packed_width)
    cap = np.zeros(B, np.uint8) if capture_rows is None else np.asarray(capture_rows, np.uint8)
    rows = np.asarray(sorted(results))
    out = BatchResult(
        tokens=np.full(B, -1, np.int32),
        support_ids=np.full((B, W), -1, np.int32),
        support_logprobs=np.full((B, W), np.nan),
        lengths=np.zeros(B, np.int32),
        selected_logprob=np.full(B, np.nan),
        row_status=np.zeros(B, np.int32),
        support_size=np.zeros(B, np.int64),
        margins=np.full((B, 3), np.inf),
        rows=rows,
        support_mask=np.zeros((B, (V + 31) // 32), np.uint32) if want_mask else None,
    )
    for r in rows:
        res = results[int(r)]
        out.tokens[r] = res.token
        out.row_status[r] = res.status
        out.margins[r] = (res.margin_top_p, res.margin_min_p, res.margin_race)
        if res.status == ROW_BADPARAM:
            continue
        nS = res.support.size
        out.support_size[r] = nS
        if cap[r]:
            n_out = min(nS, W)
            out.support_ids[r, :n_out] = res.support[:n_out]
            out.support_logprobs[r, :n_out] = res.support_logprobs[:n_out]
            out.lengths[r] = nS
            out.selected_logprob[r] = res.selected_logprob
            out.row_status[r] = ROW_OVERFLOW if nS > W else ROW_OK
            if want_mask and nS > W:
                out.support_mask[r] = support_bits(res.support, V)
    return out


def sample_filter_capture(logits: np.ndarray, dtype: int, temperature, top_k, top_p, min_p,
                          seed: int, step: int, capture_rows, packed_width: int,
                          rows: Optional[Iterable[int]] = None, want_mask: bool = False,
                          greedy_t0: bool = False, positional: bool = False,
                          min_p_first: bool = False) -> BatchResult:
    """Run the method on a batch. ``rows`` restricts the work to some rows (others stay at fill values).
    ``want_mask`` adds the bitmask of S for capturing rows with |S| > packed_width (the exact encoding
    of an overflowing support, "vLLM Sampling Mask（Distribution Replay）深入解析", 工作原理 Step 2)."""
    B, V = np.asarray(logits).shape
    rows = np.arange(B) if rows is None else np.asarray(sorted(set(int(r) for r in rows)))
    temperature = np.asarray(temperature, np.float32)
    top_k = np.asarray(top_k, np.int32)
    top_p = np.asarray(top_p, np.float32)
    min_p = np.asarray(min_p, np.float32)
    results = {}
    for r in rows:
        l = widen_logits(np.asarray(logits)[r], dtype)  # one row at a time: exact, and no batch-sized copy
        results[int(r)] = sample_row(l, temperature[r], int(top_k[r]), top_p[r], min_p[r], seed, step, int(r),
                                     greedy_t0, positional, min_p_first)
    return pack_results(B, V, packed_width, capture_rows, results, want_mask)
