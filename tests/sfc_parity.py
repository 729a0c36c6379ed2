"""Parity harness: run the CUDA path (through the C ABI binding) and the float64 oracle on the same
seeded inputs and compare them element by element.

Acceptance (the method's own contract):
  * tokens, row status, lengths and support ids: bit-exact;
  * support logprobs and the selected logprob: within 2e-5 absolute;
  * the selected logprob equals the drawn token's support logprob bitwise (same capture);
on rows whose floating-point decisions clear the oracle's margins (top-p mass 1e-5, min-p 1e-5 in z
units, race score 1e-4). Rows that do not are regenerated with a new salt (only their logits change)
until they do.
"""
from __future__ import annotations

import os

import numpy as np

import oracle
from top_support_capture_gb300 import workloads as wl

LOGPROB_ATOL = 2e-5
MARGINS = (1e-5, 1e-5, 1e-4)  # top-p mass, min-p (z units), race score


def to_device(w: wl.Workload, device="cuda"):
    import torch

    if w.dtype == wl.DT_BF16:
        logits = torch.from_numpy(w.logits.view(np.int16)).to(device).view(torch.bfloat16)
    else:
        logits = torch.from_numpy(w.logits).to(device)
    return dict(
        logits=logits,
        temperature=torch.from_numpy(w.temperature).to(device),
        top_k=torch.from_numpy(w.top_k).to(device),
        top_p=torch.from_numpy(w.top_p).to(device),
        min_p=torch.from_numpy(w.min_p).to(device),
        capture_rows=torch.from_numpy(w.capture).to(device),
    )


def gpu_run(w: wl.Workload, support_logprobs: bool = True, capture: bool = True, device="cuda", dev=None, **call_kw):
    """Returns the outputs as numpy arrays (None where an output was not requested). ``call_kw`` goes to
    the binding (mode flags, the top-k hint)."""
    import torch

    import top_support_capture_gb300 as sfc

    d = dev if dev is not None else to_device(w, device)
    out = sfc.sample_filter_capture(d["logits"], d["temperature"], d["top_k"], d["top_p"], d["min_p"], w.seed,
                                    w.step, d["capture_rows"] if capture else None, w.packed_width,
                                    support_logprobs=support_logprobs, **call_kw)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in out._asdict().items()}


# ------------------------------------------------------------------------------------------------
# The oracle over many rows: a process pool (started with spawn, so that no worker inherits the
# parent's CUDA context) runs rows in parallel; each task gets one row's raw logits and parameters.
# ------------------------------------------------------------------------------------------------
_POOL = None
PARALLEL_MIN_ELEMENTS = 4_000_000  # below this many logits the oracle runs in-process


def _pool():
    global _POOL
    if _POOL is None:
        import multiprocessing

        _POOL = multiprocessing.get_context("spawn").Pool(max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def _oracle_rows_task(task):
    """One chunk of rows: (raw rows, row indices, dtype, per-row parameters, seed, step, mode) -> results."""
    raw, idx, dtype, T, k, tp, mp, seed, step, mode = task
    out = {}
    for j, r in enumerate(idx):
        out[int(r)] = oracle.sample_row(oracle.widen_logits(raw[j], dtype), T[j], int(k[j]), tp[j], mp[j], seed, step,
                                        int(r), **mode)
    return out


def oracle_results(w: wl.Workload, rows, **mode) -> dict:
    """{row: RowResult} for the given rows of the workload, in a process pool when the rows are many."""
    rows = sorted(set(int(r) for r in rows))
    chunk = max(1, len(rows) // (4 * (os.cpu_count() or 1)))
    tasks = [(np.ascontiguousarray(w.logits[idx]), idx, w.dtype, w.temperature[idx], w.top_k[idx], w.top_p[idx],
              w.min_p[idx], w.seed, w.step, mode)
             for idx in (rows[i:i + chunk] for i in range(0, len(rows), chunk))]
    out = {}
    if len(rows) * w.V < PARALLEL_MIN_ELEMENTS:
        for t in tasks:
            out.update(_oracle_rows_task(t))
    else:
        for part in _pool().map(_oracle_rows_task, tasks):
            out.update(part)
    return out


def oracle_run(w: wl.Workload, rows=None, want_mask: bool = False, **mode) -> oracle.BatchResult:
    rows = range(w.B) if rows is None else rows
    return oracle.pack_results(w.B, w.V, w.packed_width, w.capture, oracle_results(w, rows, **mode), want_mask)


def margin_fail(ref: oracle.BatchResult, rows):
    m = ref.margins
    return [int(r) for r in rows
            if ref.row_status[r] != oracle.ROW_BADPARAM
            and (m[r, 0] < MARGINS[0] or m[r, 1] < MARGINS[1] or m[r, 2] < MARGINS[2])]


def _margins_bad(results: dict, rows):
    bad = []
    for r in rows:
        x = results[r]
        if x.status != oracle.ROW_BADPARAM and (x.margin_top_p < MARGINS[0] or x.margin_min_p < MARGINS[1]
                                                 or x.margin_race < MARGINS[2]):
            bad.append(r)
    return bad


def clear_margins(make, B: int, rows, max_tries: int = 16, **mode):
    """Regenerate rows whose decisions sit within rounding distance of a threshold.

    ``make(salt=...)`` builds the workload; ``mode`` goes to the oracle (greedy_t0, positional);
    returns (workload, oracle result, rows still failing). Only regenerated rows are run again: every
    row's inputs and noise depend on that row alone."""
    rows = sorted(set(int(r) for r in rows))
    salt = np.zeros(B, dtype=np.int64)
    w = make(salt=salt)
    res = oracle_results(w, rows, **mode)
    bad = _margins_bad(res, rows)
    for _ in range(max_tries):
        if not bad:
            break
        salt[bad] += 1
        w = make(salt=salt.copy())
        res.update(oracle_results(w, bad, **mode))
        bad = _margins_bad(res, bad)
    return w, oracle.pack_results(w.B, w.V, w.packed_width, w.capture, res), bad


def compare(w: wl.Workload, ref: oracle.BatchResult, got: dict, rows, capture: bool = True,
            support_logprobs: bool = True) -> int:
    """Assert parity on ``rows``; returns the number of rows compared."""
    W = w.packed_width
    n = 0
    for r in rows:
        r = int(r)
        cap = capture and bool(w.capture[r])
        st = int(ref.row_status[r])
        if st == oracle.ROW_BADPARAM:
            assert got["row_status"][r] == -1, r
            assert got["tokens"][r] == -1, r
            if got["lengths"] is not None:
                assert got["lengths"][r] == 0, r
            if cap:
                assert np.isnan(got["selected_logprob"][r]), r
            n += 1
            continue
        assert got["tokens"][r] == ref.tokens[r], (r, got["tokens"][r], ref.tokens[r])
        if cap:
            assert got["row_status"][r] == st, (r, got["row_status"][r], st)
            assert got["lengths"][r] == ref.lengths[r], (r, got["lengths"][r], ref.lengths[r])
            k = min(int(ref.lengths[r]), W)
            gi = got["support_ids"][r, :k]
            assert np.array_equal(gi, ref.support_ids[r, :k]), (r, np.flatnonzero(gi != ref.support_ids[r, :k])[:5])
            sel = float(got["selected_logprob"][r])
            assert abs(sel - ref.selected_logprob[r]) <= LOGPROB_ATOL, (r, sel, ref.selected_logprob[r])
            if support_logprobs:
                gl = got["support_logprobs"][r, :k].astype(np.float64)
                err = np.abs(gl - ref.support_logprobs[r, :k]).max() if k else 0.0
                assert err <= LOGPROB_ATOL, (r, err)
                pos = np.flatnonzero(gi == got["tokens"][r])
                if pos.size:
                    assert got["support_logprobs"][r, pos[0]] == got["selected_logprob"][r], r
        else:
            assert got["row_status"][r] == 0, r
            if got["lengths"] is not None:
                assert got["lengths"][r] == 0, r
        n += 1
    return n
