"""Reference packing of captured supports into one realized-size run (CSR layout).

TEST INFRASTRUCTURE (see the package header): only tests/, __graft_entry__.smoke() and bench.py's
baseline legs may use it.

Source: "[Sampling] Stream sampling masks as per-request arrays" (SGLang PR #40986), section Limitations:
the device-to-host copy of the packed masks is sized by the batch's capacity, [B, W], not by the
supports actually captured; a realized-size copy moves only sum_r min(|S_r|, W) entries.

Layout read here: offsets[0] = 0, offsets[r + 1] = offsets[r] + n_r with n_r = min(max(lengths[r], 0), W);
row r's entries are ids[offsets[r] : offsets[r + 1]] = support_ids[r, :n_r] (and the same for the
log-probabilities).
"""
from __future__ import annotations

import numpy as np


def pack_supports(lengths, support_ids, support_logprobs, packed_width: int):
    W = int(packed_width)
    n = np.clip(np.asarray(lengths, np.int64), 0, W)
    offsets = np.zeros(n.size + 1, np.int64)
    offsets[1:] = np.cumsum(n)
    ids = np.concatenate([np.asarray(support_ids)[r, :n[r]] for r in range(n.size)]) if n.size else np.zeros(0)
    lps = None
    if support_logprobs is not None:
        lps = np.concatenate([np.asarray(support_logprobs)[r, :n[r]] for r in range(n.size)])
    return offsets, ids.astype(np.int32), None if lps is None else lps.astype(np.float32)
