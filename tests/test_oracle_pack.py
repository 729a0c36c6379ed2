"""Pins of the reference packing: offsets are the running sums of min(|S|, W), the packed run is the rows'
first entries back to back, and unpacking gives back every row's captured prefix."""
import numpy as np

import oracle


def test_pack_round_trip_and_offsets():
    rng = np.random.default_rng(8)
    B, W = 9, 16
    lengths = np.array([0, 3, 16, 40, 1, 0, 7, 16, 2], np.int32)  # 40 > W: an overflowing row
    ids = rng.integers(0, 1000, size=(B, W)).astype(np.int32)
    lps = rng.standard_normal((B, W)).astype(np.float32)
    off, pid, plp = oracle.pack_supports(lengths, ids, lps, W)
    n = np.minimum(lengths, W)
    assert off[0] == 0 and off[-1] == n.sum() and (np.diff(off) == n).all()
    assert pid.size == plp.size == n.sum()
    for r in range(B):
        np.testing.assert_array_equal(pid[off[r]:off[r + 1]], ids[r, :n[r]])
        np.testing.assert_array_equal(plp[off[r]:off[r + 1]], lps[r, :n[r]])


def test_pack_of_a_capture():
    """Packing the capture oracle's outputs keeps exactly the realized entries (no -1 fill)."""
    from top_support_capture_gb300 import workloads as wl

    w = wl.config2()
    cap = oracle.sample_filter_capture(w.logits, w.dtype, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, w.step,
                                       w.capture, w.packed_width)
    off, pid, _ = oracle.pack_supports(cap.lengths, cap.support_ids, None, w.packed_width)
    assert (pid >= 0).all()
    assert off[-1] == np.minimum(cap.lengths, w.packed_width).sum()
