"""GPU check of sharded batches (row_offset): the race's counter takes the row's global index, so a batch
cut into several calls, each passing the index of its first row, reproduces one call over the whole
batch bit for bit, and matches the oracle run on the whole batch."""
import numpy as np
import pytest

import oracle
from top_support_capture_gb300 import workloads as wl
from sfc_parity import clear_margins, compare, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_support_capture_gb300 as sfc

    sfc.load_library()


def _call(d, w, r0, r1, row_offset, **kw):
    import top_support_capture_gb300 as sfc

    out = sfc.sample_filter_capture(d["logits"][r0:r1], d["temperature"][r0:r1], d["top_k"][r0:r1], d["top_p"][r0:r1],
                                    d["min_p"][r0:r1], w.seed, w.step, d["capture_rows"][r0:r1], w.packed_width,
                                    row_offset=row_offset, **kw)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in out._asdict().items()}


@pytest.mark.parametrize("make,cuts", [(lambda salt: wl.config2(salt=salt), [0, 16, 40, 41, 64]),
                                       (lambda salt: wl.config3(B=24, salt=salt), [0, 8, 24])])
def test_shards_reproduce_the_whole_batch(make, cuts):
    B = cuts[-1]
    w, ref, left = clear_margins(make, B, list(range(B)))
    assert not left
    d = to_device(w)
    whole = _call(d, w, 0, B, 0)
    compare(w, ref, whole, range(B))
    parts = [_call(d, w, a, b, a) for a, b in zip(cuts[:-1], cuts[1:])]
    for key in ("tokens", "lengths", "row_status", "support_ids", "support_logprobs", "selected_logprob"):
        joined = np.concatenate([p[key] for p in parts])
        valid = whole["lengths"] if key == "support_ids" or key == "support_logprobs" else None
        if key == "selected_logprob":  # written on capturing rows only
            cap = w.capture.astype(bool)
            assert np.array_equal(joined[cap], whole[key][cap]), key
        elif valid is None:
            assert np.array_equal(joined, whole[key]), key
        else:
            for r in range(B):
                n = min(int(valid[r]), w.packed_width)
                assert np.array_equal(joined[r, :n], whole[key][r, :n]), (key, r)


def test_offset_changes_the_draw_and_matches_the_oracle():
    """A large offset (near the top of the 32-bit row word) keys the race on the global row: the oracle,
    given the same global rows, draws the same tokens."""
    w0 = wl.config2()
    B = 16
    w = wl.Workload(**{**w0.__dict__, "logits": np.ascontiguousarray(w0.logits[:B]),
                       "temperature": w0.temperature[:B].copy(), "top_k": w0.top_k[:B].copy(),
                       "top_p": w0.top_p[:B].copy(), "min_p": w0.min_p[:B].copy(), "capture": np.ones(B, np.uint8)})
    off = (1 << 32) - B
    d = to_device(w)
    got = _call(d, w, 0, B, off)
    L = oracle.widen_logits(w.logits, w.dtype)
    n_ok = 0
    for r in range(B):
        res = oracle.sample_row(L[r], w.temperature[r], int(w.top_k[r]), w.top_p[r], w.min_p[r], w.seed, w.step, off + r)
        if min(res.margin_top_p, res.margin_min_p) < 1e-5 or res.margin_race < 1e-4:
            continue
        assert got["tokens"][r] == res.token, r
        assert got["lengths"][r] == res.support.size, r
        n_ok += 1
    assert n_ok >= 12
    base = _call(d, w, 0, B, 0)
    assert not np.array_equal(base["tokens"], got["tokens"])  # the offset reaches the noise
