"""GPU tests of the C ABI boundary itself: the plain sfc_sample_filter_capture called through ctypes (not
through the binding's extended call), and the header's promise that the call writes nothing it does not
define.

Every output array is filled with a sentinel and followed by a guard region of sentinels before the
call. Afterwards:
  * the guards past the end of every array are intact;
  * rows that do not capture leave support_ids, support_logprobs and selected_logprob untouched;
  * capturing rows leave the entries past min(|S|, W) untouched;
  * the support bitmask is written only for overflowing capturing rows;
and the outputs match the float64 oracle. These canaries stand in for a memory checker, which is not
available on the test machines.
"""
import ctypes

import numpy as np
import pytest

import oracle
from top_support_capture_gb300 import workloads as wl
from sfc_parity import clear_margins, compare, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GUARD = 4096
SENT_I = 0x7EADBEEF
SENT_F_BITS = 0x7FBADBAD  # float outputs: a NaN with a recognisable payload


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_support_capture_gb300 as sfc

    return sfc.load_library()


def _guarded(n, dtype):
    """n elements followed by GUARD more, all holding the sentinel bit pattern."""
    t = torch.full((n + GUARD,), SENT_I if dtype == torch.int32 else SENT_F_BITS, dtype=torch.int32, device="cuda")
    return t if dtype == torch.int32 else t.view(torch.float32)


def _p(t):
    return ctypes.c_void_p(int(t.data_ptr()))


def _run_plain(lib, w, d):
    import top_support_capture_gb300 as sfc

    B, W = w.B, w.packed_width
    outs = dict(tokens=_guarded(B, torch.int32), ids=_guarded(B * W, torch.int32), lps=_guarded(B * W, torch.float32),
                lens=_guarded(B, torch.int32), sel=_guarded(B, torch.float32), st=_guarded(B, torch.int32))
    need = sfc.workspace_size(B, w.V, W, w.dtype)
    ws = sfc.allocate_workspace(need, "cuda")
    L = d["logits"]
    rc = lib.sfc_sample_filter_capture(
        _p(L), w.dtype, B, w.V, int(L.stride(0)), _p(d["temperature"]), _p(d["top_k"]), _p(d["top_p"]),
        _p(d["min_p"]), w.seed, w.step, _p(d["capture_rows"]), W, _p(outs["tokens"]), _p(outs["ids"]), _p(outs["lps"]),
        _p(outs["lens"]), _p(outs["sel"]), _p(outs["st"]), None if ws is None else _p(ws), need,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == sfc.SFC_OK, sfc.strerror(rc)
    torch.cuda.synchronize()
    h = {k: v.view(torch.int32).cpu().numpy() for k, v in outs.items()}
    return h, need


def _check_canaries(w, h, ref):
    B, W = w.B, w.packed_width
    for k in h:
        assert (h[k][-GUARD:] == SENT_I if k in ("tokens", "ids", "lens", "st") else h[k][-GUARD:] == SENT_F_BITS).all(), k
    ids = h["ids"][: B * W].reshape(B, W)
    lps = h["lps"][: B * W].reshape(B, W)
    for r in range(B):
        if not w.capture[r]:
            assert (ids[r] == SENT_I).all(), r
            assert (lps[r] == SENT_F_BITS).all(), r
            assert h["sel"][r] == SENT_F_BITS, r
        else:
            n = min(int(ref.support_size[r]), W) if ref.row_status[r] != oracle.ROW_BADPARAM else 0
            assert (ids[r, n:] == SENT_I).all(), (r, n)
            assert (lps[r, n:] == SENT_F_BITS).all(), (r, n)


def _as_got(w, h):
    B, W = w.B, w.packed_width
    return dict(tokens=h["tokens"][:B], support_ids=h["ids"][: B * W].reshape(B, W),
                support_logprobs=h["lps"][: B * W].view(np.float32).reshape(B, W), lengths=h["lens"][:B],
                selected_logprob=h["sel"][:B].view(np.float32), row_status=h["st"][:B])


@pytest.mark.parametrize("make,B,splits", [(lambda salt: wl.config2(step=4, salt=salt), 64, False),
                                           (lambda salt: wl.config3(B=24, step=2, salt=salt), 24, True)])
def test_plain_entry_point_matches_the_oracle_and_writes_only_what_it_defines(lib, make, B, splits):
    w, ref, left = clear_margins(make, B, list(range(B)))
    assert not left
    h, need = _run_plain(lib, w, to_device(w))
    assert (need > 0) == splits  # the 24-row batch of long rows is split into slices (a workspace)
    _check_canaries(w, h, ref)
    assert compare(w, ref, _as_got(w, h), range(B)) == B


def test_support_mask_written_only_for_overflowing_rows(lib):
    """W = 20 on the 151936-token workload: top_k 1024 rows overflow, top_k 20 / 50 rows may not; the mask
    rows of the others keep their sentinel, and so does a guard after the mask."""
    import top_support_capture_gb300 as sfc

    w0 = wl.config3(B=9)
    w = wl.Workload(**{**w0.__dict__, "packed_width": 20,
                       "capture": np.array([1, 1, 1, 0, 1, 1, 0, 1, 1], np.uint8)})
    d = to_device(w)
    ref = oracle.sample_filter_capture(w.logits, w.dtype, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, w.step,
                                       w.capture, w.packed_width, want_mask=True)
    nw = (w.V + 31) // 32
    mask = torch.full((w.B * nw + GUARD,), SENT_I, dtype=torch.int32, device="cuda")
    out = sfc.allocate_outputs(w.B, w.packed_width, "cuda")
    out = out._replace(support_mask=mask[: w.B * nw].view(w.B, nw))
    sfc.sample_filter_capture_into(out, d["logits"], d["temperature"], d["top_k"], d["top_p"], d["min_p"], w.seed,
                                   w.step, d["capture_rows"], w.packed_width)
    torch.cuda.synchronize()
    m = mask.cpu().numpy()
    assert (m[-GUARD:] == SENT_I).all()
    m = m[: w.B * nw].reshape(w.B, nw).view(np.uint32)
    st = out.row_status.cpu().numpy()
    for r in range(w.B):
        if w.capture[r] and st[r] == 1:
            assert np.array_equal(m[r], ref.support_mask[r]), r
        else:
            assert (m[r] == np.uint32(SENT_I)).all(), r
