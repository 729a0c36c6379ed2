"""GPU check of sfc_sample_filter_capture_noalloc, the decode-step call for callers that cannot allocate
device memory: code whose buffers are all planned by a framework that forbids other allocations, or that
cannot afford cudaMalloc's implicit synchronisation on its hot path. Instead of a caller's workspace it
uses a scratch array inside the library, shared by every call on the device. Its outputs must equal the
regular entry point's (with a caller-allocated workspace) on the same inputs, call after call, including
when consecutive calls split different batch sizes over that one array."""
import ctypes

import numpy as np
import pytest

from top_support_capture_gb300 import workloads as wl
from sfc_parity import LOGPROB_ATOL, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_support_capture_gb300 as sfc

    return sfc.load_library()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(int(t.data_ptr()))


def _noalloc(lib, d, w, out, slices=0):
    """One call of the no-allocation entry point through the C ABI, on torch's current stream."""
    L = d["logits"]
    return lib.sfc_sample_filter_capture_noalloc(
        _ptr(L), w.dtype, w.B, w.V, int(L.stride(0)), _ptr(d["temperature"]), _ptr(d["top_k"]), _ptr(d["top_p"]),
        _ptr(d["min_p"]), w.seed, w.step, _ptr(d["capture_rows"]), w.packed_width, _ptr(out.tokens),
        _ptr(out.support_ids), _ptr(out.support_logprobs), _ptr(out.lengths), _ptr(out.selected_logprob),
        _ptr(out.row_status), slices, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _regular(d, w):
    """The same step through the regular entry point with a workspace the caller allocated."""
    import top_support_capture_gb300 as sfc

    out = sfc.allocate_outputs(w.B, w.packed_width, "cuda")
    ws = sfc.allocate_workspace(sfc.workspace_size(w.B, w.V, w.packed_width, w.dtype), "cuda")
    sfc.sample_filter_capture_into(out, d["logits"], d["temperature"], d["top_k"], d["top_p"], d["min_p"], w.seed,
                                   w.step, d["capture_rows"], w.packed_width, workspace=ws)
    return out


def _np(out):
    return {k: (None if v is None else v.cpu().numpy()) for k, v in out._asdict().items()}


def _same(a, b, w):
    for k in ("tokens", "row_status", "lengths"):
        assert np.array_equal(a[k], b[k]), k
    cap = w.capture.astype(bool)
    assert np.abs(a["selected_logprob"][cap] - b["selected_logprob"][cap]).max() <= LOGPROB_ATOL
    for r in np.flatnonzero(cap):
        n = min(int(a["lengths"][r]), w.packed_width)
        assert np.array_equal(a["support_ids"][r, :n], b["support_ids"][r, :n]), r
        if n:
            assert np.abs(a["support_logprobs"][r, :n] - b["support_logprobs"][r, :n]).max() <= LOGPROB_ATOL, r


def test_noalloc_matches_the_workspace_call_on_consecutive_calls(lib):
    import top_support_capture_gb300 as sfc

    # 2 rows of 151936 tokens split 4 ways (tickets in bytes 0-8, slice records from byte 256), then 100 rows
    # split 3 ways, whose tickets (bytes 0-400) lie over the first call's records: wrong unless cleared;
    # then 32 rows of 262144 tokens split 8 ways
    cases = [wl.config3(B=2), wl.config3(B=100, step=1), wl.config5(B=32, step=2)]
    for w in cases:
        assert 0 < sfc.workspace_size(w.B, w.V, w.packed_width, w.dtype) <= sfc.STATIC_SCRATCH_BYTES
    devs = [to_device(w) for w in cases]
    outs = [sfc.allocate_outputs(w.B, w.packed_width, "cuda") for w in cases]
    for d, w, o in zip(devs, cases, outs):  # back to back on one stream, nothing in between
        assert _noalloc(lib, d, w, o) == sfc.SFC_OK
    torch.cuda.synchronize()
    got = [_np(o) for o in outs]
    for d, w, g in zip(devs, cases, got):
        ref = _regular(d, w)
        torch.cuda.synchronize()
        _same(g, _np(ref), w)
    # the first call repeated: the same bits
    again = sfc.allocate_outputs(cases[0].B, cases[0].packed_width, "cuda")
    assert _noalloc(lib, devs[0], cases[0], again) == sfc.SFC_OK
    torch.cuda.synchronize()
    a = _np(again)
    for k in ("tokens", "lengths", "row_status"):
        assert np.array_equal(a[k], got[0][k]), k


def test_noalloc_rejects_a_split_larger_than_its_scratch(lib):
    """300 rows of 262144 tokens forced into 8 slices need far more than the array: refused, nothing runs."""
    import types

    import top_support_capture_gb300 as sfc

    B, V, W = 300, 262144, 1024
    assert sfc.workspace_size(B, V, W, sfc.SFC_BF16, 8) > sfc.STATIC_SCRATCH_BYTES
    cuda = dict(device="cuda")
    d = dict(logits=torch.zeros((B, V), dtype=torch.bfloat16, **cuda), temperature=torch.ones(B, **cuda),
             top_k=torch.full((B,), 5, dtype=torch.int32, **cuda), top_p=torch.ones(B, **cuda),
             min_p=torch.zeros(B, **cuda), capture_rows=torch.ones(B, dtype=torch.uint8, **cuda))
    w = types.SimpleNamespace(B=B, V=V, dtype=sfc.SFC_BF16, seed=0, step=0, packed_width=W)
    out = sfc.allocate_outputs(B, W, "cuda")
    out.tokens.fill_(-7)
    assert _noalloc(lib, d, w, out, slices=8) == sfc.SFC_EWORKSPACE
    torch.cuda.synchronize()
    assert (out.tokens == -7).all()  # nothing ran
