"""sample · filter · capture for one LLM decode step, GB300 (sm_103a).

Thin Python binding over the C ABI of ``libsfc.so`` (declared in ``include/sfc.h``). This module only
marshals arguments: every step of the method runs in the CUDA kernels of the library. PyTorch supplies
device memory and the current stream. There is no CPU fallback; without the built library every call
raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import NamedTuple, Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsfc.so")

SFC_BF16 = 0
SFC_F32 = 1
SFC_OK = 0
SFC_EINVAL = -1
SFC_EWORKSPACE = -2
SFC_ECUDA = -3
ROW_OK = 0
ROW_OVERFLOW = 1
ROW_BADPARAM = -1
ROW_TIMEOUT = -2
ROW_OUTSIDE = 2
FLAG_GREEDY_T0 = 1
FLAG_POSITIONAL = 2
FLAG_MIN_P_FIRST = 4
FLAG_TEST_STALL = 8
MAX_PACKED_WIDTH = 16384

MAX_SLICES = 8

EXPORTED = ("sfc_sample_filter_capture", "sfc_sample_filter_capture_ex", "sfc_workspace_size",
            "sfc_workspace_size_ex", "sfc_strerror", "sfc_replay_logprob", "sfc_pack_supports",
            "sfc_sample_filter_capture_noalloc")
STATIC_SCRATCH_BYTES = 5 * 1024 * 1024

_lib = None


class SfcError(RuntimeError):
    pass


def library_path() -> str:
    return LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load libsfc.so (built by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise SfcError(f"{LIB_PATH} is not built; run __graft_entry__.build() (needs nvcc for sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    c = ctypes
    lib.sfc_sample_filter_capture.restype = c.c_int
    lib.sfc_sample_filter_capture.argtypes = [
        c.c_void_p, c.c_int, c.c_int64, c.c_int64, c.c_int64,  # logits, dtype, B, V, row_stride
        c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p,  # temperature, top_k, top_p, min_p
        c.c_uint64, c.c_uint64, c.c_void_p, c.c_int32,  # seed, step, capture_rows, packed_width
        c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p,  # outputs
        c.c_void_p, c.c_size_t, c.c_void_p,  # workspace, workspace_bytes, stream
    ]
    lib.sfc_sample_filter_capture_ex.restype = c.c_int
    lib.sfc_sample_filter_capture_ex.argtypes = (lib.sfc_sample_filter_capture.argtypes[:19] +
                                                 # support_mask, flags, max_top_k, row_offset, slices
                                                 [c.c_void_p, c.c_uint32, c.c_int32, c.c_int64, c.c_int32] +
                                                 lib.sfc_sample_filter_capture.argtypes[19:])
    lib.sfc_workspace_size.restype = c.c_size_t
    lib.sfc_workspace_size.argtypes = [c.c_int64, c.c_int64, c.c_int32, c.c_int]
    # the call for callers that cannot allocate: no workspace arguments, a slices count before the stream
    lib.sfc_sample_filter_capture_noalloc.restype = c.c_int
    lib.sfc_sample_filter_capture_noalloc.argtypes = (lib.sfc_sample_filter_capture.argtypes[:19] +
                                                      [c.c_int32, c.c_void_p])
    lib.sfc_workspace_size_ex.restype = c.c_size_t
    lib.sfc_workspace_size_ex.argtypes = [c.c_int64, c.c_int64, c.c_int32, c.c_int, c.c_int32]
    lib.sfc_strerror.restype = c.c_char_p
    lib.sfc_strerror.argtypes = [c.c_int]
    lib.sfc_pack_supports.restype = c.c_int
    lib.sfc_pack_supports.argtypes = [
        c.c_void_p, c.c_void_p, c.c_void_p, c.c_int64, c.c_int32,  # lengths, ids, logprobs, B, W
        c.c_void_p, c.c_void_p, c.c_void_p, c.c_int64, c.c_void_p,  # offsets, ids_out, lps_out, capacity, stream
    ]
    lib.sfc_replay_logprob.restype = c.c_int
    lib.sfc_replay_logprob.argtypes = [
        c.c_void_p, c.c_int, c.c_int64, c.c_int64, c.c_int64,  # logits, dtype, B, V, row_stride
        c.c_void_p, c.c_void_p, c.c_void_p, c.c_int32, c.c_void_p,  # temperature, ids, lengths, W, tokens
        c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p,  # token_logprob, support_logprobs, row_status, stream
    ]
    _lib = lib
    return lib


def strerror(code: int) -> str:
    return load_library().sfc_strerror(int(code)).decode()


class SfcOutput(NamedTuple):
    tokens: "object"  # int32 [B]
    support_ids: "object"  # int32 [B, W]
    support_logprobs: "object"  # float32 [B, W] or None (selected mode)
    lengths: "object"  # int32 [B]
    selected_logprob: "object"  # float32 [B]
    row_status: "object"  # int32 [B]
    support_mask: "object" = None  # int32 [B, ceil(V / 32)] bit words (overflowing rows), or None


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return SFC_BF16
    if t.dtype == torch.float32:
        return SFC_F32
    raise SfcError(f"logits must be bfloat16 or float32, got {t.dtype}")


def workspace_size(B: int, V: int, packed_width: int, dtype: int, slices: int = 0) -> int:
    """Bytes of workspace a call needs (0: none). See include/sfc.h: zero-filled before first use, one
    call at a time."""
    return int(load_library().sfc_workspace_size_ex(B, V, packed_width, dtype, slices))


def allocate_workspace(nbytes: int, device):
    """A zero-filled workspace of at least ``nbytes`` bytes (uint8 CUDA tensor), or None for 0 bytes."""
    import torch

    if nbytes <= 0:
        return None
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


# Workspaces the binding supplies when the caller passes none: one per (device, stream), so that calls
# on different streams never share one. Each call leaves its workspace ready for the next.
_workspaces = {}


def _default_workspace(nbytes: int, device, stream):
    import torch

    key = (device.index, int(stream.cuda_stream))
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        if torch.cuda.is_current_stream_capturing():
            raise SfcError("a CUDA graph is being captured and no workspace of this size exists for the stream: "
                           "pass workspace= (allocate_workspace(workspace_size(...))) or call once before capture")
        ws = allocate_workspace(nbytes, device)
        _workspaces[key] = ws
    return ws


def _check_tensor(name, t, device, dtype, numel=None, shape=None):
    """Reject what the kernels would misread: a tensor on another device or the host, of another dtype,
    not contiguous, or smaller than the call reads or writes."""
    if t is None:
        return
    if t.device != device:
        raise SfcError(f"{name} must be on {device}, got {t.device}")
    if t.dtype != dtype:
        raise SfcError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise SfcError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise SfcError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if numel is not None and t.numel() < numel:
        raise SfcError(f"{name} must hold at least {numel} elements, got {t.numel()}")


def allocate_outputs(B: int, packed_width: int, device, capture: bool = True, support_logprobs: bool = True,
                     mask_V: int = 0):
    """Output tensors for one call (uninitialised: the kernels write every entry they define).
    ``mask_V`` > 0 adds the support-mask words of a V-token vocabulary."""
    import torch

    i32, f32 = torch.int32, torch.float32
    return SfcOutput(
        tokens=torch.empty(B, dtype=i32, device=device),
        support_ids=torch.empty((B, packed_width), dtype=i32, device=device) if capture else None,
        support_logprobs=torch.empty((B, packed_width), dtype=f32, device=device) if (capture and support_logprobs) else None,
        lengths=torch.empty(B, dtype=i32, device=device),
        selected_logprob=torch.empty(B, dtype=f32, device=device) if capture else None,
        row_status=torch.empty(B, dtype=i32, device=device),
        support_mask=torch.empty((B, (mask_V + 31) // 32), dtype=i32, device=device) if (capture and mask_V > 0) else None,
    )


def check_call_tensors(out: SfcOutput, logits, temperature, top_k, top_p, min_p, capture_rows,
                       packed_width: int) -> None:
    """The host-side checks of one call's tensors: logits on a CUDA device, then check_call_layout."""
    if not logits.is_cuda:
        raise SfcError(f"logits must be a CUDA tensor, got {logits.device}")
    check_call_layout(out, logits, temperature, top_k, top_p, min_p, capture_rows, packed_width)


def check_call_layout(out: SfcOutput, logits, temperature, top_k, top_p, min_p, capture_rows,
                      packed_width: int) -> None:
    """Every tensor on the logits' device, with the dtype, contiguity and size the kernels assume."""
    import torch

    if logits.dim() != 2:
        raise SfcError("logits must be a [B, V] tensor")
    B, V = int(logits.shape[0]), int(logits.shape[1])
    dev = logits.device
    if logits.stride(1) != 1:
        raise SfcError("logits rows must be contiguous")
    _dtype_code(logits)
    i32, f32, u8 = torch.int32, torch.float32, torch.uint8
    for name, t, dt in (("temperature", temperature, f32), ("top_k", top_k, i32), ("top_p", top_p, f32),
                        ("min_p", min_p, f32)):
        if t is None:
            raise SfcError(f"{name} is required")
        _check_tensor(name, t, dev, dt, numel=B)
    _check_tensor("capture_rows", capture_rows, dev, u8, numel=B)
    W = int(packed_width)
    if capture_rows is not None and (out.support_ids is None or out.lengths is None or out.selected_logprob is None):
        raise SfcError("capturing rows need support_ids, lengths and selected_logprob outputs")
    _check_tensor("out.tokens", out.tokens, dev, i32, numel=B)
    _check_tensor("out.row_status", out.row_status, dev, i32, numel=B)
    _check_tensor("out.lengths", out.lengths, dev, i32, numel=B)
    _check_tensor("out.selected_logprob", out.selected_logprob, dev, f32, numel=B)
    _check_tensor("out.support_ids", out.support_ids, dev, i32, shape=(B, W))
    _check_tensor("out.support_logprobs", out.support_logprobs, dev, f32, shape=(B, W))
    if out.support_mask is not None:
        _check_tensor("out.support_mask", out.support_mask, dev, out.support_mask.dtype, shape=(B, (V + 31) // 32))
        if out.support_mask.element_size() != 4:
            raise SfcError("out.support_mask must have 32-bit elements")


def sample_filter_capture_into(out: SfcOutput, logits, temperature, top_k, top_p, min_p, seed: int, step: int,
                               capture_rows=None, packed_width: int = 1024, stream=None, workspace=None,
                               greedy_t0: bool = False, max_top_k: int = 0, positional: bool = False,
                               min_p_first: bool = False, row_offset: int = 0, slices: int = 0,
                               test_stall: bool = False) -> None:
    """Enqueue one call writing into preallocated ``out`` (all CUDA tensors, contiguous). ``workspace``
    (a zero-filled uint8 CUDA tensor of ``workspace_size(...)`` bytes, used by one call at a time) may be
    omitted: the binding then keeps one per device and stream."""
    import torch

    lib = load_library()
    check_call_tensors(out, logits, temperature, top_k, top_p, min_p, capture_rows, packed_width)
    B, V = int(logits.shape[0]), int(logits.shape[1])
    dt = _dtype_code(logits)
    if stream is None:
        stream = torch.cuda.current_stream(logits.device)
    need = workspace_size(B, V, packed_width, dt, slices)
    if workspace is None and need > 0:
        workspace = _default_workspace(need, logits.device, stream)
    if workspace is not None:
        _check_tensor("workspace", workspace, logits.device, workspace.dtype)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with torch.cuda.device(logits.device):
        rc = _call(lib, logits, dt, B, V, temperature, top_k, top_p, min_p, seed, step, capture_rows, packed_width,
                   out, workspace, ws_bytes, stream,
                   (FLAG_GREEDY_T0 if greedy_t0 else 0) | (FLAG_POSITIONAL if positional else 0)
                   | (FLAG_MIN_P_FIRST if min_p_first else 0) | (FLAG_TEST_STALL if test_stall else 0), max_top_k,
                   row_offset, slices)
    if rc != SFC_OK:
        raise SfcError(f"sfc_sample_filter_capture: {strerror(rc)} ({rc})")


def _call(lib, logits, dt, B, V, temperature, top_k, top_p, min_p, seed, step, capture_rows, packed_width, out,
          workspace, ws_bytes, stream, flags=0, max_top_k=0, row_offset=0, slices=0) -> int:
    return lib.sfc_sample_filter_capture_ex(
        _ptr(logits), dt, B, V, int(logits.stride(0)),
        _ptr(temperature), _ptr(top_k), _ptr(top_p), _ptr(min_p),
        int(seed) & 0xFFFFFFFFFFFFFFFF, int(step) & 0xFFFFFFFFFFFFFFFF, _ptr(capture_rows), int(packed_width),
        _ptr(out.tokens), _ptr(out.support_ids), _ptr(out.support_logprobs), _ptr(out.lengths),
        _ptr(out.selected_logprob), _ptr(out.row_status), _ptr(out.support_mask), int(flags), int(max_top_k), int(row_offset),
        int(slices), _ptr(workspace), ws_bytes, int(stream.cuda_stream))


def sample_filter_capture(logits, temperature, top_k, top_p, min_p, seed: int, step: int, capture_rows=None,
                          packed_width: int = 1024, support_logprobs: bool = True,
                          support_mask: bool = False, greedy_t0: bool = False, max_top_k: int = 0,
                          positional: bool = False, min_p_first: bool = False, row_offset: int = 0,
                          slices: int = 0) -> SfcOutput:
    """One decode step on CUDA tensors: ``logits`` [B, V] bf16/f32; per-row ``temperature`` f32,
    ``top_k`` int32, ``top_p`` f32, ``min_p`` f32; ``capture_rows`` uint8 [B] or None;
    ``support_mask`` adds the bitmask of overflowing rows' supports; ``max_top_k`` (the largest top_k,
    if known) lets a short batch stream each row with a cluster of CTAs; ``positional`` makes top-k and
    top-p truncate by position (the PyTorch producer's reading) instead of keeping threshold ties;
    ``min_p_first`` applies min-p before top-k/top-p (the vLLM sampler's order: top-p then measures masses
    renormalised over the min-p survivors); ``row_offset`` is the global index of the first row when a batch
    is sharded over calls (the race's noise is keyed on it); ``slices`` (0: the library's choice) sets how
    many CTAs stream each row.
    Returns freshly allocated outputs (see include/sfc.h for their meaning)."""
    B = int(logits.shape[0])
    capture = capture_rows is not None
    out = allocate_outputs(B, packed_width, logits.device, capture, support_logprobs,
                           int(logits.shape[1]) if support_mask else 0)
    sample_filter_capture_into(out, logits, temperature, top_k, top_p, min_p, seed, step, capture_rows,
                               packed_width, greedy_t0=greedy_t0, max_top_k=max_top_k, positional=positional,
                               min_p_first=min_p_first, row_offset=row_offset, slices=slices)
    return out


class ReplayOutput(NamedTuple):
    token_logprob: "object"  # float32 [B]
    support_logprobs: "object"  # float32 [B, W] or None
    row_status: "object"  # int32 [B]


def replay_logprob(logits, temperature, support_ids, lengths, tokens, support_logprobs: bool = False,
                   stream=None) -> ReplayOutput:
    """The sampled tokens' log-probabilities under ``logits`` [B, V] (bf16/f32 CUDA) renormalised over
    captured supports ``support_ids`` [B, W] int32 with ``lengths`` [B] int32 (see include/sfc.h)."""
    import torch

    lib = load_library()
    if logits.dim() != 2 or not logits.is_cuda or logits.stride(1) != 1:
        raise SfcError("logits must be a CUDA [B, V] tensor with contiguous rows")
    B, V = int(logits.shape[0]), int(logits.shape[1])
    dev = logits.device
    if support_ids.dim() != 2 or int(support_ids.shape[0]) != B:
        raise SfcError("support_ids must be [B, W]")
    W = int(support_ids.shape[1])
    _check_tensor("support_ids", support_ids, dev, torch.int32, shape=(B, W))
    _check_tensor("temperature", temperature, dev, torch.float32, numel=B)
    _check_tensor("lengths", lengths, dev, torch.int32, numel=B)
    _check_tensor("tokens", tokens, dev, torch.int32, numel=B)
    out = ReplayOutput(torch.empty(B, dtype=torch.float32, device=dev),
                       torch.empty(B, W, dtype=torch.float32, device=dev) if support_logprobs else None,
                       torch.empty(B, dtype=torch.int32, device=dev))
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        rc = lib.sfc_replay_logprob(_ptr(logits), _dtype_code(logits), B, V, int(logits.stride(0)),
                                    _ptr(temperature), _ptr(support_ids), _ptr(lengths), W, _ptr(tokens),
                                    _ptr(out.token_logprob), _ptr(out.support_logprobs), _ptr(out.row_status),
                                    int(stream.cuda_stream))
    if rc != SFC_OK:
        raise SfcError(f"sfc_replay_logprob: {strerror(rc)} ({rc})")
    return out


def pack_supports_into(lengths, support_ids, support_logprobs, offsets, ids_out, lps_out=None, stream=None) -> None:
    """Pack captured supports into one realized-size run (see include/sfc.h). ``offsets`` [B + 1] int64,
    ``ids_out`` / ``lps_out`` may be CUDA tensors or pinned host tensors (the device writes them directly)."""
    import torch

    lib = load_library()
    if support_ids.dim() != 2:
        raise SfcError("support_ids must be [B, W]")
    B, W = int(support_ids.shape[0]), int(support_ids.shape[1])
    dev = support_ids.device
    _check_tensor("support_ids", support_ids, dev, torch.int32, shape=(B, W))
    _check_tensor("lengths", lengths, dev, torch.int32, numel=B)
    if lps_out is not None:
        _check_tensor("support_logprobs", support_logprobs, dev, torch.float32, shape=(B, W))
    for name, t, dt, n in (("offsets", offsets, torch.int64, B + 1), ("ids_out", ids_out, torch.int32, 0),
                           ("lps_out", lps_out, torch.float32, 0)):
        if t is None:
            continue
        if t.dtype != dt or not t.is_contiguous() or t.numel() < n:
            raise SfcError(f"{name} must be a contiguous {dt} tensor of at least {n} elements")
        if not t.is_cuda and not t.is_pinned():
            raise SfcError(f"{name} must be a CUDA tensor or pinned host memory")
    if stream is None:
        stream = torch.cuda.current_stream(support_ids.device)
    # entries past the smaller of the two outputs are not written
    cap = int(ids_out.numel()) if lps_out is None else min(int(ids_out.numel()), int(lps_out.numel()))
    with torch.cuda.device(support_ids.device):
        rc = lib.sfc_pack_supports(_ptr(lengths), _ptr(support_ids), _ptr(support_logprobs) if lps_out is not None else None,
                                   B, W, _ptr(offsets), _ptr(ids_out), _ptr(lps_out), cap, int(stream.cuda_stream))
    if rc != SFC_OK:
        raise SfcError(f"sfc_pack_supports: {strerror(rc)} ({rc})")
