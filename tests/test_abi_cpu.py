"""CPU-side checks of the C ABI library: it builds, loads, and exports what include/sfc.h declares.

No compute call is made here (there is no GPU in this environment); only the host-only helpers
sfc_strerror and sfc_workspace_size are called.
"""
import os
import re
import subprocess

import pytest

import top_support_capture_gb300 as sfc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sfc.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sfc_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(sfc.library_path()):
        from top_support_capture_gb300 import build

        build.build()
    return sfc.load_library()


def test_header_declares_the_entry_points():
    assert _declared() == sorted(sfc.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", sfc.library_path()], capture_output=True, text=True)
    if out.returncode == 0:
        exported = set(re.findall(r"\bT (sfc_[a-z_0-9]+)\b", out.stdout))
        assert set(_declared()) <= exported


def test_strerror_and_workspace(lib):
    assert sfc.strerror(sfc.SFC_OK) == "success"
    for code in (sfc.SFC_EINVAL, sfc.SFC_EWORKSPACE, sfc.SFC_ECUDA):
        assert sfc.strerror(code) and sfc.strerror(code) != "success"


def _slice_bytes(B, S, cap=2048):
    pad = lambda x: (x + 255) // 256 * 256
    return pad(4 * B) + pad(16 * B * S) + 8 * B * S * cap


def test_workspace_size_follows_the_slice_count(lib):
    """Short batches of long rows are split into slices that meet in the workspace; long batches, short
    rows and wide packed outputs are not (0 bytes)."""
    bf16, f32 = sfc.SFC_BF16, sfc.SFC_F32
    # only while every slice of every row fits the GPU's 304 CTA slots at once, each slice two 32 KB stages
    assert sfc.workspace_size(1, 262144, 1024, bf16) == _slice_bytes(1, 8)      # at most 8 slices
    assert sfc.workspace_size(32, 262144, 1024, bf16) == _slice_bytes(32, 8)    # 256 CTAs
    assert sfc.workspace_size(128, 262144, 1024, bf16) == _slice_bytes(128, 2)  # 256 CTAs
    assert sfc.workspace_size(100, 151936, 1024, bf16) == _slice_bytes(100, 3)  # 300 CTAs
    assert sfc.workspace_size(2, 151936, 1024, bf16) == _slice_bytes(2, 4)      # 18992 vectors: 4 slices
    assert sfc.workspace_size(256, 151936, 1024, bf16) == 0                     # a full wave already
    assert sfc.workspace_size(512, 262144, 1024, bf16) == 0
    assert sfc.workspace_size(64, 32000, 1024, bf16) == 0                       # rows too short to split
    assert sfc.workspace_size(256, 129280, 8192, f32) == 0                      # the wide class
    # an explicit slice count
    assert sfc.workspace_size(256, 151936, 1024, bf16, 1) == 0
    assert sfc.workspace_size(256, 151936, 1024, bf16, 2) == _slice_bytes(256, 2)
    assert sfc.workspace_size(6, 9, 64, f32, 8) == _slice_bytes(6, 2)  # 9 floats: two 16-byte vectors
    assert sfc.workspace_size(6, 3, 64, f32, 8) == 0                   # no whole vector: one CTA
    assert sfc.workspace_size(256, 151936, 1024, bf16, 9) == 0          # out of range
    assert sfc.workspace_size(0, 151936, 1024, bf16) == 0


def test_header_constants_match_binding():
    src = open(HEADER).read()
    consts = dict(re.findall(r"#define (SFC_[A-Z_0-9]+) \(?(-?\d+)\)?", src))
    assert int(consts["SFC_BF16"]) == sfc.SFC_BF16 and int(consts["SFC_F32"]) == sfc.SFC_F32
    assert int(consts["SFC_EINVAL"]) == sfc.SFC_EINVAL and int(consts["SFC_ECUDA"]) == sfc.SFC_ECUDA
    assert int(consts["SFC_ROW_OVERFLOW"]) == sfc.ROW_OVERFLOW and int(consts["SFC_ROW_BADPARAM"]) == sfc.ROW_BADPARAM
    assert int(consts["SFC_MAX_PACKED_WIDTH"]) == sfc.MAX_PACKED_WIDTH


def test_invalid_arguments_rejected_on_host(lib):
    """Argument checks run before any CUDA call, so they work without a GPU."""
    f = lib.sfc_sample_filter_capture
    fake = 0x1000  # never dereferenced: the checks reject the call first
    args = dict(logits=fake, dtype=0, B=4, V=16, stride=16, T=fake, k=fake, tp=fake, mp=fake, seed=0, step=0,
                cap=None, W=8, tok=fake, ids=fake, lps=fake, lens=fake, sel=fake, st=fake, ws=None, wsb=0, stream=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return f(a["logits"], a["dtype"], a["B"], a["V"], a["stride"], a["T"], a["k"], a["tp"], a["mp"], a["seed"],
                 a["step"], a["cap"], a["W"], a["tok"], a["ids"], a["lps"], a["lens"], a["sel"], a["st"], a["ws"],
                 a["wsb"], a["stream"])

    assert call(logits=None) == sfc.SFC_EINVAL
    assert call(dtype=7) == sfc.SFC_EINVAL
    assert call(B=0) == sfc.SFC_EINVAL
    assert call(V=0) == sfc.SFC_EINVAL
    assert call(stride=15) == sfc.SFC_EINVAL
    assert call(W=0) == sfc.SFC_EINVAL
    assert call(W=sfc.MAX_PACKED_WIDTH + 1) == sfc.SFC_EINVAL
    assert call(T=None) == sfc.SFC_EINVAL
    assert call(tok=None) == sfc.SFC_EINVAL
    assert call(cap=fake, ids=None) == sfc.SFC_EINVAL
    assert call(cap=fake, lens=None) == sfc.SFC_EINVAL
    assert call(logits=fake + 1) == sfc.SFC_EINVAL  # bf16 logits must be 2-byte aligned
    # rows split into slices need the workspace: missing, too small or unaligned
    big = dict(B=2, V=151936, stride=151936)
    need = sfc.workspace_size(2, 151936, 8, sfc.SFC_BF16)
    assert need > 0
    assert call(**big) == sfc.SFC_EWORKSPACE
    assert call(**big, ws=fake, wsb=need - 1) == sfc.SFC_EWORKSPACE
    assert call(**big, ws=fake + 8, wsb=need) == sfc.SFC_EINVAL


def test_ex_invalid_flags_and_row_offset_rejected_on_host(lib):
    """The extended call's own arguments: unknown flag bits, a negative row offset, and an offset that
    pushes the last row past the counter's 32-bit row word."""
    f = lib.sfc_sample_filter_capture_ex
    fake = 0x1000  # never dereferenced: the checks reject the call first

    def call(flags=0, row_offset=0, B=4, mask=None, cap=None, slices=0, V=16, ws=None, wsb=0):
        return f(fake, 0, B, V, V, fake, fake, fake, fake, 0, 0, cap, 8, fake, fake, fake, fake, fake, fake, mask,
                 flags, 0, row_offset, slices, ws, wsb, None)

    assert call(flags=16) == sfc.SFC_EINVAL
    assert call(flags=1 << 31) == sfc.SFC_EINVAL
    assert call(row_offset=-1) == sfc.SFC_EINVAL
    assert call(row_offset=(1 << 32) - 3, B=4) == sfc.SFC_EINVAL
    assert call(B=4, mask=fake) == sfc.SFC_EINVAL  # a support mask needs capture_rows
    assert call(slices=-1) == sfc.SFC_EINVAL
    assert call(slices=9) == sfc.SFC_EINVAL
    assert call(slices=2, V=64) == sfc.SFC_EWORKSPACE  # an explicit split of 8-vector rows needs a workspace


def test_replay_invalid_arguments_rejected_on_host(lib):
    f = lib.sfc_replay_logprob
    fake = 0x1000  # never dereferenced
    args = dict(logits=fake, dtype=1, B=4, V=16, stride=16, T=fake, ids=fake, lens=fake, W=8, tok=fake, out=fake,
                lps=None, st=fake, stream=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return f(a["logits"], a["dtype"], a["B"], a["V"], a["stride"], a["T"], a["ids"], a["lens"], a["W"],
                 a["tok"], a["out"], a["lps"], a["st"], a["stream"])

    for bad in (dict(logits=None), dict(dtype=3), dict(B=0), dict(V=0), dict(stride=8), dict(W=0),
                dict(W=sfc.MAX_PACKED_WIDTH + 1), dict(T=None), dict(ids=None), dict(lens=None), dict(tok=None),
                dict(out=None), dict(st=None), dict(logits=fake + 2)):
        assert call(**bad) == sfc.SFC_EINVAL, bad


def test_replay_status_constant_matches_binding():
    consts = dict(re.findall(r"#define (SFC_[A-Z_0-9]+) \(?(-?\d+)\)?", open(HEADER).read()))
    assert int(consts["SFC_ROW_OUTSIDE"]) == sfc.ROW_OUTSIDE
    import oracle

    assert oracle.ROW_OUTSIDE == sfc.ROW_OUTSIDE


def test_pack_invalid_arguments_rejected_on_host(lib):
    f = lib.sfc_pack_supports
    fake = 0x1000  # never dereferenced
    args = dict(lens=fake, ids=fake, lps=fake, B=4, W=8, off=fake, ido=fake, lpo=fake, cap=10, stream=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return f(a["lens"], a["ids"], a["lps"], a["B"], a["W"], a["off"], a["ido"], a["lpo"], a["cap"], a["stream"])

    for bad in (dict(lens=None), dict(ids=None), dict(off=None), dict(ido=None), dict(lps=None), dict(lpo=None),
                dict(B=0), dict(W=0), dict(W=sfc.MAX_PACKED_WIDTH + 1), dict(cap=-1)):
        assert call(**bad) == sfc.SFC_EINVAL, bad


def test_flag_constant_matches_binding():
    src = open(HEADER).read()
    for name in ("GREEDY_T0", "POSITIONAL", "MIN_P_FIRST", "TEST_STALL"):
        assert int(re.search(rf"#define SFC_FLAG_{name} (\d+)u", src).group(1)) == getattr(sfc, f"FLAG_{name}"), name


# ------------------------------------------------------------------------------------------------
# The binding's argument checks (on CPU tensors: the same checks run before a CUDA call)
# ------------------------------------------------------------------------------------------------

def _cpu_call_args(B=4, V=40, W=8):
    import torch

    out = sfc.SfcOutput(tokens=torch.empty(B, dtype=torch.int32), support_ids=torch.empty((B, W), dtype=torch.int32),
                        support_logprobs=torch.empty((B, W)), lengths=torch.empty(B, dtype=torch.int32),
                        selected_logprob=torch.empty(B), row_status=torch.empty(B, dtype=torch.int32))
    args = dict(logits=torch.zeros((B, V), dtype=torch.bfloat16), temperature=torch.ones(B),
                top_k=torch.full((B,), 5, dtype=torch.int32), top_p=torch.ones(B), min_p=torch.zeros(B),
                capture_rows=torch.ones(B, dtype=torch.uint8), packed_width=W)
    return out, args


def test_binding_accepts_a_well_formed_call():
    out, a = _cpu_call_args()
    sfc.check_call_layout(out, **a)


@pytest.mark.parametrize("bad", ["int64_top_k", "float64_T", "short_top_p", "int32_capture", "strided_min_p",
                                 "narrow_ids", "short_tokens", "f16_logprobs", "no_lengths", "float16_logits",
                                 "1d_logits", "column_logits", "narrow_mask"])
def test_binding_rejects_malformed_tensors(bad):
    """Tensors the kernels would misread (int64 read as int32 pairs, too-short per-row arrays, outputs
    narrower than the packed width, strided arrays) are refused on the host."""
    import torch

    out, a = _cpu_call_args()
    B, V, W = 4, 40, 8
    if bad == "int64_top_k":
        a["top_k"] = torch.full((B,), 5, dtype=torch.int64)
    elif bad == "float64_T":
        a["temperature"] = torch.ones(B, dtype=torch.float64)
    elif bad == "short_top_p":
        a["top_p"] = torch.ones(B - 1)
    elif bad == "int32_capture":
        a["capture_rows"] = torch.ones(B, dtype=torch.int32)
    elif bad == "strided_min_p":
        a["min_p"] = torch.zeros(2 * B)[::2]
    elif bad == "narrow_ids":
        out = out._replace(support_ids=torch.empty((B, W - 1), dtype=torch.int32))
    elif bad == "short_tokens":
        out = out._replace(tokens=torch.empty(B - 1, dtype=torch.int32))
    elif bad == "f16_logprobs":
        out = out._replace(support_logprobs=torch.empty((B, W), dtype=torch.float16))
    elif bad == "no_lengths":
        out = out._replace(lengths=None)
    elif bad == "float16_logits":
        a["logits"] = torch.zeros((B, V), dtype=torch.float16)
    elif bad == "1d_logits":
        a["logits"] = torch.zeros(V, dtype=torch.bfloat16)
    elif bad == "column_logits":
        a["logits"] = torch.zeros((V, B), dtype=torch.bfloat16).t()
    elif bad == "narrow_mask":
        out = out._replace(support_mask=torch.empty((B, (V + 31) // 32 - 1), dtype=torch.int32))
    with pytest.raises(sfc.SfcError):
        sfc.check_call_layout(out, **a)


def test_binding_requires_cuda_logits():
    out, a = _cpu_call_args()
    with pytest.raises(sfc.SfcError, match="CUDA"):
        sfc.check_call_tensors(out, **a)
