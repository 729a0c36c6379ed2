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
    assert sfc.workspace_size(256, 151936, 1024, sfc.SFC_BF16) == 0


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


def test_ex_invalid_flags_and_row_offset_rejected_on_host(lib):
    """The extended call's own arguments: unknown flag bits, a negative row offset, and an offset that
    pushes the last row past the counter's 32-bit row word."""
    f = lib.sfc_sample_filter_capture_ex
    fake = 0x1000  # never dereferenced: the checks reject the call first

    def call(flags=0, row_offset=0, B=4, mask=None, cap=None):
        return f(fake, 0, B, 16, 16, fake, fake, fake, fake, 0, 0, cap, 8, fake, fake, fake, fake, fake, fake, mask,
                 flags, 0, row_offset, None, 0, None)

    assert call(flags=8) == sfc.SFC_EINVAL
    assert call(flags=1 << 31) == sfc.SFC_EINVAL
    assert call(row_offset=-1) == sfc.SFC_EINVAL
    assert call(row_offset=(1 << 32) - 3, B=4) == sfc.SFC_EINVAL
    assert call(B=4, mask=fake) == sfc.SFC_EINVAL  # a support mask needs capture_rows


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
    for name in ("GREEDY_T0", "POSITIONAL", "MIN_P_FIRST"):
        assert int(re.search(rf"#define SFC_FLAG_{name} (\d+)u", src).group(1)) == getattr(sfc, f"FLAG_{name}"), name
