"""GPU parity of rows split into independent slices: each row is streamed by S ordinary CTAs that publish
their candidates, sample threshold and softmax statistics in the workspace; the CTA that arrives last (an
atomic ticket per row) merges them in slice order and finishes the row. Every finish path is reached
through the merge: value bins (bf16), the sorting finishes (f32), and the multi-pass path (slices whose
candidates do not fit, top-k disabled)."""
import numpy as np
import pytest

from top_support_capture_gb300 import workloads as wl
from sfc_parity import clear_margins, compare, gpu_run, margin_fail, oracle_run, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_support_capture_gb300 as sfc

    sfc.load_library()


def _check(w, rows=None, **kw):
    rows = list(range(w.B)) if rows is None else rows
    ref = oracle_run(w, rows, **{k: v for k, v in kw.items() if k in ("positional", "min_p_first", "greedy_t0")})
    ok = [r for r in rows if r not in set(margin_fail(ref, rows))]
    got = gpu_run(w, **kw)
    return compare(w, ref, got, ok, support_logprobs=kw.get("support_logprobs", True)), got


@pytest.mark.parametrize("S", [2, 3, 4, 8])
def test_long_vocabulary_rows_forced_slices(S):
    """B=24 rows of the 151936-token workload (ties at every cut, top_k 20 / 50 / 1024)."""
    w, ref, left = clear_margins(lambda salt: wl.config3(B=24, salt=salt), 24, list(range(24)))
    assert not left
    assert compare(w, ref, gpu_run(w, slices=S), range(24)) == 24


@pytest.mark.parametrize("S", [2, 5, 8])
def test_262144_token_rows_forced_slices(S):
    w, ref, left = clear_margins(lambda salt: wl.config5(B=8, salt=salt), 8, list(range(8)))
    assert not left
    assert compare(w, ref, gpu_run(w, slices=S), range(8)) == 8


@pytest.mark.parametrize("S", [2, 3, 7])
def test_short_rows_many_slices(S):
    """32000-token rows: slices far shorter than the ring (one partial stage each)."""
    w, ref, left = clear_margins(lambda salt: wl.config2(salt=salt), 64, list(range(64)))
    assert not left
    assert compare(w, ref, gpu_run(w, slices=S), range(64)) == 64


@pytest.mark.parametrize("S", [2, 4])
def test_float_rows_forced_slices(S):
    """fp32 rows (the sorting finishes) with top_k up to 1500 and packed width 2048."""
    B = 12
    def make(salt):
        w0 = wl.config4(B=B, salt=salt)
        k = np.array([20, 300, 1500, 8192, 64, 1000] * 2, np.int32)
        return wl.Workload(**{**w0.__dict__, "top_k": k, "packed_width": 2048, "capture": np.ones(B, np.uint8)})
    w, ref, left = clear_margins(make, B, list(range(B)))
    assert not left
    assert compare(w, ref, gpu_run(w, slices=S), range(B)) == B


@pytest.mark.parametrize("dtype", [wl.DT_BF16, wl.DT_F32])
def test_slices_of_unaligned_strided_rows(dtype):
    """Odd row stride (unaligned row starts), a ragged end: the first slice reads the head scalars, the
    last the tail."""
    rng = np.random.default_rng(21)
    B, V, stride = 5, 50021, 50027
    base = (rng.standard_normal((B, stride)) * 1.5).astype(np.float32)
    full = wl.f32_to_bf16_bits(base) if dtype == wl.DT_BF16 else base
    k = np.array([1, 7, 50, 400, 0], np.int32)
    tp = np.array([0.9, 1.0, 0.95, 0.8, 0.7], np.float32)
    w = wl.Workload("edge", dtype, np.ascontiguousarray(full[:, :V]), np.ones(B, np.float32), k, tp,
                    np.zeros(B, np.float32), np.ones(B, np.uint8), 512, 9, 0)
    ref = oracle_run(w)
    ok = [r for r in range(B) if r not in set(margin_fail(ref, range(B)))]
    d = to_device(w)
    big = (torch.from_numpy(full.view(np.int16)).cuda().view(torch.bfloat16) if dtype == wl.DT_BF16
           else torch.from_numpy(full).cuda())
    d["logits"] = big[:, :V]
    for S in (3, 6):
        assert compare(w, ref, gpu_run(w, dev=d, slices=S), ok) == len(ok)


def test_top_k_disabled_and_huge_ties_take_the_multi_pass_path():
    """Slices whose candidates cannot be bounded (top_k off) or overflow (one tie group over the row)."""
    B, V = 4, 70000
    l = np.zeros((B, V), np.float32)
    l[0] = np.random.default_rng(3).standard_normal(V)
    l[1] = np.random.default_rng(4).standard_normal(V)
    l[3, 777] = 1.0
    w = wl.Workload("mp", wl.DT_BF16, wl.f32_to_bf16_bits(l), np.ones(B, np.float32),
                    np.array([0, 0, 5, 2], np.int32), np.array([0.6, 0.9, 1.0, 1.0], np.float32),
                    np.zeros(B, np.float32), np.ones(B, np.uint8), 1024, 5, 0)
    n, got = _check(w, slices=4)
    assert n >= 3
    assert got["lengths"][2] == V and got["row_status"][2] == 1


@pytest.mark.parametrize("mode", [dict(positional=True), dict(min_p_first=True), dict(support_logprobs=False)])
def test_modes_through_slices(mode):
    w0 = wl.config5(B=8)
    w = wl.Workload(**{**w0.__dict__, "top_p": np.linspace(0.5, 0.99, 8).astype(np.float32)})
    n, _ = _check(w, slices=4, **mode)
    assert n >= 6


def test_greedy_rows_through_slices():
    w0 = wl.config3(B=6)
    T = np.array([0, 1, 0, 1, 0, 1], np.float32)
    w = wl.Workload(**{**w0.__dict__, "temperature": T})
    n, got = _check(w, slices=4, greedy_t0=True)
    assert n == 6
    assert (got["lengths"][T == 0] == 1).all()


def test_support_mask_through_slices():
    """Overflowing rows (top_k 1024, W = 1000) also write S's bitmask from the merged support."""
    w0 = wl.config3(B=6)
    w = wl.Workload(**{**w0.__dict__, "packed_width": 1000})
    ref = oracle_run(w, want_mask=True)
    got = gpu_run(w, slices=4, support_mask=True)
    ok = [r for r in range(6) if r not in set(margin_fail(ref, range(6)))]
    compare(w, ref, got, ok)
    mask = got["support_mask"].view(np.uint32)
    for r in ok:
        if ref.row_status[r] == 1:
            assert np.array_equal(mask[r], ref.support_mask[r]), r


def test_slices_agree_with_one_cta_per_row():
    """The split changes only the order in which partial softmax sums merge: tokens, ids, lengths and
    statuses are identical to one CTA per row; logprobs agree within the tolerance; a repeat of the same
    split is bit-identical (the workspace is all zero again after every call)."""
    import top_support_capture_gb300 as sfc

    w = wl.config3(B=48, step=5)
    d = to_device(w)
    one = gpu_run(w, dev=d, slices=1)
    ws = sfc.allocate_workspace(sfc.workspace_size(w.B, w.V, w.packed_width, w.dtype, 4), "cuda")
    runs = []
    for _ in range(3):
        out = sfc.sample_filter_capture(d["logits"], d["temperature"], d["top_k"], d["top_p"], d["min_p"], w.seed,
                                        w.step, d["capture_rows"], w.packed_width, slices=4)
        torch.cuda.synchronize()
        runs.append({k: (None if v is None else v.cpu().numpy()) for k, v in out._asdict().items()})
    for k in ("tokens", "lengths", "row_status"):
        assert np.array_equal(runs[0][k], one[k]), k
    for r in range(w.B):
        n = min(int(one["lengths"][r]), w.packed_width)
        assert np.array_equal(runs[0]["support_ids"][r, :n], one["support_ids"][r, :n]), r
        assert np.abs(runs[0]["support_logprobs"][r, :n] - one["support_logprobs"][r, :n]).max() <= 2e-5, r
        for rr in runs[1:]:
            assert np.array_equal(rr["support_ids"][r, :n], runs[0]["support_ids"][r, :n])
            assert np.array_equal(rr["support_logprobs"][r, :n].view(np.uint32),
                                  runs[0]["support_logprobs"][r, :n].view(np.uint32))
    for rr in runs[1:]:
        assert np.array_equal(rr["tokens"], runs[0]["tokens"])
        assert np.array_equal(rr["selected_logprob"].view(np.uint32), runs[0]["selected_logprob"].view(np.uint32))
    # an explicit workspace: every byte is zero again after the call (tickets, records, pools)
    out = sfc.allocate_outputs(w.B, w.packed_width, "cuda")
    sfc.sample_filter_capture_into(out, d["logits"], d["temperature"], d["top_k"], d["top_p"], d["min_p"], w.seed,
                                   w.step, d["capture_rows"], w.packed_width, workspace=ws, slices=4)
    torch.cuda.synchronize()
    assert int((ws != 0).sum().item()) == 0
    assert np.array_equal(out.tokens.cpu().numpy(), runs[0]["tokens"])


@pytest.mark.parametrize("make,B,S", [(lambda salt: wl.config5(B=32, salt=salt), 32, 8),
                                      (lambda salt: wl.config3(B=100, salt=salt), 100, 3)])
def test_default_split_of_short_batches(make, B, S):
    """The library's own choice: short batches of long rows split while all slices fit the CTA slots
    (32 x 262144 -> 8 slices, 100 x 151936 -> 3), every row compared."""
    import top_support_capture_gb300 as sfc

    w, ref, left = clear_margins(make, B, list(range(B)))
    assert not left
    assert sfc.workspace_size(B, w.V, w.packed_width, w.dtype) == sfc.workspace_size(B, w.V, w.packed_width, w.dtype, S)
    assert sfc.workspace_size(B, w.V, w.packed_width, w.dtype) > 0
    assert compare(w, ref, gpu_run(w), range(B)) == B


def test_one_workspace_serves_calls_of_every_size():
    """Calls of growing batch size on one workspace: each call's tickets lie where earlier, smaller calls
    kept records and candidates, which they returned to zero."""
    import top_support_capture_gb300 as sfc

    sizes = [(2, 4), (6, 4), (30, 8), (100, 3)]
    need = max(sfc.workspace_size(B, 151936, 1024, sfc.SFC_BF16, S) for B, S in sizes)
    ws = sfc.allocate_workspace(need, "cuda")
    for B, S in sizes:
        w, ref, left = clear_margins(lambda salt: wl.config3(B=B, step=B, salt=salt), B, list(range(B)))
        assert not left
        d = to_device(w)
        out = sfc.allocate_outputs(B, w.packed_width, "cuda")
        sfc.sample_filter_capture_into(out, d["logits"], d["temperature"], d["top_k"], d["top_p"], d["min_p"], w.seed,
                                       w.step, d["capture_rows"], w.packed_width, workspace=ws, slices=S)
        torch.cuda.synchronize()
        got = {k: (None if v is None else v.cpu().numpy()) for k, v in out._asdict().items()}
        assert compare(w, ref, got, range(B)) == B
        assert int((ws != 0).sum().item()) == 0
