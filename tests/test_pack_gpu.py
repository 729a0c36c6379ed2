"""GPU parity of the realized-size packing against the reference packing, into device memory and
directly into pinned host memory, with a capacity that cuts the run short."""
import numpy as np
import pytest

import oracle
from top_support_capture_gb300 import workloads as wl
from sfc_parity import gpu_run

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import top_support_capture_gb300 as sfc

    sfc.load_library()


def _capture(w):
    import top_support_capture_gb300 as sfc
    from sfc_parity import to_device

    d = to_device(w)
    return sfc.sample_filter_capture(d["logits"], d["temperature"], d["top_k"], d["top_p"], d["min_p"], w.seed, w.step,
                                     d["capture_rows"], w.packed_width)


@pytest.mark.parametrize("where", ["device", "pinned_host"])
@pytest.mark.parametrize("make", [lambda: wl.config2(), lambda: wl.config3(B=24)])
def test_pack_matches_reference(where, make):
    import top_support_capture_gb300 as sfc

    w = make()
    out = _capture(w)
    torch.cuda.synchronize()
    lens, ids, lps = (x.cpu().numpy() for x in (out.lengths, out.support_ids, out.support_logprobs))
    ref_off, ref_ids, ref_lps = oracle.pack_supports(lens, ids, lps, w.packed_width)
    total = int(ref_off[-1])
    alloc = (lambda n, dt: torch.full((n,), -7, dtype=dt, device="cuda")) if where == "device" else \
            (lambda n, dt: torch.full((n,), -7, dtype=dt).pin_memory())
    off = alloc(w.B + 1, torch.int64)
    pid = alloc(total, torch.int32)
    plp = alloc(total, torch.float32)
    sfc.pack_supports_into(out.lengths, out.support_ids, out.support_logprobs, off, pid, plp)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(off.cpu().numpy(), ref_off)
    np.testing.assert_array_equal(pid.cpu().numpy(), ref_ids)
    np.testing.assert_array_equal(plp.cpu().numpy(), ref_lps)


def test_pack_capacity_cut_and_ids_only():
    import top_support_capture_gb300 as sfc

    w = wl.config3(B=9)
    out = _capture(w)
    torch.cuda.synchronize()
    lens, ids = out.lengths.cpu().numpy(), out.support_ids.cpu().numpy()
    ref_off, ref_ids, _ = oracle.pack_supports(lens, ids, None, w.packed_width)
    cap = int(ref_off[-1]) // 2
    off = torch.zeros(w.B + 1, dtype=torch.int64, device="cuda")
    pid = torch.full((cap + 5,), -7, dtype=torch.int32, device="cuda")
    sfc.pack_supports_into(out.lengths, out.support_ids, None, off, pid[:cap])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(off.cpu().numpy(), ref_off)  # the full offsets even when cut short
    got = pid.cpu().numpy()
    np.testing.assert_array_equal(got[:cap], ref_ids[:cap])
    assert (got[cap:] == -7).all()
