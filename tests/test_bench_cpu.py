"""bench.py's host arithmetic, on CPU: the algorithmic bytes behind the roofline fraction, the DRAM
traffic figure taken from a committed ncu summary only while the kernel sources are unchanged, and the
peak the fraction divides by."""
import json
import os

import numpy as np
import pytest

import bench


def test_algorithmic_bytes_by_hand():
    # 2 rows of 10 bf16 logits, packed width 4; row 0 captures a 6-member support (4 packed), row 1 does not
    got = bench.algorithmic_bytes(2, 10, 2, 4, np.array([1, 0], np.uint8), np.array([6, 0]))
    reads = 2 * 10 * 2 + 2 * (4 + 4 + 4 + 4 + 1)  # logits; T, top_k, top_p, min_p, capture flag
    writes = 2 * (4 + 4 + 4) + 1 * 4 + 4 * (4 + 4)  # token, status, length; selected logprob; 4 packed entries
    assert got == reads + writes == 134


def test_headline_bytes_from_the_oracles_support_sizes():
    """The bench workload's bytes per launch with the support sizes the oracle finds at step 0 (the bench
    takes them from the kernel's first call, which parity makes the same): one read of 256 x 151936 bf16
    logits and the row parameters, the per-row outputs, and 8 bytes per packed support entry."""
    import oracle
    from top_support_capture_gb300 import workloads as wl

    w = wl.config3(step=0)
    r = oracle.sample_filter_capture(w.logits, w.dtype, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, 0,
                                     w.capture, w.packed_width)
    got = bench.algorithmic_bytes(w.B, w.V, 2, w.packed_width, w.capture, r.lengths)
    packed = sum(min(int(n), 1024) for n in r.lengths)  # every row captures
    assert 1024 * 85 < packed < 1024 * 256  # the top_k 1024 rows fill their packed width
    assert got == 256 * 151936 * 2 + 256 * 17 + 256 * 12 + 256 * 4 + packed * 8


def _profile(tmp_path, sha, traffic="123456789"):
    d = tmp_path / "profiles"
    d.mkdir(exist_ok=True)
    (d / "fused_kernel_T_ncu_full.md").write_text(
        f"# summary\n\nsource_sha256: {sha}\ntraffic_bytes_per_launch: {traffic}\n\n| metric | value |\n")


def test_traffic_only_while_the_sources_match(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha256", lambda: "a" * 64)
    assert bench.profiled_traffic("T") is None  # no summary
    _profile(tmp_path, "a" * 64)
    assert bench.profiled_traffic("T") == 123456789
    _profile(tmp_path, "b" * 64)  # captured from other sources
    assert bench.profiled_traffic("T") is None
    _profile(tmp_path, "a" * 64, traffic="n/a")
    assert bench.profiled_traffic("T") is None


def test_source_hash_covers_the_kernel_and_its_header(tmp_path, monkeypatch):
    base = bench.kernel_source_sha256()
    assert len(base) == 64 and base == bench.kernel_source_sha256()
    for rel in (("top_support_capture_gb300", "csrc"), ("include",)):
        (tmp_path.joinpath(*rel)).mkdir(parents=True, exist_ok=True)
    csrc = tmp_path / "top_support_capture_gb300" / "csrc"
    (csrc / "k.cuh").write_text("kernel")
    (tmp_path / "include" / "sfc.h").write_text("header")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_sha256()
    (csrc / "k.cuh").write_text("kernel, changed")
    h1 = bench.kernel_source_sha256()
    (tmp_path / "include" / "sfc.h").write_text("header, changed")
    h2 = bench.kernel_source_sha256()
    assert len({h0, h1, h2}) == 3


def test_peak_is_the_measured_copy_bandwidth(tmp_path, monkeypatch):
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            assert bench.measured_hbm_peak() == (float(json.load(f)["hbm_gbs"]), "measured")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))  # no measurement: the recipe's fallback
    assert bench.measured_hbm_peak() == (6800.0, "fallback")
