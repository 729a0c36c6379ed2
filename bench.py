"""Benchmark: decode steps/s of the fused sample · filter · capture call on GB300.

Workload (one "step" = one call over the whole batch): B=256 rows x V=151936 bf16 logits, quantised to
1/16-logit steps so ties form at every cut; top_k cycling {20, 50, 1024}, top_p 0.95, min_p 0, T 1; every
row captures its support, packed width 1024. This is the batch the method's HBM-roofline target is stated
on. Synthetic, seeded inputs (no dataset is involved).

  value          device throughput: a CUDA graph of G steps is replayed until K steps ran; every step reads
                 one of NB input buffers (NB x 77.8 MB > 2 x the 129 MB L2), so no step finds its logits in L2.
  e2e            the same metric through the public Python API with host buffers: per step a pinned-host ->
                 device copy of the logits and parameters, the call, and a device -> pinned-host copy of every
                 output (the captured supports realized-size: packed by the library straight into pinned
                 host memory); all inside the timed region, double-buffered so that step i + 1's input copy
                 overlaps step i's call and readback.
  roofline       algorithmic bytes per launch (one read of the logits + per-row parameters + the packed
                 outputs actually written) / average launch time, against the measured HBM copy bandwidth.
  cpu_baseline   the float64 oracle as it stands, on the host's cores: whole steps of the same workload over a
                 process pool of every core (median of 3), and a 32-row sample on one core.
  per_config     the other synthetic workloads (config 2, config 4, config 5 at B = 1, 32, 128, 512), each
                 timed the same way: us/step, rows/s, GB/s and fraction of the measured HBM bandwidth.

Multi-GPU: rows are independent, so each rank runs its own batch (weak scaling, no collective on the
data path); rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode steps/s (B rows x V vocab) with mask capture; % of HBM roofline"
UNIT = "steps/s"
CONFIG = {"workload": "B=256 x V=151936 bf16 logits quantised to 1/16 (ties), top_k {20,50,1024}, top_p 0.95, "
                      "all rows capture, packed_width 1024",
          "B": 256, "V": 151936, "dtype": "bf16", "packed_width": 1024,
          "l2": "inputs larger than L2: 4 rotating 77.8 MB logits buffers"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="sfc", choices=["sfc", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--buffers", type=int, default=4)
    ap.add_argument("--no-per-config", action="store_true", help="skip the other workloads' timings")
    ap.add_argument("--only", choices=["replay", "pack", "config4"],
                    help="time one other library kernel or workload alone (for profiling)")
    return ap.parse_args()


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    """Polls SM clock, max clock and clock-event reasons through NVML (ctypes) every millisecond."""

    # clock-event reason bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        self.samples = []
        self.t0 = self.t1 = None
        self.stop_flag = False
        self.ok = False
        try:
            import ctypes

            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            cudart = None
            for name in ("libcudart.so.13", "libcudart.so"):
                try:
                    cudart = ctypes.CDLL(name)
                    break
                except OSError:
                    continue
            bus = ctypes.create_string_buffer(64)
            if cudart is None or cudart.cudaDeviceGetPCIBusId(bus, 64, cuda_index) != 0:
                return
            self.handle = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.value, ctypes.byref(self.handle)) != 0:
                return
            mx = ctypes.c_uint()
            self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx))
            self.max_mhz = float(mx.value)
            self.ok = True
        except OSError:
            self.ok = False

    def _poll(self):
        import ctypes

        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self.stop_flag:
            self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk))
            self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.handle, ctypes.byref(rs))
            self.samples.append((time.time(), float(clk.value), int(rs.value)))
            time.sleep(0.001)

    def start(self):
        if self.ok:
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if not self.ok:
            return None
        self.stop_flag = True
        self.thread.join(timeout=2)
        sel = [(c, r) for t, c, r in self.samples if self.t0 <= t <= self.t1]
        if not sel:  # a very short region: take the samples nearest to it
            sel = [(c, r) for t, c, r in self.samples if self.t0 - 0.05 <= t <= self.t1 + 0.05]
        reasons = sorted({name for _, r in sel for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median([c for c, _ in sel]) if sel else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(sel), "source": "nvml"}


# ------------------------------------------------------------------------------------------------
def measured_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def kernel_source_sha256() -> str:
    import glob
    import hashlib

    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(ROOT, "top_support_capture_gb300", "csrc", "*")))
    files.append(os.path.join(ROOT, "include", "sfc.h"))
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(tag: str):
    """DRAM bytes per launch from the committed ncu summary of this workload, if the kernel sources are
    unchanged since that capture (else None)."""
    path = os.path.join(ROOT, "profiles", f"fused_kernel_{tag}_ncu_full.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    fields = dict(line.split(": ", 1) for line in text.splitlines() if ": " in line and line.split(": ", 1)[0] in
                  ("source_sha256", "traffic_bytes_per_launch"))
    if fields.get("source_sha256", "").strip() != kernel_source_sha256():
        return None
    try:
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def algorithmic_bytes(B, V, elt, W, capture, lengths):
    """One read of the logits and the per-row inputs; every output element the call must write."""
    rd = B * V * elt + B * (4 + 4 + 4 + 4 + 1)  # logits, T, top_k, top_p, min_p, capture flag
    wr = B * (4 + 4 + 4)  # tokens, row_status, lengths
    cap = capture.astype(bool)
    wr += int(cap.sum()) * 4  # selected logprob
    wr += int(np.minimum(lengths[cap], W).sum()) * 8  # packed ids + logprobs
    return rd + wr


# ------------------------------------------------------------------------------------------------
# The float64 oracle on the host cores (the CPU baseline and the reference arm). Rows are independent,
# so a step's rows are spread over a process pool (spawn: no worker inherits a CUDA context); each
# task gets a chunk of rows' raw logits and parameters and runs the oracle's own per-row function.
# ------------------------------------------------------------------------------------------------
def _oracle_chunk(task):
    import oracle

    raw, idx, dtype, T, k, tp, mp, seed, step = task
    for j, r in enumerate(idx):
        oracle.sample_row(oracle.widen_logits(raw[j], dtype), T[j], int(k[j]), tp[j], mp[j], seed, step, int(r))
    return len(idx)


def _oracle_tasks(w, rows, step, chunk):
    return [(np.ascontiguousarray(w.logits[idx]), idx, w.dtype, w.temperature[idx], w.top_k[idx], w.top_p[idx],
             w.min_p[idx], w.seed, step)
            for idx in (rows[i:i + chunk] for i in range(0, len(rows), chunk))]


def oracle_step_seconds(w, step, pool=None, rows=None):
    """Wall time of the oracle over `rows` (default: every row) of one step, on the pool or in-process."""
    rows = list(range(w.B)) if rows is None else list(rows)
    n = 1 if pool is None else pool._processes
    tasks = _oracle_tasks(w, rows, step, max(1, len(rows) // (4 * n)))
    t = time.perf_counter()
    if pool is None:
        for task in tasks:
            _oracle_chunk(task)
    else:
        pool.map(_oracle_chunk, tasks)
    return time.perf_counter() - t


def oracle_pool():
    import multiprocessing

    cores = os.cpu_count() or 1
    return multiprocessing.get_context("spawn").Pool(cores), cores


def cpu_baseline(w):
    """The oracle as it stands on this host: every row of a step over all cores (median of 3 steps), and a
    32-row sample on one core (median of 3, scaled to whole steps)."""
    pool, cores = oracle_pool()
    try:
        oracle_step_seconds(w, 0, pool, rows=range(min(w.B, 2 * cores)))  # start the workers
        all_s = statistics.median(oracle_step_seconds(w, i, pool) for i in range(3))
    finally:
        pool.close()
        pool.join()
    sample = list(range(0, w.B, max(1, w.B // 32)))[:32]
    one_s = statistics.median(oracle_step_seconds(w, i, None, rows=sample) for i in range(3)) * (w.B / len(sample))
    return {"value": 1.0 / all_s, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"all {w.B} rows of one step over {cores} processes, median of 3 steps ({all_s:.2f} s/step); "
                      f"float64 numpy, one full-row sort per row",
            "single_core": {"value": 1.0 / one_s, "unit": UNIT, "cores": 1,
                            "sample": f"{len(sample)} of {w.B} rows on one core, median of 3, scaled to {w.B} rows "
                                      f"({one_s:.2f} s/step)"}}


def shard_rows(rank: int, rows_per_rank: int):
    """This rank's rows of the job's batch (world x rows_per_rank rows, rank-major): [row0, row1). row0 is
    also the call's row_offset, so each row's race noise is keyed by its index in the job's batch and the
    shards together draw what one call over the whole batch draws."""
    row0 = rank * rows_per_rank
    return row0, row0 + rows_per_rank


def aggregate_ranks(local_ms: float, local_steps: int, device=None):
    """Whole-job throughput over the ranks of the default process group (or this process alone):
    every rank ran `local_steps` independent steps; the job time is the slowest rank's time.
    Returns (steps/s over all ranks, max ms over ranks)."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    max_ms = float(t.item())
    return world * local_steps / (max_ms / 1e3), max_ms


def per_config_timings(dev, peak):
    """The other synthetic workloads, each timed like the headline one (CUDA graph, CUDA events on the
    launching stream, enough rotating copies of the inputs to exceed twice the L2): config 2, config 4 and
    config 5's sweep B in {1, 32, 128, 512} (the smaller batches are the first rows of the 512-row one)."""
    import torch

    import top_support_capture_gb300 as sfc
    from top_support_capture_gb300 import workloads as wl

    def run(name, w):
        if w.dtype == wl.DT_BF16:
            L0 = torch.from_numpy(w.logits.view(np.int16)).to(dev).view(torch.bfloat16)
        else:
            L0 = torch.from_numpy(w.logits).to(dev)
        nb = int(min(512, max(1, -(-2 * 129e6 // w.logits.nbytes))))
        Ls = [L0] + [L0.clone() for _ in range(nb - 1)]
        t = lambda a: torch.from_numpy(a).to(dev)
        T, K, P, M, C = t(w.temperature), t(w.top_k), t(w.top_p), t(w.min_p), t(w.capture)
        out = sfc.allocate_outputs(w.B, w.packed_width, dev)
        ws = sfc.allocate_workspace(sfc.workspace_size(w.B, w.V, w.packed_width, w.dtype), dev)
        s = torch.cuda.Stream(dev)
        calls = max(nb, 20)
        with torch.cuda.stream(s):
            for i in range(3):
                sfc.sample_filter_capture_into(out, Ls[i % nb], T, K, P, M, w.seed, i, C, w.packed_width, stream=s,
                                               workspace=ws)
        torch.cuda.synchronize()
        lengths = out.lengths.cpu().numpy()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for i in range(calls):
                    sfc.sample_filter_capture_into(out, Ls[i % nb], T, K, P, M, w.seed, i, C, w.packed_width,
                                                   stream=s, workspace=ws)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ms = []
        rs = torch.cuda.current_stream(dev)  # the stream a replay runs on, and the events' stream
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(rs)
            g.replay()
            e1.record(rs)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1) / calls)
        us = 1e3 * statistics.median(ms)
        alg = algorithmic_bytes(w.B, w.V, 2 if w.dtype == wl.DT_BF16 else 4, w.packed_width, w.capture, lengths)
        gbs = alg / (us * 1e-6) / 1e9
        del Ls, g
        torch.cuda.empty_cache()
        return name, {"B": w.B, "V": w.V, "dtype": "bf16" if w.dtype == wl.DT_BF16 else "f32",
                      "packed_width": w.packed_width, "us_per_step": round(us, 2), "steps_per_s": round(1e6 / us, 1),
                      "rows_per_s": round(w.B * 1e6 / us, 1), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                      "input_copies": nb}

    res = dict([run("config2", wl.config2()), run("config4", wl.config4())])
    w5 = wl.config5(B=512)
    for B in (1, 32, 128, 512):
        w = wl.Workload(**{**w5.__dict__, "logits": np.ascontiguousarray(w5.logits[:B]),
                           **{k: getattr(w5, k)[:B].copy() for k in ("temperature", "top_k", "top_p", "min_p", "capture")}})
        res.update([run(f"config5_B{B}", w)])
    return res


def run_only(args):
    """One library kernel alone, for profiling and a quick timing: `replay` (the training-side replay of
    captured supports: 512 rows of the 151936-token workload, 155 MB of logits, larger than L2), `pack`
    (the realized-size packing of the 256-row batch's captured supports into pinned host memory) or
    `config4` (the wide class's call on config 4). Prints one JSON line with the mean time per call over
    --steps calls after --warmup calls."""
    import torch

    import top_support_capture_gb300 as sfc
    from top_support_capture_gb300 import workloads as wl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sfc.load_library()
    if args.only == "config4":  # the wide class: 256 x 129280 f32, W = 8192, two rotating inputs (> L2)
        ws = [wl.config4(step=i) for i in range(2)]
        t = lambda a: torch.from_numpy(a).to(dev)
        Ls = [torch.from_numpy(x.logits).to(dev) for x in ws]
        w = ws[0]
        T, K, P, M, C = t(w.temperature), t(w.top_k), t(w.top_p), t(w.min_p), t(w.capture)
        out = sfc.allocate_outputs(w.B, w.packed_width, dev)
        i = [0]

        def fn():
            sfc.sample_filter_capture_into(out, Ls[i[0] % 2], T, K, P, M, w.seed, i[0], C, w.packed_width)
            i[0] += 1
        work = f"config 4: {w.B} rows x V={w.V} f32, top_k 8192, W={w.packed_width}, a quarter of the rows capture"
        return _time_only(args, fn, work)
    w = wl.config3(B=512 if args.only == "replay" else 256)
    L = torch.from_numpy(w.logits.view(np.int16)).to(dev).view(torch.bfloat16)
    t = lambda a: torch.from_numpy(a).to(dev)
    T, K, P, M, C = t(w.temperature), t(w.top_k), t(w.top_p), t(w.min_p), t(w.capture)
    cap = sfc.sample_filter_capture(L, T, K, P, M, w.seed, 0, C, w.packed_width)
    lens = torch.clamp(cap.lengths, 1, w.packed_width).to(torch.int32)
    if args.only == "replay":
        fn = lambda: sfc.replay_logprob(L, T, cap.support_ids, lens, cap.tokens, support_logprobs=True)
        work = f"replay of {w.B} rows x V={w.V} bf16, supports of W={w.packed_width} (lengths 20-1080)"
    else:
        B, W = w.B, w.packed_width
        off = torch.empty(B + 1, dtype=torch.int64).pin_memory()
        ids = torch.empty(B * W, dtype=torch.int32).pin_memory()
        lps = torch.empty(B * W, dtype=torch.float32).pin_memory()
        fn = lambda: sfc.pack_supports_into(cap.lengths, cap.support_ids, cap.support_logprobs, off, ids, lps)
        work = f"packing of {B} captured supports (W={W}) into pinned host memory"
    return _time_only(args, fn, work)


def _time_only(args, fn, work):
    import torch

    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    print(json.dumps({"only": args.only, "workload": work, "calls": args.steps,
                      "us_per_call": round(1e3 * e0.elapsed_time(e1) / args.steps, 2)}))
    return 0


def run_reference(args):
    """The reference arm: the float64 oracle as it stands, on the host cores. Each step is one whole step of
    the workload (every row, over a process pool of all cores), so the reported time per step is measured,
    not extrapolated. If W + K steps would not end within about two minutes, only the steps that do are
    timed and the line says how many."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from top_support_capture_gb300 import workloads as wl

    w = wl.config3()
    pool, cores = oracle_pool()
    budget_s = 120.0
    times = []
    try:
        t_start = time.perf_counter()
        for i in range(args.warmup + args.steps):
            dt = oracle_step_seconds(w, i, pool)
            if i >= args.warmup:
                times.append(dt)
            if time.perf_counter() - t_start > budget_s and len(times) >= 3:
                break
    finally:
        pool.close()
        pool.join()
    total = sum(times)
    value = len(times) / total
    sample = (f"every one of the {w.B} rows of each step (step index i keys the race), over {cores} processes; "
              f"{len(times)} timed steps of {args.steps} asked (two-minute budget)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": len(times), "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": CONFIG,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.only:
        return run_only(args)

    import torch
    import torch.distributed as dist

    import top_support_capture_gb300 as sfc
    from top_support_capture_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sfc.load_library()

    # ---- inputs: NB decode steps of the workload, resident in HBM ----
    NB = args.buffers
    ws = [wl.config3(step=i, seed=3 + 1000 * rank) for i in range(NB)]
    w0 = ws[0]
    B, V, W = w0.B, w0.V, w0.packed_width
    row0, _ = shard_rows(rank, B)  # this rank's first row in the job's batch (keys the race's noise)
    logits = [torch.from_numpy(w.logits.view(np.int16)).to(dev).view(torch.bfloat16) for w in ws]
    t = lambda a: torch.from_numpy(a).to(dev)
    T, K, P, M, C = t(w0.temperature), t(w0.top_k), t(w0.top_p), t(w0.min_p), t(w0.capture)
    out = sfc.allocate_outputs(B, W, dev)
    stream = torch.cuda.current_stream(dev)

    def step_call(i):
        sfc.sample_filter_capture_into(out, logits[i % NB], T, K, P, M, w0.seed, i, C, W, stream=stream,
                                       row_offset=row0)

    # sanity (bench-time checks of the contract): every drawn token is in its row's support
    step_call(0)
    torch.cuda.synchronize()
    tok = out.tokens.cpu().numpy()
    ids = out.support_ids.cpu().numpy()
    lens = out.lengths.cpu().numpy()
    st = out.row_status.cpu().numpy()
    assert (st >= 0).all()
    for r in range(B):
        n = min(int(lens[r]), W)
        assert tok[r] in ids[r, :n] or lens[r] > W, r
    lengths0 = lens.copy()

    # ---- warm-up, then capture G steps in a CUDA graph ----
    for i in range(args.warmup):
        step_call(i)
    torch.cuda.synchronize()
    G = min(200, args.steps)
    reps = max(1, args.steps // G)
    K_steps = G * reps
    graph = torch.cuda.CUDAGraph()
    cap_stream = torch.cuda.Stream(dev)
    cap_stream.wait_stream(stream)
    with torch.cuda.stream(cap_stream):
        with torch.cuda.graph(graph, stream=cap_stream):
            for i in range(G):
                sfc.sample_filter_capture_into(out, logits[i % NB], T, K, P, M, w0.seed, i, C, W, stream=cap_stream,
                                               row_offset=row0)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.05)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gstream = torch.cuda.current_stream(dev)
    if sampler:
        sampler.mark(True)
    ev0.record(gstream)
    for _ in range(reps):
        graph.replay()
    ev1.record(gstream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(False)
    if world > 1:
        dist.barrier()
    dev_ms = ev0.elapsed_time(ev1)
    clocks = sampler.stop() if sampler else None

    value, dev_ms_max = aggregate_ranks(dev_ms, K_steps, device=dev)
    ms_per_step = dev_ms_max / K_steps

    # ---- roofline of the (single) kernel ----
    peak, peak_kind = measured_hbm_peak()
    alg = algorithmic_bytes(B, V, 2, W, w0.capture, lengths0)
    achieved = alg / (ms_per_step * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": profiled_traffic("B256_V151936_bf16"),
                "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind,
                "algorithmic_bytes_per_launch": alg}

    # ---- end to end through the public API with host buffers ----
    # Double-buffered: the host -> device copy of step i + 1 (copy stream) overlaps the call of step i
    # (compute stream) and the device -> host read of step i's outputs (readback stream); every step's
    # copies are still inside the timed region.
    host_logits = [torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16).pin_memory() for w in ws]
    host_par = [torch.from_numpy(a).pin_memory() for a in (w0.temperature, w0.top_k, w0.top_p, w0.min_p, w0.capture)]
    NBUF = 2
    d_logits = [torch.empty((B, V), dtype=torch.bfloat16, device=dev) for _ in range(NBUF)]
    d_par = [[torch.empty_like(h, device=dev) for h in host_par] for _ in range(NBUF)]
    outs = [sfc.allocate_outputs(B, W, dev) for _ in range(NBUF)]
    # per-row outputs copied back as they are; the supports move realized-size: the packing kernels
    # write CSR offsets and the captured entries straight into pinned host memory
    small = lambda o: [o.tokens, o.lengths, o.selected_logprob, o.row_status]
    host_out = [[torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in small(o)] for o in outs]
    realized = int(np.minimum(lengths0, W).sum())
    host_off = [torch.empty(B + 1, dtype=torch.int64).pin_memory() for _ in range(NBUF)]
    host_ids = [torch.empty(B * W, dtype=torch.int32).pin_memory() for _ in range(NBUF)]
    host_lps = [torch.empty(B * W, dtype=torch.float32).pin_memory() for _ in range(NBUF)]
    h2d = host_logits[0].numel() * 2 + sum(h.numel() * h.element_size() for h in host_par)
    d2h = sum(h.numel() * h.element_size() for h in host_out[0]) + (B + 1) * 8 + realized * 8
    s_copy, s_comp, s_back = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(NBUF)]    # inputs of buffer j landed
    ev_used = [torch.cuda.Event() for _ in range(NBUF)]  # the call on buffer j has read its inputs
    ev_out = [torch.cuda.Event() for _ in range(NBUF)]   # buffer j's outputs are written
    ev_read = [torch.cuda.Event() for _ in range(NBUF)]  # buffer j's outputs are on the host

    def e2e_step(i):
        j = i % NBUF
        with torch.cuda.stream(s_copy):
            s_copy.wait_event(ev_used[j])
            d_logits[j].copy_(host_logits[i % NB], non_blocking=True)
            for dpar, h in zip(d_par[j], host_par):
                dpar.copy_(h, non_blocking=True)
            ev_in[j].record(s_copy)
        s_comp.wait_event(ev_in[j])
        s_comp.wait_event(ev_read[j])  # the previous outputs of buffer j have been read back
        dp = d_par[j]
        sfc.sample_filter_capture_into(outs[j], d_logits[j], dp[0], dp[1], dp[2], dp[3], w0.seed, i, dp[4], W,
                                       stream=s_comp, row_offset=row0)
        ev_used[j].record(s_comp)
        ev_out[j].record(s_comp)
        with torch.cuda.stream(s_back):
            s_back.wait_event(ev_out[j])
            for h, d in zip(host_out[j], small(outs[j])):
                h.copy_(d, non_blocking=True)
            sfc.pack_supports_into(outs[j].lengths, outs[j].support_ids, outs[j].support_logprobs, host_off[j],
                                   host_ids[j], host_lps[j], stream=s_back)
            ev_read[j].record(s_back)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for i in range(args.e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_value, _ = aggregate_ranks(e2e_s * 1e3, args.e2e_steps, device=dev)

    line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K_steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": CONFIG,
            "rows_per_s": round(value * B, 1), "gpu_launches": K_steps,
            "roofline": roofline,
            "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": args.e2e_steps},
            "clocks": clocks}
    if rank == 0 and world == 1 and not args.no_per_config:
        line["per_config"] = per_config_timings(dev, peak)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w0)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
