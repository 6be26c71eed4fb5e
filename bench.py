"""Benchmark of the BEV-pooling hot path on one GB300 (or N independent replicas).

A step is one pass of the whole hot path over one synthetic frame:
bevpool_build_map (compaction and a counting sort by cell with the frustum
order restored inside each run, index derivation, intervals) followed by
bevpool_forward (interval-owned scatter-reduce).  L2 is flushed (a 256 MiB
buffer is written) before the map build and again before the forward, so
both run from HBM; each is bracketed by CUDA events on the
stream it is launched on.  The headline value is the forward's device time in
microseconds per call (lower is better); the map build and the whole step are
reported beside it.

Also reported, on one line of JSON:
  roofline      for a working set within half the L2 (the L2-resident
                regime): the gather-level bytes of one forward / its warm-L2
                CUDA-graph time, against the L2 copy bandwidth measured in the
                same run (bevpool_probe_l2), with the fraction of the ncu L2
                ceiling beside it; otherwise the forward's compulsory bytes /
                its L2-flushed event time against the measured HBM copy
                bandwidth;
  roofline_hbm  the HBM form of the above for every workload;
  dram_batch    (canonical runs) the DRAM-bound batch configuration's forward
                timed the same way, with its HBM roofline;
  e2e           the same forward driven from pinned host buffers through the
                C ABI (H2D of depth+feat, forward, D2H of the output), two
                frames in flight on two streams (one frame's D2H overlapping
                the next one's H2D and forward); the serial per-frame time
                is reported beside it;
  cpu_baseline  the FP64 oracle (single thread) on the same workload;
  extra         map-build time, warm-L2 CUDA-graph replay of the forward
                (the timing method of the pages' Table 1), L2-level gather GB/s.

--impl reference times the oracle alone (the reference arm of this build).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "BEV-pool forward µs/call and GB/s vs L2/HBM roofline (209K pts, C=80, FP16/FP8)"
FLUSH_BYTES = 256 << 20
REFERENCE_BUDGET_S = 150.0
FALLBACK_HBM_GBS = 6800.0
# ncu ceilings of the GB300 L2 for SM traffic (lts__t_sectors_srcunit_tex_op_read /
# _op_write peak_sustained: 2 and 1 sectors of 32 B per cycle on each of 188
# slices at the 1.979 GHz L2 clock of the canonical capture)
NCU_L2_READ_GBS = 188 * 2 * 32 * 1.979
NCU_L2_WRITE_GBS = 188 * 1 * 32 * 1.979
FORWARD_SOURCES = ["forward_impl.cuh", "forward_f16.cu", "forward_e4m3.cu", "forward_f16_e4m3out.cu",
                   "forward_e4m3_e4m3out.cu", "forward_nvfp4.cu", "forward_nvfp4_e4m3out.cu", "bevpool_internal.cuh"]


def forward_source_hash() -> str:
    """Hash of the forward's code (comments stripped, so editing a comment
    keeps the ncu records that were taken on the same code)."""
    import re

    h = hashlib.sha1()
    for f in FORWARD_SOURCES:
        with open(os.path.join(ROOT, "depth_weighted_scatter_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(line.rstrip() for line in text.splitlines() if line.strip()).encode())
    return h.hexdigest()[:16]


def measured_peaks() -> tuple:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(workload: str, key: str = "dram_bytes_per_launch"):
    """Bytes per forward launch from a committed ncu capture (DRAM bytes with
    caches flushed, or with key="l2_bytes_warm" the L2 bytes of a warm
    launch), if it was taken on the current forward source."""
    p = os.path.join(ROOT, "profiles", "forward_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("source_hash") == forward_source_hash() and key in e:
            return float(e[key])
    except Exception:
        pass
    return None


def bytes_model(wl, n_points: int, n_intervals: int, out_bytes: int = 2) -> dict:
    """Bytes one forward must move.  'footprint' = every array the forward
    touches, once (the compulsory HBM traffic after an L2 flush);
    'gather' = what the owners actually read per point (L2-level)."""
    eb = 2 if wl.dtype == "f16" else 1
    row = wl.C // 2 + wl.C // 16 if wl.dtype == "nvfp4" else wl.C * eb   # NVFP4: E2M1 pairs + block scales
    idx = 12 * n_points                  # ranks_depth, ranks_feat, ranks_bev
    iv = 8 * n_intervals                 # interval_starts, interval_lengths
    depth = wl.n_frustum * eb
    feat = wl.n_feat_rows * row
    out = wl.n_cells * wl.C * out_bytes
    footprint = idx + iv + depth + feat + out
    gather = idx + iv + n_points * eb + n_points * row + out
    return dict(index=idx, intervals=iv, depth=depth, feat=feat, out=out, footprint=footprint, gather=gather)


def l2_probe(device, stream, mib: int = 64, passes: int = 16, reps: int = 5) -> dict:
    """L2 bandwidth of a buffer resident in L2 (bevpool_probe_l2): read, write
    and copy of `mib` MiB, `passes` passes per launch, best of `reps` launches,
    GB/s.  Copy counts the bytes read plus the bytes written (a STREAM copy,
    the convention of the HBM peak)."""
    import torch

    from depth_weighted_scatter_gb300 import bevpool

    buf = torch.ones(mib << 18, dtype=torch.int32, device=device)
    sink = torch.zeros(1, dtype=torch.int32, device=device)
    nbytes = buf.numel() * 4
    out = {"buffer_mib": mib, "passes": passes, "launches": reps}
    for name, mode in (("read", bevpool.PROBE_READ), ("write", bevpool.PROBE_WRITE), ("copy", bevpool.PROBE_COPY)):
        bevpool.probe_l2(buf, 2, mode=mode, sink=sink, stream=stream)      # brings the buffer into L2
        best = float("inf")
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            bevpool.probe_l2(buf, passes, mode=mode, sink=sink, stream=stream)
            b.record(stream)
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b) * 1e-3)
        out[f"{name}_gbs"] = passes * nbytes / best / 1e9
    return out


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled while it runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu_index), "-lms", str(self.period_ms)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def nvtx_push(name: str) -> None:
    try:
        import torch

        torch.cuda.nvtx.range_push(name)
    except Exception:
        pass


def nvtx_pop() -> None:
    try:
        import torch

        torch.cuda.nvtx.range_pop()
    except Exception:
        pass


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, world: int, device):
    """Element-wise max of a list of floats over all ranks."""
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist

    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def config_dict(wl, n_pts: int, n_int: int, world: int, out_dtype: str = "f16", device_run: bool = True) -> dict:
    d = {"workload": f"{wl.name}: NC={wl.NC} D={wl.D} H={wl.H} W={wl.W} C={wl.C} grid={wl.grid} "
                     f"points={n_pts} intervals={n_int}"}
    if device_run:
        d["l2"] = "flushed (256 MiB written) before the map build and before the forward"
        d["parallelism"] = f"replicas x{world}" if world > 1 else "single GPU"
    else:
        d["host"] = "FP64 C oracle, one thread on the host CPU; no GPU involved"
    if out_dtype == "e4m3":
        d["output"] = "E4M3 codes of value / out_scale, out_scale = max|output| / 448 (calibrated once, untimed)"
    return d


def oracle_call(wl, out_scale=None):
    """One oracle forward of the workload (with the E4M3 output when out_scale is given)."""
    import oracle

    if wl.dtype == "nvfp4":
        fwd = lambda: oracle.forward_nvfp4(wl.cell_ids, *wl.dims(), wl.n_cells, wl.C, wl.depth, wl.feat,
                                           wl.feat_block, wl.depth_scale, wl.feat_scale)
        if out_scale is None:
            return fwd
        return lambda: oracle.e4m3_from_double(fwd() / out_scale)
    if out_scale is None:
        return lambda: oracle.forward(wl.dtype, wl.cell_ids, *wl.dims(), wl.n_cells, wl.C, wl.depth, wl.feat,
                                      wl.depth_scale, wl.feat_scale)
    return lambda: oracle.forward_e4m3_out(wl.dtype, wl.cell_ids, *wl.dims(), wl.n_cells, wl.C, wl.depth, wl.feat,
                                           wl.depth_scale, wl.feat_scale, out_scale)


def host_cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine() or "unknown"


def cpu_oracle_time(wl, budget_s: float = 10.0, max_reps: int = 50, out_scale=None) -> dict:
    """Times the oracle's forward on the full workload, single-threaded."""
    import oracle

    oracle.build()
    call = oracle_call(wl, out_scale)
    call()                                              # load + page in
    times = []
    t_start = time.perf_counter()
    while len(times) < max_reps and (time.perf_counter() - t_start < budget_s or len(times) < 3):
        t0 = time.perf_counter()
        call()
        times.append(time.perf_counter() - t0)
    return {"value": statistics.mean(times) * 1e6, "unit": "us/call", "cores": 1, "kind": "oracle",
            "median": statistics.median(times) * 1e6, "cpu_model": host_cpu_model(),
            "sample": f"full {wl.name} workload ({wl.n_kept} points, C={wl.C}), {len(times)} calls of the "
                      f"single-threaded FP64 C oracle forward; host has {os.cpu_count()} cores"}


def run_reference(args) -> None:
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from depth_weighted_scatter_gb300 import workloads
    import oracle

    wl = workloads.make(args.config)
    oracle.build()
    m = oracle.build_map(wl.cell_ids, *wl.dims(), wl.n_cells)
    out_scale = None
    if args.out_dtype == "e4m3":                        # the same calibration as the GPU arm: max|output| / 448
        ref = oracle_call(wl)()
        out_scale = float(np.abs(ref).max()) / 448.0 or 1.0
    call = oracle_call(wl, out_scale)
    t0 = time.perf_counter()
    call()
    t_call = time.perf_counter() - t0
    for _ in range(args.warmup - 1):
        call()
    steps = max(1, min(args.steps, int(REFERENCE_BUDGET_S / max(t_call, 1e-6))))   # a few minutes at most
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        call()
        times.append(time.perf_counter() - t0)
    v = statistics.mean(times) * 1e6
    line = {"metric": METRIC, "value": v, "unit": "us/call", "impl": "reference", "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": v / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(wl, m["n_points"], m["n_intervals"], world, args.out_dtype, device_run=False),
            "cpu_baseline": {"value": v, "unit": "us/call", "cores": 1, "kind": "oracle",
                             "median": statistics.median(times) * 1e6, "cpu_model": host_cpu_model(),
                             "sample": f"each step one full {wl.name} forward of the single-threaded FP64 C oracle; "
                                       f"host has {os.cpu_count()} cores"},
            "e2e": {"value": v, "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def pipelined_e2e_us(bevpool, m, wl, dt, cap, out_scale, ref_out, depth_h, feat_h, block_h, frames, stream,
                     reps: int = 3):
    """Frames from pinned host buffers through the C ABI, two in flight: frame
    i's D2H on one stream overlaps frame i + 1's H2D and forward on another.
    Returns µs per frame (the median over `reps` runs of `frames` frames, after
    3 untimed ones) and checks that the last frame's output read back equals
    ref_out (same inputs)."""
    import torch

    dev = ref_out.device
    nb = 2
    d_in = [(torch.empty_like(depth_h, device=dev), torch.empty_like(feat_h, device=dev),
             torch.empty_like(block_h, device=dev) if block_h is not None else None) for _ in range(nb)]
    d_out = [torch.empty_like(ref_out) for _ in range(nb)]
    h_out = [torch.empty(ref_out.shape, dtype=ref_out.dtype).pin_memory() for _ in range(nb)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    read_done = [None] * nb

    def frame(i):
        k = i % nb
        dd, ff, bb = d_in[k]
        with torch.cuda.stream(s_in):
            dd.copy_(depth_h, non_blocking=True)
            ff.copy_(feat_h, non_blocking=True)
            if bb is not None:
                bb.copy_(block_h, non_blocking=True)
            if read_done[k] is not None:           # d_out[k] is free once frame i - 2 has been read back
                s_in.wait_event(read_done[k])
            bevpool.forward(m, dd, ff, wl.C, dtype=dt, depth_scale=wl.depth_scale, feat_scale=wl.feat_scale,
                            out=d_out[k], capacity=cap, out_scale=out_scale, feat_block=bb, stream=s_in)
            done = torch.cuda.Event()
            done.record(s_in)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done)
            h_out[k].copy_(d_out[k], non_blocking=True)
            read_done[k] = torch.cuda.Event()
            read_done[k].record(s_out)

    for i in range(3):
        frame(i)
    torch.cuda.synchronize()
    per_frame = []
    nxt = 3
    for _ in range(reps):                            # the median of `reps` timed runs of `frames` frames
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for i in range(nxt, nxt + frames):
            frame(i)
        nxt += frames
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
        b.record(stream)
        torch.cuda.synchronize()
        per_frame.append(a.elapsed_time(b) * 1e3 / frames)
    if not torch.equal(h_out[(nxt - 1) % nb], ref_out.cpu()):
        raise RuntimeError("pipelined e2e: the output read back differs from the device-timed forward's")
    return statistics.median(per_frame)


def device_inputs(wl, device):
    """Pinned host copies and device copies of a workload's depth, features and
    (NVFP4) block scales, as the raw bytes the C ABI takes."""
    import torch

    view = np.uint16 if wl.dtype == "f16" else np.uint8
    depth_h = torch.from_numpy(np.ascontiguousarray(wl.depth).reshape(-1).view(view).copy()).pin_memory()
    feat_h = torch.from_numpy(np.ascontiguousarray(wl.feat).reshape(-1).view(view).copy()).pin_memory()
    block_h = (torch.from_numpy(np.ascontiguousarray(wl.feat_block).reshape(-1).copy()).pin_memory()
               if wl.feat_block is not None else None)
    return (depth_h, feat_h, block_h, depth_h.to(device), feat_h.to(device),
            block_h.to(device) if block_h is not None else None)


def time_flushed(call, flush, stream, steps: int) -> list:
    """Device time (ms) of `steps` calls, each after an L2 flush, by CUDA
    events on `stream` around the call alone."""
    import torch

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    torch.cuda._sleep(20_000_000)            # let the host queue calls ahead of the GPU
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def graph_us(call, stream, calls: int = 100, reps: int = 10) -> float:
    """Median per-call time of a CUDA graph of `calls` back-to-back calls
    (warm L2 where the working set fits), replayed `reps` times."""
    import torch

    g_stream = torch.cuda.Stream()
    g_stream.wait_stream(stream)
    with torch.cuda.stream(g_stream):
        for _ in range(3):
            call()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=g_stream):
            for _ in range(calls):
                call()
    stream.wait_stream(g_stream)
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        out.append(a.elapsed_time(b) * 1e3 / calls)
    return statistics.median(out)


def l2_gather_roofline(bm: dict, time_us: float, probe: dict, time_note: str) -> dict:
    """The L2 roofline of the gather-level bytes (what the owners read and
    write at the L2) over a forward time, against the probe's copy bandwidth."""
    achieved = bm["gather"] / (time_us * 1e-6) / 1e9
    return {"bound": "l2", "achieved": achieved, "peak": probe["copy_gbs"], "unit": "GB/s",
            "frac": achieved / probe["copy_gbs"], "bytes_per_launch": bm["gather"], "time_us": time_us,
            "time": time_note, "peak_source": "bevpool_probe_l2 copy (read + write bytes), 64 MiB resident, this run"}


def dram_batch_forward(device, stream, flush, steps: int, probe=None) -> dict:
    """The DRAM-bound batch configuration (4 x canonical frustum, C = 128,
    [4, 512, 512, 128] output, ~334 MB of compulsory traffic, above the L2):
    its forward timed with L2 flushed before each call, and its HBM roofline."""
    import torch

    from depth_weighted_scatter_gb300 import bevpool, workloads

    wl = workloads.make("dram_batch")
    _, _, _, depth, feat, _ = device_inputs(wl, device)
    cells = torch.from_numpy(wl.cell_ids).to(device)
    m = bevpool.build_map(cells, *wl.dims(), wl.n_cells, sync=True)
    cap = (m.n_points, m.n_intervals)
    out = torch.empty((wl.n_cells, wl.C), dtype=torch.float16, device=device)
    call = lambda: bevpool.forward(m, depth, feat, wl.C, dtype=bevpool.BEVPOOL_F16, out=out, capacity=cap)
    for _ in range(3):
        flush.zero_()
        call()
    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    ms = time_flushed(call, flush, stream, steps)
    clocks = sampler.stop()
    back_to_back = graph_us(call, stream, calls=20, reps=5)
    bm = bytes_model(wl, m.n_points, m.n_intervals)
    us = statistics.mean(ms) * 1e3
    peak, peak_kind = measured_peaks()
    achieved = bm["footprint"] / (us * 1e-6) / 1e9
    roof_l2 = (l2_gather_roofline(bm, us, probe, "mean event time per call, L2 flushed before each")
               if probe is not None else None)
    return {"workload": f"{wl.name}: NC={wl.NC} D={wl.D} H={wl.H} W={wl.W} C={wl.C} grid={wl.grid} "
                        f"points={m.n_points} intervals={m.n_intervals}",
            "forward_us": us, "forward_us_median": statistics.median(ms) * 1e3, "calls": steps,
            "l2": "flushed (256 MiB written) before every call; the working set (334 MB) exceeds the L2",
            "forward_us_back_to_back_graph": back_to_back,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": recorded_traffic("dram_batch"), "kernel": "k_forward",
                         "bytes_per_launch": bm["footprint"],
                         "peak_source": f"hbm_gbs of MEASURED_PEAKS.json ({peak_kind})"},
            "roofline_l2_gather": roof_l2,
            "clocks": clocks}


def run_ours(args) -> None:
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)

    from depth_weighted_scatter_gb300 import bevpool, workloads

    wl = workloads.make(args.config)
    dt = {"f16": bevpool.BEVPOOL_F16, "e4m3": bevpool.BEVPOOL_E4M3, "nvfp4": bevpool.BEVPOOL_NVFP4}[wl.dtype]
    depth_h, feat_h, block_h, depth, feat, block = device_inputs(wl, device)
    cells = torch.from_numpy(wl.cell_ids).to(device)

    ws = bevpool.workspace_for(*wl.dims(), wl.n_cells, device)
    m = bevpool.ScatterMap.allocate(*wl.dims(), wl.n_cells, device)
    bevpool.build_map(cells, *wl.dims(), wl.n_cells, out=m, workspace=ws, sync=True)
    n_pts, n_int = m.n_points, m.n_intervals
    cap = (n_pts, n_int)
    e4m3_out = args.out_dtype == "e4m3"
    out_scale = None
    if e4m3_out:                                        # calibration (untimed): max|output| / 448
        probe = bevpool.forward(m, depth, feat, wl.C, dtype=dt, depth_scale=wl.depth_scale,
                                feat_scale=wl.feat_scale, capacity=cap, feat_block=block)
        out_scale = float(probe.float().abs().max().item()) / 448.0 or 1.0
        del probe
    out = torch.empty((wl.n_cells, wl.C), dtype=torch.uint8 if e4m3_out else torch.float16, device=device)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def fwd(o=out):
        bevpool.forward(m, depth, feat, wl.C, dtype=dt, depth_scale=wl.depth_scale, feat_scale=wl.feat_scale,
                        out=o, capacity=cap, out_scale=out_scale, feat_block=block)

    def build():
        bevpool.build_map(cells, *wl.dims(), wl.n_cells, out=m, workspace=ws, sync=False)

    if args.ncu_warm_calls:
        # for a profiler: forwards back to back, L2 warm (nothing between them), no timing
        for _ in range(args.ncu_warm_calls):
            fwd()
        torch.cuda.synchronize()
        return

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        build()
        flush.zero_()
        fwd()
    torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = bevpool.bevpool_kernel_launches()
    nvtx_push("timed")
    torch.cuda._sleep(20_000_000)            # let the host queue steps ahead of the GPU (outside every event pair)
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        build()
        ev[i][1].record(stream)
        flush.zero_()
        ev[i][2].record(stream)
        fwd()
        ev[i][3].record(stream)
    torch.cuda.synchronize()
    nvtx_pop()
    if world > 1:
        torch.distributed.barrier()
    launches = bevpool.bevpool_kernel_launches() - launches0
    clocks = sampler.stop()

    build_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    fwd_ms = [ev[i][2].elapsed_time(ev[i][3]) for i in range(args.steps)]
    fwd_mean, build_mean = statistics.mean(fwd_ms), statistics.mean(build_ms)
    fwd_mean, build_mean = max_over_ranks([fwd_mean, build_mean], world, device)

    # Correctness guard: the timed map must be the one built up front.
    counts = m.d_counts.cpu().tolist()
    if counts[0] != n_pts or counts[1] != n_int:
        raise RuntimeError(f"map counts changed during timing: {counts} vs {(n_pts, n_int)}")

    # Warm-L2 CUDA-graph replay of the forward (the pages' Table 1 method).
    try:
        warm_us = graph_us(fwd, stream)
    except Exception as e:  # graph capture is an extra, never the headline
        warm_us = f"unavailable: {type(e).__name__}"
    g_stream = torch.cuda.Stream()

    # One frame with its own geometry (bevpool_pool_frame: map build + forward,
    # no host sync) replayed from a CUDA graph, warm L2.
    frame_us = None
    if not e4m3_out and wl.dtype != "nvfp4":
        try:
            fm = bevpool.ScatterMap.allocate(*wl.dims(), wl.n_cells, device)
            fout = torch.empty_like(out)
            frame = lambda: bevpool.pool_frame(cells, depth, feat, *wl.dims(), wl.n_cells, wl.C, dtype=dt,
                                               depth_scale=wl.depth_scale, feat_scale=wl.feat_scale, out=fout,
                                               map_out=fm, workspace=ws, stream=g_stream)
            with torch.cuda.stream(g_stream):
                g_stream.wait_stream(stream)
                for _ in range(3):
                    frame()
                fgraph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(fgraph, stream=g_stream):
                    for _ in range(20):
                        frame()
            stream.wait_stream(g_stream)
            torch.cuda.synchronize()
            reps = []
            for _ in range(10):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fgraph.replay()
                b.record(stream)
                torch.cuda.synchronize()
                reps.append(a.elapsed_time(b) * 1e3 / 20)
            frame_us = statistics.median(reps)
        except Exception as e:
            frame_us = f"unavailable: {type(e).__name__}"

    # L2 roofline (working set resident in L2): the gather-level bytes of one
    # forward over the warm-L2 graph time, against the L2 copy bandwidth the
    # probe measures on this GPU in this run, and against the ncu ceiling of
    # the L2 for the same mix of reads and writes.
    roof_l2 = None
    l2_bytes = torch.cuda.get_device_properties(device).L2_cache_size
    bm0 = bytes_model(wl, n_pts, n_int, 1 if e4m3_out else 2)
    probe = l2_probe(device, stream)
    if bm0["footprint"] <= l2_bytes // 2 and isinstance(warm_us, float):
        achieved_l2 = bm0["gather"] / (warm_us * 1e-6) / 1e9
        rd, wr = bm0["gather"] - bm0["out"], bm0["out"]
        ceiling = (rd + wr) / (rd / NCU_L2_READ_GBS + wr / NCU_L2_WRITE_GBS)
        gather_probe = None
        row_bytes = wl.C // 2 if wl.dtype == "nvfp4" else wl.C * (2 if wl.dtype == "f16" else 1)
        if row_bytes % 16 == 0 and row_bytes <= 512 and n_pts > 0:
            # the forward's row gather alone over this map's ranks_feat (what its walk can reach)
            rows = m.ranks_feat[:n_pts]
            g_us = graph_us(lambda: bevpool.probe_gather(feat, row_bytes, rows, ctas_per_sm=3), stream, calls=20,
                            reps=5)
            gather_probe = {"time_us": g_us, "bytes": n_pts * row_bytes,
                            "gbs": n_pts * row_bytes / (g_us * 1e-6) / 1e9,
                            "what": "bevpool_probe_gather: the forward's feature-row gather alone (16-byte lanes, "
                                    "8 rows in flight, 3 CTAs per SM) over this map's ranks_feat, warm L2, "
                                    "CUDA-graph median per launch"}
        roof_l2 = {"bound": "l2", "achieved": achieved_l2, "peak": probe["copy_gbs"], "unit": "GB/s",
                   "frac": achieved_l2 / probe["copy_gbs"], "traffic": None, "kernel": "k_forward",
                   "bytes_per_launch": bm0["gather"], "time_us": warm_us,
                   "time": "warm-L2 CUDA-graph median per call (100 forwards back to back)",
                   "peak_source": "bevpool_probe_l2 copy (read + write bytes), 64 MiB resident, best of 5, "
                                  "this run",
                   "ncu_ceiling_gbs": ceiling, "frac_of_ncu_ceiling": achieved_l2 / ceiling,
                   "ncu_ceiling_source": "188 L2 slices x (2 read | 1 write) sectors of 32 B per cycle x "
                                         "1.979 GHz, weighted by this forward's read and write bytes",
                   "probe": probe, "gather_probe": gather_probe}

    dram_batch = None
    if wl.name == "canonical" and not args.no_dram_batch and not e4m3_out:
        dram_batch = dram_batch_forward(device, stream, flush, steps=max(3, min(args.steps, 50)), probe=probe)

    # End to end through the C ABI from pinned host buffers: every frame copies
    # its depth and features in, runs the forward and reads its output back.
    # Serial: one frame at a time on one stream, L2 flushed before each (the
    # latency of a frame).  Pipelined (the e2e value): two buffer sets, frame
    # i's output read on a second stream while frame i + 1's inputs are copied
    # in and its forward runs; time per frame = the loop's time / frames.
    out_h = torch.empty((wl.n_cells, wl.C), dtype=out.dtype).pin_memory()
    e2e_steps = min(args.steps, 200)
    e2e_ms = []
    for i in range(e2e_steps + 3):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        depth.copy_(depth_h, non_blocking=True)
        feat.copy_(feat_h, non_blocking=True)
        if block is not None:
            block.copy_(block_h, non_blocking=True)
        fwd()
        out_h.copy_(out, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            e2e_ms.append(a.elapsed_time(b))
    e2e_serial_us = max_over_ranks([statistics.mean(e2e_ms) * 1e3], world, device)[0]
    e2e_us = max_over_ranks([pipelined_e2e_us(bevpool, m, wl, dt, cap, out_scale, out, depth_h, feat_h, block_h,
                                              e2e_steps, stream)], world, device)[0]
    h2d = depth_h.numel() * depth_h.element_size() + feat_h.numel() * feat_h.element_size()
    if block_h is not None:
        h2d += block_h.numel()
    d2h = out_h.numel() * out_h.element_size()

    if rank != 0:
        return
    bm = bytes_model(wl, n_pts, n_int, 1 if e4m3_out else 2)
    traffic_key = wl.name + ("_e4m3out" if e4m3_out else "")
    peak, peak_kind = measured_peaks()
    fwd_s = fwd_mean / 1e3
    achieved = bm["footprint"] / fwd_s / 1e9
    roof_hbm = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": recorded_traffic(traffic_key), "kernel": "k_forward", "bytes_per_launch": bm["footprint"],
                "time_us": fwd_mean * 1e3, "time": "mean event time per call, L2 flushed before each",
                "peak_source": f"hbm_gbs of MEASURED_PEAKS.json ({peak_kind})"}
    if roof_l2 is not None:
        roof_l2["traffic"] = roof_hbm["traffic"]
        roof_l2["traffic_note"] = "DRAM bytes of one launch with caches flushed (ncu); l2_traffic: L2 bytes of a warm launch"
        roof_l2["l2_traffic"] = recorded_traffic(traffic_key, "l2_bytes_warm")
    line = {
        "metric": METRIC,
        "value": fwd_mean * 1e3,
        "unit": "us/call",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": build_mean + fwd_mean,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype + ("->e4m3" if e4m3_out else ""),
        "data": "synthetic (seeded generator shaped like the pages' workload; nuScenes not used)",
        "config": config_dict(wl, n_pts, n_int, world, args.out_dtype),
        "roofline": roof_l2 if roof_l2 is not None else roof_hbm,
        "roofline_hbm": roof_hbm,
        "roofline_l2_gather": (l2_gather_roofline(bm, fwd_mean * 1e3, probe, "mean event time per call, L2 flushed "
                                                  "before each (the working set exceeds half the L2)")
                               if roof_l2 is None else None),
        "dram_batch": dram_batch,
        "cpu_baseline": (cpu_oracle_time(wl, out_scale=out_scale)
                         if (world == 1 and not args.no_cpu_baseline) else None),
        "e2e": {"value": e2e_us, "unit": "us/call", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "mode": "pipelined: two frames in flight, one frame's D2H overlapping the next one's H2D and forward",
                "serial_us": e2e_serial_us},
        "gpu_launches": launches,
        "clocks": clocks,
        "extra": {
            "forward_us_median": statistics.median(fwd_ms) * 1e3,
            "build_map_us": build_mean * 1e3,
            "forward_us_warm_l2_graph": warm_us,
            "frame_us_warm_l2_graph": frame_us,
            "gather_bytes": bm["gather"],
            "gather_gbs_cold": bm["gather"] / fwd_s / 1e9,
            "gather_gbs_warm": (bm["gather"] / (warm_us * 1e-6) / 1e9) if isinstance(warm_us, float) else None,
            "bytes_model": bm,
            "forward_source_hash": forward_source_hash(),
            "pages_context_us": {"v3_fp16_rtx_pro_6000": 17.3, "v3_fp8_rtx_pro_6000": 16.4,
                                 "v2_fp16_rtx_pro_6000": 274.0, "v3_fp16_a6000_dram_tuned": 90.0},
        },
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    from depth_weighted_scatter_gb300 import workloads

    ap.add_argument("--config", default="canonical", choices=workloads.ALL_NAMES)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dram-batch", action="store_true",
                    help="canonical runs: skip timing the DRAM-bound batch configuration beside it")
    ap.add_argument("--ncu-warm-calls", type=int, default=0,
                    help="for a profiler: run this many forwards back to back (L2 warm), print nothing, exit")
    ap.add_argument("--out-dtype", choices=["f16", "e4m3"], default="f16",
                    help="output of the forward: fp16, or E4M3 codes (bevpool_forward_e4m3_out)")
    args = ap.parse_args()
    if args.impl == "reference":
        # each reference step is one full oracle forward (~80 ms canonical, ~1 s
        # for the DRAM batch): run_reference caps the step count so the timed
        # steps take at most REFERENCE_BUDGET_S; the warm-up count is the one given
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
