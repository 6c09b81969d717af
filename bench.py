"""Benchmark: frames/s and achieved HBM GB/s of bit-exact float_moment +
float_psnr on 16-bit 3840x2160 frame pairs (one fused call per step).

python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference]

A step is one pass of the whole path (exact row sums, look-back, runs, walk,
finalisation for both features) over one batch of 16 seeded synthetic frame
pairs already resident in HBM: one library call on its own workspace and
outputs. Steps run as a stream of batches does: CUDA graphs of sixteen calls
(api.FrameGraph), the workspaces cleared first and each kernel launched to
overlap the one before it (programmatic dependent launch). The
batch (531 MB) is larger than L2. Under
torchrun every rank runs its own batch on its own GPU (frames shard with no
collective; weak scaling); rank 0 prints one JSON line. ``--impl
reference`` times the CPU oracle on the host cores instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "frames/s and achieved HBM GB/s (fraction of peak), 16-bit 3840x2160, bit-exact"
WORKLOAD = "C4"
PROFILE = os.path.join(ROOT, "profiles", "frames_kernel_c4.json")
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, the vendor's figure (context only)
GRAPH_DEPTH = 16          # calls per graph replay in the timed stream of batches, at least


def graph_plan(steps: int):
    """Depths of the graphs that K steps run as: as many graphs as hold at
    least GRAPH_DEPTH calls each, the steps shared out evenly (so every graph
    holds 16 to 31 calls once K >= 16), or one graph of K calls below that."""
    if steps < GRAPH_DEPTH:
        return [steps]
    n = steps // GRAPH_DEPTH
    base, extra = divmod(steps, n)
    return [base + 1] * extra + [base] * (n - extra)
KERNEL_SOURCES = [os.path.join(ROOT, "exact_reductions_gb300", "csrc", f)
                  for f in ("vmx_kernels.cu", "ordsum.cuh", "vmx_internal.h")]


def kernel_hash() -> str:
    """Hash of the kernel sources' code: comments and whitespace stripped,
    so that a comment edit does not retire the profiled traffic."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def profiled_traffic():
    """Per-launch DRAM bytes from the committed ncu summary (a small JSON
    record beside its text), or None when it is missing or was taken on other
    kernel sources."""
    try:
        with open(PROFILE) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_sources_sha256_16") != kernel_hash():
        return None
    v = rec.get("traffic_bytes_per_launch")
    return int(v) if isinstance(v, int) else None


def host_cpu():
    """The host's CPU model and machine name, as the system reports them."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as fh:
                for line in fh:
                    if line.lower().startswith(("model name", "cpu part")):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"cpu_model": model or platform.processor() or "unknown",
            "uname_m": platform.machine()}


class Clocks:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        with open(self.file.name) as fh:
            rows = [r.split(",") for r in fh.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() in ("active", "1"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def frame_indices(rank: int, frames: int) -> range:
    """Rank r takes frames r*F .. r*F+F-1 of the workload's seeded stream."""
    return range(rank * frames, (rank + 1) * frames)


def max_over_ranks(x: float, pg) -> float:
    """The largest x over the ranks of pg (x itself when pg is None)."""
    if pg is None:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=pg)
    return float(t[0])


def whole_job_rate(world: int, frames_per_rank: int, steps: int, seconds: float) -> float:
    """Frames of all ranks over the slowest rank's time."""
    return world * frames_per_rank * steps / seconds


def make_batch(rank: int):
    from exact_reductions_gb300 import synth
    wl = synth.WORKLOADS[WORKLOAD]
    F = wl.frames
    ref = np.empty((F, wl.height, wl.width), dtype=np.uint16)
    dis = np.empty_like(ref)
    for i, f in enumerate(frame_indices(rank, F)):
        ref[i], dis[i] = wl.frame(f)
    return wl, ref, dis


def cpu_baseline(ref, dis, bpc, target_s: float = 2.0):
    """The oracle, as it stands, on the host cores: one frame per thread,
    repeated until about target_s of wall time (bounded sample); then one
    frame on one core, five times (median). Returns the baseline record and
    the oracle's results of the frames it computed (moments, mse, psnr_rows)."""
    import oracle
    threads = os.cpu_count() or 1
    n = min(threads, ref.shape[0])
    sub_r, sub_d = np.ascontiguousarray(ref[:n]), np.ascontiguousarray(dis[:n])
    oracle.batch(sub_r[:1], sub_d[:1], bpc, threads=1)  # warm (build, page-in)
    done, t0 = 0, time.perf_counter()
    while True:
        want = oracle.batch(sub_r, sub_d, bpc, threads=threads)
        done += n
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    one = []
    for _ in range(5):
        t1 = time.perf_counter()
        oracle.batch(sub_r[:1], sub_d[:1], bpc, threads=1)
        one.append(time.perf_counter() - t1)
    rec = {"value": done / el, "unit": "frames/s", "cores": min(threads, n), "kind": "oracle",
           "sample": f"{done} frame computations (float_moment + float_psnr) of the first {n} "
                     f"frames of the workload, {min(threads, n)} threads, {el:.1f} s wall",
           "single_thread_ms_per_frame": 1e3 * statistics.median(one),
           "single_thread_sample": "frame 0, one thread, median of 5",
           "pages_cpu_ms_per_frame": 17.0,
           "pages_cpu_note": "the pages' CPU extractor on their unnamed host, 16-bit 3840x2160 "
                             "(context only)"}
    rec.update(host_cpu())
    return rec, want


def oracle_accumulators(ref, dis, bpc, frames):
    """The oracle's rounded accumulators in units (second moments of ref and
    dis, psnr noise) of the given frames, one frame per thread."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    def one(f):
        s = oracle.moment_sums(ref[f], dis[f], bpc)
        return (s[2], s[3]), oracle.psnr_noise_sum(ref[f], dis[f], bpc)

    with ThreadPoolExecutor(max_workers=min(len(frames), os.cpu_count() or 1)) as ex:
        res = list(ex.map(one, frames))
    return (np.array([r[0] for r in res], dtype=np.uint64),
            np.array([r[1] for r in res], dtype=np.uint64))


def timed_outputs_exact(outs, want, s2_want, noise_want) -> bool:
    """Every output of the timed calls equal, bit for bit, to the oracle's:
    the last call's moments, MSE, psnr row sums and accumulators against the
    oracle, and every other call's outputs against the last call's."""
    import torch

    def u64(t):
        return t.cpu().view(torch.int64).numpy().view(np.uint64)

    last = outs[-1]
    n = want["moments"].shape[0]
    ok = (np.array_equal(last["moments"].cpu().numpy()[:n].view(np.uint64),
                         want["moments"].view(np.uint64)) and
          np.array_equal(last["mse"].cpu().numpy()[:n].view(np.uint64), want["mse"].view(np.uint64)) and
          np.array_equal(u64(last["psnr_rows"])[:n], want["psnr_rows"]) and
          np.array_equal(u64(last["s2_sums"])[:n], s2_want) and
          np.array_equal(u64(last["noise_sums"])[:n], noise_want))
    def bits(t):
        return t.view(torch.int64)  # doubles and uint64 compared as their bits

    for o in outs[:-1]:
        ok = ok and all(torch.equal(bits(o[k]), bits(last[k])) for k in last)
    return bool(ok)


def h2d_rate(pinned, dev, reps: int = 5) -> float:
    """Page-locked host to device copy rate (GB/s) of one batch, best of reps."""
    import torch
    dst = torch.empty(pinned.shape, dtype=pinned.dtype, device=dev)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = 0.0
    for _ in range(reps):
        s.record()
        dst.copy_(pinned, non_blocking=True)
        e.record()
        torch.cuda.synchronize()
        best = max(best, pinned.numel() * pinned.element_size() / (s.elapsed_time(e) / 1e3) / 1e9)
    return best


def run_reference(args, rank, world, budget_s: float = 150.0):
    """The oracle on the host cores, as it stands. Each step computes the
    first m rows of n frames (one frame per thread); m is chosen so that
    warm-up plus the timed steps take about budget_s. Throughput is counted
    in frame equivalents (rows / height)."""
    from exact_reductions_gb300 import synth
    if rank != 0:
        return
    import oracle
    wl = synth.WORKLOADS[WORKLOAD]
    threads = os.cpu_count() or 1
    n = min(threads, wl.frames)
    ref = np.stack([wl.frame(f)[0] for f in range(n)])
    dis = np.stack([wl.frame(f)[1] for f in range(n)])
    oracle.batch(ref[:1], dis[:1], wl.bpc, threads=1)  # build and page in
    t0 = time.perf_counter()
    oracle.batch(ref, dis, wl.bpc, threads=threads)
    full_step = time.perf_counter() - t0
    per_step = budget_s / max(1, args.steps + args.warmup)
    m = max(1, min(wl.height, int(wl.height * per_step / max(full_step, 1e-9))))
    sub_r = np.ascontiguousarray(ref[:, :m, :])
    sub_d = np.ascontiguousarray(dis[:, :m, :])
    for _ in range(args.warmup):
        oracle.batch(sub_r, sub_d, wl.bpc, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.batch(sub_r, sub_d, wl.bpc, threads=threads)
    el = time.perf_counter() - t0
    value = n * (m / wl.height) * args.steps / el
    sample = (f"each step: rows 0..{m - 1} of the first {n} frames of the workload "
              f"(float_moment + float_psnr, one frame per thread); frames counted as rows / "
              f"{wl.height}")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "frames/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config(wl, wl.frames),
        "cpu_baseline": {"value": value, "unit": "frames/s", "cores": n, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "frames/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config(wl, frames):
    return {"workload": f"{wl.name}: {frames} frame pairs, 16-bit {wl.width}x{wl.height} "
                        f"full-range uniform noise (seed {wl.seed})",
            "frames_per_gpu": frames, "width": wl.width, "height": wl.height, "bpc": wl.bpc,
            "features": "float_moment + float_psnr (fused)",
            "l2": f"inputs larger than L2 ({frames * wl.frame_pair_bytes / 1e6:.1f} MB per step)"}


def run_ours(args, rank, local_rank, world, pg):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    from exact_reductions_gb300 import api

    __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl, ref_h, dis_h = make_batch(rank)
    F = ref_h.shape[0]
    ref = torch.from_numpy(ref_h).to(dev)
    dis = torch.from_numpy(dis_h).to(dev)
    # The step: one fused call on the resident batch. Steps go in CUDA graphs
    # of 16 to 31 calls each (api.FrameGraph; graph_plan), each kernel
    # launched to overlap the one before it, as a stream of batches runs;
    # every call does the whole work on its own workspace and outputs.
    plan = graph_plan(args.steps)
    depths = sorted(set(plan), reverse=True)
    made = {d: api.FrameGraph(ref, dis, wl.bpc, features=3, depth=d, sums=True) for d in depths}
    graphs = [(made[d], plan.count(d)) for d in depths]
    stream = torch.cuda.current_stream(dev)
    kernels_per_step = 1

    schedule = [fg for fg, n in graphs for _ in range(n)]
    starts = [torch.cuda.Event(enable_timing=True) for _ in schedule]
    ends = [torch.cuda.Event(enable_timing=True) for _ in schedule]

    with Clocks(local_rank) as clocks:
        # The warm-up runs once the clock sampler is up, so that the timed
        # steps start on a busy GPU rather than after its pause.
        for _ in range(max(args.warmup, 3)):
            for fg, _ in graphs:
                fg.replay()
        torch.cuda.synchronize()
        assert all(fg.status() == 0 for fg, _ in graphs), "bounded device wait gave up"
        if pg is not None:
            dist.barrier(group=pg)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i, fg in enumerate(schedule):
            starts[i].record(stream)
            fg.replay()
            ends[i].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        if pg is not None:
            dist.barrier(group=pg)
    launches = kernels_per_step * args.steps  # graph replays: one kernel per call
    assert all(fg.status() == 0 for fg, _ in graphs), "bounded device wait gave up"
    last_outs = schedule[-1].outs  # the outputs of the last replay's calls
    device_ms = max_over_ranks(starts[0].elapsed_time(ends[-1]), pg)
    per_call_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps
    value = whole_job_rate(world, F, args.steps, device_ms / 1e3)

    # End to end through the host-memory entry point: pinned host frames in
    # (read in place by the kernel over the host link), results out, all
    # inside the timed call; one launch for the 16 frames.
    pin_r = torch.from_numpy(ref_h).pin_memory()
    pin_d = torch.from_numpy(dis_h).pin_memory()
    e2e_steps = max(1, min(args.steps, 10))
    hws = api.workspace(api.host_workspace_bytes(wl.width, wl.height, wl.width * 2, wl.bpc, F, 3),
                        dev)
    out = api.frames_host(pin_r.numpy(), pin_d.numpy(), wl.bpc, features=3, chunk_frames=F, ws=hws)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    for _ in range(e2e_steps):
        out = api.frames_host(pin_r.numpy(), pin_d.numpy(), wl.bpc, features=3, chunk_frames=F,
                              ws=hws)
    e2e_s = max_over_ranks((time.perf_counter() - t1) / e2e_steps, pg)
    h2d, d2h = api.host_traffic(wl.width, wl.height, wl.width * 2, wl.bpc, F, 3)
    link_gbs = h2d_rate(pin_r, dev)
    if rank != 0:
        return

    bytes_per_launch = F * wl.frame_pair_bytes
    avg_ms = per_call_ms
    achieved = bytes_per_launch / (avg_ms / 1e3) / 1e9
    peak, peak_kind = peak_hbm()
    e2e_value = whole_job_rate(world, F, 1, e2e_s)
    line = {
        "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": device_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u64", "data": "synthetic",
        "config": dict(config(wl, F), parallelism=f"replicas x{world}",
                       mode="stream of batches: " + ", ".join(
                           f"{plan.count(d)} CUDA graph(s) of {d} overlapping calls" for d in depths)),
        "hbm_gbs": bytes_per_launch * args.steps / (device_ms / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(),
                     "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "frac_nominal": achieved / NOMINAL_HBM_GBS,
                     "peak_nominal": NOMINAL_HBM_GBS,
                     "nominal_source": "nominal: GB300 HBM3e spec bandwidth",
                     "kernel": "frames_kernel (one launch per step)",
                     "algorithmic_bytes_per_launch": bytes_per_launch,
                     "avg_launch_ms": avg_ms},
        "e2e": {"value": e2e_value, "unit": "frames/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "host_link_h2d_gbs": link_gbs,
                "frac_of_host_link": e2e_value * wl.frame_pair_bytes / 1e9 / link_gbs,
                "host_link_source": "page-locked host to device copy of the batch, best of 5, "
                                    "same run"},
        "gpu_launches": int(launches),
        "clocks": clocks.summary(),
        "wall_s": wall,
    }
    base, want = cpu_baseline(ref_h, dis_h, wl.bpc, target_s=args.cpu_seconds)
    line["cpu_baseline"] = base
    n = want["moments"].shape[0]
    s2_want, noise_want = oracle_accumulators(ref_h, dis_h, wl.bpc, list(range(n)))
    exact = timed_outputs_exact(last_outs, want, s2_want, noise_want)
    line["bit_exact"] = exact
    line["frames_checked"] = n
    line["bit_exact_note"] = (f"the last timed replay's {len(last_outs)} calls: every output of the "
                              f"last call (moments, MSE, psnr row sums, second-moment and noise "
                              f"accumulators) of frames 0..{n - 1} equal to the oracle's bit for "
                              f"bit, and every call's outputs equal to the last call's")
    print(json.dumps(line), flush=True)
    if not exact:
        raise SystemExit("bench: the timed outputs differ from the oracle")


def phase_split(R, D, bpc):
    """Where one call's time goes, from the timing build of the library
    (VMX_PHASE_TIMES=1, vmx_phase_times): warp-microseconds per phase summed
    over the warps (SM cycles at the device's clock rate), and when the warps
    ran out of items and the walks ended, from the first warp's start."""
    import torch

    from exact_reductions_gb300 import _lib, api, build

    with _lib.using(build.build_variant("phase_times", ["VMX_PHASE_TIMES=1"])) as lib:
        out = api.frames(R, D, bpc, features=3)  # the first call allocates
        torch.cuda.synchronize()
        _lib.check(lib.vmx_phase_times(None, 1), "phase times")
        api.frames(R, D, bpc, features=3, ws=out["_workspace"])
        torch.cuda.synchronize()
        c = np.zeros(16, dtype=np.uint64)
        _lib.check(lib.vmx_phase_times(c.ctypes.data, 1), "phase times")
    c = [int(x) for x in c]
    mhz = c[15] / 1e3
    t0 = c[0]
    return {
        "span_us": (c[1] - t0) / 1e3,
        "first_warp_out_of_items_us": (c[7] - t0) / 1e3,
        "last_warp_out_of_items_us": (c[6] - t0) / 1e3,
        "last_walk_end_us": (c[9] - t0) / 1e3 if c[10] else None,
        "warp_us": {"streaming": c[2] / mhz, "look_back": c[3] / mhz, "plans_and_runs": c[4] / mhz,
                    "completion": c[5] / mhz, "walks": c[8] / mhz},
        "items": c[11], "row_runs": c[14], "walks": c[10],
        "longest_walk_us": c[12] / mhz,
        "clock_note": f"cycles at the device's {mhz:.0f} MHz clock rate",
    }


def run_configs(args):
    """One JSON line per workload (C1..C5c): GPU frames/s and GB/s with
    inputs resident (calls one at a time, and as a stream of batches), the
    oracle on the host cores (one core, and all cores one frame per thread),
    and whether the GPU outputs equal the oracle's on the frames the oracle
    computed."""
    import torch

    import __graft_entry__
    import oracle
    from exact_reductions_gb300 import api, synth

    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    peak, peak_kind = peak_hbm()
    threads = os.cpu_count() or 1
    keys = ("C1", "C2", "C3", "C4", "C5a", "C5b", "C5c")
    if args.only:
        keys = [k for k in keys if k in args.only.split(",")]
    for key in keys:
        wl = synth.WORKLOADS[key]
        ref, dis = wl.batch(args.frames) if args.frames > 0 else wl.batch()
        F = ref.shape[0]
        R = torch.from_numpy(ref).to(dev)
        D = torch.from_numpy(dis).to(dev)
        out = api.frames(R, D, wl.bpc, features=3)
        ws = out["_workspace"]
        for _ in range(3):
            out = api.frames(R, D, wl.bpc, features=3, ws=ws)
        torch.cuda.synchronize()
        reps = args.steps if args.steps < 50 else 20
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):  # back to back, as a stream of batches runs
            out = api.frames(R, D, wl.bpc, features=3, ws=ws)
        e.record()
        torch.cuda.synchronize()
        t = s.elapsed_time(e) / 1e3 / reps
        status = api.workspace_status(ws)
        walk = [int(x) for x in api.workspace_stats(ws)]  # the last call's walks
        split = phase_split(R, D, wl.bpc) if args.phase_times else None
        # The same calls as a stream of batches: graphs of sixteen calls,
        # each kernel overlapping the one before (the bench's mode).
        fg = api.FrameGraph(R, D, wl.bpc, features=3, depth=16)
        for _ in range(2):
            fg.replay()
        torch.cuda.synchronize()
        greps = max(1, reps // 4)
        s.record()
        for _ in range(greps):
            fg.replay()
        e.record()
        torch.cuda.synchronize()
        tg = s.elapsed_time(e) / 1e3 / (16 * greps)
        status = status or fg.status()
        del fg
        got_m = out["moments"].cpu().numpy()
        got_mse = out["mse"].cpu().numpy()
        # The oracle: one frame on one core, then min(cores, F) frames at once.
        n1 = 1
        t0 = time.perf_counter()
        oracle.batch(ref[:n1], dis[:n1], wl.bpc, threads=1)
        one_core = (time.perf_counter() - t0) / n1
        n = min(threads, F)
        t0 = time.perf_counter()
        want = oracle.batch(ref[:n], dis[:n], wl.bpc, threads=threads)
        all_cores = n / (time.perf_counter() - t0)
        exact = bool(np.array_equal(want["moments"].view(np.uint64), got_m[:n].view(np.uint64)) and
                     np.array_equal(want["mse"].view(np.uint64), got_mse[:n].view(np.uint64)))
        gbs = F * wl.frame_pair_bytes / t / 1e9
        print(json.dumps({
            "workload": f"{key}: {F} x {wl.width}x{wl.height} {wl.bpc}-bit", "frames_per_s": F / t,
            "ms_per_call": t * 1e3, "gb_per_s": gbs, "frac_of_peak": gbs / peak,
            "peak": f"{peak} GB/s ({peak_kind})",
            "stream_frames_per_s": F / tg, "stream_frac_of_peak": F * wl.frame_pair_bytes / tg / 1e9 / peak,
            "oracle_ms_per_frame_1core": one_core * 1e3,
            "oracle_frames_per_s_all_cores": all_cores, "oracle_cores": min(threads, n),
            "bit_exact_frames_checked": n, "bit_exact": exact and status == 0,
            "walk_rows": {"exact": walk[0], "closed_form_or_run": walk[1], "by_terms": walk[2],
                          "search_passes": walk[3]},
            **({"phase_times": split} if split else {})}), flush=True)
        del R, D, out, ws
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--configs", action="store_true",
                    help="one line per workload C1..C5c (GPU, oracle, bit-exactness) instead")
    ap.add_argument("--only", default="",
                    help="with --configs: these workloads only (comma-separated, e.g. C4,C5c)")
    ap.add_argument("--frames", type=int, default=0,
                    help="with --configs: frame pairs per call instead of each workload's own")
    ap.add_argument("--phase-times", action="store_true",
                    help="with --configs: add where one call's warp time goes (a timing build)")
    args = ap.parse_args()
    if args.configs:
        run_configs(args)
        return
    rank, local_rank, world = dist_env()
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist.group.WORLD
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, local_rank, world, pg)
    if pg is not None:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
