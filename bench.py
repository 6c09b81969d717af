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
PROFILE = os.path.join(ROOT, "profiles", "frames_kernel_c4.md")
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
    """Per-launch DRAM bytes from the committed ncu summary, or None when the
    summary is missing or was taken on other kernel sources."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    h = re.search(r"kernel_sources_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != kernel_hash():
        return None
    return int(m.group(1))


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
    repeated until about target_s of wall time (bounded sample)."""
    import oracle
    threads = os.cpu_count() or 1
    n = min(threads, ref.shape[0])
    sub_r, sub_d = np.ascontiguousarray(ref[:n]), np.ascontiguousarray(dis[:n])
    oracle.batch(sub_r[:1], sub_d[:1], bpc, threads=1)  # warm (build, page-in)
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.batch(sub_r, sub_d, bpc, threads=threads)
        done += n
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    return {"value": done / el, "unit": "frames/s", "cores": min(threads, n), "kind": "oracle",
            "sample": f"{done} frame computations (float_moment + float_psnr) of the first {n} "
                      f"frames of the workload, {min(threads, n)} threads, {el:.1f} s wall"}


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
    # of `depth` calls (api.FrameGraph; 16 when the step count allows), each
    # kernel launched to overlap the one before it, as a stream of batches
    # runs; every call does the whole work on its own workspace and outputs.
    depth = next(d for d in (16, 8, 4, 2, 1) if args.steps % d == 0)
    fg = api.FrameGraph(ref, dis, wl.bpc, features=3, depth=depth)
    stream = torch.cuda.current_stream(dev)
    kernels_per_step = 1

    def replay():
        return fg.replay()

    for _ in range(max(args.warmup, 3)):
        replay()
    torch.cuda.synchronize()
    assert fg.status() == 0, "bounded device wait gave up"

    replays = args.steps // depth
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(replays)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(replays)]

    with Clocks(local_rank) as clocks:
        if pg is not None:
            dist.barrier(group=pg)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(replays):
            starts[i].record(stream)
            replay()
            ends[i].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        if pg is not None:
            dist.barrier(group=pg)
    launches = kernels_per_step * args.steps  # graph replays: one kernel each
    assert fg.status() == 0, "bounded device wait gave up"
    per = [s.elapsed_time(e) / depth for s, e in zip(starts, ends)]  # ms per call
    device_ms = max_over_ranks(starts[0].elapsed_time(ends[-1]), pg)
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
    if rank != 0:
        return

    bytes_per_launch = F * wl.frame_pair_bytes
    avg_ms = statistics.mean(per)
    achieved = bytes_per_launch / (avg_ms / 1e3) / 1e9
    peak, peak_kind = peak_hbm()
    line = {
        "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": device_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u64", "data": "synthetic",
        "config": dict(config(wl, F), parallelism=f"replicas x{world}"),
        "hbm_gbs": bytes_per_launch * args.steps / (device_ms / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(),
                     "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "kernel": "frames_kernel (one launch per step)",
                     "algorithmic_bytes_per_launch": bytes_per_launch,
                     "avg_launch_ms": avg_ms},
        "e2e": {"value": whole_job_rate(world, F, 1, e2e_s), "unit": "frames/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "clocks": clocks.summary(),
        "wall_s": wall,
    }
    line["cpu_baseline"] = cpu_baseline(ref_h, dis_h, wl.bpc, target_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)


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
    for key in ("C1", "C2", "C3", "C4", "C5a", "C5b", "C5c"):
        wl = synth.WORKLOADS[key]
        ref, dis = wl.batch()
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
            "bit_exact_frames_checked": n, "bit_exact": exact and status == 0}), flush=True)
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
