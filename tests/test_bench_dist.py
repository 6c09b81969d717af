"""bench.py's multi-rank host logic on CPU: two gloo ranks (no GPU).

Each rank takes its own frames of the seeded stream, the ranks agree on the
slowest rank's time, the whole-job rate counts every rank's frames, and the
reference arm runs on rank 0 only.
"""

import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    pg = dist.group.WORLD
    slowest = bench.max_over_ranks(1.5 + rank, pg)
    frames = list(bench.frame_indices(rank, 16))

    class Args:
        steps, warmup, gpus = 3, 3, world

    returned = bench.run_reference(Args, rank, world) if rank != 0 else None
    dist.barrier(group=pg)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as fh:
        json.dump({"slowest": slowest, "frames": frames, "returned": returned}, fh)


def test_two_gloo_ranks(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    # Both ranks see the slowest rank's time.
    assert res[0]["slowest"] == res[1]["slowest"] == 2.5
    # Disjoint, contiguous frames of the one seeded stream.
    assert res[0]["frames"] == list(range(0, 16))
    assert res[1]["frames"] == list(range(16, 32))
    # The reference arm returns at once on ranks other than 0.
    assert res[1]["returned"] is None


def test_whole_job_rate():
    sys.path.insert(0, ROOT)
    import bench
    # Two ranks, 16 frames each, 10 steps, slowest rank 0.5 s: 640 frames/s.
    assert bench.whole_job_rate(2, 16, 10, 0.5) == 640.0
    assert bench.max_over_ranks(3.25, None) == 3.25


def test_kernel_hash_ignores_comments(tmp_path, monkeypatch):
    """The profiled traffic stays keyed to the kernel code: a comment or
    whitespace edit keeps the hash, a code edit changes it."""
    sys.path.insert(0, ROOT)
    import bench
    src = tmp_path / "k.cu"
    src.write_text("int f(int x) { return x + 1; }  // one\n/* two */\n")
    monkeypatch.setattr(bench, "KERNEL_SOURCES", [str(src)])
    h0 = bench.kernel_hash()
    src.write_text("// a new comment\nint f(int x)\n{\n    return x + 1;  /* same code */\n}\n")
    assert bench.kernel_hash() == h0
    src.write_text("int f(int x) { return x + 2; }\n")
    assert bench.kernel_hash() != h0


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the keys the benchmark contract names."""
    import subprocess
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--steps", "3", "--warmup", "3"], capture_output=True, text=True,
                          timeout=600, cwd=ROOT)
    assert proc.returncode == 0, proc.stderr[-2000:]
    lines = [l for l in proc.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_profiled_traffic_reads_the_json_record(tmp_path, monkeypatch):
    """roofline.traffic comes from the JSON record beside the ncu summary,
    and only while its source hash matches the kernel code."""
    sys.path.insert(0, ROOT)
    import bench
    rec = tmp_path / "k.json"
    monkeypatch.setattr(bench, "PROFILE", str(rec))
    assert bench.profiled_traffic() is None  # no record
    rec.write_text(json.dumps({"traffic_bytes_per_launch": 538512128,
                               "kernel_sources_sha256_16": bench.kernel_hash()}))
    assert bench.profiled_traffic() == 538512128
    rec.write_text(json.dumps({"traffic_bytes_per_launch": 538512128,
                               "kernel_sources_sha256_16": "0" * 16}))
    assert bench.profiled_traffic() is None  # taken on other sources
    rec.write_text("not json")
    assert bench.profiled_traffic() is None


def test_host_cpu_names_the_machine():
    sys.path.insert(0, ROOT)
    import platform

    import bench
    d = bench.host_cpu()
    assert d["uname_m"] == platform.machine() and d["cpu_model"]


def test_timed_outputs_check_catches_one_flipped_bit():
    """The bench's exactness check compares the timed calls' outputs with the
    oracle's bit for bit: a single changed bit in any output, or a call that
    differs from the last, fails it (CPU tensors stand in for the device's)."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch

    import bench
    import oracle
    from exact_reductions_gb300 import synth
    wl = synth.WORKLOADS["T1"]
    ref, dis = wl.batch(1)
    ref, dis = ref[:, :64, :256].copy(), dis[:, :64, :256].copy()
    want = oracle.batch(ref, dis, 16, threads=1)
    s2, noise = bench.oracle_accumulators(ref, dis, 16, [0])

    def as_u64(a):
        return torch.from_numpy(np.array(a, copy=True).view(np.int64)).view(torch.uint64)

    def outs():
        return {"moments": torch.from_numpy(want["moments"].copy()),
                "mse": torch.from_numpy(want["mse"].copy()),
                "psnr_rows": as_u64(want["psnr_rows"]), "s2_sums": as_u64(s2),
                "noise_sums": as_u64(noise)}

    good = [outs(), outs()]
    assert bench.timed_outputs_exact(good, want, s2, noise)
    for key in ("moments", "mse", "psnr_rows", "s2_sums", "noise_sums"):
        bad = [outs(), outs()]
        v = bad[-1][key].view(torch.int64).view(-1)
        v[0] ^= 1
        assert not bench.timed_outputs_exact(bad, want, s2, noise), key
        first = [outs(), outs()]
        w = first[0][key].view(torch.int64).view(-1)
        w[0] ^= 1
        assert not bench.timed_outputs_exact(first, want, s2, noise), key


def test_graph_plan_keeps_every_graph_at_least_sixteen_deep():
    """Every step count of 16 or more runs as graphs of 16 to 31 calls (the
    same mode for the driver's 20 steps and a long run); fewer steps run as
    one graph."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.graph_plan(20) == [20]
    assert bench.graph_plan(2000) == [16] * 125
    assert bench.graph_plan(35) == [18, 17]
    assert bench.graph_plan(5) == [5]
    for k in range(1, 400):
        plan = bench.graph_plan(k)
        assert sum(plan) == k
        if k >= 16:
            assert all(16 <= d <= 31 for d in plan), (k, plan)
