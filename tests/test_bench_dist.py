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
