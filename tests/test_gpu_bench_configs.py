"""`bench.py --configs` on the two smallest workloads, restricted with
--only and --frames, with --phase-times: one JSON line per workload, the
GPU doubles bit-exact against the oracle, and a phase split that accounts
for the call (its items, its walks, warp time in streaming)."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_configs_lines_restricted_and_split():
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--configs", "--only", "C1,C2",
                           "--frames", "2", "--phase-times", "--steps", "3"],
                          capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert proc.returncode == 0, proc.stderr[-2000:]
    lines = [json.loads(l) for l in proc.stdout.splitlines() if l.startswith("{")]
    assert [l["workload"].split(":")[0] for l in lines] == ["C1", "C2"]
    for line in lines:
        assert line["bit_exact"] is True
        assert line["workload"].split(":")[1].strip().startswith("2 x")  # --frames 2
        assert line["frames_per_s"] > 0 and line["stream_frames_per_s"] > 0
        pt = line["phase_times"]
        assert pt["items"] > 0 and pt["walks"] == 3 * 2  # two frames, three walks each
        assert pt["warp_us"]["streaming"] > 0
        assert pt["warp_us"]["look_back"] == 0 and pt["row_runs"] == 0  # below 2^55
        assert 0 < pt["first_warp_out_of_items_us"] <= pt["last_warp_out_of_items_us"] <= pt["span_us"]
