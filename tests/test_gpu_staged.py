"""The kernel built with its rows streamed through shared memory (bulk
asynchronous copies into per-warp chunk buffers, mbarrier phases; the
VMX_STAGES compile-time option, off in the default build because direct
16-byte loads measure faster) against the oracle: a 16-bit 3840x2160 batch,
a frame past 2^55 (look-back and runs), and rows with a chunk remainder and a
padded stride."""

import numpy as np
import pytest

from exact_reductions_gb300 import _lib, build, synth
from gpu_helpers import run_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def staged():
    return _lib.bind(build.build_variant("staged3", ["VMX_STAGES=3", "VMX_MAX_REGS=128"]))


def test_staged_rows_match_oracle(monkeypatch, staged):
    monkeypatch.setattr(_lib, "_lib", staged)
    ref, dis = synth.WORKLOADS["C4"].batch(3)
    run_and_check(ref, dis, 16)
    ref, dis = synth.WORKLOADS["T2"].batch(1)
    run_and_check(ref, dis, 16)
    rng = np.random.default_rng(77)
    W, S, H = 2049, 2056, 23  # two whole chunks per row, then 33 vectors
    ref, dis = synth.random_plane_pair(rng, W, H, 16, stride_samples=S)
    run_and_check(ref[None], dis[None], 16, width=W)
