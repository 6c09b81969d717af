"""libvmx against the CPU oracle on a GB300: every double bit for bit, every
uint64 row sum and accumulator exactly (ADR-1497 / ADR-1499: the CPU's bits
on every frame). Inputs are the seeded workloads of ``synth``."""

import numpy as np
import pytest
import torch

from exact_reductions_gb300 import api, synth
from gpu_helpers import run_and_check, to_device, u64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("key", ["C1", "C2", "C3"])
def test_small_depths_all_frames(key):
    """8-, 10- and 12-bit batches: exact sums, no ordered-sum work."""
    wl = synth.WORKLOADS[key]
    ref, dis = wl.batch()
    run_and_check(ref, dis, wl.bpc)


def test_c4_full_range_noise_all_frames():
    """16 frames of 16-bit 3840x2160 noise: every second moment passes 2^53
    units and goes through runs; every frame identical."""
    wl = synth.WORKLOADS["C4"]
    ref, dis = wl.batch()
    out, stats = run_and_check(ref, dis, 16)
    exact, by_run, walked = int(stats[0]), int(stats[1]), int(stats[2])
    assert by_run > 16 * 2 * 300, stats
    assert walked <= 16 * 2 * 4, stats


@pytest.mark.parametrize("key", ["C5a", "C5b", "T1", "T2", "T3", "T4"])
def test_stress_frames(key):
    """Half-range noise (psnr past 2^53), the 2^53 boundary frames, frames
    past 2^53 and 2^55, 2^54 followed by dropped terms, parity stress."""
    wl = synth.WORKLOADS[key]
    ref, dis = wl.batch()
    run_and_check(ref, dis, 16)


@pytest.mark.parametrize("features", [1, 2])
def test_single_feature_calls(features):
    wl = synth.WORKLOADS["C5a"]
    ref, dis = wl.batch(2)
    run_and_check(ref, dis, 16, features=features)


@pytest.mark.parametrize("features", [1, 2])
def test_single_feature_calls_past_2_55(features):
    """Moments alone on a frame past 2^55 (the look-back and the row runs
    without psnr), and psnr alone on it (no look-back: only the moments
    need one)."""
    wl = synth.WORKLOADS["T2"]
    ref, dis = wl.batch(1)
    run_and_check(ref, dis, 16, features=features)


def test_c5c_8k_batch_sampled():
    """64 frames of 16-bit 7680x4320 noise (four binade ranges): the full
    batch in one call, frames 0, 31 and 63 against the oracle."""
    wl = synth.WORKLOADS["C5c"]
    ref, dis = wl.batch()
    run_and_check(ref, dis, 16, frames=[0, 31, 63])
