"""The lane-order variant of the second moment (a non-target) against the
oracle's raster loop: equal with one lane, equal with any number of lanes
while the sum stays at or below 2^53 units, different past 2^53 (the page
on the exact second-moment sum, "Neutral / follow-ups": the NEON and SVE2
paths of the CPU extractor add in lanes). The library reproduces the raster
loop, not this."""

import numpy as np

import oracle
from exact_reductions_gb300 import synth


def _bits(x: float) -> int:
    return int(np.float64(x).view(np.uint64))


def test_one_lane_is_the_scalar_loop():
    ref, dis = synth.WORKLOADS["T1"].batch(1)
    m = oracle.moment(ref[0], dis[0], 16)
    assert _bits(oracle.second_moment_lanes(ref[0], 16, 1)) == _bits(m[2])
    assert _bits(oracle.second_moment_lanes(dis[0], 16, 1)) == _bits(m[3])


def test_lanes_agree_at_or_below_2_53():
    ref, dis = synth.WORKLOADS["C2"].batch(1)
    m = oracle.moment(ref[0], dis[0], 10)
    for lanes in (2, 4, 8):
        assert _bits(oracle.second_moment_lanes(ref[0], 10, lanes)) == _bits(m[2]), lanes


def _past_2_53_frame() -> np.ndarray:
    # 1050 rows of full-scale 16-bit samples take the raster sum past 2^53
    # units; the 50 rows of ones after them are odd terms that the raster
    # loop rounds away (ties to even), while each of two or more lanes
    # stays below 2^53 and adds them exactly.
    plane = np.ones((1100, 2048), dtype=np.uint16)
    plane[:1050] = 65535
    return plane


def test_lanes_differ_past_2_53():
    plane = _past_2_53_frame()
    m = oracle.moment(plane, plane, 16)
    sums = oracle.moment_sums(plane, plane, 16)
    assert sums[2] > 1 << 53
    raster = oracle.second_moment_lanes(plane, 16, 1)
    assert _bits(raster) == _bits(m[2])
    for lanes in (2, 4, 8):
        lane = oracle.second_moment_lanes(plane, 16, lanes)
        # Lanes keep the ones the raster loop dropped: a larger mean.
        assert lane > raster, lanes
        n = plane.size
        dropped_units = (lane - raster) * n * 65536.0
        assert 0.4 * 50 * 2048 < dropped_units < 1.1 * 50 * 2048, (lanes, dropped_units)
