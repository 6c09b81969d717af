"""Checks that pin the CPU oracle to what the pages and the mathematics fix.

Each ``pin_*`` function runs the oracle (optionally a planted-mistake build)
and raises AssertionError when it disagrees with an independent statement:
exact integer brute force, closed forms, the constructed 2^53 frames of the
pages, or a full enumeration. ``tests/test_oracle_pins.py`` runs them on the
real oracle; ``tests/test_oracle_mutations.py`` shows that each planted
mistake fails at least one of them.
"""

from __future__ import annotations

import os
from functools import lru_cache

import numpy as np

import oracle
from exact import (diff_squares_units, moment_model, ordered_sum, psnr_model, rnd24,
                   scaled_mean, squares_units)
from exact_reductions_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "constructed_frames.txt")


def read_golden():
    out = {}
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            name, exact, cpu = line.split()
            out[name] = (int(exact), int(cpu))
    return out


def _eq(a, b, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, what
    assert np.array_equal(a.view(np.uint64), b.view(np.uint64)), f"{what}: {a} != {b}"


def pin_tiny_bruteforce(mutation=0, seeds=range(24)):
    """Random tiny frames of every bit depth against the integer model."""
    for s in seeds:
        rng = np.random.default_rng((1234, s))
        bpc = [8, 9, 10, 12, 14, 16][s % 6]
        w = int(rng.integers(1, 18))
        h = int(rng.integers(1, 10))
        mode = ["uniform", "extreme", "small", "overrange"][s % 4]
        ref, dis = synth.random_plane_pair(rng, w, h, bpc, mode=mode)
        want, want_rows = moment_model(ref, dis, bpc)
        got, got_rows = oracle.moment(ref, dis, bpc, rows=True, mutation=mutation)
        _eq(got, want, f"moments seed {s} bpc {bpc} {w}x{h}")
        sums = oracle.moment_sums(ref, dis, bpc, mutation=mutation)
        assert sums[2:] == tuple(ordered_sum(squares_units(x).ravel()) for x in (ref, dis))
        assert np.array_equal(got_rows, want_rows), f"s2 rows seed {s}"
        prow, pmse = psnr_model(ref, dis, bpc)
        grow, gmse = oracle.psnr(ref, dis, bpc, mutation=mutation)
        assert np.array_equal(grow, prow), f"psnr rows seed {s}"
        _eq(gmse, pmse, f"mse seed {s}")


@lru_cache(maxsize=None)
def _all_codewords_frame():
    p = np.random.default_rng(99).permutation(65536).astype(np.uint16).reshape(256, 256)
    return p, p[::-1].copy()


def pin_all_codewords(mutation=0):
    """Every 16-bit codeword once: each row of squares equals the integer
    rounding of the squares (full enumeration of the 65 536 samples)."""
    ref, dis = _all_codewords_frame()
    got, rows = oracle.moment(ref, dis, 16, rows=True, mutation=mutation)
    want, want_rows = moment_model(ref, dis, 16)
    assert np.array_equal(rows, want_rows), "row sums of all codewords"
    _eq(got, want, "moments of all codewords")
    prow, pmse = psnr_model(ref, dis, 16)
    grow, gmse = oracle.psnr(ref, dis, 16, mutation=mutation)
    assert np.array_equal(grow, prow)
    _eq(gmse, pmse, "mse of all codewords")


def pin_8bit_exact(mutation=0):
    """8-bit sums are exact integers (Research-2081 "Finding")."""
    wl = synth.WORKLOADS["C1"]
    ref, dis = wl.frame(0)
    n = ref.size
    r64, d64 = ref.astype(np.int64), dis.astype(np.int64)
    got = oracle.moment(ref, dis, 8, mutation=mutation)
    want = [float(r64.sum()) / n, float(d64.sum()) / n,
            float((r64 * r64).sum()) / n, float((d64 * d64).sum()) / n]
    _eq(got, want, "8-bit moments")
    rows, mse = oracle.psnr(ref, dis, 8, mutation=mutation)
    diff = (r64 - d64) ** 2
    assert np.array_equal(rows, diff.sum(axis=1).astype(np.uint64))
    _eq(mse, float(diff.sum()) / n, "8-bit mse")


@lru_cache(maxsize=None)
def _t1():
    return synth.WORKLOADS["T1"].frame(0)


def pin_past_2_53_bruteforce(mutation=0):
    """A 2560x1440 16-bit frame past 2^53 units (ADR-1497 "Context"): the
    second moments equal the raster-order integer recurrence; the first
    moments the exact quotient."""
    for ref, dis in (_t1(), _parity()):
        got = oracle.moment(ref, dis, 16, mutation=mutation)
        want, _ = moment_model(ref, dis, 16)
        _eq(got, want, "moments of a frame past 2^53")
        sums = oracle.moment_sums(ref, dis, 16, mutation=mutation)
        assert sums[2:] == tuple(ordered_sum(squares_units(x).ravel()) for x in (ref, dis)), \
            "second-moment sums of a frame past 2^53"


@lru_cache(maxsize=None)
def _parity():
    return synth.WORKLOADS["T4"].frame(0)


@lru_cache(maxsize=None)
def _half_range():
    return synth.WORKLOADS["C5a"].frame(0)


def pin_psnr_row_order(mutation=0):
    """Half-range 16-bit 3840x2160 noise: the psnr noise passes 2^53 units and
    the CPU adds exact rows in row order (ADR-1499 "Context"/"Decision")."""
    ref, dis = _half_range()
    prow, pmse = psnr_model(ref, dis, 16)
    assert int(prow.sum(dtype=np.uint64)) > 2**53
    grow, gmse = oracle.psnr(ref, dis, 16, mutation=mutation)
    assert np.array_equal(grow, prow), "psnr rows of the half-range frame"
    _eq(gmse, pmse, "mse of the half-range frame")
    assert oracle.psnr_noise_sum(ref, dis, 16, mutation=mutation) == ordered_sum(prow)


def pin_constructed_frames(mutation=0):
    """The 2^53 boundary frames: the oracle's sums are the pages' CPU sums."""
    golden = read_golden()
    n = 3840 * 2160
    frames = [("2^53-1", synth.WORKLOADS["C5b"].frame(0)),
              ("2^53", synth.WORKLOADS["C5b"].frame(1)),
              ("2^53+3ties", synth.WORKLOADS["C5b"].frame(2)),
              ("2^54+7drops", synth.WORKLOADS["T3"].frame(0))]
    for name, (ref, dis) in frames:
        exact, cpu = golden[name]
        t = squares_units(ref)
        assert int(t.sum(dtype=np.uint64)) == exact, name
        got = oracle.moment(ref, dis, 16, mutation=mutation)
        _eq(got[2], scaled_mean(cpu, 16, n), f"second moment {name}")
        assert oracle.moment_sums(ref, dis, 16, mutation=mutation)[2] == cpu, name
        assert oracle.psnr_noise_sum(ref, dis, 16, mutation=mutation) == cpu, name
        _eq(got[3], 0.0, f"dis second moment {name}")
        rows, mse = oracle.psnr(ref, dis, 16, mutation=mutation)
        assert int(rows.sum(dtype=np.uint64)) == exact, name
        _eq(mse, scaled_mean(cpu, 16, n), f"mse {name}")


def pin_first_moment_closed_form(mutation=0):
    """First moments are exact quotients of the integer sums (sums of p are
    below 2^41 units, exact in a double) on 10- and 12-bit frames."""
    for key in ("C2", "C3"):
        wl = synth.WORKLOADS[key]
        ref, dis = wl.frame(0)
        n = ref.size
        got = oracle.moment(ref, dis, wl.bpc, mutation=mutation)
        k = wl.bpc - 8
        want = [scaled_mean(int(ref.astype(np.uint64).sum()), k, n),
                scaled_mean(int(dis.astype(np.uint64).sum()), k, n)]
        _eq(got[:2], want, f"first moments {key}")
        # Below 2^53 the second moment is the exact sum, rounded once.
        s2 = [int(squares_units(x).sum(dtype=np.uint64)) for x in (ref, dis)]
        _eq(got[2:], [scaled_mean(s, 2 * k, n) for s in s2], f"second moments {key}")


def pin_psnr_closed_form(mutation=0):
    """PSNR reading at points with exact values: peak^2 / mse == 1 gives 0 dB,
    an 8-bit mse of 650.25 (= 255^2 / 100) gives 20 dB, the 1e-10 floor and
    the cap. The formula's constants are a reading (the pages give none)."""
    for bpc in (8, 10, 12, 16):
        peak = ((1 << bpc) - 1) / (1 << (bpc - 8))
        assert oracle.psnr_db(peak * peak, bpc, 0.0, mutation=mutation) == 0.0
        floor = oracle.psnr_db(1e-10, bpc, 0.0, mutation=mutation)
        assert oracle.psnr_db(0.0, bpc, 0.0, mutation=mutation) == floor
        assert oracle.psnr_db(1e-12, bpc, 0.0, mutation=mutation) == floor
        assert oracle.psnr_db(0.0, bpc, 60.0, mutation=mutation) == 60.0
        assert oracle.psnr_db(1.0, bpc, 0.0) > oracle.psnr_db(2.0, bpc, 0.0)
    assert oracle.psnr_db(650.25, 8, 0.0, mutation=mutation) == 20.0


def pin_integer_psnr_bruteforce(mutation=0, seeds=range(12)):
    """integer_psnr against exact integer brute force in numpy: every row's
    sum of squared codeword differences, the plane's sum and the MSE (the
    sum, converted to double once, over the pixel count), on random planes
    of every depth, including container values past the depth and padded
    strides."""
    for s in seeds:
        rng = np.random.default_rng(900 + s)
        bpc = [8, 10, 12, 16][s % 4]
        h, w = int(rng.integers(1, 9)), int(rng.integers(1, 40))
        mode = ["uniform", "extreme", "small", "overrange"][(s // 4) % 4]
        ref, dis = synth.random_plane_pair(rng, w, h, bpc, stride_samples=w + 3, mode=mode)
        rows, sse, mse = oracle.integer_psnr(ref, dis, bpc, mutation=mutation, width=w)
        d = ref[:, :w].astype(np.int64) - dis[:, :w].astype(np.int64)
        want_rows = (d * d).sum(axis=1).astype(np.uint64)
        assert np.array_equal(rows, want_rows), (s, rows, want_rows)
        assert sse == int((d * d).sum()), s
        assert mse == float(int((d * d).sum())) / float(w * h), s


def pin_integer_psnr_closed_forms(mutation=0):
    """Constant planes a and b: every row adds W (a - b)^2 and the MSE is
    (a - b)^2 exactly; where every difference is below 4096 the squares are
    exact in binary32, so the rows equal float_psnr's rows (both in units of
    a codeword squared); a difference past 4096 makes them differ."""
    for bpc, a, b in ((8, 255, 0), (10, 3, 1000), (16, 65535, 0), (16, 40000, 39000)):
        dt = np.uint8 if bpc == 8 else np.uint16
        ref = np.full((5, 7), a, dtype=dt)
        dis = np.full((5, 7), b, dtype=dt)
        rows, sse, mse = oracle.integer_psnr(ref, dis, bpc, mutation=mutation)
        assert np.all(rows == 7 * (a - b) ** 2), (bpc, rows)
        assert sse == 35 * (a - b) ** 2 and mse == float((a - b) ** 2), (bpc, sse, mse)
    rng = np.random.default_rng(77)
    ref = rng.integers(0, 4096, size=(6, 50)).astype(np.uint16)
    dis = rng.integers(0, 4096, size=(6, 50)).astype(np.uint16)
    irows, _, _ = oracle.integer_psnr(ref, dis, 16, mutation=mutation)
    frows, _ = oracle.psnr(ref, dis, 16)
    assert np.array_equal(irows, frows)
    ref[2, 3], dis[2, 3] = 65535, 100  # 65435^2 needs more than 24 bits
    irows, _, _ = oracle.integer_psnr(ref, dis, 16, mutation=mutation)
    frows, _ = oracle.psnr(ref, dis, 16)
    assert irows[2] != frows[2] and np.array_equal(np.delete(irows, 2), np.delete(frows, 2))


ALL_PINS = [pin_tiny_bruteforce, pin_all_codewords, pin_8bit_exact,
            pin_first_moment_closed_form, pin_psnr_closed_form, pin_constructed_frames,
            pin_psnr_row_order, pin_past_2_53_bruteforce, pin_integer_psnr_bruteforce,
            pin_integer_psnr_closed_forms]
