"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""

import numpy as np
import pytest

import oracle
import oracle_pins as pins
from exact import rnd24, rnd53, rnd53_u64


def test_oracle_builds_without_mutation():
    assert oracle.load(0).vmx_oracle_mutation() == 0


def test_rnd24_is_binary32_square_for_every_codeword():
    """All 65 536 codewords: the binary32 square is the integer square
    rounded to 24 significant bits, ties to even (the terms of ADR-1497
    "Context" are integers below 2^32 in units of 1/scaler^2)."""
    p = np.arange(65536, dtype=np.uint64)
    f = p.astype(np.float32)
    sq = (f * f).astype(np.float64).astype(np.uint64)
    assert np.array_equal(sq, rnd24(p * p))
    assert int(rnd24(np.array([0xFFFE0001], dtype=np.uint64))[0]) == 0xFFFE0000
    assert np.all(sq < 2**32)
    assert np.array_equal(sq[:4096], p[:4096] * p[:4096])


def test_one_term_step_is_double_add():
    """rnd53(S + t) == double(S) + double(t) on 400 000 random pairs and the
    boundary pairs (ADR-1497 "Decision": the one-term step)."""
    rng = np.random.default_rng(7)
    e = rng.integers(50, 58, size=400_000)
    s = (rng.integers(0, 2**50, size=e.size, dtype=np.uint64) | np.uint64(2**50))
    s = s << (e - 50).astype(np.uint64)
    s = rnd53_u64(s)
    t = rng.integers(0, 2**32, size=e.size, dtype=np.uint64)
    want = s.astype(np.float64) + t.astype(np.float64)
    got = rnd53_u64(s + t)
    assert np.array_equal(got.astype(np.float64), want)
    assert np.array_equal(got, want.astype(np.uint64))
    # Boundary pairs.
    starts = [2**53 - 1, 2**53, 2**53 - 2, 2**53 + 2, 2**54 - 2, 2**54, 2**54 - 4,
              2**55 - 4, 2**55, 2**56 - 8, 2**57 - 16]
    for S in starts:
        u = max(1, 1 << max(S.bit_length() - 53, 0))
        for t in (0, 1, u // 2 - 1, u // 2, u // 2 + 1, u - 1, u, u + u // 2,
                  2**32 - 2**17, 3, 5, 7):
            if t < 0:
                continue
            assert rnd53(S + t) == int(float(S) + float(t)), (S, t)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_exactness_window_closed_form():
    """ADR-1497 "Context": the exact sum stays at or below 2^53 units for every
    16-bit frame up to 2^21 pixels and every 8/10/12-bit frame up to 2^29."""
    assert 2**21 * int(rnd24(np.array([65535**2], dtype=np.uint64))[0]) <= 2**53
    assert 2**29 * 4095**2 <= 2**53
    # ... and a row of 2^15 terms stays below 2^47 (ADR-1499 "Decision" 1).
    assert 2**15 * (2**32 - 1) < 2**47
