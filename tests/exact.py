"""Exact integer models used to pin the oracle (test helpers).

Everything here is integer arithmetic on Python ints or numpy uint64 arrays;
no double adds. It restates what the pages fix, independently of the oracle's
C loops:

- a binary32 product of two integers below 2^16 is the integer square rounded
  to 24 significant bits, ties to even (``rnd24``);
- in units of 1/scaler^2 each step of the CPU's double loop is the exact
  integer sum rounded to 53 significant bits, ties to even (``rnd53``;
  ADR-1497 "Decision", first point);
- the first moment and every row sum are exact integers (ADR-1499 "Decision"
  point 1).
"""

from __future__ import annotations

from typing import List, Tuple

import numpy as np


def bit_length_u64(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.uint64)
    bl = np.zeros(x.shape, dtype=np.int64)
    for k in range(64):
        bl += (x >> np.uint64(k)) > 0
    return bl


def rnd24(x: np.ndarray) -> np.ndarray:
    """Round each integer 0 <= x < 2^40 to 24 significant bits, ties to even."""
    x = np.asarray(x, dtype=np.uint64)
    shift = np.maximum(bit_length_u64(x) - 24, 0).astype(np.uint64)
    q = x >> shift
    r = x & ((np.uint64(1) << shift) - np.uint64(1))
    half = (np.uint64(1) << shift) >> np.uint64(1)
    up = (shift > 0) & ((r > half) | ((r == half) & ((q & np.uint64(1)) == 1)))
    return (q + up.astype(np.uint64)) << shift


def rnd53(x: int) -> int:
    """Round a non-negative Python int to 53 significant bits, ties to even."""
    bl = x.bit_length()
    if bl <= 53:
        return x
    s = bl - 53
    q, r = x >> s, x & ((1 << s) - 1)
    half = 1 << (s - 1)
    if r > half or (r == half and q & 1):
        q += 1
    return q << s


def rnd53_u64(x: np.ndarray) -> np.ndarray:
    """Vectorised ``rnd53`` for uint64 arrays."""
    x = np.asarray(x, dtype=np.uint64)
    shift = np.maximum(bit_length_u64(x) - 53, 0).astype(np.uint64)
    q = x >> shift
    r = x & ((np.uint64(1) << shift) - np.uint64(1))
    half = (np.uint64(1) << shift) >> np.uint64(1)
    up = (shift > 0) & ((r > half) | ((r == half) & ((q & np.uint64(1)) == 1)))
    return (q + up.astype(np.uint64)) << shift


def ordered_sum(terms: np.ndarray, start: int = 0) -> int:
    """S <- rnd53(S + t) over the terms in order (the CPU's double loop in
    integer units). Exact below 2^53, so that part is one exact cumsum."""
    t = np.asarray(terms, dtype=np.uint64).ravel()
    s = start
    if s <= 2**53 and t.size:
        cs = np.cumsum(t, dtype=np.uint64) + np.uint64(s)
        k = int(np.searchsorted(cs, np.uint64(2**53), side="right"))
        if k:
            s = int(cs[k - 1])
        t = t[k:]
    for v in t.tolist():
        s = rnd53(s + v)
    return s


def squares_units(p: np.ndarray) -> np.ndarray:
    """rnd24(p^2) for unsigned codewords: the binary32 square in units."""
    p = np.asarray(p, dtype=np.uint64)
    return rnd24(p * p)


def diff_squares_units(r: np.ndarray, d: np.ndarray) -> np.ndarray:
    dd = np.abs(np.asarray(r, dtype=np.int64) - np.asarray(d, dtype=np.int64)).astype(np.uint64)
    return rnd24(dd * dd)


def scaled_mean(units: int, k2: int, n: int) -> float:
    """The double (units * 2^-k2) / n, correctly rounded."""
    return (float(units) * 2.0 ** (-k2)) / n


def moment_model(ref: np.ndarray, dis: np.ndarray, bpc: int) -> Tuple[List[float], np.ndarray]:
    """The four float_moment doubles and the [2][h] exact row sums, from the
    integer recurrence (raster order)."""
    k = bpc - 8
    h, w = ref.shape
    n = w * h
    out = []
    for plane in (ref, dis):
        out.append(scaled_mean(int(np.asarray(plane, dtype=np.uint64).sum()), k, n))
    rows = np.zeros((2, h), dtype=np.uint64)
    for i, plane in enumerate((ref, dis)):
        t = squares_units(plane)
        rows[i] = t.sum(axis=1, dtype=np.uint64)
        out.append(scaled_mean(ordered_sum(t.ravel()), 2 * k, n))
    return out, rows


def psnr_model(ref: np.ndarray, dis: np.ndarray, bpc: int) -> Tuple[np.ndarray, float]:
    """Exact row sums and the mse double from the row-order recurrence."""
    k = bpc - 8
    h, w = ref.shape
    rows = diff_squares_units(ref, dis).sum(axis=1, dtype=np.uint64)
    d = ordered_sum(rows)
    return rows, scaled_mean(d, 2 * k, w * h)
