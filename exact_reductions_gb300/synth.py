"""Seeded synthetic luma planes for the float_moment / float_psnr workloads.

This module only draws and arranges samples. It holds none of the method's
arithmetic (no float squares, no rounding rules, no sums in units): both the
CUDA path's tests and the CPU oracle take their inputs from here.

Every frame is drawn from its own generator, ``numpy.random.default_rng((seed,
frame))`` (PCG64 seeded through a SeedSequence), so that one frame of a large
batch can be rebuilt alone. Within a frame the reference plane is drawn first,
then the distorted plane.

The workloads follow the five configurations the float_moment / float_psnr
exact-sum pages are measured on (ADR-1497 "Consequences", ADR-1499
"Consequences"): 8-, 10-, 12- and 16-bit luma, 3840x2160 and 7680x4320 16-bit
noise, and frames built to reach 2^53 units exactly. The public clips those
pages also use (the Netflix pair, Big Buck Bunny) are not reproduced; seeded
noise and gradients of the same sizes and bit depths stand in for them.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List, Optional, Tuple

import numpy as np

# The largest sample whose square has at most 16 significant bits and so is an
# exact float: 65280 = 255 * 256, square = 255^2 * 2^16.
_EXACT_BIG = 65280


@dataclass(frozen=True)
class Workload:
    """A batch of frame pairs: sizes, bit depth, frame count and its recipe."""

    name: str
    width: int
    height: int
    bpc: int
    frames: int
    seed: int
    recipe: str

    @property
    def bytes_per_sample(self) -> int:
        return 1 if self.bpc == 8 else 2

    @property
    def dtype(self):
        return np.uint8 if self.bpc == 8 else np.uint16

    @property
    def frame_pair_bytes(self) -> int:
        return 2 * self.width * self.height * self.bytes_per_sample

    def frame(self, f: int) -> Tuple[np.ndarray, np.ndarray]:
        """Return (ref, dis) of frame ``f`` as packed (height, width) arrays."""
        return _RECIPES[self.recipe](self, f)

    def batch(self, frames: Optional[int] = None) -> Tuple[np.ndarray, np.ndarray]:
        """Return (ref, dis) of the first ``frames`` frames, shape (F, H, W)."""
        n = self.frames if frames is None else frames
        ref = np.empty((n, self.height, self.width), dtype=self.dtype)
        dis = np.empty_like(ref)
        for f in range(n):
            ref[f], dis[f] = self.frame(f)
        return ref, dis


def _rng(seed: int, f: int) -> np.random.Generator:
    return np.random.default_rng((seed, f))


def _uniform_pair(lo_r, hi_r, lo_d, hi_d):
    def make(wl: Workload, f: int):
        g = _rng(wl.seed, f)
        shape = (wl.height, wl.width)
        ref = g.integers(lo_r, hi_r + 1, size=shape, dtype=np.uint16)
        dis = g.integers(lo_d, hi_d + 1, size=shape, dtype=np.uint16)
        return ref, dis
    return make


def _c1(wl: Workload, f: int):
    # 8 bpc: ref uniform in [0, 255]; dis = clip(ref + rint(N(0, 8^2)), 0, 255).
    g = _rng(wl.seed, f)
    shape = (wl.height, wl.width)
    ref = g.integers(0, 256, size=shape, dtype=np.uint8)
    noise = np.rint(g.normal(0.0, 8.0, size=shape)).astype(np.int32)
    dis = np.clip(ref.astype(np.int32) + noise, 0, 255).astype(np.uint8)
    return ref, dis


def _c2(wl: Workload, f: int):
    # 10 bpc: ref uniform in [0, 1023]; on odd columns a sample whose low two
    # bits are both zero gets its lowest bit set, so no odd pixel is a
    # multiple of 4 (the codeword is fractional on the 8-bit scale);
    # dis = clip(ref + rint(N(0, 16^2)), 0, 1023).
    g = _rng(wl.seed, f)
    shape = (wl.height, wl.width)
    ref = g.integers(0, 1024, size=shape, dtype=np.uint16)
    odd = ref[:, 1::2]
    odd[(odd & 3) == 0] |= 1
    noise = np.rint(g.normal(0.0, 16.0, size=shape)).astype(np.int32)
    dis = np.clip(ref.astype(np.int32) + noise, 0, 1023).astype(np.uint16)
    return ref, dis


def _c3(wl: Workload, f: int):
    # 12 bpc: ref = clip(floor(x * 4095 / (w - 1)) + U[-64, 64], 0, 4095);
    # dis = clip(rint-blur(ref) + rint(N(0, 32^2)), 0, 4095) where the blur is
    # the horizontal 5-tap [1, 4, 6, 4, 1] / 16 with replicated edges, rounded
    # as (s + 8) >> 4.
    g = _rng(wl.seed, f)
    h, w = wl.height, wl.width
    x = np.arange(w, dtype=np.int64)
    grad = (x * 4095) // max(w - 1, 1)
    jitter = g.integers(-64, 65, size=(h, w), dtype=np.int64)
    ref = np.clip(grad[None, :] + jitter, 0, 4095)
    pad = np.concatenate([ref[:, :1], ref[:, :1], ref, ref[:, -1:], ref[:, -1:]], axis=1)
    s = pad[:, 0:w] + 4 * pad[:, 1:w + 1] + 6 * pad[:, 2:w + 2] + 4 * pad[:, 3:w + 3] + pad[:, 4:w + 4]
    blur = (s + 8) >> 4
    noise = np.rint(g.normal(0.0, 32.0, size=(h, w))).astype(np.int64)
    dis = np.clip(blur + noise, 0, 4095)
    return ref.astype(np.uint16), dis.astype(np.uint16)


def exact_square_fill(target: int, width: int, height: int, even_only: bool = False,
                      tail_ones: int = 0) -> np.ndarray:
    """A 16-bit plane whose squares add to exactly ``target`` at a row end.

    Only samples with an exactly representable float square are used: 65280
    (square 255^2 * 2^16) fills the plane in raster order, then the remainder
    is reached greedily with multiples of 256 and with samples below 4096
    (squares of at most 24 bits). The greedy samples sit at the end of the
    row where the prefix stops (or the next row), so the running sum meets
    ``target`` exactly at that row's end. ``even_only`` keeps every square a
    multiple of 4. After that row, ``tail_ones`` rows each hold one sample 1
    in column 0. Everything else is 0.
    """
    big = _EXACT_BIG * _EXACT_BIG
    n_big = target // big
    rem = target - n_big * big
    greedy: List[int] = []
    candidates = [256 * m for m in range(255, 0, -1)] + list(range(4095, 0, -1))
    if even_only:
        candidates = [p for p in candidates if p % 2 == 0]
    for p in candidates:
        while p * p <= rem:
            greedy.append(p)
            rem -= p * p
    if rem:
        raise ValueError("target not reachable with the chosen samples")
    plane = np.zeros(width * height, dtype=np.uint16)
    plane[:n_big] = _EXACT_BIG
    # The row holding the last big sample, or the next one when it is full.
    last = n_big - 1
    row = last // width if n_big else 0
    if n_big and (last % width) + 1 + len(greedy) > width:
        row += 1
    if len(greedy) > width:
        raise ValueError("row too short for the greedy samples")
    end = (row + 1) * width
    if greedy:
        plane[end - len(greedy):end] = np.array(greedy, dtype=np.uint16)
    for i in range(tail_ones):
        plane[(row + 1 + i) * width] = 1
    if (row + 1 + tail_ones) > height:
        raise ValueError("plane too small")
    sq = plane.astype(np.int64)
    assert int((sq * sq).sum()) == target + tail_ones
    return plane.reshape(height, width)


def _c5b(wl: Workload, f: int):
    # Frames whose exact second-moment (and psnr, dis = 0) sum is 2^53 - 1,
    # 2^53, and 2^53 followed by three rows each holding one sample 1.
    targets = [(2**53 - 1, 0), (2**53, 0), (2**53, 3)]
    t, ones = targets[f % 3]
    ref = exact_square_fill(t, wl.width, wl.height, tail_ones=ones)
    return ref, np.zeros_like(ref)


def _t54(wl: Workload, f: int):
    # 2^54 reached exactly with squares that are multiples of 4, then seven
    # rows each holding one sample 1 (test-only frame of ADR-1497 "Decision").
    ref = exact_square_fill(2**54, wl.width, wl.height, even_only=True, tail_ones=7)
    return ref, np.zeros_like(ref)


def _parity_stress(wl: Workload, f: int):
    # Past 2^55 units with codeword 65535, then a seeded mix whose squares
    # tie at the last place 8 (p = 2 mod 4 below 4096), move the parity of
    # S / 8 (p in [8192, 11585), squares that are odd multiples of 8 about
    # half the time) or round down (odd p below 4096). dis: the same recipe
    # with another draw, past 2^54 only.
    g = _rng(wl.seed, f)
    n = wl.width * wl.height
    planes = []
    for fill in (8388864 + 4096, 4194432 + 64 * 4096):
        plane = np.zeros(n, dtype=np.uint16)
        plane[:fill] = 65535
        m = n - fill
        kind = g.integers(0, 3, size=m)
        tie = 4 * g.integers(0, 1024, size=m) + 2
        flip = g.integers(8192, 11585, size=m)
        down = 2 * g.integers(0, 2048, size=m) + 1
        plane[fill:] = np.where(kind == 0, tie, np.where(kind == 1, flip, down))
        planes.append(plane.reshape(wl.height, wl.width))
    return planes[0], planes[1]


_RECIPES: dict = {
    "c1": _c1,
    "c2": _c2,
    "c3": _c3,
    "uniform16": _uniform_pair(0, 65535, 0, 65535),
    "halfrange16": _uniform_pair(32768, 65535, 0, 32767),
    "c5b": _c5b,
    "past53": _uniform_pair(40000, 65535, 40000, 65535),
    "past55": _uniform_pair(60000, 65535, 60000, 65535),
    "t54": _t54,
    "parity": _parity_stress,
}

WORKLOADS = {
    "C1": Workload("C1", 320, 240, 8, 1, 0, "c1"),
    "C2": Workload("C2", 1920, 1080, 10, 16, 1, "c2"),
    "C3": Workload("C3", 2560, 1440, 12, 16, 2, "c3"),
    "C4": Workload("C4", 3840, 2160, 16, 16, 3, "uniform16"),
    "C5a": Workload("C5a", 3840, 2160, 16, 8, 4, "halfrange16"),
    "C5b": Workload("C5b", 3840, 2160, 16, 3, 0, "c5b"),
    "C5c": Workload("C5c", 7680, 4320, 16, 64, 5, "uniform16"),
    # Extra frames named on the pages (ADR-1497 "Consequences"/guards).
    "T1": Workload("T1", 2560, 1440, 16, 1, 6, "past53"),
    "T2": Workload("T2", 4096, 2560, 16, 1, 7, "past55"),
    "T3": Workload("T3", 3840, 2160, 16, 1, 0, "t54"),
    # Parity stress: binade 55 with ties and parity changes in every row.
    "T4": Workload("T4", 4096, 2560, 16, 2, 8, "parity"),
}


def random_plane_pair(rng: np.random.Generator, width: int, height: int, bpc: int,
                      stride_samples: Optional[int] = None,
                      mode: str = "uniform") -> Tuple[np.ndarray, np.ndarray]:
    """Small random (ref, dis) planes for edge-case tests.

    ``mode``: "uniform" over the full container range of the bit depth,
    "extreme" (only 0, 1, max and max-1 codewords), "small" (below 4096),
    "overrange" (uint16 samples above 2^bpc - 1). Returns arrays of shape
    (height, stride_samples) whose padding columns hold random garbage.
    """
    dt = np.uint8 if bpc == 8 else np.uint16
    top = (1 << bpc) - 1
    ss = width if stride_samples is None else stride_samples
    cont = 255 if bpc == 8 else 65535
    ref = rng.integers(0, cont + 1, size=(height, ss), dtype=np.int64)
    dis = rng.integers(0, cont + 1, size=(height, ss), dtype=np.int64)
    body = (slice(None), slice(0, width))
    if mode == "uniform":
        ref[body] = rng.integers(0, top + 1, size=(height, width))
        dis[body] = rng.integers(0, top + 1, size=(height, width))
    elif mode == "extreme":
        choices = np.array([0, 1, top, top - 1])
        ref[body] = rng.choice(choices, size=(height, width))
        dis[body] = rng.choice(choices, size=(height, width))
    elif mode == "small":
        ref[body] = rng.integers(0, min(top, 4095) + 1, size=(height, width))
        dis[body] = rng.integers(0, min(top, 4095) + 1, size=(height, width))
    elif mode == "overrange":
        ref[body] = rng.integers(0, cont + 1, size=(height, width))
        dis[body] = rng.integers(0, cont + 1, size=(height, width))
    else:
        raise ValueError(mode)
    return ref.astype(dt), dis.astype(dt)
