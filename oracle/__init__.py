"""ctypes access to the CPU oracle (plain C raster loops, ``vmx_oracle.c``).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg import this package. The library under
``exact_reductions_gb300`` never does, and shares no code with it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Tuple

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD = os.path.join(HERE, "_build")
SRC = os.path.join(HERE, "vmx_oracle.c")
CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fno-tree-vectorize",
          "-fPIC", "-shared", "-std=c11", "-Wall", "-Wextra"]

_lock = threading.Lock()
_libs: dict = {}


def lib_path(mutation: int = 0) -> str:
    name = "libvmx_oracle.so" if mutation == 0 else f"libvmx_oracle_mut{mutation}.so"
    return os.path.join(BUILD, name)


def build(mutation: int = 0, force: bool = False) -> str:
    """Compile the oracle (or a planted-mistake copy) with gcc; return its path."""
    out = lib_path(mutation)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= max(
            os.path.getmtime(SRC), os.path.getmtime(os.path.join(HERE, "vmx_oracle.h"))):
        return out
    os.makedirs(BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, f"-DORACLE_MUTATION={mutation}", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(path: str) -> ctypes.CDLL:
    lib = ctypes.CDLL(path)
    vp, i32, i64, dp, u64p = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                              ctypes.POINTER(ctypes.c_double),
                              ctypes.POINTER(ctypes.c_uint64))
    lib.vmx_oracle_moment.argtypes = [vp, vp, i32, i32, i64, i32, dp, u64p]
    lib.vmx_oracle_moment.restype = None
    lib.vmx_oracle_moment_acc.argtypes = [vp, vp, i32, i32, i64, i32, dp]
    lib.vmx_oracle_moment_acc.restype = None
    lib.vmx_oracle_psnr_noise.argtypes = [vp, vp, i32, i32, i64, i32, u64p]
    lib.vmx_oracle_psnr_noise.restype = ctypes.c_double
    lib.vmx_oracle_psnr.argtypes = [vp, vp, i32, i32, i64, i32, u64p, dp]
    lib.vmx_oracle_psnr.restype = None
    lib.vmx_oracle_psnr_db.argtypes = [ctypes.c_double, i32, ctypes.c_double]
    lib.vmx_oracle_psnr_db.restype = ctypes.c_double
    lib.vmx_oracle_moment_batch.argtypes = [vp, vp, i32, i32, i64, i32, i32, i32, dp]
    lib.vmx_oracle_moment_batch.restype = None
    lib.vmx_oracle_psnr_batch.argtypes = [vp, vp, i32, i32, i64, i32, i32, i32, u64p, dp]
    lib.vmx_oracle_psnr_batch.restype = None
    lib.vmx_oracle_second_moment_lanes.argtypes = [vp, i32, i32, i64, i32, i32]
    lib.vmx_oracle_second_moment_lanes.restype = ctypes.c_double
    lib.vmx_oracle_integer_psnr.argtypes = [vp, vp, i32, i32, i64, i32, u64p, u64p, dp]
    lib.vmx_oracle_integer_psnr.restype = None
    lib.vmx_oracle_integer_psnr_batch.argtypes = [vp, vp, i32, i32, i64, i32, i32, i32, u64p,
                                                  u64p, dp]
    lib.vmx_oracle_integer_psnr_batch.restype = None
    lib.vmx_oracle_mutation.argtypes = []
    lib.vmx_oracle_mutation.restype = i32
    return lib


def load(mutation: int = 0) -> ctypes.CDLL:
    with _lock:
        if mutation not in _libs:
            _libs[mutation] = _bind(build(mutation))
        return _libs[mutation]


def _plane_args(ref: np.ndarray, dis: np.ndarray, width: Optional[int]):
    """(ptr_ref, ptr_dis, width, height, stride_bytes) of 2-D planes.

    The planes may be column slices of wider arrays (padded stride)."""
    assert ref.shape == dis.shape and ref.dtype == dis.dtype and ref.ndim == 2
    assert ref.strides == dis.strides and ref.strides[1] == ref.itemsize
    h, w = ref.shape
    return (ref.ctypes.data, dis.ctypes.data, w if width is None else width, h,
            ref.strides[0])


def moment(ref: np.ndarray, dis: np.ndarray, bpc: int, rows: bool = False,
           mutation: int = 0, width: Optional[int] = None):
    """float_moment of one frame pair: array [ref1, dis1, ref2, dis2] (and the
    [2][height] exact row sums of the float squares when ``rows``)."""
    lib = load(mutation)
    pr, pd, w, h, s = _plane_args(ref, dis, width)
    out = np.zeros(4, dtype=np.float64)
    r = np.zeros((2, h), dtype=np.uint64) if rows else None
    lib.vmx_oracle_moment(pr, pd, w, h, s, bpc,
                          out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                          r.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)) if rows else None)
    return (out, r) if rows else out


def second_moment_lanes(plane: np.ndarray, bpc: int, lanes: int) -> float:
    """Not the CPU's result: the second moment added in `lanes` interleaved
    double accumulators, as a SIMD path that adds in lanes would (kept to
    measure how far that is from the scalar sum past 2^53 units)."""
    lib = load(0)
    plane = np.ascontiguousarray(plane)
    h, w = plane.shape
    return float(lib.vmx_oracle_second_moment_lanes(plane.ctypes.data, w, h, plane.strides[0],
                                                    bpc, lanes))


def moment_sums(ref: np.ndarray, dis: np.ndarray, bpc: int, mutation: int = 0,
                width: Optional[int] = None) -> Tuple[int, int, int, int]:
    """The CPU's four accumulators after the last pixel, as exact integers in
    units: (sum p / scaler in 1/scaler, same for dis, second-moment sums of
    ref and dis in 1/scaler^2)."""
    lib = load(mutation)
    pr, pd, w, h, s = _plane_args(ref, dis, width)
    acc = np.zeros(4, dtype=np.float64)
    lib.vmx_oracle_moment_acc(pr, pd, w, h, s, bpc,
                              acc.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    k = bpc - 8
    return (_units(acc[0], k), _units(acc[1], k), _units(acc[2], 2 * k), _units(acc[3], 2 * k))


def psnr_noise_sum(ref: np.ndarray, dis: np.ndarray, bpc: int, mutation: int = 0,
                   width: Optional[int] = None) -> int:
    """The CPU's row-order noise accumulator as an exact integer in units."""
    lib = load(mutation)
    pr, pd, w, h, s = _plane_args(ref, dis, width)
    noise = lib.vmx_oracle_psnr_noise(pr, pd, w, h, s, bpc, None)
    return _units(noise, 2 * (bpc - 8))


def _units(x: float, shift: int) -> int:
    """A double holding a multiple of 2^-shift, as that integer multiple."""
    import math
    if x == 0.0:
        return 0
    m, e = math.frexp(x)
    mant = int(m * 2**53)  # exact: 53 significant bits
    sh = e - 53 + shift
    v = mant << sh if sh >= 0 else mant >> -sh
    assert sh >= 0 or mant & ((1 << -sh) - 1) == 0, "not a multiple of the unit"
    return v


def psnr(ref: np.ndarray, dis: np.ndarray, bpc: int, mutation: int = 0,
         width: Optional[int] = None) -> Tuple[np.ndarray, float]:
    """float_psnr of one frame pair: (row sums [height] in units, mse)."""
    lib = load(mutation)
    pr, pd, w, h, s = _plane_args(ref, dis, width)
    rows = np.zeros(h, dtype=np.uint64)
    mse = ctypes.c_double(0.0)
    lib.vmx_oracle_psnr(pr, pd, w, h, s, bpc,
                        rows.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)),
                        ctypes.byref(mse))
    return rows, mse.value


def integer_psnr(ref: np.ndarray, dis: np.ndarray, bpc: int, mutation: int = 0,
                 width: Optional[int] = None) -> Tuple[np.ndarray, int, float]:
    """integer_psnr of one plane pair: (exact row sums [height] of squared
    codeword differences, the plane's sum, mse in codeword units)."""
    lib = load(mutation)
    pr, pd, w, h, s = _plane_args(ref, dis, width)
    rows = np.zeros(h, dtype=np.uint64)
    sse = ctypes.c_uint64(0)
    mse = ctypes.c_double(0.0)
    lib.vmx_oracle_integer_psnr(pr, pd, w, h, s, bpc,
                                rows.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)),
                                ctypes.byref(sse), ctypes.byref(mse))
    return rows, int(sse.value), mse.value


def integer_psnr_batch(ref: np.ndarray, dis: np.ndarray, bpc: int,
                       width: Optional[int] = None):
    """integer_psnr over a (F, H, W) batch: dict with ``rows`` [F][H],
    ``sse`` [F], ``mse`` [F]."""
    lib = load(0)
    ref = np.ascontiguousarray(ref)
    dis = np.ascontiguousarray(dis)
    F, h, ss = ref.shape
    w = ss if width is None else width
    rows = np.zeros((F, h), dtype=np.uint64)
    sse = np.zeros(F, dtype=np.uint64)
    mse = np.zeros(F, dtype=np.float64)
    u64 = ctypes.POINTER(ctypes.c_uint64)
    lib.vmx_oracle_integer_psnr_batch(ref.ctypes.data, dis.ctypes.data, w, h, ref.strides[1],
                                      bpc, 0, F, rows.ctypes.data_as(u64), sse.ctypes.data_as(u64),
                                      mse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return {"rows": rows, "sse": sse, "mse": mse}


def psnr_db(mse: float, bpc: int, psnr_max: float = 0.0, mutation: int = 0) -> float:
    return load(mutation).vmx_oracle_psnr_db(mse, bpc, psnr_max)


def batch(ref: np.ndarray, dis: np.ndarray, bpc: int, threads: Optional[int] = None,
          moments: bool = True, psnr_rows: bool = True):
    """Oracle over a (F, H, W) batch, one frame per thread.

    Returns dict with ``moments`` [F][4], ``mse`` [F], ``psnr_rows`` [F][H]."""
    lib = load(0)
    assert ref.ndim == 3 and ref.shape == dis.shape and ref.flags.c_contiguous
    F, h, w = ref.shape
    stride = ref.strides[1]
    out_m = np.zeros((F, 4), dtype=np.float64)
    out_mse = np.zeros(F, dtype=np.float64)
    out_rows = np.zeros((F, h), dtype=np.uint64) if psnr_rows else None
    dp = ctypes.POINTER(ctypes.c_double)
    u64p = ctypes.POINTER(ctypes.c_uint64)

    def one(f: int):
        if moments:
            lib.vmx_oracle_moment_batch(ref.ctypes.data, dis.ctypes.data, w, h, stride, bpc,
                                        f, 1, out_m[f:].ctypes.data_as(dp))
        lib.vmx_oracle_psnr_batch(ref.ctypes.data, dis.ctypes.data, w, h, stride, bpc, f, 1,
                                  out_rows[f:].ctypes.data_as(u64p) if psnr_rows else None,
                                  out_mse[f:].ctypes.data_as(dp))

    n = threads or os.cpu_count() or 1
    if n <= 1 or F == 1:
        for f in range(F):
            one(f)
    else:
        # ctypes releases the GIL during the foreign call, so threads run the
        # C loops in parallel (one frame per thread; no fork involved).
        with ThreadPoolExecutor(max_workers=min(n, F)) as ex:
            list(ex.map(one, range(F)))
    return {"moments": out_m, "mse": out_mse, "psnr_rows": out_rows}
