"""Helpers of the GPU parity tests: run libvmx on device tensors and the CPU
oracle on the same arrays, then compare every output exactly."""

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
from exact_reductions_gb300 import api


def u64(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int64).numpy().view(np.uint64)


def to_device(arr: np.ndarray, misalign: int = 0) -> torch.Tensor:
    """Copy a (F, H, S) array to cuda:0, optionally `misalign` samples past a
    16-byte boundary (the planes then take the scalar-load path)."""
    arr = np.ascontiguousarray(arr)
    t = torch.from_numpy(arr)
    if not misalign:
        return t.to("cuda:0")
    flat = torch.empty(arr.size + 16, dtype=t.dtype, device="cuda:0")
    view = flat[misalign:misalign + arr.size].view(arr.shape)
    view.copy_(t.to("cuda:0"))
    return view


def oracle_frame(ref2d, dis2d, bpc, width=None):
    m, rows = oracle.moment(ref2d, dis2d, bpc, rows=True, width=width)
    prow, mse = oracle.psnr(ref2d, dis2d, bpc, width=width)
    sums = oracle.moment_sums(ref2d, dis2d, bpc, width=width)
    noise = oracle.psnr_noise_sum(ref2d, dis2d, bpc, width=width)
    return {"moments": m, "s2_rows": rows, "psnr_rows": prow, "mse": mse,
            "s2_sums": np.array(sums[2:], dtype=np.uint64), "noise_sum": noise}


def oracle_frames(ref, dis, bpc, frames, width=None, threads=16):
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda f: oracle_frame(ref[f], dis[f], bpc, width), frames))


def same_doubles(a, b) -> bool:
    a = np.ascontiguousarray(a, dtype=np.float64)
    b = np.ascontiguousarray(b, dtype=np.float64)
    return a.shape == b.shape and np.array_equal(a.view(np.uint64), b.view(np.uint64))


def run_and_check(ref, dis, bpc, width=None, features=3, frames=None, misalign=0,
                  expect_runs=None):
    """Run libvmx on the whole batch and compare frames `frames` (default:
    all) with the oracle: every double bit for bit, every uint64 exactly."""
    r = to_device(ref, misalign)
    d = to_device(dis, misalign)
    out = api.frames(r, d, bpc, features=features, width=width, s2_rows=True, sums=True)
    torch.cuda.synchronize()
    assert api.workspace_status(out["_workspace"]) == 0
    stats = api.workspace_stats(out["_workspace"])
    F = ref.shape[0]
    idx = list(range(F)) if frames is None else list(frames)
    want = oracle_frames(ref, dis, bpc, idx, width)
    got = {k: v for k, v in out.items() if not k.startswith("_")}
    for f, w in zip(idx, want):
        if features & 1:
            assert same_doubles(got["moments"].cpu().numpy()[f], w["moments"]), \
                (f, got["moments"].cpu().numpy()[f], w["moments"])
            assert np.array_equal(u64(got["s2_rows"])[f], w["s2_rows"]), f
            assert np.array_equal(u64(got["s2_sums"])[f], w["s2_sums"]), \
                (f, u64(got["s2_sums"])[f], w["s2_sums"])
        if features & 2:
            assert np.array_equal(u64(got["psnr_rows"])[f], w["psnr_rows"]), f
            assert same_doubles(got["mse"].cpu().numpy()[f], w["mse"]), f
            assert int(u64(got["noise_sums"])[f]) == w["noise_sum"], f
    return out, stats
