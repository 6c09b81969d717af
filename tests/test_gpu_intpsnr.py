"""integer_psnr on the GPU against the oracle, plane by plane (psnr_y,
psnr_cb, psnr_cr; the page on the Metal kernel batch T8-1c..k, "Feature
scope"): every row sum and plane sum exactly, every MSE double bit for bit,
on luma and 4:2:0 chroma shapes, every depth, ragged widths, padded strides,
misaligned planes, container values past the depth, and sums past 2^53."""

import numpy as np
import pytest
import torch

import oracle
from exact_reductions_gb300 import api, synth
from gpu_helpers import to_device, u64

pytestmark = pytest.mark.gpu


def _check(ref, dis, bpc, width=None, misalign=0):
    out = api.integer_psnr(to_device(ref, misalign), to_device(dis, misalign), bpc, width=width,
                           rows=True)
    torch.cuda.synchronize()
    want = oracle.integer_psnr_batch(ref, dis, bpc, width=width)
    assert np.array_equal(u64(out["rows"]), want["rows"])
    assert np.array_equal(u64(out["sse"]), want["sse"])
    assert np.array_equal(out["mse"].cpu().numpy().view(np.uint64), want["mse"].view(np.uint64))
    return out, want


def _batch(seed, F, H, W, bpc, mode="uniform", stride=None):
    rng = np.random.default_rng(seed)
    pairs = [synth.random_plane_pair(rng, W, H, bpc, stride_samples=stride, mode=mode)
             for _ in range(F)]
    return np.stack([p[0] for p in pairs]), np.stack([p[1] for p in pairs])


@pytest.mark.parametrize("bpc", [8, 10, 12, 16])
def test_luma_and_chroma_planes(bpc):
    """A 4:2:0 frame's three planes, one call each."""
    H, W = 240, 320
    planes = {"y": _batch(bpc, 3, H, W, bpc), "cb": _batch(bpc + 1, 3, H // 2, W // 2, bpc),
              "cr": _batch(bpc + 2, 3, H // 2, W // 2, bpc)}
    for name, (r, d) in planes.items():
        _check(r, d, bpc)
    got = api.integer_psnr_planes({k: (torch.from_numpy(r).cuda(), torch.from_numpy(d).cuda())
                                   for k, (r, d) in planes.items()}, bpc)
    for name, (r, d) in planes.items():
        want = oracle.integer_psnr_batch(r, d, bpc)
        db = api.integer_psnr_db(got[name]["mse"].cpu().numpy(), bpc)
        for f in range(3):
            ref_db = oracle.psnr_db(want["mse"][f] / 4.0 ** (bpc - 8), bpc)
            assert db[f] == ref_db, (name, f)


@pytest.mark.parametrize("bpc", [8, 16])
@pytest.mark.parametrize("W,H", [(1, 1), (7, 5), (255, 3), (1001, 17), (2049, 9), (32768, 2)])
def test_ragged_shapes(W, H, bpc):
    for mode in ("uniform", "extreme"):
        ref, dis = _batch(W + H + bpc, 2, H, W, bpc, mode)
        _check(ref, dis, bpc)


@pytest.mark.parametrize("bpc", [8, 12, 16])
def test_padded_stride_misaligned_and_overrange(bpc):
    W, S, H = 1000, 1032, 21
    ref, dis = _batch(60 + bpc, 2, H, W, bpc, "overrange" if bpc > 8 else "uniform", stride=S)
    _check(ref, dis, bpc, width=W)
    _check(ref, dis, bpc, width=W, misalign=1)


def test_sums_past_2_53():
    """16-bit 3840x2160 frames far apart (ref in [32768, 65535], dis in
    [0, 32767]): each plane's sum passes 2^53 and the MSE rounds it once."""
    wl = synth.WORKLOADS["C5a"]
    ref, dis = wl.batch(2)
    _, want = _check(ref, dis, 16)
    assert int(want["sse"].min()) > 1 << 53
