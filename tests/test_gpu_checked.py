"""The checked build (VMX_CHECK=1: every index the kernels compute into one of
their arrays is compared with the array's extent before the access; an index
out of range is reported and the access skipped, never trapped) on the edge
cases of the other GPU tests: every output equal to the oracle's and no
check failed. Then a test-only setting makes the kernels take the per-plane
row arrays as one element shorter than they are: the checks fire, the calls
report VMX_ECHECK, nothing goes out of bounds, and the next call is exact."""

import numpy as np
import pytest
import torch

import oracle
from exact_reductions_gb300 import _lib, api, build, synth
from gpu_helpers import run_and_check, to_device, u64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked():
    lib = _lib.bind(build.build_variant("checked", ["VMX_CHECK=1"]))
    assert lib.vmx_checked_build() == 1
    return lib


def _pair(seed, F, H, S, bpc, mode="uniform", W=None):
    rng = np.random.default_rng(seed)
    refs, diss = [], []
    for _ in range(F):
        r, d = synth.random_plane_pair(rng, W or S, H, bpc, stride_samples=S, mode=mode)
        refs.append(r)
        diss.append(d)
    return np.stack(refs), np.stack(diss)


def _no_integer_psnr_check_failed(lib):
    assert lib.vmx_check_status(torch.cuda.current_stream().cuda_stream) == _lib.VMX_OK


@pytest.mark.parametrize("bpc", [8, 10, 16])
@pytest.mark.parametrize("W,H", [(1, 1), (37, 1), (7, 5), (257, 9), (2049, 11)])
def test_checked_ragged_shapes(monkeypatch, checked, W, H, bpc):
    monkeypatch.setattr(_lib, "_lib", checked)
    for mode in ("uniform", "extreme"):
        ref, dis = _pair(W * 131 + H + bpc, 2, H, W, bpc, mode)
        run_and_check(ref, dis, bpc)


@pytest.mark.parametrize("bpc", [8, 16])
def test_checked_padded_and_misaligned(monkeypatch, checked, bpc):
    monkeypatch.setattr(_lib, "_lib", checked)
    W, S, H = 1000, 1024 + 8, 40
    ref, dis = _pair(5, 3, H, S, bpc, W=W)
    run_and_check(ref, dis, bpc, width=W)
    ref, dis = _pair(6, 2, 64, 640, bpc)
    run_and_check(ref, dis, bpc, misalign=1)


@pytest.mark.parametrize("key,frames", [("T1", 1), ("T2", 1), ("T3", 1), ("T4", 2), ("C4", 2)])
def test_checked_past_2_53_and_2_55(monkeypatch, checked, key, frames):
    """The walks, the closed forms, the look-back and the runs."""
    monkeypatch.setattr(_lib, "_lib", checked)
    wl = synth.WORKLOADS[key]
    ref, dis = wl.batch(frames)
    run_and_check(ref, dis, wl.bpc)


def test_checked_widest_rows_and_single_column(monkeypatch, checked):
    monkeypatch.setattr(_lib, "_lib", checked)
    rng = np.random.default_rng(91)
    ref, dis = synth.random_plane_pair(rng, 32768, 3, 16)
    run_and_check(ref[None], dis[None], 16)
    ref, dis = synth.random_plane_pair(rng, 1, 300, 16)
    run_and_check(ref[None], dis[None], 16)


@pytest.mark.parametrize("bpc,W,H,S", [(8, 37, 5, 37), (10, 1000, 17, 1024), (16, 3840, 64, 3840),
                                        (16, 257, 9, 264)])
def test_checked_integer_psnr(monkeypatch, checked, bpc, W, H, S):
    monkeypatch.setattr(_lib, "_lib", checked)
    ref, dis = _pair(300 + W, 3, H, S, bpc, W=W)
    out = api.integer_psnr(to_device(ref), to_device(dis), bpc, width=W, rows=True)
    torch.cuda.synchronize()
    _no_integer_psnr_check_failed(checked)
    for f in range(ref.shape[0]):
        rows, sse, mse = oracle.integer_psnr(ref[f], dis[f], bpc, width=W)
        assert np.array_equal(u64(out["rows"])[f], rows)
        assert int(u64(out["sse"])[f]) == sse
        assert out["mse"].cpu().numpy()[f] == mse


def test_checks_fire_and_skip_without_faulting(monkeypatch, checked):
    """With the row arrays taken as one element short, the last row's record
    is an index out of range: the frame call reports VMX_ECHECK (a status
    word, not a trap), integer_psnr's flag reports it too, and once the
    setting is gone the next calls are exact."""
    monkeypatch.setattr(_lib, "_lib", checked)
    wl = synth.WORKLOADS["T1"]
    ref, dis = wl.batch(1)
    R, D = to_device(ref), to_device(dis)
    monkeypatch.setenv("VMX_TEST_CHECK_SHRINK", "1")
    out = api.frames(R, D, 16, s2_rows=True, sums=True)
    torch.cuda.synchronize()
    assert api.workspace_status(out["_workspace"]) == _lib.VMX_ECHECK
    api.integer_psnr(R, D, 16, rows=True)
    torch.cuda.synchronize()
    assert checked.vmx_check_status(torch.cuda.current_stream().cuda_stream) == _lib.VMX_ECHECK
    monkeypatch.delenv("VMX_TEST_CHECK_SHRINK")
    _no_integer_psnr_check_failed(checked)  # the flag was cleared by the read
    run_and_check(ref, dis, 16)
    api.integer_psnr(R, D, 16, rows=True)
    torch.cuda.synchronize()
    _no_integer_psnr_check_failed(checked)
