"""vmx_frames_noalloc against vmx_moment_psnr_frames, both through the C ABI.

The no-alloc call keeps its scratch in a fixed static device array; these
tests run it twice in a row on each batch and hold every output to the
workspace call's, bit for bit (the library's tolerance for every output is
exact equality), and the first and last frames straight to the oracle's.
The file is collected last so that it also runs after all other GPU tests
in one process; it needs nothing they set up.
"""

import ctypes

import numpy as np
import pytest

from exact_reductions_gb300 import _lib, synth


def test_noalloc_rejects_without_touching_the_device():
    """Shape errors come back before any CUDA call (runs without a GPU)."""
    lib = _lib.load()
    fake = ctypes.c_void_p(256)
    # A batch of 16-bit 3840x2160 frames too large for the fixed scratch.
    big = 1024
    need = lib.vmx_workspace_bytes(3840, 2160, 16, big, 3)
    assert need > _lib.NOALLOC_SCRATCH_BYTES
    before = lib.vmx_kernel_launches()
    rc = lib.vmx_frames_noalloc(fake, fake, 3840, 2160, 7680, 16, big, 3, fake, None, None,
                                fake, fake, None, None, None)
    assert rc == _lib.VMX_ESCRATCH
    assert b"scratch" in lib.vmx_strerror(rc)
    rc = lib.vmx_frames_noalloc(fake, fake, 0, 2160, 7680, 16, 1, 3, fake, None, None,
                                fake, fake, None, None, None)
    assert rc == _lib.VMX_EINVAL
    # Null planes, a short or odd stride, a missing output, a misaligned
    # 16-bit plane: all argument errors, found before the device lookup (this
    # test runs without a GPU, so any CUDA call would have failed otherwise).
    odd = ctypes.c_void_p(257)
    for args in [(None, fake, 64, 8, 128, 16, 1, 3, fake, None, None, fake, fake),
                 (fake, None, 64, 8, 128, 16, 1, 3, fake, None, None, fake, fake),
                 (fake, fake, 64, 8, 126, 16, 1, 3, fake, None, None, fake, fake),
                 (fake, fake, 64, 8, 129, 16, 1, 3, fake, None, None, fake, fake),
                 (fake, fake, 64, 8, 128, 16, 1, 3, None, None, None, fake, fake),
                 (fake, fake, 64, 8, 128, 16, 1, 3, fake, None, None, None, fake),
                 (fake, fake, 64, 8, 128, 16, 1, 3, fake, None, None, fake, None),
                 (odd, fake, 64, 8, 128, 16, 1, 3, fake, None, None, fake, fake),
                 (fake, fake, 64, 8, 128, 16, 1, 4, fake, None, None, fake, fake)]:
        assert lib.vmx_frames_noalloc(*args, None, None, None) == _lib.VMX_EINVAL, args
    assert lib.vmx_kernel_launches() == before


@pytest.mark.gpu
@pytest.mark.parametrize("key,frames", [("C2", 16), ("T1", 1), ("T2", 1), ("C4", 4)])
def test_noalloc_matches_workspace_call(key, frames):
    import torch

    from gpu_helpers import oracle_frames

    lib = _lib.load()
    wl = synth.WORKLOADS[key]
    ref, dis = wl.batch(frames)
    F, H, W = ref.shape
    stride = W * ref.itemsize
    R = torch.from_numpy(ref).to("cuda:0")
    D = torch.from_numpy(dis).to("cuda:0")
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.vmx_workspace_bytes(W, H, wl.bpc, F, 3) <= _lib.NOALLOC_SCRATCH_BYTES

    def outputs():
        return {"moments": torch.empty(F * 4, dtype=torch.float64, device="cuda:0"),
                "s2_rows": torch.empty(F * 2 * H, dtype=torch.int64, device="cuda:0"),
                "s2_sums": torch.empty(F * 2, dtype=torch.int64, device="cuda:0"),
                "psnr_rows": torch.empty(F * H, dtype=torch.int64, device="cuda:0"),
                "mse": torch.empty(F, dtype=torch.float64, device="cuda:0"),
                "noise_sums": torch.empty(F, dtype=torch.int64, device="cuda:0")}

    # The call every other test holds to the oracle, with a caller workspace.
    want = outputs()
    nbytes = lib.vmx_workspace_bytes(W, H, wl.bpc, F, 3)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda:0")
    rc = lib.vmx_moment_psnr_frames(
        R.data_ptr(), D.data_ptr(), W, H, stride, wl.bpc, F, want["moments"].data_ptr(),
        want["s2_rows"].data_ptr(), want["s2_sums"].data_ptr(), want["psnr_rows"].data_ptr(),
        want["mse"].data_ptr(), want["noise_sums"].data_ptr(), ws.data_ptr(), nbytes, stream)
    assert rc == _lib.VMX_OK
    assert lib.vmx_workspace_status(ws.data_ptr(), stream) == _lib.VMX_OK

    # Two no-alloc calls in a row into the same (pre-poisoned) outputs.
    got = outputs()
    status = torch.full((1,), 7, dtype=torch.int32, device="cuda:0")
    for call in range(2):
        for t in got.values():
            t.fill_(-1)
        status.fill_(7)
        before = lib.vmx_kernel_launches()
        rc = lib.vmx_frames_noalloc(
            R.data_ptr(), D.data_ptr(), W, H, stride, wl.bpc, F, 3, got["moments"].data_ptr(),
            got["s2_rows"].data_ptr(), got["s2_sums"].data_ptr(), got["psnr_rows"].data_ptr(),
            got["mse"].data_ptr(), got["noise_sums"].data_ptr(), status.data_ptr(), stream)
        assert rc == _lib.VMX_OK, lib.vmx_strerror(rc)
        assert lib.vmx_kernel_launches() == before + 1
        torch.cuda.synchronize()
        assert int(status.item()) == 0, call
        for name in want:
            a = want[name].cpu().numpy().view(np.uint64)
            b = got[name].cpu().numpy().view(np.uint64)
            assert np.array_equal(a, b), (call, name)

    # And straight against the oracle on the first and last frames.
    for f, w in zip(sorted({0, F - 1}), oracle_frames(ref, dis, wl.bpc, sorted({0, F - 1}))):
        m = got["moments"].cpu().numpy().reshape(F, 4)[f]
        assert np.array_equal(m.view(np.uint64), w["moments"].view(np.uint64)), f
        rows = got["s2_rows"].cpu().numpy().view(np.uint64).reshape(F, 2, H)[f]
        assert np.array_equal(rows, w["s2_rows"]), f
        sums = got["s2_sums"].cpu().numpy().view(np.uint64).reshape(F, 2)[f]
        assert np.array_equal(sums, w["s2_sums"]), f
        prow = got["psnr_rows"].cpu().numpy().view(np.uint64).reshape(F, H)[f]
        assert np.array_equal(prow, w["psnr_rows"]), f
        mse = got["mse"].cpu().numpy()[f]
        assert np.array_equal(np.float64(mse).view(np.uint64), np.float64(w["mse"]).view(np.uint64)), f
        assert int(got["noise_sums"].cpu().numpy().view(np.uint64)[f]) == w["noise_sum"], f
