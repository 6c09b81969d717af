"""libvmx loads, exports every symbol include/vmx.h declares, and its host
logic behaves, all without a GPU (no compute call reaches the device)."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from exact_reductions_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "vmx.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vmx_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build_lib()
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names == sorted(_lib.SIGNATURES)
    for name in names:
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"{name} has no binding"


def test_version_and_strerror(lib):
    assert lib.vmx_version() == 10200
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.vmx_strerror(code) and lib.vmx_strerror(code) != b"unknown status"
    assert lib.vmx_strerror(-99) == b"unknown status"


def test_default_build_has_no_phase_times(lib):
    """Only a timing build (VMX_PHASE_TIMES=1) keeps phase counters; the
    default library refuses the call without touching the GPU."""
    import numpy as np
    out = np.zeros(16, dtype=np.uint64)
    assert lib.vmx_phase_times(out.ctypes.data, 1) == _lib.VMX_EINVAL
    assert lib.vmx_phase_times(None, 0) == _lib.VMX_EINVAL


def test_default_build_is_not_checked(lib):
    """The default library compiles its index checks to nothing: it says so,
    and vmx_check_status has nothing to report (no CUDA call is made)."""
    assert lib.vmx_checked_build() == 0
    assert lib.vmx_check_status(None) == _lib.VMX_OK


@pytest.mark.parametrize("args", [
    (0, 16, 16, 1, 3), (32769, 1, 16, 1, 3), (16, 0, 16, 1, 3), (16, 16, 7, 1, 3),
    (16, 16, 17, 1, 3), (16, 16, 16, 0, 3), (16, 16, 16, 1, 0), (16, 16, 16, 1, 4),
    (8192, 8192, 16, 1, 3)])
def test_workspace_rejects_bad_shapes(lib, args):
    assert lib.vmx_workspace_bytes(*args) == 0


def test_workspace_sizes(lib):
    small = lib.vmx_workspace_bytes(320, 240, 8, 1, 3)
    assert small > 0 and small % 256 == 0
    # Frames above 2^21 pixels with second moments keep per-row sums and odd
    # counts; above 2^23 pixels also per-row runs.
    a = lib.vmx_workspace_bytes(3840, 2160, 16, 16, 3)
    b = lib.vmx_workspace_bytes(3840, 2160, 16, 16, 2)
    assert a >= b + 16 * 2 * 2160 * (8 + 4)
    assert lib.vmx_workspace_bytes(3840, 2160, 16, 32, 3) > a
    big = lib.vmx_workspace_bytes(7680, 4320, 16, 1, 3)
    assert big >= 2 * 4320 * (8 + 4 + 16)


def test_argument_errors_launch_nothing(lib):
    """Bad arguments come back as VMX_EINVAL before any CUDA call."""
    launches = lib.vmx_kernel_launches()
    buf = ctypes.create_string_buffer(64)
    p = ctypes.addressof(buf)
    E = _lib.VMX_EINVAL
    # null planes, stride too small, odd uint16 stride, bpc out of range
    assert lib.vmx_moment_frames(None, p, 4, 4, 8, 16, 1, p, None, None, p, 1 << 20, None) == E
    assert lib.vmx_moment_frames(p, p, 4, 4, 6, 16, 1, p, None, None, p, 1 << 20, None) == E
    assert lib.vmx_moment_frames(p, p, 4, 4, 9, 16, 1, p, None, None, p, 1 << 20, None) == E
    assert lib.vmx_moment_frames(p, p, 4, 4, 8, 17, 1, p, None, None, p, 1 << 20, None) == E
    # missing outputs, zero frames, workspace too small
    assert lib.vmx_moment_frames(p, p, 4, 4, 8, 16, 1, None, None, None, p, 1 << 20, None) == E
    assert lib.vmx_float_psnr_frames(p, p, 4, 4, 8, 16, 1, None, p, None, p, 1 << 20, None) == E
    assert lib.vmx_moment_psnr_frames(p, p, 4, 4, 8, 16, 0, p, None, None, p, p, None, p,
                                      1 << 20, None) == E
    aligned = (p + 255) & ~255
    assert lib.vmx_moment_frames(p, p, 4, 4, 8, 16, 1, p, None, None, aligned, 16, None) == E
    assert lib.vmx_frames_host(None, p, 4, 4, 8, 16, 1, 3, p, None, p, p, None, 0.0, 1, None, 0,
                               None) == E
    # integer_psnr: null planes or outputs, stride, depth, odd uint16 stride, width, frames
    assert lib.vmx_integer_psnr_frames(None, p, 4, 4, 8, 16, 1, p, p, None, None) == E
    assert lib.vmx_integer_psnr_frames(p, p, 4, 4, 8, 16, 1, None, p, None, None) == E
    assert lib.vmx_integer_psnr_frames(p, p, 4, 4, 8, 16, 1, p, None, None, None) == E
    assert lib.vmx_integer_psnr_frames(p, p, 4, 4, 6, 16, 1, p, p, None, None) == E
    assert lib.vmx_integer_psnr_frames(p, p, 4, 4, 8, 7, 1, p, p, None, None) == E
    assert lib.vmx_integer_psnr_frames(p, p, 4, 4, 9, 16, 1, p, p, None, None) == E
    assert lib.vmx_integer_psnr_frames(p, p, 32769, 1, 1 << 17, 16, 1, p, p, None, None) == E
    assert lib.vmx_integer_psnr_frames(p, p, 4, 4, 8, 16, 0, p, p, None, None) == E
    assert lib.vmx_kernel_launches() == launches


def test_injected_launch_failure(lib, monkeypatch):
    """VMX_TEST_FAIL_AT makes a stage fail on the host; the error surfaces."""
    buf = ctypes.create_string_buffer(1 << 16)
    p = (ctypes.addressof(buf) + 255) & ~255
    monkeypatch.setenv("VMX_TEST_FAIL_AT", "launch")
    st = lib.vmx_moment_frames(p, p, 4, 4, 8, 16, 1, p, None, None, p, 1 << 15, None)
    assert st == _lib.VMX_ECUDA and b"injected" in lib.vmx_strerror(st)
    st = lib.vmx_integer_psnr_frames(p, p, 4, 4, 8, 16, 1, p, p, None, None)
    assert st == _lib.VMX_ECUDA and b"injected" in lib.vmx_strerror(st)
    monkeypatch.setenv("VMX_TEST_FAIL_AT", "alloc")
    st = lib.vmx_moment_frames(p, p, 4, 4, 8, 16, 1, p, None, None, None, 0, None)
    assert st == _lib.VMX_ENOMEM
    monkeypatch.setenv("VMX_TEST_FAIL_AT", "status")
    assert lib.vmx_workspace_status(p, None) == _lib.VMX_ETIMEOUT
    with pytest.raises(_lib.VmxError):
        _lib.check(lib.vmx_workspace_status(p, None), "status")


def test_psnr_db_matches_oracle(lib):
    """The host PSNR step equals the oracle's on the same MSE values."""
    rng = np.random.default_rng(11)
    mse = np.concatenate([[0.0, 1e-12, 1e-10, 1.0], rng.uniform(0, 400, 200),
                          10.0 ** rng.uniform(-9, 4, 200)])
    for bpc in (8, 10, 12, 16):
        for cap in (0.0, 60.0):
            out = np.zeros_like(mse)
            assert lib.vmx_psnr_db(mse.ctypes.data, mse.size, bpc, cap, out.ctypes.data) == 0
            want = np.array([oracle.psnr_db(m, bpc, cap) for m in mse])
            assert np.array_equal(out.view(np.uint64), want.view(np.uint64))


def test_integer_psnr_db_is_the_same_ratio(lib):
    """integer_psnr's PSNR (vmx_integer_psnr_db, through the C ABI and the
    binding): the MSE in codeword units over 4^(bpc - 8) goes through the
    same host step, and equals the oracle's PSNR of that normalised MSE bit
    for bit (the division by a power of two is exact)."""
    from exact_reductions_gb300 import api
    rng = np.random.default_rng(12)
    for bpc in (8, 10, 12, 16):
        mse = np.concatenate([[0.0, 1.0], rng.uniform(0, 4.0 ** bpc, 100)])
        for cap in (0.0, 60.0):
            want = np.array([oracle.psnr_db(m / 4.0 ** (bpc - 8), bpc, cap) for m in mse])
            out = np.zeros_like(mse)
            assert lib.vmx_integer_psnr_db(mse.ctypes.data, mse.size, bpc, cap,
                                           out.ctypes.data) == _lib.VMX_OK
            assert np.array_equal(out.view(np.uint64), want.view(np.uint64)), (bpc, cap)
            got = api.integer_psnr_db(mse, bpc, cap)
            assert np.array_equal(got.view(np.uint64), want.view(np.uint64)), (bpc, cap)
        peak = float((1 << bpc) - 1)
        assert api.integer_psnr_db(np.array([peak * peak]), bpc)[0] == 0.0
    x = np.zeros(1)
    assert lib.vmx_integer_psnr_db(None, 1, 16, 0.0, x.ctypes.data) == _lib.VMX_EINVAL
    assert lib.vmx_integer_psnr_db(x.ctypes.data, 1, 17, 0.0, x.ctypes.data) == _lib.VMX_EINVAL
    assert lib.vmx_integer_psnr_db(x.ctypes.data, -1, 16, 0.0, x.ctypes.data) == _lib.VMX_EINVAL


def test_host_traffic(lib):
    h2d, d2h = ctypes.c_uint64(), ctypes.c_uint64()
    lib.vmx_frames_host_traffic(3840, 2160, 7680, 16, 16, 3, 0, ctypes.addressof(h2d),
                                ctypes.addressof(d2h))
    assert h2d.value == 2 * 16 * 2160 * 7680
    assert d2h.value == 16 * 4 * 8 + 16 * 2160 * 8 + 16 * 8


def test_pipelining_flags_are_checked_before_any_cuda_call():
    """Unknown flags, or flags without a workspace, are argument errors."""
    lib = _lib.load()
    p = ctypes.c_void_p(256)
    assert lib.vmx_frames_ex(p, p, 64, 8, 128, 16, 1, 3, p, None, None, p, p, None, p, 1 << 20,
                             4, None) == _lib.VMX_EINVAL
    assert lib.vmx_frames_ex(p, p, 64, 8, 128, 16, 1, 3, p, None, None, p, p, None, None, 0,
                             _lib.FLAG_CLEARED, None) == _lib.VMX_EINVAL
    assert lib.vmx_workspace_clear(None, 1 << 20, 64, 8, 16, 1, 3, None) == _lib.VMX_EINVAL
    assert lib.vmx_workspace_clear(p, 16, 64, 8, 16, 1, 3, None) == _lib.VMX_EINVAL
    # the clear of workspaces back to back: pointer, count, spacing (a
    # multiple of 256, at least one workspace), shape
    ok = 1 << 20
    assert lib.vmx_workspace_clear_n(None, ok, 2, 64, 8, 16, 1, 3, None) == _lib.VMX_EINVAL
    assert lib.vmx_workspace_clear_n(p, ok, 0, 64, 8, 16, 1, 3, None) == _lib.VMX_EINVAL
    assert lib.vmx_workspace_clear_n(p, ok + 16, 2, 64, 8, 16, 1, 3, None) == _lib.VMX_EINVAL
    assert lib.vmx_workspace_clear_n(p, 256, 2, 64, 8, 16, 1, 3, None) == _lib.VMX_EINVAL
    assert lib.vmx_workspace_clear_n(ctypes.c_void_p(272), ok, 2, 64, 8, 16, 1, 3, None) == _lib.VMX_EINVAL
    assert lib.vmx_workspace_clear_n(p, ok, 2, 64, 8, 7, 1, 3, None) == _lib.VMX_EINVAL

