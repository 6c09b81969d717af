"""ctypes binding of libvmx (``include/vmx.h``): argument marshalling only.

The shared library is built in-tree by ``exact_reductions_gb300.build``; if it
is missing, importing anything that needs it raises, naming the build step.
There is no fallback: every step of the computation runs in libvmx's CUDA
kernels.
"""

from __future__ import annotations

import contextlib
import ctypes
import os

from . import build as _build

VMX_OK = 0
VMX_EINVAL = -1
VMX_ENOMEM = -2
VMX_ECUDA = -3
VMX_ETIMEOUT = -4
VMX_ESCRATCH = -5
VMX_ECHECK = -6
NOALLOC_SCRATCH_BYTES = 16 << 20
FEATURE_MOMENT = 1
FEATURE_PSNR = 2
FLAG_CLEARED = 1
FLAG_OVERLAP = 2

# Every symbol include/vmx.h declares: name -> (restype, argtypes).
_vp, _i32, _i64, _sz, _u64, _dbl = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                    ctypes.c_size_t, ctypes.c_uint64, ctypes.c_double)
SIGNATURES = {
    "vmx_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "vmx_moment_frames": (_i32, [_vp, _vp, _i32, _i32, _i64, _i32, _i32, _vp, _vp, _vp, _vp, _sz,
                                 _vp]),
    "vmx_float_psnr_frames": (_i32, [_vp, _vp, _i32, _i32, _i64, _i32, _i32, _vp, _vp, _vp, _vp,
                                     _sz, _vp]),
    "vmx_moment_psnr_frames": (_i32, [_vp, _vp, _i32, _i32, _i64, _i32, _i32, _vp, _vp, _vp, _vp,
                                      _vp, _vp, _vp, _sz, _vp]),
    "vmx_workspace_clear": (_i32, [_vp, _sz, _i32, _i32, _i32, _i32, _i32, _vp]),
    "vmx_workspace_clear_n": (_i32, [_vp, _sz, _sz, _i32, _i32, _i32, _i32, _i32, _vp]),
    "vmx_integer_psnr_frames": (_i32, [_vp, _vp, _i32, _i32, _i64, _i32, _i32, _vp, _vp, _vp,
                                       _vp]),
    "vmx_frames_ex": (_i32, [_vp, _vp, _i32, _i32, _i64, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp,
                             _vp, _vp, _sz, ctypes.c_uint, _vp]),
    "vmx_workspace_status": (_i32, [_vp, _vp]),
    "vmx_workspace_stats": (_i32, [_vp, _vp, _vp]),
    "vmx_psnr_db": (_i32, [_vp, _i32, _i32, _dbl, _vp]),
    "vmx_integer_psnr_db": (_i32, [_vp, _i32, _i32, _dbl, _vp]),
    "vmx_host_workspace_bytes": (_sz, [_i32, _i32, _i64, _i32, _i32, _i32]),
    "vmx_frames_host": (_i32, [_vp, _vp, _i32, _i32, _i64, _i32, _i32, _i32, _vp, _vp, _vp, _vp,
                               _vp, _dbl, _i32, _vp, _sz, _vp]),
    "vmx_frames_host_traffic": (None, [_i32, _i32, _i64, _i32, _i32, _i32, _i32, _vp, _vp]),
    "vmx_frames_noalloc": (_i32, [_vp, _vp, _i32, _i32, _i64, _i32, _i32, _i32, _vp, _vp, _vp,
                                  _vp, _vp, _vp, _vp, _vp]),
    "vmx_checked_build": (_i32, []),
    "vmx_check_status": (_i32, [_vp]),
    "vmx_phase_times": (_i32, [_vp, _i32]),
    "vmx_strerror": (ctypes.c_char_p, [_i32]),
    "vmx_kernel_launches": (_u64, []),
    "vmx_version": (_i32, []),
}

_lib = None


def lib_path() -> str:
    return _build.LIB


def bind(path: str) -> ctypes.CDLL:
    """Open a libvmx build at `path` with every entry point's signature set."""
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load() -> ctypes.CDLL:
    """Load libvmx.so (built by ``exact_reductions_gb300.build.build_lib()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise ImportError(
            f"libvmx is not built ({path} missing): run "
            "`python -c 'import __graft_entry__ as g; g.build()'` first")
    _lib = bind(path)
    return _lib


@contextlib.contextmanager
def using(path: str):
    """Run the enclosed calls on the libvmx build at `path` (a variant such as
    a timing or checked build), then go back to the default library."""
    global _lib
    old = _lib
    _lib = bind(path)
    try:
        yield _lib
    finally:
        _lib = old


class VmxError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = load().vmx_strerror(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def check(status: int, where: str) -> None:
    if status != VMX_OK:
        raise VmxError(status, where)
