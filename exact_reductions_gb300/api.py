"""Torch-facing calls of libvmx: tensors in, tensors out, marshalling only.

Planes are CUDA tensors of shape (frames, height, stride_samples), dtype
uint8 (8 bpc) or uint16 (9..16 bpc), rows ``stride_samples`` apart;
``width`` (default: the last dimension) is how many samples of each row
count. Work runs on the current CUDA stream of the tensors' device. The
PSNR (a host function of the MSE) is ``psnr_db`` (``integer_psnr_db`` for
``integer_psnr``, one plane a call).
"""

from __future__ import annotations

import ctypes
from typing import Dict, Optional

import numpy as np
import torch

from . import _lib

_ALIGN = 256


def _dtype_ok(t: torch.Tensor, bpc: int) -> None:
    want = torch.uint8 if bpc == 8 else torch.uint16
    if t.dtype != want:
        raise TypeError(f"bpc {bpc} needs {want} samples, got {t.dtype}")


def _geometry(ref: torch.Tensor, dis: torch.Tensor, bpc: int, width: Optional[int]):
    if ref.dim() == 2:
        ref, dis = ref.unsqueeze(0), dis.unsqueeze(0)
    if ref.dim() != 3 or ref.shape != dis.shape:
        raise ValueError("ref and dis must both be (frames, height, stride) tensors")
    _dtype_ok(ref, bpc)
    _dtype_ok(dis, bpc)
    if ref.stride(2) != 1 or ref.stride() != dis.stride():
        raise ValueError("rows must be contiguous and both planes laid out alike")
    F, H, S = ref.shape
    if F > 1 and ref.stride(0) != H * ref.stride(1):
        raise ValueError("frames must follow each other at height * stride")
    w = S if width is None else int(width)
    return ref, dis, F, H, w, ref.stride(1) * ref.element_size()


def workspace(nbytes: int, device) -> torch.Tensor:
    """A device byte buffer whose data pointer is 256-byte aligned."""
    buf = torch.empty(nbytes + _ALIGN, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % _ALIGN
    return buf[off:off + nbytes]


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def host_workspace_bytes(width: int, height: int, stride_bytes: int, bpc: int, chunk_frames: int,
                         features: int) -> int:
    return int(_lib.load().vmx_host_workspace_bytes(width, height, stride_bytes, bpc, chunk_frames,
                                                    features))


def workspace_bytes(width: int, height: int, bpc: int, frames: int, features: int) -> int:
    return int(_lib.load().vmx_workspace_bytes(width, height, bpc, frames, features))


def frames(ref: torch.Tensor, dis: torch.Tensor, bpc: int, features: int = 3,
           width: Optional[int] = None, s2_rows: bool = False, sums: bool = False,
           ws: Optional[torch.Tensor] = None) -> Dict[str, torch.Tensor]:
    """float_moment and/or float_psnr (``features`` bits 1 and 2) of a batch.

    Returns device tensors: ``moments`` [F, 4] (ref1, dis1, ref2, dis2),
    ``psnr_rows`` [F, H] (uint64 units), ``mse`` [F], and when asked
    ``s2_rows`` [F, 2, H], ``s2_sums`` [F, 2], ``noise_sums`` [F]."""
    lib = _lib.load()
    ref, dis, F, H, W, stride = _geometry(ref, dis, bpc, width)
    dev = ref.device
    need = int(lib.vmx_workspace_bytes(W, H, bpc, F, features))
    if need == 0:
        raise ValueError("shape rejected by libvmx")
    if ws is None or ws.numel() < need:
        ws = workspace(need, dev)
    out: Dict[str, torch.Tensor] = {}
    m = bool(features & _lib.FEATURE_MOMENT)
    p = bool(features & _lib.FEATURE_PSNR)
    u64 = torch.uint64
    if m:
        out["moments"] = torch.empty((F, 4), dtype=torch.float64, device=dev)
        if s2_rows:
            out["s2_rows"] = torch.empty((F, 2, H), dtype=u64, device=dev)
        if sums:
            out["s2_sums"] = torch.empty((F, 2), dtype=u64, device=dev)
    if p:
        out["psnr_rows"] = torch.empty((F, H), dtype=u64, device=dev)
        out["mse"] = torch.empty((F,), dtype=torch.float64, device=dev)
        if sums:
            out["noise_sums"] = torch.empty((F,), dtype=u64, device=dev)
    st = _stream(dev)
    args = (ref.data_ptr(), dis.data_ptr(), W, H, stride, bpc, F)
    if m and p:
        status = lib.vmx_moment_psnr_frames(
            *args, _ptr(out["moments"]), _ptr(out.get("s2_rows")), _ptr(out.get("s2_sums")),
            _ptr(out["psnr_rows"]), _ptr(out["mse"]), _ptr(out.get("noise_sums")),
            ws.data_ptr(), ws.numel(), st)
    elif m:
        status = lib.vmx_moment_frames(
            *args, _ptr(out["moments"]), _ptr(out.get("s2_rows")), _ptr(out.get("s2_sums")),
            ws.data_ptr(), ws.numel(), st)
    else:
        status = lib.vmx_float_psnr_frames(
            *args, _ptr(out["psnr_rows"]), _ptr(out["mse"]), _ptr(out.get("noise_sums")),
            ws.data_ptr(), ws.numel(), st)
    _lib.check(status, "vmx frames")
    out["_workspace"] = ws
    return out


class FrameGraph:
    """Calls of the fused kernel on fixed device tensors, captured as one CUDA
    graph, for a stream of batches of one shape.

    ``depth`` batches per replay, each with its own workspace and outputs
    (``self.outs[i]``; ``self.out`` is the last): the workspaces (one
    allocation) are cleared first by one strided set
    (``vmx_workspace_clear_n``), then the kernels run back to back, each
    launched to overlap the one before it (``vmx_frames_ex`` with
    ``VMX_FLAG_OVERLAP``).
    ``refs``/``diss`` give each batch's input tensors (copy new frames into
    them between replays); by default every batch reads ``ref``/``dis``.
    Bounded device waits that give up are reported by ``status()``."""

    def __init__(self, ref: torch.Tensor, dis: torch.Tensor, bpc: int, features: int = 3,
                 width: Optional[int] = None, s2_rows: bool = False, sums: bool = False,
                 depth: int = 1, refs=None, diss=None):
        lib = _lib.load()
        refs = list(refs) if refs is not None else [ref] * depth
        diss = list(diss) if diss is not None else [dis] * depth
        if len(refs) != depth or len(diss) != depth:
            raise ValueError("refs and diss need one tensor per batch")
        geo = [_geometry(r, d, bpc, width) for r, d in zip(refs, diss)]
        _, _, F, H, W, stride = geo[0]
        dev = refs[0].device
        need = int(lib.vmx_workspace_bytes(W, H, bpc, F, features))
        if need == 0:
            raise ValueError("shape rejected by libvmx")
        m = bool(features & _lib.FEATURE_MOMENT)
        p = bool(features & _lib.FEATURE_PSNR)
        # One allocation for the batches' workspaces, back to back, so that
        # one strided clear (one graph node) readies them all.
        self.ws_bytes = (need + _ALIGN - 1) // _ALIGN * _ALIGN
        self.ws_all = workspace(self.ws_bytes * depth, dev)
        self.ws = [self.ws_all[i * self.ws_bytes:(i + 1) * self.ws_bytes] for i in range(depth)]
        self.outs = []
        for _ in range(depth):
            o: Dict[str, torch.Tensor] = {}
            if m:
                o["moments"] = torch.empty((F, 4), dtype=torch.float64, device=dev)
                if s2_rows:
                    o["s2_rows"] = torch.empty((F, 2, H), dtype=torch.uint64, device=dev)
                if sums:
                    o["s2_sums"] = torch.empty((F, 2), dtype=torch.uint64, device=dev)
            if p:
                o["psnr_rows"] = torch.empty((F, H), dtype=torch.uint64, device=dev)
                o["mse"] = torch.empty((F,), dtype=torch.float64, device=dev)
                if sums:
                    o["noise_sums"] = torch.empty((F,), dtype=torch.uint64, device=dev)
            self.outs.append(o)
        self.out = self.outs[-1]

        def enqueue():
            st = _stream(dev)
            _lib.check(lib.vmx_workspace_clear_n(self.ws_all.data_ptr(), self.ws_bytes, depth, W, H, bpc,
                                                 F, features, st), "vmx workspace_clear_n")
            for i, ((r, d, _, _, _, _), o, w) in enumerate(zip(geo, self.outs, self.ws)):
                flags = _lib.FLAG_CLEARED | (_lib.FLAG_OVERLAP if i else 0)
                _lib.check(lib.vmx_frames_ex(
                    r.data_ptr(), d.data_ptr(), W, H, stride, bpc, F, features,
                    _ptr(o.get("moments")), _ptr(o.get("s2_rows")), _ptr(o.get("s2_sums")),
                    _ptr(o.get("psnr_rows")), _ptr(o.get("mse")), _ptr(o.get("noise_sums")),
                    w.data_ptr(), w.numel(), flags, st), "vmx frames_ex")

        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            enqueue()  # loads the kernels, outside the capture
        torch.cuda.current_stream(dev).wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            enqueue()

    def replay(self) -> Dict[str, torch.Tensor]:
        self.graph.replay()
        return self.out

    def status(self) -> int:
        """VMX_OK, or the first nonzero status of the batches' workspaces."""
        for w in self.ws:
            st = workspace_status(w)
            if st:
                return st
        return 0


def integer_psnr(ref: torch.Tensor, dis: torch.Tensor, bpc: int, width: Optional[int] = None,
                 rows: bool = False) -> Dict[str, torch.Tensor]:
    """integer_psnr of a batch of one plane (luma or one chroma plane).

    Returns device tensors ``sse`` [F] (uint64: exact sums of squared
    codeword differences), ``mse`` [F] (sse / pixels) and, when asked,
    ``rows`` [F, H]. PSNR in dB: ``integer_psnr_db(mse, bpc)``."""
    lib = _lib.load()
    ref, dis, F, H, W, stride = _geometry(ref, dis, bpc, width)
    dev = ref.device
    out = {"sse": torch.empty((F,), dtype=torch.uint64, device=dev),
           "mse": torch.empty((F,), dtype=torch.float64, device=dev)}
    if rows:
        out["rows"] = torch.empty((F, H), dtype=torch.uint64, device=dev)
    status = lib.vmx_integer_psnr_frames(ref.data_ptr(), dis.data_ptr(), W, H, stride, bpc, F,
                                         _ptr(out["sse"]), _ptr(out["mse"]), _ptr(out.get("rows")),
                                         _stream(dev))
    _lib.check(status, "vmx integer_psnr")
    return out


def integer_psnr_planes(planes: Dict[str, tuple], bpc: int) -> Dict[str, Dict[str, torch.Tensor]]:
    """integer_psnr of several planes, e.g. ``{"y": (ref_y, dis_y), "cb": ...,
    "cr": ...}`` (psnr_y, psnr_cb, psnr_cr): one call per plane, each with
    its own shape."""
    return {name: integer_psnr(r, d, bpc) for name, (r, d) in planes.items()}


def integer_psnr_db(mse, bpc: int, psnr_max: float = 0.0) -> np.ndarray:
    """PSNR in dB of integer_psnr MSE values (codeword units), computed by
    ``vmx_integer_psnr_db`` on the host."""
    mse = np.ascontiguousarray(np.asarray(mse, dtype=np.float64))
    out = np.zeros_like(mse)
    _lib.check(_lib.load().vmx_integer_psnr_db(mse.ctypes.data, mse.size, bpc, float(psnr_max),
                                               out.ctypes.data), "vmx integer psnr")
    return out


def moment_frames(ref, dis, bpc, **kw) -> Dict[str, torch.Tensor]:
    return frames(ref, dis, bpc, features=_lib.FEATURE_MOMENT, **kw)


def float_psnr_frames(ref, dis, bpc, **kw) -> Dict[str, torch.Tensor]:
    return frames(ref, dis, bpc, features=_lib.FEATURE_PSNR, **kw)


def moment_psnr_frames(ref, dis, bpc, **kw) -> Dict[str, torch.Tensor]:
    return frames(ref, dis, bpc, features=3, **kw)


def workspace_status(ws: torch.Tensor) -> int:
    return int(_lib.load().vmx_workspace_status(ws.data_ptr(), _stream(ws.device)))


def workspace_stats(ws: torch.Tensor) -> np.ndarray:
    out = np.zeros(4, dtype=np.uint64)
    _lib.check(_lib.load().vmx_workspace_stats(ws.data_ptr(), _stream(ws.device),
                                               out.ctypes.data), "vmx stats")
    return out


def psnr_db(mse, bpc: int, psnr_max: float = 0.0) -> np.ndarray:
    """PSNR in dB of host MSE values (library reading of the formula)."""
    mse = np.ascontiguousarray(np.asarray(mse, dtype=np.float64))
    out = np.zeros_like(mse)
    _lib.check(_lib.load().vmx_psnr_db(mse.ctypes.data, mse.size, bpc, float(psnr_max),
                                       out.ctypes.data), "vmx psnr")
    return out


def frames_host(ref: np.ndarray, dis: np.ndarray, bpc: int, features: int = 3,
                width: Optional[int] = None, chunk_frames: int = 2, psnr_max: float = 0.0,
                s2_rows: bool = False, ws: Optional[torch.Tensor] = None,
                device: int = 0) -> Dict[str, np.ndarray]:
    """Host-memory entry point: host arrays (F, H, stride) in, host arrays out.

    The copies to the device and back are part of the call."""
    lib = _lib.load()
    if ref.ndim == 2:
        ref, dis = ref[None], dis[None]
    if ref.shape != dis.shape or ref.dtype != dis.dtype or not ref.flags.c_contiguous \
            or not dis.flags.c_contiguous:
        raise ValueError("ref and dis must be C-contiguous (frames, height, stride) arrays")
    F, H, S = ref.shape
    W = S if width is None else int(width)
    stride = S * ref.itemsize
    dev = torch.device("cuda", device)
    need = int(lib.vmx_host_workspace_bytes(W, H, stride, bpc, chunk_frames, features))
    if need == 0:
        raise ValueError("shape rejected by libvmx")
    if ws is None or ws.numel() < need:
        ws = workspace(need, dev)
    m = bool(features & _lib.FEATURE_MOMENT)
    p = bool(features & _lib.FEATURE_PSNR)
    out = {}
    out["moments"] = np.zeros((F, 4), dtype=np.float64) if m else None
    out["s2_rows"] = np.zeros((F, 2, H), dtype=np.uint64) if (m and s2_rows) else None
    out["psnr_rows"] = np.zeros((F, H), dtype=np.uint64) if p else None
    out["mse"] = np.zeros(F, dtype=np.float64) if p else None
    out["psnr"] = np.zeros(F, dtype=np.float64) if p else None

    def ptr(a):
        return None if a is None else a.ctypes.data

    status = lib.vmx_frames_host(ref.ctypes.data, dis.ctypes.data, W, H, stride, bpc, F, features,
                                 ptr(out["moments"]), ptr(out["s2_rows"]), ptr(out["psnr_rows"]),
                                 ptr(out["mse"]), ptr(out["psnr"]), float(psnr_max),
                                 int(chunk_frames), ws.data_ptr(), ws.numel(), _stream(dev))
    _lib.check(status, "vmx frames_host")
    return {k: v for k, v in out.items() if v is not None}


def host_traffic(width: int, height: int, stride_bytes: int, bpc: int, frames_: int,
                 features: int, want_s2_rows: bool = False):
    h2d, d2h = ctypes.c_uint64(0), ctypes.c_uint64(0)
    _lib.load().vmx_frames_host_traffic(width, height, stride_bytes, bpc, frames_, features,
                                        int(want_s2_rows), ctypes.addressof(h2d),
                                        ctypes.addressof(d2h))
    return int(h2d.value), int(d2h.value)


def kernel_launches() -> int:
    return int(_lib.load().vmx_kernel_launches())
