"""Thin ctypes binding over libgdn (include/gdn.h): argument marshalling only.

Every step of the method runs in the CUDA kernels behind the C ABI. Torch is
used here only to own device memory (outputs, workspace) and to name the
current stream. If ``libgdn.so`` is missing the first call raises: there is no
CPU fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_F32, GDN_BF16 = 0, 1
GDN_FLAG_QK_L2NORM = 1
GDN_FLAG_BUILD_CHUNK_INDICES = 2
GDN_FLAG_CHANNEL_GATES = 4
GDN_FLAG_WORKSPACE_GUARDS = 8
GDN_NUM_STAGE_EVENTS = 5
DEV_STATUS_BITS = {1: "bad cu_seqlens", 2: "chunk overflow", 4: "bad chunk table",
                   8: "on-chip wait timed out", 16: "non-finite state or output",
                   32: "index out of range (GDN_DEBUG build)"}
GDN_DEV_DEBUG_INDEX = 32

# Every entry point include/gdn.h declares.
EXPORTED = ("gdn_check_desc", "gdn_nt_max", "gdn_workspace_size", "gdn_build_chunk_indices",
            "gdn_chunk_fwd", "gdn_read_status", "gdn_status_string", "gdn_chunk_fwd_noalloc",
            "gdn_noalloc_read_status", "gdn_test_scan_timeout", "gdn_workspace_regions",
            "gdn_debug_build", "gdn_test_debug_poison",
            "gdn_recurrent_fwd", "gdn_conv_front", "gdn_bwd_workspace_size", "gdn_chunk_bwd")
GDN_NOALLOC_SCRATCH_BYTES = 64 << 20


class GdnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = f"{what}: " if what else ""
        super().__init__(f"{msg}libgdn status {status} ({status_string(status)})")


class GdnDesc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("N", ctypes.c_int32), ("H", ctypes.c_int32),
                ("Hv", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("chunk_size", ctypes.c_int32), ("nt_max", ctypes.c_int32),
                ("qkv_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("l2norm_eps", ctypes.c_float),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("stage_events", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load libgdn.so (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise GdnError(-6, f"{path} is missing (build it with __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        vp, i32, P = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER
        lib.gdn_check_desc.argtypes = [P(GdnDesc)]
        lib.gdn_check_desc.restype = ctypes.c_int
        lib.gdn_nt_max.argtypes = [i32, i32, i32]
        lib.gdn_nt_max.restype = i32
        lib.gdn_workspace_size.argtypes = [P(GdnDesc)]
        lib.gdn_workspace_size.restype = ctypes.c_size_t
        lib.gdn_build_chunk_indices.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
        lib.gdn_build_chunk_indices.restype = ctypes.c_int
        lib.gdn_chunk_fwd.argtypes = [P(GdnDesc), vp, vp, vp, vp, vp, ctypes.c_float, vp, vp,
                                      vp, vp, vp, vp]
        lib.gdn_chunk_fwd.restype = ctypes.c_int
        lib.gdn_chunk_fwd_noalloc.argtypes = lib.gdn_chunk_fwd.argtypes
        lib.gdn_chunk_fwd_noalloc.restype = ctypes.c_int
        lib.gdn_noalloc_read_status.argtypes = [vp, vp]
        lib.gdn_noalloc_read_status.restype = ctypes.c_int
        lib.gdn_debug_build.argtypes = []
        lib.gdn_debug_build.restype = ctypes.c_int
        lib.gdn_test_debug_poison.argtypes = [i32]
        lib.gdn_test_debug_poison.restype = None
        lib.gdn_test_scan_timeout.argtypes = [ctypes.c_uint32]
        lib.gdn_test_scan_timeout.restype = None
        lib.gdn_workspace_regions.argtypes = [P(GdnDesc), vp, vp, ctypes.c_int]
        lib.gdn_workspace_regions.restype = ctypes.c_int
        lib.gdn_recurrent_fwd.argtypes = [P(GdnDesc), vp, vp, vp, vp, vp, ctypes.c_float, vp,
                                          vp, vp, vp, vp]
        lib.gdn_recurrent_fwd.restype = ctypes.c_int
        lib.gdn_conv_front.argtypes = [P(GdnDesc), vp, vp, i32, vp, vp, vp, vp, vp, vp, vp,
                                       i32, vp]
        lib.gdn_conv_front.restype = ctypes.c_int
        lib.gdn_bwd_workspace_size.argtypes = [P(GdnDesc)]
        lib.gdn_bwd_workspace_size.restype = ctypes.c_size_t
        lib.gdn_chunk_bwd.argtypes = [P(GdnDesc), vp, vp, vp, vp, vp, ctypes.c_float, vp, vp,
                                      vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.gdn_chunk_bwd.restype = ctypes.c_int
        lib.gdn_read_status.argtypes = [P(GdnDesc), vp, vp]
        lib.gdn_read_status.restype = ctypes.c_int
        lib.gdn_status_string.argtypes = [ctypes.c_int]
        lib.gdn_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load_library().gdn_status_string(int(status)).decode()
    except Exception:
        return "unknown"


gdn_status_string = status_string


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return GDN_F32
    if dt == torch.bfloat16:
        return GDN_BF16
    raise TypeError(f"unsupported dtype {dt}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def make_desc(T: int, N: int, H: int, Hv: int, qkv_dtype: torch.dtype,
              out_dtype: Optional[torch.dtype] = None, nt_max: int = 0, flags: int = 0,
              l2norm_eps: float = 0.0, dk: int = 128, dv: int = 128) -> GdnDesc:
    return GdnDesc(T=T, N=N, H=H, Hv=Hv, dk=dk, dv=dv, chunk_size=64, nt_max=nt_max,
                   qkv_dtype=_dtype_code(qkv_dtype),
                   out_dtype=_dtype_code(out_dtype or qkv_dtype), flags=flags,
                   l2norm_eps=l2norm_eps, workspace=None, workspace_bytes=0, stage_events=None)


def gdn_check_desc(desc: GdnDesc) -> int:
    return load_library().gdn_check_desc(ctypes.byref(desc))


def gdn_nt_max(T: int, N: int, chunk_size: int = 64) -> int:
    return load_library().gdn_nt_max(T, N, chunk_size)


def gdn_workspace_size(desc: GdnDesc) -> int:
    return int(load_library().gdn_workspace_size(ctypes.byref(desc)))


def alloc_workspace(desc: GdnDesc, device) -> torch.Tensor:
    n = gdn_workspace_size(desc)
    if n == 0:
        raise GdnError(load_library().gdn_check_desc(ctypes.byref(desc)), "workspace size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def gdn_build_chunk_indices(cu_seqlens: Optional[torch.Tensor], T: int, nt_max: int,
                            N: Optional[int] = None, status: Optional[torch.Tensor] = None,
                            stream=None):
    """Build the [nt_max, 2] chunk table and [N+1] chunk offsets on the device."""
    dev = cu_seqlens.device if cu_seqlens is not None else torch.device("cuda")
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else (N or 1)
    table = torch.empty(nt_max, 2, dtype=torch.int32, device=dev)
    offsets = torch.empty(N + 1, dtype=torch.int32, device=dev)
    rc = load_library().gdn_build_chunk_indices(_ptr(cu_seqlens), N, T, nt_max, _ptr(table),
                                                _ptr(offsets), _ptr(status),
                                                _stream_handle(stream))
    if rc != 0:
        raise GdnError(rc, "gdn_build_chunk_indices")
    return table, offsets


def gdn_chunk_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                  beta: torch.Tensor, scale: Optional[float] = None,
                  initial_state: Optional[torch.Tensor] = None,
                  cu_seqlens: Optional[torch.Tensor] = None,
                  chunk_indices: Optional[torch.Tensor] = None,
                  output_final_state: bool = True, out_dtype: Optional[torch.dtype] = None,
                  use_qk_l2norm: bool = False, l2norm_eps: float = 0.0,
                  build_chunk_indices: bool = False, nt_max: int = 0,
                  out: Optional[torch.Tensor] = None, final_state: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None, stream=None,
                  stage_events=None, return_desc: bool = False, extra_flags: int = 0):
    """Chunked gated-delta-rule forward through the C ABI.

    q, k [T, H, d]; v [T, Hv, d] with d = 128 or 64 (fp32 or bf16, CUDA,
    contiguous); beta fp32 [T, Hv]; g fp32 [T, Hv] (one gate per token) or
    [T, Hv, d] (one gate per key channel); initial_state fp32 [N, Hv, d, d] or
    None; cu_seqlens int32 [N + 1] or None. Returns (out [T, Hv, d], final_state
    or None).
    """
    T, H, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    flags = (GDN_FLAG_QK_L2NORM if use_qk_l2norm else 0) | (
        GDN_FLAG_BUILD_CHUNK_INDICES if build_chunk_indices else 0) | (
        GDN_FLAG_CHANNEL_GATES if g.dim() == 3 else 0) | extra_flags
    out_dtype = out_dtype or (out.dtype if out is not None else q.dtype)
    desc = make_desc(T, N, H, Hv, q.dtype, out_dtype, nt_max=nt_max, flags=flags,
                     l2norm_eps=l2norm_eps, dk=dk, dv=dv)
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if out is None:
        out = torch.empty(T, Hv, dv, dtype=out_dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty(N, Hv, dv, dk, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(desc, q.device)
    desc.workspace = workspace.data_ptr()
    desc.workspace_bytes = workspace.numel()
    ev_arr = None
    if stage_events is not None:
        ev_arr = (ctypes.c_void_p * GDN_NUM_STAGE_EVENTS)(*[int(e) for e in stage_events])
        desc.stage_events = ctypes.cast(ev_arr, ctypes.c_void_p)
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    rc = load_library().gdn_chunk_fwd(
        ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
        _ptr(initial_state), _ptr(cu_seqlens), _ptr(chunk_indices), _ptr(out),
        _ptr(final_state), _stream_handle(stream))
    if rc != 0:
        raise GdnError(rc, "gdn_chunk_fwd")
    if return_desc:
        return out, final_state, desc, workspace
    return out, final_state


def gdn_recurrent_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                      beta: torch.Tensor, scale: Optional[float] = None,
                      initial_state: Optional[torch.Tensor] = None,
                      cu_seqlens: Optional[torch.Tensor] = None,
                      output_final_state: bool = True, out_dtype: Optional[torch.dtype] = None,
                      use_qk_l2norm: bool = False, l2norm_eps: float = 0.0,
                      out: Optional[torch.Tensor] = None,
                      final_state: Optional[torch.Tensor] = None,
                      status: Optional[torch.Tensor] = None, stream=None,
                      return_desc: bool = False):
    """Token-serial forward (decode / speculative verify) through the C ABI.

    Same tensors as gdn_chunk_fwd. `status`, if given, is a 256-byte-aligned
    device buffer of at least 4 bytes that receives the device status word
    (read it with gdn_read_status on the returned descriptor).
    Returns (out, final_state) or (out, final_state, desc).
    """
    T, H, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    out_dtype = out_dtype or (out.dtype if out is not None else q.dtype)
    desc = make_desc(T, N, H, Hv, q.dtype, out_dtype,
                     flags=GDN_FLAG_QK_L2NORM if use_qk_l2norm else 0,
                     l2norm_eps=l2norm_eps, dk=dk, dv=dv)
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if out is None:
        out = torch.empty(T, Hv, dv, dtype=out_dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty(N, Hv, dv, dk, dtype=torch.float32, device=q.device)
    if status is not None:
        desc.workspace = status.data_ptr()
        desc.workspace_bytes = status.numel() * status.element_size()
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    rc = load_library().gdn_recurrent_fwd(
        ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
        _ptr(initial_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
        _stream_handle(stream))
    if rc != 0:
        raise GdnError(rc, "gdn_recurrent_fwd")
    if return_desc:
        return out, final_state, desc
    return out, final_state


def gdn_conv_front(x: torch.Tensor, conv_w: torch.Tensor, H: int, Hv: int,
                   conv_state: Optional[torch.Tensor] = None,
                   cu_seqlens: Optional[torch.Tensor] = None, use_qk_l2norm: bool = False,
                   l2norm_eps: float = 0.0, output_state: bool = True,
                   conv_state_out: Optional[torch.Tensor] = None, n_snapshots: int = 0,
                   status: Optional[torch.Tensor] = None, stream=None,
                   return_desc: bool = False, q: Optional[torch.Tensor] = None,
                   k: Optional[torch.Tensor] = None, v: Optional[torch.Tensor] = None):
    """Front end through the C ABI: x [T, C] (C = 2*H*128 + Hv*128, bf16 or fp32),
    conv_w fp32 [C, d_conv], conv_state fp32 [N, C, d_conv - 1] or None.
    Returns (q, k, v, conv_state_out or None, snapshots or None[, desc])."""
    T, C = x.shape
    d_conv = conv_w.shape[1]
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    desc = make_desc(T, N, H, Hv, x.dtype, x.dtype,
                     flags=GDN_FLAG_QK_L2NORM if use_qk_l2norm else 0, l2norm_eps=l2norm_eps)
    for name, t in (("x", x), ("conv_w", conv_w)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    q = torch.empty(T, H, 128, dtype=x.dtype, device=x.device) if q is None else q
    k = torch.empty(T, H, 128, dtype=x.dtype, device=x.device) if k is None else k
    v = torch.empty(T, Hv, 128, dtype=x.dtype, device=x.device) if v is None else v
    if conv_state_out is None and output_state:
        conv_state_out = torch.empty(N, C, d_conv - 1, dtype=torch.float32, device=x.device)
    snaps = (torch.empty(N, n_snapshots, C, d_conv - 1, dtype=torch.float32, device=x.device)
             if n_snapshots > 0 else None)
    if status is not None:
        desc.workspace = status.data_ptr()
        desc.workspace_bytes = status.numel() * status.element_size()
    rc = load_library().gdn_conv_front(
        ctypes.byref(desc), _ptr(x), _ptr(conv_w), int(d_conv), _ptr(conv_state),
        _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v), _ptr(conv_state_out), _ptr(snaps),
        int(n_snapshots), _stream_handle(stream))
    if rc != 0:
        raise GdnError(rc, "gdn_conv_front")
    if return_desc:
        return q, k, v, conv_state_out, snaps, desc
    return q, k, v, conv_state_out, snaps


def gdn_chunk_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                  beta: torch.Tensor, d_out: torch.Tensor, scale: Optional[float] = None,
                  initial_state: Optional[torch.Tensor] = None,
                  cu_seqlens: Optional[torch.Tensor] = None,
                  d_final_state: Optional[torch.Tensor] = None,
                  chunk_indices: Optional[torch.Tensor] = None, nt_max: int = 0,
                  workspace: Optional[torch.Tensor] = None, stream=None,
                  return_desc: bool = False, grads: Optional[dict] = None,
                  stage_events=None):
    """Backward of gdn_chunk_fwd through the C ABI (scalar gates, no L2 norm).

    Same inputs as the forward call plus d_out [T, Hv, d] (fp32 or bf16) and
    d_final_state fp32 [N, Hv, d, d] or None. Returns a dict of fp32 gradients
    dq, dk [T, H, d], dv [T, Hv, d], dg, dbeta [T, Hv] and d_initial_state
    [N, Hv, d, d]."""
    T, H, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    desc = make_desc(T, N, H, Hv, q.dtype, d_out.dtype, nt_max=nt_max, dk=dk, dv=dv,
                     flags=GDN_FLAG_CHANNEL_GATES if g.dim() == 3 else 0)
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("d_out", d_out)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    dev = q.device
    f32 = torch.float32
    grads = grads if grads is not None else dict(dq=torch.zeros(T, H, dk, dtype=f32, device=dev),
                 dk=torch.zeros(T, H, dk, dtype=f32, device=dev),
                 dv=torch.zeros(T, Hv, dv, dtype=f32, device=dev),
                 dg=torch.zeros(T, Hv, dtype=f32, device=dev),
                 dbeta=torch.zeros(T, Hv, dtype=f32, device=dev),
                 d_initial_state=torch.empty(N, Hv, dv, dk, dtype=f32, device=dev))
    if workspace is None:
        n = int(load_library().gdn_bwd_workspace_size(ctypes.byref(desc)))
        if n == 0:
            raise GdnError(load_library().gdn_check_desc(ctypes.byref(desc)), "bwd workspace")
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    desc.workspace = workspace.data_ptr()
    desc.workspace_bytes = workspace.numel()
    ev_arr = None
    if stage_events is not None:
        ev_arr = (ctypes.c_void_p * GDN_NUM_STAGE_EVENTS)(*[int(e) for e in stage_events])
        desc.stage_events = ctypes.cast(ev_arr, ctypes.c_void_p)
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    rc = load_library().gdn_chunk_bwd(
        ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
        _ptr(initial_state), _ptr(cu_seqlens), _ptr(chunk_indices), _ptr(d_out),
        _ptr(d_final_state), _ptr(grads["dq"]), _ptr(grads["dk"]), _ptr(grads["dv"]),
        _ptr(grads["dg"]), _ptr(grads["dbeta"]), _ptr(grads["d_initial_state"]),
        _stream_handle(stream))
    if rc != 0:
        raise GdnError(rc, "gdn_chunk_bwd")
    if return_desc:
        return grads, desc, workspace
    return grads


def gdn_read_status(desc: GdnDesc, stream=None) -> int:
    """Copy the device status word of the last call on desc.workspace (synchronizes)."""
    host = torch.zeros(1, dtype=torch.int32).pin_memory()
    rc = load_library().gdn_read_status(ctypes.byref(desc), _ptr(host), _stream_handle(stream))
    if rc != 0:
        raise GdnError(rc, "gdn_read_status")
    (torch.cuda.current_stream() if stream is None else stream).synchronize()
    return int(host.item())


def gdn_chunk_fwd_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                          beta: torch.Tensor, scale: Optional[float] = None,
                          initial_state: Optional[torch.Tensor] = None,
                          cu_seqlens: Optional[torch.Tensor] = None,
                          out: Optional[torch.Tensor] = None,
                          final_state: Optional[torch.Tensor] = None,
                          out_dtype: Optional[torch.dtype] = None, stream=None):
    """The forward pass through gdn_chunk_fwd_noalloc: the library's own static
    scratch replaces the workspace (for callers that cannot allocate device
    memory; here torch only provides the caller's inputs and outputs)."""
    T, H, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    out_dtype = out_dtype or (out.dtype if out is not None else q.dtype)
    desc = make_desc(T, N, H, Hv, q.dtype, out_dtype, dk=dk, dv=dv,
                     flags=GDN_FLAG_CHANNEL_GATES if g.dim() == 3 else 0)
    if out is None:
        out = torch.empty(T, Hv, dv, dtype=out_dtype, device=q.device)
    if final_state is None:
        final_state = torch.empty(N, Hv, dv, dk, dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    rc = load_library().gdn_chunk_fwd_noalloc(
        ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
        _ptr(initial_state), _ptr(cu_seqlens), None, _ptr(out), _ptr(final_state),
        _stream_handle(stream))
    if rc != 0:
        raise GdnError(rc, "gdn_chunk_fwd_noalloc")
    return out, final_state


def gdn_noalloc_read_status(stream=None) -> int:
    """Device status word of the last gdn_chunk_fwd_noalloc call on the current device
    (it lives in the library's static scratch; synchronizes the stream)."""
    host = torch.zeros(1, dtype=torch.int32).pin_memory()
    rc = load_library().gdn_noalloc_read_status(_ptr(host), _stream_handle(stream))
    if rc != 0:
        raise GdnError(rc, "gdn_noalloc_read_status")
    (torch.cuda.current_stream() if stream is None else stream).synchronize()
    return int(host.item())


def gdn_test_scan_timeout(polls: int) -> None:
    """Testing hook: with polls > 0 the bf16 scan waits that many polls on an event that
    never happens and takes its timeout path (GDN_DEV_TIMEOUT); 0 turns it off."""
    load_library().gdn_test_scan_timeout(int(polls))


def gdn_debug_build() -> bool:
    """Whether the loaded library is the GDN_DEBUG build (device-side index checks)."""
    return bool(load_library().gdn_debug_build())


def gdn_test_debug_poison(on: bool) -> None:
    """Testing hook of the GDN_DEBUG build: aim one intra CTA's M copies one slot past the
    end of their region, which the device check must catch (GDN_DEV_DEBUG_INDEX)."""
    load_library().gdn_test_debug_poison(1 if on else 0)


def gdn_workspace_regions(desc: GdnDesc):
    """[(begin, end)] byte ranges of the workspace regions for this descriptor."""
    b = (ctypes.c_size_t * 16)()
    e = (ctypes.c_size_t * 16)()
    n = load_library().gdn_workspace_regions(ctypes.byref(desc), b, e, 16)
    if n < 0:
        raise GdnError(n, "gdn_workspace_regions")
    return [(int(b[i]), int(e[i])) for i in range(n)]
