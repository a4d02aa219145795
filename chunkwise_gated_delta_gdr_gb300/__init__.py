"""Python binding of the GB300 chunkwise gated delta rule forward library.

A thin ctypes layer over ``include/gdr.h``: it marshals torch tensors'
device pointers, sizes and the current CUDA stream into the C ABI and turns
status codes into exceptions. Every step of the computation runs in the CUDA
kernels of ``libgdr.so``; there is no fallback, and every call raises if the
library has not been built (``python -c "import __graft_entry__ as g; g.build()"``).

Main entry points (same names as the C ABI):
  chunk_fwd(q, k, v, g, beta, initial_state=None, ...) -> (o, final_state)
  chunk_fwd_host(...)      the same on host (pinned) tensors, copies inside
  chunk_fwd_workspace_size(...), chunk_fwd_path(...), stream_status(...)
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libgdr.so")

GDR_OK, GDR_ERR_INVALID_ARG, GDR_ERR_UNSUPPORTED, GDR_ERR_ALIGNMENT = 0, 1, 2, 3
GDR_ERR_WORKSPACE, GDR_ERR_CUDA, GDR_ERR_TIMEOUT = 4, 5, 6
GDR_F32, GDR_BF16 = 0, 1
GDR_GATE_SCALAR, GDR_GATE_PER_KEY, GDR_GATE_NONE = 0, 1, 2

EXPORTED = (
    "gdr_chunk_fwd", "gdr_chunk_prepare", "gdr_chunk_recur", "gdr_chunk_fwd_workspace_size",
    "gdr_chunk_fwd_host",
    "gdr_chunk_fwd_host_buffer_size", "gdr_stream_status", "gdr_status_string",
    "gdr_chunk_fwd_path", "gdr_version", "gdr_chunk_fwd_noalloc", "gdr_recurrent_fwd",
    "gdr_ssd_chunk_fwd", "gdr_ssd_chunk_fwd_workspace_size", "gdr_chunk_fwd_segmented",
    "gdr_chunk_fwd_segmented_workspace_size", "gdr_noalloc_stream_status",
    "gdr_set_flag_wait_limit",
)
# Size of the library-owned scratch used by gdr_chunk_fwd_noalloc (per device).
GDR_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


class GdrError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class gdr_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("HV", ctypes.c_int), ("K", ctypes.c_int), ("V", ctypes.c_int),
                ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def load_library(path: Optional[str] = None):
    """Load libgdr.so (raises if it is missing: there is no fallback path)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libgdr.so not built ({p}); run chunkwise_gated_delta_gdr_gb300.build")
        lib = ctypes.CDLL(p)
        vp, ip, fp, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        dp = ctypes.POINTER(gdr_dims)
        fwd_args = [vp, vp, vp, vp, vp, vp, ip, fp, ip, ip, vp, vp, dp, vp, sz, vp]
        lib.gdr_chunk_fwd.argtypes = fwd_args
        lib.gdr_chunk_fwd.restype = ip
        lib.gdr_chunk_fwd_host.argtypes = fwd_args
        lib.gdr_chunk_fwd_host.restype = ip
        lib.gdr_chunk_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, ip, fp, ip, ip, vp, vp, dp, vp]
        lib.gdr_chunk_fwd_noalloc.restype = ip
        lib.gdr_chunk_prepare.argtypes = [vp, vp, vp, vp, vp, ip, fp, ip, ip, dp, vp, sz, vp]
        lib.gdr_chunk_prepare.restype = ip
        lib.gdr_chunk_recur.argtypes = [vp, vp, vp, ip, fp, ip, ip, vp, vp, dp, vp, sz, vp]
        lib.gdr_chunk_recur.restype = ip
        lib.gdr_chunk_fwd_workspace_size.argtypes = [dp, ip, ip]
        lib.gdr_chunk_fwd_workspace_size.restype = sz
        lib.gdr_chunk_fwd_host_buffer_size.argtypes = [dp, ip, ip, ip, ip]
        lib.gdr_chunk_fwd_host_buffer_size.restype = sz
        lib.gdr_stream_status.argtypes = [vp, vp]
        lib.gdr_stream_status.restype = ip
        lib.gdr_status_string.argtypes = [ip]
        lib.gdr_status_string.restype = ctypes.c_char_p
        lib.gdr_chunk_fwd_path.argtypes = [dp, ip, ip, ctypes.POINTER(ctypes.c_int)]
        lib.gdr_chunk_fwd_path.restype = ip
        lib.gdr_recurrent_fwd.argtypes = [vp, vp, vp, vp, vp, vp, fp, ip, ip, vp, dp, vp]
        lib.gdr_recurrent_fwd.restype = ip
        lib.gdr_ssd_chunk_fwd.argtypes = [vp, vp, vp, vp, vp, ip, fp, ip, ip, vp, vp, dp, vp, sz, vp]
        lib.gdr_ssd_chunk_fwd.restype = ip
        lib.gdr_ssd_chunk_fwd_workspace_size.argtypes = [dp, ip, ip]
        lib.gdr_ssd_chunk_fwd_workspace_size.restype = sz
        lib.gdr_chunk_fwd_segmented.argtypes = [vp, vp, vp, vp, vp, vp, ip, fp, ip, ip, ip, vp,
                                                 vp, dp, vp, sz, vp]
        lib.gdr_chunk_fwd_segmented.restype = ip
        lib.gdr_chunk_fwd_segmented_workspace_size.argtypes = [dp, ip, ip, ip]
        lib.gdr_chunk_fwd_segmented_workspace_size.restype = sz
        lib.gdr_version.argtypes = []
        lib.gdr_version.restype = ip
        lib.gdr_noalloc_stream_status.argtypes = [vp]
        lib.gdr_noalloc_stream_status.restype = ip
        lib.gdr_set_flag_wait_limit.argtypes = [ctypes.c_int64]
        lib.gdr_set_flag_wait_limit.restype = ctypes.c_int64
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().gdr_status_string(int(status)).decode()


def _dtype_code(dt) -> int:
    import torch
    if dt == torch.bfloat16:
        return GDR_BF16
    if dt == torch.float32:
        return GDR_F32
    raise TypeError(f"unsupported dtype {dt}")


def make_dims(B, T, H, HV, K, V, in_dtype, out_dtype) -> gdr_dims:
    return gdr_dims(int(B), int(T), int(H), int(HV), int(K), int(V), int(in_dtype),
                    int(out_dtype))


def chunk_fwd_workspace_size(dims: gdr_dims, chunk_size: int, gate_mode: int) -> int:
    return int(load_library().gdr_chunk_fwd_workspace_size(ctypes.byref(dims), chunk_size,
                                                            gate_mode))


def chunk_fwd_path(dims: gdr_dims, chunk_size: int, gate_mode: int) -> int:
    st = ctypes.c_int(0)
    r = load_library().gdr_chunk_fwd_path(ctypes.byref(dims), chunk_size, gate_mode,
                                          ctypes.byref(st))
    if r < 0:
        raise GdrError(st.value, "gdr_chunk_fwd_path")
    return int(r)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _shapes(q, v, g):
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    if g is None:
        gate_mode = GDR_GATE_NONE               # ungated delta rule
    else:
        gate_mode = GDR_GATE_PER_KEY if g.dim() == 4 else GDR_GATE_SCALAR
    return B, T, H, HV, K, V, gate_mode


def chunk_fwd(q, k, v, g, beta, initial_state=None, *, chunk_size: int = 64,
              scale: Optional[float] = None, use_qk_l2norm: bool = True,
              output_final_state: bool = True, out_dtype=None, out=None, final_state=None,
              workspace=None, stream=None):
    """Chunkwise gated delta rule forward on CUDA tensors.

    q, k [B,T,H,K], v [B,T,HV,V] (bf16 or fp32); g fp32 [B,T,HV] (scalar gate),
    [B,T,HV,K] (per-key gate) or None (ungated); beta fp32 [B,T,HV]; initial_state fp32 [B,HV,K,V]
    or None. scale defaults to 1/sqrt(K), out_dtype to q's dtype. Returns
    (o [B,T,HV,V], final_state [B,HV,K,V] fp32 or None). Buffers not passed in
    are allocated with torch on q's device; the call is asynchronous on
    ``stream`` (default: torch's current stream).
    """
    import torch
    B, T, H, HV, K, V, gate_mode = _shapes(q, v, g)
    out_dtype = q.dtype if out_dtype is None else out_dtype
    scale = 1.0 / math.sqrt(K) if scale is None else float(scale)
    dims = make_dims(B, T, H, HV, K, V, _dtype_code(q.dtype), _dtype_code(out_dtype))
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta),
                    ("initial_state", initial_state)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if out is None:
        out = torch.empty(B, T, HV, V, dtype=out_dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty(B, HV, K, V, dtype=torch.float32, device=q.device)
    ws_bytes = chunk_fwd_workspace_size(dims, chunk_size, gate_mode)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    st = load_library().gdr_chunk_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state), int(chunk_size),
        ctypes.c_float(scale), int(bool(use_qk_l2norm)), gate_mode, _ptr(out), _ptr(final_state),
        ctypes.byref(dims), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
        _stream_handle(stream))
    if st != GDR_OK:
        raise GdrError(st, "gdr_chunk_fwd")
    return out, final_state


def chunk_fwd_segmented_workspace_size(dims: gdr_dims, chunk_size: int, gate_mode: int,
                                       segments: int) -> int:
    return int(load_library().gdr_chunk_fwd_segmented_workspace_size(
        ctypes.byref(dims), chunk_size, gate_mode, segments))


def chunk_fwd_segmented(q, k, v, g, beta, initial_state=None, *, segments: int,
                        chunk_size: int = 64, scale: Optional[float] = None,
                        use_qk_l2norm: bool = True, output_final_state: bool = True,
                        out_dtype=None, out=None, final_state=None, workspace=None, stream=None):
    """chunk_fwd with each sequence split into ``segments`` parts whose
    recurrences run at the same time (gdr_chunk_fwd_segmented). Same arguments
    and results as chunk_fwd."""
    import torch
    B, T, H, HV, K, V, gate_mode = _shapes(q, v, g)
    out_dtype = q.dtype if out_dtype is None else out_dtype
    scale = 1.0 / math.sqrt(K) if scale is None else float(scale)
    dims = make_dims(B, T, H, HV, K, V, _dtype_code(q.dtype), _dtype_code(out_dtype))
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta),
                    ("initial_state", initial_state)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if out is None:
        out = torch.empty(B, T, HV, V, dtype=out_dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty(B, HV, K, V, dtype=torch.float32, device=q.device)
    ws_bytes = chunk_fwd_segmented_workspace_size(dims, chunk_size, gate_mode, segments)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    st = load_library().gdr_chunk_fwd_segmented(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state), int(chunk_size),
        ctypes.c_float(scale), int(bool(use_qk_l2norm)), gate_mode, int(segments), _ptr(out),
        _ptr(final_state), ctypes.byref(dims), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
        _stream_handle(stream))
    if st != GDR_OK:
        raise GdrError(st, "gdr_chunk_fwd_segmented")
    return out, final_state


def chunk_prepare(q, k, v, g, beta, *, workspace, chunk_size: int = 64,
                  scale: Optional[float] = None, use_qk_l2norm: bool = True, out_dtype=None,
                  stream=None):
    """First stage of chunk_fwd: the chunk-local kernel fills ``workspace``."""
    B, T, H, HV, K, V, gate_mode = _shapes(q, v, g)
    out_dtype = q.dtype if out_dtype is None else out_dtype
    scale = 1.0 / math.sqrt(K) if scale is None else float(scale)
    dims = make_dims(B, T, H, HV, K, V, _dtype_code(q.dtype), _dtype_code(out_dtype))
    st = load_library().gdr_chunk_prepare(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), int(chunk_size), ctypes.c_float(scale),
        int(bool(use_qk_l2norm)), gate_mode, ctypes.byref(dims), _ptr(workspace),
        ctypes.c_size_t(workspace.numel()), _stream_handle(stream))
    if st != GDR_OK:
        raise GdrError(st, "gdr_chunk_prepare")


def chunk_recur(q, k, initial_state=None, *, workspace, out, final_state=None, HV: int, V: int,
                gate_mode: int, chunk_size: int = 64, scale: Optional[float] = None,
                use_qk_l2norm: bool = True, stream=None):
    """Second stage of chunk_fwd: the state recurrence over a prepared workspace."""
    B, T, H, K = q.shape
    scale = 1.0 / math.sqrt(K) if scale is None else float(scale)
    dims = make_dims(B, T, H, HV, K, V, _dtype_code(q.dtype), _dtype_code(out.dtype))
    st = load_library().gdr_chunk_recur(
        _ptr(q), _ptr(k), _ptr(initial_state), int(chunk_size), ctypes.c_float(scale),
        int(bool(use_qk_l2norm)), int(gate_mode), _ptr(out), _ptr(final_state), ctypes.byref(dims),
        _ptr(workspace), ctypes.c_size_t(workspace.numel()), _stream_handle(stream))
    if st != GDR_OK:
        raise GdrError(st, "gdr_chunk_recur")
    return out, final_state


def chunk_fwd_noalloc(q, k, v, g, beta, initial_state=None, *, out, final_state=None,
                      chunk_size: int = 64, scale: Optional[float] = None,
                      use_qk_l2norm: bool = True, stream=None):
    """chunk_fwd on the library's own fixed scratch (no workspace is passed or
    allocated). For callers that cannot provide device memory; limited to
    problems whose workspace fits GDR_NOALLOC_SCRATCH_BYTES. Calls on one device
    share that scratch, so they must not overlap on the GPU."""
    B, T, H, HV, K, V, gate_mode = _shapes(q, v, g)
    scale = 1.0 / math.sqrt(K) if scale is None else float(scale)
    dims = make_dims(B, T, H, HV, K, V, _dtype_code(q.dtype), _dtype_code(out.dtype))
    st = load_library().gdr_chunk_fwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state), int(chunk_size),
        ctypes.c_float(scale), int(bool(use_qk_l2norm)), gate_mode, _ptr(out), _ptr(final_state),
        ctypes.byref(dims), _stream_handle(stream))
    if st != GDR_OK:
        raise GdrError(st, "gdr_chunk_fwd_noalloc")
    return out, final_state


def ssd_chunk_fwd(q, k, v, g, initial_state=None, *, chunk_size: int = 64,
                  scale: Optional[float] = None, use_qk_l2norm: bool = True, out_dtype=None,
                  output_final_state: bool = True, stream=None):
    """Chunkwise Mamba2 SSD forward (S <- diag(exp g) S + k v^T, o = S^T scale q):
    the gated recurrence without the delta erase and without beta. Shapes as
    for chunk_fwd. Returns (o, final_state)."""
    import torch
    B, T, H, HV, K, V, gate_mode = _shapes(q, v, g)
    out_dtype = q.dtype if out_dtype is None else out_dtype
    scale = 1.0 / math.sqrt(K) if scale is None else float(scale)
    dims = make_dims(B, T, H, HV, K, V, _dtype_code(q.dtype), _dtype_code(out_dtype))
    out = torch.empty(B, T, HV, V, dtype=out_dtype, device=q.device)
    final_state = (torch.empty(B, HV, K, V, dtype=torch.float32, device=q.device)
                   if output_final_state else None)
    lib = load_library()
    ws_bytes = lib.gdr_ssd_chunk_fwd_workspace_size(ctypes.byref(dims), int(chunk_size), gate_mode)
    if ws_bytes == 0 and B * T > 0:
        raise GdrError(GDR_ERR_UNSUPPORTED, "gdr_ssd_chunk_fwd_workspace_size")
    workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    st = lib.gdr_ssd_chunk_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(initial_state), int(chunk_size),
        ctypes.c_float(scale), int(bool(use_qk_l2norm)), gate_mode, _ptr(out), _ptr(final_state),
        ctypes.byref(dims), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
        _stream_handle(stream))
    if st != GDR_OK:
        raise GdrError(st, "gdr_ssd_chunk_fwd")
    return out, final_state


def recurrent_fwd(q, k, v, g, beta, state, *, scale: Optional[float] = None,
                  use_qk_l2norm: bool = True, out=None, out_dtype=None, stream=None):
    """Token-by-token recurrence (decode step for T = 1) on CUDA tensors.

    Shapes as for chunk_fwd; ``state`` fp32 [B,HV,K,V] is updated in place
    (the state before the first token on entry, after the last token on
    return). Returns o [B,T,HV,V]."""
    import torch
    B, T, H, HV, K, V, gate_mode = _shapes(q, v, g)
    out_dtype = q.dtype if out_dtype is None else out_dtype
    scale = 1.0 / math.sqrt(K) if scale is None else float(scale)
    dims = make_dims(B, T, H, HV, K, V, _dtype_code(q.dtype), _dtype_code(out_dtype))
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("state", state)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if out is None:
        out = torch.empty(B, T, HV, V, dtype=out_dtype, device=q.device)
    st = load_library().gdr_recurrent_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), ctypes.c_float(scale),
        int(bool(use_qk_l2norm)), gate_mode, _ptr(out), ctypes.byref(dims), _stream_handle(stream))
    if st != GDR_OK:
        raise GdrError(st, "gdr_recurrent_fwd")
    return out


def chunk_fwd_host_buffer_size(dims: gdr_dims, chunk_size: int, gate_mode: int,
                               with_initial_state: bool, with_final_state: bool) -> int:
    return int(load_library().gdr_chunk_fwd_host_buffer_size(
        ctypes.byref(dims), chunk_size, gate_mode, int(with_initial_state),
        int(with_final_state)))


def chunk_fwd_host(q, k, v, g, beta, initial_state=None, *, out, final_state=None,
                   device_buffer, chunk_size: int = 64, scale: Optional[float] = None,
                   use_qk_l2norm: bool = True, stream=None):
    """Forward pass on HOST tensors (pinned for asynchronous copies).

    The C library copies the inputs into ``device_buffer`` (a CUDA uint8 tensor
    of chunk_fwd_host_buffer_size bytes), runs the forward pass and copies o
    and the final state back into ``out`` / ``final_state`` (host tensors), all
    on ``stream``. Synchronise the stream before reading the outputs.
    """
    B, T, H, HV, K, V, gate_mode = _shapes(q, v, g)
    scale = 1.0 / math.sqrt(K) if scale is None else float(scale)
    dims = make_dims(B, T, H, HV, K, V, _dtype_code(q.dtype), _dtype_code(out.dtype))
    st = load_library().gdr_chunk_fwd_host(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state), int(chunk_size),
        ctypes.c_float(scale), int(bool(use_qk_l2norm)), gate_mode, _ptr(out), _ptr(final_state),
        ctypes.byref(dims), _ptr(device_buffer), ctypes.c_size_t(device_buffer.numel()),
        _stream_handle(stream))
    if st != GDR_OK:
        raise GdrError(st, "gdr_chunk_fwd_host")
    return out, final_state


def set_flag_wait_limit(polls: int) -> int:
    """gdr_set_flag_wait_limit: bound (polls, about 64 ns apart) of the
    one-launch forward's waits on chunk flags for later calls; polls < 0 leaves
    it unchanged. Returns the previous bound."""
    return int(load_library().gdr_set_flag_wait_limit(int(polls)))


def noalloc_stream_status(stream=None) -> int:
    """gdr_noalloc_stream_status: synchronise the stream and report the last
    gdr_chunk_fwd_noalloc call's device-side status on the current device."""
    return int(load_library().gdr_noalloc_stream_status(_stream_handle(stream)))


def stream_status(stream=None, workspace=None) -> int:
    """Synchronise the stream and return its gdr_status (see gdr.h)."""
    return int(load_library().gdr_stream_status(_stream_handle(stream), _ptr(workspace)))
