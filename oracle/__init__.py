"""float64 CPU oracle for the gated delta rule forward pass (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package. The CUDA library never imports, links or
calls it, and it shares no code with the CUDA sources. The arithmetic lives in
``gdr_oracle.c`` (float64, plain loops); this module only builds that file with
gcc, marshals arrays through ctypes and reshapes the per-sequence outputs.

Functions (all return float64 numpy arrays):
  recurrent(...)          the token recurrence, the method's definition
  chunkwise(...)          chunk form, beta on the columns of A_kk (lecture notes)
  chunkwise_rowbeta(...)  chunk form, beta on the rows (blog §2.3 / optimisation script)
  bruteforce(...)         explicit products of the one-step maps (tiny T, K)
  unit_lower_inverse(L, method)  (I + L)^{-1}: 0 solve, 1 Neumann, 2 row recursion

Inputs are torch CPU tensors or numpy arrays laid out as
q, k [B,T,H,K]; v [B,T,HV,V]; g [B,T,HV] (gate_mode 0) or [B,T,HV,K] (gate_mode 1);
beta [B,T,HV]; s0 [B,HV,K,V] or None. q, k, v may be float64, float32 or bfloat16;
g, beta, s0 float64 or float32 (they are read exactly, never rounded).
``sel`` optionally lists flat sequence indices b*HV + hv; the outputs are then
o [nsel, T, V] and S [nsel, K, V]. Without it they are o [B,T,HV,V], S [B,HV,K,V].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdr_oracle.so")
_lock = threading.Lock()
_lib = None

F64, F32, BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile gdr_oracle.c into a shared library with gcc (OpenMP, -O3)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           "-Wno-unused-function", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        vp, ip, dp = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        common = [vp] * 6 + [ip] * 2 + [ip] * 7 + [dp, ip]
        lib.gdr_oracle_recurrent.argtypes = common + [vp, ip, vp, vp, ip, ip]
        lib.gdr_oracle_chunkwise.argtypes = common + [ip, ip, vp, ip, vp, vp, ip]
        lib.gdr_oracle_chunkwise_rowbeta.argtypes = common + [ip, ip, vp, ip, vp, vp, ip]
        lib.gdr_oracle_bruteforce.argtypes = common + [vp, vp]
        lib.gdr_oracle_unit_lower_inverse.argtypes = [vp, ip, ip, vp]
        lib.gdr_oracle_ssd_recurrent.argtypes = [vp] * 5 + [ip] * 2 + [ip] * 7 + [dp, ip] + \
            [vp, ip, vp, vp, ip]
        for f in (lib.gdr_oracle_recurrent, lib.gdr_oracle_chunkwise,
                  lib.gdr_oracle_chunkwise_rowbeta, lib.gdr_oracle_bruteforce,
                  lib.gdr_oracle_unit_lower_inverse, lib.gdr_oracle_ssd_recurrent):
            f.restype = ctypes.c_int
        _lib = lib
        return lib


def _as_array(x, allowed):
    """Return (contiguous numpy array, dtype code) without rounding any value."""
    if x is None:
        return None, F64
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                if BF16 not in allowed:
                    raise TypeError("bfloat16 is not accepted for this input")
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            x = x.numpy()
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float64:
        return x, F64
    if x.dtype == np.float32:
        return x, F32
    raise TypeError(f"unsupported dtype {x.dtype}")


def _prepare(q, k, v, g, beta, s0):
    qa, qd = _as_array(q, (F64, F32, BF16))
    ka, kd = _as_array(k, (F64, F32, BF16))
    va, vd = _as_array(v, (F64, F32, BF16))
    if not (qd == kd == vd):
        raise TypeError("q, k and v must share one element type")
    ga, gd = _as_array(g, (F64, F32))
    ba, bd = _as_array(beta, (F64, F32))
    sa, sd = _as_array(s0, (F64, F32))
    # g, beta and s0 share one element-type code in the C interface.
    gate_dtype = gd
    if ba is not None and bd != gd:
        ba = ba.astype(np.float64) if gd == F64 else ba.astype(np.float32)
    if sa is not None and sd != gd:
        sa = sa.astype(np.float64) if gd == F64 else sa.astype(np.float32)
    B, T, H, K = qa.shape
    HV, V = va.shape[2], va.shape[3]
    gate_mode = 1 if ga.ndim == 4 else 0
    return (qa, ka, va, ga, ba, sa), qd, gate_dtype, (B, T, H, HV, K, V), gate_mode


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _sel_array(sel, B, HV):
    if sel is None:
        return None, B * HV
    s = np.ascontiguousarray(np.asarray(sel, dtype=np.int32))
    if s.size and (s.min() < 0 or s.max() >= B * HV):
        raise ValueError("sequence index out of range")
    return s, int(s.size)


def _reshape_out(o, S, sel, B, T, HV, K, V):
    if sel is not None:
        return o, S
    o = o.reshape(B, HV, T, V).transpose(0, 2, 1, 3).copy()
    S = S.reshape(B, HV, K, V)
    return o, S


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name} rejected its arguments (code {rc})")


def recurrent(q, k, v, g, beta, s0=None, *, scale=None, use_qk_l2norm=True, sel=None,
              nthreads=0, mutation=0):
    """The token recurrence in float64 (the definition the chunk form must equal)."""
    arrs, qd, gd, (B, T, H, HV, K, V), gm = _prepare(q, k, v, g, beta, s0)
    scale = K ** -0.5 if scale is None else float(scale)
    sarr, nseq = _sel_array(sel, B, HV)
    o = np.zeros((nseq, T, V), np.float64)
    S = np.zeros((nseq, K, V), np.float64)
    rc = _load().gdr_oracle_recurrent(*[_ptr(a) for a in arrs], qd, gd, B, T, H, HV, K, V, gm,
                                      scale, int(bool(use_qk_l2norm)), _ptr(sarr), nseq,
                                      _ptr(o), _ptr(S), int(nthreads), int(mutation))
    _check(rc, "gdr_oracle_recurrent")
    return _reshape_out(o, S, sel, B, T, HV, K, V)


def ssd_recurrent(q, k, v, g, s0=None, *, scale=None, use_qk_l2norm=True, sel=None, nthreads=0):
    """The Mamba2 SSD recurrence in float64: S <- diag(exp g_t) S + k_t v_t^T,
    o_t = S^T (scale q_t), with no delta erase and no beta."""
    arrs, qd, gd, (B, T, H, HV, K, V), gm = _prepare(q, k, v, g, None, s0)
    qa, ka, va, ga, _, sa = arrs
    scale = K ** -0.5 if scale is None else float(scale)
    sarr, nseq = _sel_array(sel, B, HV)
    o = np.zeros((nseq, T, V), np.float64)
    S = np.zeros((nseq, K, V), np.float64)
    rc = _load().gdr_oracle_ssd_recurrent(_ptr(qa), _ptr(ka), _ptr(va), _ptr(ga), _ptr(sa), qd, gd,
                                          B, T, H, HV, K, V, gm, scale, int(bool(use_qk_l2norm)),
                                          _ptr(sarr), nseq, _ptr(o), _ptr(S), int(nthreads))
    _check(rc, "gdr_oracle_ssd_recurrent")
    return _reshape_out(o, S, sel, B, T, HV, K, V)


def _chunk_call(fname, q, k, v, g, beta, s0, scale, use_qk_l2norm, chunk_size, solve_method,
                sel, nthreads):
    arrs, qd, gd, (B, T, H, HV, K, V), gm = _prepare(q, k, v, g, beta, s0)
    scale = K ** -0.5 if scale is None else float(scale)
    sarr, nseq = _sel_array(sel, B, HV)
    o = np.zeros((nseq, T, V), np.float64)
    S = np.zeros((nseq, K, V), np.float64)
    rc = getattr(_load(), fname)(*[_ptr(a) for a in arrs], qd, gd, B, T, H, HV, K, V, gm, scale,
                                 int(bool(use_qk_l2norm)), int(chunk_size), int(solve_method),
                                 _ptr(sarr), nseq, _ptr(o), _ptr(S), int(nthreads))
    _check(rc, fname)
    return _reshape_out(o, S, sel, B, T, HV, K, V)


def chunkwise(q, k, v, g, beta, s0=None, *, scale=None, use_qk_l2norm=True, chunk_size=64,
              solve_method=0, sel=None, nthreads=0):
    """Chunk form with beta on the columns of A_kk (lecture notes), in float64."""
    return _chunk_call("gdr_oracle_chunkwise", q, k, v, g, beta, s0, scale, use_qk_l2norm,
                       chunk_size, solve_method, sel, nthreads)


def chunkwise_rowbeta(q, k, v, g, beta, s0=None, *, scale=None, use_qk_l2norm=True,
                      chunk_size=64, solve_method=0, sel=None, nthreads=0):
    """Chunk form with beta on the rows (UT transform of the blog, §2.3), in float64."""
    return _chunk_call("gdr_oracle_chunkwise_rowbeta", q, k, v, g, beta, s0, scale,
                       use_qk_l2norm, chunk_size, solve_method, sel, nthreads)


def bruteforce(q, k, v, g, beta, s0=None, *, scale=None, use_qk_l2norm=True):
    """Explicit products of the per-token maps (I - beta k k^T) diag(exp g); tiny sizes only."""
    arrs, qd, gd, (B, T, H, HV, K, V), gm = _prepare(q, k, v, g, beta, s0)
    scale = K ** -0.5 if scale is None else float(scale)
    o = np.zeros((B * HV, T, V), np.float64)
    S = np.zeros((B * HV, K, V), np.float64)
    rc = _load().gdr_oracle_bruteforce(*[_ptr(a) for a in arrs], qd, gd, B, T, H, HV, K, V, gm,
                                       scale, int(bool(use_qk_l2norm)), _ptr(o), _ptr(S))
    _check(rc, "gdr_oracle_bruteforce")
    return _reshape_out(o, S, None, B, T, HV, K, V)


def unit_lower_inverse(L, method=0):
    """(I + L)^{-1} for a strictly lower-triangular L (float64)."""
    L = np.ascontiguousarray(np.asarray(L, dtype=np.float64))
    C = L.shape[0]
    X = np.zeros_like(L)
    _check(_load().gdr_oracle_unit_lower_inverse(_ptr(L), C, int(method), _ptr(X)),
           "gdr_oracle_unit_lower_inverse")
    return X
