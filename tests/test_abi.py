"""C-ABI tests that need no GPU: the library builds, loads, exports every
function include/gdr.h declares, and rejects bad arguments before it touches
the device (argument errors return synchronously and enqueue nothing)."""
import ctypes
import os
import re

import pytest

import chunkwise_gated_delta_gdr_gb300 as gdr
from chunkwise_gated_delta_gdr_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gdr.load_library()


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(gdr_\w+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"gdr_chunk_fwd", "gdr_chunk_fwd_workspace_size", "gdr_stream_status",
            "gdr_status_string"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(gdr.EXPORTED) <= names


def test_status_strings(lib):
    for code in range(7):
        s = gdr.status_string(code)
        assert s.startswith("GDR_")
    assert "unknown" in gdr.status_string(99)


def test_version(lib):
    assert lib.gdr_version() >= (0 << 16) | (1 << 8)


def dims(**kw):
    base = dict(B=1, T=256, H=2, HV=4, K=128, V=128, in_dtype=gdr.GDR_BF16,
                out_dtype=gdr.GDR_F32)
    base.update(kw)
    return gdr.make_dims(**base)


def test_workspace_size_valid_and_invalid(lib):
    assert gdr.chunk_fwd_workspace_size(dims(), 64, 0) > 256
    assert gdr.chunk_fwd_workspace_size(dims(), 48, 0) == 0          # bad chunk size
    assert gdr.chunk_fwd_workspace_size(dims(HV=3), 64, 0) == 0      # HV % H != 0
    assert gdr.chunk_fwd_workspace_size(dims(K=257), 64, 0) == 0     # head dim
    assert gdr.chunk_fwd_workspace_size(dims(K=256, V=256), 64, 0) > 0
    assert gdr.chunk_fwd_workspace_size(dims(T=-1), 64, 0) == 0
    assert gdr.chunk_fwd_workspace_size(dims(), 64, 3) == 0          # gate mode
    small = gdr.chunk_fwd_workspace_size(dims(T=64), 64, 0)
    big = gdr.chunk_fwd_workspace_size(dims(T=4096), 64, 0)
    assert big > small


def test_path_choice(lib):
    assert gdr.chunk_fwd_path(dims(K=32, V=32), 16, 0) == 0
    assert gdr.chunk_fwd_path(dims(in_dtype=gdr.GDR_F32), 64, 0) == 0
    with pytest.raises(gdr.GdrError):
        gdr.chunk_fwd_path(dims(HV=3), 64, 0)


def _call(lib, d, q=16, k=16, v=16, g=16, beta=16, s0=None, out=16, sT=None, C=64, scale=0.1,
          gate=0, ws=None, ws_bytes=0):
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.gdr_chunk_fwd(P(q), P(k), P(v), P(g), P(beta), P(s0), C, ctypes.c_float(scale), 1,
                             gate, P(out), P(sT), ctypes.byref(d), P(ws), ctypes.c_size_t(ws_bytes),
                             None)


def test_argument_errors_are_synchronous(lib):
    # Fake, never-dereferenced addresses: every case is rejected before any CUDA call.
    A = 1 << 20
    d = dims()
    assert _call(lib, d, q=None, k=A, v=A, g=A, beta=A, out=A) == gdr.GDR_ERR_INVALID_ARG
    assert _call(lib, d, q=A, k=A, v=A, g=A, beta=A, out=None) == gdr.GDR_ERR_INVALID_ARG
    assert _call(lib, d, q=A + 8, k=A, v=A, g=A, beta=A, out=A) == gdr.GDR_ERR_ALIGNMENT
    assert _call(lib, d, q=A, k=A, v=A, g=A, beta=A, out=A, scale=0.0) == gdr.GDR_ERR_INVALID_ARG
    assert _call(lib, d, q=A, k=A, v=A, g=A, beta=A, out=A, scale=float("nan")) == \
        gdr.GDR_ERR_INVALID_ARG
    assert _call(lib, d, q=A, k=A, v=A, g=A, beta=A, out=A, C=48) == gdr.GDR_ERR_UNSUPPORTED
    assert _call(lib, dims(HV=3), q=A, k=A, v=A, g=A, beta=A, out=A) == gdr.GDR_ERR_INVALID_ARG
    assert _call(lib, dims(V=300), q=A, k=A, v=A, g=A, beta=A, out=A) == gdr.GDR_ERR_UNSUPPORTED
    assert _call(lib, d, q=A, k=A, v=A, g=A, beta=A, out=A, ws=None) == gdr.GDR_ERR_WORKSPACE
    need = gdr.chunk_fwd_workspace_size(d, 64, 0)
    assert _call(lib, d, q=A, k=A, v=A, g=A, beta=A, out=A, ws=A, ws_bytes=need - 1) == \
        gdr.GDR_ERR_WORKSPACE
    assert _call(lib, d, q=A, k=A, v=A, g=A, beta=A, out=A, ws=A + 16, ws_bytes=need) == \
        gdr.GDR_ERR_ALIGNMENT
    assert _call(lib, dims(B=0), q=None, k=None, v=None, g=None, beta=None, out=None) == gdr.GDR_OK


def test_host_buffer_size(lib):
    d = dims()
    base = gdr.chunk_fwd_host_buffer_size(d, 64, 0, False, False)
    with_states = gdr.chunk_fwd_host_buffer_size(d, 64, 0, True, True)
    assert base > gdr.chunk_fwd_workspace_size(d, 64, 0)
    assert with_states - base == 2 * 4 * 128 * 128 * 4


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        gdr.load_library(str(tmp_path / "nope.so"))


def test_ungated_mode_and_chunk_size_128_sizes(lib):
    d = dims()
    scalar = gdr.chunk_fwd_workspace_size(d, 64, gdr.GDR_GATE_SCALAR)
    assert gdr.chunk_fwd_workspace_size(d, 64, gdr.GDR_GATE_NONE) == scalar
    assert gdr.chunk_fwd_workspace_size(d, 64, 3) == 0
    # The ungated host buffer carries no gate array.
    g_bytes = 1 * 256 * 4 * 4
    assert (gdr.chunk_fwd_host_buffer_size(d, 64, gdr.GDR_GATE_SCALAR, False, False) -
            gdr.chunk_fwd_host_buffer_size(d, 64, gdr.GDR_GATE_NONE, False, False)) == g_bytes
    # C = 128 and head dims up to 256 run on the general path.
    assert gdr.chunk_fwd_workspace_size(dims(K=64, V=64), 128, 0) > 0
    assert gdr.chunk_fwd_path(dims(K=64, V=64), 128, 1) == 0
    assert gdr.chunk_fwd_path(dims(), 128, 0) == 0
    assert gdr.chunk_fwd_path(dims(K=256, V=64), 64, 1) == 0
    assert gdr.chunk_fwd_workspace_size(dims(K=64, V=257), 128, 0) == 0


def test_gate_array_required_unless_ungated(lib):
    A = 1 << 20
    d = dims()
    assert _call(lib, d, q=A, k=A, v=A, g=None, beta=A, out=A, gate=gdr.GDR_GATE_SCALAR) == \
        gdr.GDR_ERR_INVALID_ARG
    assert _call(lib, d, q=A, k=A, v=A, g=None, beta=A, out=A, gate=gdr.GDR_GATE_PER_KEY) == \
        gdr.GDR_ERR_INVALID_ARG
    assert _call(lib, d, q=A, k=A, v=A, g=A, beta=A, out=A, gate=3) == gdr.GDR_ERR_INVALID_ARG
    assert _call(lib, d, q=A, k=A, v=A, g=A, beta=A, out=A, C=96) == gdr.GDR_ERR_UNSUPPORTED


def test_recurrent_argument_errors(lib):
    A = 1 << 20
    P = ctypes.c_void_p
    def rec(d, g=A, gate=0, scale=0.1, q=A):
        return lib.gdr_recurrent_fwd(P(q) if q else None, P(A), P(A), P(g) if g else None, P(A),
                                     P(A), ctypes.c_float(scale), 1, gate, P(A), ctypes.byref(d),
                                     None)
    assert rec(dims(T=1), q=None) == gdr.GDR_ERR_INVALID_ARG
    assert rec(dims(T=1), g=None) == gdr.GDR_ERR_INVALID_ARG
    assert rec(dims(T=1), gate=3) == gdr.GDR_ERR_INVALID_ARG
    assert rec(dims(T=1), scale=0.0) == gdr.GDR_ERR_INVALID_ARG
    assert rec(dims(T=1, HV=3)) == gdr.GDR_ERR_INVALID_ARG
    assert rec(dims(T=1, K=257)) == gdr.GDR_ERR_UNSUPPORTED
    assert rec(dims(T=0)) == gdr.GDR_OK
    assert rec(dims(B=0, T=1)) == gdr.GDR_OK


def test_ssd_workspace_and_arguments(lib):
    d = dims()
    assert lib.gdr_ssd_chunk_fwd_workspace_size(ctypes.byref(d), 64, 0) > 256
    assert lib.gdr_ssd_chunk_fwd_workspace_size(ctypes.byref(d), 48, 0) == 0
    A = 1 << 20
    P = ctypes.c_void_p
    st = lib.gdr_ssd_chunk_fwd(P(A), P(A), P(A), None, None, 64, ctypes.c_float(0.1), 1, 0, P(A),
                               None, ctypes.byref(d), P(A), ctypes.c_size_t(1 << 40), None)
    assert st == gdr.GDR_ERR_INVALID_ARG                    # g required for a gated mode


def test_segmented_sizes_and_arguments(lib):
    d = dims(T=4096)
    plain = gdr.chunk_fwd_workspace_size(d, 64, 0)
    assert gdr.chunk_fwd_segmented_workspace_size(d, 64, 0, 1) == plain
    seg = gdr.chunk_fwd_segmented_workspace_size(d, 64, 0, 4)
    assert seg > plain                                                     # + states + o scratch
    assert gdr.chunk_fwd_segmented_workspace_size(d, 64, 0, 0) == 0        # segments >= 1
    assert gdr.chunk_fwd_segmented_workspace_size(dims(T=4000), 64, 0, 4) == 0   # T % (P C)
    assert gdr.chunk_fwd_segmented_workspace_size(dims(T=4096, V=64), 64, 0, 4) == 0  # K != V
    P = ctypes.c_void_p
    A = 1 << 20
    def seg(dd, segments, q=A, ws=None, nbytes=0):
        return lib.gdr_chunk_fwd_segmented(P(q) if q else None, P(A), P(A), P(A), P(A), None, 64,
                                           ctypes.c_float(0.1), 1, 0, segments, P(A), None,
                                           ctypes.byref(dd), P(ws) if ws else None,
                                           ctypes.c_size_t(nbytes), None)
    assert seg(d, 0) == gdr.GDR_ERR_INVALID_ARG
    assert seg(dims(T=4000), 4) == gdr.GDR_ERR_UNSUPPORTED
    assert seg(dims(T=4096, V=64), 4) == gdr.GDR_ERR_UNSUPPORTED
    assert seg(d, 4, q=None) == gdr.GDR_ERR_INVALID_ARG
    assert seg(d, 4) == gdr.GDR_ERR_WORKSPACE                               # nothing launched
