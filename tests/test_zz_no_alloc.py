"""gdr_chunk_fwd_noalloc: the forward pass for callers that cannot provide
device memory (it runs on a fixed scratch array owned by the library).

Checked through the C ABI against gdr_chunk_fwd with a caller workspace, on
two calls in a row with different inputs (the second call must not see the
first one's leftovers), within the parity tolerance of the other GPU tests:
on the scalar-gate and per-key-gate tensor-core paths and the general fp32
path, on calls that alternate between the gate kinds (each path lays the
scratch out differently), and on the size the header documents as fitting.
gdr_noalloc_stream_status reports a device-side timeout of a no-alloc call.
The file is named so that pytest collects it last.
"""
import math

import numpy as np
import pytest
import torch

import chunkwise_gated_delta_gdr_gb300 as gdr
from chunkwise_gated_delta_gdr_gb300 import inputs as gin

pytestmark = pytest.mark.gpu


def _relerr(a, b):
    rms = math.sqrt(float(np.mean(np.asarray(b, np.float64) ** 2)))
    return float(np.max(np.abs(np.asarray(a, np.float64) - b))) / (rms if rms > 0 else 1.0)


def _compare(name, ov, seed_shift):
    """One no-alloc call against gdr_chunk_fwd with a workspace, same inputs."""
    dev = torch.device("cuda:0")
    tol = 2e-3 if gin.WORKLOADS[name].dtype == torch.bfloat16 else 1e-4
    w = gin.shrink(gin.WORKLOADS[name], seed=gin.WORKLOADS[name].seed + seed_shift, **ov)
    x = {n: (t.to(dev) if t is not None else None) for n, t in gin.make_inputs(w).items()}
    s0 = torch.randn(w.B, w.HV, w.K, w.V, generator=torch.Generator().manual_seed(seed_shift),
                     ).to(dev) * 0.05
    o_ref, S_ref = gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], s0,
                                 chunk_size=w.C, scale=w.scale, out_dtype=torch.float32)
    out = torch.full((w.B, w.T, w.HV, w.V), float("nan"), device=dev)
    fin = torch.full((w.B, w.HV, w.K, w.V), float("nan"), device=dev)
    gdr.chunk_fwd_noalloc(x["q"], x["k"], x["v"], x["g"], x["beta"], s0, out=out,
                          final_state=fin, chunk_size=w.C, scale=w.scale)
    assert gdr.noalloc_stream_status() == gdr.GDR_OK
    o, S = out.cpu().numpy(), fin.cpu().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
    assert _relerr(o, o_ref.cpu().numpy()) <= tol
    assert _relerr(S, S_ref.cpu().numpy()) <= tol


CASES = {
    "gdn": ("gdn_t4096_h12", dict(T=700, H=3, HV=3)),                 # scalar gate, tensor cores
    "kda": ("kda_gqa_t8192", dict(B=1, T=300, H=2, HV=4)),            # per-key gate, tensor cores
    "fp32": ("tiny_fp32", dict()),                                    # general fp32 path
}


@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_matches_workspace_entry_point(case):
    name, ov = CASES[case]
    for seed_shift in (0, 7):                      # two calls in a row, different inputs
        _compare(name, ov, seed_shift)


def test_noalloc_alternating_paths():
    """Scalar gate, per-key gate, scalar gate again: each call overwrites what
    the previous path left in the shared scratch."""
    for i, case in enumerate(("gdn", "kda", "gdn", "kda")):
        name, ov = CASES[case]
        _compare(name, ov, 3 + i)


def test_noalloc_documented_size():
    """The examples the header gives: B=1, T=4096, 4 value heads, K=V=128,
    C=64, scalar gate, bf16 inputs fits the scratch (and runs); 5 value heads
    does not."""
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], H=4, HV=4)
    assert (w.B, w.T, w.HV, w.K, w.V, w.C) == (1, 4096, 4, 128, 128, 64)
    dims = gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V, gdr.GDR_BF16, gdr.GDR_F32)
    size = gdr.chunk_fwd_workspace_size(dims, w.C, w.gate_mode)
    assert size <= gdr.GDR_NOALLOC_SCRATCH_BYTES and abs(size / 1e6 - 54.8) < 0.05
    dims5 = gdr.make_dims(w.B, w.T, 5, 5, w.K, w.V, gdr.GDR_BF16, gdr.GDR_F32)
    size5 = gdr.chunk_fwd_workspace_size(dims5, w.C, w.gate_mode)
    assert size5 > gdr.GDR_NOALLOC_SCRATCH_BYTES and abs(size5 / 1e6 - 68.5) < 0.05
    _compare("gdn_t4096_h12", dict(H=4, HV=4), 0)


def test_noalloc_reports_a_device_timeout():
    """A flag wait of the no-alloc call that runs out (bound 0 polls) shows in
    gdr_noalloc_stream_status; the next call clears it."""
    dev = torch.device("cuda:0")
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], T=700, H=3, HV=3)
    x = {n: (t.to(dev) if t is not None else None) for n, t in gin.make_inputs(w).items()}
    out = torch.empty(w.B, w.T, w.HV, w.V, device=dev)
    old = gdr.set_flag_wait_limit(0)
    try:
        gdr.chunk_fwd_noalloc(x["q"], x["k"], x["v"], x["g"], x["beta"], None, out=out,
                              chunk_size=w.C, scale=w.scale)
        status = gdr.noalloc_stream_status()
    finally:
        gdr.set_flag_wait_limit(old)
    assert status == gdr.GDR_ERR_TIMEOUT
    _compare("gdn_t4096_h12", dict(T=700, H=3, HV=3), 11)


def test_noalloc_rejects_sizes_beyond_the_scratch():
    dev = torch.device("cuda:0")
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], T=16384, H=12, HV=12)   # ~250 MB workspace
    dims = gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V, gdr.GDR_BF16, gdr.GDR_F32)
    assert gdr.chunk_fwd_workspace_size(dims, w.C, w.gate_mode) > gdr.GDR_NOALLOC_SCRATCH_BYTES
    q = torch.zeros(w.B, w.T, w.H, w.K, dtype=torch.bfloat16, device=dev)
    v = torch.zeros(w.B, w.T, w.HV, w.V, dtype=torch.bfloat16, device=dev)
    g = torch.zeros(w.B, w.T, w.HV, device=dev)
    out = torch.zeros(w.B, w.T, w.HV, w.V, device=dev)
    with pytest.raises(gdr.GdrError) as e:
        gdr.chunk_fwd_noalloc(q, q, v, g, g, None, out=out, chunk_size=w.C)
    assert e.value.status == gdr.GDR_ERR_WORKSPACE
