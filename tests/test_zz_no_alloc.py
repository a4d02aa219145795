"""gdr_chunk_fwd_noalloc: the forward pass for callers that cannot provide
device memory (it runs on a fixed scratch array owned by the library).

Checked through the C ABI against gdr_chunk_fwd with a caller workspace, on
two calls in a row with different inputs (the second call must not see the
first one's leftovers), within the parity tolerance of the other GPU tests.
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


@pytest.mark.parametrize("name,ov", [
    ("gdn_t4096_h12", dict(T=700, H=3, HV=3)),          # tensor-core path
    ("tiny_fp32", dict()),                             # general fp32 path
])
def test_noalloc_matches_workspace_entry_point(name, ov):
    dev = torch.device("cuda:0")
    tol = 2e-3 if gin.WORKLOADS[name].dtype == torch.bfloat16 else 1e-4
    for seed_shift in (0, 7):                      # two calls in a row, different inputs
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
        assert gdr.stream_status() == gdr.GDR_OK
        o, S = out.cpu().numpy(), fin.cpu().numpy()
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
        assert _relerr(o, o_ref.cpu().numpy()) <= tol
        assert _relerr(S, S_ref.cpu().numpy()) <= tol


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
