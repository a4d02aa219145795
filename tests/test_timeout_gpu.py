"""Bounded device waits: the error word and a wait that really runs out.

The one-launch forward (scalar gate, tensor-core path, few enough chains) has
chain CTAs wait for chunk flags that worker CTAs of the same launch raise.
Every such wait is bounded (gdr_set_flag_wait_limit). These tests check the
whole error path on the GPU without faulting or hanging it: a wait that gives
up records a code in the workspace error word, gdr_stream_status reports it as
GDR_ERR_TIMEOUT, the launch still ends by itself, and the device and the
library work normally afterwards.
"""
import math

import numpy as np
import pytest
import torch

import chunkwise_gated_delta_gdr_gb300 as gdr
from chunkwise_gated_delta_gdr_gb300 import inputs as gin
import oracle

pytestmark = pytest.mark.gpu


def _relerr(a, b):
    rms = math.sqrt(float(np.mean(np.asarray(b, np.float64) ** 2)))
    return float(np.max(np.abs(np.asarray(a, np.float64) - b))) / rms


def test_error_word_reads_as_timeout():
    """A nonzero error word in the workspace header is GDR_ERR_TIMEOUT; a zero
    one (or no workspace) is GDR_OK."""
    dev = torch.device("cuda:0")
    ws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    assert gdr.stream_status(None, ws) == gdr.GDR_OK
    assert gdr.stream_status(None, None) == gdr.GDR_OK
    ws[:4] = torch.tensor([8, 0, 0, 0], dtype=torch.uint8, device=dev)
    assert gdr.stream_status(None, ws) == gdr.GDR_ERR_TIMEOUT


def test_flag_wait_runs_out_then_device_is_usable():
    """With the flag-wait bound at 0 polls the chains give up on the first
    chunk flag (its producer needs microseconds), record the timeout and run
    to their end; the next call, with the default bound, on the same workspace
    matches the oracle."""
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], T=700, H=3, HV=3)
    x = gin.make_inputs(w)
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    dims = gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V, gdr.GDR_BF16, gdr.GDR_F32)
    assert gdr.chunk_fwd_path(dims, w.C, 0) == 2            # the one-launch form
    ws = torch.empty(gdr.chunk_fwd_workspace_size(dims, w.C, 0), dtype=torch.uint8, device=dev)
    old = gdr.set_flag_wait_limit(0)
    try:
        assert gdr.set_flag_wait_limit(-1) == 0              # read back, unchanged
        gdr.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, chunk_size=w.C,
                      scale=w.scale, out_dtype=torch.float32, workspace=ws)
        status = gdr.stream_status(None, ws)
    finally:
        gdr.set_flag_wait_limit(old)
    assert status == gdr.GDR_ERR_TIMEOUT
    assert gdr.set_flag_wait_limit(-1) == old
    o, S = gdr.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, chunk_size=w.C,
                         scale=w.scale, out_dtype=torch.float32, workspace=ws)
    assert gdr.stream_status(None, ws) == gdr.GDR_OK
    ro, rS = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], None, scale=w.scale)
    assert _relerr(o.cpu().numpy(), ro) <= 2e-3
    assert _relerr(S.cpu().numpy(), rS) <= 2e-3
