"""GPU parity of the token-by-token form (gdr_recurrent_fwd, the decode step)
against the float64 oracle recurrence, which is the same definition."""
import math

import numpy as np
import pytest
import torch

import chunkwise_gated_delta_gdr_gb300 as gdr
from chunkwise_gated_delta_gdr_gb300 import inputs as gin
import oracle

pytestmark = pytest.mark.gpu


def relerr(a, b):
    rms = math.sqrt(float(np.mean(np.asarray(b, np.float64) ** 2)))
    return float(np.max(np.abs(np.asarray(a, np.float64) - b))) / (rms if rms > 0 else 1.0)


def inputs(name, seed=7, s0=0.05, **ov):
    w = gin.shrink(gin.WORKLOADS[name], seed=seed, **ov)
    x = gin.make_inputs(w)
    if x["s0"] is None:
        gen = torch.Generator().manual_seed(seed + 100)
        x["s0"] = torch.randn(w.B, w.HV, w.K, w.V, generator=gen) * s0
    return w, x


def run_gpu(w, x, gate=True, out_dtype=torch.float32):
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    state = d["s0"].clone()
    o = gdr.recurrent_fwd(d["q"], d["k"], d["v"], d["g"] if gate else None, d["beta"], state,
                          scale=w.scale, use_qk_l2norm=w.use_qk_l2norm, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), state.cpu().numpy()


def oracle_run(w, x, gate=True):
    g = x["g"] if gate else torch.zeros(w.B, w.T, w.HV)
    return oracle.recurrent(x["q"], x["k"], x["v"], g, x["beta"], x["s0"], scale=w.scale,
                            use_qk_l2norm=w.use_qk_l2norm)


CASES = [
    ("gdn_t4096_h12", dict(T=1, H=4, HV=8)),                    # decode step, GQA
    ("gdn_t4096_h12", dict(T=9, H=2, HV=2)),
    ("kda_gqa_t8192", dict(B=2, T=1, H=2, HV=4)),                # per-key gate
    ("kda_many_b64", dict(B=3, T=6, H=2, HV=2)),
    ("gdn_long_t65000", dict(T=3, H=2, HV=2, K=64, V=96)),       # K != V
    ("tiny_fp32", dict(T=11)),                                   # fp32 inputs, K = V = 32
    ("tiny_fp32", dict(T=4, K=20, V=40)),                        # ragged rows and columns
    ("tiny_fp32", dict(T=3, K=16, V=30)),                        # V % 4 != 0: fallback kernel
    ("gdn_t4096_h12", dict(B=2, T=2, H=3, HV=6, K=128, V=72)),   # ragged last V tile
    ("gdn_t4096_h12", dict(T=3, H=1, HV=2, K=256, V=128)),      # K = 256: 16 rows per warp
    ("kda_many_b64", dict(B=2, T=2, H=1, HV=2, K=200, V=40)),    # per-key, K between 128 and 256
]


@pytest.mark.parametrize("name,ov", CASES)
def test_recurrent_matches_oracle(name, ov):
    w, x = inputs(name, **ov)
    o, S = run_gpu(w, x)
    ro, rS = oracle_run(w, x)
    tol = 2e-3 if w.dtype == torch.bfloat16 else 1e-4
    assert relerr(o, ro) <= tol and relerr(S, rS) <= tol, (relerr(o, ro), relerr(S, rS))


@pytest.mark.parametrize("name", ["gdn_t4096_h12", "tiny_fp32"])
def test_recurrent_ungated(name):
    w, x = inputs(name, **(dict(T=5, H=2, HV=2) if name != "tiny_fp32" else dict(T=5)))
    o, S = run_gpu(w, x, gate=False)
    ro, rS = oracle_run(w, x, gate=False)
    tol = 2e-3 if w.dtype == torch.bfloat16 else 1e-4
    assert relerr(o, ro) <= tol and relerr(S, rS) <= tol


def test_recurrent_without_l2norm_and_bf16_output():
    w, x = inputs("gdn_t4096_h12", T=4, H=2, HV=2)
    x["q"] = torch.nn.functional.normalize(x["q"].float(), dim=-1).to(torch.bfloat16)
    x["k"] = torch.nn.functional.normalize(x["k"].float(), dim=-1).to(torch.bfloat16)
    import dataclasses
    w = dataclasses.replace(w, use_qk_l2norm=False)
    o32, S = run_gpu(w, x)
    o16, _ = run_gpu(w, x, out_dtype=torch.bfloat16)
    ro, rS = oracle_run(w, x)
    assert relerr(o32, ro) <= 2e-3 and relerr(S, rS) <= 2e-3
    assert np.array_equal(o16, torch.tensor(o32).to(torch.bfloat16).float().numpy())


def test_decode_continues_a_chunked_prefill():
    """chunk_fwd over T tokens, then one recurrent step, equals chunk_fwd over
    T + 1 tokens (last output and final state)."""
    w, x = inputs("gdn_t4096_h12", T=130, H=2, HV=4)
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    T = w.T
    cut = lambda t, a, b: t[:, a:b].contiguous()
    o_all, S_all = gdr.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["s0"], scale=w.scale,
                                 out_dtype=torch.float32)
    _, S_pre = gdr.chunk_fwd(cut(d["q"], 0, T - 1), cut(d["k"], 0, T - 1), cut(d["v"], 0, T - 1),
                             cut(d["g"], 0, T - 1), cut(d["beta"], 0, T - 1), d["s0"],
                             scale=w.scale, out_dtype=torch.float32)
    o_last = gdr.recurrent_fwd(cut(d["q"], T - 1, T), cut(d["k"], T - 1, T), cut(d["v"], T - 1, T),
                               cut(d["g"], T - 1, T), cut(d["beta"], T - 1, T), S_pre,
                               scale=w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert relerr(o_last[:, 0].cpu().numpy(), o_all[:, T - 1].cpu().numpy()) <= 2e-3
    assert relerr(S_pre.cpu().numpy(), S_all.cpu().numpy()) <= 2e-3


def test_steps_compose():
    """T tokens in one call equal T calls of one token (same fp32 arithmetic)."""
    w, x = inputs("kda_many_b64", B=2, T=5, H=2, HV=2)
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    S1 = d["s0"].clone()
    o1 = gdr.recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], S1, scale=w.scale,
                           out_dtype=torch.float32)
    S2 = d["s0"].clone()
    outs = []
    for t in range(w.T):
        sl = lambda a: a[:, t:t + 1].contiguous()
        outs.append(gdr.recurrent_fwd(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]), sl(d["beta"]),
                                      S2, scale=w.scale, out_dtype=torch.float32))
    torch.cuda.synchronize()
    assert torch.equal(o1, torch.cat(outs, dim=1)) and torch.equal(S1, S2)


# Many heads: several per CTA (1024 heads on 152 CTAs), both warp groups of the
# streaming kernel busy, its three-stage ring wrapping, also with several
# tokens per head; and fewer heads than CTAs (the second group idle).
@pytest.mark.parametrize("B,T,H,HV", [(64, 1, 16, 16), (40, 3, 8, 16), (7, 2, 3, 3)])
def test_many_heads_per_cta(B, T, H, HV):
    w = gin.shrink(gin.DECODE_WORKLOADS["decode_b64_h16"], B=B, T=T, H=H, HV=HV)
    x = gin.make_inputs(w)
    o, S = run_gpu(w, x)
    ro, rS = oracle_run(w, x)
    assert relerr(o, ro) <= 2e-3 and relerr(S, rS) <= 2e-3, (relerr(o, ro), relerr(S, rS))
