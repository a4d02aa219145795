"""GPU parity: the CUDA library against the float64 oracle, element by element.

Tolerances (the accuracy bound the method's statement sets for this forward
pass): max|o_gpu - o_ref| <= tol * rms(o_ref) and, separately,
max|S_gpu - S_ref| <= tol * rms(S_ref), with tol = 2e-3 for bf16 q/k/v and
1e-4 for fp32 q/k/v. o is compared in fp32 (rounding o itself to bf16 moves it
by up to half a bf16 ulp, about 8x more than the bound allows; the bf16-output
path is checked against the fp32-output path instead).

Sizes: every named workload shrunk so the oracle finishes in seconds while the
sequence still spans several chunks and ends in a ragged chunk, and every
named workload at full size with a sample of its (batch, head) sequences
recomputed by the oracle.
"""
import math

import numpy as np
import pytest
import torch

import chunkwise_gated_delta_gdr_gb300 as gdr
from chunkwise_gated_delta_gdr_gb300 import inputs as gin
import oracle

pytestmark = pytest.mark.gpu


def tol_for(w):
    return 2e-3 if w.dtype == torch.bfloat16 else 1e-4


def relerr(a, b):
    rms = math.sqrt(float(np.mean(np.asarray(b, np.float64) ** 2)))
    return float(np.max(np.abs(np.asarray(a, np.float64) - b))) / (rms if rms > 0 else 1.0)


def gpu_run(x, w, out_dtype=torch.float32, **kw):
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o, S = gdr.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["s0"], chunk_size=w.C,
                         scale=w.scale, use_qk_l2norm=w.use_qk_l2norm, out_dtype=out_dtype, **kw)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), S.cpu().numpy()


def check_against_oracle(w, x, sel=None, out_dtype=torch.float32):
    o, S = gpu_run(x, w, out_dtype)
    ro, rS = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["s0"], scale=w.scale,
                              use_qk_l2norm=w.use_qk_l2norm, sel=sel)
    if sel is not None:
        o = np.stack([o[s // w.HV, :, s % w.HV] for s in sel])
        S = np.stack([S[s // w.HV, s % w.HV] for s in sel])
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
    eo, es = relerr(o, ro), relerr(S, rS)
    tol = tol_for(w)
    assert eo <= tol, f"{w.name}: output error {eo:.3e} > {tol}"
    assert es <= tol, f"{w.name}: final-state error {es:.3e} > {tol}"
    return eo, es


SMALL = {
    "tiny_fp32": {},
    "gdn_t4096_h12": dict(T=300, H=2, HV=2),
    "kda_gqa_t8192": dict(B=1, T=200, H=2, HV=4),
    "gdn_long_t65000": dict(T=333, H=2, HV=2),
    "kda_many_b64": dict(B=3, T=130, H=2, HV=2),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_workloads(name):
    w = gin.shrink(gin.WORKLOADS[name], **SMALL[name])
    check_against_oracle(w, gin.make_inputs(w))


FULL_SAMPLES = {
    "tiny_fp32": None,
    "gdn_t4096_h12": None,                       # all 12 sequences
    "kda_gqa_t8192": [0, 1, 33, 63],             # (b, hv) = (0,0) (0,1) (1,1) (1,31)
    "gdn_long_t65000": [0, 31],
    "kda_many_b64": [0, 17, 512, 1023],
}


@pytest.mark.parametrize("name", list(FULL_SAMPLES))
def test_full_workloads_sampled(name):
    w = gin.WORKLOADS[name]
    check_against_oracle(w, gin.make_inputs(w), sel=FULL_SAMPLES[name])


# The one-launch forward's chunk counts around its own structure: the chain
# CTAs of a sequence produce its first four chunks, the workers the rest, and
# the output items wait for export marks every 16 chunks (every 4 in the last
# 16): one chunk, fewer chunks than chain CTAs, exactly four, one more, a
# ragged tail past the first mark, and several sequences with a carried state.
ONE_LAUNCH_SHAPES = [
    dict(T=1, H=3, HV=3),
    dict(T=64, H=2, HV=2),
    dict(T=130, H=2, HV=4),
    dict(T=256, H=1, HV=3),
    dict(T=257, H=3, HV=3),
    dict(T=1100, H=1, HV=2),
    dict(B=2, T=700, H=2, HV=2, s0_std=0.02),
]


@pytest.mark.parametrize("ov", ONE_LAUNCH_SHAPES, ids=lambda ov: "-".join(f"{k}{v}" for k, v in ov.items()))
def test_one_launch_chunk_counts(ov):
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], **ov)
    dims = gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V, gdr.GDR_BF16, gdr.GDR_F32)
    assert gdr.chunk_fwd_path(dims, w.C, 0) == 2          # the one-launch form
    check_against_oracle(w, gin.make_inputs(w))


@pytest.mark.parametrize("name", ["gdn_t4096_h12", "kda_gqa_t8192"])
def test_bf16_output_is_fp32_output_rounded(name):
    w = gin.shrink(gin.WORKLOADS[name], B=1, T=257, H=1, HV=2)
    x = gin.make_inputs(w)
    o32, S32 = gpu_run(x, w, torch.float32)
    o16, S16 = gpu_run(x, w, torch.bfloat16)
    ref = torch.from_numpy(o32).to(torch.bfloat16).float().numpy()
    ulp = np.abs(ref) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(o16 - ref) <= ulp)
    assert np.array_equal(S16, S32)


@pytest.mark.parametrize("T", [1, 5, 63, 64, 65, 129])
@pytest.mark.parametrize("name", ["gdn_long_t65000", "kda_many_b64"])
def test_short_and_boundary_lengths(name, T):
    w = gin.shrink(gin.WORKLOADS[name], B=1, T=T, H=1, HV=2, s0_std=0.02)
    check_against_oracle(w, gin.make_inputs(w))


def test_per_key_initial_state():
    """Per-key gate with a carried fp32 state, several chunks, GQA."""
    w = gin.shrink(gin.WORKLOADS["kda_gqa_t8192"], B=2, T=300, H=1, HV=2, s0_std=0.05)
    x = gin.make_inputs(w)
    assert x["s0"] is not None
    check_against_oracle(w, x)


@pytest.mark.parametrize("name", ["gdn_t4096_h12", "kda_many_b64"])
def test_zero_length_returns_initial_state(name):
    w = gin.shrink(gin.WORKLOADS[name], T=0, B=2, H=2, HV=2)
    x = gin.make_inputs(w)
    s0 = torch.randn(2, 2, w.K, w.V)
    x["s0"] = s0
    o, S = gpu_run(x, w)
    assert o.shape == (2, 0, 2, w.V)
    assert np.array_equal(S, s0.numpy())
    x["s0"] = None
    _, S = gpu_run(x, w)
    assert np.all(S == 0)


@pytest.mark.parametrize("name", ["gdn_long_t65000", "kda_many_b64"])
def test_final_state_may_alias_initial_state(name):
    w = gin.shrink(gin.WORKLOADS[name], B=1, T=150, H=2, HV=2, s0_std=0.02)
    x = gin.make_inputs(w)
    o_ref, S_ref = gpu_run(x, w)
    dev = torch.device("cuda:0")
    d = {n: t.to(dev) for n, t in x.items()}
    state = d["s0"].clone()
    o, S = gdr.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], state, chunk_size=w.C,
                         scale=w.scale, out_dtype=torch.float32, final_state=state)
    torch.cuda.synchronize()
    assert np.array_equal(S.cpu().numpy(), S_ref)
    assert np.array_equal(o.cpu().numpy(), o_ref)


def test_without_l2norm_prenormalised_keys():
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], T=200, H=2, HV=2, use_qk_l2norm=False)
    x = gin.make_inputs(w)
    for n in ("q", "k"):
        f = x[n].float()
        x[n] = (f / f.norm(dim=-1, keepdim=True)).to(w.dtype)
    check_against_oracle(w, x)


def test_reset_limit_gate():
    """g = -1000: every decay is exactly 0; nothing may turn into NaN."""
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], T=200, H=2, HV=2)
    x = gin.make_inputs(w)
    x["g"] = torch.full_like(x["g"], -1000.0)
    check_against_oracle(w, x)


def test_positive_small_gate():
    """g = 0.1 N(0,1) (gates may exceed 1, as in the optimisation script's smoke run)."""
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], T=256, H=2, HV=2)
    x = gin.make_inputs(w)
    x["g"] = torch.randn(x["g"].shape, generator=torch.Generator().manual_seed(9)) * 0.1
    check_against_oracle(w, x)


# Scalar-gate recipes for the tensor-core chunk kernel: a chunk whose gate
# cumsum strays more than 80 from its middle row's takes the decays element by
# element, the others as a row factor times a column factor; these cover both
# forms, and both within one sequence.
SCALAR_GATES = {
    "steep": lambda shape, gen: torch.full(shape, -4.0),            # spans ~250: element form
    "moderate": lambda shape, gen: torch.full(shape, -1.2),         # |G_i - G_m| <= 39: split form
    "mixed_spans": lambda shape, gen: -torch.randn(shape, generator=gen).abs() * 3.0,
    "alternating_chunks": lambda shape, gen: torch.where(
        (torch.arange(shape[1]) // 64) % 2 == 0, torch.tensor(-4.0), torch.tensor(-0.05)
    ).view(1, -1, 1).expand(shape).clone(),
}


@pytest.mark.parametrize("recipe", list(SCALAR_GATES))
def test_scalar_gate_ranges(recipe):
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], T=264, H=2, HV=2, s0_std=0.02)
    x = gin.make_inputs(w)
    x["g"] = SCALAR_GATES[recipe](tuple(x["g"].shape), torch.Generator().manual_seed(22)).float()
    check_against_oracle(w, x)


# Per-key gate recipes for the factorised decayed dots: a 16-row block whose
# gate span exceeds the factor limit is computed element by element, so these
# cover both branches and their mix within one chunk.
KDA_GATES = {
    "reset_limit": lambda shape, gen: torch.full(shape, -1000.0),
    "steep_half_channels": lambda shape, gen: torch.where(
        torch.arange(shape[-1]) % 2 == 0, torch.tensor(-5.0), torch.tensor(-0.01)).expand(shape).clone(),
    "mixed_spans": lambda shape, gen: -torch.randn(shape, generator=gen).abs() * 3.0,
    "positive_small": lambda shape, gen: torch.randn(shape, generator=gen) * 0.1,
}


@pytest.mark.parametrize("recipe", list(KDA_GATES))
def test_per_key_gate_ranges(recipe):
    w = gin.shrink(gin.WORKLOADS["kda_gqa_t8192"], B=1, T=200, H=1, HV=2)
    x = gin.make_inputs(w)
    x["g"] = KDA_GATES[recipe](tuple(x["g"].shape), torch.Generator().manual_seed(21)).float()
    check_against_oracle(w, x)


def test_split_sequence_matches_single_call():
    w = gin.shrink(gin.WORKLOADS["kda_gqa_t8192"], B=1, T=320, H=1, HV=2)
    x = gin.make_inputs(w)
    o, S = gpu_run(x, w)
    t1 = 100
    first = {n: (t[:, :t1].contiguous() if n != "s0" and t is not None else t) for n, t in x.items()}
    o1, S1 = gpu_run(first, w)
    second = {n: (t[:, t1:].contiguous() if n != "s0" and t is not None else t) for n, t in x.items()}
    second["s0"] = torch.from_numpy(S1)
    o2, S2 = gpu_run(second, w)
    tol = tol_for(w)
    assert relerr(np.concatenate([o1, o2], axis=1), o) <= tol
    assert relerr(S2, S) <= tol


def test_host_entry_point_matches_device_call():
    w = gin.shrink(gin.WORKLOADS["gdn_long_t65000"], T=200, H=2, HV=2)
    x = gin.make_inputs(w)
    o_ref, S_ref = gpu_run(x, w)
    pin = {n: t.pin_memory() for n, t in x.items()}
    dims = gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V, gdr.GDR_BF16, gdr.GDR_F32)
    nbytes = gdr.chunk_fwd_host_buffer_size(dims, w.C, w.gate_mode, True, True)
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda:0")
    out = torch.empty(w.B, w.T, w.HV, w.V, dtype=torch.float32).pin_memory()
    fin = torch.empty(w.B, w.HV, w.K, w.V, dtype=torch.float32).pin_memory()
    gdr.chunk_fwd_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"], pin["s0"], out=out,
                       final_state=fin, device_buffer=buf, chunk_size=w.C, scale=w.scale)
    assert gdr.stream_status() == gdr.GDR_OK
    assert np.array_equal(out.numpy(), o_ref)
    assert np.array_equal(fin.numpy(), S_ref)


def test_stream_status_ok_after_call():
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], T=128, H=1, HV=1)
    x = {n: (t.cuda() if t is not None else None) for n, t in gin.make_inputs(w).items()}
    dims = gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V, gdr.GDR_BF16, gdr.GDR_F32)
    ws = torch.empty(gdr.chunk_fwd_workspace_size(dims, w.C, w.gate_mode), dtype=torch.uint8,
                     device="cuda:0")
    gdr.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], None, chunk_size=w.C,
                  out_dtype=torch.float32, workspace=ws)
    assert gdr.stream_status(workspace=ws) == gdr.GDR_OK


@pytest.mark.parametrize("name", ["gdn_t4096_h12", "kda_gqa_t8192", "tiny_fp32"])
def test_prepare_then_recur_with_two_states(name):
    """prepare + recur equals chunk_fwd, and one prepared workspace serves two
    different initial states (the slabs do not depend on the state)."""
    w = gin.shrink(gin.WORKLOADS[name], B=1, T=150, H=1, HV=2)
    x = gin.make_inputs(w)
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    dims = gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V, gdr.GDR_BF16 if w.dtype == torch.bfloat16
                         else gdr.GDR_F32, gdr.GDR_F32)
    ws = torch.empty(gdr.chunk_fwd_workspace_size(dims, w.C, w.gate_mode), dtype=torch.uint8,
                     device=dev)
    gdr.chunk_prepare(d["q"], d["k"], d["v"], d["g"], d["beta"], workspace=ws, chunk_size=w.C,
                      scale=w.scale, out_dtype=torch.float32)
    for seed in (1, 2):
        s0 = torch.randn(w.B, w.HV, w.K, w.V, generator=torch.Generator().manual_seed(seed)) * 0.1
        out = torch.empty(w.B, w.T, w.HV, w.V, device=dev)
        fin = torch.empty(w.B, w.HV, w.K, w.V, device=dev)
        gdr.chunk_recur(d["q"], d["k"], s0.to(dev), workspace=ws, out=out, final_state=fin,
                        HV=w.HV, V=w.V, gate_mode=w.gate_mode, chunk_size=w.C, scale=w.scale)
        x2 = dict(x, s0=s0)
        o_ref, S_ref = gpu_run(x2, w)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), o_ref)
        assert np.array_equal(fin.cpu().numpy(), S_ref)


# ---- ungated delta rule (gate_mode none) and chunk size 128 ----------------------
# Ungated: the call passes g = None; the oracle runs the recurrence with g = 0,
# i.e. every decay factor 1 (plain DeltaNet).

def check_ungated(w, x):
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o, S = gdr.chunk_fwd(d["q"], d["k"], d["v"], None, d["beta"], d["s0"], chunk_size=w.C,
                         scale=w.scale, use_qk_l2norm=w.use_qk_l2norm, out_dtype=torch.float32)
    torch.cuda.synchronize()
    g0 = torch.zeros(w.B, w.T, w.HV, dtype=torch.float32)
    ro, rS = oracle.recurrent(x["q"], x["k"], x["v"], g0, x["beta"], x["s0"], scale=w.scale,
                              use_qk_l2norm=w.use_qk_l2norm)
    o, S = o.cpu().numpy(), S.cpu().numpy()
    tol = tol_for(w)
    assert relerr(o, ro) <= tol and relerr(S, rS) <= tol, (relerr(o, ro), relerr(S, rS))


@pytest.mark.parametrize("name,ov", [
    ("gdn_t4096_h12", dict(T=300, H=2, HV=2)),                   # tensor-core path
    ("gdn_long_t65000", dict(T=200, H=2, HV=4)),                 # with an initial state
    ("tiny_fp32", {}),                                           # general fp32 path
])
def test_ungated(name, ov):
    w = gin.shrink(gin.WORKLOADS[name], **ov)
    x = gin.make_inputs(w)
    assert gdr.chunk_fwd_path(gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V,
                                            gdr.GDR_BF16 if w.dtype == torch.bfloat16 else gdr.GDR_F32,
                                            gdr.GDR_F32), w.C, gdr.GDR_GATE_NONE) in \
        ((1, 2) if name != "tiny_fp32" else (0,))
    check_ungated(w, x)


def test_ungated_equals_zero_gate():
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], T=200, H=2, HV=2)
    x = gin.make_inputs(w)
    x0 = dict(x, g=torch.zeros_like(x["g"]))
    o0, S0 = gpu_run(x0, w)
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o1, S1 = gdr.chunk_fwd(d["q"], d["k"], d["v"], None, d["beta"], None, chunk_size=w.C,
                           scale=w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert np.array_equal(o0, o1.cpu().numpy()) and np.array_equal(S0, S1.cpu().numpy())


@pytest.mark.parametrize("name,ov", [
    ("gdn_t4096_h12", dict(T=300, H=2, HV=2, K=64, V=64, C=128)),
    ("gdn_long_t65000", dict(T=260, H=1, HV=2, K=64, V=48, C=128)),     # K != V, carried state
    ("kda_gqa_t8192", dict(B=1, T=200, H=1, HV=2, K=64, V=64, C=128)),
    ("tiny_fp32", dict(T=300, C=128)),
])
def test_chunk_size_128(name, ov):
    w = gin.shrink(gin.WORKLOADS[name], **ov)
    dims = gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V,
                         gdr.GDR_BF16 if w.dtype == torch.bfloat16 else gdr.GDR_F32, gdr.GDR_F32)
    assert gdr.chunk_fwd_path(dims, 128, w.gate_mode) == 0          # general path
    check_against_oracle(w, gin.make_inputs(w))


# Head dims up to 256 and C = 128 with full head dims: the general path streams
# the head dims through shared memory in 32-channel tiles.
LARGE_HEADS = [
    ("gdn_t4096_h12", dict(T=200, H=1, HV=2, K=256, V=256)),
    ("kda_gqa_t8192", dict(B=1, T=150, H=1, HV=2, K=256, V=128)),
    ("gdn_t4096_h12", dict(T=300, H=1, HV=2, K=128, V=128, C=128)),
    ("kda_many_b64", dict(B=2, T=200, H=1, HV=2, K=128, V=256, C=128, s0_std=0.02)),
    ("gdn_long_t65000", dict(T=170, H=1, HV=1, K=96, V=200, C=32)),
    ("tiny_fp32", dict(T=100, K=256, V=256, C=32)),
]


# Head dims that are not multiples of the general state kernel's 32-channel
# tiles or of its 4-wide register blocks in the value columns.
ODD_HEADS = [
    ("tiny_fp32", dict(T=77, K=20, V=36, C=16)),
    ("gdn_t4096_h12", dict(T=150, H=1, HV=2, K=100, V=60)),
    ("kda_gqa_t8192", dict(B=1, T=90, H=1, HV=2, K=36, V=50, C=32)),
]


@pytest.mark.parametrize("name,ov", ODD_HEADS)
def test_odd_head_dims(name, ov):
    w = gin.shrink(gin.WORKLOADS[name], **ov)
    assert gdr.chunk_fwd_path(gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V, 1, 0), w.C,
                              w.gate_mode) == 0
    check_against_oracle(w, gin.make_inputs(w))


@pytest.mark.parametrize("name,ov", LARGE_HEADS)
def test_large_head_dims(name, ov):
    w = gin.shrink(gin.WORKLOADS[name], **ov)
    assert gdr.chunk_fwd_path(gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V, 1, 0), w.C,
                              w.gate_mode) == 0
    check_against_oracle(w, gin.make_inputs(w))


def test_chunk_size_128_equals_64():
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], T=256, H=1, HV=1, K=64, V=64, C=128)
    x = gin.make_inputs(w)
    o128, S128 = gpu_run(x, w)
    o64, S64 = gpu_run(x, dataclasses_replace(w, C=64))
    assert relerr(o128, o64) <= 2e-3 and relerr(S128, S64) <= 2e-3


def dataclasses_replace(w, **kw):
    import dataclasses
    return dataclasses.replace(w, **kw)


# ---- Mamba2 SSD (no delta erase, no beta) on the chunk machinery ------------------

# The scalar-gate bf16 SSD runs the tensor-core path: the chunk-local stage forms
# each chunk's state increment and the chain is a scan of them. Its shapes: one
# token, fewer chunks than chain CTAs, batch with GQA and a ragged tail, a tail
# past the first export mark, and the two multi-launch forms (96 chains: chunk
# kernel, then chains beside the output items; 160 chains: chunk, chain and
# output kernels).
SSD_SHAPES = [
    ("gdn_t4096_h12", dict(T=300, H=2, HV=2)),                 # bf16, scalar gate, C = 64
    ("gdn_long_t65000", dict(T=200, H=2, HV=4)),               # carried state
    ("kda_gqa_t8192", dict(B=1, T=150, H=1, HV=2)),            # per-key gate
    ("tiny_fp32", {}),                                         # fp32, C = 16
    ("gdn_t4096_h12", dict(T=260, H=1, HV=2, K=64, V=64, C=128)),
    ("ssd_t4096_h12", dict(T=1, H=2, HV=2)),
    ("ssd_t4096_h12", dict(T=130, H=3, HV=3, s0_std=0.02)),
    ("ssd_t4096_h12", dict(B=2, T=700, H=2, HV=4, s0_std=0.02)),
    ("ssd_t4096_h12", dict(T=1100, H=1, HV=2)),
    ("ssd_t4096_h12", dict(T=200, H=24, HV=24)),
    ("ssd_t4096_h12", dict(T=130, H=40, HV=40)),
]


@pytest.mark.parametrize("name,ov", SSD_SHAPES)
def test_ssd_matches_oracle(name, ov):
    w = gin.shrink({**gin.WORKLOADS, **gin.SSD_WORKLOADS}[name], **ov)
    x = gin.make_inputs(w)
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o, S = gdr.ssd_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["s0"], chunk_size=w.C,
                             scale=w.scale, use_qk_l2norm=w.use_qk_l2norm, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ro, rS = oracle.ssd_recurrent(x["q"], x["k"], x["v"], x["g"], x["s0"], scale=w.scale,
                                  use_qk_l2norm=w.use_qk_l2norm)
    tol = tol_for(w)
    eo, es = relerr(o.cpu().numpy(), ro), relerr(S.cpu().numpy(), rS)
    assert eo <= tol and es <= tol, (eo, es)


def test_ssd_full_size():
    """The SSD workload at its full size (12 sequences of 4096 tokens), every
    sequence against the oracle, in the one-launch form the bench times."""
    w = gin.SSD_WORKLOADS["ssd_t4096_h12"]
    dims = gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V, gdr.GDR_BF16, gdr.GDR_F32)
    assert gdr.chunk_fwd_path(dims, w.C, 0) == 2
    x = gin.make_inputs(w)
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o, S = gdr.ssd_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["s0"], chunk_size=w.C,
                             scale=w.scale, use_qk_l2norm=w.use_qk_l2norm, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ro, rS = oracle.ssd_recurrent(x["q"], x["k"], x["v"], x["g"], x["s0"], scale=w.scale,
                                  use_qk_l2norm=w.use_qk_l2norm)
    o, S = o.cpu().numpy(), S.cpu().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
    tol = tol_for(w)
    eo, es = relerr(o, ro), relerr(S, rS)
    assert eo <= tol and es <= tol, (eo, es)


# ---- the fused recurrence on further shapes ---------------------------------------

@pytest.mark.parametrize("ov", [
    dict(B=3, T=200, H=2, HV=4),            # batch > 1, GQA, carried state below
    dict(B=2, T=64, H=1, HV=3),             # exactly one chunk
    dict(B=1, T=1000, H=4, HV=8),           # 64 chains, 16 chunks, ragged tail
])
def test_fused_recurrence_shapes(ov):
    w = gin.shrink(gin.WORKLOADS["gdn_long_t65000"], **ov)
    check_against_oracle(w, gin.make_inputs(w))


def test_fused_recurrence_reuses_its_flags():
    """One prepare, then three recurrences on the same workspace: each must wait
    for its own chains (the progress flags are reset per launch)."""
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], T=700, H=3, HV=3)
    x = gin.make_inputs(w)
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    dims = gdr.make_dims(w.B, w.T, w.H, w.HV, w.K, w.V, gdr.GDR_BF16, gdr.GDR_F32)
    ws = torch.empty(gdr.chunk_fwd_workspace_size(dims, w.C, 0), dtype=torch.uint8, device=dev)
    gdr.chunk_prepare(d["q"], d["k"], d["v"], d["g"], d["beta"], workspace=ws, scale=w.scale,
                      out_dtype=torch.float32)
    ro, rS = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], None, scale=w.scale)
    for rep in range(3):
        o = torch.full((w.B, w.T, w.HV, w.V), float("nan"), device=dev)
        S = torch.empty(w.B, w.HV, w.K, w.V, device=dev)
        gdr.chunk_recur(d["q"], d["k"], None, workspace=ws, out=o, final_state=S, HV=w.HV, V=w.V,
                        gate_mode=0, scale=w.scale)
        torch.cuda.synchronize()
        assert gdr.stream_status(None, ws) == gdr.GDR_OK
        assert relerr(o.cpu().numpy(), ro) <= 2e-3 and relerr(S.cpu().numpy(), rS) <= 2e-3


# ---- segmented scan (gdr_chunk_fwd_segmented) ---------------------------------------
SEGMENTED = [
    ("gdn_t4096_h12", dict(T=1024, H=2, HV=2, s0_std=0.02), 4),        # tensor-core path
    ("gdn_long_t65000", dict(T=2048, H=1, HV=2), 8),                   # carried state, long
    ("kda_gqa_t8192", dict(B=2, T=512, H=1, HV=2), 4),                 # per-key gate
    ("kda_many_b64", dict(B=1, T=256, H=1, HV=1, s0_std=0.02), 2),     # strong per-key decay
    ("tiny_fp32", dict(T=128), 2),                                     # fp32 general path
    ("gdn_t4096_h12", dict(T=512, H=1, HV=1, K=64, V=64, C=32), 4),    # general path, C = 32
]


@pytest.mark.parametrize("name,ov,segments", SEGMENTED)
def test_segmented_matches_oracle(name, ov, segments):
    w = gin.shrink(gin.WORKLOADS[name], **ov)
    x = gin.make_inputs(w)
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o, S = gdr.chunk_fwd_segmented(d["q"], d["k"], d["v"], d["g"], d["beta"], d["s0"],
                                   segments=segments, chunk_size=w.C, scale=w.scale,
                                   use_qk_l2norm=w.use_qk_l2norm, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ro, rS = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["s0"], scale=w.scale,
                              use_qk_l2norm=w.use_qk_l2norm)
    o, S = o.cpu().numpy(), S.cpu().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
    tol = tol_for(w)
    assert relerr(o, ro) <= tol and relerr(S, rS) <= tol
    # and close to the unsegmented call
    po, pS = gpu_run(x, w)
    assert relerr(o, po) <= tol and relerr(S, pS) <= tol


def test_segmented_one_segment_is_chunk_fwd():
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], T=300, H=2, HV=2)
    x = gin.make_inputs(w)
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o, S = gdr.chunk_fwd_segmented(d["q"], d["k"], d["v"], d["g"], d["beta"], None, segments=1,
                                   chunk_size=w.C, scale=w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    po, pS = gpu_run(x, w)
    assert np.array_equal(o.cpu().numpy(), po) and np.array_equal(S.cpu().numpy(), pS)


def test_segmented_aliased_state_bf16_output():
    """final_state aliasing initial_state and bf16 output (two batches, GQA): the
    bf16 output is the fp32 output rounded, the state the same bits."""
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], B=2, T=512, H=1, HV=2, s0_std=0.02)
    x = gin.make_inputs(w)
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o32, S32 = gdr.chunk_fwd_segmented(d["q"], d["k"], d["v"], d["g"], d["beta"], d["s0"],
                                       segments=4, chunk_size=w.C, scale=w.scale,
                                       out_dtype=torch.float32)
    state = d["s0"].clone()
    o16, S16 = gdr.chunk_fwd_segmented(d["q"], d["k"], d["v"], d["g"], d["beta"], state,
                                       segments=4, chunk_size=w.C, scale=w.scale,
                                       out_dtype=torch.bfloat16, final_state=state)
    torch.cuda.synchronize()
    assert S16.data_ptr() == state.data_ptr()
    ref = o32.to(torch.bfloat16).float().cpu().numpy()
    assert np.all(np.abs(o16.float().cpu().numpy() - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30)
    assert np.array_equal(state.cpu().numpy(), S32.cpu().numpy())
    ro, rS = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["s0"], scale=w.scale)
    tol = tol_for(w)
    assert relerr(o32.cpu().numpy(), ro) <= tol and relerr(state.cpu().numpy(), rS) <= tol


def test_segmented_more_chains_than_sms():
    """64 segments x 2 value heads x 8 column tiles = 1024 chains: the states-only
    launches of the recurrence run in waves; the outputs-only launch covers every SM."""
    w = gin.shrink(gin.WORKLOADS["gdn_long_t65000"], T=4096, H=1, HV=2)
    x = gin.make_inputs(w)
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o, S = gdr.chunk_fwd_segmented(d["q"], d["k"], d["v"], d["g"], d["beta"], d["s0"],
                                   segments=64, chunk_size=w.C, scale=w.scale,
                                   out_dtype=torch.float32)
    torch.cuda.synchronize()
    ro, rS = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["s0"], scale=w.scale)
    tol = tol_for(w)
    assert relerr(o.cpu().numpy(), ro) <= tol and relerr(S.cpu().numpy(), rS) <= tol


def test_segmented_ungated():
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], T=512, H=2, HV=2, s0_std=0.02)
    x = gin.make_inputs(w)
    dev = torch.device("cuda:0")
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o, S = gdr.chunk_fwd_segmented(d["q"], d["k"], d["v"], None, d["beta"], d["s0"], segments=4,
                                   chunk_size=w.C, scale=w.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    g0 = torch.zeros(w.B, w.T, w.HV, dtype=torch.float32)
    ro, rS = oracle.recurrent(x["q"], x["k"], x["v"], g0, x["beta"], x["s0"], scale=w.scale)
    tol = tol_for(w)
    assert relerr(o.cpu().numpy(), ro) <= tol and relerr(S.cpu().numpy(), rS) <= tol
