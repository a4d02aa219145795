"""Pins for the float64 oracle (CPU only).

The oracle is checked against things other than itself: a second and a third
formulation of the chunk form (beta on columns / on rows), brute-force
products of the per-token maps, three ways of inverting the triangular system,
closed forms of special cases worked out by hand, invariants of the
recurrence, and structural properties. ``test_planted_mistakes`` shows that a
plausible mistake in the recurrence (a dropped term, a wrong sign or index, a
transposed operand) fails at least one of these pins.

Sources: "分块并行计算（Chunkwise）" lecture notes (the recurrence, the chunk
equations and the listings naive_chunk_kda / inter-chunk loop),
"Chunkwise 并行算法 —— 线性注意力" (§1.1 gated linear attention form,
§2.1 Householder form, §2.3 UT transform, Neumann series and row recursion),
"DeltaNet chunk kernel optimization" (_l2norm, padding, default scale).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from chunkwise_gated_delta_gdr_gb300 import inputs as gin


def relerr(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    rms = math.sqrt(float(np.mean(b * b))) if b.size else 1.0
    if a.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b))) / (rms if rms > 0 else 1.0)


def rand_problem(seed, B=1, T=37, H=2, HV=4, K=16, V=12, gate_mode=0, g_mean=0.0, g_std=1.0,
                 s0=True, dtype=np.float64):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, K)).astype(dtype)
    k = rng.standard_normal((B, T, H, K)).astype(dtype)
    v = rng.standard_normal((B, T, HV, V)).astype(dtype)
    gshape = (B, T, HV) if gate_mode == 0 else (B, T, HV, K)
    x = rng.standard_normal(gshape) * g_std + g_mean
    g = -np.logaddexp(0.0, -x)                          # logsigmoid
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, HV))))
    S0 = rng.standard_normal((B, HV, K, V)) * 0.1 if s0 else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, s0=S0)


def run(fn, p, **kw):
    return fn(p["q"], p["k"], p["v"], p["g"], p["beta"], p["s0"], **kw)


# ---------------------------------------------------------------- P-1, P-3
@pytest.mark.parametrize("gate_mode", [0, 1])
@pytest.mark.parametrize("C", [1, 4, 16, 64])
def test_chunkwise_equals_recurrence(gate_mode, C):
    """Chunk form (lecture notes) equals the token recurrence to 1e-10 in float64.

    T=37 leaves a ragged last chunk for every C > 1; HV=2H exercises GQA; a
    non-zero initial state exercises the inter-chunk term. C=1 is the case
    M = I, W = exp(g) k, U = v, which must reproduce the recurrence exactly.
    """
    p = rand_problem(10 + C + gate_mode, gate_mode=gate_mode)
    o_r, s_r = run(oracle.recurrent, p)
    o_c, s_c = run(oracle.chunkwise, p, chunk_size=C)
    assert relerr(o_c, o_r) <= 1e-10
    assert relerr(s_c, s_r) <= 1e-10


@pytest.mark.parametrize("gate_mode", [0, 1])
def test_row_beta_equals_column_beta(gate_mode):
    """beta on the columns of A_kk (notes) and on the rows (blog §2.3) agree:
    diag(beta) (I + L_col)^{-1} = (I + L_row)^{-1} diag(beta)."""
    p = rand_problem(3 + gate_mode, gate_mode=gate_mode, T=50)
    o_c, s_c = run(oracle.chunkwise, p, chunk_size=16)
    o_r, s_r = run(oracle.chunkwise_rowbeta, p, chunk_size=16)
    assert relerr(o_r, o_c) <= 1e-12
    assert relerr(s_r, s_c) <= 1e-12


@pytest.mark.parametrize("method", [1, 2])
def test_chunkwise_solve_methods(method):
    """The chunk form gives the same result whichever way M^{-1} is applied."""
    p = rand_problem(21, T=40, gate_mode=1)
    o0, s0 = run(oracle.chunkwise, p, chunk_size=16, solve_method=0)
    o1, s1 = run(oracle.chunkwise, p, chunk_size=16, solve_method=method)
    assert relerr(o1, o0) <= 1e-12
    assert relerr(s1, s0) <= 1e-12


# ---------------------------------------------------------------- P-4
@pytest.mark.parametrize("C", [1, 2, 16, 64])
def test_unit_lower_inverse_three_ways(C):
    """(I + L)^{-1}: forward substitution, Neumann series sum (-L)^n, row recursion."""
    rng = np.random.default_rng(C)
    L = np.tril(rng.standard_normal((C, C)) * 0.3, -1)
    X = [oracle.unit_lower_inverse(L, m) for m in (0, 1, 2)]
    ident = np.eye(C)
    for Xi in X:
        assert np.max(np.abs(Xi @ (ident + L) - ident)) <= 1e-12
        assert np.max(np.abs((ident + L) @ Xi - ident)) <= 1e-12
        assert np.allclose(np.triu(Xi, 1), 0.0)
        assert np.allclose(np.diag(Xi), 1.0)
    assert np.max(np.abs(X[1] - X[0])) <= 1e-12
    assert np.max(np.abs(X[2] - X[0])) <= 1e-12


def test_unit_lower_inverse_closed_form():
    """Bidiagonal L = -a on the first subdiagonal: (I + L)^{-1}[i, j] = a^(i-j)."""
    C, a = 9, 0.7
    L = np.diag(np.full(C - 1, -a), -1)
    expect = np.array([[a ** (i - j) if i >= j else 0.0 for j in range(C)] for i in range(C)])
    for m in (0, 1, 2):
        assert np.max(np.abs(oracle.unit_lower_inverse(L, m) - expect)) <= 1e-14


# ---------------------------------------------------------------- P-2
@pytest.mark.parametrize("gate_mode", [0, 1])
@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_bruteforce_products(gate_mode, T):
    """The recurrence equals the explicit product form of the gated
    Householder maps S_t = (I - beta_t k_t k_t^T) diag(exp g_t) S_{t-1} + beta_t k_t v_t^T."""
    p = rand_problem(40 + T, T=T, K=6, V=5, H=1, HV=2, gate_mode=gate_mode)
    o_b, s_b = run(oracle.bruteforce, p)
    o_r, s_r = run(oracle.recurrent, p)
    assert relerr(o_r, o_b) <= 1e-12
    assert relerr(s_r, s_b) <= 1e-12


# ---------------------------------------------------------------- ungated mode
@pytest.mark.parametrize("C", [1, 16, 128])
def test_ungated_is_householder_deltanet(C):
    """With g = 0 (the library's ungated mode) the method is plain DeltaNet:
    in the value-by-key convention of the Chunkwise blog (section 2.1),
    S_t = S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T and o_t = S_t q_t.
    Computed here in that transposed form, per head, and compared with the
    oracle's recurrence and chunk form run with a zero gate."""
    p = rand_problem(71, T=150, K=8, V=6, H=1, HV=2)
    p["g"] = np.zeros_like(p["g"])
    B, T, H, K = p["q"].shape
    HV, V = p["v"].shape[2], p["v"].shape[3]
    scale = 1.0 / math.sqrt(K)
    o_ref = np.zeros((B, T, HV, V))
    s_ref = np.zeros((B, HV, K, V))
    for hv in range(HV):
        St = p["s0"][0, hv].T.copy()                       # V x K
        for t in range(T):
            kk = p["k"][0, t, 0] / math.sqrt(np.sum(p["k"][0, t, 0] ** 2) + 1e-6)
            qq = p["q"][0, t, 0] / math.sqrt(np.sum(p["q"][0, t, 0] ** 2) + 1e-6)
            b = p["beta"][0, t, hv]
            St = St @ (np.eye(K) - b * np.outer(kk, kk)) + b * np.outer(p["v"][0, t, hv], kk)
            o_ref[0, t, hv] = St @ (scale * qq)
        s_ref[0, hv] = St.T
    o_r, s_r = run(oracle.recurrent, p, scale=scale)
    assert o_r.shape == o_ref.shape and relerr(o_r, o_ref) <= 1e-12
    assert relerr(s_r, s_ref) <= 1e-12
    o_c, s_c = run(oracle.chunkwise, p, scale=scale, chunk_size=C)
    assert relerr(o_c, o_r) <= 1e-10 and relerr(s_c, s_r) <= 1e-10


# ---------------------------------------------------------------- Mamba2 SSD (NEXT row)
def _ssd_block_expansion(p, hv, scale, per_key):
    """Block expansion of the SSD recurrence (Chunkwise blog, section 1.2),
    written as whole-sequence matrix algebra for one head:
      O   = ((Q~ K^T) (.) Gamma) V + (Q~ (.) exp G) S0,  Gamma_ij = exp(G_i - G_j), j <= i
      S_T = K^T diag(exp(G_T - G)) V + diag(exp G_T) S0
    with G the cumulative sum of the log-decays (per key channel if per_key)."""
    q = p["q"][0, :, 0]
    k = p["k"][0, :, 0]
    qn = q / np.sqrt(np.sum(q ** 2, 1, keepdims=True) + 1e-6) * scale
    kn = k / np.sqrt(np.sum(k ** 2, 1, keepdims=True) + 1e-6)
    v = p["v"][0, :, hv]
    S0 = p["s0"][0, hv]
    T = q.shape[0]
    if not per_key:
        G = np.cumsum(p["g"][0, :, hv])
        Gam = np.tril(np.exp(G[:, None] - G[None, :]))
        O = ((qn @ kn.T) * Gam) @ v + (qn * np.exp(G)[:, None]) @ S0
        ST = kn.T @ (np.exp(G[-1] - G)[:, None] * v) + np.exp(G[-1]) * S0
    else:
        G = np.cumsum(p["g"][0, :, hv], axis=0)                     # T x K
        A = np.einsum("ic,jc,ijc->ij", qn, kn, np.exp(G[:, None, :] - G[None, :, :]))
        O = np.tril(A) @ v + (qn * np.exp(G)) @ S0
        ST = (kn * np.exp(G[-1][None, :] - G)).T @ v + np.exp(G[-1])[:, None] * S0
    return O, ST


@pytest.mark.parametrize("gate_mode", [0, 1])
def test_ssd_equals_block_expansion(gate_mode):
    p = rand_problem(91, T=33, K=7, V=5, H=1, HV=2, gate_mode=gate_mode)
    scale = 0.37
    o, S = oracle.ssd_recurrent(p["q"], p["k"], p["v"], p["g"], p["s0"], scale=scale)
    for hv in range(2):
        O, ST = _ssd_block_expansion(p, hv, scale, gate_mode == 1)
        assert relerr(o[0, :, hv], O) <= 1e-12
        assert relerr(S[0, hv], ST) <= 1e-12


def test_ssd_without_decay_is_causal_linear_attention():
    """alpha = 1 and a zero initial state: O = tril(Q K^T) V (no normalisation)."""
    p = rand_problem(92, T=20, K=6, V=4, H=1, HV=1, s0=False)
    p["g"] = np.zeros_like(p["g"])
    o, S = oracle.ssd_recurrent(p["q"], p["k"], p["v"], p["g"], None, scale=1.0,
                                use_qk_l2norm=False)
    q, k, v = p["q"][0, :, 0], p["k"][0, :, 0], p["v"][0, :, 0]
    assert relerr(o[0, :, 0], np.tril(q @ k.T) @ v) <= 1e-12
    assert relerr(S[0, 0], k.T @ v) <= 1e-12


# ---------------------------------------------------------------- P-9, hand-worked cases
def test_single_token_closed_form():
    """T = 1: S_1 = (I - beta k k^T) D S_0 + beta k v^T, o = S_1^T (scale q)."""
    p = rand_problem(7, T=1, K=8, V=3, H=1, HV=1, gate_mode=1)
    o, S = run(oracle.recurrent, p)
    q = p["q"][0, 0, 0]
    k = p["k"][0, 0, 0]
    qn = q / math.sqrt(q @ q + 1e-6)
    kn = k / math.sqrt(k @ k + 1e-6)
    b = p["beta"][0, 0, 0]
    D = np.diag(np.exp(p["g"][0, 0, 0]))
    S1 = (np.eye(8) - b * np.outer(kn, kn)) @ D @ p["s0"][0, 0] + b * np.outer(kn, p["v"][0, 0, 0])
    assert np.max(np.abs(S[0, 0] - S1)) <= 1e-14
    assert np.max(np.abs(o[0, 0, 0] - S1.T @ (qn / math.sqrt(8)))) <= 1e-14


def _hand(q, k, v, g, beta, s0):
    a = lambda x: np.asarray(x, np.float64)
    return dict(q=a(q), k=a(k), v=a(v), g=a(g), beta=a(beta), s0=a(s0))


def test_hand_worked_scalar_gate():
    """Two tokens worked by hand (scale 1, keys already unit, K = V = 2).

    S0 = [[1,0],[0,2]]. Token 1: decay 1/2 -> [[1/2,0],[0,1]]; k=(1,0), v=(3,4),
    beta=1/2: S^T k = (1/2,0), residual (5/2,4), S += 1/2 k (5/2,4) ->
    [[7/4,2],[0,1]]; q=(1,1) gives o_1 = (7/4, 3).
    Token 2: decay 1; k=(0.6,0.8), v=(1,0), beta=1: S^T k = (1.05, 2),
    residual (-0.05,-2), S = [[1.72,0.8],[-0.04,-0.6]] (and S^T k = v exactly);
    q=(0,1) gives o_2 = (-0.04, -0.6).
    """
    p = _hand(q=[[[[1, 1]], [[0, 1]]]], k=[[[[1, 0]], [[0.6, 0.8]]]],
              v=[[[[3, 4]], [[1, 0]]]], g=[[[math.log(0.5)], [0.0]]],
              beta=[[[0.5], [1.0]]], s0=[[[[1, 0], [0, 2]]]])
    for fn in (oracle.recurrent, oracle.bruteforce):
        o, S = run(fn, p, scale=1.0, use_qk_l2norm=False)
        assert np.max(np.abs(o[0, :, 0] - np.array([[1.75, 3.0], [-0.04, -0.6]]))) <= 1e-14
        assert np.max(np.abs(S[0, 0] - np.array([[1.72, 0.8], [-0.04, -0.6]]))) <= 1e-14
    for C in (1, 2):
        o, S = run(oracle.chunkwise, p, scale=1.0, use_qk_l2norm=False, chunk_size=C)
        assert np.max(np.abs(S[0, 0] - np.array([[1.72, 0.8], [-0.04, -0.6]]))) <= 1e-14


def test_hand_worked_per_key_gate():
    """Per-key decay worked by hand (K = 2, V = 1, scale 1).

    S0 = (2, 4). Token 1: decays (1/2, 1/4) -> (1, 1); k=(1,0), v=5, beta=1:
    residual 4, S = (5, 1); q=(1,2) gives o_1 = 7.
    Token 2: decays (1, 1/2) -> (5, 1/2); k=(0,1), v=3, beta=1/2: residual 5/2,
    S = (5, 7/4); q=(2,2) gives o_2 = 13.5.
    """
    p = _hand(q=[[[[1, 2]], [[2, 2]]]], k=[[[[1, 0]], [[0, 1]]]], v=[[[[5]], [[3]]]],
              g=[[[[math.log(0.5), math.log(0.25)]], [[0.0, math.log(0.5)]]]],
              beta=[[[1.0], [0.5]]], s0=[[[[2], [4]]]])
    for fn in (oracle.recurrent, oracle.bruteforce):
        o, S = run(fn, p, scale=1.0, use_qk_l2norm=False)
        assert np.max(np.abs(o[0, :, 0, 0] - np.array([7.0, 13.5]))) <= 1e-14
        assert np.max(np.abs(S[0, 0, :, 0] - np.array([5.0, 1.75]))) <= 1e-14
    o, S = run(oracle.chunkwise, p, scale=1.0, use_qk_l2norm=False, chunk_size=2)
    assert np.max(np.abs(o[0, :, 0, 0] - np.array([7.0, 13.5]))) <= 1e-14


def test_hand_worked_l2norm_and_head_groups():
    """L2 norm with eps inside the root, and two value heads sharing one q/k head.

    q=(3,4), k=(0,2): q_hat = (0.6,0.8)/sqrt(1+4e-8), k_hat = (0,1)/sqrt(1+2.5e-7).
    S0 = 0, g = 0, scale 1. Head 0: v=1, beta=1 -> o = 0.8 c_q c_k.
    Head 1: v=3, beta=1/2 -> o = 1.2 c_q c_k.
    """
    p = _hand(q=[[[[3, 4]]]], k=[[[[0, 2]]]], v=[[[[1], [3]]]], g=[[[0.0, 0.0]]],
              beta=[[[1.0, 0.5]]], s0=np.zeros((1, 2, 2, 1)))
    cq = 1.0 / math.sqrt(1.0 + 4e-8)
    ck = 1.0 / math.sqrt(1.0 + 2.5e-7)
    o, _ = run(oracle.recurrent, p, scale=1.0, use_qk_l2norm=True)
    assert abs(o[0, 0, 0, 0] - 0.8 * cq * ck) <= 1e-15
    assert abs(o[0, 0, 1, 0] - 1.2 * cq * ck) <= 1e-15


# ---------------------------------------------------------------- P-5
def test_beta_zero_only_decays_the_state():
    """beta = 0: o_t = S0^T (exp(G_t) * scale q_t), G the running cumsum of g."""
    p = rand_problem(11, T=20, K=8, V=6, H=1, HV=1, gate_mode=1)
    p["beta"] = np.zeros_like(p["beta"])
    o, S = run(oracle.recurrent, p)
    q = p["q"][0, :, 0]
    qn = q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6)
    G = np.cumsum(p["g"][0, :, 0], axis=0)
    expect = (np.exp(G) * qn / math.sqrt(8)) @ p["s0"][0, 0]
    assert relerr(o[0, :, 0], expect) <= 1e-12
    assert relerr(S[0, 0], np.exp(G[-1])[:, None] * p["s0"][0, 0]) <= 1e-12


def test_beta_zero_gate_zero_is_a_read():
    """beta = 0 and g = 0: o_t = S0^T (scale q_hat_t)."""
    p = rand_problem(12, T=9, K=8, V=6, H=1, HV=1)
    p["beta"] = np.zeros_like(p["beta"])
    p["g"] = np.zeros_like(p["g"])
    o, _ = run(oracle.recurrent, p)
    q = p["q"][0, :, 0]
    qn = q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6)
    assert relerr(o[0, :, 0], (qn / math.sqrt(8)) @ p["s0"][0, 0]) <= 1e-12


def test_unit_beta_stores_the_pair():
    """beta = 1, unit keys, g = 0: after the write S_t^T k_t = v_t exactly.
    With q = k and scale 1 the output is o_t = S_t^T k_t = v_t."""
    p = rand_problem(13, T=15, K=8, V=6, H=1, HV=1)
    k = p["k"] / np.linalg.norm(p["k"], axis=-1, keepdims=True)
    p.update(k=k, q=k.copy(), beta=np.ones_like(p["beta"]), g=np.zeros_like(p["g"]))
    o, _ = run(oracle.recurrent, p, scale=1.0, use_qk_l2norm=False)
    assert np.max(np.abs(o[0, :, 0] - p["v"][0, :, 0])) <= 1e-12
    o, _ = run(oracle.chunkwise, p, scale=1.0, use_qk_l2norm=False, chunk_size=4)
    assert np.max(np.abs(o[0, :, 0] - p["v"][0, :, 0])) <= 1e-12


# ---------------------------------------------------------------- P-6
@pytest.mark.parametrize("gate_mode", [0, 1])
def test_orthonormal_keys_reduce_to_gated_linear_attention(gate_mode):
    """Distinct one-hot keys never interfere, so nothing is erased and the rule
    becomes gated linear attention, O = ((Q K^T) * Gamma * causal) diag(beta) V
    with Gamma[t, u] = exp(G_t - G_u) (blog §1.1, Mamba2 form; per channel of
    the key's one-hot index for the per-key gate)."""
    T, K, V = 12, 16, 5
    rng = np.random.default_rng(5)
    perm = rng.permutation(K)[:T]
    p = rand_problem(14, T=T, K=K, V=V, H=1, HV=1, gate_mode=gate_mode, s0=False)
    k = np.zeros((1, T, 1, K))
    k[0, np.arange(T), 0, perm] = 1.0
    p["k"] = k
    p["s0"] = None
    scale = 0.37
    q = p["q"][0, :, 0] * scale
    G = np.cumsum(p["g"][0, :, 0], axis=0)
    b = p["beta"][0, :, 0]
    expect = np.zeros((T, V))
    for t in range(T):
        for u in range(t + 1):
            c = perm[u]
            gam = math.exp((G[t] - G[u]) if gate_mode == 0 else (G[t, c] - G[u, c]))
            expect[t] += q[t, c] * gam * b[u] * p["v"][0, u, 0]
    for fn, kw in ((oracle.recurrent, {}), (oracle.chunkwise, {"chunk_size": 4})):
        o, _ = run(fn, p, scale=scale, use_qk_l2norm=False, **kw)
        assert relerr(o[0, :, 0], expect) <= 1e-12


# ---------------------------------------------------------------- P-7
def test_reset_limit():
    """g = -1000: every decay underflows to exactly 0, so each token sees only
    itself: o_t = scale * beta_t (q_hat_t . k_hat_t) v_t (no NaN from exp range)."""
    p = rand_problem(15, T=23, K=8, V=6, H=1, HV=2)
    p["g"] = np.full_like(p["g"], -1000.0)
    q = p["q"][0, :, 0]
    k = p["k"][0, :, 0]
    qn = q / np.sqrt((q * q).sum(-1, keepdims=True) + 1e-6)
    kn = k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
    dots = (qn * kn).sum(-1) / math.sqrt(8)
    for fn, kw in ((oracle.recurrent, {}), (oracle.chunkwise, {"chunk_size": 8})):
        o, _ = run(fn, p, **kw)
        assert np.all(np.isfinite(o))
        for hv in range(2):
            expect = (dots * p["beta"][0, :, hv])[:, None] * p["v"][0, :, hv]
            assert relerr(o[0, :, hv], expect) <= 1e-12


# ---------------------------------------------------------------- P-8
def test_split_sequence_with_carried_state():
    """Running T tokens at once equals running the first part, then the rest
    starting from the carried state (mid-chunk split)."""
    p = rand_problem(16, T=45, gate_mode=1)
    o, S = run(oracle.recurrent, p)
    t1 = 19
    first = {n: (x[:, :t1] if n not in ("s0",) and x is not None else x) for n, x in p.items()}
    o1, S1 = run(oracle.chunkwise, first, chunk_size=8)
    second = {n: (x[:, t1:] if n not in ("s0",) and x is not None else x) for n, x in p.items()}
    second["s0"] = S1
    o2, S2 = run(oracle.chunkwise, second, chunk_size=8)
    assert relerr(np.concatenate([o1, o2], axis=1), o) <= 1e-10
    assert relerr(S2, S) <= 1e-10


def test_zero_tokens_are_padding():
    """Appending tokens with q = k = v = 0, g = 0, beta = 0 (the padding of
    the optimisation script) changes neither the outputs nor the final state."""
    p = rand_problem(17, T=21)
    o, S = run(oracle.recurrent, p)
    padded = {}
    for n, x in p.items():
        if n == "s0":
            padded[n] = x
            continue
        pad_shape = list(x.shape)
        pad_shape[1] = 11
        padded[n] = np.concatenate([x, np.zeros(pad_shape)], axis=1)
    o2, S2 = run(oracle.recurrent, padded)
    assert np.max(np.abs(o2[:, :21] - o)) <= 1e-13
    assert np.max(np.abs(o2[:, 21:])) == 0.0
    assert np.max(np.abs(S2 - S)) <= 1e-13


def test_gqa_equals_explicit_repeat():
    """HV = 2H equals the same run with q and k repeated per value head
    (repeat_interleave: value head hv reads q/k head hv // (HV/H))."""
    p = rand_problem(18, T=30, H=2, HV=6, gate_mode=1)
    o, S = run(oracle.recurrent, p)
    rep = dict(p)
    rep["q"] = np.repeat(p["q"], 3, axis=2)
    rep["k"] = np.repeat(p["k"], 3, axis=2)
    o2, S2 = run(oracle.recurrent, rep)
    assert np.max(np.abs(o2 - o)) <= 1e-13
    assert np.max(np.abs(S2 - S)) <= 1e-13


def test_per_key_gate_with_equal_channels_is_scalar_gate():
    p = rand_problem(19, T=33, gate_mode=0)
    o, S = run(oracle.recurrent, p)
    kda = dict(p)
    kda["g"] = np.repeat(p["g"][..., None], p["q"].shape[-1], axis=-1)
    o2, S2 = run(oracle.chunkwise, kda, chunk_size=8)
    assert relerr(o2, o) <= 1e-10
    assert relerr(S2, S) <= 1e-10


def test_linear_in_values_and_state():
    """For fixed q, k, g, beta the outputs and final state are linear in (v, S0)."""
    p1 = rand_problem(20, T=26, gate_mode=1)
    p2 = rand_problem(21, T=26, gate_mode=1)
    a, b = 0.7, -1.3
    mix = dict(p1)
    mix["v"] = a * p1["v"] + b * p2["v"]
    mix["s0"] = a * p1["s0"] + b * p2["s0"]
    p2 = dict(p1, v=p2["v"], s0=p2["s0"])
    o1, S1 = run(oracle.recurrent, p1)
    o2, S2 = run(oracle.recurrent, p2)
    om, Sm = run(oracle.recurrent, mix)
    assert relerr(om, a * o1 + b * o2) <= 1e-12
    assert relerr(Sm, a * S1 + b * S2) <= 1e-12


def test_selection_matches_full_run():
    p = rand_problem(22, B=2, T=17, H=2, HV=4)
    o, S = run(oracle.recurrent, p)
    sel = [5, 0, 7]
    os_, Ss = run(oracle.recurrent, p, sel=sel)
    for i, s in enumerate(sel):
        b, hv = divmod(s, 4)
        assert np.array_equal(os_[i], o[b, :, hv])
        assert np.array_equal(Ss[i], S[b, hv])


def test_empty_sequence():
    p = rand_problem(23, T=0)
    o, S = run(oracle.recurrent, p)
    assert o.shape == (1, 0, 4, 12)
    assert np.array_equal(S, p["s0"])
    o, S = run(oracle.chunkwise, p, chunk_size=16)
    assert np.array_equal(S, p["s0"])


def test_bf16_inputs_are_read_exactly():
    """bf16 q/k/v are widened exactly: the run equals one on the same values in float64."""
    w = gin.shrink(gin.WORKLOADS["gdn_t4096_h12"], T=40, H=2, HV=2, K=16, V=16)
    x = gin.make_inputs(w)
    o1, S1 = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], None)
    o2, S2 = oracle.recurrent(x["q"].double(), x["k"].double(), x["v"].double(),
                              x["g"].double(), x["beta"].double(), None)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


def test_workload_shapes_and_chunk_form():
    """Every named workload, shrunk in T and heads, keeps the chunk form equal
    to the recurrence with its own C, dtype, gate and state."""
    for name, w in gin.WORKLOADS.items():
        small = gin.shrink(w, B=min(w.B, 2), T=min(w.T, 3 * w.C + 5), H=min(w.H, 2),
                           HV=min(w.HV, 2 * min(w.H, 2) if w.HV > w.H else min(w.H, 2)),
                           K=min(w.K, 32), V=min(w.V, 24))
        x = gin.make_inputs(small)
        o_r, s_r = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["s0"],
                                    scale=small.scale)
        o_c, s_c = oracle.chunkwise(x["q"], x["k"], x["v"], x["g"], x["beta"], x["s0"],
                                    scale=small.scale, chunk_size=small.C)
        assert relerr(o_c, o_r) <= 1e-10, name
        assert relerr(s_c, s_r) <= 1e-10, name
        assert np.all(np.isfinite(o_r)), name


# ---------------------------------------------------------------- planted mistakes
def _pin_battery(recurrent):
    """Run the recurrence-facing pins against `recurrent`; return the names that fail."""
    failed = []
    p = rand_problem(30, T=21, K=8, V=8, H=2, HV=4, gate_mode=1)
    o_ref, s_ref = run(oracle.chunkwise, p, chunk_size=4)
    o, s = run(recurrent, p)
    if relerr(o, o_ref) > 1e-10 or relerr(s, s_ref) > 1e-10:
        failed.append("chunk form")
    pb = rand_problem(31, T=5, K=8, V=8, H=1, HV=2, gate_mode=0)
    o_b, s_b = run(oracle.bruteforce, pb)
    o, s = run(recurrent, pb)
    if relerr(o, o_b) > 1e-12 or relerr(s, s_b) > 1e-12:
        failed.append("brute force")
    ph = _hand(q=[[[[1, 1]], [[0, 1]]]], k=[[[[1, 0]], [[0.6, 0.8]]]],
               v=[[[[3, 4]], [[1, 0]]]], g=[[[math.log(0.5)], [0.0]]],
               beta=[[[0.5], [1.0]]], s0=[[[[1, 0], [0, 2]]]])
    o, _ = run(recurrent, ph, scale=1.0, use_qk_l2norm=False)
    if np.max(np.abs(o[0, :, 0] - np.array([[1.75, 3.0], [-0.04, -0.6]]))) > 1e-14:
        failed.append("hand-worked")
    return failed


def test_faithful_oracle_passes_battery():
    assert _pin_battery(oracle.recurrent) == []


@pytest.mark.parametrize("mutation", range(1, 10))
def test_planted_mistakes(mutation):
    """Each planted mistake in the recurrence fails at least one pin."""
    mutant = lambda *a, **kw: oracle.recurrent(*a, mutation=mutation, **kw)
    assert _pin_battery(mutant), f"mutation {mutation} was not caught"


# ---------------------------------------------------------------- regression fixtures
@pytest.mark.parametrize("name", ["oracle_gdn_small", "oracle_kda_gqa_small",
                                  "oracle_long_state_small"])
def test_golden_regression(name):
    """The oracle still reproduces the fixtures written by tests/golden/make_golden.py."""
    import importlib.util
    import os
    spec = importlib.util.spec_from_file_location(
        "make_golden", os.path.join(os.path.dirname(__file__), "golden", "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    o_ref, S_ref = mg.read(name)
    _, o, S = mg.compute(name)
    assert np.max(np.abs(o - o_ref)) <= 1e-13
    assert np.max(np.abs(S - S_ref)) <= 1e-13
