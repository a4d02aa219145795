// gdr_general.cu -- general chunkwise gated delta rule forward on CUDA cores (fp32).
//
// Two kernels, for head dims K, V <= 256 and chunk sizes 16/32/64/128, fp32
// or bf16 inputs, both gate kinds and the ungated mode (g == NULL reads as
// zero). The chunk kernel streams the head dims through shared memory in tiles
// of 32 channels, so its footprint depends on C only. All arithmetic is fp32,
// which is what the fp32-input accuracy bound needs; the bf16 K = V = 128,
// C = 64 workloads take the tensor-core path instead (gdr_tc.cu).
//
//  general_prep_kernel   one CTA per chunk (n, hv, b): L2 norm and scale of q/k,
//                        gate cumsum G, decayed dots A_kk / A_qk, the unit
//                        lower-triangular inverse X = M^-1 (blocked: 16 x 16
//                        diagonal blocks by substitution, the rest by doubling),
//                        W = X (exp(G) k) and U = X v, and the
//                        per-chunk factors the state pass needs ("分块并行计算（Chunkwise）" notes, section
//                        "chunk 内的 cumsum 与下三角解" and listing naive_chunk_kda).
//  general_state_kernel  one CTA per (V tile, hv, b), serial over chunks: the
//                        inter-chunk loop r = U - W S, o = (q exp(G)) S + A_qk r,
//                        S = exp(G_last) S + (exp(G_last - G) k)^T (beta r)
//                        (same notes, listing of the inter-chunk loop).
//
// Padding: tokens t >= T read as q = k = v = g = beta = 0 (the zero padding of
// "DeltaNet chunk kernel optimization", "Pad to chunk boundary"); their rows
// are never stored.
#include "gdr_internal.cuh"

namespace gdr {
namespace {

constexpr int kThreads = 256;
constexpr int kVt = 32;  // value columns per state CTA

// Workspace arrays (fp32), one slab per chunk (b, hv, n), chunk index
// ((b * HV + hv) * N + n):
//   W  [C][K]  M^-1 (exp(G) k_hat)
//   U  [C][V]  M^-1 v
//   QE [C][K]  scale q_hat exp(G)
//   KD [C][K]  beta_i k_hat exp(G_last - G_i)
//   AQ [C][C]  A_qk with beta on its columns, zero above the diagonal
//   GM [K]     exp(G_last) per channel (entry 0 only for a scalar gate)
struct Slabs {
  float* W;
  float* U;
  float* QE;
  float* KD;
  float* AQ;
  float* GM;
};

struct Sizes {
  size_t w, u, aq, gm, nchunks;
};

Sizes slab_sizes(const Problem& p) {
  Sizes s;
  s.nchunks = (size_t)p.B * p.HV * p.N;
  s.w = (size_t)p.C * p.K;
  s.u = (size_t)p.C * p.V;
  s.aq = (size_t)p.C * p.C;
  s.gm = (size_t)p.K;
  return s;
}

Slabs carve(const Problem& p, void* ws) {
  Sizes s = slab_sizes(p);
  char* base = static_cast<char*>(ws);
  Slabs out;
  out.W = reinterpret_cast<float*>(base);
  base += align_up(s.nchunks * s.w * sizeof(float));
  out.U = reinterpret_cast<float*>(base);
  base += align_up(s.nchunks * s.u * sizeof(float));
  out.QE = reinterpret_cast<float*>(base);
  base += align_up(s.nchunks * s.w * sizeof(float));
  out.KD = reinterpret_cast<float*>(base);
  base += align_up(s.nchunks * s.w * sizeof(float));
  out.AQ = reinterpret_cast<float*>(base);
  base += align_up(s.nchunks * s.aq * sizeof(float));
  out.GM = reinterpret_cast<float*>(base);
  return out;
}

__device__ __forceinline__ float ld_in(const void* p, long i, int bf16) {
  if (bf16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  return static_cast<const float*>(p)[i];
}

struct Args {
  Problem p;
  Slabs s;
};

constexpr int kTk = 32;  // channel tile (keys or values) of the chunk kernel

// Shared memory of the chunk kernel depends on C only: the head dims are
// streamed in tiles of kTk channels.
size_t prep_smem_bytes(const Problem& p) {
  const int C = p.C;
  return sizeof(float) * ((size_t)2 * C * C + (size_t)3 * C * (kTk + 1) + (size_t)4 * C);
}

// Loads channels [c0, c0 + tw) of chunk rows [t0, t0 + C) of a [B, T, heads, D]
// tensor into t[C][kTk + 1]; rows past T and columns past tw read as zero.
__device__ __forceinline__ void load_tile(float* t, const void* src, int bf16, const Problem& p,
                                          int b, int head, int heads, int D, int t0, int c0,
                                          int tw) {
  const int C = p.C;
  for (int idx = threadIdx.x; idx < C * kTk; idx += kThreads) {
    const int i = idx / kTk, c = idx % kTk, tt = t0 + i;
    t[i * (kTk + 1) + c] = (tt < p.T && c < tw)
        ? ld_in(src, (((long)b * p.T + tt) * heads + head) * D + c0 + c, bf16) : 0.f;
  }
}

// Per-key gate: channels [c0, c0 + tw) of g for the chunk, cumulated over the
// chunk rows (G), into t[C][kTk + 1]. g == NULL (ungated) reads as zero.
__device__ __forceinline__ void load_gate_tile(float* t, const Problem& p, int b, int hv, int t0,
                                               int c0, int tw) {
  const int C = p.C;
  for (int idx = threadIdx.x; idx < C * kTk; idx += kThreads) {
    const int i = idx / kTk, c = idx % kTk, tt = t0 + i;
    t[i * (kTk + 1) + c] = (p.g && tt < p.T && c < tw)
        ? p.g[(((long)b * p.T + tt) * p.HV + hv) * p.K + c0 + c] : 0.f;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < kTk; c += kThreads) {
    float acc = 0.f;
    for (int i = 0; i < C; ++i) {
      acc += t[i * (kTk + 1) + c];
      t[i * (kTk + 1) + c] = acc;
    }
  }
}

__global__ void __launch_bounds__(kThreads) general_prep_kernel(Args a) {
  extern __shared__ float sm[];
  const Problem& p = a.p;
  const int n = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
  const int C = p.C, K = p.K, V = p.V, TP = kTk + 1;
  const int h = hv / (p.HV / p.H);
  const int t0 = n * C;
  const int tid = threadIdx.x;
  const long chunk = ((long)b * p.HV + hv) * p.N + n;

  float* Aq = sm;              // [C][C] q.k dots, later X = M^-1
  float* Lm = Aq + C * C;      // [C][C] k.k dots, later the strictly lower part of M
  float* tq = Lm + C * C;      // [C][TP] q tile, later the W right-hand side
  float* tk = tq + C * TP;     // [C][TP] k tile, later the v tile
  float* tg = tk + C * TP;     // [C][TP] per-key gate cumsum of the tile
  float* Gs = tg + C * TP;     // [C] scalar-gate cumsum
  float* bb = Gs + C;          // [C] beta
  float* nq = bb + C;          // [C] sum q^2, then scale / ||q||
  float* nk = nq + C;          // [C] sum k^2, then 1 / ||k||

  for (int idx = tid; idx < C * C; idx += kThreads) Aq[idx] = Lm[idx] = 0.f;
  for (int i = tid; i < C; i += kThreads) {
    const int t = t0 + i;
    // SSD: beta = 1 everywhere (padded rows carry k = v = 0).
    bb[i] = p.ssd ? 1.f : (t < p.T) ? p.beta[((long)b * p.T + t) * p.HV + hv] : 0.f;
    nq[i] = nk[i] = 0.f;
  }
  if (p.gate_mode == 0 && tid == 0) {
    float acc = 0.f;
    for (int i = 0; i < C; ++i) {
      const int t = t0 + i;
      acc += (p.g && t < p.T) ? p.g[((long)b * p.T + t) * p.HV + hv] : 0.f;
      Gs[i] = acc;
    }
  }

  // Raw dots and squared norms, accumulated over channel tiles. The per-key
  // decay sits inside the dot; L2 norms and the scalar decay are applied after.
  for (int c0 = 0; c0 < K; c0 += kTk) {
    const int tw = min(kTk, K - c0);
    __syncthreads();
    load_tile(tq, p.q, p.in_bf16, p, b, h, p.H, K, t0, c0, tw);
    load_tile(tk, p.k, p.in_bf16, p, b, h, p.H, K, t0, c0, tw);
    if (p.gate_mode) load_gate_tile(tg, p, b, hv, t0, c0, tw);
    __syncthreads();
    if (tid < 2 * C) {
      const float* row = (tid < C ? tq : tk) + (tid % C) * TP;
      float s2 = 0.f;
      for (int c = 0; c < kTk; ++c) s2 = fmaf(row[c], row[c], s2);
      (tid < C ? nq : nk)[tid % C] += s2;
    }
    for (int idx = tid; idx < C * C; idx += kThreads) {
      const int i = idx / C, j = idx % C;
      if (j > i) continue;
      float dq = 0.f, dk = 0.f;
      if (p.gate_mode == 0) {
        for (int c = 0; c < kTk; ++c) {
          const float kj = tk[j * TP + c];
          dq = fmaf(tq[i * TP + c], kj, dq);
          dk = fmaf(tk[i * TP + c], kj, dk);
        }
      } else {
        for (int c = 0; c < kTk; ++c) {
          const float kj = tk[j * TP + c] * expf(tg[i * TP + c] - tg[j * TP + c]);
          dq = fmaf(tq[i * TP + c], kj, dq);
          dk = fmaf(tk[i * TP + c], kj, dk);
        }
      }
      Aq[idx] += dq;
      Lm[idx] += dk;
    }
  }
  __syncthreads();
  for (int i = tid; i < C; i += kThreads) {
    nq[i] = p.use_l2 ? p.scale / sqrtf(nq[i] + 1e-6f) : p.scale;
    nk[i] = p.use_l2 ? 1.f / sqrtf(nk[i] + 1e-6f) : 1.f;
  }
  __syncthreads();
  // A_qk (beta on its columns, diagonal kept) -> workspace; M's strictly lower
  // part L = tril(A_kk beta_j, -1) in place (listing naive_chunk_kda).
  float* AQ = a.s.AQ + chunk * (long)C * C;
  for (int idx = tid; idx < C * C; idx += kThreads) {
    const int i = idx / C, j = idx % C;
    const float e = (p.gate_mode == 0) ? expf(Gs[i] - Gs[j]) : 1.f;
    const float f = nk[j] * e * bb[j];
    AQ[idx] = (j <= i) ? Aq[idx] * nq[i] * f : 0.f;
    Lm[idx] = (j < i && !p.ssd) ? Lm[idx] * nk[i] * f : 0.f;   // SSD: no erase, M = I
  }
  __syncthreads();
  // X = M^-1, M = I + L (L strictly lower, in Lm), blocked: the 16 x 16
  // diagonal blocks by forward substitution on their unit columns (one column
  // per thread), then the blocks below them by doubling. For adjacent s-blocks
  // J (rows and columns [2 k s, 2 k s + s)) and I (the next s), the inverse of
  // [[M_JJ, 0], [L_IJ, M_II]] has the lower block X_IJ = -X_II (L_IJ X_JJ), both
  // products in fp32 (T = L_IJ X_JJ in the dead q tile).
  for (int idx = tid; idx < C * C; idx += kThreads) Aq[idx] = 0.f;
  __syncthreads();
  for (int col = tid; col < C; col += kThreads) {
    const int o = col & ~15;
    for (int i = col; i < o + 16; ++i) {
      float acc = (i == col) ? 1.f : 0.f;
      for (int m = col; m < i; ++m) acc = fmaf(-Lm[i * C + m], Aq[m * C + col], acc);
      Aq[i * C + col] = acc;
    }
  }
  float* Tm = tq;   // pairs x s x s <= C s / 2 <= C (kTk + 1) floats
  for (int sz = 16; sz < C; sz *= 2) {
    const int pairs = C / (2 * sz), ss = sz * sz;
    __syncthreads();
    for (int idx = tid; idx < pairs * ss; idx += kThreads) {
      const int pr = idx / ss, e = idx % ss, i = e / sz, j = e % sz;
      const int rI = 2 * pr * sz + sz, cJ = 2 * pr * sz;
      float acc = 0.f;
      for (int m = j; m < sz; ++m)   // X_JJ is lower triangular
        acc = fmaf(Lm[(rI + i) * C + cJ + m], Aq[(cJ + m) * C + cJ + j], acc);
      Tm[idx] = acc;
    }
    __syncthreads();
    for (int idx = tid; idx < pairs * ss; idx += kThreads) {
      const int pr = idx / ss, e = idx % ss, i = e / sz, j = e % sz;
      const int rI = 2 * pr * sz + sz, cJ = 2 * pr * sz;
      float acc = 0.f;
      for (int m = 0; m <= i; ++m)   // X_II is lower triangular
        acc = fmaf(Aq[(rI + i) * C + rI + m], Tm[pr * ss + m * sz + j], acc);
      Aq[(rI + i) * C + cJ + j] = -acc;
    }
  }
  // Per-chunk factors of the state pass and W = X (exp(G) k_hat), tile by tile.
  float* W = a.s.W + chunk * (long)C * K;
  float* QE = a.s.QE + chunk * (long)C * K;
  float* KD = a.s.KD + chunk * (long)C * K;
  for (int c0 = 0; c0 < K; c0 += kTk) {
    const int tw = min(kTk, K - c0);
    __syncthreads();
    load_tile(tq, p.q, p.in_bf16, p, b, h, p.H, K, t0, c0, tw);
    load_tile(tk, p.k, p.in_bf16, p, b, h, p.H, K, t0, c0, tw);
    if (p.gate_mode) load_gate_tile(tg, p, b, hv, t0, c0, tw);
    __syncthreads();
    for (int idx = tid; idx < C * kTk; idx += kThreads) {
      const int i = idx / kTk, c = idx % kTk;
      const float gi = p.gate_mode ? tg[i * TP + c] : Gs[i];
      const float gl = p.gate_mode ? tg[(C - 1) * TP + c] : Gs[C - 1];
      const float kh = tk[i * TP + c] * nk[i];
      if (c < tw) {
        QE[(long)i * K + c0 + c] = tq[i * TP + c] * nq[i] * expf(gi);
        KD[(long)i * K + c0 + c] = kh * expf(gl - gi) * bb[i];
        if (i == 0 && (p.gate_mode || c0 + c == 0))
          a.s.GM[chunk * K + c0 + c] = expf(gl);
      }
      tq[i * TP + c] = kh * expf(gi);   // right-hand side of W
    }
    __syncthreads();
    for (int idx = tid; idx < C * tw; idx += kThreads) {
      const int i = idx / tw, c = idx % tw;
      float acc = 0.f;
      for (int m = 0; m <= i; ++m) acc = fmaf(Aq[i * C + m], tq[m * TP + c], acc);
      W[(long)i * K + c0 + c] = p.ssd ? 0.f : acc;   // SSD: r = U - W S = v
    }
  }
  // U = X v, tile by tile.
  float* U = a.s.U + chunk * (long)C * V;
  for (int c0 = 0; c0 < V; c0 += kTk) {
    const int tw = min(kTk, V - c0);
    __syncthreads();
    load_tile(tk, p.v, p.in_bf16, p, b, hv, p.HV, V, t0, c0, tw);
    __syncthreads();
    for (int idx = tid; idx < C * tw; idx += kThreads) {
      const int i = idx / tw, c = idx % tw;
      float acc = 0.f;
      for (int m = 0; m <= i; ++m) acc = fmaf(Aq[i * C + m], tk[m * TP + c], acc);
      U[(long)i * V + c0 + c] = acc;
    }
  }
}

// State kernel: per chunk three phases over the CTA's kVt = 32 value columns,
// each thread accumulating a 4 x 4 block in registers (column group cg =
// tid % 8: columns 4 cg .. 4 cg + 3; row group rg = tid / 8: rows, or state
// channels, 4 rg .. 4 rg + 3, and 4 rg + 128 .. for K > 128):
//   r  = U - W S            rows i of the chunk
//   o  = QE S + A_qk r      rows i
//   S' = GM S + KD^T r      state channels c
// Each phase streams its per-chunk matrix through shared memory in tiles of
// kSt = 64 channels (or 64 chunk rows for KD^T and A_qk), staged with coalesced
// loads (W, QE and A_qk transposed, so that a thread's four rows are one
// 16-byte read); every step of an inner product then takes one 16-byte read
// of each operand for 16 FMAs. S is padded to a multiple of kSt channels and
// r to a multiple of kSt rows, with zeros.
constexpr int kSt = 64;                 // channel / row tile of the state kernel (32 measured 5 % slower)
constexpr int kChPass = 2;              // passes of 128 state channels (K <= 256)
constexpr int kStageRegs = 256 * kSt / 256;   // a thread's share of one tile (K <= 256)

__host__ __device__ inline int round_st(int x) { return (x + kSt - 1) / kSt * kSt; }

// Shared memory: S [Kp][kVt], r [Cp][kVt], exp(G_last) [Kp], and one tile:
// transposed [kSt][Cp + 4] or [kSt][Kp + 4].
size_t state_smem_bytes(const Problem& p) {
  const size_t Kp = round_st(p.K), Cp = round_st(p.C);
  return sizeof(float) * (Kp * kVt + Cp * kVt + Kp + kSt * ((Kp > Cp ? Kp : Cp) + 4));
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

__global__ void __launch_bounds__(kThreads) general_state_kernel(Args a) {
  extern __shared__ float sm[];
  const Problem& p = a.p;
  const int vt = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
  const int C = p.C, K = p.K, V = p.V;
  const int Kp = round_st(K), Cp = round_st(C);
  const int LC = Cp + 4, LK = Kp + 4;     // tile row strides (16-byte multiples)
  const int v0 = vt * kVt;
  const int vw = min(kVt, V - v0);
  const int tid = threadIdx.x, cg = tid & 7, rg = tid >> 3;
  const int j0 = 4 * cg;                  // this thread's first column

  float* S = sm;                  // [Kp][kVt]
  float* r = S + Kp * kVt;        // [Cp][kVt]
  float* gm = r + Cp * kVt;       // [Kp]
  float* tile = gm + Kp;          // [kSt][LC] (transposed rows) or [kSt][LK]

  const long seq = (long)b * p.HV + hv;
  for (int idx = tid; idx < Kp * kVt; idx += kThreads) {
    const int c = idx / kVt, jj = idx % kVt;
    S[idx] = (p.s0 && c < K && jj < vw) ? p.s0[(seq * K + c) * V + v0 + jj] : 0.f;
  }
  for (int idx = tid; idx < Cp * kVt; idx += kThreads) r[idx] = 0.f;
  const int i0 = 4 * rg;                  // this thread's first row (r and o phases)
  const bool rows_ok = i0 < C;            // (C is a multiple of 16)

  // acc += tile^T x X over the kSt staged steps: this thread's 4 rows
  // (tile[cc][i0 ..]) times 4 columns of X (rows x0 + cc of [.][kVt]).
  auto tile_product = [&](float (&acc)[4][4], const float* X, int x0, float sign) {
#pragma unroll 4
    for (int cc = 0; cc < kSt; ++cc) {
      const float4 xv = ld4(X + (x0 + cc) * kVt + j0);
      const float4 tv = ld4(tile + cc * LC + i0);
      const float xs[4] = {xv.x, xv.y, xv.z, xv.w};
      const float ts[4] = {sign * tv.x, sign * tv.y, sign * tv.z, sign * tv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int f = 0; f < 4; ++f) acc[e][f] = fmaf(ts[e], xs[f], acc[e][f]);
    }
  };
  // The chunks' tiles form one sequence of stages: per chunk nK tiles of W,
  // nK of QE, nC of A_qk, nC of KD. The values of stage q + 1 are loaded into
  // registers (a thread's share, at most kStageRegs) while stage q is
  // computed, so that the round trip to L2 or DRAM overlaps the arithmetic.
  const int nK = (K + kSt - 1) / kSt, nC = (C + kSt - 1) / kSt;
  const int per_chunk = 2 * nK + 2 * nC;
  const long nstages = (long)p.N * per_chunk;
  float nxt[kStageRegs];
  // Source of stage q: which matrix, its leading dimension, column count and
  // first column (or first KD row).
  auto load_stage = [&](long q) {
    const long chunk = seq * p.N + q / per_chunk;
    const int s = (int)(q % per_chunk);
    if (s < 2 * nK + nC) {   // W, QE or A_qk columns, read along the row
      const float* M;
      int ld, cols, c0;
      if (s < nK) { M = a.s.W + chunk * (long)C * K; ld = K; cols = K; c0 = kSt * s; }
      else if (s < 2 * nK) { M = a.s.QE + chunk * (long)C * K; ld = K; cols = K; c0 = kSt * (s - nK); }
      else { M = a.s.AQ + chunk * (long)C * C; ld = C; cols = C; c0 = kSt * (s - 2 * nK); }
#pragma unroll
      for (int kk = 0; kk < kStageRegs; ++kk) {
        const int idx = tid + kThreads * kk;
        const int i = idx / kSt, cc = idx % kSt;
        nxt[kk] = (i < C && c0 + cc < cols) ? M[(long)i * ld + c0 + cc] : 0.f;
      }
    } else {                 // KD rows m0 .. m0 + 31, all K channels
      const float* KD = a.s.KD + chunk * (long)C * K;
      const int m0 = kSt * (s - 2 * nK - nC);
#pragma unroll
      for (int kk = 0; kk < kStageRegs; ++kk) {
        const int idx = tid + kThreads * kk;
        const int mm = idx / K, c = idx % K;
        nxt[kk] = (mm < kSt && m0 + mm < C) ? KD[(long)(m0 + mm) * K + c] : 0.f;
      }
    }
  };
  // The loaded values into the tile: W, QE and A_qk transposed ([cc][i]), KD
  // as is ([mm][c], channels K .. Kp + 3 zero).
  auto store_stage = [&](long q) {
    const int s = (int)(q % per_chunk);
    if (s < 2 * nK + nC) {
#pragma unroll
      for (int kk = 0; kk < kStageRegs; ++kk) {
        const int idx = tid + kThreads * kk;
        const int i = idx / kSt, cc = idx % kSt;
        if (i < C) tile[cc * LC + i] = nxt[kk];
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < kStageRegs; ++kk) {
        const int idx = tid + kThreads * kk;
        const int mm = idx / K, c = idx % K;
        if (mm < kSt) tile[mm * LK + c] = nxt[kk];
      }
      for (int idx = tid; idx < kSt * (LK - K); idx += kThreads) {
        const int mm = idx / (LK - K), c = K + idx % (LK - K);
        tile[mm * LK + c] = 0.f;
      }
    }
  };
  float acc[4][4], acc2[kChPass][4][4];
  if (nstages > 0) load_stage(0);
  for (long q = 0; q < nstages; ++q) {
    const int n = (int)(q / per_chunk), s = (int)(q % per_chunk);
    const long chunk = seq * p.N + n;
    __syncthreads();   // the tile's previous readers (and S and r writers) are done
    store_stage(q);
    if (s == 0)
      for (int c = tid; c < Kp; c += kThreads)
        gm[c] = c < K ? a.s.GM[chunk * K + (p.gate_mode ? c : 0)] : 0.f;
    __syncthreads();
    if (q + 1 < nstages) load_stage(q + 1);
    if (s == 0 || s == nK) {
      // r = U - W S starts from U; o = QE S + A_qk r from zero.
      const float* U = a.s.U + chunk * (long)C * V;
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int f = 0; f < 4; ++f)
          acc[e][f] = (s == 0 && rows_ok && j0 + f < vw && !p.zero_u)
                          ? U[(long)(i0 + e) * V + v0 + j0 + f] : 0.f;
    }
    if (s < nK) {
      if (rows_ok) tile_product(acc, S, kSt * s, -1.f);
      if (s == nK - 1 && rows_ok) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          *reinterpret_cast<float4*>(r + (i0 + e) * kVt + j0) =
              make_float4(acc[e][0], acc[e][1], acc[e][2], acc[e][3]);
      }
    } else if (s < 2 * nK) {
      if (rows_ok) tile_product(acc, S, kSt * (s - nK), 1.f);
    } else if (s < 2 * nK + nC) {
      if (rows_ok) tile_product(acc, r, kSt * (s - 2 * nK), 1.f);
      if (s == 2 * nK + nC - 1 && rows_ok) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = n * C + i0 + e;
          if (t >= p.T) continue;
          const long off = (((long)b * p.T + t) * p.HV + hv) * V + v0 + j0;
#pragma unroll
          for (int f = 0; f < 4; ++f) {
            if (j0 + f >= vw) continue;
            if (p.out_bf16)
              static_cast<__nv_bfloat16*>(p.out)[off + f] = __float2bfloat16_rn(acc[e][f]);
            else
              static_cast<float*>(p.out)[off + f] = acc[e][f];
          }
        }
      }
    } else {
      const int m0 = kSt * (s - 2 * nK - nC);
      if (m0 == 0) {
        // S' = GM S + KD^T r: this thread's channels c = 4 rg + 128 q' + e.
#pragma unroll
        for (int qq = 0; qq < kChPass; ++qq)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 4 * rg + 128 * qq + e;
#pragma unroll
            for (int f = 0; f < 4; ++f)
              acc2[qq][e][f] = c < Kp ? gm[c] * S[c * kVt + j0 + f] : 0.f;
          }
      }
#pragma unroll 4
      for (int mm = 0; mm < kSt; ++mm) {
        const float4 rv = ld4(r + (m0 + mm) * kVt + j0);
        const float rs[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
        for (int qq = 0; qq < kChPass; ++qq) {
          const int c = 4 * rg + 128 * qq;
          if (c >= Kp) continue;
          const float4 kv = ld4(tile + mm * LK + c);
          const float ks[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int f = 0; f < 4; ++f) acc2[qq][e][f] = fmaf(ks[e], rs[f], acc2[qq][e][f]);
        }
      }
      if (s == per_chunk - 1) {
        __syncthreads();   // every read of this chunk's S is done
#pragma unroll
        for (int qq = 0; qq < kChPass; ++qq) {
          const int c = 4 * rg + 128 * qq;
          if (c >= Kp) continue;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            *reinterpret_cast<float4*>(S + (c + e) * kVt + j0) =
                make_float4(acc2[qq][e][0], acc2[qq][e][1], acc2[qq][e][2], acc2[qq][e][3]);
        }
      }
    }
  }
  __syncthreads();
  if (p.sT) {
    for (int idx = tid; idx < K * kVt; idx += kThreads) {
      const int c = idx / kVt, jj = idx % kVt;
      if (jj < vw) p.sT[(seq * K + c) * V + v0 + jj] = S[idx];
    }
  }
}

}  // namespace

size_t general_workspace_bytes(const Problem& p) {
  Sizes s = slab_sizes(p);
  return align_up(s.nchunks * s.w * sizeof(float)) * 3 +
         align_up(s.nchunks * s.u * sizeof(float)) +
         align_up(s.nchunks * s.aq * sizeof(float)) +
         align_up(s.nchunks * s.gm * sizeof(float));
}

gdr_status launch_general(const Problem& p, void* ws_body, cudaStream_t stream, int stage) {
  Args a;
  a.p = p;
  a.s = carve(p, ws_body);
  const size_t prep_smem = prep_smem_bytes(p);
  const size_t state_smem = state_smem_bytes(p);
  if (cudaFuncSetAttribute(general_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)prep_smem) != cudaSuccess)
    return GDR_ERR_CUDA;
  if (cudaFuncSetAttribute(general_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)state_smem) != cudaSuccess)
    return GDR_ERR_CUDA;
  if (stage & 1) {
    dim3 g1(p.N, p.HV, p.B);
    general_prep_kernel<<<g1, kThreads, prep_smem, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return GDR_ERR_CUDA;
  }
  if (stage & 2) {
    dim3 g2((p.V + kVt - 1) / kVt, p.HV, p.B);
    general_state_kernel<<<g2, kThreads, state_smem, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return GDR_ERR_CUDA;
  }
  return GDR_OK;
}

}  // namespace gdr
