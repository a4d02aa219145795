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
//                        lower-triangular inverse X = M^-1 (substitution on the
//                        unit columns), W = X (exp(G) k) and U = X v, and the
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
  // X = M^-1 by forward substitution on the unit columns, one column per thread.
  for (int col = tid; col < C; col += kThreads) {
    for (int i = 0; i < C; ++i) {
      float acc = (i == col) ? 1.f : 0.f;
      for (int m = col; m < i; ++m) acc = fmaf(-Lm[i * C + m], Aq[m * C + col], acc);
      Aq[i * C + col] = acc;
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

// State kernel: per chunk three phases over the CTA's kVt = 32 value columns
// (lane = column j; warp w of 8 takes rows i = w + 8 m of the chunk and
// channels c = w + 8 m of the state, accumulating in registers):
//   r  = U - W S            rows i
//   o  = QE S + A_qk r      rows i
//   S' = GM S + KD^T r      channels c
// Each phase streams its per-chunk matrix through shared memory in tiles of
// 32 channels (or 32 chunk rows for KD^T and A_qk), staged with coalesced
// loads, so every term of the inner products comes from shared memory (the
// matrix element is a broadcast within the warp). S is padded to a multiple
// of 32 channels and r to a multiple of 32 rows, with zeros.
constexpr int kSt = 32;                 // channel / row tile of the state kernel
constexpr int kRowAcc = 128 / 8;        // rows per thread (C <= 128)
constexpr int kChAcc = 256 / 8;         // channels per thread (K <= 256)

__host__ __device__ inline int round32(int x) { return (x + 31) & ~31; }

// Shared memory: S [Kp][kVt], r [Cp][kVt], exp(G_last) [Kp], one tile of
// max(Cp, Kp) x 32 floats.
size_t state_smem_bytes(const Problem& p) {
  const size_t Kp = round32(p.K), Cp = round32(p.C);
  return sizeof(float) * (Kp * kVt + Cp * kVt + Kp + (Kp > Cp ? Kp : Cp) * kSt);
}

__global__ void __launch_bounds__(kThreads) general_state_kernel(Args a) {
  extern __shared__ float sm[];
  const Problem& p = a.p;
  const int vt = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
  const int C = p.C, K = p.K, V = p.V;
  const int Kp = round32(K), Cp = round32(C);
  const int v0 = vt * kVt;
  const int vw = min(kVt, V - v0);
  const int tid = threadIdx.x, w = tid >> 5, j = tid & 31;

  float* S = sm;                  // [Kp][kVt]
  float* r = S + Kp * kVt;        // [Cp][kVt]
  float* gm = r + Cp * kVt;       // [Kp]
  float* tile = gm + Kp;          // [max(Cp, Kp)][kSt] or [kSt][Kp]

  const long seq = (long)b * p.HV + hv;
  for (int idx = tid; idx < Kp * kVt; idx += kThreads) {
    const int c = idx / kVt, jj = idx % kVt;
    S[idx] = (p.s0 && c < K && jj < vw) ? p.s0[(seq * K + c) * V + v0 + jj] : 0.f;
  }
  for (int idx = tid; idx < Cp * kVt; idx += kThreads) r[idx] = 0.f;

  for (int n = 0; n < p.N; ++n) {
    const long chunk = seq * p.N + n;
    const float* W = a.s.W + chunk * (long)C * K;
    const float* QE = a.s.QE + chunk * (long)C * K;
    const float* KD = a.s.KD + chunk * (long)C * K;
    const float* U = a.s.U + chunk * (long)C * V;
    const float* AQ = a.s.AQ + chunk * (long)C * C;
    __syncthreads();   // the previous chunk's S and r are written
    for (int c = tid; c < Kp; c += kThreads)
      gm[c] = c < K ? a.s.GM[chunk * K + (p.gate_mode ? c : 0)] : 0.f;
    // [C rows][32 columns c0 ..] of a row-major [C][ld] matrix into the tile.
    // (unrolled, so that a thread has several loads in flight: one at a time
    // each would wait for its own round trip to L2)
    auto stage_rows = [&](const float* M, int ld, int cols, int c0) {
      __syncthreads();   // the tile's previous readers are done
#pragma unroll 8
      for (int idx = tid; idx < C * kSt; idx += kThreads) {
        const int i = idx >> 5, cc = idx & 31;
        tile[idx] = c0 + cc < cols ? M[(long)i * ld + c0 + cc] : 0.f;
      }
      __syncthreads();
    };
    // ---- r = U - W S
    float acc[kRowAcc];
#pragma unroll
    for (int m = 0; m < kRowAcc; ++m) {
      const int i = w + 8 * m;
      acc[m] = (i < C && j < vw && !p.zero_u) ? U[(long)i * V + v0 + j] : 0.f;
    }
    for (int c0 = 0; c0 < K; c0 += kSt) {
      stage_rows(W, K, K, c0);
#pragma unroll 4
      for (int cc = 0; cc < kSt; ++cc) {
        const float sv = S[(c0 + cc) * kVt + j];
#pragma unroll
        for (int m = 0; m < kRowAcc; ++m)
          if (w + 8 * m < C) acc[m] = fmaf(-tile[(w + 8 * m) * kSt + cc], sv, acc[m]);
      }
    }
#pragma unroll
    for (int m = 0; m < kRowAcc; ++m)
      if (w + 8 * m < C) r[(w + 8 * m) * kVt + j] = acc[m];
    // ---- o = QE S + A_qk r
#pragma unroll
    for (int m = 0; m < kRowAcc; ++m) acc[m] = 0.f;
    for (int c0 = 0; c0 < K; c0 += kSt) {
      stage_rows(QE, K, K, c0);
#pragma unroll 4
      for (int cc = 0; cc < kSt; ++cc) {
        const float sv = S[(c0 + cc) * kVt + j];
#pragma unroll
        for (int m = 0; m < kRowAcc; ++m)
          if (w + 8 * m < C) acc[m] = fmaf(tile[(w + 8 * m) * kSt + cc], sv, acc[m]);
      }
    }
    for (int m0 = 0; m0 < C; m0 += kSt) {
      stage_rows(AQ, C, C, m0);   // (the barrier in it also makes r visible)
#pragma unroll 4
      for (int mm = 0; mm < kSt; ++mm) {
        const float rv = r[(m0 + mm) * kVt + j];
#pragma unroll
        for (int m = 0; m < kRowAcc; ++m)
          if (w + 8 * m < C) acc[m] = fmaf(tile[(w + 8 * m) * kSt + mm], rv, acc[m]);
      }
    }
#pragma unroll
    for (int m = 0; m < kRowAcc; ++m) {
      const int i = w + 8 * m, t = n * C + i;
      if (i >= C || j >= vw || t >= p.T) continue;
      const long off = (((long)b * p.T + t) * p.HV + hv) * V + v0 + j;
      if (p.out_bf16)
        static_cast<__nv_bfloat16*>(p.out)[off] = __float2bfloat16_rn(acc[m]);
      else
        static_cast<float*>(p.out)[off] = acc[m];
    }
    // ---- S' = GM S + KD^T r: the tile holds KD rows m0 .. m0 + 31, all K channels.
    float acc2[kChAcc];
#pragma unroll
    for (int m = 0; m < kChAcc; ++m) {
      const int c = w + 8 * m;
      acc2[m] = c < K ? gm[c] * S[c * kVt + j] : 0.f;
    }
    for (int m0 = 0; m0 < C; m0 += kSt) {
      __syncthreads();
#pragma unroll 8
      for (int idx = tid; idx < kSt * K; idx += kThreads) {
        const int mm = idx / K, c = idx % K;
        tile[idx] = m0 + mm < C ? KD[(long)(m0 + mm) * K + c] : 0.f;
      }
      __syncthreads();
#pragma unroll 4
      for (int mm = 0; mm < kSt; ++mm) {
        const float rv = r[(m0 + mm) * kVt + j];
#pragma unroll
        for (int m = 0; m < kChAcc; ++m)
          if (w + 8 * m < K) acc2[m] = fmaf(tile[mm * K + w + 8 * m], rv, acc2[m]);
      }
    }
    __syncthreads();   // every read of this chunk's S is done
#pragma unroll
    for (int m = 0; m < kChAcc; ++m)
      if (w + 8 * m < K) S[(w + 8 * m) * kVt + j] = acc2[m];
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
