// gdr_general.cu -- general chunkwise gated delta rule forward on CUDA cores (fp32).
//
// Two kernels, for any head dims K, V <= 128 (K + V <= 256), chunk sizes
// 16/32/64 (and 128 for K, V <= 64), fp32 or bf16 inputs, both gate kinds and
// the ungated mode (g == NULL reads as zero). All arithmetic is fp32,
// which is what the fp32-input accuracy bound needs; the bf16 K = V = 128,
// C = 64 workloads take the tensor-core path instead (gdr_tc.cu).
//
//  general_prep_kernel   one CTA per chunk (n, hv, b): L2 norm and scale of q/k,
//                        gate cumsum G, decayed dots A_kk / A_qk, the unit
//                        lower-triangular solve for W = M^-1 (exp(G) k) and
//                        U = M^-1 v, and the per-chunk factors the state pass
//                        needs ("分块并行计算（Chunkwise）" notes, section
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

size_t prep_smem_bytes(const Problem& p) {
  const int KP = p.K + 1, VP = p.V + 1, C = p.C;
  const int GP = p.gate_mode ? KP : 1;
  return sizeof(float) * ((size_t)2 * C * KP + (size_t)C * VP + (size_t)C * GP +
                          (size_t)C * C + 3 * (size_t)C);
}

__global__ void __launch_bounds__(kThreads) general_prep_kernel(Args a) {
  extern __shared__ float sm[];
  const Problem& p = a.p;
  const int n = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
  const int C = p.C, K = p.K, V = p.V;
  const int KP = K + 1, VP = V + 1;
  const int KG = p.gate_mode ? K : 1, GP = p.gate_mode ? KP : 1;
  const int h = hv / (p.HV / p.H);
  const int t0 = n * C;
  const int tid = threadIdx.x;
  const long chunk = ((long)b * p.HV + hv) * p.N + n;

  float* qs = sm;             // [C][KP]  scaled normalised q
  float* ks = qs + C * KP;    // [C][KP]  normalised k, later the W right-hand side / solution
  float* vs = ks + C * KP;    // [C][VP]  v, later U
  float* G = vs + C * VP;     // [C][GP]  in-chunk cumsum of g
  float* L = G + C * GP;      // [C][C]   strictly lower part of M
  float* bb = L + C * C;      // [C]      beta
  float* nq = bb + C;         // [C]      scale / ||q||
  float* nk = nq + C;         // [C]      1 / ||k||

  for (int idx = tid; idx < C * K; idx += kThreads) {
    const int i = idx / K, c = idx % K, t = t0 + i;
    float qv = 0.f, kv = 0.f;
    if (t < p.T) {
      const long off = (((long)b * p.T + t) * p.H + h) * K + c;
      qv = ld_in(p.q, off, p.in_bf16);
      kv = ld_in(p.k, off, p.in_bf16);
    }
    qs[i * KP + c] = qv;
    ks[i * KP + c] = kv;
  }
  for (int idx = tid; idx < C * V; idx += kThreads) {
    const int i = idx / V, c = idx % V, t = t0 + i;
    vs[i * VP + c] = (t < p.T) ? ld_in(p.v, (((long)b * p.T + t) * p.HV + hv) * V + c, p.in_bf16)
                               : 0.f;
  }
  for (int idx = tid; idx < C * KG; idx += kThreads) {
    const int i = idx / KG, c = idx % KG, t = t0 + i;
    G[i * GP + c] = (p.g && t < p.T) ? p.g[(((long)b * p.T + t) * p.HV + hv) * KG + c] : 0.f;
  }
  for (int i = tid; i < C; i += kThreads) {
    const int t = t0 + i;
    // SSD: beta = 1 everywhere (padded rows carry k = v = 0).
    bb[i] = p.ssd ? 1.f : (t < p.T) ? p.beta[((long)b * p.T + t) * p.HV + hv] : 0.f;
  }
  __syncthreads();

  // L2 norms (x / sqrt(sum x^2 + 1e-6)), one warp per row.
  const int warp = tid >> 5, lane = tid & 31;
  for (int i = warp; i < C; i += kThreads / 32) {
    float sq = 0.f, sk = 0.f;
    for (int c = lane; c < K; c += 32) {
      sq += qs[i * KP + c] * qs[i * KP + c];
      sk += ks[i * KP + c] * ks[i * KP + c];
    }
    for (int o = 16; o > 0; o >>= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    if (lane == 0) {
      nq[i] = p.use_l2 ? p.scale / sqrtf(sq + 1e-6f) : p.scale;
      nk[i] = p.use_l2 ? 1.f / sqrtf(sk + 1e-6f) : 1.f;
    }
  }
  // Gate cumsum within the chunk, per channel.
  __syncthreads();
  for (int c = tid; c < KG; c += kThreads) {
    float acc = 0.f;
    for (int i = 0; i < C; ++i) {
      acc += G[i * GP + c];
      G[i * GP + c] = acc;
    }
  }
  for (int idx = tid; idx < C * K; idx += kThreads) {
    const int i = idx / K, c = idx % K;
    qs[i * KP + c] *= nq[i];
    ks[i * KP + c] *= nk[i];
  }
  __syncthreads();

  // Decayed dots. A_kk feeds M = I + tril(A_kk * beta_j, -1); A_qk keeps its
  // diagonal and carries beta on its columns (listing naive_chunk_kda).
  float* AQ = a.s.AQ + chunk * (long)C * C;
  for (int idx = tid; idx < C * C; idx += kThreads) {
    const int i = idx / C, j = idx % C;
    float akk = 0.f, aqk = 0.f;
    if (j <= i) {
      if (p.gate_mode == 0) {
        float dq = 0.f, dk = 0.f;
        for (int c = 0; c < K; ++c) {
          const float kj = ks[j * KP + c];
          dq = fmaf(qs[i * KP + c], kj, dq);
          dk = fmaf(ks[i * KP + c], kj, dk);
        }
        const float e = expf(G[i] - G[j]);
        aqk = dq * e;
        akk = dk * e;
      } else {
        for (int c = 0; c < K; ++c) {
          const float e = expf(G[i * GP + c] - G[j * GP + c]) * ks[j * KP + c];
          aqk = fmaf(qs[i * KP + c], e, aqk);
          akk = fmaf(ks[i * KP + c], e, akk);
        }
      }
    }
    L[idx] = (j < i && !p.ssd) ? akk * bb[j] : 0.f;   // SSD: no erase, M = I
    AQ[idx] = (j <= i) ? aqk * bb[j] : 0.f;
  }

  // Per-chunk factors of the state pass.
  float* QE = a.s.QE + chunk * (long)C * K;
  float* KD = a.s.KD + chunk * (long)C * K;
  for (int idx = tid; idx < C * K; idx += kThreads) {
    const int i = idx / K, c = idx % K;
    const int gc = p.gate_mode ? c : 0;
    const float gi = G[i * GP + gc], gl = G[(C - 1) * GP + gc];
    QE[idx] = qs[i * KP + c] * expf(gi);
    KD[idx] = ks[i * KP + c] * expf(gl - gi) * bb[i];
  }
  for (int c = tid; c < KG; c += kThreads) a.s.GM[chunk * K + c] = expf(G[(C - 1) * GP + c]);
  __syncthreads();
  // Right-hand side of W: exp(G) * k_hat, in place.
  for (int idx = tid; idx < C * K; idx += kThreads) {
    const int i = idx / K, c = idx % K;
    ks[i * KP + c] *= expf(G[i * GP + (p.gate_mode ? c : 0)]);
  }
  __syncthreads();

  // Forward substitution, one right-hand-side column per thread, in place.
  for (int col = tid; col < K + V; col += kThreads) {
    float* x = (col < K) ? ks + col : vs + (col - K);
    const int st = (col < K) ? KP : VP;
    for (int i = 1; i < C; ++i) {
      float a0 = x[i * st], a1 = 0.f, a2 = 0.f, a3 = 0.f;
      const float* Li = L + i * C;
      int m = 0;
      for (; m + 3 < i; m += 4) {
        a0 = fmaf(-Li[m], x[m * st], a0);
        a1 = fmaf(-Li[m + 1], x[(m + 1) * st], a1);
        a2 = fmaf(-Li[m + 2], x[(m + 2) * st], a2);
        a3 = fmaf(-Li[m + 3], x[(m + 3) * st], a3);
      }
      for (; m < i; ++m) a0 = fmaf(-Li[m], x[m * st], a0);
      x[i * st] = (a0 + a1) + (a2 + a3);
    }
  }
  __syncthreads();
  float* W = a.s.W + chunk * (long)C * K;
  float* U = a.s.U + chunk * (long)C * V;
  for (int idx = tid; idx < C * K; idx += kThreads)
    W[idx] = p.ssd ? 0.f : ks[(idx / K) * KP + idx % K];   // SSD: r = U - W S = v
  for (int idx = tid; idx < C * V; idx += kThreads) U[idx] = vs[(idx / V) * VP + idx % V];
}

size_t state_smem_bytes(const Problem& p) {
  const int KP = p.K + 1, C = p.C;
  return sizeof(float) * ((size_t)p.K * kVt * 2 + (size_t)C * kVt + 3 * (size_t)C * KP +
                          (size_t)C * C + (size_t)p.K);
}

__global__ void __launch_bounds__(kThreads) general_state_kernel(Args a) {
  extern __shared__ float sm[];
  const Problem& p = a.p;
  const int vt = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
  const int C = p.C, K = p.K, V = p.V, KP = K + 1;
  const int KG = p.gate_mode ? K : 1;
  const int v0 = vt * kVt;
  const int vw = min(kVt, V - v0);
  const int tid = threadIdx.x;

  float* S = sm;                  // [K][kVt]
  float* S2 = S + K * kVt;        // [K][kVt] next state
  float* r = S2 + K * kVt;        // [C][kVt]
  float* Ws = r + C * kVt;        // [C][KP]
  float* QEs = Ws + C * KP;       // [C][KP]
  float* KDs = QEs + C * KP;      // [C][KP]
  float* Aq = KDs + C * KP;       // [C][C]
  float* gm = Aq + C * C;         // [K]

  const long seq = (long)b * p.HV + hv;
  for (int idx = tid; idx < K * kVt; idx += kThreads) {
    const int c = idx / kVt, j = idx % kVt;
    S[idx] = (p.s0 && j < vw) ? p.s0[(seq * K + c) * V + v0 + j] : 0.f;
  }

  for (int n = 0; n < p.N; ++n) {
    const long chunk = seq * p.N + n;
    const float* W = a.s.W + chunk * (long)C * K;
    const float* QE = a.s.QE + chunk * (long)C * K;
    const float* KD = a.s.KD + chunk * (long)C * K;
    const float* U = a.s.U + chunk * (long)C * V;
    const float* AQ = a.s.AQ + chunk * (long)C * C;
    __syncthreads();
    for (int idx = tid; idx < C * K; idx += kThreads) {
      const int i = idx / K, c = idx % K;
      Ws[i * KP + c] = W[idx];
      QEs[i * KP + c] = QE[idx];
      KDs[i * KP + c] = KD[idx];
    }
    for (int idx = tid; idx < C * C; idx += kThreads) Aq[idx] = AQ[idx];
    for (int c = tid; c < K; c += kThreads) gm[c] = a.s.GM[chunk * K + (p.gate_mode ? c : 0)];
    __syncthreads();
    // r = U - W S
    for (int idx = tid; idx < C * kVt; idx += kThreads) {
      const int i = idx / kVt, j = idx % kVt;
      float acc = (j < vw) ? U[i * V + v0 + j] : 0.f;
      for (int c = 0; c < K; ++c) acc = fmaf(-Ws[i * KP + c], S[c * kVt + j], acc);
      r[idx] = acc;
    }
    __syncthreads();
    // o = (q exp(G)) S + A_qk r, and the next state into S2.
    for (int idx = tid; idx < C * kVt; idx += kThreads) {
      const int i = idx / kVt, j = idx % kVt;
      const int t = n * C + i;
      if (j >= vw || t >= p.T) continue;
      float acc = 0.f;
      for (int c = 0; c < K; ++c) acc = fmaf(QEs[i * KP + c], S[c * kVt + j], acc);
      for (int m = 0; m <= i; ++m) acc = fmaf(Aq[i * C + m], r[m * kVt + j], acc);
      const long off = (((long)b * p.T + t) * p.HV + hv) * V + v0 + j;
      if (p.out_bf16)
        static_cast<__nv_bfloat16*>(p.out)[off] = __float2bfloat16_rn(acc);
      else
        static_cast<float*>(p.out)[off] = acc;
    }
    for (int idx = tid; idx < K * kVt; idx += kThreads) {
      const int c = idx / kVt, j = idx % kVt;
      float acc = gm[c] * S[idx];
      for (int m = 0; m < C; ++m) acc = fmaf(KDs[m * KP + c], r[m * kVt + j], acc);
      S2[idx] = acc;
    }
    __syncthreads();
    for (int idx = tid; idx < K * kVt; idx += kThreads) S[idx] = S2[idx];
  }
  __syncthreads();
  (void)KG;
  if (p.sT) {
    for (int idx = tid; idx < K * kVt; idx += kThreads) {
      const int c = idx / kVt, j = idx % kVt;
      if (j < vw) p.sT[(seq * K + c) * V + v0 + j] = S[idx];
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
