// gdr_chunk_simt.cu -- CUDA-core producer of the fast-path chunk slabs.
//
// Same outputs as the tcgen05 chunk-local kernel (gdr_chunk_tc.cu), computed
// with fp32 FMAs: it is the reference the tensor-core producer is tested
// against, and the producer used when the tensor-core one is switched off.
// One CTA per chunk (n, hv, b), 256 threads. Per chunk (the "分块并行计算
// （Chunkwise）" notes, section "chunk 内的 cumsum 与下三角解" and listing
// naive_chunk_kda): L2-normalise q and k, cumsum the gate, form the decayed
// dots A_kk / A_qk, solve M = I + tril(A_kk beta, -1) for W and U by forward
// substitution, and write the slab described in gdr_fast.cuh.
#include <cuda_bf16.h>

#include "gdr_fast.cuh"

namespace gdr {
namespace fast {
namespace {

constexpr int THREADS = 256;
constexpr int KP = K + 1;

__device__ __forceinline__ void split_store(__nv_bfloat16* hi, __nv_bfloat16* lo, float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  *hi = h;
  *lo = __float2bfloat16_rn(x - __bfloat162float(h));
}

template <int GATE>
__global__ void __launch_bounds__(THREADS) chunk_simt_kernel(Params p) {
  extern __shared__ float sm[];
  const int n = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
  const int h = hv / (p.HV / p.H);
  const int t0 = n * C;
  const int tid = threadIdx.x;
  constexpr int GP = GATE ? KP : 1;
  float* qs = sm;             // [C][KP]
  float* ks = qs + C * KP;    // [C][KP]
  float* vs = ks + C * KP;    // [C][V + 1]
  float* G = vs + C * (V + 1);
  float* L = G + C * GP;      // [C][C]
  float* bb = L + C * C;
  float* nq = bb + C;
  float* nk = nq + C;
  uint8_t* slab = p.slabs + slab_index(p, b, hv, n) * p.slab_bytes;

  for (int idx = tid; idx < C * K; idx += THREADS) {
    const int i = idx / K, c = idx % K, t = t0 + i;
    float qv = 0.f, kv = 0.f, vv = 0.f;
    if (t < p.T) {
      const size_t off = (((size_t)b * p.T + t) * p.H + h) * K + c;
      qv = __bfloat162float(p.q[off]);
      kv = __bfloat162float(p.k[off]);
      vv = __bfloat162float(p.v[(((size_t)b * p.T + t) * p.HV + hv) * V + c]);
    }
    qs[i * KP + c] = qv;
    ks[i * KP + c] = kv;
    vs[i * (V + 1) + c] = vv;
  }
  for (int idx = tid; idx < C * (GATE ? K : 1); idx += THREADS) {
    const int kg = GATE ? K : 1;
    const int i = idx / kg, c = idx % kg, t = t0 + i;
    G[i * GP + c] = (t < p.T) ? p.g[(((size_t)b * p.T + t) * p.HV + hv) * kg + c] : 0.f;
  }
  for (int i = tid; i < C; i += THREADS) {
    const int t = t0 + i;
    bb[i] = (t < p.T) ? p.beta[((size_t)b * p.T + t) * p.HV + hv] : 0.f;
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  for (int i = warp; i < C; i += THREADS / 32) {
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
      nq[i] = p.use_l2 ? 1.f / sqrtf(sq + 1e-6f) : 1.f;
      nk[i] = p.use_l2 ? 1.f / sqrtf(sk + 1e-6f) : 1.f;
    }
  }
  __syncthreads();
  for (int c = tid; c < (GATE ? K : 1); c += THREADS) {
    float acc = 0.f;
    for (int i = 0; i < C; ++i) {
      acc += G[i * GP + c];
      G[i * GP + c] = acc;
    }
  }
  for (int idx = tid; idx < C * K; idx += THREADS) {
    const int i = idx / K, c = idx % K;
    qs[i * KP + c] *= nq[i] * p.scale;
    ks[i * KP + c] *= nk[i];
  }
  __syncthreads();

  __nv_bfloat16* aq = reinterpret_cast<__nv_bfloat16*>(slab + Slab::AQ2);
  for (int idx = tid; idx < C * C; idx += THREADS) {
    const int i = idx / C, j = idx % C;
    float akk = 0.f, aqk = 0.f;
    if (j <= i) {
      if (GATE == 0) {
        float dq = 0.f, dk = 0.f;
        for (int c = 0; c < K; ++c) {
          dq = fmaf(qs[i * KP + c], ks[j * KP + c], dq);
          dk = fmaf(ks[i * KP + c], ks[j * KP + c], dk);
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
    L[idx] = (j < i) ? akk * bb[j] : 0.f;
    split_store(aq + idx, aq + C * C + idx, (j <= i) ? aqk * bb[j] : 0.f);
  }
  float* vec = reinterpret_cast<float*>(slab + Slab::VEC);
  if (GATE == 0) {
    const float gl = G[(C - 1) * GP];
    for (int i = tid; i < C; i += THREADS) {
      vec[i] = p.scale * nq[i] * expf(G[i * GP]);
      vec[C + i] = bb[i] * nk[i] * expf(gl - G[i * GP]);
    }
    for (int c = tid; c < K; c += THREADS) vec[2 * C + c] = expf(gl);
  } else {
    __nv_bfloat16* qb = reinterpret_cast<__nv_bfloat16*>(slab + Slab::QB2);
    __nv_bfloat16* kb = reinterpret_cast<__nv_bfloat16*>(slab + Slab::KB2);
    for (int idx = tid; idx < C * K; idx += THREADS) {
      const int i = idx / K, c = idx % K;
      const float gi = G[i * GP + c], gl = G[(C - 1) * GP + c];
      split_store(qb + idx, qb + C * K + idx, qs[i * KP + c] * expf(gi));
      split_store(kb + idx, kb + C * K + idx, ks[i * KP + c] * expf(gl - gi) * bb[i]);
    }
    for (int i = tid; i < C; i += THREADS) {
      vec[i] = 1.f;
      vec[C + i] = 1.f;
    }
    for (int c = tid; c < K; c += THREADS) vec[2 * C + c] = expf(G[(C - 1) * GP + c]);
  }
  __syncthreads();
  for (int idx = tid; idx < C * K; idx += THREADS) {
    const int i = idx / K, c = idx % K;
    ks[i * KP + c] *= expf(G[i * GP + (GATE ? c : 0)]);
  }
  __syncthreads();
  for (int col = tid; col < K + V; col += THREADS) {
    float* x = (col < K) ? ks + col : vs + (col - K);
    const int st = (col < K) ? KP : V + 1;
    for (int i = 1; i < C; ++i) {
      float a0 = x[i * st], a1 = 0.f;
      const float* Li = L + i * C;
      int m = 0;
      for (; m + 1 < i; m += 2) {
        a0 = fmaf(-Li[m], x[m * st], a0);
        a1 = fmaf(-Li[m + 1], x[(m + 1) * st], a1);
      }
      if (m < i) a0 = fmaf(-Li[m], x[m * st], a0);
      x[i * st] = a0 + a1;
    }
  }
  __syncthreads();
  __nv_bfloat16* w2 = reinterpret_cast<__nv_bfloat16*>(slab + Slab::W2);
  float* u = reinterpret_cast<float*>(slab + Slab::U);
  for (int idx = tid; idx < C * K; idx += THREADS) {
    const int i = idx / K, c = idx % K;
    split_store(w2 + idx, w2 + C * K + idx, -ks[i * KP + c]);
    u[idx] = vs[i * (V + 1) + c];
  }
}

template <int GATE>
gdr_status launch_simt(const Params& p, cudaStream_t stream) {
  constexpr int GP = GATE ? KP : 1;
  const size_t smem = sizeof(float) * ((size_t)2 * C * KP + (size_t)C * (V + 1) + (size_t)C * GP +
                                       (size_t)C * C + 3 * C);
  auto kern = chunk_simt_kernel<GATE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return GDR_ERR_CUDA;
  dim3 grid(p.N, p.HV, p.B);
  kern<<<grid, THREADS, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

}  // namespace

gdr_status launch_chunk_simt(const Params& p, cudaStream_t stream) {
  return p.gate_mode ? launch_simt<1>(p, stream) : launch_simt<0>(p, stream);
}

}  // namespace fast
}  // namespace gdr
