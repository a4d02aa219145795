// gdr_chunk_tc.cu -- chunk-local kernel of the fast path on tcgen05 tensor cores.
//
// One CTA (4 warps) per chunk (n, hv, b), scalar gate, bf16 inputs, C = 64,
// K = V = 128. It computes, for one chunk of the "分块并行计算（Chunkwise）"
// notes (section "chunk 内的 cumsum 与下三角解", listing naive_chunk_kda):
//   G     = cumsum(g)                                 (in-chunk gate cumsum)
//   P, Q  = k k^T, q k^T       one tcgen05 MMA, A = [k; q] stacked to M = 128
//   A_kk  = P |k_i|^-1 |k_j|^-1 exp(G_i - G_j)        (L2 norm and decay as fp32
//   A_qk  = Q scale |q_i|^-1 |k_j|^-1 exp(G_i - G_j) beta_j   epilogue factors;
//                                                      the bf16 inputs are exact)
//   M     = I + tril(A_kk beta_j, -1),  X = M^-1      (fp32, 16x16 diagonal blocks
//                                                      by substitution, off-diagonal
//                                                      blocks by block products)
//   W     = X diag(exp(G_j) |k_j|^-1) k,  U = X v     two tcgen05 MMAs with A =
//                                                      [X_hi; X_lo] stacked to M = 128
//                                                      and the raw bf16 k / v tile as B
// and writes the slab of gdr_fast.cuh. q, k and v arrive by TMA (128-byte
// swizzle, zero fill past the end of the sequence, which is the zero padding of
// the last chunk); accumulators live in TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "gdr_fast.cuh"

namespace gdr {
namespace fast {
namespace {

constexpr int THREADS = 128;
constexpr uint32_t TMEM_COLS = 256;
constexpr long kWaitLimit = 1L << 24;   // bounded spin: ~tens of ms, then error word
constexpr unsigned int kErrTmaWait = 1u, kErrMmaWait = 2u;

// Shared-memory map (bytes from a 1024-aligned base).
constexpr int OFF_K0 = 0;          // k cols 0-63   (8 KB, SW128)
constexpr int OFF_Q0 = 8192;       // q cols 0-63
constexpr int OFF_K1 = 16384;      // k cols 64-127
constexpr int OFF_Q1 = 24576;      // q cols 64-127
constexpr int OFF_V0 = 32768;      // v cols 0-63
constexpr int OFF_V1 = 40960;      // v cols 64-127
constexpr int OFF_L = 49152;       // L fp32 [64][64]; later XW = [X'hi; X'lo] (M=128, K=64)
constexpr int OFF_X = 65536;       // X fp32 [64][64]; later XU = [Xhi; Xlo]
constexpr int OFF_SMALL = 81920;   // G, nq, nk, beta (4 x 64 fp32)
constexpr int OFF_BAR = 82944;     // mbarriers + TMEM slot
constexpr int SMEM_BYTES = OFF_BAR + 64 + 1024;  // + alignment slack
// After the W / U MMAs complete, [0, 65536) holds the two fp32 exchange tiles.
constexpr int OFF_XCH_W = 0;       // [64][128] fp32
constexpr int OFF_XCH_U = 32768;   // [64][128] fp32

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint32_t swz128(uint32_t off) { return off ^ (((off >> 7) & 7u) << 4); }

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  // tcgen05 shared-memory matrix descriptor, 128-byte swizzle, version 1.
  return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  // kind::f16 instruction descriptor: D f32, A/B bf16, dense.
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, int acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (long i = 0; i < kWaitLimit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}
__device__ __forceinline__ void tma_load4(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                          int c2, int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t pack_bf16(float x, float y) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&h);
}

struct TcArgs {
  Params p;
};

__global__ void __launch_bounds__(THREADS, 2)
    chunk_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, TcArgs args) {
  const Params& p = args.p;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int n = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
  const int h = hv / (p.HV / p.H);
  const int t0 = n * C;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  float* L = reinterpret_cast<float*>(sm + OFF_L);
  float* X = reinterpret_cast<float*>(sm + OFF_X);
  float* G = reinterpret_cast<float*>(sm + OFF_SMALL);
  float* nq = G + C;
  float* nk = nq + C;
  float* bb = nk + C;
  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* bar_mma = bar_tma + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_tma + 2);
  uint8_t* slab = p.slabs + slab_index(p, b, hv, n) * p.slab_bytes;

  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tslot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tslot;

  if (tid == 0) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar_tma)),
                 "r"(6 * 8192)
                 : "memory");
    tma_load4(smem_u32(sm + OFF_K0), &map_k, 0, h, t0, b, bar_tma);
    tma_load4(smem_u32(sm + OFF_K1), &map_k, 64, h, t0, b, bar_tma);
    tma_load4(smem_u32(sm + OFF_Q0), &map_q, 0, h, t0, b, bar_tma);
    tma_load4(smem_u32(sm + OFF_Q1), &map_q, 64, h, t0, b, bar_tma);
    tma_load4(smem_u32(sm + OFF_V0), &map_v, 0, hv, t0, b, bar_tma);
    tma_load4(smem_u32(sm + OFF_V1), &map_v, 64, hv, t0, b, bar_tma);
  }
  // beta (plain loads; zero past the end of the sequence).
  if (tid < C) {
    const int t = t0 + tid;
    bb[tid] = (t < p.T) ? p.beta[((size_t)b * p.T + t) * p.HV + hv] : 0.f;
  }
  bool ok = __all_sync(0xffffffffu, mbar_wait(bar_tma, 0));
  if (!ok && lane == 0) atomicOr(p.error_word, kErrTmaWait);

  // ---- MMA 1: D[0:128, 0:64] = [k; q] k^T ------------------------------------
  if (ok && tid == 0) {
    fence_after();
    const uint32_t id = idesc_bf16(128, 64, 0, 0);
    const uint32_t base = smem_u32(sm + OFF_K0);
#pragma unroll
    for (int s = 0; s < K / 16; ++s) {
      const uint32_t a = base + (s >> 2) * 16384 + (s & 3) * 32;
      umma(tmem, sdesc(a, 16, 1024), sdesc(a, 16, 1024), id, s > 0);
    }
    umma_commit(bar_mma);
  }
  // Row norms (threads 0-63: k rows, 64-127: q rows) and the gate cumsum, while
  // the MMA runs.
  {
    const int r = tid & 63;
    const uint8_t* t0p = sm + (tid < 64 ? OFF_K0 : OFF_Q0);
    const uint8_t* t1p = sm + (tid < 64 ? OFF_K1 : OFF_Q1);
    float ss = 0.f;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      const uint32_t off = swz128((uint32_t)(r * 128 + ch * 16));
      const uint4 u0 = *reinterpret_cast<const uint4*>(t0p + off);
      const uint4 u1 = *reinterpret_cast<const uint4*>(t1p + off);
      const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
        ss = fmaf(lo, lo, fmaf(hi, hi, ss));
      }
    }
    const float inv = p.use_l2 ? 1.f / sqrtf(ss + 1e-6f) : 1.f;
    if (tid < 64) nk[r] = inv; else nq[r] = inv;
  }
  if (warp == 0) {
    // Inclusive scan of the 64 gate values of the chunk, two per lane (zero
    // past the end of the sequence).
    const int ta = t0 + 2 * lane;
    const float a0 = (ta < p.T) ? p.g[((size_t)b * p.T + ta) * p.HV + hv] : 0.f;
    const float a1 = (ta + 1 < p.T) ? p.g[((size_t)b * p.T + ta + 1) * p.HV + hv] : 0.f;
    float s = a0 + a1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    const float excl = s - (a0 + a1);
    G[2 * lane] = excl + a0;
    G[2 * lane + 1] = excl + a0 + a1;
  }
  __syncthreads();

  // ---- epilogue 1: A_kk -> L (smem), A_qk -> slab ------------------------------
  if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_mma, 0));
  if (!ok && tid == 0) atomicOr(p.error_word, kErrMmaWait);
  fence_after();
  if (ok) {
    const int r = tid & 63;
    const bool is_q = tid >= 64;
    const float Gi = G[r];
    const float rowf = is_q ? p.scale * nq[r] : nk[r];
    __nv_bfloat16* aq = reinterpret_cast<__nv_bfloat16*>(slab + Slab::AQ2);
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      float v[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + cc * 32, v);
      if (!is_q) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int j = cc * 32 + e;
          L[r * C + j] = (j < r) ? v[e] * rowf * nk[j] * __expf(Gi - G[j]) * bb[j] : 0.f;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int f = 0; f < 8; f += 2) {
            float a2[2];
#pragma unroll
            for (int z = 0; z < 2; ++z) {
              const int j = cc * 32 + e + f + z;
              a2[z] = (j <= r) ? v[e + f + z] * rowf * nk[j] * __expf(Gi - G[j]) * bb[j] : 0.f;
            }
            __nv_bfloat162 hb = __floats2bfloat162_rn(a2[0], a2[1]);
            const float2 hf = __bfloat1622float2(hb);
            hi[f / 2] = *reinterpret_cast<uint32_t*>(&hb);
            lo[f / 2] = pack_bf16(a2[0] - hf.x, a2[1] - hf.y);
          }
          const int j0 = cc * 32 + e;
          *reinterpret_cast<uint4*>(aq + r * C + j0) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(aq + C * C + r * C + j0) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
    }
  }
  fence_before();
  __syncthreads();

  // ---- X = (I + L)^-1 ---------------------------------------------------------
  // Diagonal 16x16 blocks: thread (blk, col) runs forward substitution down one column.
  if (tid < 64) {
    const int blk = tid >> 4, col = tid & 15, o = blk * 16;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = (i == col) ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < i; ++m) acc = fmaf(-L[(o + i) * C + o + m], x[m], acc);
      x[i] = acc;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) X[(o + i) * C + o + col] = x[i];
  } else {
    // Zero the strictly upper blocks of X.
    for (int idx = tid - 64; idx < C * C; idx += 64) {
      const int i = idx / C, j = idx % C;
      if ((j >> 4) > (i >> 4)) X[idx] = 0.f;
    }
  }
  __syncthreads();
  // Off-diagonal blocks, by distance d = I - J: X_IJ = -X_II sum_{m=J}^{I-1} L_Im X_mJ.
  // T_IJ is staged in the strictly upper blocks of L (unused by then).
#pragma unroll 1
  for (int d = 1; d < 4; ++d) {
    const int nblk = 4 - d;
    for (int idx = tid; idx < nblk * 256; idx += THREADS) {
      const int J = idx >> 8, e = idx & 255, i = e >> 4, j = e & 15, I = J + d;
      float acc = 0.f;
      for (int m = 16 * J; m < 16 * I; ++m) acc = fmaf(L[(16 * I + i) * C + m], X[m * C + 16 * J + j], acc);
      L[(16 * J + i) * C + 16 * I + j] = acc;   // block (J, I) of L is above the diagonal
    }
    __syncthreads();
    for (int idx = tid; idx < nblk * 256; idx += THREADS) {
      const int J = idx >> 8, e = idx & 255, i = e >> 4, j = e & 15, I = J + d;
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m)
        acc = fmaf(X[(16 * I + i) * C + 16 * I + m], L[(16 * J + m) * C + 16 * I + j], acc);
      X[(16 * I + i) * C + 16 * J + j] = -acc;
    }
    __syncthreads();
  }

  // ---- A operands of the W / U MMAs: XW = [X'hi; X'lo], XU = [Xhi; Xlo] ---------
  // X' = X diag(exp(G_j) |k_j|^-1). Thread: row r = tid >> 1, columns 32 (tid & 1) ..
  {
    const int r = tid >> 1, c0 = (tid & 1) * 32;
    float xv[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) xv[e] = X[r * C + c0 + e];
    __syncthreads();   // X and L are overwritten below
    uint8_t* xw = sm + OFF_L;
    uint8_t* xu = sm + OFF_X;
#pragma unroll
    for (int e = 0; e < 32; e += 8) {
      uint32_t whi[4], wlo[4], uhi[4], ulo[4];
#pragma unroll
      for (int f = 0; f < 8; f += 2) {
        const int j = c0 + e + f;
        const float w0 = xv[e + f] * __expf(G[j]) * nk[j];
        const float w1 = xv[e + f + 1] * __expf(G[j + 1]) * nk[j + 1];
        __nv_bfloat162 wb = __floats2bfloat162_rn(w0, w1);
        float2 wf = __bfloat1622float2(wb);
        whi[f / 2] = *reinterpret_cast<uint32_t*>(&wb);
        wlo[f / 2] = pack_bf16(w0 - wf.x, w1 - wf.y);
        __nv_bfloat162 ub = __floats2bfloat162_rn(xv[e + f], xv[e + f + 1]);
        float2 uf = __bfloat1622float2(ub);
        uhi[f / 2] = *reinterpret_cast<uint32_t*>(&ub);
        ulo[f / 2] = pack_bf16(xv[e + f] - uf.x, xv[e + f + 1] - uf.y);
      }
      const uint32_t off_hi = swz128((uint32_t)(r * 128 + (c0 + e) * 2));
      const uint32_t off_lo = swz128((uint32_t)((r + 64) * 128 + (c0 + e) * 2));
      *reinterpret_cast<uint4*>(xw + off_hi) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
      *reinterpret_cast<uint4*>(xw + off_lo) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
      *reinterpret_cast<uint4*>(xu + off_hi) = make_uint4(uhi[0], uhi[1], uhi[2], uhi[3]);
      *reinterpret_cast<uint4*>(xu + off_lo) = make_uint4(ulo[0], ulo[1], ulo[2], ulo[3]);
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  fence_before();
  __syncthreads();

  // ---- MMA 2/3: D_W = [X'hi; X'lo] k (cols 0-127), D_U = [Xhi; Xlo] v (cols 128-255) --
  if (ok && tid == 0) {
    fence_after();
    const uint32_t id = idesc_bf16(128, 128, 0, 1);
    const uint32_t xw = smem_u32(sm + OFF_L), xu = smem_u32(sm + OFF_X);
    const uint32_t kb = smem_u32(sm + OFF_K0), vb = smem_u32(sm + OFF_V0);
#pragma unroll
    for (int s = 0; s < C / 16; ++s) {
      umma(tmem, sdesc(xw + s * 32, 16, 1024), sdesc(kb + s * 2048, 16384, 1024), id, s > 0);
      umma(tmem + 128, sdesc(xu + s * 32, 16, 1024), sdesc(vb + s * 2048, 8192, 1024), id, s > 0);
    }
    umma_commit(bar_mma);
  }
  // Per-row factors of the state pass, while the MMAs run.
  {
    float* vec = reinterpret_cast<float*>(slab + Slab::VEC);
    const float gl = G[C - 1];
    if (tid < C) {
      vec[tid] = p.scale * nq[tid] * __expf(G[tid]);
      vec[C + tid] = bb[tid] * nk[tid] * __expf(gl - G[tid]);
    }
    vec[2 * C + tid] = __expf(gl);
  }
  if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_mma, 1));
  if (!ok && tid == 0) atomicOr(p.error_word, kErrMmaWait);
  fence_after();

  // ---- epilogue 2: W = D_W[0:64] + D_W[64:128], U = D_U[0:64] + D_U[64:128] ------
  // Warps 2-3 hand their W halves to warps 0-1 through shared memory; warps 0-1
  // hand their U halves to warps 2-3.
  float* xch_w = reinterpret_cast<float*>(sm + OFF_XCH_W);
  float* xch_u = reinterpret_cast<float*>(sm + OFF_XCH_U);
  const int r = tid & 63;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  if (ok) {
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      float v[32];
      tmem_ld32(tmem + lane_base + (tid < 64 ? 128 : 0) + cc * 32, v);
      float* dst = (tid < 64 ? xch_u : xch_w) + r * 128 + cc * 32;
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        *reinterpret_cast<float4*>(dst + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
    }
  }
  fence_before();
  __syncthreads();
  if (ok) {
    __nv_bfloat16* w2 = reinterpret_cast<__nv_bfloat16*>(slab + Slab::W2);
    float* u = reinterpret_cast<float*>(slab + Slab::U);
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      float v[32];
      tmem_ld32(tmem + lane_base + (tid < 64 ? 0 : 128) + cc * 32, v);
      const float* other = (tid < 64 ? xch_w : xch_u) + r * 128 + cc * 32;
      if (tid < 64) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int f = 0; f < 8; f += 2) {
            const float w0 = -(v[e + f] + other[e + f]);
            const float w1 = -(v[e + f + 1] + other[e + f + 1]);
            __nv_bfloat162 hb = __floats2bfloat162_rn(w0, w1);
            const float2 hf = __bfloat1622float2(hb);
            hi[f / 2] = *reinterpret_cast<uint32_t*>(&hb);
            lo[f / 2] = pack_bf16(w0 - hf.x, w1 - hf.y);
          }
          const int c = cc * 32 + e;
          *reinterpret_cast<uint4*>(w2 + r * K + c) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(w2 + C * K + r * K + c) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 s4 = make_float4(v[e] + other[e], v[e + 1] + other[e + 1],
                                        v[e + 2] + other[e + 2], v[e + 3] + other[e + 3]);
          *reinterpret_cast<float4*>(u + r * V + cc * 32 + e) = s4;
        }
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS));
  }
}

// ---------------------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 4-D map over a [B, T, heads, 128] bf16 tensor; box = 64 channels x 1 head x
// 64 tokens x 1 batch row, 128-byte swizzle, zero fill out of bounds.
bool encode_bthd(CUtensorMap* map, const void* base, int B, int T, int heads) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[4] = {128, (cuuint64_t)heads, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {128 * 2, (cuuint64_t)heads * 128 * 2,
                                 (cuuint64_t)T * heads * 128 * 2};
  const cuuint32_t box[4] = {64, 1, 64, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool chunk_tc_available() { return get_encode() != nullptr; }

gdr_status launch_chunk_tc(const Params& p, cudaStream_t stream) {
  if (p.gate_mode != 0) return launch_chunk_simt(p, stream);
  CUtensorMap mq, mk, mv;
  if (!encode_bthd(&mq, p.q, p.B, p.T, p.H) || !encode_bthd(&mk, p.k, p.B, p.T, p.H) ||
      !encode_bthd(&mv, p.v, p.B, p.T, p.HV))
    return GDR_ERR_CUDA;
  if (cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SMEM_BYTES) != cudaSuccess)
    return GDR_ERR_CUDA;
  TcArgs a{p};
  dim3 grid(p.N, p.HV, p.B);
  chunk_tc_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(mq, mk, mv, a);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

}  // namespace fast
}  // namespace gdr
