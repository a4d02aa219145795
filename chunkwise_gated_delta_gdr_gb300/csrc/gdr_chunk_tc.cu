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
constexpr int OFF_K0 = 0;          // k cols 0-63   (8 KB, 128-byte swizzle, from TMA)
constexpr int OFF_Q0 = 8192;       // q cols 0-63
constexpr int OFF_K1 = 16384;      // k cols 64-127
constexpr int OFF_Q1 = 24576;      // q cols 64-127
constexpr int OFF_V0 = 32768;      // v cols 0-63
constexpr int OFF_V1 = 40960;      // v cols 64-127
constexpr int LDL = 68;            // fp32 row stride of L (272 B: float4 rows, conflict-free)
constexpr int OFF_L = 49152;       // L [64][LDL] fp32; later XW (16 KB)
constexpr int LDQ = 72;            // bf16 row stride of the A_qk staging tiles
constexpr int OFF_AQS = 66560;     // A_qk hi / lo staging [2][64][LDQ] bf16
constexpr int OFF_XU = 65536;      // XU (16 KB), written once L and the A_qk staging are dead
constexpr int LDX = 68;            // fp32 row stride of X
constexpr int OFF_X = 84992;       // X = (I + L)^-1 [64][LDX] fp32
constexpr int OFF_T = 8192;        // block-product scratch [32][36] fp32 (in the dead q tile)
constexpr int OFF_SMALL = 102400;  // G, nq, nk, beta, column factor (5 x 64 fp32)
constexpr int OFF_BAR = 103680;    // mbarriers + TMEM slot
constexpr int SMEM_BYTES = OFF_BAR + 64 + 1024;  // + alignment slack
// Epilogue-2 staging (after the W / U MMAs, over the dead operand tiles).
constexpr int LDWS = 136;          // bf16 row stride of the -W staging tiles
constexpr int OFF_WS = 0;          // -W hi / lo [2][64][LDWS] bf16 (34816 B)
constexpr int LDUS = 132;          // fp32 row stride of the U staging tile
constexpr int OFF_US = 34816;      // U [64][LDUS] fp32 (33792 B)
static_assert(OFF_AQS + 2 * 64 * LDQ * 2 <= OFF_SMALL, "A_qk staging overlaps");
static_assert(OFF_L + 64 * LDL * 4 <= OFF_AQS, "L overlaps");
static_assert(OFF_US + 64 * LDUS * 4 <= OFF_X, "U staging overlaps X");
static_assert(OFF_X + 64 * LDX * 4 <= OFF_SMALL, "X overlaps");
static_assert(OFF_T + 32 * 36 * 4 <= OFF_K1, "scratch overlaps the k tile");

// Rows of the stacked A operands [X_hi; X_lo] of the W / U MMAs are
// interleaved in blocks of 16 so that the hi and lo products of output row i
// land in the same warp's TMEM lanes (lanes 32 w + t and 32 w + 16 + t):
//   row i, hi part -> A row 32 (i / 16) + (i % 16); lo part -> that + 16.
__host__ __device__ constexpr int stacked_row(int i, int lo) { return 32 * (i >> 4) + (i & 15) + 16 * lo; }

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
  float* T = reinterpret_cast<float*>(sm + OFF_T);
  __nv_bfloat16* aqs = reinterpret_cast<__nv_bfloat16*>(sm + OFF_AQS);
  float* G = reinterpret_cast<float*>(sm + OFF_SMALL);
  float* nq = G + C;
  float* nk = nq + C;
  float* bb = nk + C;
  float* cfac = bb + C;
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
  // Gate and beta (plain loads, issued before the TMA wait; zero past the end).
  float ga = 0.f, gb = 0.f;
  if (warp == 0) {
    const int ta = t0 + 2 * lane;
    if (ta < p.T) ga = p.g[((size_t)b * p.T + ta) * p.HV + hv];
    if (ta + 1 < p.T) gb = p.g[((size_t)b * p.T + ta + 1) * p.HV + hv];
  }
  if (tid < C) {
    const int t = t0 + tid;
    bb[tid] = (t < p.T) ? p.beta[((size_t)b * p.T + t) * p.HV + hv] : 0.f;
  }
  bool ok = __all_sync(0xffffffffu, mbar_wait(bar_tma, 0));
  if (!ok && lane == 0) atomicOr(p.error_word, kErrTmaWait);

  // ---- MMA 1: D[0:128, 0:64] = [k; q] k^T -------------------------------------
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
  // Row norms (threads 0-63: k rows, 64-127: q rows) and the gate cumsum while
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
    // Inclusive scan of the chunk's 64 gate values, two per lane.
    float s = ga + gb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    const float excl = s - (ga + gb);
    G[2 * lane] = excl + ga;
    G[2 * lane + 1] = excl + ga + gb;
  }
  __syncthreads();

  // ---- epilogue 1: A_kk -> L (fp32, smem), A_qk -> bf16 hi/lo staging -----------
  if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_mma, 0));
  if (!ok && tid == 0) atomicOr(p.error_word, kErrMmaWait);
  fence_after();
  if (ok) {
    const int r = tid & 63;
    const bool is_q = tid >= 64;
    const float Gi = G[r];
    const float rowf = is_q ? p.scale * nq[r] : nk[r];
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
      float v[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + cc * 32, v);
      if (!is_q) {
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          float a4[4];
#pragma unroll
          for (int z = 0; z < 4; ++z) {
            const int j = cc * 32 + e + z;
            a4[z] = (j < r) ? v[e + z] * rowf * nk[j] * __expf(Gi - G[j]) * bb[j] : 0.f;
          }
          *reinterpret_cast<float4*>(L + r * LDL + cc * 32 + e) = make_float4(a4[0], a4[1], a4[2], a4[3]);
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
          *reinterpret_cast<uint4*>(aqs + r * LDQ + j0) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(aqs + 64 * LDQ + r * LDQ + j0) =
              make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
    }
  }
  fence_before();
  __syncthreads();

  // A_qk slab rows out (coalesced) and the per-row factors of the state pass.
  {
    __nv_bfloat16* aq = reinterpret_cast<__nv_bfloat16*>(slab + Slab::AQ2);
#pragma unroll 2
    for (int idx = tid; idx < 2 * C * (C / 8); idx += THREADS) {
      const int half = idx / (C * C / 8), rem = idx % (C * C / 8);
      const int r = rem >> 3, c8 = (rem & 7) * 8;
      *reinterpret_cast<uint4*>(aq + half * C * C + r * C + c8) =
          *reinterpret_cast<const uint4*>(aqs + half * 64 * LDQ + r * LDQ + c8);
    }
    float* vec = reinterpret_cast<float*>(slab + Slab::VEC);
    const float gl = G[C - 1];
    if (tid < C) {
      vec[tid] = p.scale * nq[tid] * __expf(G[tid]);
      vec[C + tid] = bb[tid] * nk[tid] * __expf(gl - G[tid]);
      cfac[tid] = __expf(G[tid]) * nk[tid];   // column factor of X' = X diag(exp(G) |k|^-1)
    }
    vec[2 * C + tid] = __expf(gl);
  }

  // ---- X = (I + L)^-1, blocked --------------------------------------------------
  // Level 0: the four 16x16 diagonal blocks, one column per thread (threads 0-63),
  // by forward substitution x_i = delta_ij - sum_{m<i} L_im x_m.
  if (tid < 64) {
    const int o = (tid >> 4) * 16, col = tid & 15;
    float xd[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = (i == col) ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < i; ++m) acc = fmaf(-L[(o + i) * LDL + o + m], xd[m], acc);
      xd[i] = acc;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) X[(o + i) * LDX + o + col] = xd[i];
  }
  __syncthreads();
  // Level 1: X_10 = -X_11 (L_10 X_00) and X_32 = -X_33 (L_32 X_22), 16x16 blocks;
  // each thread one row segment of 4 columns.
  {
    const int which = tid >> 6, e = tid & 63, i = e >> 2, j0 = (e & 3) * 4;
    const int I = 16 * (2 * which + 1), J = I - 16;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float l = L[(I + i) * LDL + J + m];
      const float4 xv = *reinterpret_cast<const float4*>(X + (J + m) * LDX + J + j0);
      acc.x = fmaf(l, xv.x, acc.x); acc.y = fmaf(l, xv.y, acc.y);
      acc.z = fmaf(l, xv.z, acc.z); acc.w = fmaf(l, xv.w, acc.w);
    }
    *reinterpret_cast<float4*>(T + (which * 16 + i) * 36 + j0) = acc;
    __syncthreads();
    float4 r4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float xv = X[(I + i) * LDX + I + m];
      const float4 t4 = *reinterpret_cast<const float4*>(T + (which * 16 + m) * 36 + j0);
      r4.x = fmaf(xv, t4.x, r4.x); r4.y = fmaf(xv, t4.y, r4.y);
      r4.z = fmaf(xv, t4.z, r4.z); r4.w = fmaf(xv, t4.w, r4.w);
    }
    *reinterpret_cast<float4*>(X + (I + i) * LDX + J + j0) = make_float4(-r4.x, -r4.y, -r4.z, -r4.w);
  }
  __syncthreads();
  // Level 2: X[32:64, 0:32] = -X[32:64, 32:64] (L[32:64, 0:32] X[0:32, 0:32]); each
  // thread one row segment of 8 columns. Entries above the diagonal of X are
  // never written and read as zero through the masks below.
  {
    const int i = tid >> 2, j0 = (tid & 3) * 8;
    float a[8];
#pragma unroll
    for (int z = 0; z < 8; ++z) a[z] = 0.f;
#pragma unroll 8
    for (int m = 0; m < 32; ++m) {
      const float l = L[(32 + i) * LDL + m];
      const float4 x0 = *reinterpret_cast<const float4*>(X + m * LDX + j0);
      const float4 x1 = *reinterpret_cast<const float4*>(X + m * LDX + j0 + 4);
      const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int z = 0; z < 8; ++z) a[z] = fmaf(l, (j0 + z <= m) ? xs[z] : 0.f, a[z]);
    }
    __syncthreads();   // every thread is past its reads of the level-1 scratch
#pragma unroll
    for (int z = 0; z < 8; z += 4)
      *reinterpret_cast<float4*>(T + i * 36 + j0 + z) = make_float4(a[z], a[z + 1], a[z + 2], a[z + 3]);
    __syncthreads();
    float r8[8];
#pragma unroll
    for (int z = 0; z < 8; ++z) r8[z] = 0.f;
#pragma unroll 8
    for (int m = 0; m < 32; ++m) {
      const float xv = (m <= i) ? X[(32 + i) * LDX + 32 + m] : 0.f;
      const float4 t0 = *reinterpret_cast<const float4*>(T + m * 36 + j0);
      const float4 t1 = *reinterpret_cast<const float4*>(T + m * 36 + j0 + 4);
      const float ts[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
      for (int z = 0; z < 8; ++z) r8[z] = fmaf(xv, ts[z], r8[z]);
    }
#pragma unroll
    for (int z = 0; z < 8; z += 4)
      *reinterpret_cast<float4*>(X + (32 + i) * LDX + j0 + z) =
          make_float4(-r8[z], -r8[z + 1], -r8[z + 2], -r8[z + 3]);
  }
  __syncthreads();   // X complete; L and the A_qk staging are dead from here on

  // ---- A operands XW = [X' hi/lo], XU = [X hi/lo] (rows interleaved, see stacked_row)
  // Each thread: one row i, 8 consecutive columns, 4 items.
  {
    uint8_t* xw = sm + OFF_L;
    uint8_t* xu = sm + OFF_XU;
#pragma unroll 2
    for (int it = tid; it < C * 8; it += THREADS) {
      const int i = it >> 3, c8 = (it & 7) * 8;
      const float4 x0 = *reinterpret_cast<const float4*>(X + i * LDX + c8);
      const float4 x1 = *reinterpret_cast<const float4*>(X + i * LDX + c8 + 4);
      const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      uint32_t whi[4], wlo[4], uhi[4], ulo[4];
#pragma unroll
      for (int z = 0; z < 8; z += 2) {
        const float u0 = (c8 + z <= i) ? xs[z] : 0.f;
        const float u1 = (c8 + z + 1 <= i) ? xs[z + 1] : 0.f;
        const float w0 = u0 * cfac[c8 + z], w1 = u1 * cfac[c8 + z + 1];
        __nv_bfloat162 wb = __floats2bfloat162_rn(w0, w1);
        const float2 wf = __bfloat1622float2(wb);
        whi[z / 2] = *reinterpret_cast<uint32_t*>(&wb);
        wlo[z / 2] = pack_bf16(w0 - wf.x, w1 - wf.y);
        __nv_bfloat162 ub = __floats2bfloat162_rn(u0, u1);
        const float2 uf = __bfloat1622float2(ub);
        uhi[z / 2] = *reinterpret_cast<uint32_t*>(&ub);
        ulo[z / 2] = pack_bf16(u0 - uf.x, u1 - uf.y);
      }
      const uint32_t o_hi = swz128((uint32_t)(stacked_row(i, 0) * 128 + c8 * 2));
      const uint32_t o_lo = swz128((uint32_t)(stacked_row(i, 1) * 128 + c8 * 2));
      *reinterpret_cast<uint4*>(xw + o_hi) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
      *reinterpret_cast<uint4*>(xw + o_lo) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
      *reinterpret_cast<uint4*>(xu + o_hi) = make_uint4(uhi[0], uhi[1], uhi[2], uhi[3]);
      *reinterpret_cast<uint4*>(xu + o_lo) = make_uint4(ulo[0], ulo[1], ulo[2], ulo[3]);
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  fence_before();
  __syncthreads();

  // ---- MMA 2/3: D_W = XW k (TMEM cols 0-127), D_U = XU v (cols 128-255) ----------
  if (ok && tid == 0) {
    fence_after();
    const uint32_t id = idesc_bf16(128, 128, 0, 1);
    const uint32_t xw = smem_u32(sm + OFF_L), xu = smem_u32(sm + OFF_XU);
    const uint32_t kb = smem_u32(sm + OFF_K0), vb = smem_u32(sm + OFF_V0);
#pragma unroll
    for (int s = 0; s < C / 16; ++s) {
      umma(tmem, sdesc(xw + s * 32, 16, 1024), sdesc(kb + s * 2048, 16384, 1024), id, s > 0);
      umma(tmem + 128, sdesc(xu + s * 32, 16, 1024), sdesc(vb + s * 2048, 8192, 1024), id, s > 0);
    }
    umma_commit(bar_mma);
  }
  if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_mma, 1));
  if (!ok && tid == 0) atomicOr(p.error_word, kErrMmaWait);
  fence_after();

  // ---- epilogue 2: W = hi + lo rows, U likewise; -W hi/lo and U staged in smem ----
  // Lane t < 16 of warp w holds the hi product of row r = 16 w + t, lane t + 16
  // the lo product of the same row: one shuffle per value sums them, after which
  // lane t keeps columns [0,16) and lane t + 16 columns [16,32) of each 32-block.
  __nv_bfloat16* ws_hi = reinterpret_cast<__nv_bfloat16*>(sm + OFF_WS);
  __nv_bfloat16* ws_lo = ws_hi + 64 * LDWS;
  float* us = reinterpret_cast<float*>(sm + OFF_US);
  if (ok) {
    const int r = 16 * warp + (lane & 15);
    const int half = lane >> 4;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
#pragma unroll 1
    for (int blk = 0; blk < 8; ++blk) {
      const bool is_u = blk >= 4;
      const int cc = blk & 3;
      float v[32];
      tmem_ld32(tmem + lane_base + (is_u ? 128 : 0) + cc * 32, v);
      float s[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float send = half ? v[e] : v[16 + e];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
        s[e] = (half ? v[16 + e] : v[e]) + recv;
      }
      const int c0 = cc * 32 + half * 16;
      if (!is_u) {
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const float w0 = -s[e], w1 = -s[e + 1];
          __nv_bfloat162 hb = __floats2bfloat162_rn(w0, w1);
          const float2 hf = __bfloat1622float2(hb);
          hi[e / 2] = *reinterpret_cast<uint32_t*>(&hb);
          lo[e / 2] = pack_bf16(w0 - hf.x, w1 - hf.y);
        }
        *reinterpret_cast<uint4*>(ws_hi + r * LDWS + c0) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(ws_hi + r * LDWS + c0 + 8) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
        *reinterpret_cast<uint4*>(ws_lo + r * LDWS + c0) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        *reinterpret_cast<uint4*>(ws_lo + r * LDWS + c0 + 8) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
      } else {
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<float4*>(us + r * LDUS + c0 + e) = make_float4(s[e], s[e + 1], s[e + 2], s[e + 3]);
      }
    }
  }
  fence_before();
  __syncthreads();
  // Coalesced copy-out of the staged -W (hi, lo) and U rows into the slab.
  {
    __nv_bfloat16* w2 = reinterpret_cast<__nv_bfloat16*>(slab + Slab::W2);
    float* u = reinterpret_cast<float*>(slab + Slab::U);
#pragma unroll 4
    for (int idx = tid; idx < 2 * C * (K / 8); idx += THREADS) {
      const int half = idx / (C * K / 8), rem = idx % (C * K / 8);
      const int r = rem >> 4, c8 = (rem & 15) * 8;
      *reinterpret_cast<uint4*>(w2 + half * C * K + r * K + c8) =
          *reinterpret_cast<const uint4*>(ws_hi + half * 64 * LDWS + r * LDWS + c8);
    }
#pragma unroll 4
    for (int idx = tid; idx < C * (V / 4); idx += THREADS) {
      const int r = idx >> 5, c4 = (idx & 31) * 4;
      *reinterpret_cast<float4*>(u + r * V + c4) = *reinterpret_cast<const float4*>(us + r * LDUS + c4);
    }
  }
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
