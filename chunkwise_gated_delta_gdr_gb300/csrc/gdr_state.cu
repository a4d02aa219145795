// gdr_state.cu -- scalar-gate state recurrence for shapes the fused kernel
// does not take (fallback of gdr_recur.cu), and the dispatch of the recurrence.
//
// One CTA per (batch b, value head hv, 16-column V tile), serial over the
// chunks of the sequence. Per chunk n it applies the inter-chunk loop of the
// "分块并行计算（Chunkwise）" notes (listing of the chunk 间递推 section):
//     r   = U - W S
//     o   = (q exp(G)) S + A_qk r
//     S   = exp(G_last) S + (exp(G_last - G) k)^T (beta r)
// in the transposed form, so that every product has the 16 value columns of
// the tile as its M dimension and each accumulator can feed the next product
// straight from registers:
//     r^T  = U^T - S^T W^T                      (16 x 64,  K = 128)
//     o^T  = diag-scaled S^T q^T + r^T A_qk^T   (16 x 64)
//     S^T <- gamma S^T + (kscale r)^T k         (16 x 128, K = 64)
// The state S^T stays in fp32 registers for the whole sequence. Products run
// on the tensor cores with mma.sync m16n8k16 (bf16 in, fp32 accumulate); an
// fp32-valued operand x is fed as x_hi + x_lo with x_hi = bf16(x),
// x_lo = bf16(x - x_hi), and the lo * lo term is dropped, which keeps about 16
// significant bits per product. Every split term accumulates into its own
// register tile. The per-key gate runs on tcgen05 instead (gdr_state_kda.cu).
//
// Chunk operands arrive by TMA (128-byte swizzled tiles, read conflict-free
// by ldmatrix), one chunk ahead, counted on mbarriers.
#include <string.h>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "gdr_fast.cuh"
#include "gdr_ptx.cuh"

namespace gdr {
namespace fast {
namespace {

using namespace ptx;

constexpr int LDW = K + 8;   // bf16 row stride of the S^T exchange tiles (272 B)
constexpr int LDA = C + 8;   // bf16 row stride of the r^T exchange tiles (144 B)
constexpr long kWaitLimit = 1L << 24;
constexpr unsigned int kErrStateWait = 4u;

// Byte address of element (r, c) (c a multiple of 8) of a swizzled bf16 tile
// stored as 64-column boxes of 8 KB.
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int r, int c) {
  return base + (uint32_t)((c >> 6) * 8192 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4));
}

struct Maps {
  CUtensorMap q, k, w2, aq2, u;
};

// ---------------------------------------------------------------------------
// Scalar gate, warp-specialised. Warps 0-3 ("chain") run the serial part:
// publish S^T, r^T = U^T - S^T W^T, publish r^T / rho^T, S^T update. Warps 4-7
// ("output") trail by up to one chunk and compute o^T = diag(qscale) S^T q^T +
// r^T A_qk^T from double-buffered copies of the S^T and r^T tiles, so the
// output products leave the chain's critical path. Each group prefetches its
// own operand tiles one chunk ahead with TMA. Named barriers:
//   1: chain warps among themselves; 2: output warps among themselves;
//   3+s: S^T tile s ready (chain arrives, output waits);
//   5+s: r^T tile s ready (chain arrives, output waits);
//   7+s: chunk in buffer s consumed by the output warps (output arrives, chain waits).
namespace ws {
// Chain warps, output warps, and two producer warps that only issue TMA loads
// (one for each buffer ring), so that no compute warp waits on the issue.
constexpr int CW = 4, OW = 4, PW = 2, XT = (CW + OW) * 32, THREADS = XT + PW * 32;
// Chain-side buffer: W hi, W lo, k, U tile [64][16] fp32, VEC.
constexpr int C_W_HI = 0, C_W_LO = 16384, C_K = 32768, C_U = 49152, C_VEC = 53248, C_BYTES = 55296;
constexpr uint32_t C_TX = 32768 + 16384 + 4096 + 1024;
// Output-side buffer: q, A_qk hi, A_qk lo, qscale.
constexpr int O_Q = 0, O_AQ_HI = 16384, O_AQ_LO = 24576, O_QS = 32768, O_BYTES = 33792;
constexpr uint32_t O_TX = 16384 + 16384 + 256;
constexpr int XS_BYTES = 2 * 16 * LDW * 2;     // S^T hi + lo
constexpr int XR_BYTES = 2 * 16 * LDA * 2;     // r^T hi + lo (or rho^T)
constexpr int OFF_C = 0, OFF_O = 2 * C_BYTES, OFF_XS = OFF_O + 2 * O_BYTES,
              OFF_XR = OFF_XS + 2 * XS_BYTES, OFF_XP = OFF_XR + 2 * XR_BYTES,
              OFF_XO = OFF_XP + XR_BYTES, OFF_BAR = OFF_XO + OW * 16 * 16 * 4,
              TOTAL = OFF_BAR + 64 + 1024;
static_assert(TOTAL <= 232448, "shared memory plan too large");

__device__ __forceinline__ void nb_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void nb_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
}  // namespace ws

__global__ void __launch_bounds__(ws::THREADS) state_ws_kernel(const __grid_constant__ Maps maps,
                                                                Params p) {
  using namespace ws;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int vt = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
  const int h = hv / (p.HV / p.H);
  const int v0 = vt * VT;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const size_t seq = (size_t)b * p.HV + hv;
  const int chunk0 = (int)(seq * p.N);
  uint64_t* cfull = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* ofull = cfull + 2;
  uint64_t* cempty = cfull + 4;
  uint64_t* oempty = cfull + 6;
  const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int acol = (lane >> 4) * 8;
  const int brow = (lane & 7);
  const int bcol = (lane >> 3) * 8;

  auto xs = [&](int s, int lo) {
    return reinterpret_cast<__nv_bfloat16*>(sm + OFF_XS + s * XS_BYTES) + lo * 16 * LDW;
  };
  auto xr = [&](int s, int lo) {
    return reinterpret_cast<__nv_bfloat16*>(sm + OFF_XR + s * XR_BYTES) + lo * 16 * LDA;
  };
  __nv_bfloat16* xp_hi = reinterpret_cast<__nv_bfloat16*>(sm + OFF_XP);
  __nv_bfloat16* xp_lo = xp_hi + 16 * LDA;

  auto issue_chain = [&](int n) {
    const int s = n & 1, idx = chunk0 + n;
    const uint32_t base = smem_u32(sm + OFF_C + s * C_BYTES);
    mbar_expect_tx(&cfull[s], C_TX);
    tma_load3(base + C_W_HI, &maps.w2, 0, 0, idx, &cfull[s]);
    tma_load3(base + C_W_HI + 8192, &maps.w2, 64, 0, idx, &cfull[s]);
    tma_load3(base + C_W_LO, &maps.w2, 0, 64, idx, &cfull[s]);
    tma_load3(base + C_W_LO + 8192, &maps.w2, 64, 64, idx, &cfull[s]);
    tma_load4(base + C_K, &maps.k, 0, h, n * C, b, &cfull[s]);
    tma_load4(base + C_K + 8192, &maps.k, 64, h, n * C, b, &cfull[s]);
    tma_load3(base + C_U, &maps.u, v0, 0, idx, &cfull[s]);
    bulk_load(base + C_VEC, p.slabs + (size_t)idx * p.slab_bytes + Slab::VEC, 1024, &cfull[s]);
  };
  auto issue_output = [&](int n) {
    const int s = n & 1, idx = chunk0 + n;
    const uint32_t base = smem_u32(sm + OFF_O + s * O_BYTES);
    mbar_expect_tx(&ofull[s], O_TX);
    tma_load4(base + O_Q, &maps.q, 0, h, n * C, b, &ofull[s]);
    tma_load4(base + O_Q + 8192, &maps.q, 64, h, n * C, b, &ofull[s]);
    tma_load3(base + O_AQ_HI, &maps.aq2, 0, 0, idx, &ofull[s]);
    tma_load3(base + O_AQ_LO, &maps.aq2, 0, 64, idx, &ofull[s]);
    bulk_load(base + O_QS, p.slabs + (size_t)idx * p.slab_bytes + Slab::VEC, 256, &ofull[s]);
  };

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&cfull[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&cempty[i], CW);
      mbar_init(&oempty[i], OW);
    }
    mbar_fence_init();
  }
  __syncthreads();
  bool ok = true;

  if (warp >= CW + OW) {
    // ============================== producer warps ===============================
    // Stage s of a ring is refilled with chunk n once the consumers have released
    // chunk n - 2 from it (completion (n >> 1) - 1 of its empty barrier).
    if (lane == 0) {
      const bool chain = warp == CW + OW;
      uint64_t* empty = chain ? cempty : oempty;
      for (int n = 0; n < p.N; ++n) {
        if (n >= 2) ok = ok && mbar_wait(&empty[n & 1], ((n >> 1) - 1) & 1, kWaitLimit);
        if (!ok) break;
        if (chain)
          issue_chain(n);
        else
          issue_output(n);
      }
      if (!ok) atomicOr(p.error_word, kErrStateWait);
    }
  } else if (warp < CW) {
    // ================================ chain warps ================================
    const int jw = 16 * warp, cw = 32 * warp;          // r^T j-tiles, state channels
    const int krow = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int kcol = cw + (lane >> 4) * 8;
    float S[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int c = cw + 8 * nt + 2 * t4;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int vv = g + (e >> 1) * 8, cc = c + (e & 1);
        S[nt][e] = p.s0 ? p.s0[(seq * K + cc) * V + v0 + vv] : 0.f;
      }
    }
    for (int n = 0; n < p.N; ++n) {
      const int s = n & 1;
      uint8_t* cb = sm + OFF_C + s * C_BYTES;
      const uint32_t w_hi = smem_u32(cb + C_W_HI), w_lo = smem_u32(cb + C_W_LO);
      const uint32_t k_t = smem_u32(cb + C_K);
      const float* su = reinterpret_cast<const float*>(cb + C_U);
      const float* ks = reinterpret_cast<const float*>(cb + C_VEC) + C;
      const float* gam = ks + C;
      if (n >= 2) nb_sync(7 + s, XT);                  // output done with chunk n-2's tiles
      __nv_bfloat16* xsh = xs(s, 0);
      __nv_bfloat16* xsl = xs(s, 1);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int c = cw + 8 * nt + 2 * t4;
        uint32_t hi, lo;
        split_pair(S[nt][0], S[nt][1], hi, lo);
        *reinterpret_cast<uint32_t*>(xsh + g * LDW + c) = hi;
        *reinterpret_cast<uint32_t*>(xsl + g * LDW + c) = lo;
        split_pair(S[nt][2], S[nt][3], hi, lo);
        *reinterpret_cast<uint32_t*>(xsh + (g + 8) * LDW + c) = hi;
        *reinterpret_cast<uint32_t*>(xsl + (g + 8) * LDW + c) = lo;
      }
      ok = ok && mbar_wait(&cfull[s], (n >> 1) & 1, kWaitLimit);
      nb_sync(1, CW * 32);                             // S^T complete
      nb_arrive(3 + s, XT);
      // r^T = U^T - S^T W^T, j in [jw, jw + 16)
      float Rhh[2][4], Rlh[2][4], Rhl[2][4];
#pragma unroll
      for (int jt = 0; jt < 2; ++jt) {
        const int j = jw + 8 * jt + 2 * t4;
        const float uf = p.zero_u ? 0.f : 1.f;
        Rhh[jt][0] = uf * su[j * VT + g];
        Rhh[jt][1] = uf * su[(j + 1) * VT + g];
        Rhh[jt][2] = uf * su[j * VT + g + 8];
        Rhh[jt][3] = uf * su[(j + 1) * VT + g + 8];
#pragma unroll
        for (int e = 0; e < 4; ++e) Rlh[jt][e] = Rhl[jt][e] = 0.f;
      }
#pragma unroll
      for (int ks2 = 0; ks2 < K / 16; ks2 += 2) {
        uint32_t ah[2][4], al[2][4];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          ldsm_x4(ah[h2], smem_u32(xsh + arow * LDW + 16 * (ks2 + h2) + acol));
          ldsm_x4(al[h2], smem_u32(xsl + arow * LDW + 16 * (ks2 + h2) + acol));
        }
#pragma unroll
        for (int jt = 0; jt < 2; ++jt) {
          uint32_t wh[4], wl[4];
          ldsm_x4(wh, tile_addr(w_hi, jw + 8 * jt + brow, 16 * ks2 + bcol));
          ldsm_x4(wl, tile_addr(w_lo, jw + 8 * jt + brow, 16 * ks2 + bcol));
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            mma_bf16_16816(Rhh[jt], ah[h2], wh[2 * h2], wh[2 * h2 + 1]);
            mma_bf16_16816(Rlh[jt], al[h2], wh[2 * h2], wh[2 * h2 + 1]);
            mma_bf16_16816(Rhl[jt], ah[h2], wl[2 * h2], wl[2 * h2 + 1]);
          }
        }
      }
      __nv_bfloat16* xrh = xr(s, 0);
      __nv_bfloat16* xrl = xr(s, 1);
#pragma unroll
      for (int jt = 0; jt < 2; ++jt) {
        const int j = jw + 8 * jt + 2 * t4;
        float R[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) R[e] = Rhh[jt][e] + (Rlh[jt][e] + Rhl[jt][e]);
        uint32_t hi, lo;
        split_pair(R[0], R[1], hi, lo);
        *reinterpret_cast<uint32_t*>(xrh + g * LDA + j) = hi;
        *reinterpret_cast<uint32_t*>(xrl + g * LDA + j) = lo;
        split_pair(R[2], R[3], hi, lo);
        *reinterpret_cast<uint32_t*>(xrh + (g + 8) * LDA + j) = hi;
        *reinterpret_cast<uint32_t*>(xrl + (g + 8) * LDA + j) = lo;
        const float k0 = ks[j], k1 = ks[j + 1];
        split_pair(R[0] * k0, R[1] * k1, hi, lo);
        *reinterpret_cast<uint32_t*>(xp_hi + g * LDA + j) = hi;
        *reinterpret_cast<uint32_t*>(xp_lo + g * LDA + j) = lo;
        split_pair(R[2] * k0, R[3] * k1, hi, lo);
        *reinterpret_cast<uint32_t*>(xp_hi + (g + 8) * LDA + j) = hi;
        *reinterpret_cast<uint32_t*>(xp_lo + (g + 8) * LDA + j) = lo;
      }
      nb_sync(1, CW * 32);                             // r^T, rho^T complete
      nb_arrive(5 + s, XT);
      // S^T = gamma S^T + rho^T k, c in [cw, cw + 32)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int c = cw + 8 * nt + 2 * t4;
        const float g0 = gam[c], g1 = gam[c + 1];
        S[nt][0] *= g0;
        S[nt][1] *= g1;
        S[nt][2] *= g0;
        S[nt][3] *= g1;
      }
      float Dl[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) Dl[nt][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks) {
        uint32_t ph[4], pl[4];
        ldsm_x4(ph, smem_u32(xp_hi + arow * LDA + 16 * ks + acol));
        ldsm_x4(pl, smem_u32(xp_lo + arow * LDA + 16 * ks + acol));
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          uint32_t kh[4];
          ldsm_x4_t(kh, tile_addr(k_t, 16 * ks + krow, kcol + 16 * np));
          mma_bf16_16816(S[2 * np], ph, kh[0], kh[1]);
          mma_bf16_16816(S[2 * np + 1], ph, kh[2], kh[3]);
          mma_bf16_16816(Dl[2 * np], pl, kh[0], kh[1]);
          mma_bf16_16816(Dl[2 * np + 1], pl, kh[2], kh[3]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) S[nt][e] += Dl[nt][e];
      __syncwarp();
      if (lane == 0) mbar_arrive(&cempty[s]);          // this warp is done with the stage
    }
    if (!ok) atomicOr(p.error_word, kErrStateWait);
    // Balance the consumed-barrier generations of the last two chunks.
    for (int n = (p.N >= 2 ? p.N - 2 : 0); n < p.N; ++n) nb_sync(7 + (n & 1), XT);
    if (p.sT) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int c = cw + 8 * nt + 2 * t4;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int vv = g + (e >> 1) * 8, cc = c + (e & 1);
          p.sT[(seq * K + cc) * V + v0 + vv] = S[nt][e];
        }
      }
    }
  } else {
    // ================================ output warps ===============================
    const int ow = warp - CW, iw = 16 * ow;            // o^T rows i in [iw, iw + 16)
    float* xo = reinterpret_cast<float*>(sm + OFF_XO) + ow * 256;
    for (int n = 0; n < p.N; ++n) {
      const int s = n & 1;
      uint8_t* ob = sm + OFF_O + s * O_BYTES;
      const uint32_t q_t = smem_u32(ob + O_Q);
      const uint32_t aq_hi = smem_u32(ob + O_AQ_HI), aq_lo = smem_u32(ob + O_AQ_LO);
      const float* qs = reinterpret_cast<const float*>(ob + O_QS);
      ok = ok && mbar_wait(&ofull[s], (n >> 1) & 1, kWaitLimit);
      nb_sync(3 + s, XT);                              // S^T of chunk n published
      const __nv_bfloat16* xsh = xs(s, 0);
      const __nv_bfloat16* xsl = xs(s, 1);
      float Oh[2][4], Ol[2][4];
#pragma unroll
      for (int it = 0; it < 2; ++it)
#pragma unroll
        for (int e = 0; e < 4; ++e) Oh[it][e] = Ol[it][e] = 0.f;
#pragma unroll
      for (int ks2 = 0; ks2 < K / 16; ks2 += 2) {
        uint32_t ah[2][4], al[2][4];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          ldsm_x4(ah[h2], smem_u32(xsh + arow * LDW + 16 * (ks2 + h2) + acol));
          ldsm_x4(al[h2], smem_u32(xsl + arow * LDW + 16 * (ks2 + h2) + acol));
        }
#pragma unroll
        for (int it = 0; it < 2; ++it) {
          uint32_t qh[4];
          ldsm_x4(qh, tile_addr(q_t, iw + 8 * it + brow, 16 * ks2 + bcol));
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            mma_bf16_16816(Oh[it], ah[h2], qh[2 * h2], qh[2 * h2 + 1]);
            mma_bf16_16816(Ol[it], al[h2], qh[2 * h2], qh[2 * h2 + 1]);
          }
        }
      }
      float O[2][4];
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int i = iw + 8 * it + 2 * t4;
        const float q0 = qs[i], q1 = qs[i + 1];
        O[it][0] = (Oh[it][0] + Ol[it][0]) * q0;
        O[it][1] = (Oh[it][1] + Ol[it][1]) * q1;
        O[it][2] = (Oh[it][2] + Ol[it][2]) * q0;
        O[it][3] = (Oh[it][3] + Ol[it][3]) * q1;
      }
      nb_sync(5 + s, XT);                              // r^T of chunk n published
      const __nv_bfloat16* xrh = xr(s, 0);
      const __nv_bfloat16* xrl = xr(s, 1);
      float Phh[2][4], Plh[2][4], Phl[2][4];
#pragma unroll
      for (int it = 0; it < 2; ++it)
#pragma unroll
        for (int e = 0; e < 4; ++e) Phh[it][e] = Plh[it][e] = Phl[it][e] = 0.f;
#pragma unroll
      for (int ks2 = 0; ks2 < C / 16; ks2 += 2) {
        uint32_t rh[2][4], rl[2][4];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          ldsm_x4(rh[h2], smem_u32(xrh + arow * LDA + 16 * (ks2 + h2) + acol));
          ldsm_x4(rl[h2], smem_u32(xrl + arow * LDA + 16 * (ks2 + h2) + acol));
        }
#pragma unroll
        for (int it = 0; it < 2; ++it) {
          uint32_t ah[4], al[4];
          ldsm_x4(ah, tile_addr(aq_hi, iw + 8 * it + brow, 16 * ks2 + bcol));
          ldsm_x4(al, tile_addr(aq_lo, iw + 8 * it + brow, 16 * ks2 + bcol));
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            mma_bf16_16816(Phh[it], rh[h2], ah[2 * h2], ah[2 * h2 + 1]);
            mma_bf16_16816(Plh[it], rl[h2], ah[2 * h2], ah[2 * h2 + 1]);
            mma_bf16_16816(Phl[it], rh[h2], al[2 * h2], al[2 * h2 + 1]);
          }
        }
      }
      // The S^T, r^T copies and this chunk's output tiles are no longer read.
      __syncwarp();
      if (lane == 0) mbar_arrive(&oempty[s]);          // q, A_qk, qscale of the stage read
      nb_sync(2, OW * 32);
      nb_arrive(7 + s, XT);
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int i = 8 * it + 2 * t4;
        xo[i * 16 + g] = O[it][0] + (Phh[it][0] + (Plh[it][0] + Phl[it][0]));
        xo[(i + 1) * 16 + g] = O[it][1] + (Phh[it][1] + (Plh[it][1] + Phl[it][1]));
        xo[i * 16 + g + 8] = O[it][2] + (Phh[it][2] + (Plh[it][2] + Phl[it][2]));
        xo[(i + 1) * 16 + g + 8] = O[it][3] + (Phh[it][3] + (Plh[it][3] + Phl[it][3]));
      }
      __syncwarp();
#pragma unroll
      for (int rep = 0; rep < 2; ++rep) {
        const int i = 8 * rep + (lane >> 2), c4 = (lane & 3) * 4;
        const int t = n * C + iw + i;
        if (t < p.T) {
          const float4 val = *reinterpret_cast<const float4*>(xo + i * 16 + c4);
          const size_t off = (((size_t)b * p.T + t) * p.HV + hv) * V + v0 + c4;
          if (p.out_bf16) {
            uint2 pk;
            pk.x = pack_bf16(val.x, val.y);
            pk.y = pack_bf16(val.z, val.w);
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + off) = pk;
          } else {
            *reinterpret_cast<float4*>(static_cast<float*>(p.out) + off) = val;
          }
        }
      }
      __syncwarp();
    }
    if (!ok) atomicOr(p.error_word, kErrStateWait);
  }
}

// ---------------------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

bool encode(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base,
            const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
            CUtensorMapSwizzle swz) {
  auto enc = encoder();
  if (!enc) return false;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(map, type, rank, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Slab array viewed as [nchunks][rows][cols] of `esize`-byte elements.
bool encode_slab(CUtensorMap* map, const Params& p, size_t offset, CUtensorMapDataType type,
                 int esize, int cols, int rows, int box_cols, CUtensorMapSwizzle swz) {
  const cuuint64_t nch = (cuuint64_t)p.B * p.HV * p.N;
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, nch};
  const cuuint64_t strides[2] = {(cuuint64_t)cols * esize, (cuuint64_t)p.slab_bytes};
  const cuuint32_t box[3] = {(cuuint32_t)box_cols, 64, 1};
  return encode(map, type, 3, p.slabs + offset, dims, strides, box, swz);
}

bool encode_bthd(CUtensorMap* map, const void* base, int B, int T, int heads) {
  const cuuint64_t dims[4] = {128, (cuuint64_t)heads, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {128 * 2, (cuuint64_t)heads * 128 * 2,
                                 (cuuint64_t)T * heads * 128 * 2};
  const cuuint32_t box[4] = {64, 1, 64, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_128B);
}

gdr_status launch_ws(const Params& p, cudaStream_t stream) {
  Maps m;
  memset(&m, 0, sizeof m);
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const bool ok =
      encode_slab(&m.w2, p, Slab::W2, BF, 2, K, 2 * C, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
      encode_slab(&m.aq2, p, Slab::AQ2, BF, 2, C, 2 * C, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
      encode_slab(&m.u, p, Slab::U, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, V, C, VT,
                  CU_TENSOR_MAP_SWIZZLE_NONE) &&
      encode_bthd(&m.q, p.q, p.B, p.T, p.H) && encode_bthd(&m.k, p.k, p.B, p.T, p.H);
  if (!ok) return GDR_ERR_CUDA;
  if (cudaFuncSetAttribute(state_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           ws::TOTAL) != cudaSuccess)
    return GDR_ERR_CUDA;
  dim3 grid(V / VT, p.HV, p.B);
  state_ws_kernel<<<grid, ws::THREADS, ws::TOTAL, stream>>>(m, p);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

}  // namespace

gdr_status launch_state(const Params& p, cudaStream_t stream) {
  // Kernels that write the outputs with the states have no separate output pass.
  if (p.gate_mode) return p.recur_mode == 2 ? GDR_OK : launch_state_kda_tc(p, stream);
  // Scalar gate: the fused chain + output launch when the chains leave SMs
  // for the outputs, else chain and outputs in the same CTAs.
  const gdr_status st = launch_recur(p, stream);
  if (st != GDR_ERR_UNSUPPORTED) return st;
  return p.recur_mode == 2 ? GDR_OK : launch_ws(p, stream);
}

}  // namespace fast
}  // namespace gdr
