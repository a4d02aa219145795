// gdr_state.cu -- inter-chunk state recurrence of the fast path.
//
// One CTA per (batch b, value head hv, 16-column V tile), 8 warps, serial over
// the chunks of the sequence. Per chunk n it applies the inter-chunk loop of
// the "分块并行计算（Chunkwise）" notes (listing of the chunk 间递推 section):
//     r   = U - W S
//     o   = (q exp(G)) S + A_qk r
//     S   = exp(G_last) S + (exp(G_last - G) k)^T (beta r)
// in the transposed form, so that every product has the 16 value columns of
// the tile as its M dimension and each accumulator can feed the next product
// straight from registers:
//     r^T  = U^T - S^T W^T                      (16 x 64,  K = 128)
//     o^T  = diag-scaled S^T q^T + r^T A_qk^T   (16 x 64)
//     S^T <- gamma S^T + (kscale r)^T k         (16 x 128, K = 64)
// The state S^T stays in fp32 registers for the whole sequence (each warp owns
// 16 of its 128 key channels). Products run on the tensor cores with
// mma.sync m16n8k16 (bf16 in, fp32 accumulate); an fp32-valued operand x is
// fed as x_hi + x_lo with x_hi = bf16(x), x_lo = bf16(x - x_hi), and the
// lo * lo term is dropped, which keeps about 16 significant bits per product.
// Every split term accumulates into its own register tile.
//
// Chunk operands arrive by TMA (128-byte swizzled tiles, read conflict-free
// by ldmatrix), one chunk ahead, counted on mbarriers; the only per-chunk
// exchanges are two shared-memory tiles (S^T and r^T) and two CTA barriers.
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
#ifndef KDA_MG
#define KDA_MG 4
#endif
constexpr long kWaitLimit = 1L << 24;
constexpr unsigned int kErrStateWait = 4u;

// Byte address of element (r, c) (c a multiple of 8) of a swizzled bf16 tile
// stored as 64-column boxes of 8 KB.
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int r, int c) {
  return base + (uint32_t)((c >> 6) * 8192 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4));
}

struct Maps {
  CUtensorMap q, k, w2, aq2, u, qb2, kb2;
};

// ---------------------------------------------------------------------------
// Per-key gate. One CTA per (b, hv, 16 MG value columns): MG groups of 4 warps,
// group m owning value rows 16 m .. 16 m + 15 of the CTA's S^T tile. All groups
// read the same chunk operands from one shared buffer, so a chunk's W, QB, KB
// and A_qk cross from L2 once per MG 16-column tiles.
//
// Operand tiles of one chunk, 128-byte swizzled [64][128] bf16 tiles as two
// 8 KB boxes. Group 1 (read by the r and o products): W hi/lo, QB hi/lo, plus
// the U tile and VEC in the small buffer. Group 2 (read by the state update and
// the second o product): KB hi/lo, A_qk hi/lo.
namespace kda {
constexpr int WARPS = 4;                          // per group
constexpr int JT = C / 8 / WARPS, CT = K / 8 / WARPS;
constexpr int W_HI = 0, W_LO = 16384, Q_HI = 32768, Q_LO = 49152;
constexpr int K_HI = 65536, K_LO = 81920, AQ_HI = 98304, AQ_LO = 106496, BIG = 114688;
constexpr uint32_t kGroup2Bytes = 32768 + 16384;

template <int MG>
struct Layout {
  static constexpr int VTK = 16 * MG;                     // value columns per CTA
  static constexpr int SMALL_U = BIG;                     // U tile [C][VTK] fp32
  static constexpr int SMALL_VEC = SMALL_U + C * VTK * 4; // qscale, kscale, gamma
  static constexpr int XS = SMALL_VEC + 1024;             // S^T hi / lo [VTK][LDW]
  static constexpr int XR = XS + 2 * VTK * LDW * 2;       // r^T, rho^T hi / lo [VTK][LDA]
  static constexpr int XO = XR + 4 * VTK * LDA * 2;       // o staging, per warp
  static constexpr int BARS = XO + MG * WARPS * (8 * JT * 16) * 4;
  static constexpr int TOTAL = BARS + 64 + 1024;
  static constexpr uint32_t kGroup1Bytes = 32768 + 32768 + C * VTK * 4 + 1024;
};
}  // namespace kda

template <int MG>
__global__ void __launch_bounds__(MG * kda::WARPS * 32, 1)
    state_kda_kernel(const __grid_constant__ Maps maps, Params p) {
  using namespace kda;
  using LY = Layout<MG>;
  constexpr int VTK = LY::VTK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int vt = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
  const int v0 = vt * VTK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mg = warp / WARPS, wi = warp % WARPS;
  const int vr = 16 * mg;                                 // this group's rows of S^T
  const int g = lane >> 2, t4 = lane & 3;

  __nv_bfloat16* xs_hi = reinterpret_cast<__nv_bfloat16*>(sm + LY::XS);
  __nv_bfloat16* xs_lo = xs_hi + VTK * LDW;
  __nv_bfloat16* xr_hi = reinterpret_cast<__nv_bfloat16*>(sm + LY::XR);
  __nv_bfloat16* xr_lo = xr_hi + VTK * LDA;
  __nv_bfloat16* xp_hi = xr_lo + VTK * LDA;
  __nv_bfloat16* xp_lo = xp_hi + VTK * LDA;
  float* xo = reinterpret_cast<float*>(sm + LY::XO) + warp * (8 * JT * 16);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + LY::BARS);   // [0] group 1, [1] group 2
  const float* su = reinterpret_cast<const float*>(sm + LY::SMALL_U);
  const float* vec = reinterpret_cast<const float*>(sm + LY::SMALL_VEC);

  const size_t seq = (size_t)b * p.HV + hv;
  const int chunk0 = (int)(seq * p.N);

  // Loads of chunk n, issued by one thread. Group 1 is reissued as soon as
  // every warp is past the products that read it (the CTA barrier after the
  // r^T tiles), group 2 after the chunk's last product.
  auto issue_group1 = [&](int n) {
    const int idx = chunk0 + n;
    const uint32_t big = smem_u32(sm);
    mbar_expect_tx(&bars[0], LY::kGroup1Bytes);
    tma_load3(big + W_HI, &maps.w2, 0, 0, idx, &bars[0]);
    tma_load3(big + W_HI + 8192, &maps.w2, 64, 0, idx, &bars[0]);
    tma_load3(big + W_LO, &maps.w2, 0, 64, idx, &bars[0]);
    tma_load3(big + W_LO + 8192, &maps.w2, 64, 64, idx, &bars[0]);
    tma_load3(big + Q_HI, &maps.qb2, 0, 0, idx, &bars[0]);
    tma_load3(big + Q_HI + 8192, &maps.qb2, 64, 0, idx, &bars[0]);
    tma_load3(big + Q_LO, &maps.qb2, 0, 64, idx, &bars[0]);
    tma_load3(big + Q_LO + 8192, &maps.qb2, 64, 64, idx, &bars[0]);
    tma_load3(big + LY::SMALL_U, &maps.u, v0, 0, idx, &bars[0]);
    bulk_load(big + LY::SMALL_VEC, p.slabs + (size_t)idx * p.slab_bytes + Slab::VEC, 1024, &bars[0]);
  };
  auto issue_group2 = [&](int n) {
    const int idx = chunk0 + n;
    const uint32_t big = smem_u32(sm);
    mbar_expect_tx(&bars[1], kGroup2Bytes);
    tma_load3(big + K_HI, &maps.kb2, 0, 0, idx, &bars[1]);
    tma_load3(big + K_HI + 8192, &maps.kb2, 64, 0, idx, &bars[1]);
    tma_load3(big + K_LO, &maps.kb2, 0, 64, idx, &bars[1]);
    tma_load3(big + K_LO + 8192, &maps.kb2, 64, 64, idx, &bars[1]);
    tma_load3(big + AQ_HI, &maps.aq2, 0, 0, idx, &bars[1]);
    tma_load3(big + AQ_LO, &maps.aq2, 0, 64, idx, &bars[1]);
  };

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0) {
    issue_group1(0);
    issue_group2(0);
  }

  const int jw = 8 * JT * wi, cw = 8 * CT * wi;

  float S[CT][4];
#pragma unroll
  for (int nt = 0; nt < CT; ++nt) {
    const int c = cw + 8 * nt + 2 * t4;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int vv = vr + g + (e >> 1) * 8, cc = c + (e & 1);
      S[nt][e] = p.s0 ? p.s0[(seq * K + cc) * V + v0 + vv] : 0.f;
    }
  }

  // ldmatrix lane addressing.
  const int arow = vr + (lane & 7) + ((lane >> 3) & 1) * 8;   // A fragments (this group's 16 rows)
  const int acol = (lane >> 4) * 8;
  const int brow = (lane & 7);                                // B from [n][k] tiles, 2 k-steps per x4
  const int bcol = (lane >> 3) * 8;
  const int krow = (lane & 7) + ((lane >> 3) & 1) * 8;        // B from the [j][c] k tile (.trans)
  const int kcol = cw + (lane >> 4) * 8;                      // two c-tiles per x4
  const uint32_t big = smem_u32(sm);
  bool ok = true;

  for (int n = 0; n < p.N; ++n) {
    const int t0 = n * C;

    // ---- A: publish this warp's S^T slice as bf16 hi/lo -------------------------
#pragma unroll
    for (int nt = 0; nt < CT; ++nt) {
      const int c = cw + 8 * nt + 2 * t4;
      uint32_t hi, lo;
      split_pair(S[nt][0], S[nt][1], hi, lo);
      *reinterpret_cast<uint32_t*>(xs_hi + (vr + g) * LDW + c) = hi;
      *reinterpret_cast<uint32_t*>(xs_lo + (vr + g) * LDW + c) = lo;
      split_pair(S[nt][2], S[nt][3], hi, lo);
      *reinterpret_cast<uint32_t*>(xs_hi + (vr + g + 8) * LDW + c) = hi;
      *reinterpret_cast<uint32_t*>(xs_lo + (vr + g + 8) * LDW + c) = lo;
    }
    ok = ok && mbar_wait(&bars[0], n & 1, kWaitLimit);   // W, QB, U, VEC of chunk n
    __syncthreads();          // #1: S^T tiles visible
    if (tid == 0 && !ok) atomicOr(p.error_word, kErrStateWait);

    // ---- B: r^T = U^T - S^T W^T and o^T part 1 = S^T QB^T (JT n-tiles each) -----
    float Rhh[JT][4], Rlh[JT][4], Rhl[JT][4], Oh[JT][4], Ol[JT][4], Ox[JT][4];
#pragma unroll
    for (int jt = 0; jt < JT; ++jt) {
      const int j = jw + 8 * jt + 2 * t4;
      Rhh[jt][0] = su[j * VTK + vr + g];
      Rhh[jt][1] = su[(j + 1) * VTK + vr + g];
      Rhh[jt][2] = su[j * VTK + vr + g + 8];
      Rhh[jt][3] = su[(j + 1) * VTK + vr + g + 8];
#pragma unroll
      for (int e = 0; e < 4; ++e) Rlh[jt][e] = Rhl[jt][e] = Oh[jt][e] = Ol[jt][e] = Ox[jt][e] = 0.f;
    }
#pragma unroll
    for (int ks2 = 0; ks2 < K / 16; ks2 += 2) {
      uint32_t ah[2][4], al[2][4];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        ldsm_x4(ah[h2], smem_u32(xs_hi + arow * LDW + 16 * (ks2 + h2) + acol));
        ldsm_x4(al[h2], smem_u32(xs_lo + arow * LDW + 16 * (ks2 + h2) + acol));
      }
#pragma unroll
      for (int jt = 0; jt < JT; ++jt) {
        const int rb = jw + 8 * jt + brow;
        uint32_t wh[4], wl[4], qh[4], ql[4];
        ldsm_x4(wh, tile_addr(big + W_HI, rb, 16 * ks2 + bcol));
        ldsm_x4(wl, tile_addr(big + W_LO, rb, 16 * ks2 + bcol));
        ldsm_x4(qh, tile_addr(big + Q_HI, rb, 16 * ks2 + bcol));
        ldsm_x4(ql, tile_addr(big + Q_LO, rb, 16 * ks2 + bcol));
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          mma_bf16_16816(Rhh[jt], ah[h2], wh[2 * h2], wh[2 * h2 + 1]);
          mma_bf16_16816(Rlh[jt], al[h2], wh[2 * h2], wh[2 * h2 + 1]);
          mma_bf16_16816(Rhl[jt], ah[h2], wl[2 * h2], wl[2 * h2 + 1]);
          mma_bf16_16816(Oh[jt], ah[h2], qh[2 * h2], qh[2 * h2 + 1]);
          mma_bf16_16816(Ol[jt], al[h2], qh[2 * h2], qh[2 * h2 + 1]);
          mma_bf16_16816(Ox[jt], ah[h2], ql[2 * h2], ql[2 * h2 + 1]);
        }
      }
    }

    // ---- C: publish r^T and rho^T = r^T diag(kscale) ------------------------------
    const float* qs = vec;
    const float* ks = vec + C;
    float O[JT][4];
#pragma unroll
    for (int jt = 0; jt < JT; ++jt) {
      const int j = jw + 8 * jt + 2 * t4;
      float R[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) R[e] = Rhh[jt][e] + (Rlh[jt][e] + Rhl[jt][e]);
      uint32_t hi, lo;
      split_pair(R[0], R[1], hi, lo);
      *reinterpret_cast<uint32_t*>(xr_hi + (vr + g) * LDA + j) = hi;
      *reinterpret_cast<uint32_t*>(xr_lo + (vr + g) * LDA + j) = lo;
      split_pair(R[2], R[3], hi, lo);
      *reinterpret_cast<uint32_t*>(xr_hi + (vr + g + 8) * LDA + j) = hi;
      *reinterpret_cast<uint32_t*>(xr_lo + (vr + g + 8) * LDA + j) = lo;
      const float k0 = ks[j], k1 = ks[j + 1];
      split_pair(R[0] * k0, R[1] * k1, hi, lo);
      *reinterpret_cast<uint32_t*>(xp_hi + (vr + g) * LDA + j) = hi;
      *reinterpret_cast<uint32_t*>(xp_lo + (vr + g) * LDA + j) = lo;
      split_pair(R[2] * k0, R[3] * k1, hi, lo);
      *reinterpret_cast<uint32_t*>(xp_hi + (vr + g + 8) * LDA + j) = hi;
      *reinterpret_cast<uint32_t*>(xp_lo + (vr + g + 8) * LDA + j) = lo;
      const float q0 = qs[j], q1 = qs[j + 1];
      O[jt][0] = (Oh[jt][0] + (Ol[jt][0] + Ox[jt][0])) * q0;
      O[jt][1] = (Oh[jt][1] + (Ol[jt][1] + Ox[jt][1])) * q1;
      O[jt][2] = (Oh[jt][2] + (Ol[jt][2] + Ox[jt][2])) * q0;
      O[jt][3] = (Oh[jt][3] + (Ol[jt][3] + Ox[jt][3])) * q1;
    }
    // gamma of this warp's channels, read before the group-1 buffer is reloaded.
    float gam[CT][2];
#pragma unroll
    for (int nt = 0; nt < CT; ++nt) {
      const int c = cw + 8 * nt + 2 * t4;
      gam[nt][0] = vec[2 * C + c];
      gam[nt][1] = vec[2 * C + c + 1];
    }
    ok = ok && mbar_wait(&bars[1], n & 1, kWaitLimit);   // KB, A_qk of chunk n
    __syncthreads();                           // #2: r^T / rho^T tiles visible; group 1 is free
    if (tid == 0 && n + 1 < p.N) issue_group1(n + 1);

    // ---- D: S^T = gamma S^T + rho^T KB (channels of this warp), o^T part 2 ---------
#pragma unroll
    for (int nt = 0; nt < CT; ++nt) {
      S[nt][0] *= gam[nt][0];
      S[nt][1] *= gam[nt][1];
      S[nt][2] *= gam[nt][0];
      S[nt][3] *= gam[nt][1];
    }
    float Dl[CT][4], Dx[CT][4], Phh[JT][4], Plh[JT][4], Phl[JT][4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
#pragma unroll
      for (int nt = 0; nt < CT; ++nt) Dl[nt][e] = Dx[nt][e] = 0.f;
#pragma unroll
      for (int jt = 0; jt < JT; ++jt) Phh[jt][e] = Plh[jt][e] = Phl[jt][e] = 0.f;
    }
#pragma unroll
    for (int ks = 0; ks < C / 16; ++ks) {
      uint32_t ph[4], pl[4];
      ldsm_x4(ph, smem_u32(xp_hi + arow * LDA + 16 * ks + acol));
      ldsm_x4(pl, smem_u32(xp_lo + arow * LDA + 16 * ks + acol));
#pragma unroll
      for (int np = 0; np < CT / 2; ++np) {
        uint32_t kh[4], kl[4];
        ldsm_x4_t(kh, tile_addr(big + K_HI, 16 * ks + krow, kcol + 16 * np));
        ldsm_x4_t(kl, tile_addr(big + K_LO, 16 * ks + krow, kcol + 16 * np));
        mma_bf16_16816(S[2 * np], ph, kh[0], kh[1]);
        mma_bf16_16816(S[2 * np + 1], ph, kh[2], kh[3]);
        mma_bf16_16816(Dl[2 * np], pl, kh[0], kh[1]);
        mma_bf16_16816(Dl[2 * np + 1], pl, kh[2], kh[3]);
        mma_bf16_16816(Dx[2 * np], ph, kl[0], kl[1]);
        mma_bf16_16816(Dx[2 * np + 1], ph, kl[2], kl[3]);
      }
    }
#pragma unroll
    for (int ks2 = 0; ks2 < C / 16; ks2 += 2) {
      uint32_t rh[2][4], rl[2][4];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        ldsm_x4(rh[h2], smem_u32(xr_hi + arow * LDA + 16 * (ks2 + h2) + acol));
        ldsm_x4(rl[h2], smem_u32(xr_lo + arow * LDA + 16 * (ks2 + h2) + acol));
      }
#pragma unroll
      for (int jt = 0; jt < JT; ++jt) {
        uint32_t ah[4], al[4];
        ldsm_x4(ah, tile_addr(big + AQ_HI, jw + 8 * jt + brow, 16 * ks2 + bcol));
        ldsm_x4(al, tile_addr(big + AQ_LO, jw + 8 * jt + brow, 16 * ks2 + bcol));
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          mma_bf16_16816(Phh[jt], rh[h2], ah[2 * h2], ah[2 * h2 + 1]);
          mma_bf16_16816(Plh[jt], rl[h2], ah[2 * h2], ah[2 * h2 + 1]);
          mma_bf16_16816(Phl[jt], rh[h2], al[2 * h2], al[2 * h2 + 1]);
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < CT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) S[nt][e] += Dl[nt][e] + Dx[nt][e];

    // ---- E: o rows of this warp (i in [jw, jw + 8 JT)), 16 value columns -> global
#pragma unroll
    for (int jt = 0; jt < JT; ++jt) {
      const int i = 8 * jt + 2 * t4;
      xo[i * 16 + g] = O[jt][0] + (Phh[jt][0] + (Plh[jt][0] + Phl[jt][0]));
      xo[(i + 1) * 16 + g] = O[jt][1] + (Phh[jt][1] + (Plh[jt][1] + Phl[jt][1]));
      xo[i * 16 + g + 8] = O[jt][2] + (Phh[jt][2] + (Plh[jt][2] + Phl[jt][2]));
      xo[(i + 1) * 16 + g + 8] = O[jt][3] + (Phh[jt][3] + (Plh[jt][3] + Phl[jt][3]));
    }
    __syncwarp();
#pragma unroll
    for (int rep = 0; rep < JT; ++rep) {
      const int i = 8 * rep + (lane >> 2), c4 = (lane & 3) * 4;   // 8 JT rows x 4 float4
      const int t = t0 + jw + i;
      if (t < p.T) {
        const float4 val = *reinterpret_cast<const float4*>(xo + i * 16 + c4);
        const size_t off = (((size_t)b * p.T + t) * p.HV + hv) * V + v0 + vr + c4;
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

    if (n + 1 < p.N) {
      __syncthreads();   // every warp is done with group 2 of chunk n
      if (tid == 0) issue_group2(n + 1);
    }
  }

  if (p.sT) {
#pragma unroll
    for (int nt = 0; nt < CT; ++nt) {
      const int c = cw + 8 * nt + 2 * t4;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int vv = vr + g + (e >> 1) * 8, cc = c + (e & 1);
        p.sT[(seq * K + cc) * V + v0 + vv] = S[nt][e];
      }
    }
  }
}

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
        Rhh[jt][0] = su[j * VT + g];
        Rhh[jt][1] = su[(j + 1) * VT + g];
        Rhh[jt][2] = su[j * VT + g + 8];
        Rhh[jt][3] = su[(j + 1) * VT + g + 8];
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

template <int MG>
gdr_status launch_kda(const Params& p, cudaStream_t stream) {
  using LY = kda::Layout<MG>;
  Maps m;
  memset(&m, 0, sizeof m);
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const bool ok =
      encode_slab(&m.w2, p, Slab::W2, BF, 2, K, 2 * C, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
      encode_slab(&m.aq2, p, Slab::AQ2, BF, 2, C, 2 * C, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
      encode_slab(&m.u, p, Slab::U, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, V, C, LY::VTK,
                  CU_TENSOR_MAP_SWIZZLE_NONE) &&
      encode_slab(&m.qb2, p, Slab::QB2, BF, 2, K, 2 * C, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
      encode_slab(&m.kb2, p, Slab::KB2, BF, 2, K, 2 * C, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return GDR_ERR_CUDA;
  auto kern = state_kda_kernel<MG>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::TOTAL) !=
      cudaSuccess)
    return GDR_ERR_CUDA;
  dim3 grid(V / LY::VTK, p.HV, p.B);
  kern<<<grid, MG * kda::WARPS * 32, LY::TOTAL, stream>>>(m, p);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
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
  if (p.gate_mode) return launch_kda<KDA_MG>(p, stream);
  // Scalar gate: the fused chain + output launch when the chains leave SMs
  // for the outputs, else chain and outputs in the same CTAs.
  const gdr_status st = launch_recur(p, stream);
  return st == GDR_ERR_UNSUPPORTED ? launch_ws(p, stream) : st;
}

}  // namespace fast
}  // namespace gdr
