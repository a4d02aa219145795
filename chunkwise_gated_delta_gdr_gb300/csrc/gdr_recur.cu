// gdr_recur.cu -- inter-chunk recurrence of the fast path for the scalar gate
// (Gated DeltaNet): the state chain and the chunk outputs in one launch.
//
// Per chunk n the inter-chunk recurrence of the "分块并行计算（Chunkwise）" notes
// (section "chunk 间递推") reads
//     r_n     = U_n - W_n S_n
//     o_n     = (q exp(G)) S_n + A_qk r_n
//     S_{n+1} = exp(G_last) S_n + (exp(G_last - G) k)^T (beta r_n)
// Only the S update is serial: o_n needs S_n and r_n, and nothing needs o_n.
// The launch therefore gives the SMs one of two roles.
//
//  * Chain CTAs, one per (batch, value head, 16-column V tile), keep S^T in
//    fp32 registers for the whole sequence and run r and the S update on
//    mma.sync m16n8k16 (bf16 hi / lo split operands, fp32 accumulation):
//        r^T  = U^T - S^T W^T                  (16 x 64,  K = 128)
//        S^T <- gamma S^T + (kscale r)^T k     (16 x 128, K = 64)
//    Each chunk they publish S_n^T and r_n^T (bf16 hi / lo planes) as
//    128-byte swizzled shared-memory tiles, which also feed their own
//    ldmatrix reads; a copy warp writes them to the chunk's exchange block in
//    global memory and a flag warp raises a per-chain progress flag.
//  * Output CTAs, on the SMs the chains leave free, take (chunk, head, V half)
//    items in chunk order, wait for the flags of the four chains that cover
//    the half, stage q, A_qk and the published tiles by TMA and form
//        o = diag(qscale) (q S) + A_qk r
//    as two tcgen05 accumulators (M = 64 chunk rows, N = 64 value columns) in
//    TMEM, double-buffered so that one item's epilogue overlaps the next
//    item's MMAs; o leaves through a TMA store.
//
// A chain CTA's chunk step is bound by shared-memory bandwidth (ldmatrix
// fragments and TMA fills). Taking the output products off the chain SMs
// removes about 40% of that traffic from the serial path and puts the SMs
// the chains do not use to work.
//
// Output CTAs wait on flags that chain CTAs of the same launch set, so both
// roles go in one cooperative launch (all CTAs co-resident); launch_recur
// declines (GDR_ERR_UNSUPPORTED, nothing enqueued) when the chains would not
// leave enough SMs for the outputs, and the caller runs the single-role state
// kernel instead. Every wait is bounded: one that gives up records a code in
// the workspace error word and the kernel still runs to completion.
#include <string.h>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdr_fast.cuh"
#include "gdr_ptx.cuh"
#include "gdr_tmap.cuh"

namespace gdr {
namespace fast {
namespace {

using namespace ptx;

constexpr int VTILES = V / VT;          // chains per sequence
constexpr int THREADS = 256;            // 8 warps in either role
constexpr int LDA = C + 8;              // bf16 row stride of the rho^T tile (144 B)
constexpr long kWaitLimit = 1L << 24;   // mbarrier polls before a wait gives up
constexpr long kFlagLimit = 1L << 24;   // flag polls (64 ns apart) before a wait gives up
constexpr unsigned int kErrChainWait = 4u, kErrOutputWait = 8u;

// ------------------------------------------------------------------ chain role
// Warps 0-3 carry the state: warp w owns state channels [32 w, 32 w + 32) and
// r^T columns [16 w, 16 w + 16). Warp 4 issues the TMA loads (the SM's TMA
// unit is busy with them; the published tiles leave through plain stores of
// warp 5). Warp 6 raises the chain's flag: a GPU-scope release costs about as
// much as a chunk step, so it runs apart from the copies and covers all
// chunks copied since its previous release. Warp 7 (gate) confirms each
// chunk's operand stage ahead of the chain warps.
namespace ch {
constexpr int CW = 4;
static_assert(K / 32 == CW && C / 16 == CW, "one channel pair and one j-step of 16 per chain warp");
// Operand stage (three-deep ring): -W hi, -W lo and the chunk's k rows
// ([64][128] bf16, two 128-byte swizzled 8 KB boxes each), the U tile [64][16]
// fp32 and VEC (qscale, kscale, gamma).
constexpr int W_HI = 0, W_LO = 16384, KT = 32768, U = 49152, VEC = 53248, STAGE = 55296;
constexpr uint32_t TX = 32768 + 16384 + 4096 + 1024;
constexpr int NST = 3;
// Published tiles (NXB buffers), 128-byte swizzled: S^T hi, lo as two
// [16 v][64 k] boxes each; r^T hi, lo as one [16 v][64 j] box each. rho^T
// (chain-internal) is a padded [2][16][LDA] bf16 tile.
constexpr int XS_BUF = 2 * 2 * 2048, XR_BUF = 2 * 2048, XP_BYTES = 2 * 16 * LDA * 2;
constexpr int NXB = 4;                     // published-tile buffers
constexpr int XS = NST * STAGE, XR = XS + NXB * XS_BUF, XP = XR + NXB * XR_BUF, BAR = XP + XP_BYTES;
constexpr int DONE = BAR + 2 * NST * 8;     // chunks copied out (u32)
constexpr int BYTES = DONE + 16;
constexpr int SYNC = CW * 32 + 32;         // chain warps + copy warp
// Named barriers: 1 chain warps (S^T complete); BAR_R chain warps + gate warp
// (r^T complete, and the next chunk's operands are in their stage); BAR_XS + s
// S^T of buffer s published; BAR_XR + s r^T of buffer s published; BAR_CP + s
// buffer s copied out (s < NXB).
constexpr int BAR_XS = 2, BAR_XR = BAR_XS + NXB, BAR_CP = BAR_XR + NXB, BAR_R = BAR_CP + NXB;
static_assert(BAR_R < 16, "named barrier ids");
constexpr int GATE_SYNC = CW * 32 + 32;     // chain warps + gate warp
}  // namespace ch

// ----------------------------------------------------------------- output role
// Warp 0 issues the TMA loads, warp 1 the MMAs (and owns the TMEM), warps 2-5
// run the epilogue (warp w may read TMEM lanes [32 (w % 4), 32 (w % 4) + 32)),
// warps 6 and 7 have no work.
namespace ou {
// Operand stage (double-buffered), 128-byte swizzled K-major tiles: q [64 i]
// [128 k] (two boxes), A_qk hi / lo [64 i][64 j], S^T hi / lo [64 v][128 k]
// (two boxes each), r^T hi / lo [64 v][64 j].
constexpr int Q = 0, AQ_HI = 16384, AQ_LO = 24576, S_HI = 32768, S_LO = 49152, R_HI = 65536,
              R_LO = 73728, STAGE = 81920;
constexpr uint32_t TX = STAGE;
constexpr int OST_BYTES = 16384;           // output staging [64 i][64 v], double-buffered
constexpr int OST = 2 * STAGE, BAR = OST + 2 * OST_BYTES;
constexpr int BYTES = BAR + 8 * 8 + 16;
constexpr int TMEM_COLS = 256;             // 2 x (q S: 64 columns, A_qk r: 64 columns)
constexpr int EPI = 128;                   // epilogue threads
}  // namespace ou

constexpr int SMEM_BYTES = (ch::BYTES > ou::BYTES ? ch::BYTES : ou::BYTES) + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory plan too large");
static_assert(ou::OST % 1024 == 0 && ou::STAGE % 1024 == 0 && ch::XS % 1024 == 0 &&
                  ch::XR % 1024 == 0 && ch::STAGE % 1024 == 0,
              "swizzled tiles need 1 KB alignment");

struct Maps {
  CUtensorMap k, w2, u;                  // chain role
  CUtensorMap q, aq2, xs, xr, out;       // output role
};

__device__ __forceinline__ void nb_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void nb_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Byte address of element (r, c) (c a multiple of 8) of a swizzled bf16 tile
// stored as 64-column boxes of 8 KB.
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int r, int c) {
  return base + (uint32_t)((c >> 6) * 8192 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4));
}
// Same for a 16-row tile stored as 64-column boxes of 2 KB; any even c.
__device__ __forceinline__ uint32_t tile16_off(int r, int c) {
  return (uint32_t)((c >> 6) * 2048 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}

// ============================================================================ chain
__device__ __forceinline__ void chain_role(const Maps& maps, const Params& p, uint8_t* sm,
                                           int cta) {
  using namespace ch;
  const int vt = cta % VTILES, seq = cta / VTILES;
  const int b = seq / p.HV, hv = seq % p.HV, h = hv / (p.HV / p.H);
  const int v0 = vt * VT;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int chunk0 = seq * p.N;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + BAR);
  uint64_t* empty = full + NST;
  unsigned int* done = reinterpret_cast<unsigned int*>(sm + DONE);

  if (tid == 0) {
    *done = 0;
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], CW);
    }
    mbar_fence_init();
  }
  __syncthreads();
  bool ok = true;

  if (warp == CW) {
    // ------------------------------------------------------------ TMA producer
    // Stage s = n % NST is refilled with chunk n once the chain warps released
    // chunk n - NST from it (completion n / NST - 1 of empty[s]).
    if (lane == 0) {
      for (int n = 0; n < p.N; ++n) {
        const int s = n % NST, idx = chunk0 + n;
        if (n >= NST) ok = ok && mbar_wait(&empty[s], (n / NST - 1) & 1, kWaitLimit);
        if (!ok) break;
        const uint32_t base = smem_u32(sm + s * STAGE);
        mbar_expect_tx(&full[s], p.ssd ? TX - 32768 : TX);
        if (!p.ssd) {                                  // SSD: W = 0, not loaded
          tma_load3(base + W_HI, &maps.w2, 0, 0, idx, &full[s]);
          tma_load3(base + W_HI + 8192, &maps.w2, 64, 0, idx, &full[s]);
          tma_load3(base + W_LO, &maps.w2, 0, 64, idx, &full[s]);
          tma_load3(base + W_LO + 8192, &maps.w2, 64, 64, idx, &full[s]);
        }
        tma_load4(base + KT, &maps.k, 0, h, n * C, b, &full[s]);
        tma_load4(base + KT + 8192, &maps.k, 64, h, n * C, b, &full[s]);
        tma_load3(base + U, &maps.u, v0, 0, idx, &full[s]);
        bulk_load(base + VEC, p.slabs + (size_t)idx * p.slab_bytes + Slab::VEC, 1024, &full[s]);
      }
    }
  } else if (warp == CW + 1) {
    // -------------------------------------------------------------- copy-out
    // Shared-memory loads first, then the global stores (the loads must not
    // queue behind possibly aliasing stores). Row r of a published tile keeps
    // its 16-byte chunk c at chunk c ^ (r % 8); the exchange block is plain.
    for (int n = 0; n < p.N; ++n) {
      const int s = n % NXB;
      uint8_t* blk = p.xchg + (size_t)(chunk0 + n) * Xchg::BYTES;
      nb_sync(BAR_XS + s, SYNC);
      const uint8_t* xs = sm + XS + s * XS_BUF;
      uint4 val[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {                   // 2 planes x 16 rows x 16 chunks
        const int u = lane + 32 * i, pl = u >> 8, row = (u >> 4) & 15, c = u & 15;
        val[i] = *reinterpret_cast<const uint4*>(xs + pl * 4096 + (c >> 3) * 2048 + row * 128 +
                                                 (((c & 7) ^ (row & 7)) << 4));
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int u = lane + 32 * i, pl = u >> 8, row = (u >> 4) & 15, c = u & 15;
        *reinterpret_cast<uint4*>(blk + Xchg::S_HI + pl * (Xchg::S_LO - Xchg::S_HI) +
                                  (size_t)(v0 + row) * (K * 2) + c * 16) = val[i];
      }
      nb_sync(BAR_XR + s, SYNC);
      const uint8_t* xr = sm + XR + s * XR_BUF;
#pragma unroll
      for (int i = 0; i < 8; ++i) {                    // 2 planes x 16 rows x 8 chunks
        const int u = lane + 32 * i, pl = u >> 7, row = (u >> 3) & 15, c = u & 7;
        val[i] = *reinterpret_cast<const uint4*>(xr + pl * 2048 + row * 128 + ((c ^ (row & 7)) << 4));
      }
      nb_arrive(BAR_CP + s, SYNC);                          // buffer s read: it may be overwritten
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int u = lane + 32 * i, pl = u >> 7, row = (u >> 3) & 15, c = u & 7;
        *reinterpret_cast<uint4*>(blk + Xchg::R_HI + pl * (Xchg::R_LO - Xchg::R_HI) +
                                  (size_t)(v0 + row) * (C * 2) + c * 16) = val[i];
      }
      __syncwarp();                                    // orders the lanes' stores before:
      if (lane == 0) st_release_cta_shared(done, (unsigned int)(n + 1));
    }
  } else if (warp == CW + 2) {
    // ------------------------------------------------------------------- flag
    // The chain's flag counts its chunks whose tiles are in global memory.
    if (lane == 0) {
      unsigned int* flag = p.flags + (size_t)seq * VTILES + vt;
      unsigned int raised = 0;
      long idle = 0;
      while (raised < (unsigned int)p.N) {
        const unsigned int d = ld_acquire_cta_shared(done);
        if (d > raised) {
          fence_async_global();
          red_max_release_gpu(flag, d);
          raised = d;
          idle = 0;
        } else {
          if (++idle >= kFlagLimit) {
            ok = false;
            break;
          }
          __nanosleep(32);
        }
      }
    }
  } else if (warp == CW + 3) {
    // ------------------------------------------------------------------- gate
    // Joins the chain warps' r^T barrier of step n once chunk n + 1's operands
    // are in their stage: the chain warps then start step n + 1 without
    // testing the stage's barrier themselves (the test costs about as much as
    // a barrier). It joins every generation, also after a wait gave up.
    for (int n = 0; n < p.N; ++n) {
      if (n + 1 < p.N && lane == 0)
        ok = ok && mbar_wait(&full[(n + 1) % NST], ((n + 1) / NST) & 1, kWaitLimit);
      __syncwarp();
      nb_sync(BAR_R, GATE_SYNC);
    }
  } else {
    // ------------------------------------------------------------ chain warps
    const int jw = 16 * warp, cw = 32 * warp;          // r^T j-tiles, state channels
    const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = (lane >> 4) * 8;
    const int brow = lane & 7, bcol = (lane >> 3) * 8;
    const int kcol = cw + (lane >> 4) * 8;
    __nv_bfloat16* xp_hi = reinterpret_cast<__nv_bfloat16*>(sm + XP);
    __nv_bfloat16* xp_lo = xp_hi + 16 * LDA;
    float S[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int c = cw + 8 * nt + 2 * t4;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int vv = g + (e >> 1) * 8, cc = c + (e & 1);
        S[nt][e] = p.s0 ? p.s0[((size_t)seq * K + cc) * V + v0 + vv] : 0.f;
      }
    }
    for (int n = 0; n < p.N; ++n) {
      const int s = n % NXB, st = n % NST;             // published-tile buffer, operand stage
      uint8_t* cb = sm + st * STAGE;
      const uint32_t w_hi = smem_u32(cb + W_HI), w_lo = smem_u32(cb + W_LO);
      const uint32_t k_t = smem_u32(cb + KT);
      const float* su = reinterpret_cast<const float*>(cb + U);
      const float* ks = reinterpret_cast<const float*>(cb + VEC) + C;
      const float* gam = ks + C;
      uint8_t* xsh = sm + XS + s * XS_BUF;             // S^T hi; lo at + 4096
      uint8_t* xrh = sm + XR + s * XR_BUF;             // r^T hi; lo at + 2048
      if (n >= NXB) nb_sync(BAR_CP + s, SYNC);              // chunk n - NXB copied out of buffer s
      // S^T hi / lo by stmatrix: matrix i of call q is channel tile 2 q + i / 2,
      // value rows 8 (i % 2) .. + 8. The registers stored are also this warp's
      // A fragments of its own two k-steps (channels cw + 16 q ...) of the r
      // products, which therefore run before the barrier.
      uint32_t oah[2][4], oal[2][4];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        split_pair(S[2 * q][0], S[2 * q][1], oah[q][0], oal[q][0]);
        split_pair(S[2 * q][2], S[2 * q][3], oah[q][1], oal[q][1]);
        split_pair(S[2 * q + 1][0], S[2 * q + 1][1], oah[q][2], oal[q][2]);
        split_pair(S[2 * q + 1][2], S[2 * q + 1][3], oah[q][3], oal[q][3]);
        const int mi = lane >> 3;
        const uint32_t a = smem_u32(xsh) + tile16_off(8 * (mi & 1) + (lane & 7), cw + 16 * q + 8 * (mi >> 1));
        stsm_x4(a, oah[q][0], oah[q][1], oah[q][2], oah[q][3]);
        stsm_x4(a + 4096, oal[q][0], oal[q][1], oal[q][2], oal[q][3]);
      }
      if (n == 0) ok = ok && mbar_wait(&full[st], 0, kWaitLimit);   // later chunks: the gate warp
      // r^T = U^T + S^T (-W)^T, j in [jw, jw + 16)
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
      if (!p.ssd) {                                    // SSD: r = U
        // This warp's own channels (k-steps 2 warp, 2 warp + 1) from registers.
#pragma unroll
        for (int jt = 0; jt < 2; ++jt) {
          uint32_t wh[4], wl[4];
          ldsm_x4(wh, tile_addr(w_hi, jw + 8 * jt + brow, cw + bcol));
          ldsm_x4(wl, tile_addr(w_lo, jw + 8 * jt + brow, cw + bcol));
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            mma_bf16_16816(Rhh[jt], oah[h2], wh[2 * h2], wh[2 * h2 + 1]);
            mma_bf16_16816(Rlh[jt], oal[h2], wh[2 * h2], wh[2 * h2 + 1]);
            mma_bf16_16816(Rhl[jt], oah[h2], wl[2 * h2], wl[2 * h2 + 1]);
          }
        }
      }
      nb_sync(1, CW * 32);                             // S^T complete
      nb_arrive(BAR_XS + s, SYNC);
      if (!p.ssd) {
        // The other warps' channels, from the published S^T.
#pragma unroll
        for (int kp = 1; kp < CW; ++kp) {
          const int ks2 = 2 * ((warp + kp) & (CW - 1));
          uint32_t ah[2][4], al[2][4];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            ldsm_x4(ah[h2], smem_u32(xsh) + tile16_off(arow, 16 * (ks2 + h2) + acol));
            ldsm_x4(al[h2], smem_u32(xsh) + 4096 + tile16_off(arow, 16 * (ks2 + h2) + acol));
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
      }
      float Dl[4][4];
      {
        // r^T and rho^T = (kscale r)^T hi / lo by stmatrix: matrix i is j tile
        // i / 2, value rows 8 (i % 2) .. + 8.
        uint32_t rh[4], rl[4], ph[4], pl[4];
#pragma unroll
        for (int jt = 0; jt < 2; ++jt) {
          const int j = jw + 8 * jt + 2 * t4;
          float R[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) R[e] = Rhh[jt][e] + (Rlh[jt][e] + Rhl[jt][e]);
          const float k0 = ks[j], k1 = ks[j + 1];
          split_pair(R[0], R[1], rh[2 * jt], rl[2 * jt]);
          split_pair(R[2], R[3], rh[2 * jt + 1], rl[2 * jt + 1]);
          split_pair(R[0] * k0, R[1] * k1, ph[2 * jt], pl[2 * jt]);
          split_pair(R[2] * k0, R[3] * k1, ph[2 * jt + 1], pl[2 * jt + 1]);
        }
        const int mi = lane >> 3, row = 8 * (mi & 1) + (lane & 7), col = jw + 8 * (mi >> 1);
        const uint32_t a = smem_u32(xrh) + tile16_off(row, col);
        stsm_x4(a, rh[0], rh[1], rh[2], rh[3]);
        stsm_x4(a + 2048, rl[0], rl[1], rl[2], rl[3]);
        const uint32_t b = smem_u32(xp_hi + row * LDA + col);
        stsm_x4(b, ph[0], ph[1], ph[2], ph[3]);
        stsm_x4(b + 16 * LDA * 2, pl[0], pl[1], pl[2], pl[3]);
        // S^T = gamma S^T + rho^T k, c in [cw, cw + 32); the scalar gate's decay
        // gamma is the same on every channel. ph / pl are also this warp's A
        // fragments of its own k-step (j in [jw, jw + 16)), taken before the barrier.
        const float gm = gam[0];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            S[nt][e] *= gm;
            Dl[nt][e] = 0.f;
          }
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          uint32_t kh[4];
          ldsm_x4_t(kh, tile_addr(k_t, jw + arow, kcol + 16 * np));
          mma_bf16_16816(S[2 * np], ph, kh[0], kh[1]);
          mma_bf16_16816(S[2 * np + 1], ph, kh[2], kh[3]);
          mma_bf16_16816(Dl[2 * np], pl, kh[0], kh[1]);
          mma_bf16_16816(Dl[2 * np + 1], pl, kh[2], kh[3]);
        }
      }
      nb_sync(BAR_R, GATE_SYNC);                       // r^T, rho^T complete; chunk n + 1 in place
      nb_arrive(BAR_XR + s, SYNC);
      // The other warps' j-steps, from the published rho^T.
#pragma unroll
      for (int kp = 1; kp < CW; ++kp) {
        const int kk = (warp + kp) & (CW - 1);
        uint32_t ph[4], pl[4];
        ldsm_x4(ph, smem_u32(xp_hi + arow * LDA + 16 * kk + acol));
        ldsm_x4(pl, smem_u32(xp_lo + arow * LDA + 16 * kk + acol));
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          uint32_t kh[4];
          ldsm_x4_t(kh, tile_addr(k_t, 16 * kk + arow, kcol + 16 * np));
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
      if (lane == 0) mbar_arrive(&empty[st]);          // this warp is done with stage st
    }
    // Balance the copy-out barrier generations of the last NXB chunks.
    for (int n = (p.N >= NXB ? p.N - NXB : 0); n < p.N; ++n) nb_sync(BAR_CP + n % NXB, SYNC);
    if (p.sT) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int c = cw + 8 * nt + 2 * t4;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int vv = g + (e >> 1) * 8, cc = c + (e & 1);
          p.sT[((size_t)seq * K + cc) * V + v0 + vv] = S[nt][e];
        }
      }
    }
  }
  if (!ok) atomicOr(p.error_word, kErrChainWait);
}

// =========================================================================== output
__device__ __forceinline__ void output_role(const Maps& maps, const Params& p, uint8_t* sm,
                                            int ob, int n_out) {
  using namespace ou;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + BAR);
  uint64_t* empty = full + 2;
  uint64_t* afull = full + 4;
  uint64_t* aempty = full + 6;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(full + 8);
  const int nseq = p.B * p.HV;
  const int n_items = nseq * p.N * 2;
  // Item it: V half it & 1 of sequence (it >> 1) % nseq, chunk (it >> 1) / nseq.

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&afull[i], 1);
      mbar_init(&aempty[i], 4);
    }
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tslot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int li = 0;
      for (int it = ob; it < n_items; it += n_out, ++li) {
        const int vh = it & 1, seq = (it >> 1) % nseq, n = (it >> 1) / nseq;
        const int b = seq / p.HV, hv = seq % p.HV, h = hv / (p.HV / p.H);
        const int s = li & 1, idx = seq * p.N + n;
        if (li >= 2) ok = ok && mbar_wait(&empty[s], ((li >> 1) - 1) & 1, kWaitLimit);
        const unsigned int* fl = p.flags + (size_t)seq * VTILES + (VTILES / 2) * vh;
        for (int j = 0; j < VTILES / 2 && ok; ++j) {
          long polls = 0;
          while (ld_acquire_gpu(fl + j) < (unsigned int)(n + 1)) {
            if (++polls >= kFlagLimit) {
              ok = false;
              break;
            }
            __nanosleep(64);
          }
        }
        if (!ok) break;
        fence_async_global();                          // published tiles -> TMA reads
        const uint32_t base = smem_u32(sm + s * STAGE);
        mbar_expect_tx(&full[s], TX);
        tma_load4(base + Q, &maps.q, 0, h, n * C, b, &full[s]);
        tma_load4(base + Q + 8192, &maps.q, 64, h, n * C, b, &full[s]);
        tma_load3(base + AQ_HI, &maps.aq2, 0, 0, idx, &full[s]);
        tma_load3(base + AQ_LO, &maps.aq2, 0, C, idx, &full[s]);
        tma_load3(base + S_HI, &maps.xs, 0, 64 * vh, idx, &full[s]);
        tma_load3(base + S_HI + 8192, &maps.xs, 64, 64 * vh, idx, &full[s]);
        tma_load3(base + S_LO, &maps.xs, 0, V + 64 * vh, idx, &full[s]);
        tma_load3(base + S_LO + 8192, &maps.xs, 64, V + 64 * vh, idx, &full[s]);
        tma_load3(base + R_HI, &maps.xr, 0, 64 * vh, idx, &full[s]);
        tma_load3(base + R_LO, &maps.xr, 0, V + 64 * vh, idx, &full[s]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    // Accumulator s: columns [128 s, 128 s + 64) = q S, [128 s + 64, 128 s + 128)
    // = A_qk r, both with the chunk row i in TMEM lane 32 (i / 16) + i % 16.
    if (lane == 0) {
      constexpr uint32_t ID = idesc_bf16_kk(64, 64);
      int li = 0;
      for (int it = ob; it < n_items; it += n_out, ++li) {
        const int s = li & 1;
        ok = ok && mbar_wait(&full[s], (li >> 1) & 1, kWaitLimit);
        if (li >= 2) ok = ok && mbar_wait(&aempty[s], ((li >> 1) - 1) & 1, kWaitLimit);
        if (!ok) break;
        tc_fence_after();
        const uint32_t base = smem_u32(sm + s * STAGE);
        const uint32_t d_qs = tmem + s * 128, d_ar = d_qs + 64;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
          umma_bf16(d_qs, sdesc_sw128(base + Q + off), sdesc_sw128(base + S_HI + off), ID, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
          umma_bf16(d_qs, sdesc_sw128(base + Q + off), sdesc_sw128(base + S_LO + off), ID, 1);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t off = kk * 32;
          umma_bf16(d_ar, sdesc_sw128(base + AQ_HI + off), sdesc_sw128(base + R_HI + off), ID,
                    kk > 0);
          umma_bf16(d_ar, sdesc_sw128(base + AQ_LO + off), sdesc_sw128(base + R_HI + off), ID, 1);
          umma_bf16(d_ar, sdesc_sw128(base + AQ_HI + off), sdesc_sw128(base + R_LO + off), ID, 1);
        }
        umma_commit(&empty[s]);                        // operand stage s free
        umma_commit(&afull[s]);                        // accumulator s ready
      }
    }
  } else if (warp < 6) {
    // --------------------------------------------------------------- epilogue
    const int quad = warp & 3;
    const int i = 16 * quad + (lane & 15);             // chunk row (lanes 0-15 hold it)
    const int et = tid - 64;                           // 0 .. 127
    int li = 0;
    for (int it = ob; it < n_items; it += n_out, ++li) {
      const int vh = it & 1, seq = (it >> 1) % nseq, n = (it >> 1) / nseq;
      const int b = seq / p.HV, hv = seq % p.HV;
      const int s = li & 1, idx = seq * p.N + n;
      const float qs =
          reinterpret_cast<const float*>(p.slabs + (size_t)idx * p.slab_bytes + Slab::VEC)[i];
      if (et == 0) bulk_wait_read<1>();                // store of item li - 2 left buffer s
      nb_sync(1, EPI);
      ok = ok && mbar_wait(&afull[s], (li >> 1) & 1, kWaitLimit);
      tc_fence_after();
      uint8_t* ost = sm + OST + s * OST_BYTES;
      const uint32_t taddr = tmem + ((uint32_t)(32 * quad) << 16) + s * 128;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float dq[32], da[32];
        tmem_ld32(taddr + 32 * hh, dq);
        tmem_ld32(taddr + 64 + 32 * hh, da);
        if (lane < 16) {
          if (p.out_bf16) {
            // one [64][64] bf16 box: 16-byte chunk 4 hh + c of row i
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint4 pk;
              pk.x = pack_bf16(fmaf(dq[8 * c + 0], qs, da[8 * c + 0]), fmaf(dq[8 * c + 1], qs, da[8 * c + 1]));
              pk.y = pack_bf16(fmaf(dq[8 * c + 2], qs, da[8 * c + 2]), fmaf(dq[8 * c + 3], qs, da[8 * c + 3]));
              pk.z = pack_bf16(fmaf(dq[8 * c + 4], qs, da[8 * c + 4]), fmaf(dq[8 * c + 5], qs, da[8 * c + 5]));
              pk.w = pack_bf16(fmaf(dq[8 * c + 6], qs, da[8 * c + 6]), fmaf(dq[8 * c + 7], qs, da[8 * c + 7]));
              *reinterpret_cast<uint4*>(ost + i * 128 + (((4 * hh + c) ^ (i & 7)) << 4)) = pk;
            }
          } else {
            // box hh: [64][32] fp32, 16-byte chunk c of row i
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              float4 v4;
              v4.x = fmaf(dq[4 * c + 0], qs, da[4 * c + 0]);
              v4.y = fmaf(dq[4 * c + 1], qs, da[4 * c + 1]);
              v4.z = fmaf(dq[4 * c + 2], qs, da[4 * c + 2]);
              v4.w = fmaf(dq[4 * c + 3], qs, da[4 * c + 3]);
              *reinterpret_cast<float4*>(ost + hh * 8192 + i * 128 + ((c ^ (i & 7)) << 4)) = v4;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&aempty[s]);          // accumulator s read
      fence_async_shared();
      nb_sync(1, EPI);                                 // staging tile complete
      if (et == 0) {
        const uint32_t src = smem_u32(ost);
        tma_store4(&maps.out, src, 64 * vh, hv, n * C, b);
        if (!p.out_bf16) tma_store4(&maps.out, src + 8192, 64 * vh + 32, hv, n * C, b);
        bulk_commit();
      }
    }
    if (et == 0) bulk_wait<0>();
  }
  if (!ok) atomicOr(p.error_word, kErrOutputWait);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

__global__ void __launch_bounds__(THREADS, 1)
    recur_kernel(const __grid_constant__ Maps maps, Params p, int n_chain, int n_out) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  if ((int)blockIdx.x < n_chain)
    chain_role(maps, p, sm, blockIdx.x);
  else
    output_role(maps, p, sm, blockIdx.x - n_chain, n_out);
}

struct DeviceInfo {
  int sms = 0;
  bool coop = false;
};

DeviceInfo device_info() {
  static DeviceInfo cache[64];
  static bool known[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return DeviceInfo{};
  if (dev < 64 && known[dev]) return cache[dev];
  DeviceInfo d;
  int coop = 0;
  cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  d.coop = coop != 0;
  if (dev < 64) {
    cache[dev] = d;
    known[dev] = true;
  }
  return d;
}

}  // namespace

gdr_status launch_recur(const Params& p, cudaStream_t stream) {
  if (!p.xchg || !p.flags || p.gate_mode != 0) return GDR_ERR_UNSUPPORTED;
  const int nseq = p.B * p.HV;
  const long long items = 2LL * nseq * p.N;
  const DeviceInfo dev = device_info();
  int n_chain = nseq * VTILES, n_out = 0;
  bool coop = false;
  if (p.recur_mode == 1) {
    // Chains only: they wait on nothing, so any number may run, in waves.
  } else if (p.recur_mode == 2) {
    // Outputs only, on every SM: the flags of the previous chains-only launch
    // are final, so no output CTA waits for long.
    n_chain = 0;
    n_out = (int)(items < dev.sms ? items : dev.sms);
  } else {
    // The outputs need at least an eighth as many SMs as the chains (and 8).
    const int spare = dev.sms - n_chain;
    if (!dev.coop || spare < 8 || spare * 8 < n_chain) return GDR_ERR_UNSUPPORTED;
    n_out = (int)(items < spare ? items : spare);
    coop = true;
  }

  Maps m;
  memset(&m, 0, sizeof m);
  const size_t nch = (size_t)nseq * p.N;
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  const int es = p.out_bf16 ? 2 : 4;
  const cuuint64_t od[4] = {(cuuint64_t)V, (cuuint64_t)p.HV, (cuuint64_t)p.T, (cuuint64_t)p.B};
  const cuuint64_t os[3] = {(cuuint64_t)V * es, (cuuint64_t)p.HV * V * es,
                            (cuuint64_t)p.T * p.HV * V * es};
  const cuuint32_t obox[4] = {p.out_bf16 ? 64u : 32u, 1, 64, 1};
  const bool ok =
      tmap_bthd(&m.k, p.k, p.B, p.T, p.H) && tmap_bthd(&m.q, p.q, p.B, p.T, p.H) &&
      tmap_blocks(&m.w2, p.slabs + Slab::W2, BF, 2, K, 2 * C, nch, p.slab_bytes, 64, 64, SW) &&
      tmap_blocks(&m.aq2, p.slabs + Slab::AQ2, BF, 2, C, 2 * C, nch, p.slab_bytes, 64, 64, SW) &&
      tmap_blocks(&m.u, p.slabs + Slab::U, F32, 4, V, C, nch, p.slab_bytes, VT, 64,
                  CU_TENSOR_MAP_SWIZZLE_NONE) &&
      tmap_blocks(&m.xs, p.xchg + Xchg::S_HI, BF, 2, K, 2 * V, nch, Xchg::BYTES, 64, 64, SW) &&
      tmap_blocks(&m.xr, p.xchg + Xchg::R_HI, BF, 2, C, 2 * V, nch, Xchg::BYTES, 64, 64, SW) &&
      tmap_encode(&m.out, p.out_bf16 ? BF : F32, 4, p.out, od, os, obox, SW);
  if (!ok) return GDR_ERR_CUDA;
  if (cudaFuncSetAttribute(recur_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SMEM_BYTES) != cudaSuccess)
    return GDR_ERR_CUDA;
  if (!p.zero_flags && p.recur_mode != 2 &&
      cudaMemsetAsync(p.flags, 0, (size_t)nseq * VTILES * sizeof(unsigned int), stream) !=
          cudaSuccess)
    return GDR_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_chain + n_out);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = coop ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, recur_kernel, m, p, n_chain, n_out);
  if (e == cudaSuccess) return GDR_OK;
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    (void)cudaGetLastError();
    return GDR_ERR_UNSUPPORTED;
  }
  return GDR_ERR_CUDA;
}

}  // namespace fast
}  // namespace gdr
