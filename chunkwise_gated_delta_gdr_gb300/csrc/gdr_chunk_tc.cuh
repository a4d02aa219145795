// gdr_chunk_tc.cuh -- the chunk-local stage of the fast path (scalar gate) as a
// device function, shared by the chunk kernel (gdr_chunk_tc.cu) and the
// worker CTAs of the one-launch forward (gdr_chain.cu). gdr_chunk_tc.cu has
// the description of what it computes.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "gdr_fast.cuh"
#include "gdr_ptx.cuh"
#include "gdr_tmap.cuh"
#include "gdr_trinv.cuh"

namespace gdr {
namespace fast {
namespace chunk {

using namespace ptx;

constexpr int THREADS = 256;            // one group of 8 warps per chunk
constexpr uint32_t TMEM_COLS = 256;
constexpr long kWaitLimit = 1L << 24;   // bounded spin: ~tens of ms, then error word
constexpr unsigned int kErrTmaWait = 1u, kErrMmaWait = 2u;
constexpr float kSplitSpan = 80.f;      // |G_i - G_m| bound of the split decays

// Shared-memory map of one group (bytes from a 1024-aligned base).
constexpr int OFF_K0 = 0;          // k cols 0-63   (8 KB, 128-byte swizzle, from TMA)
constexpr int OFF_Q0 = 8192;       // q cols 0-63
constexpr int OFF_K1 = 16384;      // k cols 64-127
constexpr int OFF_Q1 = 24576;      // q cols 64-127
constexpr int OFF_V0 = 32768;      // v cols 0-63
constexpr int OFF_V1 = 40960;      // v cols 64-127
constexpr int LDL = 68;            // fp32 row stride of L (272 B: float4 rows, conflict-free)
constexpr int OFF_L = 49152;       // L [64][LDL] fp32; later XW (16 KB)
constexpr int OFF_AQS = 66560;     // A_qk hi / lo staging, one stacked swizzled [128][64] bf16 box
constexpr int OFF_XU = 65536;      // XU (16 KB), written once L and the A_qk staging are dead
constexpr int LDX = 68;            // fp32 row stride of X
constexpr int OFF_X = 84992;       // X = (I + L)^-1 [64][LDX] fp32
constexpr int OFF_T = 8192;        // block-product scratch [32][36] fp32 (in the dead q tile)
constexpr int OFF_KP = 86016;      // previous chunk's k tile (16 KB), in the dead X region;
                                   // later the -T hi / lo staging box
constexpr int OFF_SMALL = 102400;  // G, nq, nk, beta, column factor (5 x 64 fp32)
constexpr int OFF_BAR = 103680;    // mbarriers + TMEM slot
constexpr int GROUP_BYTES = 104448;            // one group's region (1 KB multiple)
constexpr int SMEM_BYTES = GROUP_BYTES + 1024;  // + alignment slack
// Epilogue-2 staging (after the W / U MMAs, over the dead operand tiles):
// -W as two stacked [128][64] bf16 boxes (column halves); U as four swizzled
// [64][32] fp32 boxes.
constexpr int OFF_WS = 0;
constexpr int OFF_US = 32768;
static_assert(OFF_AQS % 1024 == 0 && OFF_AQS + 16384 <= OFF_X, "A_qk staging placement");
static_assert(OFF_XU + 16384 <= OFF_X && OFF_US + 32768 <= OFF_X, "staging overlaps X");
static_assert(OFF_X + 64 * LDX * 4 <= OFF_SMALL, "X overlaps");
static_assert(OFF_T + 32 * 36 * 4 <= OFF_K1, "scratch overlaps the k tile");
static_assert(OFF_BAR + 64 <= GROUP_BYTES, "group region");
static_assert(OFF_KP % 1024 == 0 && OFF_KP >= OFF_X && OFF_KP + 16384 <= OFF_SMALL,
              "previous k tile inside the dead X region");
// mbarriers at OFF_BAR (the caller initialises them, count 1 each): +0 k and q
// tiles, +8 MMAs, +16 TMEM slot and split flag (not a barrier), +24 v tiles,
// +32 previous chunk's k tile, +40 the T product.
constexpr int kNumBars = 6;

struct Maps {
  CUtensorMap q, k, v;          // [B, T, heads, 128] bf16 inputs
};

// Initialises the mbarriers of a group region (one thread, then an
// mbarrier-init fence; the group barrier that follows orders it before use).
__device__ __forceinline__ void init_group_bars(uint8_t* sm) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  mbar_init(bars + 0, 1);
  mbar_init(bars + 1, 1);
  mbar_init(bars + 3, 1);
  mbar_init(bars + 4, 1);
  mbar_init(bars + 5, 1);
  mbar_fence_init();
}

// Encodes the tensor maps of the chunk-local stage (false: the driver refused).
bool make_maps(Maps* m, const Params& p);

// Byte offset of 16-byte chunk c of row r in a swizzled box of 128-byte rows.
__device__ __forceinline__ uint32_t box_off(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void group_sync(int bar_id) {
  asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(THREADS) : "memory");
}

// Shared-memory offset of the B operand tile of value tile t in the SSD
// increment product (the dead q tiles, then the dead L region).
__device__ __forceinline__ int ssd_b_tile(int t) { return t < 2 ? OFF_Q0 + t * 16384 : OFF_L + (t - 2) * 8192; }
static_assert(OFF_Q1 == OFF_Q0 + 16384 && OFF_L + 16384 <= OFF_AQS && OFF_L % 1024 == 0,
              "SSD operand tiles");

// Mamba2 SSD, the rest of a chunk after its A_qk and row factors. With W = 0
// the system matrix is I, U = v, and the chunk's whole effect on the state is
//   S_{n+1} = gamma S_n + N,   N = k^T diag(kscale) v   (K x V, fp32),
// which does not depend on S: it is formed here, so that the recurrence is a
// plain scan. Per value tile t (32 columns), on tcgen05:
//   D_N[t] = k^T [(kscale v_t)_hi | (kscale v_t)_lo]   M = 128 (raw k, MN-major), N = 64, K = 64
// into TMEM columns 64 t, and N[t] = the hi half + the lo half (v is exact in
// bf16, kscale v is split). N leaves as four [128 c][32 v] fp32 boxes at
// Slab::ssd_n(t); r = v goes to the chunk's exchange block as its four r
// tiles [64 j][v 32 | 0 32] by plain stores (before the slab's flag, like the
// row factors). The TMA barriers of the previous keys and of T complete this
// chunk's phase without a transfer, so that every barrier keeps one (the
// MMA barrier two) phases per chunk.
__device__ __forceinline__ bool ssd_increment(const Params& p, uint8_t* sm, int tid, int bar_id,
                                              int idx, uint32_t ph, uint32_t tmem, bool ok) {
  const int warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, colh = warp >> 2;
  const float* G = reinterpret_cast<const float*>(sm + OFF_SMALL);
  const float* nk = G + 2 * C;
  const float* bb = G + 3 * C;
  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* bar_mma = bar_tma + 1;
  uint64_t* bar_v = bar_tma + 3;
  uint64_t* bar_kp = bar_tma + 4;
  uint64_t* bar_t = bar_tma + 5;
  uint8_t* slab = p.slabs + (size_t)idx * p.slab_bytes;
  uint8_t* xr = p.xchg + (size_t)idx * Xchg::BYTES + Xchg::R;
  if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_v, ph, kWaitLimit));
  if (!ok && lane == 0) atomicOr(p.error_word, kErrTmaWait);
  if (ok) {
    // Item (j, cc): row j, 8-column chunk cc of v, i.e. chunk cc % 4 of value tile cc / 4.
    const float gl = G[C - 1];
    for (int it = tid; it < C * 16; it += THREADS) {
      const int j = it >> 4, cc = it & 15, t = cc >> 2, qc = cc & 3;
      const uint4 raw = *reinterpret_cast<const uint4*>(sm + (cc < 8 ? OFF_V0 : OFF_V1) + box_off(j, cc & 7));
      const float ks = bb[j] * nk[j] * __expf(gl - G[j]);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int z = 0; z < 4; ++z)
        split_pair(ks * __uint_as_float(w[z] << 16), ks * __uint_as_float(w[z] & 0xffff0000u), hi[z], lo[z]);
      uint8_t* bt = sm + ssd_b_tile(t);
      *reinterpret_cast<uint4*>(bt + box_off(j, qc)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(bt + box_off(j, qc + 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      uint8_t* rt = xr + (size_t)t * Xchg::R_TILE;
      *reinterpret_cast<uint4*>(rt + box_off(j, qc)) = raw;
      *reinterpret_cast<uint4*>(rt + box_off(j, qc + 4)) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  fence_async_shared();
  tc_fence_before();
  group_sync(bar_id);
  if (tid == 0) {
    if (ok) {
      tc_fence_after();
      constexpr uint32_t id = idesc_bf16(128, 64, 1, 1);
      const uint32_t kb = smem_u32(sm + OFF_K0);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t bt = smem_u32(sm + ssd_b_tile(t));
#pragma unroll
        for (int s = 0; s < C / 16; ++s)
          umma_bf16(tmem + 64 * t, sdesc_sw128_lbo(kb + s * 2048, 16384),
                    sdesc_sw128_lbo(bt + s * 2048, 8192), id, s > 0);
      }
      umma_commit(bar_mma);
    }
    mbar_arrive(bar_kp);
    mbar_arrive(bar_t);
  }
  if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_mma, 1, kWaitLimit));
  if (!ok && tid == 0) atomicOr(p.error_word, kErrMmaWait);
  tc_fence_after();
  // Warp w: key channels c = 32 (w % 4) + lane (its TMEM lanes), value tiles
  // 2 (w / 4) and 2 (w / 4) + 1, staged as [128][32] fp32 boxes over the dead
  // key, q, v and L tiles (the products that read them are complete).
  if (ok) {
    const int c = 32 * quad + lane;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
#pragma unroll 1
    for (int u = 0; u < 2; ++u) {
      const int t = 2 * colh + u;
      float d[64];
      tmem_ld64(tmem + lane_base + 64 * t, d);
      uint8_t* nt = sm + t * 16384;
#pragma unroll
      for (int qc = 0; qc < 8; ++qc)
        *reinterpret_cast<float4*>(nt + box_off(c, qc)) =
            make_float4(d[4 * qc] + d[32 + 4 * qc], d[4 * qc + 1] + d[33 + 4 * qc],
                        d[4 * qc + 2] + d[34 + 4 * qc], d[4 * qc + 3] + d[35 + 4 * qc]);
    }
  }
  fence_async_shared();
  tc_fence_before();
  group_sync(bar_id);
  if (tid == 0) {
    bulk_store(slab + Slab::ssd_n(0), smem_u32(sm), 2 * (uint32_t)Slab::SSD_N_BOX);
    bulk_store(slab + Slab::ssd_n(2), smem_u32(sm + 2 * Slab::SSD_N_BOX), 2 * (uint32_t)Slab::SSD_N_BOX);
    bulk_commit();
  }
  return ok;
}
static_assert(4 * Slab::SSD_N_BOX <= (size_t)OFF_AQS, "SSD increment staging below the A_qk staging");

// One chunk (n, hv, b) by the 256 threads tid = 0 .. 255 of a group that
// meets on named barrier bar_id, in the group's shared-memory region sm, with
// its mbarriers (at OFF_BAR, initialised by the caller) in phase ph for this
// chunk. TMEM: 256 columns at tmem_given, or allocated by warp 1 into
// alloc_slot when that is not null. Thread 0 publishes release_flag (the
// previous chunk of the group) once that chunk's stores are complete, and
// leaves this chunk's stores in flight. Returns false if a wait gave up.
// kSsd = p.ssd (Mamba2 SSD: no erase, the state increment instead of W, U
// and T), a template argument so that each form is compiled without the
// other's code.
template <bool kSsd>
__device__ __forceinline__ bool produce_chunk(const Maps& maps, const Params& p, uint8_t* sm, int tid, int bar_id,
                              int n, int hv, int b, uint32_t ph, uint32_t tmem_given,
                              uint32_t* alloc_slot, unsigned int* release_flag) {
  const int h = hv / (p.HV / p.H);
  const int t0 = n * C;
  const int warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, colh = warp >> 2;   // TMEM lane quadrant, column half
  const int idx = (int)slab_index(p, b, hv, n);

  float* L = reinterpret_cast<float*>(sm + OFF_L);
  float* X = reinterpret_cast<float*>(sm + OFF_X);
  float* T = reinterpret_cast<float*>(sm + OFF_T);
  float* G = reinterpret_cast<float*>(sm + OFF_SMALL);
  float* nq = G + C;
  float* nk = nq + C;
  float* bb = nk + C;
  float* cfac = bb + C;
  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* bar_mma = bar_tma + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_tma + 2);
  int* split_ok = reinterpret_cast<int*>(tslot + 1);   // decay factorisation allowed
  uint64_t* bar_v = bar_tma + 3;                       // v tiles (read by MMA 3 only)
  uint64_t* bar_kp = bar_tma + 4;                      // previous chunk's k tile
  uint64_t* bar_t = bar_tma + 5;                       // T product
  uint8_t* slab = p.slabs + (size_t)idx * p.slab_bytes;

  // The input tiles are requested first: before the TMEM allocation and the
  // group barrier. The staging of the previous chunk (same thread's TMA
  // stores) must have been read before the tiles overwrite it.
  if (tid == 0) {
    bulk_wait_read<0>();
    // k and q first (MMA 1 and the norms wait for them); v on its own barrier,
    // waited for only by the MMA that reads it.
    mbar_expect_tx(bar_tma, 4 * 8192);
    tma_load4(smem_u32(sm + OFF_K0), &maps.k, 0, h, t0, b, bar_tma);
    tma_load4(smem_u32(sm + OFF_K1), &maps.k, 64, h, t0, b, bar_tma);
    tma_load4(smem_u32(sm + OFF_Q0), &maps.q, 0, h, t0, b, bar_tma);
    tma_load4(smem_u32(sm + OFF_Q1), &maps.q, 64, h, t0, b, bar_tma);
    mbar_expect_tx(bar_v, 2 * 8192);
    tma_load4(smem_u32(sm + OFF_V0), &maps.v, 0, hv, t0, b, bar_v);
    tma_load4(smem_u32(sm + OFF_V1), &maps.v, 64, hv, t0, b, bar_v);
    // The previous chunk's slab is complete in global memory once this
    // thread's bulk stores are (every bulk store of a slab is thread 0's; the
    // row factors, plain stores, came before a group barrier): publish it.
    if (release_flag) {
      bulk_wait<0>();
      fence_async_global();
      st_release_gpu(release_flag, 1u);
    }
  }
  // Gate and beta (plain loads into registers, in flight during the TMEM
  // allocation; zero past the end and for the ungated mode).
  float ga = 0.f, gb = 0.f, bv = 0.f;
  if (warp == 0) {
    const int ta = t0 + 2 * lane;
    if (p.g && ta < p.T) ga = p.g[((size_t)b * p.T + ta) * p.HV + hv];   // g == NULL: ungated
    if (p.g && ta + 1 < p.T) gb = p.g[((size_t)b * p.T + ta + 1) * p.HV + hv];
  }
  if (tid < C) {
    const int t = t0 + tid;
    // SSD: beta = 1 on real rows.
    bv = (t < p.T) ? (kSsd ? 1.f : p.beta[((size_t)b * p.T + t) * p.HV + hv]) : 0.f;
  }
  if (alloc_slot && warp == 1) tmem_alloc(alloc_slot, TMEM_COLS);   // warp 0 is issuing the loads
  tc_fence_before();
  group_sync(bar_id);
  tc_fence_after();
  const uint32_t tmem = alloc_slot ? *alloc_slot : tmem_given;
  bool ok = __all_sync(0xffffffffu, mbar_wait(bar_tma, ph, kWaitLimit));
  if (!ok && lane == 0) atomicOr(p.error_word, kErrTmaWait);
  if (tid < C) bb[tid] = bv;   // read after the next group barrier
  // The key tile's image (the recurrence's A operand k^T) goes to the slab as
  // it is; it must be read out before epilogue 2 overwrites the tile. (Mamba2
  // SSD: the recurrence reads no keys.)
  if (tid == 0 && !kSsd) {
    bulk_store(slab + Slab::K2, smem_u32(sm + OFF_K0), 8192);
    bulk_store(slab + Slab::K2 + 8192, smem_u32(sm + OFF_K1), 8192);
    bulk_commit();
  }

  // ---- MMA 1: D[0:128, 0:64] = [k; q] k^T -------------------------------------
  if (ok && tid == 0) {
    tc_fence_after();
    constexpr uint32_t id = idesc_bf16(128, 64, 0, 0);
    const uint32_t base = smem_u32(sm + OFF_K0);
#pragma unroll
    for (int s = 0; s < K / 16; ++s) {
      const uint32_t a = base + (s >> 2) * 16384 + (s & 3) * 32;
      umma_bf16(tmem, sdesc_sw128(a), sdesc_sw128(a), id, s > 0);
    }
    umma_commit(bar_mma);
  }
  // Row norms while the MMA runs: thread pair (2 r, 2 r + 1) sums the squares
  // of row r of [k; q] (r < 64: k, else q), one 64-column tile each.
  {
    const int r = tid >> 1, part = tid & 1, rr = r & 63;
    const uint8_t* tp = sm + (r < 64 ? OFF_K0 : OFF_Q0) + part * 16384;
    float ss = 0.f;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      const uint4 u = *reinterpret_cast<const uint4*>(tp + swz128((uint32_t)(rr * 128 + ch * 16)));
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
        ss = fmaf(lo, lo, fmaf(hi, hi, ss));
      }
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    const float inv = p.use_l2 ? 1.f / sqrtf(ss + 1e-6f) : 1.f;
    if (part == 0) {
      if (r < 64) nk[rr] = inv; else nq[rr] = inv;
    }
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
    const float g0 = excl + ga, g1 = excl + ga + gb;
    G[2 * lane] = g0;
    G[2 * lane + 1] = g1;
    // The decays exp(G_i - G_j) may be split at the middle row m = C/2 - 1 as
    // exp(G_i - G_m) exp(G_m - G_j) while every |G_i - G_m| <= 80: both factors
    // then stay inside the fp32 range (NaN gates fail the test).
    const float gm = __shfl_sync(0xffffffffu, g1, C / 4 - 1);
    float dev = fmaxf(fabsf(g0 - gm), fabsf(g1 - gm));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dev = fmaxf(dev, __shfl_xor_sync(0xffffffffu, dev, o));
    if (lane == 0) *split_ok = dev <= kSplitSpan ? 1 : 0;
  }
  group_sync(bar_id);
  // Split decays: column factor |k_j|^-1 beta_j exp(G_m - G_j) once per column
  // (in the column-factor array, free until the row factors below); the row and
  // column factors are multiplied before the dot, so the intermediate is the
  // size of exp(G_i - G_j).
  const bool split = *split_ok != 0;
  const float Gm = G[C / 2 - 1];
  if (split) {
    if (tid < C) cfac[tid] = nk[tid] * bb[tid] * __expf(Gm - G[tid]);
    group_sync(bar_id);
  }

  // ---- epilogue 1: A_kk -> L (fp32, smem), A_qk -> stacked hi/lo bf16 box ------
  // Warp w: TMEM lanes of quadrant w % 4 (rows of [k; q]), columns
  // [32 (w / 4), 32 (w / 4) + 32). A_qk row i, hi and lo, go to stacked rows
  // stacked_row(i, 0 / 1) of one swizzled [128][64] box.
  if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_mma, 0, kWaitLimit));
  if (!ok && tid == 0) atomicOr(p.error_word, kErrMmaWait);
  tc_fence_after();
  if (ok && split) {
    const int r = 32 * quad + lane, rr = r & 63;
    const bool is_q = r >= 64;
    const float rowe = (is_q ? p.scale * nq[rr] : nk[rr]) * __expf(G[rr] - Gm);
    float v[32];
    tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + 32 * colh, v);
    const int jb = 32 * colh;
    if (!is_q) {
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 cf = *reinterpret_cast<const float4*>(cfac + jb + e);
        const float cs[4] = {cf.x, cf.y, cf.z, cf.w};
        float a4[4];
#pragma unroll
        for (int z = 0; z < 4; ++z)
          a4[z] = (jb + e + z < rr && !kSsd) ? v[e + z] * (rowe * cs[z]) : 0.f;
        *reinterpret_cast<float4*>(L + rr * LDL + jb + e) = make_float4(a4[0], a4[1], a4[2], a4[3]);
      }
    } else {
      uint8_t* aqs = sm + OFF_AQS;
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        const float4 c0 = *reinterpret_cast<const float4*>(cfac + jb + e);
        const float4 c1 = *reinterpret_cast<const float4*>(cfac + jb + e + 4);
        const float cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int f = 0; f < 8; f += 2) {
          const float a0 = (jb + e + f <= rr) ? v[e + f] * (rowe * cs[f]) : 0.f;
          const float a1 = (jb + e + f + 1 <= rr) ? v[e + f + 1] * (rowe * cs[f + 1]) : 0.f;
          split_pair(a0, a1, hi[f / 2], lo[f / 2]);
        }
        const int c = (jb + e) >> 3;
        *reinterpret_cast<uint4*>(aqs + box_off(stacked_row(rr, 0), c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(aqs + box_off(stacked_row(rr, 1), c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
  } else if (ok) {
    // Decays too far apart to split: exp(G_i - G_j) element by element.
    const int r = 32 * quad + lane, rr = r & 63;
    const bool is_q = r >= 64;
    const float Gi = G[rr];
    const float rowf = is_q ? p.scale * nq[rr] : nk[rr];
    float v[32];
    tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + 32 * colh, v);
    const int jb = 32 * colh;
    if (!is_q) {
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        float a4[4];
#pragma unroll
        for (int z = 0; z < 4; ++z) {
          const int j = jb + e + z;
          a4[z] = (j < rr && !kSsd) ? v[e + z] * rowf * nk[j] * __expf(Gi - G[j]) * bb[j] : 0.f;
        }
        *reinterpret_cast<float4*>(L + rr * LDL + jb + e) = make_float4(a4[0], a4[1], a4[2], a4[3]);
      }
    } else {
      uint8_t* aqs = sm + OFF_AQS;
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int f = 0; f < 8; f += 2) {
          float a2[2];
#pragma unroll
          for (int z = 0; z < 2; ++z) {
            const int j = jb + e + f + z;
            a2[z] = (j <= rr) ? v[e + f + z] * rowf * nk[j] * __expf(Gi - G[j]) * bb[j] : 0.f;
          }
          split_pair(a2[0], a2[1], hi[f / 2], lo[f / 2]);
        }
        const int c = (jb + e) >> 3;
        *reinterpret_cast<uint4*>(aqs + box_off(stacked_row(rr, 0), c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(aqs + box_off(stacked_row(rr, 1), c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
  }
  fence_async_shared();
  tc_fence_before();
  group_sync(bar_id);

  // A_qk hi / lo out by a bulk copy (thread 0, like every bulk store of the
  // slab, so that its one completion wait before the flag covers them all),
  // and the per-row factors of the state pass on warps 2-7 while warps 0-1
  // run level 0 of the inverse.
  constexpr int kRowTid = 64;          // first thread of the row-factor warps
  if (tid == 0) {
    bulk_store(slab + Slab::AQ2, smem_u32(sm + OFF_AQS), 16384);
    bulk_commit();
  }
  {
    float* vec = reinterpret_cast<float*>(slab + Slab::VEC);
    const float gl = G[C - 1];
    const int e = tid - kRowTid;
    if (e >= 0 && e < C) {
      vec[e] = p.scale * nq[e] * __expf(G[e]);
      vec[C + e] = bb[e] * nk[e] * __expf(gl - G[e]);
      cfac[e] = __expf(G[e]) * nk[e];   // column factor of X' = X diag(exp(G) |k|^-1)
    }
    if (e >= 0 && e < K) vec[2 * C + e] = __expf(gl);
  }
  if (kSsd) return ssd_increment(p, sm, tid, bar_id, idx, ph, tmem, ok);

  // ---- X = (I + L)^-1, blocked (gdr_trinv.cuh) ---------------------------------
  unit_lower_inverse64<LDL, LDX>(L, X, T, tid, bar_id);
  // The A_qk staging read out (it is overwritten next); the store itself
  // completes before the slab's flag, with the others.
  if (tid == 0) bulk_wait_read<0>();
  group_sync(bar_id);   // X complete; L and the A_qk staging are dead from here on

  // ---- A operands XW = [X' hi/lo], XU = [X hi/lo] (rows interleaved, see stacked_row)
  // Each thread: one row i, 8 consecutive columns, 2 items.
  {
    uint8_t* xw = sm + OFF_L;
    uint8_t* xu = sm + OFF_XU;
#pragma unroll
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
        split_pair(u0 * cfac[c8 + z], u1 * cfac[c8 + z + 1], whi[z / 2], wlo[z / 2]);
        split_pair(u0, u1, uhi[z / 2], ulo[z / 2]);
      }
      const uint32_t o_hi = swz128((uint32_t)(stacked_row(i, 0) * 128 + c8 * 2));
      const uint32_t o_lo = swz128((uint32_t)(stacked_row(i, 1) * 128 + c8 * 2));
      *reinterpret_cast<uint4*>(xw + o_hi) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
      *reinterpret_cast<uint4*>(xw + o_lo) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
      *reinterpret_cast<uint4*>(xu + o_hi) = make_uint4(uhi[0], uhi[1], uhi[2], uhi[3]);
      *reinterpret_cast<uint4*>(xu + o_lo) = make_uint4(ulo[0], ulo[1], ulo[2], ulo[3]);
    }
  }
  fence_async_shared();
  tc_fence_before();
  group_sync(bar_id);
  // X is dead: the previous chunk's keys (for T) go where it was. The first
  // chunk of a sequence has none; its barriers complete a phase all the same,
  // so that a group's barrier phases stay one per chunk.
  if (tid == 0) {
    if (n > 0) {
      mbar_expect_tx(bar_kp, 2 * 8192);
      tma_load4(smem_u32(sm + OFF_KP), &maps.k, 0, h, t0 - C, b, bar_kp);
      tma_load4(smem_u32(sm + OFF_KP + 8192), &maps.k, 64, h, t0 - C, b, bar_kp);
    } else {
      mbar_arrive(bar_kp);
      mbar_arrive(bar_t);
    }
  }

  // ---- MMA 2/3: D_W = XW k (TMEM cols 0-127), D_U = XU v (cols 128-255) ----------
  if (tid == 0) bulk_wait_read<0>();                 // key image read out (epilogue 2 reuses the tile)
  if (ok && tid == 0) {
    ok = mbar_wait(bar_v, ph, kWaitLimit);           // the v tiles (normally long arrived)
    if (!ok) atomicOr(p.error_word, kErrTmaWait);
  }
  if (ok && tid == 0) {
    tc_fence_after();
    constexpr uint32_t id = idesc_bf16(128, 128, 0, 1);
    const uint32_t xw = smem_u32(sm + OFF_L), xu = smem_u32(sm + OFF_XU);
    const uint32_t kb = smem_u32(sm + OFF_K0), vb = smem_u32(sm + OFF_V0);
#pragma unroll
    for (int s = 0; s < C / 16; ++s) {
      umma_bf16(tmem, sdesc_sw128(xw + s * 32), sdesc_sw128_lbo(kb + s * 2048, 16384), id, s > 0);
      umma_bf16(tmem + 128, sdesc_sw128(xu + s * 32), sdesc_sw128_lbo(vb + s * 2048, 8192), id,
                s > 0);
    }
    umma_commit(bar_mma);
  }
  if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_mma, 1, kWaitLimit));
  if (!ok && tid == 0) atomicOr(p.error_word, kErrMmaWait);
  tc_fence_after();

  // ---- epilogue 2: W = hi + lo rows, U likewise; -W hi/lo and U staged --------
  // Lane t < 16 of quadrant q holds the hi product of row r = 16 q + t, lane
  // t + 16 the lo product of the same row: one shuffle per value sums them,
  // after which lane t keeps columns [0,16) and lane t + 16 columns [16,32) of
  // each 32-column block. Warps 0-3 take the W blocks, warps 4-7 the U blocks.
  // -W leaves as two stacked [128][64] boxes (column halves; rows by
  // stacked_row), U as four [64][32] fp32 boxes.
  if (ok) {
    const int r = 16 * quad + (lane & 15);
    const int half = lane >> 4;
    const bool is_u = colh == 1;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      float v[32];
      tmem_ld32(tmem + lane_base + (is_u ? 128 : 0) + cc * 32, v);
      float s[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float send = half ? v[e] : v[16 + e];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
        s[e] = (half ? v[16 + e] : v[e]) + recv;
      }
      const int c0 = cc * 32 + half * 16;   // first column of this lane's 16
      if (!is_u) {
        uint32_t hi[8], lo[8];
        // SSD keeps no erase term: W = 0 (then X = I and U = v).
        const float ws = kSsd ? 0.f : -1.f;
#pragma unroll
        for (int e = 0; e < 16; e += 2) split_pair(ws * s[e], ws * s[e + 1], hi[e / 2], lo[e / 2]);
        const int bx = c0 >> 6, c = (c0 & 63) >> 3;
        uint8_t* wb = sm + OFF_WS + bx * 16384;
        const int rh = stacked_row(r, 0), rl = stacked_row(r, 1);
        *reinterpret_cast<uint4*>(wb + box_off(rh, c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(wb + box_off(rh, c + 1)) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
        *reinterpret_cast<uint4*>(wb + box_off(rl, c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        *reinterpret_cast<uint4*>(wb + box_off(rl, c + 1)) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
      } else {
        uint8_t* ub = sm + OFF_US + cc * 8192;   // box cc: columns [32 cc, 32 cc + 32)
        const int c = (c0 & 31) >> 2;
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<float4*>(ub + box_off(r, c + e / 4)) =
              make_float4(s[e], s[e + 1], s[e + 2], s[e + 3]);
      }
    }
  }
  fence_async_shared();
  tc_fence_before();
  group_sync(bar_id);
  if (tid == 0) {
    bulk_store(slab + Slab::W2, smem_u32(sm + OFF_WS), 32768);
    bulk_store(slab + Slab::U, smem_u32(sm + OFF_US), 32768);
    bulk_commit();
  }

  // ---- T = W k_prev^T for the recurrence's look-ahead (not for the first chunk) ----
  // A = the -W hi / lo staging (stacked rows, K-major, two 64-column boxes),
  // B = the previous chunk's raw key tile (K-major: rows j, channels
  // contiguous): D_T [128 stacked rows][64 j] in TMEM columns 0-63, whose hi
  // and lo rows are added like W's. -T leaves as one stacked [128][64] box
  // staged over the (then dead) key tile.
  if (n > 0) {
    if (ok && tid == 0) {
      ok = mbar_wait(bar_kp, ph, kWaitLimit);
      if (!ok) atomicOr(p.error_word, kErrTmaWait);
    }
    if (ok && tid == 0) {
      tc_fence_after();
      constexpr uint32_t id = idesc_bf16(128, 64, 0, 0);
      const uint32_t ws = smem_u32(sm + OFF_WS), kp = smem_u32(sm + OFF_KP);
#pragma unroll
      for (int s = 0; s < K / 16; ++s)
        umma_bf16(tmem, sdesc_sw128(ws + (s >> 2) * 16384 + (s & 3) * 32),
                  sdesc_sw128(kp + (s >> 2) * 8192 + (s & 3) * 32), id, s > 0);
      umma_commit(bar_t);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_t, ph, kWaitLimit));
    if (!ok && tid == 0) atomicOr(p.error_word, kErrMmaWait);
    tc_fence_after();
    if (ok) {
      const int r = 16 * quad + (lane & 15);
      const int half = lane >> 4;
      float v[32];
      tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + 32 * colh, v);
      float t[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float send = half ? v[e] : v[16 + e];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
        t[e] = (half ? v[16 + e] : v[e]) + recv;     // (-W) k_prev^T: already -T
      }
      uint32_t hi[8], lo[8];
#pragma unroll
      for (int e = 0; e < 16; e += 2) split_pair(t[e], t[e + 1], hi[e / 2], lo[e / 2]);
      const int c = (32 * colh + 16 * half) >> 3;
      uint8_t* tb = sm + OFF_KP;
      const int rh = stacked_row(r, 0), rl = stacked_row(r, 1);
      *reinterpret_cast<uint4*>(tb + box_off(rh, c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(tb + box_off(rh, c + 1)) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
      *reinterpret_cast<uint4*>(tb + box_off(rl, c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      *reinterpret_cast<uint4*>(tb + box_off(rl, c + 1)) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
    }
    fence_async_shared();
    tc_fence_before();
    group_sync(bar_id);
    if (tid == 0) {
      bulk_store(slab + Slab::T2, smem_u32(sm + OFF_KP), 16384);
      bulk_commit();
    }
  }
  return ok;
}

}  // namespace chunk
}  // namespace fast
}  // namespace gdr
