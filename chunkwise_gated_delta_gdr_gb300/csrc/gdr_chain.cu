// gdr_chain.cu -- inter-chunk recurrence of the fast path for the scalar gate
// (Gated DeltaNet) on tcgen05 tensor cores, its output pass, and the
// one-launch forward.
//
// Per chunk n the inter-chunk loop of the "分块并行计算（Chunkwise）" notes
// (section "chunk 间递推") reads, with S_n the state at the start of chunk n,
//     r_n     = U_n - W_n S_n
//     o_n     = (q exp(G)) S_n + A_qk r_n
//     S_{n+1} = gamma_n S_n + k_n^T rho_n,     rho_n = kscale_n r_n
// (gamma_n = exp(G_last) of chunk n, kscale the row factors of
// (exp(G_last - G) k)^T beta). The serial dependence is r_n -> S_{n+1} ->
// r_{n+1}. Substituting S_n in r_n:
//     W_n S_n = gamma_{n-1} W_n S_{n-1} + T_n rho_{n-1},   T_n = W_n k_{n-1}^T (C x C)
// so with T_n formed in the chunk-local stage,
//     r_n = U_n + gamma_{n-1} (-W_n) S_{n-1} + (-T_n) rho_{n-1}
// and the only product between rho_{n-1} and r_n is (-T_n) rho_{n-1} (K = C),
// while (-W_n) S_{n-1} and the state update run one chunk ahead.
//
// Chain role: one CTA per (sequence, 32 value columns). Its operands arrive as
// the byte images the chunk-local stage stored (one bulk copy per array: on
// GB300 an SM takes in about 120 bytes per cycle this way against about 43 by
// tensor-map loads of 128-byte swizzled boxes). Per chunk, on tcgen05
// (kind::f16, fp32 accumulators in TMEM, every fp32-valued operand as a bf16
// hi + lo pair):
//     D_ws(n) = [-W_hi; -W_lo] [S_{n-1,hi} | S_{n-1,lo}]   M = 128 (stacked), N = 64, K = 128
//     D_t(n)  = [-T_hi; -T_lo] [rho_{n-1,hi} | rho_{n-1,lo}] M = 128 (stacked), N = 64, K = 64
//     D_S(n)  = k_{n-1}^T [rho_{n-1,hi} | rho_{n-1,lo}]      M = 128 (k raw bf16), N = 64, K = 64
// (for n = 0: D_ws(0) = (-W_0) S_0 with gamma := 1 and no D_t).
// Each product is issued as soon as its last input is published, by a thread
// released through a named barrier: an mbarrier hand-off costs several hundred
// cycles per product on this serial path, and the tensor pipe itself needs
// only about 1.2k cycles per chunk for the sixteen MMAs.
// Roles (16 warps):
//   warps 0-7  the state: thread (w, lane) holds channel c = 32 (w % 4) + lane
//              of S (TMEM lane c of D_S), value columns [16 h, 16 h + 16) with
//              h = w / 4, for the whole sequence: S_n = gamma_{n-1} S_{n-1} +
//              D_S(n), published as the bf16 [hi 32 | lo 32] rows of an
//              MN-major B operand.
//   warps 8-11 r: lanes 0-15 of quadrant q hold the hi rows j = 16 q + lane of
//              D_ws and D_t, lanes 16-31 the lo rows of the same j; they form
//              r_n and rho_n and publish both as tiles of the same format (rho
//              for the products, r for the output pass).
//   warp 12    TMA producer (three rings of two slots: {-W}, {-T, U, VEC}, {k}).
//   warp 14    issues D_S(n + 1) and D_t(n + 1) once the r warps have published
//              rho_n; warp 15 issues D_ws(n + 1) once the state warps have
//              published S_n. Each is released by a named barrier (the r
//              warps arrive on theirs without waiting, the state warps sync).
//   warp 13    TMEM owner and exporter: once S_n and r_n are published it copies both tiles
//              to the exchange block (bulk copies, one group per chunk, one
//              group in flight) and announces the previous chunk's tiles read
//              out (three S tiles, two r tiles). In
//              the one-launch forward it also marks the chunks exported so
//              far, every kMarkEvery chunks and a little behind the copies.
// The S_n and r_n tiles of every chunk leave by bulk copies (a plain store of a
// row-per-thread tile would touch 32 lines per instruction and hold up the
// SM's memory pipe) as the exchange block of gdr_fast.cuh; the output pass
// then forms
//     o_n = qscale (q S_n) + A_qk r_n
// per (chunk, sequence, 64 value columns) on tcgen05.
//
// Mamba2 SSD (W = 0, U = v): r_n = v_n does not depend on the state, so the
// chunk-local stage forms each chunk's whole increment N_n = k_n^T rho_n and
// writes the r tiles itself; the chain CTA then runs S_{n+1} = gamma_n S_n +
// N_n with no product (ssd_chain), exporting S_n as above.
//
// One-launch forward (launch_fused): one cooperative launch of one CTA per SM.
// The first CTAs are the chains; each first runs the chunk-local stage
// (gdr_chunk_tc.cuh) for one of its sequence's first four chunks. The other
// CTAs are workers, two groups of 8 warps each, that run the chunk-local stage
// over the remaining chunks in chunk order. Every chunk's flag is raised once
// its slab is in global memory, and a chain's TMA warp waits for chunk n's
// flag before loading it. Each
// worker group then takes output items (chunk n, sequence, 64 value columns)
// in chunk order from a counter, and forms o_n once the chains of both value
// tiles have marked chunk n exported; a chain CTA joins them once its chain
// is done. A GPU-scope acquire or release by any thread of a chain CTA waits
// until every memory operation in flight on its SM (the ring loads included)
// has completed, a microsecond or more, so the chains acquire the slab flags
// as rarely as they can (every flag already set at once) and mark their
// exports only every kMarkEvery chunks. Workers wait on chains only after
// their last slab, chains never wait on output items, and all CTAs are
// co-resident, so the waits end; every wait is bounded all the same and
// records a code in the workspace error word when it gives up, after which
// the CTA runs to its end.
#include <string.h>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdr_chunk_tc.cuh"

namespace gdr {
namespace fast {
namespace {

using namespace ptx;

constexpr int VC = 32;                  // value columns per chain CTA
constexpr int VTILES = V / VC;          // chain CTAs per sequence
constexpr int CHAIN_THREADS = 512;
constexpr int FUSED_THREADS = 512;      // worker CTA: two chunk groups of 256
constexpr long kWaitLimit = 1L << 24;   // mbarrier polls before a wait gives up
constexpr long kTmaIdleLimit = 1L << 24;  // TMA event-loop rounds (64 ns sleeps) likewise
// Slab flags the TMA producer reads at once (one acquire for all of those set).
constexpr int kFlagWindow = 32;
constexpr unsigned int kErrChainWait = 4u, kErrFlagWait = 8u, kErrOutWait = 16u, kErrXchgWait = 32u;
// One-launch forward: a chain announces its exports every kMarkEvery chunks
// and every kMarkTail chunks in the last kMarkEvery (whose outputs wait for
// the chains to end), kMarkLag bulk groups behind the newest export (by then
// long written). Each release waits for every memory operation in flight on
// the SM and can hold up the exporter for about a chain step, so the marks
// are few. (Every 32 chunks measured slower: the workers then wait longer.)
constexpr int kMarkEvery = 16;
constexpr int kMarkTail = 4;
constexpr int kMarkTailSpan = kMarkEvery;
constexpr int kMarkLag = 2;
// (Bringing the next four slabs into L2 ahead of the ring loads with bulk
// prefetches measured 14 us slower per forward.)
constexpr int kProduceBar = 4;   // named barrier of a chain CTA's chunk production (warps 0-7)
// First chunks of a sequence its chain CTAs produce, one each (two each
// measured 12 us slower per forward).
constexpr int kChainChunks = VTILES;

// Shared memory of a chain CTA (bytes from a 1024-aligned base). Three rings
// of two slots, each slot released as soon as its last reader is done:
// Ring W slot (chunk n): -W stacked [128][128] bf16 (two [128][64] boxes); free
// once D_ws(n) is complete, so chunk n + 2 streams in a step before it is used.
constexpr int W_SLOT = 32768;
constexpr uint32_t W_TX = 32768;
// Ring A slot (chunk n): -T stacked [128][64] bf16, U [64 j][32 v] fp32
// (128-byte swizzled); beside it, outside the 1 KB-aligned slots, the chunk's
// kscale[64] and gamma (the VEC entries from kscale on, 512 bytes).
constexpr int A_T = 0, A_U = 16384, A_SLOT = 24576;
constexpr int VEC_OFF = C * 4, VEC_BYTES = 512;   // slab VEC bytes the chain reads (kscale, gamma)
constexpr uint32_t A_TX = 16384 + 8192 + VEC_BYTES;
// Ring B slot (chunk n): k [64 j][128 c] bf16 (two [64][64] boxes).
constexpr int KB_SLOT = 16384;
constexpr uint32_t B_TX = 16384;
// S tiles: three, so that S_n overwrites S_{n-3}, whose readers (D_ws(n - 2)
// and its export) are long done, and the state warps wait for neither.
constexpr int S_TILES = 3;
constexpr int OFF_W = 0;
constexpr int OFF_A = OFF_W + 2 * W_SLOT;
constexpr int OFF_B = OFF_A + 2 * A_SLOT;
constexpr int OFF_S = OFF_B + 2 * KB_SLOT;          // S tiles [128 c][hi 32 | lo 32] bf16
constexpr int OFF_P = OFF_S + S_TILES * 16384;     // rho tiles [64 j][hi 32 | lo 32], x 2
constexpr int OFF_R = OFF_P + 2 * 8192;            // r tiles, the same format, x 2
constexpr int OFF_V = OFF_R + 2 * 8192;            // ring A's VEC part, x 2
constexpr int OFF_BARS = OFF_V + 2 * VEC_BYTES;
constexpr int CHAIN_SMEM = OFF_BARS + 256 + 1024;
static_assert(A_SLOT % 1024 == 0 && OFF_A % 1024 == 0 && OFF_B % 1024 == 0 && OFF_S % 1024 == 0 &&
                  OFF_P % 1024 == 0 && OFF_R % 1024 == 0 && A_T % 1024 == 0 && A_U % 1024 == 0,
              "swizzled tiles need 1 KB alignment");
static_assert(Slab::VEC % 16 == 0 && VEC_OFF % 16 == 0, "bulk copy alignment");
static_assert(CHAIN_SMEM <= 232448, "chain shared memory");
constexpr int FUSED_SMEM =
    (CHAIN_SMEM > 2 * chunk::GROUP_BYTES + 1024) ? CHAIN_SMEM : 2 * chunk::GROUP_BYTES + 1024;
static_assert(FUSED_SMEM <= 232448, "one-launch shared memory");

// TMEM columns of a chain CTA: D_ws (two buffers), D_t, D_S (two buffers).
constexpr uint32_t T_WS = 0, T_T = 128, T_S = 192, CHAIN_TMEM = 512;

// Barriers of a chain CTA (index into a uint64_t array at OFF_BARS).
enum : int {
  B_FULLA = 0,    // [2] ring A slot loaded (local arrive + transaction bytes)
  B_EMPTYA = 2,   // [2] ring A slot free: 4 r warps (after D_t of the chunk completed)
                  //     + 8 S warps
  B_FULLB = 4,    // [2] ring B slot loaded
  B_EMPTYB = 6,   // [2] ring B slot free: 8 S warps (after the D_S that read it)
  B_WS = 8,       // [2] D_ws complete (commit), buffer n % 2
  B_T = 10,       // D_t complete (commit)
  B_DS = 11,      // [2] D_S complete (commit), buffer (n - 1) % 2 for D_S(n)
  B_FULLW = 13,   // [2] ring W slot loaded
  B_EMPTYW = 15,  // [2] ring W slot free: 4 r warps (after D_ws of the chunk completed)
  B_RP = 17,      // [2] r_n tile published, barrier n % 2 (4 r warps)
  B_ES = 19,      // [3] S_n published, barrier n % 3 (8 state warps; for the exporter)
  B_XR = 22,      // [3] exports of chunk n (S and r tiles) read out, barrier n % 3 (exporter)
  B_SLOT = 25     // TMEM slot (u32)
};
static_assert((B_SLOT + 1) * 8 <= 256, "chain barrier area");
// A waiter tests an mbarrier phase by parity, so a barrier must never run two
// phases ahead of one of its waiters. The S, r and export barriers could (S_{n+1}
// may be published before chunk n is exported, and chunk n - 1 exported before
// the MMA thread checks chunk n - 2), so each has one barrier per tile: barrier
// n % T completes phase n / T for chunk n (T = S_TILES for S and the exports,
// 2 for r), and its next phase (chunk n + T) depends on the waiter having
// passed chunk n.
__device__ __forceinline__ uint32_t tile_parity(int n, int tiles) { return (uint32_t)(n / tiles) & 1u; }
constexpr int kEmptyA = 4 + 8;
constexpr int kEmptyB = 8;
constexpr int kEmptyW = 4;

__device__ __forceinline__ void nb_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Arrives on named barrier id (n threads in all) without waiting for it.
__device__ __forceinline__ void nb_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Byte offset of 16-byte chunk q of row r in 128-byte swizzled rows.
__device__ __forceinline__ uint32_t sw_off(int r, int q) {
  return (uint32_t)(r * 128 + ((q ^ (r & 7)) << 4));
}
// Bounded wait by polling (no suspension of the thread between polls).
__device__ __forceinline__ bool mbar_spin(uint64_t* bar, uint32_t parity, long limit) {
  for (long i = 0; i <= limit; ++i)
    if (mbar_test(bar, parity)) return true;
  return false;
}
// A bounded wait of a whole warp; false for every lane once any lane gave up.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, bool ok) {
  const bool r = ok && mbar_wait(bar, parity, kWaitLimit);
  return __all_sync(0xffffffffu, r);
}
// 16 fp32 values -> bf16 hi / lo chunks (two 16-byte chunks each) of row r:
// hi at chunks q0, q0 + 1, lo at chunks q0 + 4, q0 + 5 (rows [x_hi 32 | x_lo 32]).
__device__ __forceinline__ void publish16(uint8_t* tile, int r, int q0, const float* x) {
  uint32_t h[8], l[8];
#pragma unroll
  for (int z = 0; z < 8; ++z) split_pair(x[2 * z], x[2 * z + 1], h[z], l[z]);
  *reinterpret_cast<uint4*>(tile + sw_off(r, q0)) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(tile + sw_off(r, q0 + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
  *reinterpret_cast<uint4*>(tile + sw_off(r, q0 + 4)) = make_uint4(l[0], l[1], l[2], l[3]);
  *reinterpret_cast<uint4*>(tile + sw_off(r, q0 + 5)) = make_uint4(l[4], l[5], l[6], l[7]);
}
// Sums the hi and lo rows of a stacked accumulator: lane t < 16 holds the hi
// row, lane t + 16 the lo row of the same output row; in each, columns
// [0, 32) come from the B hi part and [32, 64) from the B lo part. Returns the
// 16 columns [16 half, 16 half + 16) this lane keeps.
__device__ __forceinline__ void stacked_sum(const float* d, int half, float* out) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float col_a = d[i] + d[32 + i];          // column i
    const float col_b = d[16 + i] + d[48 + i];     // column 16 + i
    const float send = half ? col_a : col_b;       // what the partner lane keeps
    const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
    out[i] = (half ? col_b : col_a) + recv;
  }
}

// Output products of one (sequence, chunk n, 64 value columns vh): o = qscale
// (q S_n) + A_qk r_n from the exchange block of chunk n (the S and r tiles of
// value tiles 2 vh, 2 vh + 1) and the slab (A_qk, qscale), with raw q by TMA.
//   D_qs = q [S_a | S_b]            M = 64,  N = 128 (two tiles of [hi 32 | lo 32]), K = 128
//   D_ar = [A_hi; A_lo] [R_a | R_b] M = 128 (stacked), N = 128, K = 64
// Shared-memory map (from a 1024-aligned base) and TMEM use of both forms that
// compute them: the output kernel and a group of 8 warps of the one-launch forward.
namespace out {
constexpr int THREADS = 128;
constexpr int Q = 0, AQ = 16384, S = 32768, R = 65536, QS = 81920, BAR = 82176;
constexpr int SMEM = BAR + 64 + 1024;
constexpr uint32_t TX = 16384 + 16384 + 32768 + 16384 + 256;
constexpr uint32_t TMEM_COLS = 256;
static_assert(QS + 256 <= chunk::OFF_SMALL, "output tiles inside a worker group region");

// Loads of an output item (one thread), completing on `bar`.
__device__ __forceinline__ void issue_loads(const CUtensorMap* qmap, const Params& p, uint32_t sb,
                                            int seq, int n, int vh, uint64_t* bar) {
  const int b = seq / p.HV, hv = seq % p.HV, h = hv / (p.HV / p.H);
  const size_t idx = (size_t)seq * p.N + n;
  const uint8_t* xb = p.xchg + idx * Xchg::BYTES;
  mbar_expect_tx(bar, TX);
  tma_load4(sb + Q, qmap, 0, h, n * C, b, bar);
  tma_load4(sb + Q + 8192, qmap, 64, h, n * C, b, bar);
  // (the exchange tiles are read once, the slab's A_qk and qscale by both
  // value halves)
  const uint64_t pol = l2_evict_first();
  bulk_load(sb + AQ, p.slabs + idx * p.slab_bytes + Slab::AQ2, 16384, bar);
  bulk_load_hint(sb + S, xb + Xchg::S + 2 * vh * Xchg::S_TILE, 2 * Xchg::S_TILE, bar, pol);
  bulk_load_hint(sb + R, xb + Xchg::R + 2 * vh * Xchg::R_TILE, 2 * Xchg::R_TILE, bar, pol);
  bulk_load(sb + QS, p.slabs + idx * p.slab_bytes + Slab::VEC, 256, bar);
}
// The two products (one thread), accumulators at TMEM columns 0-127 and 128-255.
__device__ __forceinline__ void issue_mmas(uint32_t tmem, uint32_t sb) {
  constexpr uint32_t ID_QS = idesc_bf16(64, 128, 0, 1);
  constexpr uint32_t ID_AR = idesc_bf16(128, 128, 0, 1);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    umma_bf16(tmem, sdesc_sw128(sb + Q + (kk >> 2) * 8192 + (kk & 3) * 32),
              sdesc_sw128_lbo(sb + S + kk * 2048, 16384), ID_QS, kk > 0);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    umma_bf16(tmem + 128, sdesc_sw128(sb + AQ + kk * 32),
              sdesc_sw128_lbo(sb + R + kk * 2048, 8192), ID_AR, kk > 0);
}
// Writes 16 outputs of row t (value columns v0 .. v0 + 15) of head hv.
__device__ __forceinline__ void store16(const Params& p, int b, int t, int hv, int v0, const float* o) {
  const size_t off = (((size_t)b * p.T + t) * p.HV + hv) * V + v0;
  if (p.out_bf16) {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + off);
#pragma unroll
    for (int q = 0; q < 2; ++q)
      dst[q] = make_uint4(pack_bf16(o[8 * q], o[8 * q + 1]), pack_bf16(o[8 * q + 2], o[8 * q + 3]),
                          pack_bf16(o[8 * q + 4], o[8 * q + 5]), pack_bf16(o[8 * q + 6], o[8 * q + 7]));
  } else {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + off);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
  }
}
}  // namespace out

// Output items of the one-launch forward, run by a group of 8 warps (threads
// gtid = 0 .. 255, named barrier bar_id) in a worker group region gsm with
// 256 TMEM columns at tmem, its TMA and MMA barriers (chunk layout) next in
// phases ph and mph. Items (chunk n, sequence, 64 value columns vh) are
// claimed in that order from the counter after the export marks; an item
// waits until both of its value tiles have marked chunk n exported.
__device__ __forceinline__ void output_items(const CUtensorMap* qmap, const Params& p, uint8_t* gsm,
                                             int gtid, int bar_id, uint32_t tmem, uint32_t ph,
                                             uint32_t mph) {
  const int nseq = p.B * p.HV;
  const long items = 2L * nseq * p.N;
  unsigned int* counter = p.xmark + (size_t)nseq * VTILES;
  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(gsm + chunk::OFF_BAR);
  uint64_t* bar_mma = bar_tma + 1;
  int* claim = reinterpret_cast<int*>(bar_tma + 2) + 1;   // the chunk stage's split flag word
  const uint32_t sb = smem_u32(gsm);
  const int lane = gtid & 31, gw = gtid >> 5;
  for (;;) {
    if (gtid == 0) *claim = (int)atomicAdd(counter, 1u);
    chunk::group_sync(bar_id);
    const long it = *claim;
    if (it >= items) break;
    const int n = (int)(it / (2 * nseq)), rem = (int)(it % (2 * nseq));
    const int seq = rem >> 1, vh = rem & 1;
    const int b = seq / p.HV, hv = seq % p.HV;
    if (gtid == 0) {
      const unsigned int* xm = p.xmark + (size_t)seq * VTILES + 2 * vh;
      long polls = 0;
      while (ld_acquire_gpu(xm) <= (unsigned int)n || ld_acquire_gpu(xm + 1) <= (unsigned int)n) {
        if (++polls > p.wait_limit) {
          atomicOr(p.error_word, kErrXchgWait);
          break;
        }
        __nanosleep(64);
      }
      fence_async_global();     // the exports (generic acquire) -> bulk reads
      out::issue_loads(qmap, p, sb, seq, n, vh, bar_tma);
      const bool ok = mbar_wait(bar_tma, ph, kWaitLimit);
      if (ok) {
        tc_fence_after();
        out::issue_mmas(tmem, sb);
      } else {
        atomicOr(p.error_word, kErrOutWait);
      }
      umma_commit(bar_mma);
    }
    ph ^= 1u;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar_mma, mph, kWaitLimit));
    mph ^= 1u;
    tc_fence_after();
    // Warp gw: TMEM lane quadrant gw % 4, value tile u = gw / 4. Lanes 0-15 hold
    // row i = 16 (gw % 4) + lane of D_qs and the hi rows of D_ar, lanes 16-31
    // the lo rows of D_ar; one shuffle adds the pair, after which lane half
    // keeps 16 of the tile's 32 columns.
    const int qd = gw & 3, u = gw >> 2, half = lane >> 4;
    const int i = 16 * qd + (lane & 15);
    const uint32_t lb = (uint32_t)(32 * qd) << 16;
    const float qs = reinterpret_cast<const float*>(gsm + out::QS)[i];
    float x[32];
    {
      float d[64];
      tmem_ld64(tmem + lb + 64 * u, d);
#pragma unroll
      for (int e = 0; e < 32; ++e) x[e] = half ? 0.f : qs * (d[e] + d[32 + e]);
      tmem_ld64(tmem + lb + 128 + 64 * u, d);
#pragma unroll
      for (int e = 0; e < 32; ++e) x[e] += d[e] + d[32 + e];
    }
    float o[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float send = half ? x[e] : x[16 + e];
      const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
      o[e] = (half ? x[16 + e] : x[e]) + recv;
    }
    const int t = n * C + i;
    if (ok && t < p.T) out::store16(p, b, t, hv, 64 * vh + 32 * u + 16 * half, o);
    if (!ok && lane == 0) atomicOr(p.error_word, kErrOutWait);
    tc_fence_before();
    chunk::group_sync(bar_id);   // shared memory, TMEM and the claim free for the next item
  }
}

// ============================================================================ chain
// The next slab flags of a sequence (chunk slabs written by workers of the
// same launch): kFlagWindow of them read at once, then one acquire for the
// run of those already set. True when nflag advanced. After p.wait_limit
// fruitless polls it gives up: records it and sets nflag = N, so that the
// caller runs to its end on whatever the workspace holds (in bounds) and no
// other wait runs out too.
__device__ __forceinline__ bool poll_flags(const Params& p, int chunk0, int N, int& nflag,
                                           long& polls, bool& flags_ok) {
  unsigned int f[kFlagWindow];
#pragma unroll
  for (int z = 0; z < kFlagWindow; ++z)
    f[z] = nflag + z < N ? ld_relaxed_gpu(p.flags + chunk0 + nflag + z) : 0u;
  int m = nflag;
#pragma unroll
  for (int z = 0; z < kFlagWindow; ++z)
    if (m == nflag + z && f[z] != 0u) ++m;
  if (m > nflag) {
    fence_acq_rel_gpu();     // acquire the slabs' writes
    fence_async_global();    // ... for the bulk reads
    nflag = m;
    polls = 0;
    return true;
  }
  if (++polls > p.wait_limit) {
    flags_ok = false;
    nflag = N;
    atomicOr(p.error_word, kErrFlagWait);
  }
  return false;
}
// Chunks between export marks: kMarkEvery, or for long chains about 16 marks
// in all (each holds the exporter up).
__device__ __forceinline__ int mark_period(int N) {
  return N / 16 > kMarkEvery ? ((N / 16 + kMarkTail - 1) / kMarkTail) * kMarkTail : kMarkEvery;
}
// After the export of chunk nx (its bulk group committed): chunks 0 .. done - 1
// are in global memory once all but the newest kMarkLag groups are; announce
// them every mark_every chunks, and every kMarkTail in the last kMarkTailSpan.
__device__ __forceinline__ void mark_exports(unsigned int* mark, int nx, int N, int mark_every) {
  const int done = nx + 1 - kMarkLag;
  if (mark && done > 0 && nx + 1 < N &&
      (done % mark_every == 0 || (done >= N - kMarkTailSpan && done % kMarkTail == 0))) {
    bulk_wait<kMarkLag>();
    fence_async_global();
    st_release_gpu(mark, (unsigned int)done);
  }
}

// ------------------------------------------------------------------ SSD chain
// Mamba2 SSD (W = 0): r_n = U_n = v_n does not depend on the state, and the
// chunk-local stage has formed each chunk's state increment N_n = k_n^T
// diag(kscale_n) v_n (gdr_chunk_tc.cuh, Slab::ssd_n) and written r_n to the
// exchange block, so the chain is the fp32 scan
//     S_{n+1} = gamma_n S_n + N_n
// without a product. Shared memory (from the chain's 1024-aligned base): a
// ring of SSD_SLOTS increment boxes (this CTA's 32 value columns, [128 c][32 v]
// fp32, 128-byte swizzled rows) with gamma_n beside each, then the S tiles.
// Warps 0-7 hold S as in the delta-rule chain (thread (w, lane): channel
// 32 (w % 4) + lane, columns [16 (w / 4), 16 (w / 4) + 16)) and publish each
// S_n for the export; warp 12 loads the ring (waiting for the slab flags in
// the one-launch forward); warp 13 exports the S tiles and marks them.
constexpr int SSD_SLOTS = 6;
constexpr int SSD_SLOT = (int)Slab::SSD_N_BOX;
constexpr int SSD_OFF_GAM = SSD_SLOTS * SSD_SLOT;   // 16 bytes per slot
constexpr int SSD_OFF_S = SSD_OFF_GAM + 1024;
constexpr uint32_t SSD_TX = SSD_SLOT + 16;
static_assert(SSD_SLOT == 16384 && SSD_OFF_S % 1024 == 0 && SSD_OFF_S + S_TILES * 16384 <= OFF_BARS,
              "SSD chain shared memory");
enum : int {
  SB_FULL = 0,                      // [SSD_SLOTS] ring slot loaded
  SB_EMPTY = SB_FULL + SSD_SLOTS,   // [SSD_SLOTS] ring slot read (8 state warps)
  SB_ES = SB_EMPTY + SSD_SLOTS,     // [S_TILES] S_n published, barrier n % S_TILES (8 state warps)
  SB_XR = SB_ES + S_TILES           // [S_TILES] export of S_n read out (exporter)
};
static_assert(SB_XR + S_TILES <= B_SLOT, "SSD barriers below the TMEM slot word");

__device__ __forceinline__ void ssd_init_bars(uint64_t* bars) {
  for (int i = 0; i < SSD_SLOTS; ++i) {
    mbar_init(&bars[SB_FULL + i], 1);
    mbar_init(&bars[SB_EMPTY + i], 8);
  }
  for (int i = 0; i < S_TILES; ++i) {
    mbar_init(&bars[SB_ES + i], 8);
    mbar_init(&bars[SB_XR + i], 1);
  }
}

// All threads of the chain CTA; ok turns false (for the calling thread) when
// one of its waits gave up.
__device__ __forceinline__ void ssd_chain(const Params& p, uint8_t* sm, int seq, int vt, bool wait_flags,
                                          bool marks, uint8_t* xbase, bool& ok) {
  const int N = p.N, v0 = vt * VC, chunk0 = seq * N;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BARS);
  const uint32_t sb = smem_u32(sm);
  if (warp < 8) {
    const int qd = warp & 3, h = warp >> 2;
    const int c = 32 * qd + lane;
    float S[16];
    if (p.s0) {
      const float4* src =
          reinterpret_cast<const float4*>(p.s0 + ((size_t)seq * K + c) * V + v0 + 16 * h);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 x = src[q];
        S[4 * q] = x.x; S[4 * q + 1] = x.y; S[4 * q + 2] = x.z; S[4 * q + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) S[i] = 0.f;
    }
    for (int n = 0; n < N; ++n) {
      // Chunk n's slab first, although S_n does not need it: its export (and
      // the mark after it) must come after this CTA acquired chunk n's slab,
      // whose A_qk, row factors and r tiles the output items read once the
      // mark is out.
      const int sl = n % SSD_SLOTS;
      ok = warp_wait(&bars[SB_FULL + sl], (uint32_t)(n / SSD_SLOTS) & 1u, ok);
      // S_n into tile n % S_TILES once the export of S_{n - S_TILES} from it is read out.
      if (n >= S_TILES)
        ok = warp_wait(&bars[SB_XR + n % S_TILES], tile_parity(n - S_TILES, S_TILES), ok);
      publish16(sm + SSD_OFF_S + (n % S_TILES) * 16384, c, 2 * h, S);
      fence_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[SB_ES + n % S_TILES]);
      const uint8_t* box = sm + sl * SSD_SLOT;
      const float gam = *reinterpret_cast<const float*>(sm + SSD_OFF_GAM + sl * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 x = *reinterpret_cast<const float4*>(box + sw_off(c, 4 * h + q));
        S[4 * q] = fmaf(gam, S[4 * q], x.x);
        S[4 * q + 1] = fmaf(gam, S[4 * q + 1], x.y);
        S[4 * q + 2] = fmaf(gam, S[4 * q + 2], x.z);
        S[4 * q + 3] = fmaf(gam, S[4 * q + 3], x.w);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[SB_EMPTY + sl]);
    }
    if (p.sT) {
      float4* dst = reinterpret_cast<float4*>(p.sT + ((size_t)seq * K + c) * V + v0 + 16 * h);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        dst[q] = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
    }
  } else if (warp == 12) {
    if (lane == 0) {
      // Each increment box is read once, by this CTA.
      const uint64_t pol = l2_evict_first();
      int nl = 0, nflag = wait_flags ? 0 : N;
      bool flags_ok = wait_flags;
      long idle = 0, flag_polls = 0;
      while (nl < N && ok) {
        bool progress = false, polled = false;
        if (flags_ok && nflag < N && nflag < nl + 2) {
          polled = true;
          progress = poll_flags(p, chunk0, N, nflag, flag_polls, flags_ok);
        }
        const int sl = nl % SSD_SLOTS;
        if (nl < nflag &&
            (nl < SSD_SLOTS || mbar_test(&bars[SB_EMPTY + sl], (uint32_t)(nl / SSD_SLOTS - 1) & 1u))) {
          const uint8_t* slab = p.slabs + (size_t)(chunk0 + nl) * p.slab_bytes;
          uint64_t* fb = &bars[SB_FULL + sl];
          mbar_expect_tx(fb, SSD_TX);
          bulk_load_hint(sb + sl * SSD_SLOT, slab + Slab::ssd_n(vt), SSD_SLOT, fb, pol);
          bulk_load(sb + SSD_OFF_GAM + sl * 16, slab + Slab::VEC + 2 * C * 4, 16, fb);
          ++nl;
          progress = true;
        }
        if (progress) {
          idle = 0;
        } else {
          if (!polled && ++idle > kTmaIdleLimit) ok = false;
          __nanosleep(64);
        }
      }
    }
    __syncwarp();
  } else if (warp == 13) {
    if (lane == 0) {
      const uint64_t pol_keep = l2_evict_last();   // the output items read it next
      unsigned int* mark = marks ? p.xmark + (size_t)seq * VTILES + vt : nullptr;
      const int mark_every = mark_period(N);
      for (int nx = 0; nx < N && ok; ++nx) {
        ok = mbar_wait(&bars[SB_ES + nx % S_TILES], tile_parity(nx, S_TILES), kWaitLimit);
        if (!ok) break;
        bulk_store_hint(xbase + (size_t)nx * Xchg::BYTES + Xchg::S + vt * Xchg::S_TILE,
                        sb + SSD_OFF_S + (nx % S_TILES) * 16384, 16384, pol_keep);
        bulk_commit();
        // One export in flight: the previous chunk's tile is read out once all
        // but the newest group are (the state warps rewrite a tile three
        // chunks on; two in flight measured the same).
        if (nx > 0) {
          bulk_wait_read<1>();
          mbar_arrive(&bars[SB_XR + (nx - 1) % S_TILES]);
        }
        mark_exports(mark, nx, N, mark_every);
      }
      bulk_wait<0>();
      // All chunks, also after a wait gave up (recorded): the output items
      // never wait for exports that will not come.
      if (mark) {
        fence_async_global();
        st_release_gpu(mark, (unsigned int)N);
      }
    }
    __syncwarp();
  }
}

// seq = b * HV + hv, value columns [32 vt, 32 vt + 32). With maps (the
// one-launch forward): chunk n's slab is produced in the same launch (wait for
// its flag before loading it), the CTA first produces chunk vt of its
// sequence itself, the exports are marked for the output items, and the CTA
// joins them once its chain is done. With maps but not produce (chains and
// output items after a finished chunk-local stage) only the last two.
// kSsd = p.ssd (Mamba2 SSD), a template argument so that the delta-rule
// chain is compiled without the scan's code and the other way round (one
// kernel with both measured 1-2 us slower on the delta rule).
template <bool kSsd>
__device__ __forceinline__ void chain_role(const Params& p, uint8_t* sm, int seq, int vt,
                                           const chunk::Maps* maps, bool produce) {
  const bool wait_flags = maps != nullptr && produce;
  const int v0 = vt * VC;
  const int N = p.N;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk0 = seq * N;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BARS);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + B_SLOT);

  if (tid == 0 && kSsd) {
    ssd_init_bars(bars);
    mbar_fence_init();
  } else if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_FULLA + i], 1);
      mbar_init(&bars[B_EMPTYA + i], kEmptyA);
      mbar_init(&bars[B_FULLW + i], 1);
      mbar_init(&bars[B_EMPTYW + i], kEmptyW);
      mbar_init(&bars[B_FULLB + i], 1);
      mbar_init(&bars[B_EMPTYB + i], kEmptyB);
      mbar_init(&bars[B_WS + i], 1);
      mbar_init(&bars[B_DS + i], 1);
      mbar_init(&bars[B_RP + i], 4);
    }
    for (int i = 0; i < S_TILES; ++i) {
      mbar_init(&bars[B_ES + i], 8);
      mbar_init(&bars[B_XR + i], 1);
    }
    mbar_init(&bars[B_T], 1);
    mbar_fence_init();
  }
  if (warp == 13) tmem_alloc(tslot, CHAIN_TMEM);
  tc_fence_before();
  nb_sync(1, CHAIN_THREADS);
  tc_fence_after();
  const uint32_t tmem = *tslot;
  bool ok = true;
  if (wait_flags && vt < N) {
    // The sequence's first chunks come from its own chain CTAs (chunks vt,
    // vt + 4, ... below kChainChunks here, by warps 0-7 in the worker group
    // layout over the rings, which are idle until the chain starts): their
    // SMs have nothing else in flight, and a worker's first chunk is slow.
    if (warp < 8) {
      if (tid == 0) chunk::init_group_bars(sm);
      chunk::group_sync(kProduceBar);
      uint32_t ph = 0;
      for (int n = vt; n < N && n < kChainChunks; n += VTILES) {
        chunk::produce_chunk<kSsd>(*maps, p, sm, tid, kProduceBar, n, seq % p.HV, seq / p.HV, ph, tmem,
                             nullptr, nullptr);
        if (tid == 0) {
          bulk_wait<0>();
          fence_async_global();
          st_release_gpu(p.flags + chunk0 + n, 1u);
        }
        ph ^= 1u;
      }
    }
    tc_fence_before();
    nb_sync(1, CHAIN_THREADS);
    tc_fence_after();
    if (tid == 0) {
      uint64_t* gb = reinterpret_cast<uint64_t*>(sm + chunk::OFF_BAR);
      for (int i = 0; i < chunk::kNumBars; ++i)
        if (i != 2) mbar_inval(gb + i);   // (index 2 holds the TMEM slot word, not a barrier)
    }
    nb_sync(1, CHAIN_THREADS);
  }
  uint8_t* xbase = p.xchg + (size_t)chunk0 * Xchg::BYTES;
  const uint32_t sb = smem_u32(sm);
  constexpr uint32_t ID_KMN = idesc_bf16(128, 64, 0, 1);   // A K-major, B MN-major
  constexpr uint32_t ID_MNMN = idesc_bf16(128, 64, 1, 1);  // A = k^T read MN-major

  if (kSsd) {
    ssd_chain(p, sm, seq, vt, wait_flags, maps != nullptr, xbase, ok);
  } else if (warp < 8) {
    // ---------------------------------------------------------------- state
    // After publishing S_n the eight warps meet on named barrier 2, which
    // releases the D_ws issuer (warp 15).
    const int qd = warp & 3, h = warp >> 2;
    const int c = 32 * qd + lane;                        // key channel = TMEM lane
    const uint32_t lb = (uint32_t)(32 * qd) << 16;
    float S[16];
    if (p.s0) {
      const float4* src =
          reinterpret_cast<const float4*>(p.s0 + ((size_t)seq * K + c) * V + v0 + 16 * h);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 x = src[q];
        S[4 * q] = x.x; S[4 * q + 1] = x.y; S[4 * q + 2] = x.z; S[4 * q + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) S[i] = 0.f;
    }
    float gam = 1.f;
    for (int n = 0; n <= N; ++n) {
      if (n > 0) {
        // S_n = gamma_{n-1} S_{n-1} + D_S(n) (hi and lo columns of B), from
        // D_S buffer (n - 1) % 2.
        const int bs = (n - 1) & 1;
        ok = warp_wait(&bars[B_DS + bs], ((n - 1) >> 1) & 1, ok);
        if (lane == 0) mbar_arrive(&bars[B_EMPTYB + bs]);   // k_{n-1} read
        tc_fence_after();
        float d[32];
        const uint32_t ts = tmem + lb + T_S + 64 * bs;
        tmem_ld16x2(ts + 16 * h, ts + 32 + 16 * h, d);
#pragma unroll
        for (int i = 0; i < 16; ++i) S[i] = fmaf(gam, S[i], d[i] + d[16 + i]);
        tc_fence_before();
      }
      if (n == N) break;
      // S tile n % 3 held S_{n-3}: D_ws(n - 2) read it, and completed before
      // D_ws(n - 1), whose completion the r warps saw before rho_{n-1}, the
      // operand of D_S(n); its export is checked.
      if (n >= S_TILES)
        ok = warp_wait(&bars[B_XR + n % S_TILES], tile_parity(n - S_TILES, S_TILES), ok);
      uint8_t* st = sm + OFF_S + (n % S_TILES) * 16384;
      publish16(st, c, 2 * h, S);
      fence_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_ES + n % S_TILES]);   // for the exporter
      tc_fence_before();
      // (a sync, not an arrive: a state warp that ran a step ahead could
      // otherwise complete the phase of a slower one and release D_ws early)
      nb_sync(2, 288);
      // gamma_n for S_{n+1}; then this warp is done with ring A slot n % 2.
      ok = warp_wait(&bars[B_FULLA + (n & 1)], (n >> 1) & 1, ok);
      gam = reinterpret_cast<const float*>(sm + OFF_V + (n & 1) * VEC_BYTES)[C];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_EMPTYA + (n & 1)]);
    }
    if (p.sT) {
      float4* dst = reinterpret_cast<float4*>(p.sT + ((size_t)seq * K + c) * V + v0 + 16 * h);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        dst[q] = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
    }
  } else if (warp < 12) {
    // -------------------------------------------------------------------- r
    // After publishing rho_n the four warps arrive on named barrier 3, which
    // releases the D_S / D_t issuer (warp 14).
    const int qd = warp - 8;
    const uint32_t lb = (uint32_t)(32 * qd) << 16;
    const int half = lane >> 4;
    const int j = 16 * qd + (lane & 15);                 // r row of this lane
    float gam_prev = 1.f;
    for (int n = 0; n < N; ++n) {
      const int sa = n & 1;
      const uint8_t* slot = sm + OFF_A + sa * A_SLOT;
      ok = warp_wait(&bars[B_WS + sa], (n >> 1) & 1, ok);
      if (lane == 0) mbar_arrive(&bars[B_EMPTYW + sa]);   // D_ws(n) done: W_n read
      ok = warp_wait(&bars[B_FULLA + sa], (n >> 1) & 1, ok);
      tc_fence_after();
      float r[16];
      {
        float d[64];
        tmem_ld64(tmem + lb + T_WS + 64 * sa, d);
        stacked_sum(d, half, r);
      }
      const float* vec = reinterpret_cast<const float*>(sm + OFF_V + sa * VEC_BYTES);
      const float ks = vec[j];
      const float gam_n = vec[C];
      const float uf = p.zero_u ? 0.f : 1.f;
      const uint8_t* ub = slot + A_U;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 u = *reinterpret_cast<const float4*>(ub + sw_off(j, 4 * half + q));
        r[4 * q] = fmaf(gam_prev, r[4 * q], uf * u.x);
        r[4 * q + 1] = fmaf(gam_prev, r[4 * q + 1], uf * u.y);
        r[4 * q + 2] = fmaf(gam_prev, r[4 * q + 2], uf * u.z);
        r[4 * q + 3] = fmaf(gam_prev, r[4 * q + 3], uf * u.w);
      }
      if (n > 0) {
        ok = warp_wait(&bars[B_T], (n - 1) & 1, ok);
        tc_fence_after();
        float d[64], t[16];
        tmem_ld64(tmem + lb + T_T, d);
        stacked_sum(d, half, t);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] += t[i];
      }
      tc_fence_before();
      // rho into tile n % 2: rho_{n-2} there was read by D_S(n - 1) and
      // D_t(n - 1), issued by the same thread before D_t(n), whose completion
      // this step waited for.
      float rho[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) rho[i] = r[i] * ks;
      publish16(sm + OFF_P + sa * 8192, j, 2 * half, rho);
      fence_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_EMPTYA + sa]);   // U, VEC read; D_t(n) (T_n) done
      tc_fence_before();
      // An arrive: r_{n+1} needs D_t(n + 1), issued only after this phase, so
      // no r warp can reach the next phase early.
      nb_arrive(3, 160);
      // r into its tile n % 2 once the export of r_{n-2} from it is read out.
      if (n >= 2) ok = warp_wait(&bars[B_XR + (n - 2) % S_TILES], tile_parity(n - 2, S_TILES), ok);
      publish16(sm + OFF_R + sa * 8192, j, 2 * half, r);
      fence_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_RP + (n & 1)]);
      gam_prev = gam_n;
    }
  } else if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    // Ring W takes chunk nw once its slot is free (chunk nw - 2 done), rings A
    // and B likewise; one bulk copy per array.
    if (lane == 0) {
      const uint32_t sb = smem_u32(sm);
      int nw = 0, na = 0, nb = 0, nflag = wait_flags ? 0 : N;   // nflag: flags seen
      // This CTA's U columns are read once; -W, -T and k by the four V-tile
      // CTAs of the sequence.
      const uint64_t pol_last_read = l2_evict_first();
      bool flags_ok = wait_flags;
      long idle = 0, flag_polls = 0;
      while ((nw < N || na < N || nb < N) && ok) {
        bool progress = false, polled = false;
        const int lead = nw > na ? (nw > nb ? nw : nb) : (na > nb ? na : nb);
        if (flags_ok && nflag < N && nflag < lead + 2) {
          polled = true;
          progress = poll_flags(p, chunk0, N, nflag, flag_polls, flags_ok);
        }
        if (nw < N && nw < nflag &&
            (nw < 2 || mbar_test(&bars[B_EMPTYW + (nw & 1)], ((nw >> 1) - 1) & 1))) {
          uint64_t* fb = &bars[B_FULLW + (nw & 1)];
          mbar_expect_tx(fb, W_TX);
          bulk_load(sb + OFF_W + (nw & 1) * W_SLOT, p.slabs + (size_t)(chunk0 + nw) * p.slab_bytes + Slab::W2,
                    32768, fb);
          ++nw;
          progress = true;
        }
        if (na < N && na < nflag &&
            (na < 2 || mbar_test(&bars[B_EMPTYA + (na & 1)], ((na >> 1) - 1) & 1))) {
          const uint8_t* slab = p.slabs + (size_t)(chunk0 + na) * p.slab_bytes;
          uint64_t* fb = &bars[B_FULLA + (na & 1)];
          const uint32_t slot = sb + OFF_A + (na & 1) * A_SLOT;
          mbar_expect_tx(fb, A_TX);
          bulk_load(slot + A_T, slab + Slab::T2, 16384, fb);   // (first chunk: not used)
          bulk_load_hint(slot + A_U, slab + Slab::U + vt * 8192, 8192, fb, pol_last_read);
          bulk_load(sb + OFF_V + (na & 1) * VEC_BYTES, slab + Slab::VEC + VEC_OFF, VEC_BYTES, fb);
          ++na;
          progress = true;
        }
        if (nb < N && nb < nflag &&
            (nb < 2 || mbar_test(&bars[B_EMPTYB + (nb & 1)], ((nb >> 1) - 1) & 1))) {
          uint64_t* fb = &bars[B_FULLB + (nb & 1)];
          const uint32_t slot = sb + OFF_B + (nb & 1) * KB_SLOT;
          mbar_expect_tx(fb, B_TX);
          bulk_load(slot, p.slabs + (size_t)(chunk0 + nb) * p.slab_bytes + Slab::K2, 16384, fb);
          ++nb;
          progress = true;
        }
        if (progress) {
          idle = 0;
        } else {
          // (a flag wait has its own bound, p.wait_limit polls)
          if (!polled && ++idle > kTmaIdleLimit) ok = false;
          __nanosleep(64);
        }
      }
    }
    __syncwarp();
  } else if (warp == 14) {
    // ------------------------------------------------------- D_S / D_t issuer
    // Once rho_n is published (named barrier 3): D_S(n + 1) = k_n^T rho_n into
    // D_S buffer n % 2 (read for S_{n-1}, which D_ws(n), complete before rho_n,
    // consumed), then D_t(n + 1) = (-T_{n+1}) rho_n (the last round: D_S(N)
    // alone, for the final state). (D_t first measured slower: S_{n+1}, and
    // with it D_ws(n + 2), comes later.)
    for (int n = 0; n < N; ++n) {
      nb_sync(3, 160);
      if (lane == 0 && ok) {
        const int sa = n & 1;
        ok = mbar_spin(&bars[B_FULLB + sa], (n >> 1) & 1, kWaitLimit);   // k_n
        if (ok) {
          tc_fence_after();
          const uint32_t kb = sb + OFF_B + sa * KB_SLOT;
          const uint32_t pt = sb + OFF_P + sa * 8192;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem + T_S + 64 * sa, sdesc_sw128_lbo(kb + kk * 2048, 8192),
                      sdesc_sw128_lbo(pt + kk * 2048, 8192), ID_MNMN, kk > 0);
          umma_commit(&bars[B_DS + sa]);
        }
        if (ok && n + 1 < N) {
          const int m = n + 1;
          ok = mbar_spin(&bars[B_FULLA + (m & 1)], (m >> 1) & 1, kWaitLimit);   // T_{n+1}
          if (ok) {
            const uint32_t ta = sb + OFF_A + (m & 1) * A_SLOT + A_T;
            const uint32_t pt = sb + OFF_P + sa * 8192;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16(tmem + T_T, sdesc_sw128(ta + kk * 32), sdesc_sw128_lbo(pt + kk * 2048, 8192),
                        ID_KMN, kk > 0);
            umma_commit(&bars[B_T]);
          }
        }
      }
      __syncwarp();
    }
  } else if (warp == 15) {
    // ------------------------------------------------------------ D_ws issuer
    // Once S_n is published (named barrier 2): D_ws(n + 1) = (-W_{n+1}) S_n
    // into buffer (n + 1) % 2 (after S_0 also D_ws(0) = (-W_0) S_0).
    auto issue_ws = [&](int m) {
      ok = mbar_spin(&bars[B_FULLW + (m & 1)], (m >> 1) & 1, kWaitLimit);
      if (!ok) return;
      const uint32_t wa = sb + OFF_W + (m & 1) * W_SLOT;
      const uint32_t st = sb + OFF_S + ((m > 0 ? m - 1 : 0) % S_TILES) * 16384;
      const uint32_t d = tmem + T_WS + 64 * (m & 1);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma_bf16(d, sdesc_sw128(wa + (kk >> 2) * 16384 + (kk & 3) * 32),
                  sdesc_sw128_lbo(st + kk * 2048, 8192), ID_KMN, kk > 0);
      umma_commit(&bars[B_WS + (m & 1)]);
    };
    for (int n = 0; n < N; ++n) {
      nb_sync(2, 288);
      if (lane == 0 && ok) {
        tc_fence_after();
        if (n == 0) issue_ws(0);
        if (ok && n + 1 < N) issue_ws(n + 1);
      }
      __syncwarp();
    }
  } else if (warp == 13) {
    // ---------------------------------------------------------------- exporter
    if (lane == 0) {
      // The output pass reads the exchange next: keep it in L2.
      const uint64_t pol_keep = l2_evict_last();
      unsigned int* mark = maps ? p.xmark + (size_t)seq * VTILES + vt : nullptr;
      const int mark_every = mark_period(N);
      for (int nx = 0; nx < N && ok; ++nx) {
        ok = mbar_wait(&bars[B_ES + nx % S_TILES], tile_parity(nx, S_TILES), kWaitLimit) &&
             mbar_wait(&bars[B_RP + (nx & 1)], (nx >> 1) & 1, kWaitLimit);
        if (!ok) break;
        // Both tiles of chunk nx out as one bulk group; once read out they may
        // be rewritten.
        uint8_t* xb = xbase + (size_t)nx * Xchg::BYTES;
        bulk_store_hint(xb + Xchg::S + vt * Xchg::S_TILE, sb + OFF_S + (nx % S_TILES) * 16384, 16384,
                        pol_keep);
        bulk_store_hint(xb + Xchg::R + vt * Xchg::R_TILE, sb + OFF_R + (nx & 1) * 8192, 8192, pol_keep);
        bulk_commit();
        // One export in flight: the previous chunk's tiles are read out once
        // all but the newest group are (an S tile is rewritten three chunks
        // on, an r tile two).
        if (nx > 0) {
          bulk_wait_read<1>();
          mbar_arrive(&bars[B_XR + (nx - 1) % S_TILES]);
        }
        mark_exports(mark, nx, N, mark_every);
      }
      bulk_wait<0>();
      // All chunks, also after a wait gave up (recorded): the output items
      // never wait for exports that will not come.
      if (mark) {
        fence_async_global();
        st_release_gpu(mark, (unsigned int)N);
      }
    }
    __syncwarp();
  }
  if (!ok) atomicOr(p.error_word, kErrChainWait);

  tc_fence_before();
  nb_sync(1, CHAIN_THREADS);
  if (maps) {
    // One-launch forward: the CTA joins the output work as two groups of 8
    // warps in the worker group layout, each with 256 of the chain's TMEM
    // columns (the chain's tiles and rings are dead).
    tc_fence_after();
    const int grp = warp >> 3;
    uint8_t* gsm = sm + grp * chunk::GROUP_BYTES;
    if ((tid & 255) == 0) chunk::init_group_bars(gsm);
    output_items(&maps->q, p, gsm, tid & 255, 1 + grp, tmem + 256 * grp, 0u, 0u);
    // (barrier 0: group 0 may still be on named barrier 1 with 256 threads)
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, CHAIN_TMEM);
  }
}

template <bool kSsd>
__global__ void __launch_bounds__(CHAIN_THREADS, 1) chain_kernel(Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  chain_role<kSsd>(p, sm, blockIdx.y * p.HV + blockIdx.x / VTILES, blockIdx.x % VTILES, nullptr, false);
}


// =========================================================================== worker
// Two groups of 8 warps run the chunk-local stage over chunk items in chunk
// order (item it: chunk it / (B HV) of sequence it % (B HV)); group G of NG
// takes items G, G + NG, ... (the groups 0 of all workers first). Then each
// group takes output items. (Holding group 1 back until group 0's first chunk
// was done measured 2 us slower: a worker's first chunk takes ~19 us even
// alone on its SM, against ~12 us for its later ones.)
template <bool kSsd>
__device__ __forceinline__ void worker_role(const chunk::Maps& maps, const Params& p,
                                            uint8_t* sm_base, int worker, int n_workers, bool produce) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int grp = warp >> 3, gtid = tid & 255;
  uint8_t* sm = sm_base + grp * chunk::GROUP_BYTES;
  // The CTA's TMEM allocation (both groups' 256 columns) is recorded in the
  // TMEM slot of group 0, which produce_chunk leaves alone when given its columns.
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm_base + chunk::OFF_BAR) + 4;
  if (gtid == 0) chunk::init_group_bars(sm);
  if (warp == 0) tmem_alloc(tslot, 2 * chunk::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot + grp * chunk::TMEM_COLS;
  const int nseq = p.B * p.HV;
  const long items = (long)nseq * p.N;
  const int G = grp * n_workers + worker, NG = 2 * n_workers;
  // (chunks 0 .. kChainChunks - 1 of every sequence come from its chain CTAs)
  const long first = produce ? (long)nseq * (p.N < kChainChunks ? p.N : kChainChunks) : items;
  unsigned int* pending = nullptr;
  uint32_t ph = 0;
  for (long it = first + G; it < items; it += NG) {
    const int n = (int)(it / nseq), seq = (int)(it % nseq);
    const int b = seq / p.HV, hv = seq % p.HV;
    chunk::produce_chunk<kSsd>(maps, p, sm, gtid, 1 + grp, n, hv, b, ph, tmem, nullptr, pending);
    pending = p.flags + slab_index(p, b, hv, n);
    if (it < first + NG) {
      // The first wave (the chunks the chains reach first): published at once
      // rather than at the start of the next item.
      if (gtid == 0) {
        bulk_wait<0>();
        fence_async_global();
        st_release_gpu(pending, 1u);
      }
      pending = nullptr;
    }
    ph ^= 1u;
  }
  if (gtid == 0 && pending) {
    bulk_wait<0>();
    fence_async_global();
    st_release_gpu(pending, 1u);
  }
  // Then the output items. The chunk stage's MMA barrier completed two phases
  // per item, so its next phase has parity 0; its TMA barrier one (ph).
  output_items(&maps.q, p, sm, gtid, 1 + grp, tmem, ph, 0u);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(*tslot, 2 * chunk::TMEM_COLS);
  }
}

template <bool kSsd>
__global__ void __launch_bounds__(FUSED_THREADS, 1)
    fused_kernel(const __grid_constant__ chunk::Maps maps, Params p, int n_chain, int n_workers, int produce) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int cta = blockIdx.x;
  if (cta < n_chain) {
    if (threadIdx.x < CHAIN_THREADS) chain_role<kSsd>(p, sm, cta / VTILES, cta % VTILES, &maps, produce != 0);
  } else {
    worker_role<kSsd>(maps, p, sm, cta - n_chain, n_workers, produce != 0);
  }
}

// =========================================================================== outputs
// The output pass after a finished recurrence: one CTA per (sequence, 64 value
// columns vh, chunk n), the products of namespace out.
struct OutMaps {
  CUtensorMap q;
};

__global__ void __launch_bounds__(out::THREADS, 2)
    output_kernel(const __grid_constant__ OutMaps maps, Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int vh = blockIdx.x & 1, seq = blockIdx.x >> 1, n = blockIdx.y;
  const int b = seq / p.HV, hv = seq % p.HV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + out::BAR);
  uint64_t* mma_bar = bar + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 2);
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(mma_bar, 1);
    mbar_fence_init();
    out::issue_loads(&maps.q, p, smem_u32(sm), seq, n, vh, bar);
  }
  if (warp == 1) tmem_alloc(tslot, out::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  bool ok = true;
  if (tid == 0) {
    ok = mbar_wait(bar, 0, kWaitLimit);
    if (ok) {
      tc_fence_after();
      out::issue_mmas(tmem, smem_u32(sm));
    }
    umma_commit(mma_bar);
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  ok = __all_sync(0xffffffffu, mbar_wait(mma_bar, 0, kWaitLimit)) && ok;
  tc_fence_after();
  // Warp w: rows i = 16 w + lane % 16 (lanes 0-15: D_qs rows and the hi rows of
  // D_ar; lanes 16-31: the lo rows of D_ar). Column 64 u + x of either
  // accumulator is tile u, part x / 32 (hi, lo), value column 32 u + x % 32 of
  // this CTA's 64; lane half keeps tile u = half.
  const int half = lane >> 4;
  const int i = 16 * warp + (lane & 15);
  const uint32_t lb = (uint32_t)(32 * warp) << 16;
  const float qs = reinterpret_cast<const float*>(sm + out::QS)[i];
  float x[2][32];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    float d[64];
    tmem_ld64(tmem + lb + 64 * u, d);
#pragma unroll
    for (int e = 0; e < 32; ++e) x[u][e] = half ? 0.f : qs * (d[e] + d[32 + e]);
    tmem_ld64(tmem + lb + 128 + 64 * u, d);
#pragma unroll
    for (int e = 0; e < 32; ++e) x[u][e] += d[e] + d[32 + e];
  }
  float o[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const float send = half ? x[0][e] : x[1][e];       // the partner keeps tile 1 - half
    const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
    o[e] = (half ? x[1][e] : x[0][e]) + recv;
  }
  const int t = n * C + i;
  if (ok && t < p.T) {
    const size_t off = (((size_t)b * p.T + t) * p.HV + hv) * V + 64 * vh + 32 * half;
    if (p.out_bf16) {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + off);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        dst[q] = make_uint4(pack_bf16(o[8 * q], o[8 * q + 1]), pack_bf16(o[8 * q + 2], o[8 * q + 3]),
                            pack_bf16(o[8 * q + 4], o[8 * q + 5]), pack_bf16(o[8 * q + 6], o[8 * q + 7]));
    } else {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + off);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    }
  }
  if (!ok && tid == 0) atomicOr(p.error_word, kErrOutWait);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, out::TMEM_COLS);
  }
}

struct DeviceInfo {
  int sms = 0;
  bool coop = false;
};

DeviceInfo& device_info() {
  static DeviceInfo cache[64];
  static bool known[64] = {};
  static DeviceInfo none;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    none = DeviceInfo{};
    return none;
  }
  if (known[dev]) return cache[dev];
  DeviceInfo d;
  int coop = 0;
  cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  d.coop = coop != 0;
  cache[dev] = d;
  known[dev] = true;
  return cache[dev];
}

}  // namespace

gdr_status launch_chain(const Params& p, cudaStream_t stream) {
  if (p.gate_mode != 0 || !p.xchg) return GDR_ERR_UNSUPPORTED;
  const auto kern = p.ssd ? chain_kernel<true> : chain_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           CHAIN_SMEM) != cudaSuccess)
    return GDR_ERR_CUDA;
  dim3 grid(p.HV * VTILES, p.B);
  kern<<<grid, CHAIN_THREADS, CHAIN_SMEM, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

gdr_status launch_outputs(const Params& p, cudaStream_t stream) {
  if (p.gate_mode != 0 || !p.xchg) return GDR_ERR_UNSUPPORTED;
  if (p.N > 65535) return GDR_ERR_UNSUPPORTED;
  OutMaps m;
  if (!tmap_bthd(&m.q, p.q, p.B, p.T, p.H)) return GDR_ERR_CUDA;
  if (cudaFuncSetAttribute(output_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           out::SMEM) != cudaSuccess)
    return GDR_ERR_CUDA;
  dim3 grid(2 * p.B * p.HV, p.N);
  output_kernel<<<grid, out::THREADS, out::SMEM, stream>>>(m, p);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

bool fused_fits(int B, int HV) {
  const DeviceInfo& dev = device_info();
  const long long n_chain = (long long)B * HV * VTILES;
  // The workers must produce chunks about as fast as the chains consume them:
  // at least as many worker CTAs as chain CTAs.
  return dev.coop && dev.sms > 0 && n_chain * 2 <= dev.sms;
}

namespace {

// One cooperative launch of fused_kernel: with produce, the whole forward;
// without, the chains and the output items after a finished chunk-local stage.
gdr_status launch_one(const Params& p, cudaStream_t stream, bool produce) {
  const DeviceInfo& dev = device_info();
  const int n_chain = p.B * p.HV * VTILES;
  const int n_workers = dev.sms - n_chain;
  chunk::Maps m;
  if (!chunk::make_maps(&m, p)) return GDR_ERR_CUDA;
  const auto kern = p.ssd ? fused_kernel<true> : fused_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FUSED_SMEM) != cudaSuccess)
    return GDR_ERR_CUDA;
  // Slab flags, export marks and the output item counter start at zero.
  const size_t words = (size_t)p.B * p.HV * (p.N + VTILES) + 1;
  if (!p.xmark || p.xmark != p.flags + (size_t)p.B * p.HV * p.N) return GDR_ERR_UNSUPPORTED;
  if (cudaMemsetAsync(p.flags, 0, words * sizeof(unsigned int), stream) != cudaSuccess)
    return GDR_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(dev.sms);
  cfg.blockDim = dim3(FUSED_THREADS);
  cfg.dynamicSmemBytes = FUSED_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, m, p, n_chain, n_workers, produce ? 1 : 0);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return e == cudaErrorCooperativeLaunchTooLarge ? GDR_ERR_UNSUPPORTED : GDR_ERR_CUDA;
  }
  return GDR_OK;
}

}  // namespace

gdr_status launch_fused(const Params& p, cudaStream_t stream) {
  if (p.gate_mode != 0 || !p.flags || !p.xchg || !fused_fits(p.B, p.HV)) return GDR_ERR_UNSUPPORTED;
  return launch_one(p, stream, true);
}

gdr_status launch_chain_outputs(const Params& p, cudaStream_t stream) {
  const DeviceInfo& dev = device_info();
  if (p.gate_mode != 0 || !p.flags || !p.xchg || !dev.coop || dev.sms <= 0 ||
      (long long)p.B * p.HV * VTILES > dev.sms)
    return GDR_ERR_UNSUPPORTED;
  return launch_one(p, stream, false);
}

}  // namespace fast
}  // namespace gdr
