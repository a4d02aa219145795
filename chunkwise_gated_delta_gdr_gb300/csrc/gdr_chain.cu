// gdr_chain.cu -- inter-chunk recurrence of the fast path for the scalar gate
// (Gated DeltaNet) on tcgen05 tensor cores, and the one-launch forward.
//
// Per chunk n the inter-chunk loop of the "分块并行计算（Chunkwise）" notes
// (section "chunk 间递推") reads
//     r_n     = U_n - W_n S_n
//     o_n     = (q exp(G)) S_n + A_qk r_n
//     S_{n+1} = exp(G_last) S_n + (exp(G_last - G) k)^T (beta r_n)
// Only the S update is serial. One chain CTA per (batch, value head, 32 value
// columns v0 .. v0 + 31) keeps its 128 x 32 slice of S in fp32 registers (one
// key channel per thread) for the whole sequence and forms the chunk outputs
// of its columns as it goes. Per chunk, on tcgen05 (kind::f16, fp32
// accumulators in TMEM):
//     D_r  = [-W_hi; -W_lo] [S_hi | S_lo]      M = 128 (stacked rows), N = 64, K = 128
//     r    = U + (the four quarters of D_r),   rho = kscale r        (fp32, registers)
//     D_S  = k^T [rho_hi | rho_lo]             M = 128, N = 64, K = 64 (k raw bf16)
//     S    = gamma S + (the two halves of D_S)
//     D_qs = q [S_hi | S_lo]                   M = 64,  N = 64, K = 128 (q raw bf16)
//     D_ar = [A_hi; A_lo] [r_hi | r_lo]        M = 128 (stacked rows), N = 64, K = 64
//     o    = qscale (D_qs halves) + (the four quarters of D_ar)
// Every operand holding fp32 values enters as a bf16 hi + lo pair: hi hi,
// hi lo and lo hi products (the lo lo products come along and are kept). q and
// k are exact in bf16 and carry their L2 norms, scale and decays as fp32 row
// factors (qscale, kscale), which is why their products need no lo part.
//
// Roles of a chain CTA (10 warps):
//   warps 0-3  the state: thread (w, lane) holds channel c = 32 w + lane (TMEM
//              lane c of D_S). They form r from D_r (lanes 0-15 hold the hi
//              rows j = 16 w + lane, lanes 16-31 the lo rows of the same j),
//              publish r and rho as MN-major B operands, then S from D_S, and
//              publish S (bf16 hi | lo per row, 128-byte swizzled).
//   warps 4-7  the outputs: o rows i = 16 (w - 4) + lane % 16, 16 columns per
//              lane, stored straight to global memory (rows past T skipped).
//   warp 8     TMA producer: -W (stacked), k, q, A_qk (stacked), the U tile
//              and VEC of chunk n into one of two operand stages.
//   warp 9     MMA issuer and TMEM owner, per chunk in the order D_r, D_qs,
//              D_S, D_ar: the output products run while the state warps work
//              on r and on S and never sit in front of D_r or D_S.
// TMEM: D_r 64 columns, D_S 64, two output accumulator pairs (D_qs, D_ar) of
// 128 so that one chunk's outputs are read while the next chunk's are formed.
//
// One-launch forward (launch_fused): one cooperative launch of one CTA per SM.
// The first CTAs take the chain role; the others are workers, two groups of 8
// warps each, that run the chunk-local stage (gdr_chunk_tc.cuh) over the
// chunks in chunk order and raise each chunk's flag once its slab is in
// global memory. A chain's TMA warp waits for chunk n's flag before loading
// it. Workers never wait on chains and all CTAs are co-resident, so the waits
// end; every wait is bounded all the same and records a code in the workspace
// error word when it gives up, after which the CTA runs to its end.
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
constexpr int CHAIN_THREADS = 320;
constexpr int FUSED_THREADS = 512;      // worker CTA: two chunk groups of 256
constexpr long kWaitLimit = 1L << 24;   // mbarrier polls before a wait gives up
constexpr unsigned int kErrChainWait = 4u, kErrFlagWait = 8u;

// Shared memory of a chain CTA (bytes from a 1024-aligned base). Operand stage:
constexpr int ST_W = 0;          // -W stacked [128][128] bf16: two [128][64] boxes
constexpr int ST_K = 32768;      // k [64 j][128 c] bf16: two [64][64] boxes
constexpr int ST_Q = 49152;      // q [64 i][128 c] bf16: two [64][64] boxes
constexpr int ST_AQ = 65536;     // A_qk stacked [128][64] bf16
constexpr int ST_U = 81920;      // U [64 j][32 v] fp32, 128-byte swizzled
constexpr int ST_VEC = 90112;    // qscale[64], kscale[64], gamma[128] fp32
constexpr int STAGE = 91136;
constexpr uint32_t STAGE_TX = 32768 + 16384 + 16384 + 16384 + 8192 + 1024;
constexpr int NST = 2;
constexpr int S_TILE = NST * STAGE;      // S [128 c][S_hi 32 | S_lo 32] bf16, swizzled rows
constexpr int R_TILE = S_TILE + 16384;   // r [64 j][r_hi 32 | r_lo 32]
constexpr int P_TILE = R_TILE + 8192;    // rho [64 j][rho_hi 32 | rho_lo 32]
constexpr int BARS = P_TILE + 8192;
constexpr int CHAIN_SMEM = BARS + 256 + 1024;
static_assert(STAGE % 1024 == 0 && S_TILE % 1024 == 0 && R_TILE % 1024 == 0 &&
                  P_TILE % 1024 == 0,
              "swizzled tiles need 1 KB alignment");
static_assert(CHAIN_SMEM <= 232448, "chain shared memory");
constexpr int FUSED_SMEM =
    (CHAIN_SMEM > 2 * chunk::GROUP_BYTES + 1024) ? CHAIN_SMEM : 2 * chunk::GROUP_BYTES + 1024;
static_assert(FUSED_SMEM <= 232448, "one-launch shared memory");

// TMEM columns.
constexpr uint32_t T_R = 0, T_S = 64, T_O = 128;   // output pair b: D_qs at T_O + 128 b, D_ar + 64
constexpr uint32_t TMEM_COLS = 512;

__device__ __forceinline__ void nb_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Byte offset of 16-byte chunk q of row r in 128-byte swizzled rows.
__device__ __forceinline__ uint32_t sw_off(int r, int q) {
  return (uint32_t)(r * 128 + ((q ^ (r & 7)) << 4));
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

// ============================================================================ chain
// seq = b * HV + hv, value columns [32 vt, 32 vt + 32). wait_flags: chunk n's
// slab is produced in the same launch (wait for its flag before loading it).
__device__ __forceinline__ void chain_role(const chunk::Maps& maps, const Params& p, uint8_t* sm,
                                           int seq, int vt, bool wait_flags) {
  const int b = seq / p.HV, hv = seq % p.HV, h = hv / (p.HV / p.H);
  const int v0 = vt * VC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk0 = seq * p.N;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + BARS);
  uint64_t* full = bars;           // [NST] operand stage loaded
  uint64_t* empty = bars + 2;      // [NST] stage free: MMA commit + 4 output warps (VEC read)
  uint64_t* s_ready = bars + 4;    // S tile published (4 state warps)
  uint64_t* rho_ready = bars + 5;  // r and rho tiles published (4 state warps)
  uint64_t* r_done = bars + 6;     // D_r complete (commit)
  uint64_t* ds_done = bars + 7;    // D_S complete (commit)
  uint64_t* o_full = bars + 8;     // [2] output pair complete (commit)
  uint64_t* o_empty = bars + 10;   // [2] output pair read (4 output warps)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 12);

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 5);
    }
    mbar_init(s_ready, 4);
    mbar_init(rho_ready, 4);
    mbar_init(r_done, 1);
    mbar_init(ds_done, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&o_full[i], 1);
      mbar_init(&o_empty[i], 4);
    }
    mbar_fence_init();
  }
  if (warp == 9) tmem_alloc(tslot, TMEM_COLS);
  tc_fence_before();
  nb_sync(1, CHAIN_THREADS);
  tc_fence_after();
  const uint32_t tmem = *tslot;
  bool ok = true;

  if (warp < 4) {
    // ---------------------------------------------------------------- state
    const int c = 32 * warp + lane;                      // key channel = TMEM lane
    const uint32_t lb = (uint32_t)(32 * warp) << 16;
    const int half = lane >> 4;
    const int j = 16 * warp + (lane & 15);               // r row of this lane's D_r lane
    uint8_t* stile = sm + S_TILE;
    float S[32];
    if (p.s0) {
      const float4* src = reinterpret_cast<const float4*>(p.s0 + ((size_t)seq * K + c) * V + v0);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 x = src[q];
        S[4 * q] = x.x; S[4 * q + 1] = x.y; S[4 * q + 2] = x.z; S[4 * q + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) S[i] = 0.f;
    }
    publish16(stile, c, 0, S);
    publish16(stile, c, 2, S + 16);
    fence_async_shared();
    __syncwarp();
    if (lane == 0) mbar_arrive(s_ready);
    for (int n = 0; n < p.N; ++n) {
      const uint8_t* stg = sm + (n % NST) * STAGE;
      // r = U + D_r; rho = kscale r.
      ok = warp_wait(r_done, n & 1, ok);
      tc_fence_after();
      float gam;
      {
        float d[64];
        tmem_ld64(tmem + lb + T_R, d);
        // Lanes 0-15: hi row j (cols 0-31 W_hi S_hi, 32-63 W_hi S_lo); lanes
        // 16-31: lo row j. Lane t keeps columns [16 half, 16 half + 16).
        float r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float col_a = d[i] + d[32 + i];          // column i
          const float col_b = d[16 + i] + d[48 + i];     // column 16 + i
          const float send = half ? col_a : col_b;       // what the partner lane keeps
          const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
          r[i] = (half ? col_b : col_a) + recv;
        }
        const float* vec = reinterpret_cast<const float*>(stg + ST_VEC);
        const float ks = vec[C + j];
        gam = vec[2 * C + c];
        if (!p.zero_u) {
          const uint8_t* ub = stg + ST_U;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 u = *reinterpret_cast<const float4*>(ub + sw_off(j, 4 * half + q));
            r[4 * q] += u.x; r[4 * q + 1] += u.y; r[4 * q + 2] += u.z; r[4 * q + 3] += u.w;
          }
        }
        publish16(sm + R_TILE, j, 2 * half, r);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] *= ks;
        publish16(sm + P_TILE, j, 2 * half, r);
      }
      fence_async_shared();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(rho_ready);
      // S = gamma S + D_S.
      ok = warp_wait(ds_done, n & 1, ok);
      tc_fence_after();
      {
        float d[64];
        tmem_ld64(tmem + lb + T_S, d);
#pragma unroll
        for (int i = 0; i < 32; ++i) S[i] = fmaf(gam, S[i], d[i] + d[32 + i]);
      }
      tc_fence_before();
      if (n + 1 < p.N) {
        publish16(stile, c, 0, S);
        publish16(stile, c, 2, S + 16);
        fence_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_ready);
      }
    }
    if (p.sT) {
      float4* dst = reinterpret_cast<float4*>(p.sT + ((size_t)seq * K + c) * V + v0);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[q] = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
    }
  } else if (warp < 8) {
    // -------------------------------------------------------------- outputs
    const int qd = warp - 4;
    const uint32_t lb = (uint32_t)(32 * qd) << 16;
    const int half = lane >> 4;
    const int i = 16 * qd + (lane & 15);                 // chunk row
    for (int n = 0; n < p.N; ++n) {
      const int ob = n & 1, st = n % NST;
      ok = warp_wait(&o_full[ob], (n >> 1) & 1, ok);
      tc_fence_after();
      const float qs = reinterpret_cast<const float*>(sm + st * STAGE + ST_VEC)[i];
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);            // this warp is done with the stage
      float x[32];
      {
        float d[64];
        tmem_ld64(tmem + lb + T_O + 128 * ob, d);        // D_qs: lanes 0-15
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = half ? 0.f : qs * (d[e] + d[32 + e]);
        tmem_ld64(tmem + lb + T_O + 128 * ob + 64, d);   // D_ar: hi rows 0-15, lo rows 16-31
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] += d[e] + d[32 + e];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_empty[ob]);
      float o[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float send = half ? x[e] : x[16 + e];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
        o[e] = (half ? x[16 + e] : x[e]) + recv;
      }
      const int t = n * C + i;
      if (t < p.T) {
        const size_t off = (((size_t)b * p.T + t) * p.HV + hv) * V + v0 + 16 * half;
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
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t sb = smem_u32(sm);
      bool flags_ok = wait_flags;
      for (int n = 0; n < p.N; ++n) {
        const int st = n % NST, idx = chunk0 + n;
        if (n >= NST) ok = ok && mbar_wait(&empty[st], ((n / NST) - 1) & 1, kWaitLimit);
        if (!ok) break;
        if (flags_ok) {
          // The chunk's slab is written by a worker of this launch. A wait that
          // gives up records the error and stops waiting: the chain then runs
          // to its end on whatever the workspace holds (in bounds), so no
          // other wait of the launch has to run out as well.
          const unsigned int* fl = p.flags + idx;
          long polls = 0;
          while (ld_acquire_gpu(fl) == 0u) {
            if (++polls > p.wait_limit) {
              flags_ok = false;
              atomicOr(p.error_word, kErrFlagWait);
              break;
            }
            __nanosleep(64);
          }
          fence_async_global();                          // slab (generic acquire) -> TMA reads
        }
        const uint32_t stg = sb + st * STAGE;
        mbar_expect_tx(&full[st], STAGE_TX);
        tma_load3(stg + ST_W, &maps.w2, 0, 0, idx, &full[st]);
        tma_load3(stg + ST_W + 16384, &maps.w2, 64, 0, idx, &full[st]);
        tma_load4(stg + ST_K, &maps.k, 0, h, n * C, b, &full[st]);
        tma_load4(stg + ST_K + 8192, &maps.k, 64, h, n * C, b, &full[st]);
        tma_load4(stg + ST_Q, &maps.q, 0, h, n * C, b, &full[st]);
        tma_load4(stg + ST_Q + 8192, &maps.q, 64, h, n * C, b, &full[st]);
        tma_load3(stg + ST_AQ, &maps.aq2, 0, 0, idx, &full[st]);
        tma_load3(stg + ST_U, &maps.u, v0, 0, idx, &full[st]);
        bulk_load(stg + ST_VEC, p.slabs + (size_t)idx * p.slab_bytes + Slab::VEC, 1024, &full[st]);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_R = idesc_bf16(128, 64, 0, 1);    // A K-major, B MN-major
      constexpr uint32_t ID_QS = idesc_bf16(64, 64, 0, 1);
      constexpr uint32_t ID_S = idesc_bf16(128, 64, 1, 1);    // A = k^T read MN-major
      const uint32_t sb = smem_u32(sm);
      const uint32_t stile = sb + S_TILE, rtile = sb + R_TILE, ptile = sb + P_TILE;
      for (int n = 0; n < p.N; ++n) {
        const int st = n % NST, ob = n & 1;
        const uint32_t stg = sb + st * STAGE;
        const uint32_t d_qs = tmem + T_O + 128 * ob, d_ar = d_qs + 64;
        ok = ok && mbar_wait(&full[st], (n / NST) & 1, kWaitLimit);
        ok = ok && mbar_wait(s_ready, n & 1, kWaitLimit);
        tc_fence_after();
        if (ok) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_bf16(tmem + T_R, sdesc_sw128(stg + ST_W + (kk >> 2) * 16384 + (kk & 3) * 32),
                      sdesc_sw128_lbo(stile + kk * 2048, 8192), ID_R, kk > 0);
        }
        umma_commit(r_done);
        if (n >= 2) ok = ok && mbar_wait(&o_empty[ob], ((n >> 1) - 1) & 1, kWaitLimit);
        tc_fence_after();
        if (ok) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_bf16(d_qs, sdesc_sw128(stg + ST_Q + (kk >> 2) * 8192 + (kk & 3) * 32),
                      sdesc_sw128_lbo(stile + kk * 2048, 8192), ID_QS, kk > 0);
        }
        ok = ok && mbar_wait(rho_ready, n & 1, kWaitLimit);
        tc_fence_after();
        if (ok) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem + T_S, sdesc_sw128_lbo(stg + ST_K + kk * 2048, 8192),
                      sdesc_sw128_lbo(ptile + kk * 2048, 8192), ID_S, kk > 0);
        }
        umma_commit(ds_done);
        if (ok) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(d_ar, sdesc_sw128(stg + ST_AQ + kk * 32),
                      sdesc_sw128_lbo(rtile + kk * 2048, 8192), ID_R, kk > 0);
        }
        umma_commit(&o_full[ob]);
        umma_commit(&empty[st]);
      }
    }
    __syncwarp();
  }
  if (!ok) atomicOr(p.error_word, kErrChainWait);
  tc_fence_before();
  nb_sync(1, CHAIN_THREADS);
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

__global__ void __launch_bounds__(CHAIN_THREADS, 1)
    chain_kernel(const __grid_constant__ chunk::Maps maps, Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  chain_role(maps, p, sm, blockIdx.y * p.HV + blockIdx.x / VTILES, blockIdx.x % VTILES, false);
}

// =========================================================================== worker
// Two groups of 8 warps run the chunk-local stage over chunk items in chunk
// order (item it: chunk it / (B HV) of sequence it % (B HV)); group G of
// NG takes items G, G + NG, ...
__device__ __forceinline__ void worker_role(const chunk::Maps& maps, const Params& p,
                                            uint8_t* sm_base, int worker, int n_workers) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int grp = warp >> 3, gtid = tid & 255;
  uint8_t* sm = sm_base + grp * chunk::GROUP_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + chunk::OFF_BAR);
  // The CTA's TMEM allocation (both groups' 256 columns) is recorded in the
  // TMEM slot of group 0, which produce_chunk leaves alone when given its columns.
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm_base + chunk::OFF_BAR) + 4;
  if (gtid == 0) {
    mbar_init(bars, 1);       // tiles k, q
    mbar_init(bars + 1, 1);   // MMAs
    mbar_init(bars + 3, 1);   // tiles v
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(tslot, 2 * chunk::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot + grp * chunk::TMEM_COLS;
  const int nseq = p.B * p.HV;
  const long items = (long)nseq * p.N;
  const int G = 2 * worker + grp, NG = 2 * n_workers;
  unsigned int* pending = nullptr;
  uint32_t ph = 0;
  for (long it = G; it < items; it += NG) {
    const int n = (int)(it / nseq), seq = (int)(it % nseq);
    const int b = seq / p.HV, hv = seq % p.HV;
    chunk::produce_chunk(maps, p, sm, gtid, 1 + grp, n, hv, b, ph, tmem, nullptr, pending);
    pending = p.flags + slab_index(p, b, hv, n);
    ph ^= 1u;
  }
  if (gtid == 0 && pending) {
    bulk_wait<0>();
    fence_async_global();
    st_release_gpu(pending, 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(*tslot, 2 * chunk::TMEM_COLS);
  }
}

__global__ void __launch_bounds__(FUSED_THREADS, 1)
    fused_kernel(const __grid_constant__ chunk::Maps maps, Params p, int n_chain, int n_workers) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int cta = blockIdx.x;
  if (cta < n_chain) {
    if (threadIdx.x < CHAIN_THREADS) chain_role(maps, p, sm, cta / VTILES, cta % VTILES, true);
  } else {
    worker_role(maps, p, sm, cta - n_chain, n_workers);
  }
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

// Maps of the chain role: q, k inputs and the slab arrays (v is not read).
bool chain_maps(chunk::Maps* m, const Params& p) {
  memset(m, 0, sizeof *m);
  const size_t nch = (size_t)p.B * p.HV * p.N;
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
  return tmap_bthd(&m->q, p.q, p.B, p.T, p.H) && tmap_bthd(&m->k, p.k, p.B, p.T, p.H) &&
         tmap_blocks(&m->aq2, p.slabs + Slab::AQ2, BF, 2, C, 2 * C, nch, p.slab_bytes, 64, 128, SW) &&
         tmap_blocks(&m->w2, p.slabs + Slab::W2, BF, 2, K, 2 * C, nch, p.slab_bytes, 64, 128, SW) &&
         tmap_blocks(&m->u, p.slabs + Slab::U, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, V, C, nch,
                     p.slab_bytes, 32, 64, SW);
}

}  // namespace

gdr_status launch_chain(const Params& p, cudaStream_t stream) {
  if (p.gate_mode != 0) return GDR_ERR_UNSUPPORTED;
  chunk::Maps m;
  if (!chain_maps(&m, p)) return GDR_ERR_CUDA;
  if (cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           CHAIN_SMEM) != cudaSuccess)
    return GDR_ERR_CUDA;
  dim3 grid(p.HV * VTILES, p.B);
  chain_kernel<<<grid, CHAIN_THREADS, CHAIN_SMEM, stream>>>(m, p);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

bool fused_fits(int B, int HV) {
  const DeviceInfo dev = device_info();
  const long long n_chain = (long long)B * HV * VTILES;
  // The workers must produce chunks about as fast as the chains consume them:
  // at least as many worker CTAs as chain CTAs.
  return dev.coop && n_chain * 2 <= dev.sms;
}

gdr_status launch_fused(const Params& p, cudaStream_t stream) {
  if (p.gate_mode != 0 || !p.flags || !fused_fits(p.B, p.HV)) return GDR_ERR_UNSUPPORTED;
  const DeviceInfo dev = device_info();
  const long long n_chain = (long long)p.B * p.HV * VTILES;
  const int n_workers = dev.sms - (int)n_chain;
  chunk::Maps m;
  if (!chunk::make_maps(&m, p)) return GDR_ERR_CUDA;
  if (cudaFuncSetAttribute(fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           FUSED_SMEM) != cudaSuccess)
    return GDR_ERR_CUDA;
  const size_t nch = (size_t)p.B * p.HV * p.N;
  if (cudaMemsetAsync(p.flags, 0, nch * sizeof(unsigned int), stream) != cudaSuccess)
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
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fused_kernel, m, p, (int)n_chain, n_workers);
  if (e == cudaSuccess) return GDR_OK;
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    (void)cudaGetLastError();
    return GDR_ERR_UNSUPPORTED;
  }
  return GDR_ERR_CUDA;
}

}  // namespace fast
}  // namespace gdr
