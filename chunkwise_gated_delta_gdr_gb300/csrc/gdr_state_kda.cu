// gdr_state_kda.cu -- inter-chunk recurrence for the per-key gate on tcgen05.
//
// One CTA per (b, hv, 64 value columns v0 .. v0 + 63), serial over the chunks.
// Per chunk n it applies the inter-chunk loop of the "分块并行计算（Chunkwise）"
// notes (section "chunk 间递推"; gate per key channel, listing naive_chunk_kda):
//     r  = U + (-W) S                       [64 j x 64 v]
//     dS = KB^T r,   S <- gamma S + dS      [128 c x 64 v]
//     o  = QB S + A_qk r                    [64 i x 64 v]
// with KB = beta k^ exp(G_last - G), QB = q~ exp(G), gamma = exp(G_last) per
// channel (the chunk slab of gdr_fast.cuh). Every product runs on tcgen05
// (kind::f16, bf16 operands, fp32 accumulators in TMEM) with both operands
// split into bf16 hi + lo. The B operand is stacked along N as [B_hi | B_lo]
// (N = 128): per K step A_hi [B_hi | B_lo] (N = 128) and A_lo B_hi (N = 64,
// into the first half), i.e. the three terms hi hi + hi lo + lo hi; the two
// column halves of the accumulator are added in the epilogue.
//
// Roles (10 warps):
//   warps 0-7  the state: warps w and w + 4 share TMEM lane quadrant w % 4 and
//              take value columns [32 (w / 4), 32 (w / 4) + 32); thread (c, half)
//              holds those 32 columns of row c of S in fp32 registers for the
//              whole sequence. Per chunk they publish S as the hi / lo B operand
//              (MN-major, 128-byte swizzled rows), store the previous chunk's o
//              while the r products run, form r = U + D_r from TMEM and publish
//              it likewise (lanes 0-15, rows j), then apply S = gamma S + dS.
//   warp 8     TMA producer. Each operand has its own buffer and is reloaded as
//              soon as its last reader is done: W (two buffers) after the r
//              products, QB after QB S, U and gamma (two buffers) after the r
//              epilogue, KB after the dS products, A_qk after A_qk r. (An L2
//              prefetch of later chunks' slabs measured slower.)
//   warp 9     MMA issuer and TMEM owner, in the order r, QB S, dS, A_qk r: the
//              output products run on the tensor pipe while the state warps
//              work on r and on S, never in front of r or dS.
// The state and MMA warps meet on two named barriers per chunk (S published,
// r published), both sides bar.sync. Every mbarrier wait is bounded; on expiry
// the error word is set and the loops run to their end without products, so
// the CTA always terminates.
#include <cuda.h>
#include <cuda_bf16.h>

#include "gdr_fast.cuh"
#include "gdr_ptx.cuh"

namespace gdr {
namespace fast {
namespace {

using namespace ptx;

constexpr int VC = 64;                  // value columns per CTA
constexpr int THREADS = 320;
constexpr int SYNC_N = 288;             // state warps + MMA warp on the named barriers
constexpr long kWaitLimit = 1L << 24;
constexpr unsigned int kErrWait = 16u;

// Shared memory (bytes from a 1024-aligned base). bf16 [64][128] operands are
// two 8 KB boxes (columns 0-63, 64-127) per hi / lo plane.
constexpr int W_BASE = 0;                 // -W hi, lo          32 KB, x 2
constexpr int KB_BASE = 65536;            // KB hi, lo          32 KB
constexpr int QB_BASE = 98304;            // QB hi, lo          32 KB
constexpr int AQ_BASE = 131072;           // A_qk hi, lo        16 KB
constexpr int U_BASE = 147456;            // U [64 j][64 v] fp32 as two swizzled [64][32] boxes, x 2
constexpr int S_BASE = 180224;            // S hi | lo [128 c][64 v] bf16 (16 KB each)
constexpr int R_BASE = 212992;            // r hi | lo [64 j][64 v] bf16 (8 KB each)
constexpr int GAM_BASE = 229376;          // gamma [128] fp32, x 2
constexpr int BAR_BASE = 230400;
constexpr int SMEM_BYTES = BAR_BASE + 256 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
constexpr uint32_t kUBytes = 16384 + 512;

// TMEM columns (128 each: the B_hi and B_lo halves): D_r as two accumulators
// (even and odd K steps, two independent MMA chains), dS, o.
constexpr uint32_t T_R = 0, T_R2 = 128, T_DS = 256, T_O = 384, TMEM_COLS = 512;

__device__ __forceinline__ void nb_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Byte offset of 16-byte chunk q of row r in 128-byte swizzled rows.
__device__ __forceinline__ uint32_t sw_off(int r, int q) {
  return (uint32_t)(r * 128 + ((q ^ (r & 7)) << 4));
}

// 8 Q fp32 values -> 16-byte chunks q0 .. q0 + Q - 1 of row r of the hi and lo
// bf16 planes (MN-major operand, swizzled rows of 64 values).
template <int Q>
__device__ __forceinline__ void publish(uint8_t* hi, uint8_t* lo, int r, int q0, const float* x) {
#pragma unroll
  for (int qq = 0; qq < Q; ++qq) {
    const int q = q0 + qq;
    uint32_t h[4], l[4];
#pragma unroll
    for (int z = 0; z < 4; ++z) split_pair(x[8 * qq + 2 * z], x[8 * qq + 2 * z + 1], h[z], l[z]);
    *reinterpret_cast<uint4*>(hi + sw_off(r, q)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo + sw_off(r, q)) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}
__global__ void __launch_bounds__(THREADS, 1) state_kda_tc_kernel(Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int vt = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
  const int v0 = vt * VC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t seq = (size_t)b * p.HV + hv;
  const int chunk0 = (int)(seq * p.N);

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + BAR_BASE);
  uint64_t* w_full = bars + 0;      // [2]
  uint64_t* w_empty = bars + 2;     // [2], commit after the r products
  uint64_t* u_full = bars + 4;      // [2]
  uint64_t* u_empty = bars + 6;     // [2], 8 arrivals (state warps)
  uint64_t* kb_full = bars + 8;
  uint64_t* kb_empty = bars + 9;    // commit after the dS products
  uint64_t* qb_full = bars + 10;
  uint64_t* qb_empty = bars + 11;   // commit after QB S
  uint64_t* aq_full = bars + 12;
  uint64_t* aq_empty = bars + 13;   // commit after A_qk r
  uint64_t* r_done = bars + 14;
  uint64_t* ds_done = bars + 15;
  uint64_t* o_full = bars + 16;
  uint64_t* o_empty = bars + 17;    // 8 arrivals (state warps)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 20);

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&w_full[i], 1);
      mbar_init(&w_empty[i], 1);
      mbar_init(&u_full[i], 1);
      mbar_init(&u_empty[i], 8);
    }
    mbar_init(kb_full, 1);
    mbar_init(kb_empty, 1);
    mbar_init(qb_full, 1);
    mbar_init(qb_empty, 1);
    mbar_init(aq_full, 1);
    mbar_init(aq_empty, 1);
    mbar_init(o_full, 1);
    mbar_init(o_empty, 8);
    mbar_init(r_done, 1);
    mbar_init(ds_done, 1);
    mbar_fence_init();
  }
  if (warp == 9) tmem_alloc(tslot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  bool ok = true;

  if (warp < 8) {
    // ---------------------------------------------------------------- state
    const int quad = warp & 3, hf = warp >> 2;          // lane quadrant, column half
    const int c = 32 * quad + lane;                      // key channel = TMEM lane
    const int j = 16 * quad + (lane & 15);               // D_r / o row held by lanes 0-15
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const int vc = v0 + 32 * hf;                         // first value column of this thread
    float S[32];
    if (p.s0) {
      const float4* src = reinterpret_cast<const float4*>(p.s0 + (seq * K + c) * V + vc);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 x = src[q];
        S[4 * q] = x.x; S[4 * q + 1] = x.y; S[4 * q + 2] = x.z; S[4 * q + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) S[i] = 0.f;
    }
    // o of chunk m: 32 columns of row j, lanes 0-15.
    auto store_o = [&](int m) {
      ok = ok && mbar_wait(o_full, m & 1, kWaitLimit);
      tc_fence_after();
      float o[32], ol[32];
      tmem_ld32(tmem + lane_base + T_O + 32 * hf, o);
      tmem_ld32(tmem + lane_base + T_O + 64 + 32 * hf, ol);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty);
      const int t = m * C + j;
      if (lane < 16 && t < p.T) {
        const size_t off = (((size_t)b * p.T + t) * p.HV + hv) * V + vc;
        if (p.out_bf16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + off);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[q] = make_uint4(pack_bf16(o[8 * q] + ol[8 * q], o[8 * q + 1] + ol[8 * q + 1]),
                                pack_bf16(o[8 * q + 2] + ol[8 * q + 2], o[8 * q + 3] + ol[8 * q + 3]),
                                pack_bf16(o[8 * q + 4] + ol[8 * q + 4], o[8 * q + 5] + ol[8 * q + 5]),
                                pack_bf16(o[8 * q + 6] + ol[8 * q + 6], o[8 * q + 7] + ol[8 * q + 7]));
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + off);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(o[4 * q] + ol[4 * q], o[4 * q + 1] + ol[4 * q + 1],
                                 o[4 * q + 2] + ol[4 * q + 2], o[4 * q + 3] + ol[4 * q + 3]);
        }
      }
    };
    for (int n = 0; n < p.N; ++n) {
      const int s = n & 1;
      // S_n -> B operand of the r and QB S products (their previous readers
      // are done: both precede the last dS products in the MMA order).
      publish<4>(sm + S_BASE, sm + S_BASE + 16384, c, 4 * hf, S);
      fence_async_shared();
      nb_sync(1, SYNC_N);
      if (n > 0) store_o(n - 1);                          // overlaps the r products
      // r = U + D_r: lanes 0-15 of each warp hold rows j = 16 quad + lane.
      ok = ok && mbar_wait(&u_full[s], (n >> 1) & 1, kWaitLimit);
      ok = ok && mbar_wait(r_done, n & 1, kWaitLimit);
      tc_fence_after();
      const float gam = reinterpret_cast<const float*>(sm + GAM_BASE + s * 512)[c];
      {
        float r[32], rl[32];
        tmem_ld32(tmem + lane_base + T_R + 32 * hf, r);
        tmem_ld32(tmem + lane_base + T_R + 64 + 32 * hf, rl);
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] += rl[i];
        tmem_ld32(tmem + lane_base + T_R2 + 32 * hf, rl);
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] += rl[i];
        tmem_ld32(tmem + lane_base + T_R2 + 64 + 32 * hf, rl);
        if (lane < 16) {
          const uint8_t* ub = sm + U_BASE + s * 16384 + hf * 8192;
          const float uf = p.zero_u ? 0.f : 1.f;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 u = *reinterpret_cast<const float4*>(ub + sw_off(j, q));
            r[4 * q] += rl[4 * q] + uf * u.x;
            r[4 * q + 1] += rl[4 * q + 1] + uf * u.y;
            r[4 * q + 2] += rl[4 * q + 2] + uf * u.z;
            r[4 * q + 3] += rl[4 * q + 3] + uf * u.w;
          }
          publish<4>(sm + R_BASE, sm + R_BASE + 8192, j, 4 * hf, r);
        }
      }
      fence_async_shared();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&u_empty[s]);          // U and gamma of buffer s read
      nb_sync(2, SYNC_N);
      // S_{n+1} = gamma S_n + dS.
      ok = ok && mbar_wait(ds_done, n & 1, kWaitLimit);
      tc_fence_after();
      {
        float d[32], dl[32];
        tmem_ld32(tmem + lane_base + T_DS + 32 * hf, d);
        tmem_ld32(tmem + lane_base + T_DS + 64 + 32 * hf, dl);
#pragma unroll
        for (int i = 0; i < 32; ++i) S[i] = fmaf(gam, S[i], d[i] + dl[i]);
      }
      tc_fence_before();
    }
    if (p.N > 0) store_o(p.N - 1);
    if (p.sT) {
      float4* dst = reinterpret_cast<float4*>(p.sT + (seq * K + c) * V + vc);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[q] = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t sb = smem_u32(sm);
      auto slab = [&](int n) { return p.slabs + (size_t)(chunk0 + n) * p.slab_bytes; };
      // One bulk copy per array: the chunk-local stage stores each as the
      // byte image of the 128-byte swizzled boxes it takes here.
      auto issue_w = [&](int n) {
        const int s = n & 1;
        mbar_expect_tx(&w_full[s], 32768);
        bulk_load(sb + W_BASE + s * 32768, slab(n) + Slab::W2, 32768, &w_full[s]);
      };
      auto issue_u = [&](int n) {
        const int s = n & 1;
        mbar_expect_tx(&u_full[s], kUBytes);
        bulk_load(sb + U_BASE + s * 16384, slab(n) + Slab::U + (size_t)vt * 16384, 16384, &u_full[s]);
        bulk_load(sb + GAM_BASE + s * 512, slab(n) + Slab::VEC + 2 * C * sizeof(float), 512,
                  &u_full[s]);
      };
      auto issue_kb = [&](int n) {
        mbar_expect_tx(kb_full, 32768);
        bulk_load(sb + KB_BASE, slab(n) + Slab::KB2, 32768, kb_full);
      };
      auto issue_qb = [&](int n) {
        mbar_expect_tx(qb_full, 32768);
        bulk_load(sb + QB_BASE, slab(n) + Slab::QB2, 32768, qb_full);
      };
      auto issue_aq = [&](int n) {
        mbar_expect_tx(aq_full, 16384);
        bulk_load(sb + AQ_BASE, slab(n) + Slab::AQ2, 16384, aq_full);
      };
      issue_w(0);
      issue_qb(0);
      issue_u(0);
      issue_kb(0);
      issue_aq(0);
      if (p.N > 1) {
        issue_w(1);
        issue_u(1);
      }
      // Operands of chunk n + 1 (n + 2 for the two-buffer ones), in the order
      // chunk n frees their buffers.
      for (int n = 0; n + 1 < p.N && ok; ++n) {
        if (n + 2 < p.N) {
          ok = ok && mbar_wait(&w_empty[n & 1], (n >> 1) & 1, kWaitLimit);
          if (!ok) break;
          issue_w(n + 2);
        }
        ok = ok && mbar_wait(qb_empty, n & 1, kWaitLimit);
        if (!ok) break;
        issue_qb(n + 1);
        if (n + 2 < p.N) {
          ok = ok && mbar_wait(&u_empty[n & 1], (n >> 1) & 1, kWaitLimit);
          if (!ok) break;
          issue_u(n + 2);
        }
        ok = ok && mbar_wait(kb_empty, n & 1, kWaitLimit);
        if (!ok) break;
        issue_kb(n + 1);
        ok = ok && mbar_wait(aq_empty, n & 1, kWaitLimit);
        if (!ok) break;
        issue_aq(n + 1);
      }
    }
  } else {
    // ------------------------------------------------------------- MMA issuer
    constexpr uint32_t ID_KMN = idesc_bf16(64, 128, 0, 1);    // A K-major, B MN-major [hi | lo]
    constexpr uint32_t ID_KMN_H = idesc_bf16(64, 64, 0, 1);   // same, B hi only
    constexpr uint32_t ID_MNMN = idesc_bf16(128, 128, 1, 1);  // both MN-major
    constexpr uint32_t ID_MNMN_H = idesc_bf16(128, 64, 1, 1);
    const uint32_t sb = smem_u32(sm), rb = smem_u32(sm + R_BASE), sbuf = smem_u32(sm + S_BASE);
    for (int n = 0; n < p.N; ++n) {
      const uint32_t d_o = tmem + T_O;
      const uint32_t wb = sb + W_BASE + (n & 1) * 32768;
      nb_sync(1, SYNC_N);                                          // S_n published
      ok = ok && mbar_wait(&w_full[n & 1], (n >> 1) & 1, kWaitLimit);
      tc_fence_after();
      if (lane == 0) {
        if (ok) {
          // D_r = (-W) [S_hi | S_lo]: A = -W hi, lo (K-major), B MN-major (N = 128).
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ao = (kk >> 2) * 8192 + (kk & 3) * 32;
            const uint64_t bd = sdesc_sw128_lbo(sbuf + kk * 2048, 16384);
            const uint32_t dr = tmem + ((kk & 1) ? T_R2 : T_R);
            umma_bf16(dr, sdesc_sw128(wb + ao), bd, ID_KMN, kk > 1);
            umma_bf16(dr, sdesc_sw128(wb + 16384 + ao), bd, ID_KMN_H, 1);
          }
        }
        umma_commit(r_done);
        umma_commit(&w_empty[n & 1]);
      }
      __syncwarp();
      ok = ok && mbar_wait(qb_full, n & 1, kWaitLimit);
      if (n >= 1) ok = ok && mbar_wait(o_empty, (n - 1) & 1, kWaitLimit);
      tc_fence_after();
      if (lane == 0) {
        if (ok) {
          // o = QB [S_hi | S_lo] (runs during the r epilogue).
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ao = (kk >> 2) * 8192 + (kk & 3) * 32;
            const uint64_t bd = sdesc_sw128_lbo(sbuf + kk * 2048, 16384);
            umma_bf16(d_o, sdesc_sw128(sb + QB_BASE + ao), bd, ID_KMN, kk > 0);
            umma_bf16(d_o, sdesc_sw128(sb + QB_BASE + 16384 + ao), bd, ID_KMN_H, 1);
          }
        }
        umma_commit(qb_empty);
      }
      __syncwarp();
      nb_sync(2, SYNC_N);                                          // r published
      ok = ok && mbar_wait(kb_full, n & 1, kWaitLimit);
      tc_fence_after();
      if (lane == 0) {
        if (ok) {
          // dS = KB^T [r_hi | r_lo]: A = KB hi, lo read MN-major (M = c).
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = sdesc_sw128_lbo(rb + kk * 2048, 8192);
            umma_bf16(tmem + T_DS, sdesc_sw128_lbo(sb + KB_BASE + kk * 2048, 8192), bd, ID_MNMN, kk > 0);
            umma_bf16(tmem + T_DS, sdesc_sw128_lbo(sb + KB_BASE + 16384 + kk * 2048, 8192), bd, ID_MNMN_H, 1);
          }
        }
        umma_commit(ds_done);
        umma_commit(kb_empty);
      }
      __syncwarp();
      ok = ok && mbar_wait(aq_full, n & 1, kWaitLimit);
      tc_fence_after();
      if (lane == 0) {
        if (ok) {
          // o += A_qk [r_hi | r_lo] (runs while the state warps update S).
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = sdesc_sw128_lbo(rb + kk * 2048, 8192);
            umma_bf16(d_o, sdesc_sw128(sb + AQ_BASE + kk * 32), bd, ID_KMN, 1);
            umma_bf16(d_o, sdesc_sw128(sb + AQ_BASE + 8192 + kk * 32), bd, ID_KMN_H, 1);
          }
        }
        umma_commit(o_full);
        umma_commit(aq_empty);
      }
      __syncwarp();
    }
  }
  if (!ok) atomicOr(p.error_word, kErrWait);
  tc_fence_before();
  __syncthreads();
  if (warp == 9) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

gdr_status launch_state_kda_tc(const Params& p, cudaStream_t stream) {
  static_assert(Slab::W2 % 16 == 0 && Slab::U % 16 == 0 && Slab::QB2 % 16 == 0 &&
                    Slab::KB2 % 16 == 0 && Slab::AQ2 % 16 == 0,
                "bulk copies from the slab need 16-byte alignment");
  if (p.slab_bytes % 16 != 0) return GDR_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(state_kda_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SMEM_BYTES) != cudaSuccess)
    return GDR_ERR_CUDA;
  dim3 grid(V / VC, p.HV, p.B);
  state_kda_tc_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

}  // namespace fast
}  // namespace gdr
