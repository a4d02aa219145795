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
//     r^T  = U^T - S^T W^T                 (16 x 64,  K = 128)
//     o^T  = diag-scaled S^T q^T + r^T A_qk^T   (16 x 64)
//     S^T <- gamma S^T + (kscale r)^T k    (16 x 128, K = 64)
// The state S^T stays in fp32 registers for the whole sequence (each warp owns
// 16 of its 128 key channels). Products run on the tensor cores with
// mma.sync m16n8k16 (bf16 in, fp32 accumulate); an fp32-valued operand x is
// fed as x_hi + x_lo with x_hi = bf16(x), x_lo = bf16(x - x_hi), and the
// lo * lo term is dropped, which keeps about 16 significant bits per product.
// Every split term accumulates into its own register tile, so no chain of
// dependent mma.sync is longer than one product's k-steps; two warps per SM
// sub-partition hide the remaining latency.
// The only exchanges are two shared-memory tiles per chunk (S^T and r^T) and
// two CTA barriers. Chunk operands are staged in shared memory with cp.async,
// one chunk ahead.
#include <cuda_bf16.h>

#include "gdr_fast.cuh"

namespace gdr {
namespace fast {
namespace {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int LDW = K + 8;  // bf16 row stride of [*, 128] tiles (272 B: ldmatrix conflict-free)
constexpr int LDA = C + 8;  // bf16 row stride of [*, 64] tiles (144 B)

// Shared-memory plan (bytes). "Big" operand tiles are staged STAGES times.
struct Smem {
  static constexpr int TILE_W = C * LDW * 2;      // one [64][136] bf16 tile
  static constexpr int TILE_A = C * LDA * 2;      // one [64][72] bf16 tile
  // Per stage: W hi, W lo, Q (hi[, lo]), K (hi[, lo]), AQ hi, AQ lo.
  __host__ __device__ static constexpr int stage_bytes(int gate) { return TILE_W * (2 + (gate ? 4 : 2)) + 2 * TILE_A; }
  // Small double-buffered part: U tile [64][16] fp32 and VEC.
  static constexpr int SMALL = C * VT * 4 + (2 * C + K) * 4;
  // Exchange tiles: S^T hi/lo [16][136]; r^T, rho^T hi/lo [16][72]; o staging 8 x [8][16] fp32.
  static constexpr int XS = 2 * VT * LDW * 2;
  static constexpr int XR = 4 * VT * LDA * 2;
  static constexpr int XO = WARPS * 8 * 16 * 4;
  __host__ __device__ static constexpr int total(int gate, int stages) {
    return stages * stage_bytes(gate) + 2 * SMALL + XS + XR + XO;
  }
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// D += A (16x16, row) * B (16x8, col), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// bf16 pair (lo half = x) and the hi/lo split of an fp32 pair.
__device__ __forceinline__ uint32_t pack_bf16(float x, float y) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ void split_pair(float x, float y, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  float2 hf = __bfloat1622float2(h);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = pack_bf16(x - hf.x, y - hf.y);
}

// Stage pointers inside the dynamic shared memory block.
template <int GATE>
struct Stage {
  __nv_bfloat16 *w_hi, *w_lo, *q_hi, *q_lo, *k_hi, *k_lo, *aq_hi, *aq_lo;
  __device__ Stage(uint8_t* base) {
    uint8_t* p = base;
    w_hi = reinterpret_cast<__nv_bfloat16*>(p); p += Smem::TILE_W;
    w_lo = reinterpret_cast<__nv_bfloat16*>(p); p += Smem::TILE_W;
    q_hi = reinterpret_cast<__nv_bfloat16*>(p); p += Smem::TILE_W;
    if (GATE) { q_lo = reinterpret_cast<__nv_bfloat16*>(p); p += Smem::TILE_W; } else { q_lo = nullptr; }
    k_hi = reinterpret_cast<__nv_bfloat16*>(p); p += Smem::TILE_W;
    if (GATE) { k_lo = reinterpret_cast<__nv_bfloat16*>(p); p += Smem::TILE_W; } else { k_lo = nullptr; }
    aq_hi = reinterpret_cast<__nv_bfloat16*>(p); p += Smem::TILE_A;
    aq_lo = reinterpret_cast<__nv_bfloat16*>(p);
  }
};

struct Small {
  float* u;      // [64][16]
  float* qs;     // [64]
  float* ks;     // [64]
  float* gam;    // [128]
  __device__ Small(uint8_t* base) {
    u = reinterpret_cast<float*>(base);
    qs = u + C * VT;
    ks = qs + C;
    gam = ks + C;
  }
};

// Copy a [64][128] bf16 tile whose rows are `row_stride` elements apart into a
// [64][LDW] shared tile; rows >= valid_rows are zero-filled.
__device__ __forceinline__ void load_tile128(__nv_bfloat16* dst, const __nv_bfloat16* src,
                                             size_t row_stride, int valid_rows, int tid) {
  for (int idx = tid; idx < C * (K / 8); idx += THREADS) {
    const int r = idx >> 4, c8 = (idx & 15) * 8;
    const bool ok = r < valid_rows;
    const __nv_bfloat16* s = src + (ok ? (size_t)r * row_stride + c8 : 0);
    cp_async16(smem_u32(dst + r * LDW + c8), s, ok);
  }
}
__device__ __forceinline__ void load_tile64(__nv_bfloat16* dst, const __nv_bfloat16* src, int tid) {
  for (int idx = tid; idx < C * (C / 8); idx += THREADS) {
    const int r = idx >> 3, c8 = (idx & 7) * 8;
    cp_async16(smem_u32(dst + r * LDA + c8), src + r * C + c8, true);
  }
}

// Operands of chunk n from its slab (and, for the scalar gate, raw q / k).
template <int GATE>
__device__ __forceinline__ void load_big(const Params& p, const Stage<GATE>& st, const uint8_t* slab,
                                         int b, int h, int n, int tid) {
  const __nv_bfloat16* w2 = reinterpret_cast<const __nv_bfloat16*>(slab + Slab::W2);
  load_tile128(st.w_hi, w2, K, C, tid);
  load_tile128(st.w_lo, w2 + C * K, K, C, tid);
  if (GATE) {
    const __nv_bfloat16* q2 = reinterpret_cast<const __nv_bfloat16*>(slab + Slab::QB2);
    const __nv_bfloat16* k2 = reinterpret_cast<const __nv_bfloat16*>(slab + Slab::KB2);
    load_tile128(st.q_hi, q2, K, C, tid);
    load_tile128(st.q_lo, q2 + C * K, K, C, tid);
    load_tile128(st.k_hi, k2, K, C, tid);
    load_tile128(st.k_lo, k2 + C * K, K, C, tid);
  } else {
    const int t0 = n * C;
    const int valid = min(C, p.T - t0);
    const size_t rs = (size_t)p.H * K;
    const size_t off = (((size_t)b * p.T + t0) * p.H + h) * K;
    load_tile128(st.q_hi, p.q + off, rs, valid, tid);
    load_tile128(st.k_hi, p.k + off, rs, valid, tid);
  }
  const __nv_bfloat16* aq = reinterpret_cast<const __nv_bfloat16*>(slab + Slab::AQ2);
  load_tile64(st.aq_hi, aq, tid);
  load_tile64(st.aq_lo, aq + C * C, tid);
}

__device__ __forceinline__ void load_small(const Small& sm, const uint8_t* slab, int v0, int tid) {
  const float* u = reinterpret_cast<const float*>(slab + Slab::U);
  for (int idx = tid; idx < C * (VT / 4); idx += THREADS) {
    const int r = idx / (VT / 4), c4 = (idx % (VT / 4)) * 4;
    cp_async16(smem_u32(sm.u + r * VT + c4), u + r * V + v0 + c4, true);
  }
  const float* vec = reinterpret_cast<const float*>(slab + Slab::VEC);
  for (int idx = tid; idx < (2 * C + K) / 4; idx += THREADS)
    cp_async16(smem_u32(sm.qs + idx * 4), vec + idx * 4, true);
}

// Single-stage protocol (per-key gate): group 1 = W, Q and the small part,
// group 2 = K and A_qk.
__device__ __forceinline__ void load_group1(const Stage<1>& st, const Small& sm, const uint8_t* slab,
                                            int v0, int tid) {
  const __nv_bfloat16* w2 = reinterpret_cast<const __nv_bfloat16*>(slab + Slab::W2);
  load_tile128(st.w_hi, w2, K, C, tid);
  load_tile128(st.w_lo, w2 + C * K, K, C, tid);
  const __nv_bfloat16* q2 = reinterpret_cast<const __nv_bfloat16*>(slab + Slab::QB2);
  load_tile128(st.q_hi, q2, K, C, tid);
  load_tile128(st.q_lo, q2 + C * K, K, C, tid);
  load_small(sm, slab, v0, tid);
  cp_commit();
}
__device__ __forceinline__ void load_group2(const Stage<1>& st, const uint8_t* slab, int tid) {
  const __nv_bfloat16* k2 = reinterpret_cast<const __nv_bfloat16*>(slab + Slab::KB2);
  load_tile128(st.k_hi, k2, K, C, tid);
  load_tile128(st.k_lo, k2 + C * K, K, C, tid);
  const __nv_bfloat16* aq = reinterpret_cast<const __nv_bfloat16*>(slab + Slab::AQ2);
  load_tile64(st.aq_hi, aq, tid);
  load_tile64(st.aq_lo, aq + C * C, tid);
  cp_commit();
}

template <int GATE, int STAGES>
__global__ void __launch_bounds__(THREADS) state_kernel(Params p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int vt = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
  const int h = hv / (p.HV / p.H);
  const int v0 = vt * VT;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;

  uint8_t* sp = smem;
  uint8_t* const stage0 = sp;
  sp += STAGES * Smem::stage_bytes(GATE);
  uint8_t* const small0 = sp;
  sp += 2 * Smem::SMALL;
  auto stage_at = [&](int n) { return stage0 + (STAGES == 2 ? (n & 1) : 0) * Smem::stage_bytes(GATE); };
  auto small_at = [&](int n) { return small0 + (n & 1) * Smem::SMALL; };
  __nv_bfloat16* xs_hi = reinterpret_cast<__nv_bfloat16*>(sp);
  __nv_bfloat16* xs_lo = xs_hi + VT * LDW;
  sp += Smem::XS;
  __nv_bfloat16* xr_hi = reinterpret_cast<__nv_bfloat16*>(sp);
  __nv_bfloat16* xr_lo = xr_hi + VT * LDA;
  __nv_bfloat16* xp_hi = xr_lo + VT * LDA;
  __nv_bfloat16* xp_lo = xp_hi + VT * LDA;
  sp += Smem::XR;
  float* xo = reinterpret_cast<float*>(sp) + warp * 128;

  const size_t seq = (size_t)b * p.HV + hv;
  const uint8_t* slabs = p.slabs + seq * p.N * p.slab_bytes;

  // Warp roles per chunk: r^T and o^T columns j, i in [8 warp, 8 warp + 8);
  // S^T key channels c in [16 warp, 16 warp + 16) (two n-tiles of 8).
  const int jw = 8 * warp, cw = 16 * warp;

  // State S^T[v][c] (fp32) of this warp's channels.
  float S[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int c = cw + 8 * nt + 2 * t4;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int vv = g + (e >> 1) * 8, cc = c + (e & 1);
      S[nt][e] = p.s0 ? p.s0[(seq * K + cc) * V + v0 + vv] : 0.f;
    }
  }

  // Prologue: the operands of chunk 0, in the groups the loop expects.
  if constexpr (STAGES == 2) {
    Stage<GATE> st0(stage_at(0));
    load_big<GATE>(p, st0, slabs, b, h, 0, tid);
    load_small(Small(small_at(0)), slabs, v0, tid);
    cp_commit();
  } else {
    Stage<1> st0(stage_at(0));
    load_group1(st0, Small(small_at(0)), slabs, v0, tid);
    load_group2(st0, slabs, tid);
  }

  // ldmatrix lane addressing.
  const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;   // A fragments (16 rows)
  const int acol = (lane >> 4) * 8;
  const int brow = (lane & 7);                           // B from [n][k] tiles, 2 k-steps per x4
  const int bcol = (lane >> 3) * 8;
  const int krow = (lane & 7) + ((lane >> 3) & 1) * 8;   // B from the [j][c] k tile (.trans)
  const int kcol = cw + (lane >> 4) * 8;

  for (int n = 0; n < p.N; ++n) {
    const uint8_t* slab = slabs + (size_t)n * p.slab_bytes;
    Stage<GATE> st(stage_at(n));
    Small sm(small_at(n));
    const int t0 = n * C;

    // ---- A: publish this warp's S^T slice as bf16 hi/lo -------------------------
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int c = cw + 8 * nt + 2 * t4;
      uint32_t hi, lo;
      split_pair(S[nt][0], S[nt][1], hi, lo);
      *reinterpret_cast<uint32_t*>(xs_hi + g * LDW + c) = hi;
      *reinterpret_cast<uint32_t*>(xs_lo + g * LDW + c) = lo;
      split_pair(S[nt][2], S[nt][3], hi, lo);
      *reinterpret_cast<uint32_t*>(xs_hi + (g + 8) * LDW + c) = hi;
      *reinterpret_cast<uint32_t*>(xs_lo + (g + 8) * LDW + c) = lo;
    }
    if constexpr (STAGES == 2) {
      cp_wait<0>();           // chunk n operands landed (this thread's copies)
    } else {
      cp_wait<1>();           // group 1 (W, Q, small part) of chunk n landed
    }
    __syncthreads();          // #1: S^T tiles and chunk-n operands visible to all

    if constexpr (STAGES == 2) {
      if (n + 1 < p.N) {
        // Both buffers of chunk n+1 were last read in chunk n-1, before barrier #1.
        const uint8_t* nslab = slab + p.slab_bytes;
        Stage<GATE> nst(stage_at(n + 1));
        load_big<GATE>(p, nst, nslab, b, h, n + 1, tid);
        load_small(Small(small_at(n + 1)), nslab, v0, tid);
        cp_commit();
      }
    }

    // ---- B: r^T = U^T - S^T W^T and o^T part 1 = S^T q^T (one n-tile each) --------
    float Rhh[4], Rlh[4], Rhl[4], Oh[4], Ol[4], Ox[4];
    {
      const int j = jw + 2 * t4;
      Rhh[0] = sm.u[j * VT + g];
      Rhh[1] = sm.u[(j + 1) * VT + g];
      Rhh[2] = sm.u[j * VT + g + 8];
      Rhh[3] = sm.u[(j + 1) * VT + g + 8];
#pragma unroll
      for (int e = 0; e < 4; ++e) Rlh[e] = Rhl[e] = Oh[e] = Ol[e] = Ox[e] = 0.f;
    }
#pragma unroll
    for (int ks = 0; ks < K / 16; ks += 2) {
      uint32_t wh[4], wl[4], qh[4];
      ldsm_x4(wh, smem_u32(st.w_hi + (jw + brow) * LDW + 16 * ks + bcol));
      ldsm_x4(wl, smem_u32(st.w_lo + (jw + brow) * LDW + 16 * ks + bcol));
      ldsm_x4(qh, smem_u32(st.q_hi + (jw + brow) * LDW + 16 * ks + bcol));
      uint32_t ql[4];
      if (GATE) ldsm_x4(ql, smem_u32(st.q_lo + (jw + brow) * LDW + 16 * ks + bcol));
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t ah[4], al[4];
        ldsm_x4(ah, smem_u32(xs_hi + arow * LDW + 16 * (ks + h2) + acol));
        ldsm_x4(al, smem_u32(xs_lo + arow * LDW + 16 * (ks + h2) + acol));
        mma(Rhh, ah, wh[2 * h2], wh[2 * h2 + 1]);
        mma(Rlh, al, wh[2 * h2], wh[2 * h2 + 1]);
        mma(Rhl, ah, wl[2 * h2], wl[2 * h2 + 1]);
        mma(Oh, ah, qh[2 * h2], qh[2 * h2 + 1]);
        mma(Ol, al, qh[2 * h2], qh[2 * h2 + 1]);
        if (GATE) mma(Ox, ah, ql[2 * h2], ql[2 * h2 + 1]);
      }
    }

    // ---- C: publish r^T and rho^T = r^T diag(kscale); scale o part 1 -------------
    float O[4];
    {
      const int j = jw + 2 * t4;
      float R[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) R[e] = Rhh[e] + (Rlh[e] + Rhl[e]);
      uint32_t hi, lo;
      split_pair(R[0], R[1], hi, lo);
      *reinterpret_cast<uint32_t*>(xr_hi + g * LDA + j) = hi;
      *reinterpret_cast<uint32_t*>(xr_lo + g * LDA + j) = lo;
      split_pair(R[2], R[3], hi, lo);
      *reinterpret_cast<uint32_t*>(xr_hi + (g + 8) * LDA + j) = hi;
      *reinterpret_cast<uint32_t*>(xr_lo + (g + 8) * LDA + j) = lo;
      const float k0 = sm.ks[j], k1 = sm.ks[j + 1];
      split_pair(R[0] * k0, R[1] * k1, hi, lo);
      *reinterpret_cast<uint32_t*>(xp_hi + g * LDA + j) = hi;
      *reinterpret_cast<uint32_t*>(xp_lo + g * LDA + j) = lo;
      split_pair(R[2] * k0, R[3] * k1, hi, lo);
      *reinterpret_cast<uint32_t*>(xp_hi + (g + 8) * LDA + j) = hi;
      *reinterpret_cast<uint32_t*>(xp_lo + (g + 8) * LDA + j) = lo;
      const float q0 = sm.qs[j], q1 = sm.qs[j + 1];
      O[0] = (Oh[0] + (Ol[0] + Ox[0])) * q0;
      O[1] = (Oh[1] + (Ol[1] + Ox[1])) * q1;
      O[2] = (Oh[2] + (Ol[2] + Ox[2])) * q0;
      O[3] = (Oh[3] + (Ol[3] + Ox[3])) * q1;
    }
    if constexpr (STAGES == 1) cp_wait<0>();  // group 2 (K, A_qk) of chunk n landed
    __syncthreads();                           // #2: r^T / rho^T tiles visible

    // ---- D: S^T = gamma S^T + rho^T k (channels of this warp), o^T part 2 -----------
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int c = cw + 8 * nt + 2 * t4;
      const float g0 = sm.gam[c], g1 = sm.gam[c + 1];
      S[nt][0] *= g0;
      S[nt][1] *= g1;
      S[nt][2] *= g0;
      S[nt][3] *= g1;
    }
    float Dl[2][4], Dx[2][4], Phh[4], Plh[4], Phl[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      Dl[0][e] = Dl[1][e] = Dx[0][e] = Dx[1][e] = 0.f;
      Phh[e] = Plh[e] = Phl[e] = 0.f;
    }
#pragma unroll
    for (int ks = 0; ks < C / 16; ++ks) {
      uint32_t ph[4], pl[4], kh[4];
      ldsm_x4(ph, smem_u32(xp_hi + arow * LDA + 16 * ks + acol));
      ldsm_x4(pl, smem_u32(xp_lo + arow * LDA + 16 * ks + acol));
      ldsm_x4_t(kh, smem_u32(st.k_hi + (16 * ks + krow) * LDW + kcol));
      mma(S[0], ph, kh[0], kh[1]);
      mma(S[1], ph, kh[2], kh[3]);
      mma(Dl[0], pl, kh[0], kh[1]);
      mma(Dl[1], pl, kh[2], kh[3]);
      if (GATE) {
        uint32_t kl[4];
        ldsm_x4_t(kl, smem_u32(st.k_lo + (16 * ks + krow) * LDW + kcol));
        mma(Dx[0], ph, kl[0], kl[1]);
        mma(Dx[1], ph, kl[2], kl[3]);
      }
    }
#pragma unroll
    for (int ks = 0; ks < C / 16; ks += 2) {
      uint32_t ah[4], al[4];
      ldsm_x4(ah, smem_u32(st.aq_hi + (jw + brow) * LDA + 16 * ks + bcol));
      ldsm_x4(al, smem_u32(st.aq_lo + (jw + brow) * LDA + 16 * ks + bcol));
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t rh[4], rl[4];
        ldsm_x4(rh, smem_u32(xr_hi + arow * LDA + 16 * (ks + h2) + acol));
        ldsm_x4(rl, smem_u32(xr_lo + arow * LDA + 16 * (ks + h2) + acol));
        mma(Phh, rh, ah[2 * h2], ah[2 * h2 + 1]);
        mma(Plh, rl, ah[2 * h2], ah[2 * h2 + 1]);
        mma(Phl, rh, al[2 * h2], al[2 * h2 + 1]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) S[nt][e] += Dl[nt][e] + Dx[nt][e];

    // ---- E: o rows of this warp (i in [8 warp, +8)) -> global -------------------
    {
      const int i = 2 * t4;
      xo[i * 16 + g] = O[0] + (Phh[0] + (Plh[0] + Phl[0]));
      xo[(i + 1) * 16 + g] = O[1] + (Phh[1] + (Plh[1] + Phl[1]));
      xo[i * 16 + g + 8] = O[2] + (Phh[2] + (Plh[2] + Phl[2]));
      xo[(i + 1) * 16 + g + 8] = O[3] + (Phh[3] + (Plh[3] + Phl[3]));
    }
    __syncwarp();
    {
      const int i = lane >> 2, c4 = (lane & 3) * 4;   // 8 rows x 4 float4
      const int t = t0 + jw + i;
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

    if constexpr (STAGES == 1) {
      if (n + 1 < p.N) {
        // Every warp must be done with this chunk's tiles before they are
        // overwritten: a CTA barrier, then the next chunk in two groups.
        __syncthreads();
        const uint8_t* nslab = slab + p.slab_bytes;
        Stage<1> nst(stage_at(n + 1));
        load_group1(nst, Small(small_at(n + 1)), nslab, v0, tid);
        load_group2(nst, nslab, tid);
      }
    }
  }

  if (p.sT) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int c = cw + 8 * nt + 2 * t4;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int vv = g + (e >> 1) * 8, cc = c + (e & 1);
        p.sT[(seq * K + cc) * V + v0 + vv] = S[nt][e];
      }
    }
  }
}

template <int GATE, int STAGES>
gdr_status launch_one(const Params& p, cudaStream_t stream) {
  const int smem = Smem::total(GATE, STAGES);
  auto kern = state_kernel<GATE, STAGES>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return GDR_ERR_CUDA;
  dim3 grid(V / VT, p.HV, p.B);
  kern<<<grid, THREADS, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

}  // namespace

gdr_status launch_state(const Params& p, cudaStream_t stream) {
  if (p.gate_mode) return launch_one<1, 1>(p, stream);
  return launch_one<0, 2>(p, stream);
}

}  // namespace fast
}  // namespace gdr
