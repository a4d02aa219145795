// gdr_trinv.cuh -- blocked inverse of a 64x64 unit lower-triangular matrix.
//
// X = (I + L)^-1 for the in-chunk system M = I + tril(A_kk beta, -1) of the
// "分块并行计算（Chunkwise）" notes (section "chunk 内的 cumsum 与下三角解"): the
// notes solve it with a triangular solve; here it is inverted once in fp32,
// so that W = X (...) and U = X v become plain products on the tensor cores.
//   level 0: the four 16x16 diagonal blocks, by forward substitution
//            x_i = delta_ij - sum_{m<i} L_im x_m (one column per thread);
//   level 1: X_10 = -X_11 L_10 X_00 and X_32 = -X_33 L_32 X_22;
//   level 2: X[32:64, 0:32] = -X[32:64, 32:64] L[32:64, 0:32] X[0:32, 0:32].
// Only the strictly lower entries of L are read. Inside the two 32x32 diagonal
// blocks everything above the diagonal is written as exact zeros (the 16x16
// diagonal blocks' upper triangles and the blocks X_01, X_23), so the level-2
// products need no masks; X[0:32, 32:64] is never written. All 256 threads of
// the CTA call it; it synchronises the CTA between levels but not after the
// last writes (the caller does). The 256 threads meet on named barrier bar_id
// (a whole 256-thread CTA may pass 0, the barrier of __syncthreads).
#pragma once

#include "gdr_ptx.cuh"

namespace gdr {
namespace fast {

__device__ __forceinline__ void trinv_sync(int bar_id) {
  asm volatile("bar.sync %0, 256;" ::"r"(bar_id) : "memory");
}

// Level 0 for threads 0-63: column (tid & 15) of diagonal block tid >> 4, in registers.
template <int LDL>
__device__ __forceinline__ void inverse_level0(const float* L, float (&xd)[16], int tid) {
  const int o = (tid >> 4) * 16, col = tid & 15;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float acc = (i == col) ? 1.f : 0.f;
#pragma unroll
    for (int m = 0; m < i; ++m) acc = fmaf(-L[(o + i) * LDL + o + m], xd[m], acc);
    xd[i] = acc;
  }
}
// Threads 0-63 store their column; those of diagonal blocks 0 and 2 also zero
// the same column of the block to the right (X_01, X_23).
template <int LDX>
__device__ __forceinline__ void inverse_level0_store(float* X, const float (&xd)[16], int tid) {
  const int o = (tid >> 4) * 16, col = tid & 15;
  const bool zero_right = ((tid >> 4) & 1) == 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    X[(o + i) * LDX + o + col] = xd[i];
    if (zero_right) X[(o + i) * LDX + o + 16 + col] = 0.f;
  }
}

// Levels 1 and 2, once the diagonal blocks of X are in place and visible.
template <int LDL, int LDX>
__device__ __forceinline__ void inverse_levels12(const float* L, float* X, float* T, int tid,
                                                 int bar_id) {
  // Level 1: threads 0-127, each one row segment of 4 columns.
  {
    const int which = (tid >> 6) & 1, e = tid & 63, i = e >> 2, j0 = (e & 3) * 4;
    const int I = 16 * (2 * which + 1), J = I - 16;
    if (tid < 128) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float l = L[(I + i) * LDL + J + m];
        const float4 xv = *reinterpret_cast<const float4*>(X + (J + m) * LDX + J + j0);
        acc.x = fmaf(l, xv.x, acc.x); acc.y = fmaf(l, xv.y, acc.y);
        acc.z = fmaf(l, xv.z, acc.z); acc.w = fmaf(l, xv.w, acc.w);
      }
      *reinterpret_cast<float4*>(T + (which * 16 + i) * 36 + j0) = acc;
    }
    trinv_sync(bar_id);
    if (tid < 128) {
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
  }
  trinv_sync(bar_id);
  // Level 2: each thread one row segment of 4 columns. The zeros above the
  // diagonal of X[0:32, 0:32] and X[32:64, 32:64] are stored, so the products
  // run over the full 32 x 32 blocks.
  {
    const int i = tid >> 3, j0 = (tid & 7) * 4;
    float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int m = 0; m < 32; ++m) {
      const float l = L[(32 + i) * LDL + m];
      const float4 x0 = *reinterpret_cast<const float4*>(X + m * LDX + j0);
      a[0] = fmaf(l, x0.x, a[0]); a[1] = fmaf(l, x0.y, a[1]);
      a[2] = fmaf(l, x0.z, a[2]); a[3] = fmaf(l, x0.w, a[3]);
    }
    // The level-1 scratch was last read before the barrier that ends level 1.
    *reinterpret_cast<float4*>(T + i * 36 + j0) = make_float4(a[0], a[1], a[2], a[3]);
    trinv_sync(bar_id);
    float r4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int m = 0; m < 32; ++m) {
      const float xv = X[(32 + i) * LDX + 32 + m];
      const float4 t4 = *reinterpret_cast<const float4*>(T + m * 36 + j0);
      const float ts[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
      for (int z = 0; z < 4; ++z) r4[z] = fmaf(xv, ts[z], r4[z]);
    }
    *reinterpret_cast<float4*>(X + (32 + i) * LDX + j0) = make_float4(-r4[0], -r4[1], -r4[2], -r4[3]);
  }
}

// D += A B for one 16x8 tile on the tensor cores, A a 16x16 block of the fp32
// matrix A (row stride lda) at (ar, ac), B a 16x8 block of the fp32 matrix B
// (row stride ldb) at (bk, bn): both split into bf16 hi + lo, three products
// (hi hi, lo hi, hi lo; the lo lo term and the lo parts' own rounding leave a
// relative error near 2^-16). Fragment layouts of mma.m16n8k16: lane (g, t) =
// (lane / 4, lane % 4) holds A rows g, g + 8 at columns 2t, 2t + 1, 2t + 8,
// 2t + 9, and B rows 2t, 2t + 1, 2t + 8, 2t + 9 at column g.
__device__ __forceinline__ void mma16x8_split(float (&d)[4], const float* A, int lda, int ar,
                                              int ac, const float* B, int ldb, int bk, int bn,
                                              int lane) {
  const int g = lane >> 2, t = lane & 3;
  const float* a0 = A + (ar + g) * lda + ac + 2 * t;
  const float2 x0 = *reinterpret_cast<const float2*>(a0);
  const float2 x1 = *reinterpret_cast<const float2*>(a0 + 8 * lda);
  const float2 x2 = *reinterpret_cast<const float2*>(a0 + 8);
  const float2 x3 = *reinterpret_cast<const float2*>(a0 + 8 * lda + 8);
  uint32_t ah[4], al[4];
  ptx::split_pair(x0.x, x0.y, ah[0], al[0]);
  ptx::split_pair(x1.x, x1.y, ah[1], al[1]);
  ptx::split_pair(x2.x, x2.y, ah[2], al[2]);
  ptx::split_pair(x3.x, x3.y, ah[3], al[3]);
  const float* b0 = B + (bk + 2 * t) * ldb + bn + g;
  uint32_t bh0, bl0, bh1, bl1;
  ptx::split_pair(b0[0], b0[ldb], bh0, bl0);
  ptx::split_pair(b0[8 * ldb], b0[9 * ldb], bh1, bl1);
  ptx::mma_bf16_16816(d, ah, bh0, bh1);
  ptx::mma_bf16_16816(d, al, bh0, bh1);
  ptx::mma_bf16_16816(d, ah, bl0, bl1);
}

// Stores s * D of a 16x8 tile at (r0, c0) of the fp32 matrix M (row stride ld).
__device__ __forceinline__ void store16x8(float* M, int ld, int r0, int c0, const float (&d)[4],
                                          float s, int lane) {
  const int g = lane >> 2, t = lane & 3;
  float* m = M + (r0 + g) * ld + c0 + 2 * t;
  *reinterpret_cast<float2*>(m) = make_float2(s * d[0], s * d[1]);
  *reinterpret_cast<float2*>(m + 8 * ld) = make_float2(s * d[2], s * d[3]);
}

// Levels 1 and 2 as split-bf16 mma.sync products (same blocks and order as
// inverse_levels12): level 1 on warps 0-3 (block pair w / 2, 8-column tile
// w % 2), level 2 on all 8 warps (16-row tile w / 4, 8-column tile w % 4).
// The scratch T holds the 16x16 level-1 products in rows 0-31, columns 0-15,
// then the 32x32 level-2 product.
template <int LDL, int LDX>
__device__ __forceinline__ void inverse_levels12_mma(const float* L, float* X, float* T, int tid,
                                                     int bar_id) {
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int LDT = 36;
  {
    const int which = warp >> 1, nt = warp & 1;
    const int I = 16 * (2 * which + 1), J = I - 16;
    if (warp < 4) {                                   // T_w = L[I, J] X[J, J]
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      mma16x8_split(d, L, LDL, I, J, X, LDX, J, J + 8 * nt, lane);
      store16x8(T, LDT, 16 * which, 8 * nt, d, 1.f, lane);
    }
    trinv_sync(bar_id);
    if (warp < 4) {                                   // X[I, J] = -X[I, I] T_w
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      mma16x8_split(d, X, LDX, I, I, T, LDT, 16 * which, 8 * nt, lane);
      store16x8(X, LDX, I, J + 8 * nt, d, -1.f, lane);
    }
  }
  trinv_sync(bar_id);
  const int mt = warp >> 2, nt = warp & 3;
  {                                                   // T = L[32:64, 0:32] X[0:32, 0:32]
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    mma16x8_split(d, L, LDL, 32 + 16 * mt, 0, X, LDX, 0, 8 * nt, lane);
    mma16x8_split(d, L, LDL, 32 + 16 * mt, 16, X, LDX, 16, 8 * nt, lane);
    store16x8(T, LDT, 16 * mt, 8 * nt, d, 1.f, lane);
  }
  trinv_sync(bar_id);
  {                                                   // X[32:64, 0:32] = -X[32:64, 32:64] T
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    mma16x8_split(d, X, LDX, 32 + 16 * mt, 32, T, LDT, 0, 8 * nt, lane);
    mma16x8_split(d, X, LDX, 32 + 16 * mt, 48, T, LDT, 16, 8 * nt, lane);
    store16x8(X, LDX, 32 + 16 * mt, 8 * nt, d, -1.f, lane);
  }
}

// L: [64][LDL] fp32; X: [64][LDX] fp32; T: scratch [32][36] fp32. Levels 1
// and 2 on the tensor cores (inverse_levels12_mma): X then carries a relative
// error near 2^-16, the size of the residual the callers' own hi/lo split of X
// leaves.
template <int LDL, int LDX>
__device__ __forceinline__ void unit_lower_inverse64(const float* L, float* X, float* T, int tid,
                                                     int bar_id) {
  if (tid < 64) {
    float xd[16];
    inverse_level0<LDL>(L, xd, tid);
    inverse_level0_store<LDX>(X, xd, tid);
  }
  trinv_sync(bar_id);
  inverse_levels12_mma<LDL, LDX>(L, X, T, tid, bar_id);
}

}  // namespace fast
}  // namespace gdr
