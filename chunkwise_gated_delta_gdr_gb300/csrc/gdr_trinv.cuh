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
// last writes (the caller does).
#pragma once

namespace gdr {
namespace fast {

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
__device__ __forceinline__ void inverse_levels12(const float* L, float* X, float* T, int tid) {
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
    __syncthreads();
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
  __syncthreads();
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
    __syncthreads();
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

// L: [64][LDL] fp32; X: [64][LDX] fp32; T: scratch [32][36] fp32.
template <int LDL, int LDX>
__device__ __forceinline__ void unit_lower_inverse64(const float* L, float* X, float* T, int tid) {
  if (tid < 64) {
    float xd[16];
    inverse_level0<LDL>(L, xd, tid);
    inverse_level0_store<LDX>(X, xd, tid);
  }
  __syncthreads();
  inverse_levels12<LDL, LDX>(L, X, T, tid);
}

}  // namespace fast
}  // namespace gdr
