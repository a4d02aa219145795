// gdr_segment.cu -- segmented (parallel) scan of the inter-chunk recurrence.
//
// Over one chunk the state map of the chunk form is affine,
//     S' = (gamma - KB^T W) S + KB^T U,
// so over a segment of chunks it is S_out = A_p S_in + B_p with A_p the product
// of the chunks' linear parts (the "keyed scan" of the affine chunk maps that
// "DeltaNet chunk kernel optimization" observes, section on cross-chunk state
// passing). gdr_chunk_fwd_segmented splits every sequence into P equal segments
// and runs, all on the caller's stream:
//   1. the chunk-local kernel once, on the sequences viewed as B P sequences of
//      T / P tokens (a contiguous reshape of every [B, T, ...] tensor);
//   2. the recurrence from a zero state: the final states are B_p;
//   3. the recurrence from the identity with U read as zero: the final states
//      are A_p (K x K; needs K = V);
//   4. segment_combine_kernel: S_0 = initial state, S_{p+1} = A_p S_p + B_p,
//      serial over the P segments, parallel over (b, hv, 16-column tiles);
//   5. the recurrence from the S_p, which writes the outputs.
// Steps 2, 3 and 5 launch the scalar-gate recurrence with its state chains only
// (no output CTAs, so any number of chains, in waves); step 5 then launches its
// output CTAs alone, on every SM, over the exchange blocks the chains left.
// The recurrences are T / P chunks long instead of T, at the cost of two more
// of them and the combine, so it pays when the sequences are few and long (few
// chains to spread over the SMs).
#include "gdr_internal.cuh"
#include "gdr_ptx.cuh"

namespace gdr {
namespace {

constexpr int kSegThreads = 256;
constexpr int kSegCols = 16;     // state columns per CTA
constexpr int kSegRows = 64;     // rows of A_p per shared-memory block

// A[n][K][K] = identity for every one of the n states.
__global__ void segment_identity_kernel(float* A, long n, int K) {
  const long total = n * K * K;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
       i += (long)gridDim.x * blockDim.x) {
    const long e = i % ((long)K * K);
    A[i] = (e / K == e % K) ? 1.f : 0.f;
  }
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// Rows [r0, r0 + rows) of the K x K matrix src into dst (row stride ld), by cp.async.
template <bool kVec>
__device__ __forceinline__ void stage_rows(float* dst, const float* src, int r0, int rows, int K,
                                           int ld, int tid) {
  if (kVec) {
    const int per = K >> 2;
    for (int e = tid; e < rows * per; e += kSegThreads) {
      const int r = e / per, c = 4 * (e - r * per);
      ptx::cp_async16(ptx::smem_u32(dst + r * ld + c), src + (size_t)(r0 + r) * K + c, 16);
    }
  } else {
    for (int e = tid; e < rows * K; e += kSegThreads) {
      const int r = e / K, c = e - r * K;
      cp_async4(ptx::smem_u32(dst + r * ld + c), src + (size_t)(r0 + r) * K + c);
    }
  }
}

// One CTA per (16-column tile, hv, b) runs S_{p+1} = A_p S_p + B_p over the P
// segments of its column tile, with S in shared memory and A_p streamed through
// two shared-memory blocks of 64 rows (the copy of the next block overlaps the
// product on the current one). States [K][K] fp32, segment p of batch b at
// index (b P + p) HV + hv. kVec: K a multiple of 4 (16-byte copies and loads).
template <bool kVec>
__global__ void __launch_bounds__(kSegThreads) segment_combine_kernel(
    const float* A, const float* Bst, const float* s0, float* Sin, float* sT, int P, int HV,
    int K) {
  extern __shared__ __align__(16) float sm[];
  const int ld = K + 4;                              // A row stride: rows 1 apart, 4 banks apart
  float* S = sm;                                     // [K][kSegCols]
  float* S2 = S + K * kSegCols;
  float* Ab = S2 + K * kSegCols;                     // 2 x [kSegRows][ld]
  const int vt = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
  const int c0 = vt * kSegCols;
  const int cw = min(kSegCols, K - c0);
  const int tid = threadIdx.x, j = tid % kSegCols, ri = tid / kSegCols;   // ri in [0, 16)
  const size_t plane = (size_t)K * K;
  const int nrb = (K + kSegRows - 1) / kSegRows;
  const int nt = P * nrb;
  auto mat = [&](const float* X, int p) { return X + (((size_t)b * P + p) * HV + hv) * plane; };

  for (int i = tid / kSegCols; i < K; i += kSegThreads / kSegCols)
    S[i * kSegCols + j] =
        (s0 && j < cw) ? s0[((size_t)b * HV + hv) * plane + (size_t)i * K + c0 + j] : 0.f;
  stage_rows<kVec>(Ab, mat(A, 0), 0, min(kSegRows, K), K, ld, tid);
  ptx::cp_async_commit();
  __syncthreads();
  for (int t = 0; t < nt; ++t) {
    const int p = t / nrb, rb = t - p * nrb, r0 = rb * kSegRows;
    const int rows = min(kSegRows, K - r0);
    if (rb == 0 && j < cw)                           // S holds S_p
      for (int i = ri; i < K; i += kSegThreads / kSegCols)
        Sin[(mat(Sin, p) - Sin) + (size_t)i * K + c0 + j] = S[i * kSegCols + j];
    if (t + 1 < nt) {
      const int p1 = (t + 1) / nrb, r1 = ((t + 1) - p1 * nrb) * kSegRows;
      stage_rows<kVec>(Ab + ((t + 1) & 1) * kSegRows * ld, mat(A, p1), r1,
                       min(kSegRows, K - r1), K, ld, tid);
    }
    ptx::cp_async_commit();
    const float* Bp = mat(Bst, p);
    float acc[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int i = ri + 16 * m;
      acc[m] = (i < rows && j < cw) ? Bp[(size_t)(r0 + i) * K + c0 + j] : 0.f;
    }
    ptx::cp_async_wait<1>();                         // this thread's copies of block t
    __syncthreads();                                 // everyone's
    const float* Ar = Ab + (t & 1) * kSegRows * ld + ri * ld;
    // Rows past the block's end read stale (in-bounds) data and are not stored.
    if (kVec) {
      for (int c = 0; c < K; c += 4) {
        const float s_0 = S[(c + 0) * kSegCols + j], s_1 = S[(c + 1) * kSegCols + j];
        const float s_2 = S[(c + 2) * kSegCols + j], s_3 = S[(c + 3) * kSegCols + j];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float4 a = *reinterpret_cast<const float4*>(Ar + 16 * m * ld + c);
          acc[m] = fmaf(a.x, s_0, acc[m]);
          acc[m] = fmaf(a.y, s_1, acc[m]);
          acc[m] = fmaf(a.z, s_2, acc[m]);
          acc[m] = fmaf(a.w, s_3, acc[m]);
        }
      }
    } else {
      for (int c = 0; c < K; ++c) {
        const float sv = S[c * kSegCols + j];
#pragma unroll
        for (int m = 0; m < 4; ++m) acc[m] = fmaf(Ar[16 * m * ld + c], sv, acc[m]);
      }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m)
      if (ri + 16 * m < rows) S2[(r0 + ri + 16 * m) * kSegCols + j] = acc[m];
    __syncthreads();                                 // block t read; S2 rows written
    if (rb == nrb - 1) {                             // S_{p+1} complete
      float* x = S;
      S = S2;
      S2 = x;
    }
  }
  if (sT && j < cw)
    for (int i = ri; i < K; i += kSegThreads / kSegCols)
      sT[((size_t)b * HV + hv) * plane + (size_t)i * K + c0 + j] = S[i * kSegCols + j];
}

}  // namespace

gdr_status launch_segment_identity(float* A, long n, int K, cudaStream_t stream) {
  segment_identity_kernel<<<1024, 256, 0, stream>>>(A, n, K);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

gdr_status launch_segment_combine(const float* A, const float* Bst, const float* s0, float* Sin,
                                  float* sT, int B, int P, int HV, int K, cudaStream_t stream) {
  const size_t smem =
      sizeof(float) * (2 * (size_t)K * kSegCols + 2 * (size_t)kSegRows * (K + 4));
  const bool vec = (K & 3) == 0;
  const void* fn = vec ? (const void*)segment_combine_kernel<true>
                       : (const void*)segment_combine_kernel<false>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return GDR_ERR_CUDA;
  dim3 grid((K + kSegCols - 1) / kSegCols, HV, B);
  if (vec)
    segment_combine_kernel<true><<<grid, kSegThreads, smem, stream>>>(A, Bst, s0, Sin, sT, P, HV, K);
  else
    segment_combine_kernel<false><<<grid, kSegThreads, smem, stream>>>(A, Bst, s0, Sin, sT, P, HV, K);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

}  // namespace gdr
