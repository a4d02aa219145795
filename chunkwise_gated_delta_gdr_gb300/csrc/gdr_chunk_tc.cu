// gdr_chunk_tc.cu -- chunk-local stage of the fast path on tcgen05 tensor cores.
//
// One group of 8 warps per chunk (n, hv, b), scalar gate, bf16 inputs, C = 64,
// K = V = 128. It computes, for one chunk of the "分块并行计算（Chunkwise）"
// notes (section "chunk 内的 cumsum 与下三角解"):
//   G     = cumsum(g)                                 (in-chunk gate cumsum)
//   P, Q  = k k^T, q k^T       one tcgen05 MMA, A = [k; q] stacked to M = 128
//   A_kk  = P |k_i|^-1 |k_j|^-1 exp(G_i - G_j)        (L2 norm and decay as fp32
//   A_qk  = Q scale |q_i|^-1 |k_j|^-1 exp(G_i - G_j) beta_j   epilogue factors;
//                                                      the bf16 inputs are exact)
//   M     = I + tril(A_kk beta_j, -1),  X = M^-1      (fp32, 16x16 diagonal blocks
//                                                      by substitution, off-diagonal
//                                                      blocks by block products)
//   W     = X diag(exp(G_j) |k_j|^-1) k,  U = X v     two tcgen05 MMAs with A =
//                                                      [X_hi; X_lo] stacked to M = 128
//                                                      and the raw bf16 k / v tile as B
// and writes the slab of gdr_fast.cuh. q, k and v arrive by TMA (128-byte
// swizzle, zero fill past the end of the sequence, which is the zero padding of
// the last chunk); accumulators live in TMEM; A_qk, -W, U, -T and the key
// tile are staged as 128-byte swizzled tiles whose byte images leave by bulk
// copies (the recurrence loads them back the same way, which restores the
// swizzled layout without a tensor map). Each per-thread phase is
// spread over the 8 warps (two per TMEM lane quadrant, one per column half).
//
// For the Mamba2 SSD recurrence of the "Chunkwise 并行算法 —— 线性注意力" page
// (§1.1-1.2: no delta erase, beta = 1) M = I, W = 0 and U = v, so the chunk
// stops after A_qk and the row factors and forms, instead of W, U and T, its
// whole state increment N = k^T diag(kscale) v (four tcgen05 products with the
// raw keys as A), which turns the recurrence into a scan (ssd_increment).
//
// The work of one chunk is the device function produce_chunk. It runs in the
// chunk kernel below (one CTA per chunk, two CTAs per SM) and, for the
// one-launch forward, in the worker CTAs of gdr_chain.cu (two groups of 8
// warps per CTA, each taking chunks in chunk order and raising a flag per
// chunk once its slab is in global memory).
#include "gdr_chunk_tc.cuh"

namespace gdr {
namespace fast {
namespace chunk {

// Encodes the tensor maps of the chunk-local stage.
bool make_maps(Maps* m, const Params& p) {
  return tmap_bthd(&m->q, p.q, p.B, p.T, p.H) && tmap_bthd(&m->k, p.k, p.B, p.T, p.H) &&
         tmap_bthd(&m->v, p.v, p.B, p.T, p.HV);
}

}  // namespace chunk

namespace {

template <bool kSsd>
__global__ void __launch_bounds__(chunk::THREADS, 2) chunk_tc_kernel(
    const __grid_constant__ chunk::Maps maps, Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + chunk::OFF_BAR);
  if (threadIdx.x == 0) chunk::init_group_bars(sm);
  // (the first barrier inside produce_chunk orders the initialisation before
  // any wait; only thread 0 uses the barriers before it)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  chunk::produce_chunk<kSsd>(maps, p, sm, threadIdx.x, 1, blockIdx.x, blockIdx.y, blockIdx.z, 0, 0,
                       tslot, nullptr);
  if (threadIdx.x == 0) ptx::bulk_wait_read<0>();   // staging read before the smem is released
  if ((threadIdx.x >> 5) == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(*tslot, chunk::TMEM_COLS);
  }
}

}  // namespace

gdr_status launch_chunk_tc(const Params& p, cudaStream_t stream) {
  if (p.gate_mode != 0) return launch_chunk_kda(p, stream);
  chunk::Maps m;
  if (!chunk::make_maps(&m, p)) return GDR_ERR_CUDA;
  const auto kern = p.ssd ? chunk_tc_kernel<true> : chunk_tc_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           chunk::SMEM_BYTES) != cudaSuccess)
    return GDR_ERR_CUDA;
  dim3 grid(p.N, p.HV, p.B);
  kern<<<grid, chunk::THREADS, chunk::SMEM_BYTES, stream>>>(m, p);
  return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

}  // namespace fast
}  // namespace gdr
