// gdr_fast.cuh -- shared definitions of the fast path (bf16, K = V = 128, C = 64).
//
// The fast path has two stages:
//   1. a chunk-local stage (one chunk per CTA or per worker group) writes, per
//      chunk, the operands of the inter-chunk recurrence into a workspace slab:
//      gdr_chunk_tc.cu (tcgen05, scalar gate) or gdr_chunk_kda.cu (mma.sync,
//      per-key gate);
//   2. a recurrence stage runs the chunks in order per (batch, value head,
//      V tile) and writes the outputs: gdr_chain.cu (scalar gate, tcgen05) or
//      gdr_state_kda.cu (per-key gate, tcgen05).
// For the scalar gate gdr_chain.cu can also run both stages in one cooperative
// launch: worker CTAs produce the slabs in chunk order and raise one flag per
// chunk, chain CTAs consume them as they appear.
// This header fixes the slab format both stages agree on.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "gdr_internal.cuh"

namespace gdr {
namespace fast {

constexpr int C = 64;    // chunk length
constexpr int K = 128;   // key head dim
constexpr int V = 128;   // value head dim

// Rows of a stacked hi / lo operand [X_hi; X_lo] (2C rows) interleaved in
// blocks of 16: row i of the hi part is stacked row 32 (i / 16) + i % 16, row i
// of the lo part that + 16. An M = 128 tcgen05 product with this operand puts
// the hi and lo results of row i in TMEM lanes of one warp (lanes t and t + 16
// of lane quadrant i / 16), so one shuffle adds them.
__host__ __device__ constexpr int stacked_row(int i, int lo) { return 32 * (i >> 4) + (i & 15) + 16 * lo; }

// Slab of one chunk (b, hv, n), chunk index ((b * HV + hv) * N + n). All
// offsets in bytes from the slab start; every array is 16-byte aligned.
//   W2   [2C][K] bf16  hi / lo of -W, W = M^-1 (exp(G) k_hat). Scalar gate:
//                      the two parts stacked by stacked_row; per-key gate: hi
//                      rows 0 .. C-1, then lo rows.
//   AQ2  [2C][C] bf16  hi / lo of A_qk (beta on its columns, zero above the
//                      diagonal), arranged like W2.
//   U    [C][V]    fp32  U = M^-1 v
//   VEC  qscale[C], kscale[C], gamma[K] fp32
//        scalar gate: qscale_i = scale |q_i|^-1 exp(G_i), kscale_j = beta_j |k_j|^-1
//        exp(G_last - G_j), gamma = exp(G_last) on every channel;
//        per-key gate: qscale = kscale = 1, gamma_c = exp(G_last,c)
//   QB2  [2][C][K] bf16  per-key gate only: hi / lo of scale q_hat exp(G)
//   KB2  [2][C][K] bf16  per-key gate only: hi / lo of beta k_hat exp(G_last - G)
// For the scalar gate the recurrence reads raw q and k from the inputs (exact
// in bf16) and applies qscale / kscale as fp32 row factors.
struct Slab {
  static constexpr size_t W2 = 0;
  static constexpr size_t AQ2 = W2 + 2ull * C * K * 2;
  static constexpr size_t U = AQ2 + 2ull * C * C * 2;
  static constexpr size_t VEC = U + (size_t)C * V * 4;
  static constexpr size_t QB2 = VEC + (size_t)(2 * C + K) * 4;
  static constexpr size_t KB2 = QB2 + 2ull * C * K * 2;
  static constexpr size_t SCALAR_BYTES = QB2;
  static constexpr size_t PERKEY_BYTES = KB2 + 2ull * C * K * 2;
  static constexpr size_t bytes(int gate_mode) { return gate_mode ? PERKEY_BYTES : SCALAR_BYTES; }
};
static_assert(Slab::AQ2 % 16 == 0 && Slab::U % 16 == 0 && Slab::VEC % 16 == 0 &&
                  Slab::QB2 % 16 == 0 && Slab::KB2 % 16 == 0,
              "slab arrays must stay 16-byte aligned");

// Everything both stages of the fast path need.
struct Params {
  const __nv_bfloat16* q;   // [B, T, H, K]
  const __nv_bfloat16* k;   // [B, T, H, K]
  const __nv_bfloat16* v;   // [B, T, HV, V]
  const float* g;           // [B, T, HV] or [B, T, HV, K]
  const float* beta;        // [B, T, HV]
  const float* s0;          // [B, HV, K, V] or null
  void* out;                // [B, T, HV, V]
  float* sT;                // [B, HV, K, V] or null
  uint8_t* slabs;           // N * B * HV slabs
  unsigned int* flags;      // one per chunk (slab index): nonzero once its slab is written
                            // (one-launch forward of the scalar gate), else null
  unsigned int* error_word;
  int B, T, H, HV, N;
  int out_bf16, gate_mode, use_l2;
  int ssd;                  // Mamba2 SSD update: no delta erase (W = 0), beta = 1
  int zero_u;               // recurrence reads U as zero (the chunk map's linear part)
  int recur_mode;           // 0 states and outputs; 1 states (outputs too where one kernel
                            // writes both); 2 the separate output pass (gdr_internal.cuh)
  float scale;
  size_t slab_bytes;
  long wait_limit;          // polls of a chain's bounded wait on a chunk flag before it
                            // gives up (one-launch forward)
};

inline __host__ __device__ size_t slab_index(const Params& p, int b, int hv, int n) {
  return ((size_t)b * p.HV + hv) * p.N + n;
}

// Launchers.
// Scalar gate: recurrence after a finished chunk-local stage (gdr_chain.cu).
gdr_status launch_chain(const Params& p, cudaStream_t stream);
// Scalar gate: both stages in one cooperative launch (gdr_chain.cu); declines
// with GDR_ERR_UNSUPPORTED (nothing enqueued) when it does not pay.
gdr_status launch_fused(const Params& p, cudaStream_t stream);
// Whether launch_fused runs for B x HV sequences on the current device.
bool fused_fits(int B, int HV);
// Per-key gate: the recurrence on tcgen05, 64 value columns per CTA (gdr_state_kda.cu).
gdr_status launch_state_kda_tc(const Params& p, cudaStream_t stream);
// Per-key gate: chunk-local kernel on mma.sync (gdr_chunk_kda.cu).
gdr_status launch_chunk_kda(const Params& p, cudaStream_t stream);
// Chunk-local kernel (gdr_chunk_tc.cu; forwards the per-key gate to gdr_chunk_kda.cu).
gdr_status launch_chunk_tc(const Params& p, cudaStream_t stream);

}  // namespace fast
}  // namespace gdr
