// gdr_fast.cuh -- shared definitions of the fast path (bf16, K = V = 128, C = 64).
//
// The fast path has three stages:
//   1. a chunk-local stage (one chunk per CTA or per worker group) writes, per
//      chunk, the operands of the inter-chunk recurrence into a workspace slab:
//      gdr_chunk_tc.cu (tcgen05, scalar gate) or gdr_chunk_kda.cu (mma.sync,
//      per-key gate);
//   2. a recurrence stage runs the chunks in order per (batch, value head,
//      V tile): gdr_chain.cu (scalar gate, tcgen05, the state and r of every
//      chunk exported to an exchange area) or gdr_state_kda.cu (per-key gate,
//      tcgen05, outputs written with the states);
//   3. scalar gate: an output pass forms o from the exchange (gdr_chain.cu).
// For the scalar gate, all three can also run in one cooperative launch:
// worker CTAs produce the slabs in chunk order and raise one flag per chunk,
// chain CTAs consume them as they appear and mark their exports every few
// chunks, and the workers (and each chain CTA once its chain is done) form the
// outputs of the chunks already marked.
// This header fixes the slab and exchange formats the stages agree on.
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
// Scalar gate: every array except VEC is the byte image of a 128-byte swizzled
// shared-memory tile (the chunk-local stage stores its staging tiles with bulk
// copies; a bulk copy into a 1024-aligned tile restores the layout):
//   W2   -W hi / lo stacked by stacked_row: two [2C][64] bf16 boxes (channel halves)
//   AQ2  A_qk hi / lo (beta on its columns, zero above the diagonal), stacked: [2C][C] bf16
//   U    U = M^-1 v: four [C][32] fp32 boxes, box t = value columns 32 t .. 32 t + 31
//   VEC  qscale[C], kscale[C], gamma[K] fp32 (plain)
//   T2   -T hi / lo stacked, T = W k_prev^T with k_prev the raw keys of the
//        previous chunk of the sequence (not written for the first chunk): [2C][C] bf16
//   K2   the chunk's raw keys: two [C][64] bf16 boxes (channel halves)
// with qscale_i = scale |q_i|^-1 exp(G_i), kscale_j = beta_j |k_j|^-1
// exp(G_last - G_j), gamma = exp(G_last) on every channel; the recurrence
// applies them as fp32 row factors to the exact bf16 q and k.
// Mamba2 SSD (W = 0, U = v): W2, U and T2 are not written; instead the chunk's
// state increment N = k^T diag(kscale) v (K x V fp32) takes the W2, T2 and K2
// bytes as four [128 c][32 v] fp32 boxes (128-byte swizzled rows), box t =
// value columns 32 t .. 32 t + 31 at ssd_n(t), and r = v goes straight to the
// chunk's exchange block.
// Per-key gate (the byte images of the 128-byte swizzled boxes the recurrence
// loads with one bulk copy per array: [2][C][K] bf16 arrays as four [C][64]
// boxes, plane-major (hi columns 0-63, hi 64-127, lo 0-63, lo 64-127); [2][C][C]
// as two; U as four [C][32] fp32 boxes):
//   W2   [2][C][K] bf16  hi / lo of -W, W = M^-1 (exp(G) k_hat)
//   AQ2  [2][C][C] bf16  hi / lo of A_qk
//   U    [C][V]    fp32
//   VEC  qscale = kscale = 1, gamma_c = exp(G_last,c)
//   QB2  [2][C][K] bf16  hi / lo of scale q_hat exp(G)
//   KB2  [2][C][K] bf16  hi / lo of beta k_hat exp(G_last - G)
struct Slab {
  static constexpr size_t W2 = 0;
  static constexpr size_t AQ2 = W2 + 2ull * C * K * 2;
  static constexpr size_t U = AQ2 + 2ull * C * C * 2;
  static constexpr size_t VEC = U + (size_t)C * V * 4;
  static constexpr size_t T2 = VEC + (size_t)(2 * C + K) * 4;
  static constexpr size_t K2 = T2 + 2ull * C * C * 2;
  static constexpr size_t QB2 = T2;
  static constexpr size_t KB2 = QB2 + 2ull * C * K * 2;
  static constexpr size_t SCALAR_BYTES = K2 + (size_t)C * K * 2;
  static constexpr size_t PERKEY_BYTES = KB2 + 2ull * C * K * 2;
  static constexpr size_t bytes(int gate_mode) { return gate_mode ? PERKEY_BYTES : SCALAR_BYTES; }
  static constexpr size_t SSD_N_BOX = (size_t)K * 32 * 4;
  __host__ __device__ static constexpr size_t ssd_n(int t) {
    return t < 2 ? W2 + (size_t)t * SSD_N_BOX : T2 + (size_t)(t - 2) * SSD_N_BOX;
  }
};
static_assert(Slab::W2 + 2 * Slab::SSD_N_BOX <= Slab::AQ2 &&
                  Slab::T2 + 2 * Slab::SSD_N_BOX == Slab::SCALAR_BYTES,
              "SSD increment boxes in the W2, T2 and K2 bytes");
static_assert(Slab::AQ2 % 16 == 0 && Slab::U % 16 == 0 && Slab::VEC % 16 == 0 &&
                  Slab::T2 % 16 == 0 && Slab::K2 % 16 == 0 && Slab::QB2 % 16 == 0 &&
                  Slab::KB2 % 16 == 0 && Slab::SCALAR_BYTES % 16 == 0,
              "slab arrays must stay 16-byte aligned");

// Exchange block of one chunk (scalar gate): what the chain CTAs of the
// sequence export for the output pass, as the byte images of their shared
// tiles (128-byte swizzled rows, the layout the output products read):
//   S  [4 tiles][128 c][S_hi 32 | S_lo 32] bf16   the state at the chunk start,
//                                                 tile t = value columns 32 t ..
//   R  [4 tiles][64 j][r_hi 32 | r_lo 32] bf16    r = U - W S, same columns
struct Xchg {
  static constexpr size_t S_TILE = 128ull * 64 * 2;
  static constexpr size_t R_TILE = 64ull * 64 * 2;
  static constexpr size_t S = 0;
  static constexpr size_t R = S + 4 * S_TILE;
  static constexpr size_t BYTES = R + 4 * R_TILE;
};

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
  uint8_t* xchg;            // N * B * HV exchange blocks (scalar gate), else null
  unsigned int* flags;      // one per chunk (slab index): nonzero once its slab is written
                            // (one-launch forward of the scalar gate), else null
  unsigned int* xmark;      // after the flags: per (sequence, 32 value columns) the number of
                            // chunks whose exports are in global memory, then the counter of
                            // claimed output items (one-launch forward), else null
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
// Scalar gate: the output pass over the exchange of a finished recurrence.
gdr_status launch_outputs(const Params& p, cudaStream_t stream);
// Scalar gate: the whole forward in one cooperative launch (gdr_chain.cu);
// declines with GDR_ERR_UNSUPPORTED (nothing enqueued) when it does not pay.
gdr_status launch_fused(const Params& p, cudaStream_t stream);
// Scalar gate: the chains and the output items in one cooperative launch after
// a finished chunk-local stage (the outputs of chunks already exported are
// formed beside the chains); declines with GDR_ERR_UNSUPPORTED (nothing
// enqueued) when the chains do not fit on the SMs at once.
gdr_status launch_chain_outputs(const Params& p, cudaStream_t stream);
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
