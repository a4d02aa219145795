// gdr_fast.cuh -- shared definitions of the fast path (bf16, K = V = 128, C = 64).
//
// The fast path runs two kernels:
//   1. a chunk-local kernel (one CTA per chunk) writes, per chunk, the operands
//      of the inter-chunk recurrence into a workspace slab: gdr_chunk_tc.cu
//      (tcgen05, scalar gate) or gdr_chunk_kda.cu (mma.sync, per-key gate);
//   2. a recurrence kernel runs the chunks in order per (batch, value head,
//      V tile): gdr_recur.cu (scalar gate; mma.sync chains plus tcgen05 output
//      CTAs, fallback gdr_state.cu) or gdr_state_kda.cu (per-key gate, tcgen05).
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
constexpr int VT = 16;   // value columns per state CTA

// Slab of one chunk (b, hv, n), chunk index ((b * HV + hv) * N + n). All
// offsets in bytes from the slab start; every array is 16-byte aligned.
//   W2   [2][C][K] bf16  hi / lo of -W, W = M^-1 (exp(G) k_hat)
//   AQ2  [2][C][C] bf16  hi / lo of A_qk (beta on its columns, zero above the diagonal)
//   U    [C][V]    fp32  U = M^-1 v
//   VEC  qscale[C], kscale[C], gamma[K] fp32
//        scalar gate: qscale_i = scale |q_i|^-1 exp(G_i), kscale_j = beta_j |k_j|^-1
//        exp(G_last - G_j), gamma = exp(G_last) on every channel;
//        per-key gate: qscale = kscale = 1, gamma_c = exp(G_last,c)
//   QB2  [2][C][K] bf16  per-key gate only: hi / lo of scale q_hat exp(G)
//   KB2  [2][C][K] bf16  per-key gate only: hi / lo of beta k_hat exp(G_last - G)
// For the scalar gate the state kernel reads raw q and k from the inputs
// (exact in bf16) and applies qscale / kscale as fp32 row factors.
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

// Exchange block of one chunk (scalar gate): the state at the chunk start and
// the chunk's corrected values, published by the state chain for the output
// stage, as bf16 hi / lo planes, value-major (the layout the output products
// read as their K-major B operands).
//   S_HI, S_LO  [V][K] bf16   S^T at the start of the chunk
//   R_HI, R_LO  [V][C] bf16   r^T = (U - W S)^T
struct Xchg {
  static constexpr size_t S_HI = 0;
  static constexpr size_t S_LO = S_HI + (size_t)V * K * 2;
  static constexpr size_t R_HI = S_LO + (size_t)V * K * 2;
  static constexpr size_t R_LO = R_HI + (size_t)V * C * 2;
  static constexpr size_t BYTES = R_LO + (size_t)V * C * 2;
};

// Everything both kernels of the fast path need.
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
  unsigned int* flags;      // [B * HV][V / VT] chunks published per chain (scalar gate)
  unsigned int* error_word;
  int B, T, H, HV, N;
  int out_bf16, gate_mode, use_l2;
  int ssd;                  // Mamba2 SSD update: no delta erase (W = 0), beta = 1
  // Both stages in one call: the chunk kernel zeroes the chains' progress flags
  // (read only by the recurrence, which runs after it), so the recurrence
  // launch needs no separate reset.
  int zero_flags;
  int zero_u;               // recurrence reads U as zero (the chunk map's linear part)
  int recur_mode;           // 0 chains + outputs; 1 chains only; 2 outputs only (gdr_internal.cuh)
  float scale;
  size_t slab_bytes;
};

inline __host__ __device__ size_t slab_index(const Params& p, int b, int hv, int n) {
  return ((size_t)b * p.HV + hv) * p.N + n;
}

// Launchers (gdr_state.cu, gdr_chunk.cu).
gdr_status launch_state(const Params& p, cudaStream_t stream);
// Scalar gate: state chain and chunk outputs in one launch (gdr_recur.cu).
gdr_status launch_recur(const Params& p, cudaStream_t stream);
// Per-key gate: the recurrence on tcgen05, 64 value columns per CTA (gdr_state_kda.cu).
gdr_status launch_state_kda_tc(const Params& p, cudaStream_t stream);
// Per-key gate: chunk-local kernel on mma.sync (gdr_chunk_kda.cu).
gdr_status launch_chunk_kda(const Params& p, cudaStream_t stream);
gdr_status launch_chunk_tc(const Params& p, cudaStream_t stream);

}  // namespace fast
}  // namespace gdr
