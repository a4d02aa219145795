// gdr_internal.cuh -- shared host-side declarations of the CUDA library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include "gdr.h"

namespace gdr {

// One validated call of the forward pass.
struct Problem {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* s0;       // may be null (zero state)
  void* out;
  float* sT;             // may be null (not written)
  int B, T, H, HV, K, V, C;
  int N;                 // chunks per sequence, ceil(T / C)
  int in_bf16, out_bf16, gate_mode, use_l2;
  float scale;
  int ssd = 0;           // Mamba2 SSD update: no delta erase, no beta (general path only)
  int zero_u = 0;        // recurrence reads U as zero: S <- (gamma - KB^T W) S, the linear
                         // part of the chunk map (segmented scan)
  int recur_mode = 0;    // 0: states and outputs; 1: states only where the outputs are a
                         // separate pass (the fused recurrence), else both; 2: that
                         // separate output pass after a mode-1 launch (else nothing)
};

// Workspace header: first 256 bytes of every workspace.
struct WorkspaceHeader {
  unsigned int error_word;  // nonzero: a bounded device wait gave up (code in low bits)
  unsigned int reserved[63];
};
static_assert(sizeof(WorkspaceHeader) == 256, "header must stay 256 bytes");

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

// General fp32 CUDA-core path (any supported shape). stage: 1 = chunk-local
// kernel, 2 = state recurrence, 3 = both.
size_t general_workspace_bytes(const Problem& p);
gdr_status launch_general(const Problem& p, void* ws_body, cudaStream_t stream, int stage);

// Fast path (bf16, K = V = 128, C = 64): chunk-local stage and state
// recurrence on tcgen05 (the per-key gate's chunk-local stage on mma.sync).
bool tc_supported(const Problem& p);
size_t tc_workspace_bytes(const Problem& p);
gdr_status launch_tc(const Problem& p, void* ws_body, unsigned int* error_word,
                     cudaStream_t stream, int stage);
// Whether gdr_chunk_fwd takes the one-launch form of the fast path (scalar
// gate) for this problem on the current device.
bool tc_one_launch(const Problem& p);
// Bound (polls) of the one-launch forward's waits on chunk flags, for calls
// enqueued from now on (polls < 0: unchanged); returns the previous bound.
long long set_wait_limit(long long polls);

// Segmented scan helpers (gdr_segment.cu): n identity K x K states; the serial
// combine S_{p+1} = A_p S_p + B_p over the P segments of each (b, hv).
gdr_status launch_segment_identity(float* A, long n, int K, cudaStream_t stream);
gdr_status launch_segment_combine(const float* A, const float* Bst, const float* s0, float* Sin,
                                  float* sT, int B, int P, int HV, int K, cudaStream_t stream);

}  // namespace gdr
