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

// Fast path (bf16, K = V = 128, C = 64): tcgen05 chunk-local kernel and
// mma.sync state recurrence.
bool tc_supported(const Problem& p);
size_t tc_workspace_bytes(const Problem& p);
gdr_status launch_tc(const Problem& p, void* ws_body, unsigned int* error_word,
                     cudaStream_t stream, int stage);

}  // namespace gdr
