// gdr_tc.cu -- tcgen05 tensor-core path (bf16, K = V = 128, C = 64).
#include "gdr_internal.cuh"

namespace gdr {

bool tc_supported(const Problem&) { return false; }
size_t tc_workspace_bytes(const Problem&) { return 0; }
gdr_status launch_tc(const Problem&, void*, unsigned int*, cudaStream_t) {
  return GDR_ERR_UNSUPPORTED;
}

}  // namespace gdr
