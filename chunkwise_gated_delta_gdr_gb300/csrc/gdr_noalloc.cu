// gdr_noalloc.cu -- the forward pass with library-owned scratch.
//
// gdr_chunk_fwd needs a caller-provided workspace. Some callers cannot
// provide one: code running under an allocator that is not the CUDA one (or
// none at all), plugins that must not touch the device heap, or a caller that
// sits inside a region where cudaMalloc is forbidden (it synchronises the
// device and is not allowed while another stream is being captured). For them
// this file owns a fixed scratch buffer in device global memory, declared as a
// file-scope __device__ array, and gdr_chunk_fwd_noalloc runs the usual
// forward pass on it. Nothing here calls cudaMalloc, cudaFree or any allocating
// library routine.
//
// The array exists once per device that loads this library and stays
// allocated until the process exits. Its size is GDR_NOALLOC_SCRATCH_BYTES.
#include <mutex>

#include "gdr_internal.cuh"

namespace gdr {
namespace {

constexpr size_t kScratchBytes = GDR_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

// The scratch buffer itself. Host code must not use this name as an address:
// on the host it denotes a stand-in object, so the device address is looked up
// with cudaGetSymbolAddress (below) and cached per device.
__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 256;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device. Outside stream capture
// it is looked up again on every call (cheap), so a cudaDeviceReset, after
// which the module and the array may come back at another address, leaves no
// stale pointer behind; while `stream` is being captured the address cached by
// an earlier call on this device is used.
gdr_status scratch_address(cudaStream_t stream, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDR_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GDR_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    cs = cudaStreamCaptureStatusActive;     // unknown: do not touch the module
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (cs == cudaStreamCaptureStatusNone || !g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr) {
      (void)cudaGetLastError();
      return GDR_ERR_CUDA;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return GDR_OK;
}

}  // namespace
}  // namespace gdr

extern "C" gdr_status gdr_chunk_fwd_noalloc(const void* q, const void* k, const void* v,
                                            const float* g, const float* beta,
                                            const float* initial_state, int chunk_size,
                                            float scale, int use_qk_l2norm, int gate_mode,
                                            void* out, float* final_state, const gdr_dims* dims,
                                            gdr_stream_t stream) {
  if (!dims) return GDR_ERR_INVALID_ARG;
  const size_t need = gdr_chunk_fwd_workspace_size(dims, chunk_size, gate_mode);
  if (need > gdr::kScratchBytes) return GDR_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    const gdr_status st = gdr::scratch_address(reinterpret_cast<cudaStream_t>(stream), &scratch);
    if (st != GDR_OK) return st;
  }
  // need == 0 means the sizes are invalid or unsupported: gdr_chunk_fwd then
  // reports why, before touching any workspace.
  return gdr_chunk_fwd(q, k, v, g, beta, initial_state, chunk_size, scale, use_qk_l2norm,
                       gate_mode, out, final_state, dims, scratch, scratch ? gdr::kScratchBytes : 0,
                       stream);
}

// The scratch array starts with the workspace header, whose error word the
// kernels set when a bounded wait gives up: read it the way gdr_stream_status
// reads a caller's workspace.
extern "C" gdr_status gdr_noalloc_stream_status(gdr_stream_t stream) {
  void* scratch = nullptr;
  const gdr_status st = gdr::scratch_address(reinterpret_cast<cudaStream_t>(stream), &scratch);
  if (st != GDR_OK) return st;
  return gdr_stream_status(stream, scratch);
}
