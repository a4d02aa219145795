// gdr_tmap.cu -- TMA tensor-map encoding (driver entry point fetched once).
#include "gdr_tmap.cuh"

#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace gdr {
namespace fast {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

}  // namespace

bool tmap_encode(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base,
                 const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                 CUtensorMapSwizzle swz) {
  auto enc = encoder();
  if (!enc) return false;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(map, type, rank, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tmap_bthd(CUtensorMap* map, const void* base, int B, int T, int heads) {
  const cuuint64_t dims[4] = {128, (cuuint64_t)heads, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {128 * 2, (cuuint64_t)heads * 128 * 2,
                                 (cuuint64_t)T * heads * 128 * 2};
  const cuuint32_t box[4] = {64, 1, 64, 1};
  return tmap_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

bool tmap_blocks(CUtensorMap* map, const void* base, CUtensorMapDataType type, int esize,
                 int cols, int rows, size_t count, size_t block_bytes, int box_cols, int box_rows,
                 CUtensorMapSwizzle swz) {
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)count};
  const cuuint64_t strides[2] = {(cuuint64_t)cols * esize, (cuuint64_t)block_bytes};
  const cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
  return tmap_encode(map, type, 3, base, dims, strides, box, swz);
}

}  // namespace fast
}  // namespace gdr
