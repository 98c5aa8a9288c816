// Host-side tensor-map encoding for the TMA loads (the driver entry point is looked up through
// the runtime, so the library needs no link against libcuda).
#include <cudaTypedefs.h>
#include <mutex>

#include "psk_common.cuh"

namespace psk {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

bool resolve() {
  std::call_once(g_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}
}  // namespace

bool encode_cache_map(CUtensorMap *map, const void *base, int dtype, int D, int H, long long rows, int box_rows,
                      bool sw128) {
  if (!resolve()) return false;
  const int es = dtype == PSK_F32 ? 4 : 2;
  const int box_d = sw128 ? 128 / es : D;
  if (box_d > D || D % box_d != 0) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)H * D * es};
  const cuuint32_t box[3] = {(cuuint32_t)box_d, 1u, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = g_encode(map, dtype == PSK_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_matrix_map_sw128(CUtensorMap *map, const void *base, long long cols, long long rows, int box_cols,
                             int box_rows) {
  if (!resolve() || box_cols * 2 != 128) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace psk
