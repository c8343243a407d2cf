// Host side of TMA: tensor-map encoding through the driver entry point
// (no link-time dependency on libcuda).
#include <cudaTypedefs.h>
#include <mutex>

#include "wa_internal.cuh"

namespace wa {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

void resolve() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  else
    cudaGetLastError();
}
}  // namespace

wa_status make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                            uint64_t row_stride, uint32_t box_cols, uint32_t box_rows) {
  std::call_once(g_once, resolve);
  if (!g_encode) return WA_ERR_CUDA;
  if (!aligned16(base) || (row_stride * 2) % 16 != 0 || box_cols * 2 > 128 || rows == 0)
    return WA_ERR_ALIGN;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_stride * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? WA_OK : WA_ERR_CUDA;
}

wa_status make_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1,
                            uint64_t d2, uint64_t s1, uint64_t s2, uint32_t box0, uint32_t box1) {
  std::call_once(g_once, resolve);
  if (!g_encode) return WA_ERR_CUDA;
  if (!aligned16(base) || (s1 * 2) % 16 != 0 || (s2 * 2) % 16 != 0 || box0 * 2 > 128 || d1 == 0)
    return WA_ERR_ALIGN;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1 * 2, s2 * 2};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? WA_OK : WA_ERR_CUDA;
}

}  // namespace wa
