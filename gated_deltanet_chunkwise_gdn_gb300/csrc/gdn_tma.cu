// gdn_tma.cu — host helpers: the driver's tensor-map encoder, fetched once through the
// runtime (no link-time dependency on libcuda), and the 3-D row-tile maps used by the kernels.
#include <cudaTypedefs.h>

#include <mutex>

#include "gdn_common.cuh"

namespace gdn {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return g_encode;
}

// Map over a [T, heads, D] array of 16-bit elements whose box is 64 consecutive elements of one head
// for `box_rows` consecutive tokens, 128-byte swizzled in shared memory (one 128-byte row
// per token). Coordinates are (element, head, token); tokens past T read as zero.
bool make_token_tile_map(CUtensorMap* map, const void* base, int D, int heads, int64_t T, int box_rows, bool fp16) {
  auto enc = encoder();
  if (!enc || T <= 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map over a row-major [rows, inner] array of 16-bit elements; the box is box_inner x box_rows elements,
// 128-byte swizzled in shared memory when swizzle128 (box_inner must then be 64), else
// stored densely (box_inner * 2 bytes per row).
bool make_2d_tile_map(CUtensorMap* map, const void* base, int inner, int64_t rows, int box_inner, int box_rows,
                      bool swizzle128, bool fp16) {
  auto enc = encoder();
  if (!enc || rows <= 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(map, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gdn
