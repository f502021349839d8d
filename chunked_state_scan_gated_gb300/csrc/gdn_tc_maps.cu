// gdn_tc_maps.cu -- TMA tensor maps of the tensor-core path and its selector.
//
// Tensor maps describe the token-major inputs [B, T_stride, heads, 128] (bf16)
// to the TMA unit: one box is 64 tokens x 64 columns of one head, landing in
// shared memory as a 128-byte-swizzled K-major tile (the layout the tcgen05
// descriptors of gdn_tc_common.cuh expect).  The chunk size and head dim are
// the fused backend's shape of the "Linear Attention CP 融合算子 PR #1114
// 测试报告", section 3.1.
#include <cuda.h>
#include <cuda_bf16.h>
#include <mutex>

#include "gdn_internal.h"

namespace gdn {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  });
  return fn;
}

// [B, Ts, heads, 128] bf16 tensor, boxes of 64 tokens x 64 columns of one head.
bool make_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t Ts, int64_t heads) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {128, (cuuint64_t)heads, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {256, (cuuint64_t)(heads * 256), (cuuint64_t)(Ts * heads * 256)};
  cuuint32_t box[4] = {64, 1, 64, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_make_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t Ts, int64_t heads) {
  return make_map(m, ptr, B, T, Ts, heads);
}

// The same tensor, boxes of `rows` tokens x the whole 128-column head, unswizzled (rows of
// 256 bytes): the K - 1 tokens before a chunk that the Conv1D reads.
bool tc_make_map_rows(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t Ts,
                      int64_t heads, int rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rows < 1 || rows > 256) return false;
  cuuint64_t dims[4] = {128, (cuuint64_t)heads, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {256, (cuuint64_t)(heads * 256), (cuuint64_t)(Ts * heads * 256)};
  cuuint32_t box[4] = {128, 1, (cuuint32_t)rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_path(const Prob& pr) {
  return pr.dtype == GDN_BF16 && pr.dk == 128 && pr.dv == 128 && pr.B > 0 && pr.NC > 0;
}

}  // namespace gdn
