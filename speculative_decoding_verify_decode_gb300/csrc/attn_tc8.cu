// Host side of the split-KV verify attention on e4m3 (quantised) caches: the
// tensor map of the K codes (V pages move as plain bulk copies); the launch
// plan and the merge are those of the bf16 caches.  The kernel itself is in
// attn_tc_kernel.cuh.
#include "attn_tc_kernel.cuh"

namespace sdv {
namespace {

// The e4m3 K cache viewed as 3-D: x = code within a token row (256 bytes,
// contiguous), y = slot (256 B apart), z = page of one KV head (page * 4 +
// head, 4 KB apart).  A box of {128, 16, 1} is half of every row of one page:
// 2 KB, landing as 16 rows of 128 bytes.
bool code_map(CUtensorMap* map, const void* cache, int pool_pages) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)kPage, (cuuint64_t)pool_pages * kHkv};
  cuuint64_t strides[2] = {(cuuint64_t)kDim, (cuuint64_t)kDim * kPage};
  cuuint32_t box[3] = {128, (cuuint32_t)kPage, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(cache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_attn_tc8(const AttnParams& p, const BatchDesc& bd, cudaStream_t st) {
  CUtensorMap mk, unused;   // V pages move as plain bulk copies
  std::memset(&unused, 0, sizeof(unused));
  if (!code_map(&mk, p.k_cache8, p.num_pool_pages)) return cudaErrorInvalidValue;
  const cudaError_t e = launch_tc_kind<true>(mk, unused, p, bd, st);
  if (e != cudaSuccess || p.num_splits == 1) return e;
  return launch_attn_merge(p, bd, st);
}

}  // namespace sdv
