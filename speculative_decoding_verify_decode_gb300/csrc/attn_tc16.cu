// Host side of the split-KV verify attention on bf16 caches when every
// context split holds a single 128-token tile (short contexts): tensor maps of
// the paged cache and the launch of attn_tc_kernel's bf16 instances followed by
// the log-sum-exp merge.  At one tile per CTA the layer is a latency chain
// (stage the operands, one tile, epilogue, merge), and this kernel's shorter
// chain and smaller register footprint (the merge blocks fit beside its CTAs,
// so the next kernel launches early) beat the ring kernel, whose deeper
// buffering only pays off over several tiles.  The kernel itself is in
// attn_tc_kernel.cuh.
#include "attn_tc_kernel.cuh"

namespace sdv {
namespace {

// The cache viewed as 4-D: x = dim within a 64-dim block (contiguous),
// y = slot within an 8-slot half page (512 B apart), z = 64-dim block (128 B
// apart), w = half page of one KV head ((page * 4 + head) * 2 + half, 4 KB
// apart), with the 128-byte swizzle.  A box of {64, 8, 4, 2} is one page of
// one head (8 KB), landing as two 8-row groups of the group-major K/V tile.
bool bf16_page_map(CUtensorMap* map, const void* cache, int pool_pages) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {64, 8, 4, (cuuint64_t)pool_pages * kHkv * 2};
  cuuint64_t strides[3] = {(cuuint64_t)kDim * 2, 128, (cuuint64_t)kDim * 2 * 8};
  cuuint32_t box[4] = {64, 8, 4, 2};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(cache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_attn_tc16(const AttnParams& p, const BatchDesc& bd, cudaStream_t st) {
  CUtensorMap mk, mv;
  if (!bf16_page_map(&mk, p.k_cache, p.num_pool_pages) || !bf16_page_map(&mv, p.v_cache, p.num_pool_pages))
    return cudaErrorInvalidValue;
  const cudaError_t e = launch_tc_kind<false>(mk, mv, p, bd, st);
  if (e != cudaSuccess || p.num_splits == 1) return e;
  return launch_attn_merge(p, bd, st);
}

}  // namespace sdv
