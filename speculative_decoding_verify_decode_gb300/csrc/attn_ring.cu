// Host side of the split-KV verify attention on bf16 caches: tensor maps of
// the paged cache, the query-column plan, and the launch of the ring-buffered
// kernel (attn_ring_kernel.cuh) followed by the log-sum-exp merge.
#include "attn_ring_launch.cuh"

namespace sdv {
namespace {

// The driver's tensor-map encoder, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 ring_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

}  // namespace

// The cache viewed as 4-D: x = dim within a 64-dim block (contiguous),
// y = slot within an 8-slot half page (512 B apart), z = 64-dim block (128 B
// apart), w = half page of one KV head ((page * 4 + head) * 2 + half, 4 KB
// apart), with the 128-byte swizzle.  A box of {64, 8, 4, 2} is one page of
// one head (8 contiguous KB), landing as [half][block][8 slots][128 B]: two
// 8-row groups of the group-major K tile or of a V page slot (both bf16 kernels).
bool bf16_page_map(CUtensorMap* map, const void* cache, int pool_pages) {
  auto fn = ring_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[4] = {64, 8, 4, (cuuint64_t)pool_pages * kHkv * 2};
  cuuint64_t strides[3] = {(cuuint64_t)kDim * 2, 128, (cuuint64_t)kDim * 2 * 8};
  cuuint32_t box[4] = {64, 8, 4, 2};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(cache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

TcPlan ring_plan(int max_nodes) {
  TcPlan pl;
  const int opts[4] = {6, 3, 2, 1};
  pl.hpc = 1;
  for (int h : opts) {
    if (h * max_nodes <= kRingMaxNQ) { pl.hpc = h; break; }
  }
  pl.hparts = (kGroup + pl.hpc - 1) / pl.hpc;
  pl.nq = (pl.hpc * max_nodes + 15) / 16 * 16;
  if (pl.nq < 32) pl.nq = 32;
  return pl;
}

cudaError_t launch_attn_ring(const AttnParams& p, const BatchDesc& bd, cudaStream_t st) {
  CUtensorMap mk, mv;
  if (!bf16_page_map(&mk, p.k_cache, p.num_pool_pages) || !bf16_page_map(&mv, p.v_cache, p.num_pool_pages))
    return cudaErrorInvalidValue;
  const TcPlan pl = ring_plan(bd.max_nodes);
  const cudaError_t e = p.window > 0 ? launch_ring_window(mk, mv, p, bd, pl, st)
                                     : launch_ring_kind<false>(mk, mv, p, bd, pl, st);
  if (e != cudaSuccess || p.num_splits == 1) return e;
  return launch_attn_merge(p, bd, st);
}

}  // namespace sdv
