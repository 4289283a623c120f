// Host side of the split-KV verify attention on bf16 caches: tensor maps of
// the paged cache, the launch plan, and the dispatch over the compiled
// query-column widths.  The kernel itself is in attn_tc_kernel.cuh.
#include "attn_tc_kernel.cuh"

namespace sdv {
namespace {

// ---------------------------------------------------------------- host side

// The cache viewed as 4-D: x = dim within a 64-dim block (contiguous),
// y = slot within an 8-slot half page (512 B apart), z = 64-dim block (128 B
// apart), w = half page of one KV head ((page * 4 + head) * 2 + half, 4 KB
// apart).  A box of {64, 8, 4, 2} is one page of one head (8 KB) and lands
// as [half][block][8 slots][128 B] with the 128-byte swizzle: two 8-row
// groups of the group-major K/V tile.
bool cache_map(CUtensorMap* map, const void* cache, int pool_pages) {
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

size_t tc_smem_bytes(int nq) {
  // the P^T tile always spans two 64-column atoms: the PV product takes its 128 rows as M
  return (size_t)nq * 512 + 2 * (size_t)kTileB + 2 * (size_t)kAtomB + sizeof(Small);
}

TcPlan tc_plan(int max_nodes) {
  TcPlan pl;
  const int opts[4] = {6, 3, 2, 1};
  pl.hpc = 1;
  for (int h : opts) {
    if (h * max_nodes <= kTcMaxNQ) { pl.hpc = h; break; }
  }
  pl.hparts = (kGroup + pl.hpc - 1) / pl.hpc;
  pl.nq = (pl.hpc * max_nodes + 15) / 16 * 16;
  if (pl.nq < 32) pl.nq = 32;
  return pl;
}

int attn_tc_tile() { return kT; }

cudaError_t launch_attn_tc(const AttnParams& p, const BatchDesc& bd, cudaStream_t st) {
  CUtensorMap mk, mv;
  if (!cache_map(&mk, p.k_cache, p.num_pool_pages) || !cache_map(&mv, p.v_cache, p.num_pool_pages))
    return cudaErrorInvalidValue;
  const cudaError_t e = launch_tc_kind<false>(mk, mv, p, bd, st);
  if (e != cudaSuccess || p.num_splits == 1) return e;
  return launch_attn_merge(p, bd, st);
}

}  // namespace sdv
