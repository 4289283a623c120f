// Host side of the split-KV verify attention on e4m3 (quantised) caches: the
// tensor map of the K codes (V pages move as plain bulk copies), the
// query-column plan of this kernel, and the launch followed by the merge.  The
// kernel itself is in attn_tc_kernel.cuh.
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

cudaError_t launch_attn_tc8(const AttnParams& p, const BatchDesc& bd, cudaStream_t st) {
  CUtensorMap mk, unused;   // V pages move as plain bulk copies
  std::memset(&unused, 0, sizeof(unused));
  if (!code_map(&mk, p.k_cache8, p.num_pool_pages)) return cudaErrorInvalidValue;
  const cudaError_t e = launch_tc_kind<true>(mk, unused, p, bd, st);
  if (e != cudaSuccess || p.num_splits == 1) return e;
  return launch_attn_merge(p, bd, st);
}

}  // namespace sdv
