// Host side of the split-KV verify attention on e4m3 (quantised) caches: the
// pages are read by the kernel's converter warps with plain loads, so no
// tensor map is made; the launch plan and the merge are those of the bf16
// caches.  The kernel itself is in attn_tc_kernel.cuh.
#include "attn_tc_kernel.cuh"

namespace sdv {

cudaError_t launch_attn_tc8(const AttnParams& p, const BatchDesc& bd, cudaStream_t st) {
  CUtensorMap unused;   // the converter warps need no tensor map
  std::memset(&unused, 0, sizeof(unused));
  const cudaError_t e = launch_tc_kind<true>(unused, unused, p, bd, st);
  if (e != cudaSuccess || p.num_splits == 1) return e;
  return launch_attn_merge(p, bd, st);
}

}  // namespace sdv
