// Host side of the split-KV verify attention on bf16 caches when every
// context split holds a single 128-token tile (short contexts): the launch of
// attn_tc_kernel's bf16 instances (through the page map the ring kernel uses)
// followed by the log-sum-exp merge.  At one tile per CTA the layer is a
// latency chain (stage the operands, one tile, epilogue, merge), and this
// kernel's shorter chain and smaller register footprint (the merge blocks fit
// beside its CTAs, so the next kernel launches early) beat the ring kernel,
// whose deeper buffering only pays off over several tiles.  The kernel itself
// is in attn_tc_kernel.cuh.
#include "attn_tc_kernel.cuh"

namespace sdv {

cudaError_t launch_attn_tc16(const AttnParams& p, const BatchDesc& bd, cudaStream_t st) {
  CUtensorMap mk, mv;
  if (!bf16_page_map(&mk, p.k_cache, p.num_pool_pages) || !bf16_page_map(&mv, p.v_cache, p.num_pool_pages))
    return cudaErrorInvalidValue;
  const cudaError_t e = launch_tc_kind<false>(mk, mv, p, bd, st);
  if (e != cudaSuccess || p.num_splits == 1) return e;
  return launch_attn_merge(p, bd, st);
}

}  // namespace sdv
