// The sliding-window instances of the ring-buffered verify attention (their own
// translation unit, so that they compile beside the full-attention ones).
#include "attn_ring_launch.cuh"

namespace sdv {

cudaError_t launch_ring_window(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p, const BatchDesc& bd,
                               const TcPlan& pl, cudaStream_t st) {
  return launch_ring_kind<true>(mk, mv, p, bd, pl, st);
}

}  // namespace sdv
