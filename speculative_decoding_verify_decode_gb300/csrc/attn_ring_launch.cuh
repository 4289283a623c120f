// Launch of the ring-buffered verify attention for one (NQ, window) instance,
// shared by the translation units that instantiate the kernel (full attention
// in attn_ring.cu, sliding window in attn_ring_win.cu).
#pragma once

#include "attn_ring_kernel.cuh"

namespace sdv {
namespace {

template <int NQ, bool WIN>
cudaError_t launch_ring_nq(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p, const BatchDesc& bd,
                           const TcPlan& pl, cudaStream_t st) {
  const size_t smem = Ring<NQ>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(attn_ring_kernel<NQ, WIN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_splits * kHkv * pl.hparts, bd.batch);
  cfg.blockDim = dim3(kRingThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_ring_kernel<NQ, WIN>, mk, mv, p, bd, pl.hpc, pl.hparts);
}

// Dispatch over the compiled query-column widths.
template <bool WIN>
cudaError_t launch_ring_kind(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p, const BatchDesc& bd,
                             const TcPlan& pl, cudaStream_t st) {
  switch (pl.nq) {
    case 32: return launch_ring_nq<32, WIN>(mk, mv, p, bd, pl, st);
    case 48: return launch_ring_nq<48, WIN>(mk, mv, p, bd, pl, st);
    case 64: return launch_ring_nq<64, WIN>(mk, mv, p, bd, pl, st);
    case 80: return launch_ring_nq<80, WIN>(mk, mv, p, bd, pl, st);
    case 96: return launch_ring_nq<96, WIN>(mk, mv, p, bd, pl, st);
    case 112: return launch_ring_nq<112, WIN>(mk, mv, p, bd, pl, st);
    case 128: return launch_ring_nq<128, WIN>(mk, mv, p, bd, pl, st);
    case 144: return launch_ring_nq<144, WIN>(mk, mv, p, bd, pl, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace sdv
