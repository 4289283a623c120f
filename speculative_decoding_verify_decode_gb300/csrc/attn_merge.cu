// Log-sum-exp merge of split-KV partial attention outputs.
//
// Every split of a sequence wrote its normalised partial output o_s (fp32)
// and its base-2 log-sum-exp lse_s.  With M = max_s lse_s the merged result
// is o = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M) and
// lse = M + log2 sum_s 2^(lse_s - M) (reported in natural log).  Sequences
// served by a single split were written directly by the split kernel.
#include "common.cuh"
#include "kernels.h"

namespace sdv {
namespace {

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// One warp per (node row, query head): combine the active splits.
__global__ void __launch_bounds__(256) attn_merge_kernel(const AttnParams p, const BatchDesc bd) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x * 8 + warp;
  if (pair >= bd.total_nodes * kHq) return;
  const int r = pair / kHq, head = pair % kHq;
  int b = 0;
  while (b + 1 < bd.batch && bd.q_indptr[b + 1] <= r) ++b;
  int L = p.ctx_lens[b];
  L = L < 0 ? 0 : min(L, p.max_pages * kPage);
  const int ns = active_splits(L, p.chunk);
  if (ns == 1) return;  // written directly by the split kernel
  float mx = -INFINITY;
  for (int s = 0; s < ns; ++s) mx = fmaxf(mx, p.lse_part[((size_t)s * bd.total_nodes + r) * kHq + head]);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float den = 0.f;
  for (int s = 0; s < ns; ++s) {
    const size_t row = ((size_t)s * bd.total_nodes + r) * kHq + head;
    const float w = fast_exp2(p.lse_part[row] - mx);
    den += w;
    const float4* src = reinterpret_cast<const float4*>(p.o_part + row * kDim + lane * 8);
    const float4 a = src[0], c = src[1];
    acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
    acc[4] += w * c.x; acc[5] += w * c.y; acc[6] += w * c.z; acc[7] += w * c.w;
  }
  const float inv = 1.f / den;
  __nv_bfloat16* dst = p.out + ((size_t)r * kHq + head) * kDim + lane * 8;
  uint4 packed;
  packed.x = pack_bf16(acc[0] * inv, acc[1] * inv);
  packed.y = pack_bf16(acc[2] * inv, acc[3] * inv);
  packed.z = pack_bf16(acc[4] * inv, acc[5] * inv);
  packed.w = pack_bf16(acc[6] * inv, acc[7] * inv);
  *reinterpret_cast<uint4*>(dst) = packed;
  if (p.lse != nullptr && lane == 0) p.lse[(size_t)r * kHq + head] = (mx + fast_log2(den)) * kLn2;
}

}  // namespace

cudaError_t launch_attn_merge(const AttnParams& p, const BatchDesc& bd, cudaStream_t st) {
  const int pairs = bd.total_nodes * kHq;
  attn_merge_kernel<<<(pairs + 7) / 8, 256, 0, st>>>(p, bd);
  return cudaGetLastError();
}

}  // namespace sdv
