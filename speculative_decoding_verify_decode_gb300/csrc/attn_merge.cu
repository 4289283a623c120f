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

// One 64-thread block per (node row, query head).  Thread t owns dims
// 4t..4t+3; the split weights come from a block-wide max of the split LSEs.
constexpr int kMergeThreads = 64;

__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const AttnParams p, const BatchDesc bd) {
  const int pair = blockIdx.x;
  const int r = pair / kHq, head = pair % kHq;
  int b = 0;
  while (b + 1 < bd.batch && bd.q_indptr[b + 1] <= r) ++b;
  int L = p.ctx_lens[b];
  L = L < 0 ? 0 : min(L, p.max_pages * kPage);
  const int ns = active_splits(L, p.chunk);
  if (ns == 1) return;  // written directly by the split kernel
  const size_t stride = (size_t)bd.total_nodes * kHq;   // rows between splits
  const size_t row0 = (size_t)r * kHq + head;
  __shared__ float s_red[kMergeThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float mx = -INFINITY;
  for (int s = tid; s < ns; s += kMergeThreads) mx = fmaxf(mx, p.lse_part[s * stride + row0]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) s_red[warp] = mx;
  __syncthreads();
  mx = fmaxf(s_red[0], s_red[1]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  int s = 0;
  for (; s + 4 <= ns; s += 4) {
    float w[4];
    float4 o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const size_t row = (s + k) * stride + row0;
      w[k] = p.lse_part[row];
      o[k] = reinterpret_cast<const float4*>(p.o_part + row * kDim)[tid];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float wk = fast_exp2(w[k] - mx);
      den += wk;
      acc.x += wk * o[k].x; acc.y += wk * o[k].y; acc.z += wk * o[k].z; acc.w += wk * o[k].w;
    }
  }
  for (; s < ns; ++s) {
    const size_t row = s * stride + row0;
    const float wk = fast_exp2(p.lse_part[row] - mx);
    const float4 o = reinterpret_cast<const float4*>(p.o_part + row * kDim)[tid];
    den += wk;
    acc.x += wk * o.x; acc.y += wk * o.y; acc.z += wk * o.z; acc.w += wk * o.w;
  }
  const float inv = 1.f / den;
  uint2 packed;
  packed.x = pack_bf16(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2*>(p.out + row0 * kDim)[tid] = packed;
  if (p.lse != nullptr && tid == 0) p.lse[row0] = (mx + fast_log2(den)) * kLn2;
}

}  // namespace

cudaError_t launch_attn_merge(const AttnParams& p, const BatchDesc& bd, cudaStream_t st) {
  attn_merge_kernel<<<bd.total_nodes * kHq, kMergeThreads, 0, st>>>(p, bd);
  return cudaGetLastError();
}

}  // namespace sdv
