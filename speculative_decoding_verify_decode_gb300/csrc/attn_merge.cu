// Log-sum-exp merge of split-KV partial attention outputs.
//
// Every split of a sequence wrote its normalised partial output o_s (bf16)
// and its base-2 log-sum-exp lse_s.  With M = max_s lse_s the merged result
// is o = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M) and
// lse = M + log2 sum_s 2^(lse_s - M) (reported in natural log).  Sequences
// served by a single split were written directly by the split kernel.
#include "common.cuh"
#include "kernels.h"

namespace sdv {
namespace {

__device__ __forceinline__ float2 unpack_bf16(uint32_t v) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// One 256-thread block per (node row, query head): eight warps each take every
// eighth split, lane t owning dims 8t..8t+7 (16 bytes of each partial row).  A
// thread issues the loads of up to kBatch of its splits before it uses any
// (one round of memory latency for up to 8 * kBatch = 40 splits) and keeps its
// warp's running (max, sum, weighted sum) in base 2; the eight warps are
// combined once, through shared memory.  The blocks are launched while the
// split kernel runs and become resident as its CTAs exit.
constexpr int kMergeThreads = 256;
constexpr int kMergeGroups = kMergeThreads / 32;
constexpr int kBatch = 5;

__device__ __forceinline__ void add_weighted(float (&acc)[8], float wk, const uint4& o) {
  const float2 a = unpack_bf16(o.x), b = unpack_bf16(o.y), c = unpack_bf16(o.z), d = unpack_bf16(o.w);
  acc[0] += wk * a.x; acc[1] += wk * a.y; acc[2] += wk * b.x; acc[3] += wk * b.y;
  acc[4] += wk * c.x; acc[5] += wk * c.y; acc[6] += wk * d.x; acc[7] += wk * d.y;
}

__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const AttnParams p, const BatchDesc bd) {
  // The next kernel in the stream (the next layer's split kernel) may be
  // scheduled at once; it waits for this grid before it reads what this grid
  // writes, and may load context tiles meanwhile.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int pair = blockIdx.x;
  const int r = pair / kHq, head = pair % kHq;
  int lo = 0, hi = bd.batch - 1;   // sequence of node row r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (bd.q_indptr[mid] <= r) lo = mid; else hi = mid - 1;
  }
  int L = p.ctx_lens[lo];
  L = L < 0 ? 0 : min(L, p.max_pages * kPage);
  const int ns = active_splits(L, p.window, kTileTokens, p.chunk);
  // The partials are written by the split kernel launched just before.  Every
  // block waits for it, even one with nothing to merge, so that this grid
  // finishes only after the split kernel: a dependent that waits for this grid
  // then also sees the outputs the split kernel wrote directly.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (ns == 1) return;  // written directly by the split kernel
  const size_t stride = (size_t)bd.total_nodes * kHq;   // rows between splits
  const size_t row0 = (size_t)r * kHq + head;
  __shared__ float4 s_acc[kMergeGroups][2][32];
  __shared__ float s_max[kMergeGroups], s_den[kMergeGroups];
  const int grp = threadIdx.x >> 5, t = threadIdx.x & 31;
  float mx = -INFINITY, den = 0.f;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int base = 0; base < ns; base += kBatch * kMergeGroups) {
    float w[kBatch];
    uint4 o[kBatch];   // 8 bf16
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int s = base + grp + k * kMergeGroups;
      const size_t row = (size_t)min(s, ns - 1) * stride + row0;
      w[k] = s < ns ? p.lse_part[row] : -INFINITY;
      o[k] = reinterpret_cast<const uint4*>(p.o_part + row * kDim)[t];
    }
    float bm = mx;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) bm = fmaxf(bm, w[k]);
    if (bm > mx) {   // rescale what this warp has so far to the new maximum
      const float a = mx == -INFINITY ? 0.f : fast_exp2(mx - bm);
      den *= a;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] *= a;
      mx = bm;
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const float wk = w[k] == -INFINITY ? 0.f : fast_exp2(w[k] - mx);   // padding entries weigh 0
      den += wk;
      add_weighted(acc, wk, o[k]);
    }
  }
  s_acc[grp][0][t] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  s_acc[grp][1][t] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  if (t == 0) { s_max[grp] = mx; s_den[grp] = den; }
  __syncthreads();
  if (grp > 0) return;
  float m_all = s_max[0];
#pragma unroll
  for (int k = 1; k < kMergeGroups; ++k) m_all = fmaxf(m_all, s_max[k]);
  float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float d_all = 0.f;
#pragma unroll
  for (int k = 0; k < kMergeGroups; ++k) {
    const float a = s_max[k] == -INFINITY ? 0.f : fast_exp2(s_max[k] - m_all);   // a warp may hold no split
    const float4 v0 = s_acc[k][0][t], v1 = s_acc[k][1][t];
    d_all += a * s_den[k];
    sum[0] += a * v0.x; sum[1] += a * v0.y; sum[2] += a * v0.z; sum[3] += a * v0.w;
    sum[4] += a * v1.x; sum[5] += a * v1.y; sum[6] += a * v1.z; sum[7] += a * v1.w;
  }
  const float inv = 1.f / d_all;
  uint4 packed;
  packed.x = pack_bf16(sum[0] * inv, sum[1] * inv);
  packed.y = pack_bf16(sum[2] * inv, sum[3] * inv);
  packed.z = pack_bf16(sum[4] * inv, sum[5] * inv);
  packed.w = pack_bf16(sum[6] * inv, sum[7] * inv);
  reinterpret_cast<uint4*>(p.out + row0 * kDim)[t] = packed;
  if (p.lse != nullptr && t == 0) p.lse[row0] = (m_all + fast_log2(d_all)) * kLn2;
}

}  // namespace

// Launched as a programmatic dependent of the split kernel: its blocks may be
// scheduled while the split kernel runs and wait (griddepcontrol.wait) for
// that kernel's completion before they read the partials.  It lets its own
// dependents be scheduled at once (see the kernel).
cudaError_t launch_attn_merge(const AttnParams& p, const BatchDesc& bd, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(bd.total_nodes * kHq);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_merge_kernel, p, bd);
}

}  // namespace sdv
