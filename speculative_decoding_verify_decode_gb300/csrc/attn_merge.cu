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

// One 256-thread block per (node row, query head): four groups of 64
// threads each take every fourth split, thread t of a group owning dims
// 4t..4t+3 (8 bytes of each partial row).  A thread issues the loads of up to kBatch of its splits before
// it uses any (one round of memory latency for up to 4 * kBatch splits); the
// groups' sums are added in shared memory.  The split weights use the
// block-wide maximum of the split LSEs.
constexpr int kMergeThreads = 256;
constexpr int kMergeGroups = kMergeThreads / 64;
constexpr int kBatch = 12;

__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const AttnParams p, const BatchDesc bd) {
  const int pair = blockIdx.x;
  const int r = pair / kHq, head = pair % kHq;
  int lo = 0, hi = bd.batch - 1;   // sequence of node row r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (bd.q_indptr[mid] <= r) lo = mid; else hi = mid - 1;
  }
  int L = p.ctx_lens[lo];
  L = L < 0 ? 0 : min(L, p.max_pages * kPage);
  const int ns = active_splits(L, p.chunk);
  if (ns == 1) return;  // written directly by the split kernel
  // the partials are written by the split kernel launched just before
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const size_t stride = (size_t)bd.total_nodes * kHq;   // rows between splits
  const size_t row0 = (size_t)r * kHq + head;
  __shared__ float s_max[kMergeThreads / 32];
  __shared__ float4 s_acc[kMergeGroups - 1][64];
  __shared__ float s_den[kMergeGroups - 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = tid >> 6, t = tid & 63;
  // first batch of this thread's splits, in flight during the max reduction
  float w[kBatch];
  uint2 o[kBatch];   // 4 bf16
#pragma unroll
  for (int k = 0; k < kBatch; ++k) {
    const int s = grp + k * kMergeGroups;
    const size_t row = (size_t)min(s, ns - 1) * stride + row0;
    w[k] = s < ns ? p.lse_part[row] : -INFINITY;
    o[k] = reinterpret_cast<const uint2*>(p.o_part + row * kDim)[t];
  }
  float mx = -INFINITY;
  for (int s = tid; s < ns; s += kMergeThreads) mx = fmaxf(mx, p.lse_part[s * stride + row0]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) s_max[warp] = mx;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kMergeThreads / 32; ++i) mx = fmaxf(mx, s_max[i]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  for (int base = 0;;) {
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const float wk = fast_exp2(w[k] - mx);   // 0 for the padding entries (w = -inf)
      const float2 lo = unpack_bf16(o[k].x), hi = unpack_bf16(o[k].y);
      den += wk;
      acc.x += wk * lo.x; acc.y += wk * lo.y; acc.z += wk * hi.x; acc.w += wk * hi.y;
    }
    base += kBatch * kMergeGroups;
    if (base >= ns) break;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int s = base + grp + k * kMergeGroups;
      const size_t row = (size_t)min(s, ns - 1) * stride + row0;
      w[k] = s < ns ? p.lse_part[row] : -INFINITY;
      o[k] = reinterpret_cast<const uint2*>(p.o_part + row * kDim)[t];
    }
  }
  if (grp > 0) {
    s_acc[grp - 1][t] = acc;
    if (t == 0) s_den[grp - 1] = den;
  }
  __syncthreads();
  if (grp > 0) return;
#pragma unroll
  for (int k = 0; k < kMergeGroups - 1; ++k) {
    const float4 v = s_acc[k][t];
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    den += s_den[k];
  }
  const float inv = 1.f / den;
  uint2 packed;
  packed.x = pack_bf16(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2*>(p.out + row0 * kDim)[t] = packed;
  if (p.lse != nullptr && t == 0) p.lse[row0] = (mx + fast_log2(den)) * kLn2;
}

}  // namespace

// Launched as a programmatic dependent of the split kernel: its blocks may be
// scheduled while the split kernel runs and wait (griddepcontrol.wait) for
// that kernel's completion before they read the partials.
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
