// Commit of the accepted draft nodes' K/V into the paged cache, every layer
// in one launch.
//
// Accepted node path[i] becomes context position ctx + i: page
// table[(ctx + i) / 16], slot (ctx + i) % 16 — 16-token pages from one pool,
// «Qwen3.8-27B投机解码实测：从14到159 tok/s的性能断点地图» §2 and §4.  Rejected nodes
// are never written; the accepted state is written once, in place, instead of
// being copied around afterwards (the persist-kernel idea of
// «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍», 关键突破).
//
// One CTA per (layer, sequence).  It first validates everything it is about
// to touch (accept length, path ids, page ids); an invalid sequence is
// reported and skipped as a whole.  The copy moves 16-byte vectors: each
// 512-byte (node, KV head) row of K or V is one warp-wide coalesced read and
// write.
//
// e4m3 caches: the rows are quantised on the way in (the write-time
// quantisation of «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍»,
// 24 GB 显存上的 128K 上下文, here in e4m3 with one scale per layer and tensor):
// code = e4m3(x * (1 / scale)), the product rounded to fp32, then to the
// nearest e4m3 value (ties to even), finite values beyond 448 saturating.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace sdv {
namespace {

// Two fp32 values as two e4m3 codes (lo in the low byte), nearest-even, saturating.
__device__ __forceinline__ uint32_t to_e4m3x2(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b16 t; cvt.rn.satfinite.e4m3x2.f32 t, %1, %2; cvt.u32.u16 %0, t; }" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Eight bf16 (one 16-byte chunk) times `inv`, as eight e4m3 codes.
__device__ __forceinline__ uint2 quantise8(const uint4 v, float inv) {
  auto two = [inv](uint32_t w) -> uint32_t {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
    return to_e4m3x2(__fmul_rn(f.x, inv), __fmul_rn(f.y, inv));
  };
  return make_uint2(two(v.x) | (two(v.y) << 16), two(v.z) | (two(v.w) << 16));
}

// FP8: e4m3 caches (quantise on the way in); otherwise bf16 rows are copied unchanged.
template <bool FP8>
__global__ void __launch_bounds__(256) commit_kernel(const CommitParams p, const BatchDesc bd) {
  const int layer = blockIdx.x;
  const int b = blockIdx.y;
  const int q0 = bd.q_indptr[b];
  const int n = bd.q_indptr[b + 1] - q0;
  const int a = p.accept_len[b];
  const int L = p.ctx_lens[b];
  __shared__ int s_page[kMaxNodes];
  __shared__ int s_src[kMaxNodes];

  bool bad = a < 1 || a > n || a > p.max_path || L < 0 ||
             (long long)L + a > (long long)p.max_pages * kPage;
  if (!bad && threadIdx.x < a) {
    const int i = threadIdx.x;
    const int node = p.path[(size_t)b * p.max_path + i];
    const int pos = L + i;
    const int page = p.page_table[(size_t)b * p.max_pages + (pos >> 4)];
    bool ok = node >= 0 && node < n && (i != 0 || node == 0);
    if (page < 0 || page >= p.num_pool_pages) {
      ok = false;
      if (layer == 0) report(p.dev_status, SD_DEV_BAD_PAGE);
    }
    bad = !ok;
    s_page[i] = page;
    s_src[i] = q0 + node;
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0 && layer == 0) report(p.dev_status, SD_DEV_BAD_ACCEPT);
    return;
  }

  const uint4* k_src = static_cast<const uint4*>(p.k_new[layer]);
  const uint4* v_src = static_cast<const uint4*>(p.v_new[layer]);
  constexpr int kVecPerRow = kDim * 2 / 16;  // 32 x 16 B per (node, head) row
  if constexpr (FP8) {
    // a 256-code row per (node, head): 32 x 8 B
    uint2* k_dst = static_cast<uint2*>(p.k_cache[layer]);
    uint2* v_dst = static_cast<uint2*>(p.v_cache[layer]);
    const float ki = p.k_inv[layer], vi = p.v_inv[layer];
    const int tasks = a * kHkv * kVecPerRow;
    for (int t = threadIdx.x; t < tasks; t += blockDim.x) {
      const int v = t % kVecPerRow;
      const int g = (t / kVecPerRow) % kHkv;
      const int i = t / (kVecPerRow * kHkv);
      const int pos = L + i;
      const size_t src = ((size_t)s_src[i] * kHkv + g) * kVecPerRow + v;
      const size_t dst = (((size_t)s_page[i] * kHkv + g) * kPage + (pos & 15)) * kVecPerRow + v;
      k_dst[dst] = quantise8(k_src[src], ki);
      v_dst[dst] = quantise8(v_src[src], vi);
    }
    if (layer == 0 && threadIdx.x == 0 && p.new_ctx_lens != nullptr) p.new_ctx_lens[b] = L + a;
    return;
  }
  uint4* k_dst = static_cast<uint4*>(p.k_cache[layer]);
  uint4* v_dst = static_cast<uint4*>(p.v_cache[layer]);
  const int tasks = a * kHkv * kVecPerRow;
  for (int t = threadIdx.x; t < tasks; t += blockDim.x) {
    const int v = t % kVecPerRow;
    const int g = (t / kVecPerRow) % kHkv;
    const int i = t / (kVecPerRow * kHkv);
    const int pos = L + i;
    const size_t src = ((size_t)s_src[i] * kHkv + g) * kVecPerRow + v;
    const size_t dst = (((size_t)s_page[i] * kHkv + g) * kPage + (pos & 15)) * kVecPerRow + v;
    k_dst[dst] = k_src[src];
    v_dst[dst] = v_src[src];
  }
  if (layer == 0 && threadIdx.x == 0 && p.new_ctx_lens != nullptr) p.new_ctx_lens[b] = L + a;
}

}  // namespace

cudaError_t launch_commit(const CommitParams& p, const BatchDesc& bd, cudaStream_t st) {
  dim3 grid(p.num_layers, bd.batch);
  if (p.fp8)
    commit_kernel<true><<<grid, 256, 0, st>>>(p, bd);
  else
    commit_kernel<false><<<grid, 256, 0, st>>>(p, bd);
  return cudaGetLastError();
}

}  // namespace sdv
