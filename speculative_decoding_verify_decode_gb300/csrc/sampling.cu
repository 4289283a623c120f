// Sampling-based verification: speculative sampling over a chain or a token
// tree at temperature T, instead of the greedy argmax walk.
//
// The pages verify greedily and name sampling as future work
// («如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍», 补充测试 and
// 关键突破; «Qwen3.8-27B 部署技术报告» runs at temperature 0); they give no
// acceptance rule, so this is the standard one, with the multi-candidate rule
// for trees:
//   p_u = softmax(logits_u / T); the children of u were drawn from the draft
//   distribution q_u; they are tried in increasing node order, child c with
//   token x being accepted when r_c q_u(x) < p(x); after a rejection p becomes
//   max(0, p - q_u) renormalised; the walk descends into an accepted child; when
//   every child is rejected (or u is a leaf) the bonus token is drawn from the
//   current p by inverse CDF with u's uniform s_u.
//
// Kernel 1 scans 4096-entry chunks of every logits row (128-bit loads) for
// the chunk's maximum and sum of exp((x - max) / T).  Kernel 2 runs one
// 1024-thread CTA per sequence: it combines each row's chunk statistics, then
// walks the tree with block-uniform decisions.  The current distribution is
// kept as (node u, residual normalisers Z_1..Z_k): p_k(v) = max(0, p_{k-1}(v)
// - q_u(v)) / Z_k with p_0 = p_u, recomputed element by element, so a
// rejection costs one pass over the vocabulary (the next normaliser) and the
// bonus one pass for tile sums plus one tile for the final scan.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace sdv {
namespace {

constexpr int kSampleThreads = 1024;
constexpr int kTile = 1024;              // elements per tile of the inverse-CDF search
constexpr int kMaxResidual = kMaxNodes;  // residual steps at one node (at most its children)

struct MaxSum {
  float m;
  float s;
};

// combine two (max, sum of exp((x - max) * inv_t)) pairs
__device__ __forceinline__ MaxSum combine(MaxSum a, MaxSum b, float inv_t) {
  if (a.m == -INFINITY) return b;
  if (b.m == -INFINITY) return a;
  const float m = fmaxf(a.m, b.m);
  return {m, a.s * expf((a.m - m) * inv_t) + b.s * expf((b.m - m) * inv_t)};
}

template <bool kVec4>
__global__ void __launch_bounds__(256) lse_chunk_kernel(const SampleParams p) {
  const int row = blockIdx.y;
  const int chunk = blockIdx.x;
  const float* x = p.logits + (size_t)row * p.vocab;
  const int begin = chunk * kAcceptChunk;
  const int end = min(p.vocab, begin + kAcceptChunk);
  const float inv_t = p.inv_t;
  MaxSum acc = {-INFINITY, 0.f};
  bool nan = false;
  auto add = [&](float e) {
    nan |= e != e;
    if (e > acc.m) {
      acc.s = acc.m == -INFINITY ? 1.f : acc.s * expf((acc.m - e) * inv_t) + 1.f;
      acc.m = e;
    } else if (e != -INFINITY) {
      acc.s += expf((e - acc.m) * inv_t);
    }
  };
  if (kVec4) {
    for (int i = begin + threadIdx.x * 4; i < end; i += 256 * 4) {
      const float4 v = __ldcs(reinterpret_cast<const float4*>(x + i));
      add(v.x); add(v.y); add(v.z); add(v.w);
    }
  } else {
    for (int i = begin + threadIdx.x; i < end; i += 256) add(x[i]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    MaxSum o = {__shfl_xor_sync(0xffffffffu, acc.m, off), __shfl_xor_sync(0xffffffffu, acc.s, off)};
    acc = combine(acc, o, inv_t);
  }
  __shared__ MaxSum red[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = acc;
  if (__syncthreads_or(nan) && threadIdx.x == 0) report(p.dev_status, SD_DEV_NAN_LOGITS);
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) acc = combine(acc, red[w], inv_t);
    reinterpret_cast<MaxSum*>(p.partial)[(size_t)row * p.chunks + chunk] = acc;
  }
}

// Sum of one value per thread over the block; every thread gets the total.
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();   // red[] may still be read from a previous call
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < kSampleThreads / 32 ? red[lane] : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
  return t;
}

__global__ void __launch_bounds__(kSampleThreads) sample_accept_kernel(const SampleParams p, const BatchDesc bd) {
  const int b = blockIdx.x;
  const int q0 = bd.q_indptr[b];
  const int n = bd.q_indptr[b + 1] - q0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int V = p.vocab;
  const float inv_t = p.inv_t;
  __shared__ float s_m[kMaxNodes], s_s[kMaxNodes];   // per row: max, sum of exp((x - max) / T)
  __shared__ int s_par[kMaxNodes], s_path[kMaxNodes + 1], s_tok[kMaxNodes + 1];
  __shared__ float s_z[kMaxResidual];                // residual normalisers at the current node
  __shared__ float s_red[kSampleThreads / 32];
  __shared__ float s_tiles[kSampleMaxTiles];
  __shared__ int s_bad, s_pick;
  __shared__ float s_base;

  if (tid == 0) s_bad = 0;
  // each row's statistics from its chunk partials: a warp per row
  for (int row = warp; row < n; row += kSampleThreads / 32) {
    const MaxSum* part = reinterpret_cast<const MaxSum*>(p.partial) + (size_t)(q0 + row) * p.chunks;
    MaxSum acc = {-INFINITY, 0.f};
    for (int c = lane; c < p.chunks; c += 32) acc = combine(acc, part[c], inv_t);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      MaxSum o = {__shfl_xor_sync(0xffffffffu, acc.m, off), __shfl_xor_sync(0xffffffffu, acc.s, off)};
      acc = combine(acc, o, inv_t);
    }
    if (lane == 0) {
      s_m[row] = acc.m;
      s_s[row] = acc.s;
    }
  }
  if (tid < n) {
    const int pj = p.parents[q0 + tid];
    if ((tid == 0 && pj != -1) || (tid > 0 && (pj < 0 || pj >= tid))) atomicOr(&s_bad, 1);
    s_par[tid] = pj;
  }
  __syncthreads();
  // a broken tree: reported; the root is kept alone, with a bonus drawn at the root
  const bool bad = s_bad != 0;
  if (bad && tid == 0) report(p.dev_status, SD_DEV_BAD_PARENTS);

  // p_k(v) at node u with k residual steps
  auto prob = [&](int u, int k, int v) -> float {
    const float l = p.logits[(size_t)(q0 + u) * V + v];
    float x = s_s[u] > 0.f ? expf((l - s_m[u]) * inv_t) / s_s[u] : 0.f;
    const float qv = p.draft_probs[(size_t)(q0 + u) * V + v];
    for (int i = 0; i < k; ++i) x = fmaxf(x - qv, 0.f) / s_z[i];
    return x;
  };

  int u = 0, k = 0, a = 1;
  if (tid == 0) s_path[0] = 0;
  int bonus = 0;
  for (int step = 0; step < n; ++step) {
    int accepted = -1;
    for (int c = u + 1; c < n && !bad; ++c) {
      if (s_par[c] != u) continue;
      const int x = p.draft_tokens[q0 + c];
      if (x < 0 || x >= V) continue;   // not a token: never accepted
      const float px = prob(u, k, x);
      const float qx = p.draft_probs[(size_t)(q0 + u) * V + x];
      if (p.r_accept[q0 + c] * qx < px) {
        accepted = c;
        break;
      }
      // rejected: the next residual normaliser, one pass over the vocabulary
      float part = 0.f;
      for (int v = tid; v < V; v += kSampleThreads)
        part += fmaxf(prob(u, k, v) - p.draft_probs[(size_t)(q0 + u) * V + v], 0.f);
      const float z = block_sum(part, s_red);
      if (z > 0.f && k < kMaxResidual) {
        __syncthreads();
        if (tid == 0) s_z[k] = z;
        __syncthreads();
        ++k;
      }
    }
    if (accepted >= 0) {
      if (tid == 0) {
        s_path[a] = accepted;
        s_tok[a - 1] = p.draft_tokens[q0 + accepted];
      }
      ++a;
      u = accepted;
      k = 0;
      continue;
    }
    // bonus from the current distribution: tile sums (a warp per tile, lane = 32 consecutive tokens),
    // then the tile and the token where the cumulative sum first exceeds s * total
    const int tiles = (V + kTile - 1) / kTile;
    for (int t = warp; t < tiles; t += kSampleThreads / 32) {
      float ls = 0.f;
      for (int i = 0; i < 32; ++i) {
        const int v = t * kTile + lane * 32 + i;
        if (v < V) ls += prob(u, k, v);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
      if (lane == 0) s_tiles[t] = ls;
    }
    __syncthreads();
    if (tid == 0) {
      float total = 0.f;
      for (int t = 0; t < tiles; ++t) total += s_tiles[t];
      const float target = p.r_sample[q0 + u] * total;
      float run = 0.f;
      int pick = -1, last = 0;
      for (int t = 0; t < tiles; ++t) {
        if (s_tiles[t] > 0.f) last = t;
        if (pick < 0 && run + s_tiles[t] > target) pick = t;
        if (pick < 0) run += s_tiles[t];
      }
      if (pick < 0) {   // rounding left the target at the very end: the last tile with mass
        pick = last;
        run = 0.f;
        for (int t = 0; t < last; ++t) run += s_tiles[t];
      }
      s_pick = pick;
      s_base = run;
      s_red[0] = target;
    }
    __syncthreads();
    if (warp == 0) {
      const int t = s_pick;
      const float target = s_red[0];
      float w[32], ls = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int v = t * kTile + lane * 32 + i;
        w[i] = v < V ? prob(u, k, v) : 0.f;
        ls += w[i];
      }
      float incl = ls;   // inclusive scan of the lanes' sums
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const float base = s_base;
      const unsigned hit = __ballot_sync(0xffffffffu, base + incl > target);
      const unsigned has = __ballot_sync(0xffffffffu, ls > 0.f);
      int src = hit ? __ffs(hit) - 1 : (has ? 31 - __clz(has) : 0);
      int chosen = -1;
      if (lane == src) {
        float run = base + incl - ls;
        int lastpos = -1;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (w[i] > 0.f) lastpos = i;
          run += w[i];
          if (chosen < 0 && run > target && w[i] > 0.f) chosen = i;
        }
        if (chosen < 0) chosen = lastpos < 0 ? 0 : lastpos;
        chosen += t * kTile + lane * 32;
      }
      chosen = __shfl_sync(0xffffffffu, chosen, src);
      if (lane == 0) s_pick = min(chosen, V - 1);
    }
    __syncthreads();
    bonus = s_pick;
    break;
  }
  if (tid != 0) return;
  s_tok[a - 1] = bonus;
  if (a > p.max_path) report(p.dev_status, SD_DEV_PATH_OVERFLOW);
  const int a_out = min(a, p.max_path);
  p.accept_len[b] = a_out;
  int* path = p.path + (size_t)b * p.max_path;
  int* toks = p.out_tokens + (size_t)b * p.max_path;
  for (int i = 0; i < p.max_path; ++i) {
    path[i] = i < a_out ? s_path[i] : -1;
    toks[i] = i < a_out ? s_tok[i] : -1;
  }
}

}  // namespace

cudaError_t launch_sample_accept(const SampleParams& p, const BatchDesc& bd, cudaStream_t st) {
  dim3 grid(p.chunks, bd.total_nodes);
  const bool aligned = (reinterpret_cast<uintptr_t>(p.logits) & 15) == 0;
  if (p.vocab % 4 == 0 && aligned) lse_chunk_kernel<true><<<grid, 256, 0, st>>>(p);
  else lse_chunk_kernel<false><<<grid, 256, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sample_accept_kernel<<<bd.batch, kSampleThreads, 0, st>>>(p, bd);
  return cudaGetLastError();
}

}  // namespace sdv
