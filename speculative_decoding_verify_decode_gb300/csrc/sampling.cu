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
// Kernel 1 scans 1024-entry tiles of every logits row (128-bit loads) for
// the tile's maximum and sum of exp((x - max) / T).  Kernel 2 runs one
// 1024-thread CTA per sequence: it combines each row's tile statistics, then
// walks the tree with block-uniform decisions.  The current distribution is
// kept as (node u, residual normalisers Z_1..Z_k): p_k(v) = max(0, p_{k-1}(v)
// - q_u(v)) / Z_k with p_0 = p_u, recomputed element by element.  A bonus
// drawn with no residual step (the common case) needs no pass over the
// vocabulary: the tile sums of p_u come from kernel 1, and one tile is
// scanned.  Kernel 1b sums the first residual max(0, p_u - q_u) per tile for
// every row, in parallel, so a first rejection at a node (its normaliser, and a
// bonus drawn after it) needs no pass either; only a second rejection at the
// same node costs passes over the vocabulary (16-byte loads).
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace sdv {
namespace {

constexpr int kSampleThreads = 1024;
constexpr int kTile = kSampleTile;       // elements per tile (statistics and inverse-CDF search)
constexpr int kMaxResidual = kMaxNodes;  // residual steps at one node (at most its children)
constexpr float kLog2e = 1.4426950408889634f;

struct MaxSum {
  float m;
  float s;
};

// combine two (max, sum of exp((x - max) / T)) pairs; c = log2(e) / T, so exp(y / T) = 2^(y c)
__device__ __forceinline__ MaxSum combine(MaxSum a, MaxSum b, float c) {
  if (a.m == -INFINITY) return b;
  if (b.m == -INFINITY) return a;
  const float m = fmaxf(a.m, b.m);
  return {m, a.s * fast_exp2((a.m - m) * c) + b.s * fast_exp2((b.m - m) * c)};
}

template <bool kVec4>
__global__ void __launch_bounds__(256) lse_chunk_kernel(const SampleParams p) {
  const int row = blockIdx.y;
  const int chunk = blockIdx.x;
  const float* x = p.logits + (size_t)row * p.vocab;
  const int begin = chunk * kTile;
  const int end = min(p.vocab, begin + kTile);
  const float inv_t = p.inv_t * kLog2e;   // base-2 scale
  MaxSum acc = {-INFINITY, 0.f};
  bool nan = false;
  auto add = [&](float e) {
    nan |= e != e;
    if (e > acc.m) {
      acc.s = acc.m == -INFINITY ? 1.f : acc.s * fast_exp2((acc.m - e) * inv_t) + 1.f;
      acc.m = e;
    } else if (e != -INFINITY) {
      acc.s += fast_exp2((e - acc.m) * inv_t);
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

// Per (row, tile): sum of max(0, p_u(v) - q_u(v)) over the tile's tokens — the tile sums of the first
// residual at every node, from which the walk takes the first normaliser and, after one rejection, the
// bonus tile sums without a pass of its own.
template <bool kVec4>
__global__ void __launch_bounds__(256) resid_tile_kernel(const SampleParams p) {
  const int row = blockIdx.y, tile = blockIdx.x;
  const float c = p.inv_t * kLog2e;
  __shared__ float s_stat[2];
  __shared__ float red[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {   // the row's statistics from its tile partials
    const MaxSum* part = reinterpret_cast<const MaxSum*>(p.partial) + (size_t)row * p.chunks;
    MaxSum acc = {-INFINITY, 0.f};
    for (int t = lane; t < p.chunks; t += 32) acc = combine(acc, part[t], c);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      MaxSum o = {__shfl_xor_sync(0xffffffffu, acc.m, off), __shfl_xor_sync(0xffffffffu, acc.s, off)};
      acc = combine(acc, o, c);
    }
    if (lane == 0) {
      s_stat[0] = acc.m;
      s_stat[1] = acc.s > 0.f ? 1.0f / acc.s : 0.f;
    }
  }
  __syncthreads();
  const float m = s_stat[0], inv_s = s_stat[1];
  const float* lr = p.logits + (size_t)row * p.vocab;
  const float* qr = p.draft_probs + (size_t)row * p.vocab;
  const int v0 = tile * kSampleTile + threadIdx.x * 4;
  float r = 0.f;
  if (kVec4 && v0 + 4 <= p.vocab) {
    const float4 l = *reinterpret_cast<const float4*>(lr + v0);
    const float4 q = *reinterpret_cast<const float4*>(qr + v0);
    r = fmaxf(fast_exp2((l.x - m) * c) * inv_s - q.x, 0.f) + fmaxf(fast_exp2((l.y - m) * c) * inv_s - q.y, 0.f) +
        fmaxf(fast_exp2((l.z - m) * c) * inv_s - q.z, 0.f) + fmaxf(fast_exp2((l.w - m) * c) * inv_s - q.w, 0.f);
  } else {
    for (int i = 0; i < 4 && v0 + i < p.vocab; ++i)
      r += fmaxf(fast_exp2((lr[v0 + i] - m) * c) * inv_s - qr[v0 + i], 0.f);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
  if (lane == 0) red[warp] = r;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += red[w];
    p.resid[(size_t)row * p.chunks + tile] = t;
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

// kVec4: V % 4 == 0 and 16-byte aligned rows, so passes move four tokens per 16-byte load.
template <bool kVec4>
__global__ void __launch_bounds__(kSampleThreads, 1) sample_accept_kernel(const SampleParams p, const BatchDesc bd) {
  const int b = blockIdx.x;
  const int q0 = bd.q_indptr[b];
  const int n = bd.q_indptr[b + 1] - q0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int V = p.vocab;
  const float inv_t = p.inv_t * kLog2e;   // base-2 scale: exp((x - m) / T) = 2^((x - m) * inv_t)
  __shared__ float s_m[kMaxNodes], s_s[kMaxNodes];   // per row: max, 1 / sum of exp((x - max) / T) (0 if none)
  __shared__ int s_par[kMaxNodes], s_path[kMaxNodes + 1], s_tok[kMaxNodes + 1];
  __shared__ float s_z[kMaxResidual];                // reciprocals of the residual normalisers at the current node
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
      s_s[row] = acc.s > 0.f ? 1.0f / acc.s : 0.f;
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

  // p_k(v) at node u with k residual steps, from the logit l and the draft probability qv of token v
  auto prob_of = [&](int u, int k, float l, float qv) -> float {
    float x = fast_exp2((l - s_m[u]) * inv_t) * s_s[u];
    for (int i = 0; i < k; ++i) x = fmaxf(x - qv, 0.f) * s_z[i];
    return x;
  };
  auto prob = [&](int u, int k, int v) -> float {
    return prob_of(u, k, p.logits[(size_t)(q0 + u) * V + v], p.draft_probs[(size_t)(q0 + u) * V + v]);
  };
  // sum over tokens [v0, v0 + 32) of p_k (tile-sum pass) or of max(0, p_k - q) (next normaliser)
  auto sum32 = [&](int u, int k, int v0, bool resid) -> float {
    float acc = 0.f;
    const float* lr = p.logits + (size_t)(q0 + u) * V;
    const float* qr = p.draft_probs + (size_t)(q0 + u) * V;
    if (kVec4 && v0 + 32 <= V) {
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 l = *reinterpret_cast<const float4*>(lr + v0 + i);
        const float4 q = *reinterpret_cast<const float4*>(qr + v0 + i);
        const float e[4] = {l.x, l.y, l.z, l.w}, f[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float x = prob_of(u, k, e[c], f[c]);
          acc += resid ? fmaxf(x - f[c], 0.f) : x;
        }
      }
    } else {
      for (int i = 0; i < 32 && v0 + i < V; ++i) {
        const float f = qr[v0 + i];
        const float x = prob_of(u, k, lr[v0 + i], f);
        acc += resid ? fmaxf(x - f, 0.f) : x;
      }
    }
    return acc;
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
      // rejected: the next residual normaliser — the first from the residual tile sums, later ones by a
      // pass over the vocabulary (32 tokens per thread and round)
      float part = 0.f;
      if (k == 0) {
        for (int t = tid; t < p.chunks; t += kSampleThreads) part += p.resid[(size_t)(q0 + u) * p.chunks + t];
      } else {
        for (int v0 = tid * 32; v0 < V; v0 += kSampleThreads * 32) part += sum32(u, k, v0, true);
      }
      const float z = block_sum(part, s_red);
      if (z > 0.f && k < kMaxResidual) {
        __syncthreads();
        if (tid == 0) s_z[k] = 1.0f / z;
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
    // bonus from the current distribution: tile sums — from the statistics pass when no residual step
    // was taken, else one pass (a warp per tile, lane = 32 consecutive tokens) — then the tile and the
    // token where the cumulative sum first exceeds s * total
    const int tiles = (V + kTile - 1) / kTile;
    if (k == 0) {
      const MaxSum* part = reinterpret_cast<const MaxSum*>(p.partial) + (size_t)(q0 + u) * p.chunks;
      for (int t = tid; t < tiles; t += kSampleThreads) {
        const MaxSum ms = part[t];
        s_tiles[t] = ms.m == -INFINITY ? 0.f : ms.s * fast_exp2((ms.m - s_m[u]) * inv_t) * s_s[u];
      }
    } else if (k == 1) {
      for (int t = tid; t < tiles; t += kSampleThreads) s_tiles[t] = p.resid[(size_t)(q0 + u) * p.chunks + t] * s_z[0];
    } else {
      for (int t = warp; t < tiles; t += kSampleThreads / 32) {
        float ls = sum32(u, k, t * kTile + lane * 32, false);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
        if (lane == 0) s_tiles[t] = ls;
      }
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
  const bool vec = p.vocab % 4 == 0 && aligned && (reinterpret_cast<uintptr_t>(p.draft_probs) & 15) == 0;
  if (vec) resid_tile_kernel<true><<<grid, 256, 0, st>>>(p);
  else resid_tile_kernel<false><<<grid, 256, 0, st>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (vec) sample_accept_kernel<true><<<bd.batch, kSampleThreads, 0, st>>>(p, bd);
  else sample_accept_kernel<false><<<bd.batch, kSampleThreads, 0, st>>>(p, bd);
  return cudaGetLastError();
}

}  // namespace sdv
