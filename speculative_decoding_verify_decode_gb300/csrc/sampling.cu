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
constexpr int kPer = kTile / kSampleThreads;   // tokens per thread in the bonus draw
constexpr int kReqPass = 1, kReqDone = 2;      // requests of the walking warp to the rest of the block
static_assert(kTile % kSampleThreads == 0 && kTile % 1024 == 0, "tile of whole thread and load rounds");
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
  pdl_wait();
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
    // kTile / 1024 16-byte loads per thread, all issued before any is used
    constexpr int kLoads = kTile / 1024;
    float4 v[kLoads];
#pragma unroll
    for (int j = 0; j < kLoads; ++j) {
      const int i = begin + j * 1024 + threadIdx.x * 4;
      v[j] = i < end ? __ldcs(reinterpret_cast<const float4*>(x + i))
                     : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int j = 0; j < kLoads; ++j) { add(v[j].x); add(v[j].y); add(v[j].z); add(v[j].w); }
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
  pdl_wait();
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
  constexpr int kLoads = kTile / 1024;
  float r = 0.f;
  if (kVec4) {
    float4 l[kLoads], q[kLoads];
#pragma unroll
    for (int j = 0; j < kLoads; ++j) {
      const int v0 = tile * kTile + j * 1024 + threadIdx.x * 4;
      const bool in = v0 + 4 <= p.vocab;   // V % 4 == 0: a group of four is whole or absent
      l[j] = in ? *reinterpret_cast<const float4*>(lr + v0) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      q[j] = in ? *reinterpret_cast<const float4*>(qr + v0) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kLoads; ++j)   // absent groups: p = 2^-inf = 0 and q = 0 add 0
      r += fmaxf(fast_exp2((l[j].x - m) * c) * inv_s - q[j].x, 0.f) +
           fmaxf(fast_exp2((l[j].y - m) * c) * inv_s - q[j].y, 0.f) +
           fmaxf(fast_exp2((l[j].z - m) * c) * inv_s - q[j].z, 0.f) +
           fmaxf(fast_exp2((l[j].w - m) * c) * inv_s - q[j].w, 0.f);
  } else {
    for (int j = 0; j < kLoads; ++j) {
      const int v0 = tile * kTile + j * 1024 + threadIdx.x * 4;
      for (int i = 0; i < 4 && v0 + i < p.vocab; ++i)
        r += fmaxf(fast_exp2((lr[v0 + i] - m) * c) * inv_s - qr[v0 + i], 0.f);
    }
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

// Inclusive prefix sum of one value per thread over the block in thread order; every thread gets its
// own prefix and the block total.  `w` holds 32 floats of shared memory, free on entry.
__device__ __forceinline__ float block_incl_scan(float v, float* w, float& total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) w[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    float x = lane < kSampleThreads / 32 ? w[lane] : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += o;
    }
    w[lane] = x;
  }
  __syncthreads();
  total = w[31];
  return (warp > 0 ? w[warp - 1] : 0.f) + incl;
}

// kVec4: V % 4 == 0 and 16-byte aligned rows, so passes move four tokens per 16-byte load.
template <bool kVec4>
__global__ void __launch_bounds__(kSampleThreads, 1) sample_accept_kernel(const SampleParams p, const BatchDesc bd) {
  pdl_wait();
  const int b = blockIdx.x;
  const int q0 = bd.q_indptr[b];
  const int n = bd.q_indptr[b + 1] - q0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int V = p.vocab;
  const float inv_t = p.inv_t * kLog2e;   // base-2 scale: exp((x - m) / T) = 2^((x - m) * inv_t)
  __shared__ float s_m[kMaxNodes], s_s[kMaxNodes];   // per row: max, 1 / sum of exp((x - max) / T) (0 if none)
  __shared__ int s_par[kMaxNodes], s_path[kMaxNodes + 1], s_tok[kMaxNodes + 1];
  __shared__ float s_z[kMaxResidual];                // reciprocals of the residual normalisers at the current node
  __shared__ float s_z1[kMaxNodes];                  // per row: the first residual normaliser (sum of its tile sums)
  // per candidate node c (its token x in its parent's row): x, the logit and draft probability of x there, and
  // the acceptance uniform, fetched for every node at once so that the walk reads no global memory per test
  __shared__ int s_cx[kMaxNodes];
  __shared__ float s_cl[kMaxNodes], s_cq[kMaxNodes], s_cr[kMaxNodes], s_rs[kMaxNodes];
  __shared__ float s_red[kSampleThreads / 32];
  __shared__ float s_tiles[kSampleMaxTiles];
  __shared__ int s_bad, s_pick, s_last;
  __shared__ int s_req, s_req_u, s_req_k;   // requests of the walking warp (kReqPass / kReqDone)
  __shared__ float s_base, s_scan[32];

  if (tid == 0) s_bad = 0;
  // each row's statistics from its chunk partials: a warp per row
  for (int row = warp; row < n; row += kSampleThreads / 32) {
    const MaxSum* part = reinterpret_cast<const MaxSum*>(p.partial) + (size_t)(q0 + row) * p.chunks;
    const float* rs = p.resid + (size_t)(q0 + row) * p.chunks;
    MaxSum acc = {-INFINITY, 0.f};
    float z1 = 0.f;
    for (int c = lane; c < p.chunks; c += 32) {
      acc = combine(acc, part[c], inv_t);
      z1 += rs[c];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      MaxSum o = {__shfl_xor_sync(0xffffffffu, acc.m, off), __shfl_xor_sync(0xffffffffu, acc.s, off)};
      acc = combine(acc, o, inv_t);
      z1 += __shfl_xor_sync(0xffffffffu, z1, off);
    }
    if (lane == 0) {
      s_m[row] = acc.m;
      s_s[row] = acc.s > 0.f ? 1.0f / acc.s : 0.f;
      s_z1[row] = z1;
    }
  }
  if (tid < n) {
    const int pj = p.parents[q0 + tid];
    if ((tid == 0 && pj != -1) || (tid > 0 && (pj < 0 || pj >= tid))) atomicOr(&s_bad, 1);
    s_par[tid] = pj;
    const int x = p.draft_tokens[q0 + tid];
    s_cx[tid] = x;
    s_cr[tid] = p.r_accept[q0 + tid];
    s_rs[tid] = p.r_sample[q0 + tid];
    float l = 0.f, qv = 0.f;
    if (tid > 0 && pj >= 0 && pj < tid && x >= 0 && x < V) {
      l = p.logits[(size_t)(q0 + pj) * V + x];
      qv = p.draft_probs[(size_t)(q0 + pj) * V + x];
    }
    s_cl[tid] = l;
    s_cq[tid] = qv;
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

  // the next residual normaliser at (u, k >= 1): a pass of the whole block over the vocabulary
  // (32 tokens per thread and round); every thread gets the sum
  auto resid_pass = [&](int ru, int rk) -> float {
    float part = 0.f;
    for (int v0 = tid * 32; v0 < V; v0 += kSampleThreads * 32) part += sum32(ru, rk, v0, true);
    return block_sum(part, s_red);
  };

  // Warp 0 walks the tree (its lanes take the same decisions; every test reads shared memory only).
  // The other warps wait at named barrier 1 for a request: a residual normaliser that needs a pass over
  // the vocabulary (a second rejection at one node), which the whole block computes, or the end of the
  // walk, after which the whole block draws the bonus.  Warp 0 has no early exit: it always reaches
  // the final request.
  int u = 0, k = 0, a = 1;
  if (warp == 0) {
    if (lane == 0) s_path[0] = 0;
    for (int step = 0; step < n; ++step) {
      int accepted = -1;
      for (int c = u + 1; c < n && !bad; ++c) {
        if (s_par[c] != u) continue;
        const int x = s_cx[c];
        if (x < 0 || x >= V) continue;   // not a token: never accepted
        const float qx = s_cq[c];
        const float px = prob_of(u, k, s_cl[c], qx);
        if (s_cr[c] * qx < px) {
          accepted = c;
          break;
        }
        // rejected: the next residual normaliser — the first from the residual tile sums (added up per
        // row above), later ones by a pass of the whole block over the vocabulary
        float z;
        if (k == 0) {
          z = s_z1[u];
        } else {
          if (lane == 0) { s_req = kReqPass; s_req_u = u; s_req_k = k; }
          asm volatile("bar.sync 1, %0;" ::"n"(kSampleThreads) : "memory");
          z = resid_pass(u, k);
        }
        if (z > 0.f && k < kMaxResidual) {
          if (lane == 0) s_z[k] = 1.0f / z;
          __syncwarp();
          ++k;
        }
      }
      if (accepted < 0) break;   // the bonus, from the current distribution
      if (lane == 0) {
        s_path[a] = accepted;
        s_tok[a - 1] = s_cx[accepted];
      }
      ++a;
      u = accepted;
      k = 0;
    }
    if (lane == 0) { s_req = kReqDone; s_req_u = u; s_req_k = k; }
    asm volatile("bar.sync 1, %0;" ::"n"(kSampleThreads) : "memory");
  } else {
    for (;;) {
      asm volatile("bar.sync 1, %0;" ::"n"(kSampleThreads) : "memory");
      if (s_req == kReqDone) break;
      resid_pass(s_req_u, s_req_k);
    }
  }
  u = s_req_u;
  k = s_req_k;
  {
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
        float ls = 0.f;
        for (int sub = 0; sub < kTile; sub += 1024) ls += sum32(u, k, t * kTile + sub + lane * 32, false);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
        if (lane == 0) s_tiles[t] = ls;
      }
    }
    // the tile: each thread takes `per` consecutive tiles; a block prefix sum finds the first tile whose
    // cumulative sum exceeds s * total (rounding can leave none: then the last tile with mass)
    if (tid == 0) { s_pick = INT_MAX; s_last = -1; }
    __syncthreads();
    {
      const int per = (tiles + kSampleThreads - 1) / kSampleThreads;
      const int t0 = tid * per;
      float ls = 0.f;
      int lastm = -1;
      for (int j = 0; j < per; ++j) {
        const int t = t0 + j;
        if (t < tiles) {
          ls += s_tiles[t];
          if (s_tiles[t] > 0.f) lastm = t;
        }
      }
      float total;
      const float incl = block_incl_scan(ls, s_scan, total);
      const float target = s_rs[u] * total;
      float run = incl - ls;
      for (int j = 0; j < per; ++j) {
        const int t = t0 + j;
        if (t < tiles) {
          if (run + s_tiles[t] > target) { atomicMin(&s_pick, t); break; }
          run += s_tiles[t];
        }
      }
      if (lastm >= 0) atomicMax(&s_last, lastm);
      __syncthreads();
      const int pick = s_pick != INT_MAX ? s_pick : (s_last >= 0 ? s_last : 0);
      if (t0 <= pick && pick < t0 + per) {   // the owner of the tile: the sum of the tiles before it
        float base = incl - ls;
        for (int t = t0; t < pick; ++t) base += s_tiles[t];
        s_base = base;
        s_red[0] = target;
      }
      __syncthreads();
      if (tid == 0) s_pick = pick;
      __syncthreads();
    }
    // the token: thread i takes tokens 4i .. 4i + 3 of the tile; a block prefix sum in token order from the
    // tiles before finds the first token with mass whose cumulative sum exceeds the target (rounding can
    // leave none: then the last token with mass)
    {
      const int t = s_pick;
      const float target = s_red[0], base = s_base;
      const int v0 = t * kTile + tid * kPer;
      float wv[kPer], ls = 0.f;
#pragma unroll
      for (int e = 0; e < kPer; ++e) {
        wv[e] = v0 + e < V ? prob(u, k, v0 + e) : 0.f;
        ls += wv[e];
      }
      __syncthreads();   // everyone has read s_pick before it is reset
      if (tid == 0) { s_pick = INT_MAX; s_last = -1; }
      __syncthreads();
      float total;
      float run = base + block_incl_scan(ls, s_scan, total) - ls;
      int first = -1, lastm = -1;
#pragma unroll
      for (int e = 0; e < kPer; ++e) {
        run += wv[e];
        if (wv[e] > 0.f) {
          lastm = v0 + e;
          if (first < 0 && run > target) first = v0 + e;
        }
      }
      if (first >= 0) atomicMin(&s_pick, first);
      if (lastm >= 0) atomicMax(&s_last, lastm);
      __syncthreads();
      if (tid == 0) {
        const int chosen = s_pick != INT_MAX ? s_pick : (s_last >= 0 ? s_last : t * kTile);
        s_pick = min(chosen, V - 1);
      }
      __syncthreads();
    }
  }
  const int bonus = s_pick;
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
  // each kernel starts by waiting for the one before (pdl_wait): the three run as programmatic dependents
  cudaError_t e = (p.vocab % 4 == 0 && aligned) ? launch_pdl(lse_chunk_kernel<true>, grid, dim3(256), 0, st, p)
                                                : launch_pdl(lse_chunk_kernel<false>, grid, dim3(256), 0, st, p);
  if (e != cudaSuccess) return e;
  const bool vec = p.vocab % 4 == 0 && aligned && (reinterpret_cast<uintptr_t>(p.draft_probs) & 15) == 0;
  e = vec ? launch_pdl(resid_tile_kernel<true>, grid, dim3(256), 0, st, p)
          : launch_pdl(resid_tile_kernel<false>, grid, dim3(256), 0, st, p);
  if (e != cudaSuccess) return e;
  return vec ? launch_pdl(sample_accept_kernel<true>, dim3(bd.batch), dim3(kSampleThreads), 0, st, p, bd)
             : launch_pdl(sample_accept_kernel<false>, dim3(bd.batch), dim3(kSampleThreads), 0, st, p, bd);
}

}  // namespace sdv
