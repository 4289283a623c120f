// Draft-tree (DDTree) construction: per-position top-K of the draft logits,
// then a best-first token tree of `budget` nodes under the root.
//
// «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍» (blog.xiaohack.org):
// 从自回归到 DDTree — a draft block of 16 positions becomes a tree of `budget`
// nodes verified in one target forward; 关键突破 — the tree comes from the
// draft's per-position top-K (K = 32 -> 8), with a chain pre-seed; a top-K list
// handed over worst-first sends the worst token under the root.
//
// Kernel 1 scans fixed 4096-logit chunks of every (sequence, position) row
// with 128-bit loads; each thread keeps its 16 values' top 8 in registers
// (largest value first, equal values: smaller token id first), the warps merge
// theirs by 8 rounds of redux.sync argmax, and the chunk's top 8 is written with
// the chunk's (max, sum of exp(x - max)) for the log-sum-exp.
// Kernel 2 runs one block per sequence: sixteen warps merge the chunk lists of
// the positions (all of a position's records in one round of loads) and form
// log-probabilities (logit - log-sum-exp); one warp then inserts the rank-0
// chain up to depth min(positions, budget) and adds the best remaining
// candidate (kept in registers across the warp; two redux.sync maxima over an
// order-preserving score key and the inverted creation number) until the tree
// holds 1 + budget nodes.  The
// candidates are, for every inserted node, its first child (rank 0, one
// position deeper) and its next sibling (rank + 1, same parent); score = the
// summed log-probabilities of the root path; ties go to the candidate created
// first.  Node ids follow insertion order, so parent[j] < j.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace sdv {
namespace {

constexpr int kK = kDdTopKMax;      // candidates kept per chunk and per position
constexpr int kThreads1 = 256;
constexpr int kThreads2 = 512;
constexpr int kMaxCand = 3 * kMaxNodes;   // live candidates never exceed 2 per node + the chain's

// (av, ai) ranks before (bv, bi): larger value, or equal value and smaller id.
__device__ __forceinline__ bool before(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

// Insert (v, i) into a sorted top-kK list held in registers.
__device__ __forceinline__ void insert_sorted(float (&tv)[kK], int (&ti)[kK], float v, int i) {
  if (!before(v, i, tv[kK - 1], ti[kK - 1])) return;
  tv[kK - 1] = v;
  ti[kK - 1] = i;
#pragma unroll
  for (int j = kK - 1; j > 0; --j) {
    if (before(tv[j], ti[j], tv[j - 1], ti[j - 1])) {
      const float fv = tv[j]; tv[j] = tv[j - 1]; tv[j - 1] = fv;
      const int fi = ti[j]; ti[j] = ti[j - 1]; ti[j - 1] = fi;
    }
  }
}

// Order-preserving 32-bit key of a float (larger float -> larger key; -0 and +0
// must be folded by the caller, NaN excluded).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Warp-wide argmax of (value, id) pairs with ties to the smaller id: two
// redux.sync, the largest value key, then the smallest id among the lanes holding it.
__device__ __forceinline__ void warp_best(float v, int i, float& bv, int& bi) {
  const uint32_t k = order_key(v + 0.0f);                 // -0 -> +0
  const uint32_t bk = __reduce_max_sync(0xffffffffu, k);
  bi = (int)__reduce_min_sync(0xffffffffu, k == bk ? (uint32_t)i : 0xffffffffu);
  bv = key_value(bk);
}

// Warp-wide: the best of the lanes' list heads; the winning lane drops its head.
// Returns the winner (same on every lane).
__device__ __forceinline__ void warp_pop_best(float (&tv)[kK], int (&ti)[kK], float& wv, int& wi) {
  warp_best(tv[0], ti[0], wv, wi);
  if ((tv[0] + 0.0f) == wv && ti[0] == wi) {   // ids are distinct: one lane matches (padding lanes may too)
#pragma unroll
    for (int j = 0; j < kK - 1; ++j) { tv[j] = tv[j + 1]; ti[j] = ti[j + 1]; }
    tv[kK - 1] = -INFINITY;
    ti[kK - 1] = INT_MAX;
  }
}

// (max, sum of exp(x - max)) pairs: combine b into a.
__device__ __forceinline__ void lse_combine(float& am, float& as, float bm, float bs) {
  const float m = fmaxf(am, bm);
  if (m == -INFINITY) return;
  as = as * __expf(am - m) + bs * __expf(bm - m);
  am = m;
}

template <bool kVec4>
__global__ void __launch_bounds__(kThreads1) topk_chunk_kernel(const DdtreeParams p) {
  const int row = blockIdx.y;                 // sequence * positions + position
  const int chunk = blockIdx.x;
  const float* x = p.logits + (size_t)row * p.vocab;
  const int begin = chunk * kDdChunk;
  const int end = min(p.vocab, begin + kDdChunk);
  float tv[kK];
  int ti[kK];
#pragma unroll
  for (int j = 0; j < kK; ++j) { tv[j] = -INFINITY; ti[j] = INT_MAX; }
  constexpr int kPer = kDdChunk / kThreads1;  // 16 values per thread
  static_assert(kPer == 16, "one batch of four 16-byte loads per thread");
  float e[kPer];
  int ei[kPer];
  bool nan = false;
#pragma unroll
  for (int q = 0; q < kPer / 4; ++q) {
    const int i = begin + q * kThreads1 * 4 + threadIdx.x * 4;
    float4 v = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (kVec4) {
      if (i < end) v = __ldcs(reinterpret_cast<const float4*>(x + i));   // vocab % 4 == 0: 16-byte aligned
    } else {
      if (i < end) v.x = x[i];
      if (i + 1 < end) v.y = x[i + 1];
      if (i + 2 < end) v.z = x[i + 2];
      if (i + 3 < end) v.w = x[i + 3];
    }
    e[4 * q] = v.x; e[4 * q + 1] = v.y; e[4 * q + 2] = v.z; e[4 * q + 3] = v.w;
#pragma unroll
    for (int k = 0; k < 4; ++k) ei[4 * q + k] = i + k;
  }
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    nan |= e[k] != e[k];
    if (e[k] != e[k]) e[k] = -INFINITY;       // reported; ignored by the selection
    m = fmaxf(m, e[k]);
  }
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    if (e[k] != -INFINITY) s += __expf(e[k] - m);
    if (ei[k] < end) insert_sorted(tv, ti, e[k], ei[k]);
  }
  if (__any_sync(0xffffffffu, nan) && (threadIdx.x & 31) == 0) report(p.dev_status, SD_DEV_NAN_LOGITS);

  __shared__ float s_v[kThreads1 / 32][kK];
  __shared__ int s_i[kThreads1 / 32][kK];
  __shared__ float s_m[kThreads1 / 32], s_s[kThreads1 / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // warp: log-sum-exp pair and top 8
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, off), os = __shfl_xor_sync(0xffffffffu, s, off);
    lse_combine(m, s, om, os);
  }
  float rv[kK];
  int ri[kK];
#pragma unroll
  for (int k = 0; k < kK; ++k) warp_pop_best(tv, ti, rv[k], ri[k]);
  if (lane == 0) {
    s_m[warp] = m;
    s_s[warp] = s;
#pragma unroll
    for (int k = 0; k < kK; ++k) { s_v[warp][k] = rv[k]; s_i[warp][k] = ri[k]; }
  }
  __syncthreads();
  if (warp != 0) return;
  // warp 0 merges the 8 warps' lists: lane l holds entries 2l and 2l + 1 (a sorted pair)
#pragma unroll
  for (int j = 0; j < kK; ++j) { tv[j] = -INFINITY; ti[j] = INT_MAX; }
  {
    const int w = (2 * lane) / kK, k0 = (2 * lane) % kK;
    tv[0] = s_v[w][k0]; ti[0] = s_i[w][k0];
    tv[1] = s_v[w][k0 + 1]; ti[1] = s_i[w][k0 + 1];
  }
  m = lane < kThreads1 / 32 ? s_m[lane] : -INFINITY;
  s = lane < kThreads1 / 32 ? s_s[lane] : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, off), os = __shfl_xor_sync(0xffffffffu, s, off);
    lse_combine(m, s, om, os);
  }
#pragma unroll
  for (int k = 0; k < kK; ++k) warp_pop_best(tv, ti, rv[k], ri[k]);
  const size_t rec = (size_t)row * p.chunks + chunk;
  if (lane < kK) {
    float v = rv[0];
    int i = ri[0];
#pragma unroll
    for (int k = 1; k < kK; ++k) if (lane == k) { v = rv[k]; i = ri[k]; }
    p.part_v[rec * kK + lane] = v;
    p.part_i[rec * kK + lane] = i;
  }
  if (lane == 0) {
    p.part_ms[rec * 2] = m;
    p.part_ms[rec * 2 + 1] = s;
  }
}

__global__ void __launch_bounds__(kThreads2) ddtree_build_kernel(const DdtreeParams p) {
  extern __shared__ __align__(16) uint8_t dyn[];
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kThreads2 / 32;
  const int cpr = p.chunks * kK;              // candidate records per position
  float* c_v = reinterpret_cast<float*>(dyn);                // [kWarps][cpr]
  int* c_i = reinterpret_cast<int*>(c_v + kWarps * cpr);     // [kWarps][cpr]
  __shared__ int s_tok[kMaxNodes][kK];        // candidate tokens per position
  __shared__ float s_lp[kMaxNodes][kK];       // their log-probabilities
  // ---- per position (one warp each): merge the chunk lists, log-probabilities
  for (int d = warp; d < p.positions; d += kWarps) {
    const size_t row = (size_t)b * p.positions + d;
    float* wv = c_v + warp * cpr;
    int* wi = c_i + warp * cpr;
    // every record of the position in one round of loads
    constexpr int kU = 8;
    for (int r0 = lane; r0 < cpr; r0 += 32 * kU) {
      float v[kU];
      int i[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int r = min(r0 + 32 * u, cpr - 1);
        v[u] = p.part_v[row * cpr + r];
        i[u] = p.part_i[row * cpr + r];
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int r = min(r0 + 32 * u, cpr - 1);
        wv[r] = v[u];
        wi[r] = i[u];
      }
    }
    float m = -INFINITY, s = 0.f;
    for (int c = lane; c < p.chunks; c += 32) lse_combine(m, s, p.part_ms[(row * p.chunks + c) * 2],
                                                         p.part_ms[(row * p.chunks + c) * 2 + 1]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, m, off), os = __shfl_xor_sync(0xffffffffu, s, off);
      lse_combine(m, s, om, os);
    }
    const float lse = m + __logf(s);
    __syncwarp();
    // topk rounds: the best record ranked after the previous winner
    float pv = INFINITY;
    int pi = -1;
    for (int k = 0; k < p.topk; ++k) {
      float bv = -INFINITY;
      int bi = INT_MAX;
      for (int r = lane; r < cpr; r += 32) {
        const float v = wv[r];
        const int i = wi[r];
        if (before(pv, pi, v, i) && before(v, i, bv, bi)) { bv = v; bi = i; }
      }
      warp_best(bv, bi, bv, bi);
      if (lane == 0) { s_tok[d][k] = bi; s_lp[d][k] = bv - lse; }
      pv = bv;
      pi = bi;
    }
    __syncwarp();
  }
  __syncthreads();
  if (warp != 0) return;
  // ---- best-first insertion (warp 0).  Candidate number c lives in lane c % 32,
  // register slot c / 32: (score, parent's score, creation number, parent | depth << 8 | rank << 16).
  __shared__ int n_par[kMaxNodes], n_tok[kMaxNodes];
  __shared__ float n_sc[kMaxNodes];
  constexpr int kSlots = (kMaxCand + 31) / 32;
  float c_sc[kSlots], c_psc[kSlots];
  int c_seq[kSlots], c_info[kSlots];
#pragma unroll
  for (int k = 0; k < kSlots; ++k) { c_sc[k] = -INFINITY; c_psc[k] = 0.f; c_seq[k] = -1; c_info[k] = 0; }
  const int P = p.positions, K = p.topk, budget = p.budget;
  const int chain = min(P, budget);
  int ncand = 0;
  auto push = [&](int par, int dep, int rank, float par_score) {
    if (dep > P || rank >= K || ncand >= kMaxCand) return;
    const float sc = par_score + s_lp[dep - 1][rank];
    const int slot = ncand >> 5;
    if (lane == (ncand & 31)) {
#pragma unroll
      for (int k = 0; k < kSlots; ++k)
        if (k == slot) { c_sc[k] = sc; c_psc[k] = par_score; c_seq[k] = ncand; c_info[k] = par | (dep << 8) | (rank << 16); }
    }
    ++ncand;
  };
  float chain_sc = 0.f;
  if (lane == 0) {
    n_par[0] = -1;
    n_tok[0] = p.root_tokens[b];
    n_sc[0] = 0.f;
  }
  for (int d = 1; d <= chain; ++d) {        // the chain pre-seed
    const float sc = chain_sc + s_lp[d - 1][0];
    if (lane == 0) {
      n_par[d] = d - 1;
      n_tok[d] = s_tok[d - 1][0];
      n_sc[d] = sc;
    }
    chain_sc = sc;
  }
  {
    float sc = 0.f;
    for (int d = 0; d < chain; ++d) {       // second-best child of each chain node
      push(d, d + 1, 1, sc);
      sc += s_lp[d][0];
    }
    push(chain, chain + 1, 0, chain_sc);    // the chain's continuation
  }
  int nodes = 1 + chain;
  while (nodes < 1 + budget) {
    // this lane's best live candidate: largest score, then smallest creation number
    uint32_t k1 = 0u, k2 = 0u;
    int bk = -1;
    float bsc = 0.f, bpsc = 0.f;
    int binfo = 0;
#pragma unroll
    for (int k = 0; k < kSlots; ++k) {
      if (c_seq[k] < 0) continue;
      const uint32_t a1 = order_key(c_sc[k] + 0.0f), a2 = ~(uint32_t)c_seq[k];
      if (bk < 0 || a1 > k1 || (a1 == k1 && a2 > k2)) {
        k1 = a1; k2 = a2; bk = k; bsc = c_sc[k]; bpsc = c_psc[k]; binfo = c_info[k];
      }
    }
    if (__ballot_sync(0xffffffffu, bk >= 0) == 0u) break;   // no candidate left
    const uint32_t best1 = __reduce_max_sync(0xffffffffu, bk >= 0 ? k1 : 0u);
    const uint32_t best2 = __reduce_max_sync(0xffffffffu, (bk >= 0 && k1 == best1) ? k2 : 0u);
    const bool mine = bk >= 0 && k1 == best1 && k2 == best2;
    const int owner = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
    const float sc = __shfl_sync(0xffffffffu, bsc, owner);
    const float psc = __shfl_sync(0xffffffffu, bpsc, owner);
    const int info = __shfl_sync(0xffffffffu, binfo, owner);
    if (mine) {
#pragma unroll
      for (int k = 0; k < kSlots; ++k) if (k == bk) c_seq[k] = -1;   // taken
    }
    const int par = info & 0xff, dep = (info >> 8) & 0xff, rank = info >> 16;
    const int node = nodes;
    if (lane == 0) {
      n_par[node] = par;
      n_tok[node] = s_tok[dep - 1][rank];
      n_sc[node] = sc;
    }
    push(node, dep + 1, 0, sc);               // its first child
    push(par, dep, rank + 1, psc);            // its next sibling
    ++nodes;
  }
  __syncwarp();
  const int out0 = b * (1 + budget);
  for (int j = lane; j < 1 + budget; j += 32) {
    const bool live = j < nodes;
    p.parents[out0 + j] = live ? n_par[j] : -1;
    p.tokens[out0 + j] = live ? n_tok[j] : -1;
    if (p.scores != nullptr) p.scores[out0 + j] = live ? n_sc[j] : -INFINITY;
  }
}

}  // namespace

size_t ddtree_smem_bytes(int chunks) { return (size_t)(kThreads2 / 32) * chunks * kK * 8; }

cudaError_t launch_ddtree(const DdtreeParams& p, cudaStream_t st) {
  dim3 g1(p.chunks, p.batch * p.positions);
  if (p.vocab % 4 == 0) topk_chunk_kernel<true><<<g1, kThreads1, 0, st>>>(p);
  else topk_chunk_kernel<false><<<g1, kThreads1, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = ddtree_smem_bytes(p.chunks);
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(ddtree_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  ddtree_build_kernel<<<p.batch, kThreads2, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace sdv
