// Split-KV verify attention on the 5th-generation tensor cores (tcgen05,
// accumulators in tensor memory) with TMA-staged K/V pages.
//
// What it computes is the same as the tree/causal-masked grouped-query
// attention of the verify step: for sequence b, draft node j and query head
// h, softmax attention (scale 1/16) of q[j][h] over every context token of KV
// head h/6 plus the draft nodes on j's root path.  Sources, by page title:
// «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍» (为什么我们要做这个测试:
// 24 Q / 4 KV heads, head dim 256; 关键突破: the tree mask follows each node's
// parent chain) and «Qwen3.8-27B投机解码实测：从14到159 tok/s的性能断点地图» (§2, §4:
// 16-token pages from one pool; §5.3: bottom-right causal mask of a chain).
//
// Layout of the work.  A CTA owns (split s, KV head g, head part c, sequence
// b): hpc query heads of group g (6, 3, 2 or 1, so that hpc * N <= 96)
// times the sequence's N draft nodes form NQ (multiple of 16) query columns.
// For QK the tokens are the MMA's M dimension ("swap-AB"), so a 128-token K
// tile serves every query column at once; PV then takes the query columns as
// M (padded to 128) and all 256 dims as N:
//   S^T[128 tok][NQ]  = K_tile[128 tok][256] . Q^T                (K-major A and B)
//   O[128 q][256 dim] += P[128 q][128 tok] . V_tile[128 tok][256]  (MN-major A and B)
// S^T (double-buffered, 2 * NQ columns) and O (256 columns, one query column
// per tensor-memory lane) live in tensor memory.  P is the bf16 P^T tile the
// softmax writes, read as an MN-major A operand; its rows past NQ are never
// written and only reach rows of O that are never read.  The column sums of P
// (the softmax denominators) are added by the softmax warps from the same
// rounded P^T tile.  Because a thread of the epilogue holds a whole 512-byte
// output row, the rows leave tensor memory straight for global memory.  When a
// sequence needs several CTAs for its query heads (hpc < 6), the CTAs of one
// split are adjacent in launch order and read the same pages while they are
// still in L2.
//
// Operand tiles (Q^T, K, V) are "block-major": four 64-dim blocks, each
// holding every row of the tile at 128 B with the 128-byte swizzle, so the
// UMMA descriptors step 1 KB between 8-row groups.  A TMA box of 16 rows x 64
// dims (one page of one KV head, one block) writes 2 KB of a block; a
// 128-token tile takes 32 boxes.
//
// Warp roles (224 threads): warp 0 streams K tiles and warp 6 V tiles with
// TMA; warp 1 allocates tensor memory and one lane issues every tcgen05.mma,
// taking QK of tile i and PV of tile i-1 in whichever order their inputs
// arrive; warps 2-5 (one per tensor-memory lane quarter, thread = token row)
// run the online softmax: masking, a running per-column maximum that is only
// raised (and O, l rescaled) when a score exceeds it by more than 2^8, exp2,
// and the bf16 P^T tile.  Every wait on an mbarrier is bounded; on
// expiry the kernel reports SD_DEV_TIMEOUT and winds down.
//
// Quantised cache (KV8).  The context K/V pages hold e4m3 codes with one
// scale per tensor (K, V) of the layer; the key and value a code stands for is
// decode(code) * scale (the quantised KV cache of «如何在单张 RTX 3090 上让
// Qwen3.5-27B token 生成速度提升 6 倍», 24 GB 显存上的 128K 上下文, here in e4m3).
// The tensor core takes f16 operands (every e4m3 value is exact in f16), so
// each tile passes through two stages: a loader warp (8) brings e4m3 half
// tiles by TMA into two 16 KB staging slots per tensor (K: dims 0-127 or
// 128-255 of every token, one 2 KB box per page; V: pages 0-3 or 4-7, one
// 4 KB bulk copy per page), and converter warps (0 and 7 for K, 6 and 9 for
// V) widen a slot into the tensor's single f16 half-tile buffer, which the
// MMA consumes half by half (QK in two 128-dim steps, PV in two 64-token
// steps).  A slot is refilled as soon as it has been widened, so the next
// tile's codes are in flight while this tile is multiplied.  Q^T, P^T and the
// draft block are f16 too.  The K scale joins the softmax multiplier and the
// V scale the epilogue's normalisation; the draft block (not yet committed,
// so not quantised) has scale 1.
#pragma once

#include <cstddef>
#include <cstring>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace sdv {
namespace {

constexpr int kT = kTileTokens;         // tokens per tile
constexpr int kTileB = kT / 8 * kGroupB;   // 64 KB
constexpr int kAtomB = kT * 128;        // one 64-column atom of the P^T tile: 16 KB
constexpr int kThreads = 224;
constexpr int kThreads8 = 320;          // the quantised-cache instances: two more converters and a loader
constexpr int kWarpK = 0, kWarpMma = 1, kWarpV = 6;
// quantised cache: second K / V converter and the TMA loader, placed so that each of the four
// schedulers (warp % 4) runs one converter warp
constexpr int kWarpK2 = 7, kWarpV2 = 9, kWarpLoad = 8;
constexpr int kHalfB = kTileB / 2;      // quantised cache: f16 half tile (128 tokens x 128 dims, or 64 x 256)
constexpr int kSlotB = kTileB / 4;      // quantised cache: e4m3 half tile (staging slot)
constexpr float kThresh = 8.0f;         // base-2 growth of the max tolerated without rescaling
constexpr float kNoMax = -1.0e30f;      // the running maximum before any visible score

// The V tile moves in two 64-token halves (pages 0-3 and 4-7, each 32 KB
// contiguous), so that the first half of the next tile loads while the PV
// product still reads the second half of this one.
// Quantised cache: K_FULL / K_EMPTY and V_FULL0 / V_EMPTY0 guard the f16
// half-tile buffers (two phases per tile), K8_* / V8_* the e4m3 staging slots.
enum Bar { K_FULL, K_EMPTY, V_FULL0, V_FULL1, V_EMPTY0, V_EMPTY1, S_FULL0, S_FULL1, S_FREE0, S_FREE1, P_FULL, O_DONE,
           GROUP, K8_FULL0, K8_FULL1, K8_EMPTY0, K8_EMPTY1, V8_FULL0, V8_FULL1, V8_EMPTY0, V8_EMPTY1, NUM_BARS };

constexpr int kCols = 128;   // per-column arrays padded to whole 32-column groups
constexpr int kMaxStageRows = kTcMaxNQ + 2 * kMaxNodes;   // Q^T rows + the draft block's K and V rows

// Per-column arrays first: each is read with 16-byte vector loads.
struct Small {
  float m[kCols];
  float alpha[kCols];
  float red[4][kCols];
  float lsum[4][kCols];   // per softmax warp: column sums of P over its 32 token rows
  int outrow[kCols];    // output row (node row * 24 + head) of each query column (-1: padding)
  int lo_col[kCols];    // sliding window: oldest context position each query column sees
  uint64_t bar[NUM_BARS];
  unsigned long long anc[kMaxNodes];    // bit r of anc[n]: draft node r is node n or one of its ancestors
  int par[kMaxNodes];
  int depth[kMaxNodes];   // draft CTA with a window: depth of each node
  // Row copies of the staging pass: source row (null: zeros), byte offset of
  // the row's chunk 0 in the dynamic shared memory, and its 64-dim block stride.
  const __nv_bfloat16* rsrc[kMaxStageRows];
  uint32_t rdst[kMaxStageRows];
  uint32_t rblk[kMaxStageRows];
  int flag[2][4];
  uint32_t tmem;
  int abort;
};
static_assert(offsetof(Small, m) % 16 == 0 && offsetof(Small, alpha) % 16 == 0 &&
                  offsetof(Small, red) % 16 == 0 && offsetof(Small, lsum) % 16 == 0 &&
                  offsetof(Small, outrow) % 16 == 0 && offsetof(Small, lo_col) % 16 == 0,
              "per-column arrays must be 16-byte aligned");
static_assert(offsetof(Small, bar) % 8 == 0, "mbarriers must be 8-byte aligned");
static_assert(kTcMaxNQ * 512 + 2 * kTileB + 2 * kAtomB + sizeof(Small) <= 232448,
              "the widest tile configuration must fit in 227 KB of shared memory");

// ------------------------------------------------------------ quantised cache

// Eight bf16 (one 16-byte chunk) as eight f16, rounded to nearest.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4 v) {
  auto one = [](uint32_t w) -> uint32_t {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
    const __half2 h = __floats2half2_rn(f.x, f.y);
    return *reinterpret_cast<const uint32_t*>(&h);
  };
  return make_uint4(one(v.x), one(v.y), one(v.z), one(v.w));
}
// Four e4m3 codes (one 32-bit word, low byte first) as four f16 (two words;
// exact: e4m3 is a subset of f16).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t four, uint32_t& lo, uint32_t& hi) {
  asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; cvt.rn.f16x2.e4m3x2 %0, l; cvt.rn.f16x2.e4m3x2 %1, h; }"
      : "=r"(lo), "=r"(hi)
      : "r"(four));
}
// Half a page of e4m3 K codes (16 slots x 128 dims: x = 0 or 128) into shared
// memory: a 2 KB box of the 3-D code map at (x, 0, page * 4 + head).
__device__ __forceinline__ void tma_load_k8(uint32_t dst, const CUtensorMap* map, int x, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(0), "r"(z), "r"(bar), "l"(l2_evict_first())
      : "memory");
}
// `bytes` contiguous bytes (a multiple of 16, both addresses 16-byte aligned) into shared memory, read
// with the evict-first policy (context pages).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
               ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(l2_evict_first())
               : "memory");
}
// WIN: compiled with the sliding-window paths (band masks, depths); the
// instances without them serve full attention.
// KV8: the quantised-cache instance (e4m3 pages, f16 operands, converter warps).
template <int NQ, bool WIN, bool KV8>
__global__ void __launch_bounds__(KV8 ? kThreads8 : kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const AttnParams p, const BatchDesc bd, const int hpc, const int hparts) {
  constexpr int NG = (NQ + 31) / 32;          // 32-column groups
  constexpr int NATOM = (NQ + 63) / 64;       // 64-column atoms of the P^T tile the softmax writes
  constexpr int kQB = NQ * 512;               // Q^T tile: 4 blocks of NQ rows x 128 B
  constexpr uint32_t kColS0 = 0, kColO = 2 * NQ;   // tensor-memory columns
  static_assert(2 * NQ + kDim <= 512, "tensor memory holds 2 S^T buffers and O");
  // The kernel declares no static shared memory, so the dynamic window starts
  // at a 1024-byte boundary (required by the 128-byte swizzle atoms); indexing
  // it directly keeps every access a shared-space one.
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  uint8_t* sQ = dyn_smem;
  uint8_t* sK = sQ + kQB;
  uint8_t* sV = sK + (KV8 ? kHalfB : kTileB);
  uint8_t* sK8 = sV + kHalfB;        // quantised cache: two e4m3 K slots
  uint8_t* sV8 = sK8 + 2 * kSlotB;   // quantised cache: two e4m3 V slots
  uint8_t* sP = sK + 2 * kTileB;
  Small* sm = reinterpret_cast<Small*>(sP + 2 * kAtomB);   // P^T spans 128 columns: PV takes M = 128

  constexpr int NT = KV8 ? kThreads8 : kThreads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // warps that fill the K/V tiles: TMA producers, or converters for a quantised cache
  const bool producer =
      warp == kWarpK || warp == kWarpV || (KV8 && (warp == kWarpK2 || warp == kWarpV2 || warp == kWarpLoad));
  const int bid = blockIdx.x;
  const int c = bid % hparts;
  const int g = (bid / hparts) % kHkv;
  const int s = bid / (hparts * kHkv);
  const int b = blockIdx.y;
  const int q0 = bd.q_indptr[b];
  const int n_nodes = bd.q_indptr[b + 1] - q0;
  const int rows = hpc * n_nodes;
  if (c * hpc >= kGroup) return;
  // Launched as a programmatic dependent of the previous kernel in the stream.
  // By default every thread waits for that kernel before touching global
  // memory.  With ctx_stable (the caller guarantees that kernel writes neither
  // the context lengths, the page table nor the context pages) a context CTA
  // reads those and issues its first tile's loads first: its producers wait
  // once that tile is on its way, its compute warps before they read Q or the
  // parents, so the outputs and the workspace are written only after the wait.
  // The draft CTA always waits here: it reads Q and the draft block at once.
  // Then the merge kernel's blocks may be scheduled (they wait for this grid to
  // finish before reading).
  const bool early = p.ctx_stable != 0 && s != 0;
  if (smem_u32(dyn_smem) & 1023u) {  // not expected; refuse rather than mis-swizzle
    if (threadIdx.x == 0) report_dep(p.dev_status, SD_DEV_TIMEOUT);
    return;
  }
  // The draft CTA (split 0) runs to the end in every case: it takes its tensor
  // memory before the wait (no global memory involved).
  if (s == 0 && warp == kWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&sm->tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // the producers fetch their TMA descriptor while the rest of the prologue runs
  if (((!KV8 && (warp == kWarpK || warp == kWarpV)) || (KV8 && warp == kWarpLoad)) && lane == 0)
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(warp == kWarpV ? &tm_v : &tm_k))
                 : "memory");
  if (!early) asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Split 0 attends to the draft block alone; split s >= 1 to context tokens
  // [(s - 1) * chunk, s * chunk).  The producers fetch their first tile's page
  // ids beside the context length (any entry of the table row is in bounds).
  const bool has_draft = (s == 0);
  const int W = WIN ? p.window : 0;
  int page0 = -1;
  if (producer && lane < 8 && !has_draft && W <= 0) {
    const long long idx = (((long long)(s - 1) * p.chunk) >> 4) + lane;
    if (idx < p.max_pages) page0 = p.page_table[(size_t)b * p.max_pages + idx];
  }
  int L = p.ctx_lens[b];
  if (L < 0 || L > p.max_pages * kPage) {
    if (s == 0 && c == 0 && g == 0 && tid == 0) report(p.dev_status, SD_DEV_BAD_CTX);
    L = L < 0 ? 0 : p.max_pages * kPage;
  }
  // with a window the splits cover the tiles from the root's oldest visible position on
  const int base = window_base(L, W, kT);
  const int nsplit = active_splits(L, W, kT, p.chunk);
  if (s >= nsplit) return;
  const int ctx_begin = has_draft ? 0 : base + (s - 1) * p.chunk;
  if (W > 0 && producer && lane < 8 && !has_draft) {
    const long long idx = (ctx_begin >> 4) + lane;
    if (idx < p.max_pages) page0 = p.page_table[(size_t)b * p.max_pages + idx];
  }
  const int ctx_end = has_draft ? 0 : min(L, ctx_begin + p.chunk);
  const int n_tiles = has_draft ? 1 : (ctx_end - ctx_begin + kT - 1) / kT;
  const int head0 = g * kGroup + c * hpc;

  // ---------------------------------------------------------------- prologue
  if (tid == 0) {
    for (int i = 0; i < NUM_BARS; ++i) {
      // a quantised tile is complete when both of its converter warps have arrived
      const bool conv = KV8 && (i == K_FULL || i == V_FULL0 || i == K8_EMPTY0 || i == K8_EMPTY1 ||
                                i == V8_EMPTY0 || i == V8_EMPTY1);
      const uint32_t cnt = (i == S_FREE0 || i == S_FREE1 || i == P_FULL || i == GROUP) ? 4u : conv ? 2u : 1u;
      mbar_init(smem_u32(&sm->bar[i]), cnt);
    }
    sm->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int q = tid; q < kCols; q += NT) {
    // Running maxima start finite and far below any score: a column that has
    // seen no visible key yet (possible with a window) then gives masked scores
    // exp2(-inf - m) = 0, not NaN, and its first visible score takes the
    // rescaling path like any score more than 2^8 above the maximum.
    sm->m[q] = q < NQ ? kNoMax : 0.f;
    sm->alpha[q] = 1.f;
    sm->outrow[q] = q < rows ? (q0 + q / hpc) * kHq + head0 + q % hpc : -1;
  }
  // one load each; the walks below are in shared memory (every CTA needs the depths with a window)
  // (an early context CTA's compute warps load them after their wait)
  if ((has_draft || (W > 0 && !early)) && tid < n_nodes) sm->par[tid] = p.parents[q0 + tid];
  __syncthreads();  // mbarriers and per-column arrays ready
  const uint32_t bars = smem_u32(&sm->bar[0]);
  auto bar = [&](int i) { return bars + 8u * i; };

  // Staging of the operands that do not come by TMA, by `nthr` threads
  // (index t): Q^T (K-major, block-major; column q = node * hpc +
  // head-in-part, the hpc heads of a node being adjacent rows of q; zeros past
  // `rows`) and, in the draft CTA, the draft block as the K and V tiles
  // (group-major; node t = token row t).  A row table (source, destination,
  // block stride) is built first, then one pass of 16-byte copies with up to
  // 16 loads in flight per thread; the last round repeats the final chunk
  // instead of branching, so the unrolled copies stay independent.
  auto stage_operands = [&](const int t, const int nthr, const bool all_warps) {
    const float inv_hpc = 1.0f / (float)hpc;
    const int n_stage = NQ + (has_draft ? 2 * n_nodes : 0);
    for (int r = t; r < n_stage; r += nthr) {
      const __nv_bfloat16* src;
      uint32_t dst, blk;
      if (r < NQ) {
        const int node = __float2int_rz(((float)r + 0.5f) * inv_hpc);   // r / hpc, exact for r < 2^20
        src = r < rows ? p.q + ((size_t)(q0 + node) * kHq + head0 + r - node * hpc) * kDim : nullptr;
        dst = (uint32_t)(sQ - dyn_smem) + r * 128;
        blk = NQ * 128;
      } else {
        const bool is_v = r >= NQ + n_nodes;
        const int tok = r - NQ - (is_v ? n_nodes : 0);
        src = (is_v ? p.v_new : p.k_new) + ((size_t)(q0 + tok) * kHkv + g) * kDim;
        dst = (uint32_t)((is_v ? sV : sK) - dyn_smem) + (tok >> 3) * kGroupB + (tok & 7) * 128;
        blk = 1024;
      }
      sm->rsrc[r] = src;
      sm->rdst[r] = dst;
      sm->rblk[r] = blk;
    }
    if (all_warps) __syncthreads();
    else asm volatile("bar.sync 3, 160;" ::: "memory");   // the five compute warps
    constexpr int U = 16;
    const int tasks = n_stage * 32;
    for (int t0 = t; t0 - t < tasks; t0 += nthr * U) {
      uint4 v[U];
      uint32_t d[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int task = min(t0 + u * nthr, tasks - 1);
        const int r = task >> 5, c = task & 31;
        const __nv_bfloat16* src = sm->rsrc[r];
        const uint32_t off = sm->rdst[r];
        v[u] = src != nullptr ? __ldg(reinterpret_cast<const uint4*>(src) + c) : make_uint4(0, 0, 0, 0);
        d[u] = off + (c >> 3) * sm->rblk[r] + (((c & 7) ^ ((off >> 7) & 7)) << 4);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) *reinterpret_cast<uint4*>(dyn_smem + d[u]) = KV8 ? bf16x8_to_f16x8(v[u]) : v[u];
    }
  };
  if (has_draft) {
    // The draft CTA has no TMA work: all warps stage its operands.  V
    // rows from the block's end to the next 16-row boundary are zeroed (the
    // draft tile's PV product stops there; P^T is 0 on them, but 0 times stale
    // shared memory could be NaN).  S^T rows past the block are masked.
    stage_operands(tid, NT, true);
    const int v_end = (n_nodes + 15) & ~15;
    for (int i = tid; i < (v_end - n_nodes) * 32; i += NT)
      *reinterpret_cast<uint4*>(sV + kv_off(n_nodes + (i >> 5), i & 31)) = make_uint4(0, 0, 0, 0);
    fence_async_smem();   // plain stores above, read by the tensor core
    __syncthreads();
  }

  if (KV8 && producer) {
    const int n_ctx = has_draft ? 0 : n_tiles;
    int page_next = page0;   // lane l < 8: page id of page l of the coming tile, fetched a tile ahead
    // page ids of tile i (lanes 0-7; -1: not needed, or outside the pool)
    auto tile_pages = [&](int i, int& valid, bool report_bad) -> int {
      const int t0 = ctx_begin + i * kT;
      valid = min(kT, ctx_end - t0);
      int page = (lane < 8 && lane * kPage < valid) ? page_next : -1;
      if (lane < 8 && i + 1 < n_ctx && lane * kPage < ctx_end - (t0 + kT))
        page_next = p.page_table[(size_t)b * p.max_pages + (((t0 + kT) >> 4) + lane)];
      if (lane < 8 && lane * kPage < valid && (page < 0 || page >= p.num_pool_pages)) {
        if (report_bad) report_dep(p.dev_status, SD_DEV_BAD_PAGE);
        page = -1;
      }
      return page;
    };
    if (warp == kWarpLoad) {
      // ---------------------------------------------------------- loader (quantised cache)
      // Per tile, four half-tile loads (K dims 0-127, K dims 128-255, V pages
      // 0-3, V pages 4-7), each issued as soon as its slot has been widened.
      int last[4] = {-1, -1, -1, -1};
      bool ok = true;
      for (int i = 0; i < n_ctx && ok; ++i) {
        int valid;
        const int page = tile_pages(i, valid, true);
        const uint32_t need = __ballot_sync(0xffffffffu, lane < 8 && page >= 0);
        const uint32_t parity = (uint32_t)(i & 1) ^ 1u;
        int todo = 0xF;
        long long idle_since = clock64();
        while (todo != 0) {
#pragma unroll
          for (int part = 0; part < 4; ++part) {
            const bool is_k = part < 2;
            const int h = part & 1;
            if (!(todo & (1 << part))) continue;
            const uint32_t empty = bar(is_k ? K8_EMPTY0 + h : V8_EMPTY0 + h);
            const uint32_t full = bar(is_k ? K8_FULL0 + h : V8_FULL0 + h);
            const bool ready = __shfl_sync(0xffffffffu, lane == 0 ? (mbar_test(empty, parity) ? 1 : 0) : 0, 0) != 0;
            if (!ready) continue;
            const uint32_t pm = is_k ? need : (need & (0xFu << (4 * h)));
            if (lane == 0) mbar_expect_tx(full, (uint32_t)__popc(pm) * (is_k ? kSlotB / 8 : kSlotB / 4));
            __syncwarp();
            if ((pm >> lane) & 1u) {
              if (is_k)
                tma_load_k8(smem_u32(sK8 + h * kSlotB + lane * (kSlotB / 8)), &tm_k, 128 * h, page * kHkv + g, full);
              else
                bulk_load(smem_u32(sV8 + h * kSlotB + (lane - 4 * h) * (kSlotB / 4)),
                          p.v_cache8 + ((size_t)page * kHkv + g) * (kPage * kDim), kSlotB / 4, full);
            }
            todo &= ~(1 << part);
            last[part] = i;
            idle_since = clock64();
          }
          if (todo != 0) {
            if (clock64() - idle_since > kWaitCycles || *(volatile int*)&sm->abort) {
              if (lane == 0) { sm->abort = 1; report_dep(p.dev_status, SD_DEV_TIMEOUT); }
              ok = false;
              break;
            }
            // no sleep between polls: the loader's wake-up would sit on the widening chain
          }
        }
        // early context loads: the next slots free up only as the compute warps (which wait) progress
        if (early && i == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
      }
      // no copy may still be landing when the CTA ends (after an abort): wait, bounded, for the last of each slot
      if (lane == 0) {
        for (int part = 0; part < 4; ++part) {
          if (last[part] < 0) continue;
          const uint32_t full = bar(part < 2 ? K8_FULL0 + (part & 1) : V8_FULL0 + (part & 1));
          const long long t0 = clock64();
          while (!mbar_test(full, (uint32_t)(last[part] & 1)) && clock64() - t0 < kWaitCycles) {
          }
        }
      }
    } else {
      // ---------------------------------------------------------- converters (quantised cache)
      // Warp wi (0 or 1) of a tensor, thread t = 32 wi + lane, widens 16
      // chunks of 16 codes of a slot:
      //   K: token rows t/8 + 8u (u < 16), dims 16 (t%8) .. +15 of the half;
      //   V: token rows t/16 + 4u of the half (64 rows), dims 16 (t%16) .. +15.
      // Both slot layouts are linear in the row (K 128 B, V 256 B per row), so
      // each step moves the source by 1 KB and the destination by a constant
      // (K: one 8-row group, 2 KB; V: every other step one 8-row group, 4 KB,
      // the swizzle row alternating between t/16 and t/16 + 4).  Each 8-lane
      // group reads 128 contiguous bytes and writes one row's 16-byte chunks
      // (the odd chunk first where bit 2 of the chunk is set: no bank conflicts).
      const bool is_k = warp == kWarpK || warp == kWarpK2;
      const int t64 = ((warp == kWarpK || warp == kWarpV) ? 0 : 32) + lane;
      uint8_t* dst = is_k ? sK : sV;
      const int c = is_k ? (t64 & 7) : (t64 & 15);           // 16-code chunk of the row
      const int r0 = is_k ? (t64 >> 3) : (t64 >> 4);          // first row
      const bool odd_first = (c & 4) != 0;
      const uint32_t src0 = (uint32_t)(r0 * (is_k ? 128 : kDim) + c * 16);
      // destination of the first / second stored chunk for rows with r % 8 = rr, group 0
      auto dst_pair = [&](int rr, uint32_t& d_first, uint32_t& d_second) {
        const int cc_first = 2 * c + (odd_first ? 1 : 0), cc_second = 2 * c + (odd_first ? 0 : 1);
        auto off = [&](int cc) { return (uint32_t)((cc >> 3) * 1024 + rr * 128 + (((cc & 7) ^ rr) << 4)); };
        d_first = off(cc_first);
        d_second = off(cc_second);
      };
      uint32_t d1e, d2e, d1o, d2o;   // even / odd steps (V: the swizzle row alternates)
      dst_pair(r0 & 7, d1e, d2e);
      dst_pair(is_k ? (r0 & 7) : ((r0 + 4) & 7), d1o, d2o);
      const uint32_t dst_base = smem_u32(dst);
      bool ok = true;
      int uses = 0;   // phases of the f16 half-tile buffer so far
      for (int i = 0; i < n_ctx && ok; ++i) {
        int valid;
        const int page = tile_pages(i, valid, false);
        const bool whole = valid == kT && __ballot_sync(0xffffffffu, lane < 8 && page >= 0) == 0xffu;
        for (int h = 0; h < 2; ++h, ++uses) {
          // early context loads: the f16 buffer's second use waits for the compute warps (which wait)
          if (early && uses == 1) asm volatile("griddepcontrol.wait;" ::: "memory");
          const uint32_t slot_full = bar(is_k ? K8_FULL0 + h : V8_FULL0 + h);
          const uint32_t buf_empty = bar(is_k ? K_EMPTY : V_EMPTY0);
          // every lane waits (a lone waiting lane while the rest of the warp sits at a
          // warp-wide step resumes late)
          ok = mbar_wait(slot_full, (uint32_t)(i & 1), &sm->abort, p.dev_status) &&
               mbar_wait(buf_empty, (uint32_t)(uses & 1) ^ 1u, &sm->abort, p.dev_status);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          const uint32_t src_base = smem_u32((is_k ? sK8 : sV8) + h * kSlotB) + src0;
          // rows of this lane that hold codes (all of them for a whole tile)
          uint32_t live = 0xffffu;
          if (!whole) {
            live = 0u;
            for (int u = 0; u < 16; ++u) {
              const int r = r0 + (is_k ? 8 : 4) * u;
              const int pg = __shfl_sync(0xffffffffu, page, is_k ? r >> 4 : 4 * h + (r >> 4));
              const int tok = is_k ? r : 64 * h + r;
              live |= (pg >= 0 && tok < valid ? 1u : 0u) << u;
            }
          }
#pragma unroll
          for (int u0 = 0; u0 < 16; u0 += 4) {
            uint4 v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t a = src_base + (uint32_t)(u0 + k) * 1024u;
              asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(v[k].x), "=r"(v[k].y), "=r"(v[k].z), "=r"(v[k].w)
                           : "r"(a));
              if (!((live >> (u0 + k)) & 1u)) v[k] = make_uint4(0, 0, 0, 0);   // past the context / no page
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int u = u0 + k;
              // the chunk stored first: codes 8-15 (odd chunk) or 0-7
              const uint32_t f0 = odd_first ? v[k].z : v[k].x, f1 = odd_first ? v[k].w : v[k].y;
              const uint32_t s0 = odd_first ? v[k].x : v[k].z, s1 = odd_first ? v[k].y : v[k].w;
              uint4 a, b2;
              e4m3x4_to_f16x4(f0, a.x, a.y);
              e4m3x4_to_f16x4(f1, a.z, a.w);
              e4m3x4_to_f16x4(s0, b2.x, b2.y);
              e4m3x4_to_f16x4(s1, b2.z, b2.w);
              const uint32_t grp = is_k ? (uint32_t)u * (kGroupB / 2) : (uint32_t)(u >> 1) * kGroupB;
              const uint32_t o1 = dst_base + grp + ((u & 1) ? d1o : d1e);
              const uint32_t o2 = dst_base + grp + ((u & 1) ? d2o : d2e);
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(o1), "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w)
                           : "memory");
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(o2), "r"(b2.x), "r"(b2.y), "r"(b2.z),
                           "r"(b2.w)
                           : "memory");
            }
          }
          fence_async_smem();   // plain stores, read by the tensor core
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bar(is_k ? K_FULL : V_FULL0));
            mbar_arrive(bar(is_k ? K8_EMPTY0 + h : V8_EMPTY0 + h));
          }
        }
        if (__shfl_sync(0xffffffffu, sm->abort, 0)) break;
      }
    }
  } else if (!KV8 && producer) {
    // ------------------------------------------------------------ TMA producers (K or V)
    const bool is_k = warp == kWarpK;
    uint8_t* dst = is_k ? sK : sV;
    const __nv_bfloat16* cache = is_k ? p.k_cache : p.v_cache;
    const CUtensorMap* map = is_k ? &tm_k : &tm_v;
    const int nparts = is_k ? 1 : 2;           // K: one 8-page part; V: two 4-page halves
    const int ppp = 8 / nparts;                 // pages per part
    const int n_ctx = has_draft ? 0 : n_tiles;   // the draft CTA stages its block without TMA
    int page_next = page0;   // lane l < 8: page id of page l of the coming tile, fetched a tile ahead
    for (int i = 0; i < n_ctx; ++i) {
      const int t0 = ctx_begin + i * kT;
      const int valid = min(kT, ctx_end - t0);
      int page = (lane < 8 && lane * kPage < valid) ? page_next : -1;
      if (lane < 8 && i + 1 < n_ctx && lane * kPage < ctx_end - (t0 + kT))
        page_next = p.page_table[(size_t)b * p.max_pages + (((t0 + kT) >> 4) + lane)];
      if (lane < 8 && lane * kPage < valid && (page < 0 || page >= p.num_pool_pages)) {
        report_dep(p.dev_status, SD_DEV_BAD_PAGE);
        page = -1;
      }
      // a page goes by TMA when it is in range and all 16 of its tokens are valid
      const bool page_full = page >= 0 && (lane + 1) * kPage <= valid;
      const uint32_t tma_mask = __ballot_sync(0xffffffffu, lane < 8 && page_full);
      const uint32_t parity = (uint32_t)(i & 1) ^ 1u;
      bool ok = true;
      for (int part = 0; part < nparts && ok; ++part) {
        const uint32_t full = bar(is_k ? K_FULL : V_FULL0 + part), empty = bar(is_k ? K_EMPTY : V_EMPTY0 + part);
        const uint32_t part_mask = ((1u << ppp) - 1u) << (part * ppp);
        if (lane == 0) ok = mbar_wait(empty, parity, &sm->abort, p.dev_status);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        // pages that are partial, missing or out of range: plain copies, zero past the context
        for (int pi = part * ppp; pi < (part + 1) * ppp; ++pi) {
          if (tma_mask & (1u << pi)) continue;
          const int pg = __shfl_sync(0xffffffffu, page, pi);
          stage_rows(dst, pi * kPage, kPage, [&](int slot) -> const __nv_bfloat16* {
            return (pg >= 0 && pi * kPage + slot < valid) ? cache + (((size_t)pg * kHkv + g) * kPage + slot) * kDim
                                                          : nullptr;
          }, lane, 32);
        }
        if ((tma_mask & part_mask) != part_mask) fence_async_smem();   // plain copies above: visible to the MMA
        __syncwarp();
        if (lane == 0) mbar_expect_tx(full, (uint32_t)__popc(tma_mask & part_mask) * kPageB);
        __syncwarp();
        // lane l: page l of the tile, one 8 KB box
        if (((part_mask & tma_mask) >> lane) & 1u)
          tma_load_page(smem_u32(dst + lane * kPageB), map, (page * kHkv + g) * 2, full);
      }
      // early context loads: the next tile's buffers free up only as the compute warps (which wait) progress
      if (early && i == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
      if (!ok) break;
      if (__shfl_sync(0xffffffffu, sm->abort, 0)) break;
    }
  } else {
  // ---------------------------------------------------------------- compute warps (1-5)
  // While the producers fetch the first tiles, these five warps stage Q^T
  // (and split 0's draft block, tile 0) and allocate tensor memory.
  {
    const int ct = tid - 32;
    if (early) {
      // tensor memory first (no global memory), then the wait for the previous kernel
      if (warp == kWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&sm->tmem)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      // the window depths need the parents (ordered before their use by the staging barrier)
      if (W > 0)
        for (int j = ct; j < n_nodes; j += 5 * 32) sm->par[j] = p.parents[q0 + j];
    }
    if (!has_draft) stage_operands(ct, 5 * 32, false);
    if (W > 0) {
      // oldest visible context position of each query column: L + depth(node) - W + 1
      // (padding columns take the root's; an invalid parent chain stops the walk)
      const float inv_hpc = 1.0f / (float)hpc;
      for (int q = ct; q < kCols; q += 5 * 32) {
        int d = 0;
        if (q < rows) {
          for (int u = __float2int_rz(((float)q + 0.5f) * inv_hpc); u > 0 && d < kMaxNodes; ++d) {
            const int pu = sm->par[u];
            if (pu < 0 || pu >= u) break;
            u = pu;
          }
        }
        sm->lo_col[q] = L + d - W + 1;
      }
    }
    if (warp == kWarpMma && !early && s != 0) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&sm->tmem)));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    fence_async_smem();
    tc_fence_before();
    asm volatile("bar.sync 1, 160;" ::: "memory");   // the five compute warps, all arrive unconditionally
    tc_fence_after();
  }
  const uint32_t tmem = sm->tmem;
  if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescQK = f16_idesc(128, NQ, 0, 0, !KV8);
      constexpr uint32_t kIdescPV = f16_idesc(128, kDim, 1, 1, !KV8);
      const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV), p_addr = smem_u32(sP);
      int kf = 0, pf = 0, vf0 = 0, vf1 = 0;
      int pv_half = 0;   // the PV product of a context tile runs in two 64-token halves
      int qk_half = 0;   // quantised cache: the QK product of a context tile runs in two 128-dim halves
      int sfree[2] = {0, 0};
      int qk_next = 0, pv_next = 0;
      long long idle_since = clock64();
      while (pv_next < n_tiles) {
        bool progressed = false;
        // QK of the next tile: K tile landed, S^T buffer released by the softmax
        if (qk_next < n_tiles && qk_next <= pv_next + 1) {
          const int i = qk_next, sb = i & 1;
          const bool draft_qk = has_draft && i == 0;
          const bool k_ok = draft_qk || mbar_test(bar(K_FULL), kf & 1);
          const bool s_ok = qk_half == 1 || i < 2 || mbar_test(bar(S_FREE0 + sb), sfree[sb] & 1);
          if (k_ok && s_ok) {
            if (!draft_qk) ++kf;
            if (qk_half == 0 && i >= 2) ++sfree[sb];
            tc_fence_after();
            if (KV8 && !draft_qk) {
              // quantised cache: one 128-dim half from the f16 half-tile buffer (8-row groups 2 KB apart)
#pragma unroll
              for (int k8 = 0; k8 < kDim / 32; ++k8) {
                const int kk = (kDim / 32) * qk_half + k8;
                const uint32_t off = (k8 & 3) * 32;
                umma(tmem + kColS0 + sb * NQ, sw128_desc(k_addr + (k8 >> 2) * 1024 + off, 16, kGroupB / 2),
                     sw128_desc(q_addr + (kk >> 2) * NQ * 128 + off, 16, 1024), kIdescQK, kk > 0 ? 1u : 0u);
              }
              umma_commit(bar(K_EMPTY));
              if (qk_half == 1) {
                umma_commit(bar(S_FULL0 + sb));
                ++qk_next;
              }
              qk_half ^= 1;
            } else {
#pragma unroll
              for (int kk = 0; kk < kDim / 16; ++kk) {
                // A = K, K-major: 64-dim blocks 1 KB apart, 32 bytes per 16-element step, 8-row groups 4 KB apart
                // B = Q^T, K-major, block-major: 64-dim blocks NQ * 128 B apart, 8-row groups 1 KB apart
                const uint32_t off = (kk & 3) * 32;
                umma(tmem + kColS0 + sb * NQ, sw128_desc(k_addr + (kk >> 2) * 1024 + off, 16, kGroupB),
                     sw128_desc(q_addr + (kk >> 2) * NQ * 128 + off, 16, 1024),
                     kIdescQK, kk > 0 ? 1u : 0u);
              }
              umma_commit(bar(S_FULL0 + sb));
              umma_commit(bar(K_EMPTY));
              ++qk_next;
            }
            progressed = true;
          }
        }
        // PV of the oldest tile whose P^T is written, one V half at a time
        if (pv_next < qk_next) {
          const int t = pv_next;
          const bool draft = has_draft && t == 0;
          // (quantised cache: both halves pass through the one f16 half-tile buffer of V_FULL0)
          const bool ready = pv_half == 0 ? mbar_test(bar(P_FULL), pf & 1) && (draft || mbar_test(bar(V_FULL0), vf0 & 1))
                                          : (KV8 ? mbar_test(bar(V_FULL0), vf0 & 1) : mbar_test(bar(V_FULL1), vf1 & 1));
          if (ready) {
            if (pv_half == 0) {
              ++pf;
              if (!draft) ++vf0;
            } else if (KV8) {
              ++vf0;
            } else {
              ++vf1;
            }
            tc_fence_after();
            // O += P . V over 16-token steps j0 .. j0 + steps - 1 (V rows from step vj0 of the buffer on)
            auto issue_pv = [&](const int j0, const int steps, const int vj0) {
#pragma unroll
              for (int jj = 0; jj < steps; ++jj) {
                const int j = j0 + jj;
                const uint32_t acc = (t > 0 || j > 0) ? 1u : 0u;
                // A = P (the P^T tile), MN-major: 64-column atoms 16 KB apart, 8-token groups 1 KB apart;
                // B = V, MN-major: 64-dim atoms 1 KB apart, 8-token groups 4 KB apart
                umma(tmem + kColO, sw128_desc(p_addr + j * 2048, kAtomB, 1024),
                     sw128_desc(v_addr + (j - vj0) * 2 * kGroupB, 1024, kGroupB), kIdescPV, acc);
              }
            };
            if (draft) {
              // the draft tile holds n_nodes <= 64 token rows: all in the first half
              issue_pv(0, (n_nodes + 15) >> 4, 0);
              umma_commit(bar(O_DONE));
              ++pv_next;
            } else if (pv_half == 0) {
              issue_pv(0, kT / 32, 0);
              umma_commit(bar(V_EMPTY0));
              pv_half = 1;
            } else {
              issue_pv(kT / 32, kT / 32, KV8 ? kT / 32 : 0);   // quantised cache: the half-tile buffer
              umma_commit(bar(KV8 ? V_EMPTY0 : V_EMPTY1));
              umma_commit(bar(O_DONE));
              pv_half = 0;
              ++pv_next;
            }
            progressed = true;
          }
        }
        if (progressed) {
          idle_since = clock64();
        } else {
          if (clock64() - idle_since > kWaitCycles || *(volatile int*)&sm->abort) {
            sm->abort = 1;
            report(p.dev_status, SD_DEV_TIMEOUT);
            break;
          }
          // e4m3 caches: no sleep between polls (the issue sits on the per-tile chain; 32K tree layer
          // 69.4 -> 67.7 us); bf16 caches keep a short one (measured marginally faster there)
          if constexpr (!KV8) __nanosleep(32);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    // Columns are processed in groups of 32 in loops that are not unrolled;
    // S^T is re-read from tensor memory by each pass.
    const int sw = warp - 2;                 // 0..3
    // scores to base-2 softmax units; a quantised context tile carries the K scale
    const float qk_mul = (KV8 && !has_draft) ? kScaleLog2 * p.k_scale : kScaleLog2;
    const int quarter = warp & 3;            // tensor-memory lane quarter of this warp
    const int row = quarter * 32 + lane;     // token row of S^T; query column (row of O) in the epilogue
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    // Barrier of the four softmax warps on an mbarrier, so that it is bounded too.
    int gphase = 0;
    auto group_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(GROUP));
      return mbar_spin(bar(GROUP), (uint32_t)(gphase++ & 1), &sm->abort, p.dev_status);
    };
    auto load_cols = [&](const float* arr, int col, float (&w)[32]) {
      const float4* src = reinterpret_cast<const float4*>(arr + col);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 t = src[k];
        w[4 * k] = t.x; w[4 * k + 1] = t.y; w[4 * k + 2] = t.z; w[4 * k + 3] = t.w;
      }
    };
    // Column sums of P, from the bf16 P^T tile this warp wrote (the same
    // rounded weights the PV product multiplies V with): lane L sums columns
    // 64a + 8(L%8) .. +7 of atom a over token rows 32 * quarter + L/8 + 4k,
    // k < 8; the warp's lanes and the four warps are added in the epilogue.
    float csum[NATOM][8];
#pragma unroll
    for (int a = 0; a < NATOM; ++a)
#pragma unroll
      for (int j = 0; j < 8; ++j) csum[a][j] = 0.f;
    const int cs_chunk = lane & 7;
    // Draft CTA: the tree masks, built while the QK product runs.  Node
    // `row` walks its root path (its ancestor set), then, after the group
    // barrier, gathers its descendant set: bit n set when node n has `row` on
    // its root path (itself included).
    unsigned long long my_desc = 0ull;
    bool masks_ok = true;
    if (has_draft) {
      if (row < n_nodes) {
        unsigned long long a = 1ull << row;
        int d = 0;
        bool ok = row == 0 ? sm->par[0] == -1 : true;
        for (int u = row; ok && u > 0; ++d) {
          const int pu = sm->par[u];
          ok = pu >= 0 && pu < u;
          if (ok) a |= 1ull << pu;
          u = pu;
        }
        if (!ok) { report(p.dev_status, SD_DEV_BAD_PARENTS); a = 1ull << row; d = 0; }
        sm->anc[row] = a;
        sm->depth[row] = d;
      }
      masks_ok = group_sync();
      if (row < n_nodes) {
        // with a window, a descendant n more than W - 1 levels below does not see `row`
        const int dr = sm->depth[row];
        for (int n = row; n < n_nodes; ++n)
          if (W <= 0 || sm->depth[n] - dr < W) my_desc |= ((sm->anc[n] >> row) & 1ull) << n;
      }
    }
    for (int i = 0; i < n_tiles && masks_ok; ++i) {
      const int sb = i & 1;
      if (!mbar_spin(bar(S_FULL0 + sb), (i >> 1) & 1, &sm->abort, p.dev_status)) break;
      tc_fence_after();
      const uint32_t s_addr = tmem + lane_addr + kColS0 + sb * NQ;
      const bool draft_tile = has_draft;
      const int t0 = ctx_begin + i * kT;
      const int valid = draft_tile ? n_nodes : min(kT, ctx_end - t0);
      // Visibility of this thread's token row, one bit per column of each
      // 32-column group: context rows before `valid` see every query column;
      // in the draft tile, node `row` is seen by the columns of its
      // descendants (itself included; padding columns see the root only).
      uint32_t vis[NG];
#pragma unroll
      for (int gq = 0; gq < NG; ++gq) {
        const int ncol = min(32, NQ - gq * 32);
        vis[gq] = (!draft_tile && row < valid) ? (ncol >= 32 ? 0xffffffffu : ((1u << ncol) - 1u)) : 0u;
      }
      if (!draft_tile && W > 0 && t0 < L - W + 1 + kMaxNodes) {
        // tiles inside the window's band: column q sees token t0 + row from lo_col[q] on
        const int tpos = t0 + row;
#pragma unroll
        for (int gq = 0; gq < NG; ++gq) {
          uint32_t bits = 0u;
#pragma unroll 1
          for (int e = 0; e < 32; ++e) bits |= (tpos >= sm->lo_col[gq * 32 + e] ? 1u : 0u) << e;
          vis[gq] &= bits;
        }
      }
      if (draft_tile) {
        unsigned long long d = my_desc;
        while (d != 0ull) {
          const int n = __ffsll((long long)d) - 1;
          d &= d - 1ull;
#pragma unroll
          for (int gq = 0; gq < NG; ++gq) vis[gq] |= bit_range(n * hpc - gq * 32, hpc);
        }
        if (row == 0) {
#pragma unroll
          for (int gq = 0; gq < NG; ++gq) vis[gq] |= bit_range(rows - gq * 32, NQ - rows);
        }
      }
      // Scores of 32 columns of this thread's token row, base 2, masked to -inf.
      constexpr int kStep = NG == 2 ? 2 : 1;
      auto mask_scale = [&](int g32, const float (&a)[16], const float (&cc)[16], float (&v)[32]) {
        const uint32_t vm = vis_of(vis, g32);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float raw = e < 16 ? a[e] : cc[e - 16];
          v[e] = ((vm >> e) & 1u) ? raw * qk_mul : -INFINITY;
        }
      };
      // Groups g32 and g32 + 1 under one tensor-memory wait when there are
      // exactly two (each round trip costs hundreds of cycles; with three the
      // registers would spill): kStep groups per call.
      auto load_scores2 = [&](int g32, float (&v0)[32], float (&v1)[32]) {
        float a0[16], c0[16], a1[16], c1[16];
        const bool second0 = g32 * 32 + 16 < NQ;
        const bool has1 = kStep == 2 && g32 + 1 < NG;
        const bool second1 = (g32 + 1) * 32 + 16 < NQ;
        tmem_ld16(s_addr + g32 * 32, a0);
        if (second0) tmem_ld16(s_addr + g32 * 32 + 16, c0);
        if (has1) {
          tmem_ld16(s_addr + g32 * 32 + 32, a1);
          if (second1) tmem_ld16(s_addr + g32 * 32 + 48, c1);
        }
        tmem_wait_ld();
        if (!second0) {
#pragma unroll
          for (int e = 0; e < 16; ++e) c0[e] = 0.f;
        }
        mask_scale(g32, a0, c0, v0);
        if (has1) {
          if (!second1) {
#pragma unroll
            for (int e = 0; e < 16; ++e) c1[e] = 0.f;
          }
          mask_scale(g32 + 1, a1, c1, v1);
        }
      };

      // Pass 1: does any score exceed its column's running maximum by more
      // than 2^8?  (The first tile always sets the maxima.)
      bool slow = true;
      if (i > 0) {
        float dm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
        for (int g32 = 0; g32 < NG; g32 += kStep) {
          float v0[32], v1[32], mm[32];
          load_scores2(g32, v0, v1);
          load_cols(sm->m, g32 * 32, mm);
#pragma unroll
          for (int e = 0; e < 32; ++e) dm[e & 3] = fmaxf(dm[e & 3], v0[e] - mm[e]);
          if (kStep == 2) {
            load_cols(sm->m, g32 * 32 + 32, mm);
#pragma unroll
            for (int e = 0; e < 32; ++e) dm[e & 3] = fmaxf(dm[e & 3], v1[e] - mm[e]);
          }
        }
        const float dmax = fmaxf(fmaxf(dm[0], dm[1]), fmaxf(dm[2], dm[3]));
        if (lane == 0) sm->flag[i & 1][sw] = 0;
        __syncwarp();
        if (__any_sync(0xffffffffu, dmax > kThresh) && lane == 0) sm->flag[i & 1][sw] = 1;
        if (!group_sync()) break;
        slow = (sm->flag[i & 1][0] | sm->flag[i & 1][1] | sm->flag[i & 1][2] | sm->flag[i & 1][3]) != 0;
      }
      bool pv_waited = false;
      if (slow) {
        // exact column maxima of this tile, new running maxima and rescale factors
#pragma unroll 1
        for (int g32 = 0; g32 < NG; g32 += kStep) {
          float v0[32], v1[32];
          load_scores2(g32, v0, v1);
          sm->red[sw][g32 * 32 + lane] = transpose_max32(v0, lane);
          if (kStep == 2) sm->red[sw][g32 * 32 + 32 + lane] = transpose_max32(v1, lane);
        }
        if (!group_sync()) break;
        for (int q = sw * 32 + lane; q < NQ; q += 128) {
          const float mt = fmaxf(fmaxf(sm->red[0][q], sm->red[1][q]), fmaxf(sm->red[2][q], sm->red[3][q]));
          const float mo = sm->m[q];
          const float mn = fmaxf(mo, mt);
          sm->alpha[q] = (mn == -INFINITY) ? 1.f : fast_exp2(mo - mn);
          sm->m[q] = mn;
        }
        if (!group_sync()) break;
#pragma unroll
        for (int a = 0; a < NATOM; ++a) {
          const float4 f0 = reinterpret_cast<const float4*>(sm->alpha + a * 64 + cs_chunk * 8)[0];
          const float4 f1 = reinterpret_cast<const float4*>(sm->alpha + a * 64 + cs_chunk * 8)[1];
          csum[a][0] *= f0.x; csum[a][1] *= f0.y; csum[a][2] *= f0.z; csum[a][3] *= f0.w;
          csum[a][4] *= f1.x; csum[a][5] *= f1.y; csum[a][6] *= f1.z; csum[a][7] *= f1.w;
        }
        if (i > 0) {
          // O holds earlier tiles: wait for the last PV, then rescale the rows
          // (query columns) of this warp's lane quarter, 32 dims at a time
          if (!mbar_spin(bar(O_DONE), (i - 1) & 1, &sm->abort, p.dev_status)) break;
          pv_waited = true;
          tc_fence_after();
          if (quarter * 32 < NQ) {   // warp-uniform: the quarter holds query columns
            const float al = row < NQ ? sm->alpha[row] : 1.f;
#pragma unroll 1
            for (int c = 0; c < kDim; c += 32) {
              float v0[16], v1[16];
              const uint32_t a = tmem + lane_addr + kColO + c;
              tmem_ld16(a, v0);
              tmem_ld16(a + 16, v1);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) { v0[e] *= al; v1[e] *= al; }
              tmem_st16(a, v0);
              tmem_st16(a + 16, v1);
            }
            tmem_wait_st();
          }
        }
      }
      // Pass 2: P = exp2(s - m) as the bf16 P^T row of this token.
      if (i > 0 && !pv_waited) {
        if (!mbar_spin(bar(O_DONE), (i - 1) & 1, &sm->abort, p.dev_status)) break;
      }
      auto write_p = [&](int g32, const float (&v)[32]) {
        float mm[32];
        load_cols(sm->m, g32 * 32, mm);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int ch = g32 * 4 + k;      // 16-byte chunk (8 columns) of the P^T row
          if (ch * 8 < NQ) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float p0 = fast_exp2(v[k * 8 + 2 * e] - mm[k * 8 + 2 * e]);
              const float p1 = fast_exp2(v[k * 8 + 2 * e + 1] - mm[k * 8 + 2 * e + 1]);
              if constexpr (KV8) {
                const __half2 h = __floats2half2_rn(p0, p1);
                w[e] = *reinterpret_cast<const uint32_t*>(&h);
              } else {
                const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
                w[e] = *reinterpret_cast<const uint32_t*>(&h);
              }
            }
            // MN-major P^T: atom ch/8 (64 columns), token row `row`, 16-byte chunk ch%8
            *reinterpret_cast<uint4*>(sP + (ch >> 3) * kAtomB + p_off(row, ch & 7)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      };
#pragma unroll 1
      for (int g32 = 0; g32 < NG; g32 += kStep) {
        float v0[32], v1[32];
        load_scores2(g32, v0, v1);
        write_p(g32, v0);
        if (kStep == 2) write_p(g32 + 1, v1);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(S_FREE0 + sb));
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(P_FULL));
      // Column sums of this tile's P from the rows this warp just wrote, while
      // the PV product runs (the next tile overwrites P^T only after it ends).
#pragma unroll
      for (int a = 0; a < NATOM; ++a) {
        if (a * 64 + cs_chunk * 8 < NQ) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int r = quarter * 32 + (lane >> 3) + 4 * k;
            const uint4 pv = *reinterpret_cast<const uint4*>(sP + a * kAtomB + p_off(r, cs_chunk));
            const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = KV8 ? __half22float2(*reinterpret_cast<const __half2*>(&pw[e]))
                                   : __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pw[e]));
              csum[a][2 * e] += f.x;
              csum[a][2 * e + 1] += f.y;
            }
          }
        }
      }
    }

    // ------------------------------------------------------------ epilogue
    // Thread `row` of the warps whose lane quarter holds query columns owns
    // query column q = row: its 256 dims sit in one tensor-memory lane, so it
    // normalises them by the column sum l (the four warps' partial sums, added
    // from shared memory) and writes the bf16 row (the output, or this split's
    // partial for the merge) straight to global memory, 16 bytes at a time.
    if (!*(volatile int*)&sm->abort) {
      // add the warp's four row groups (lanes with the same lane % 8), then
      // publish this warp's column sums
#pragma unroll
      for (int a = 0; a < NATOM; ++a)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          csum[a][j] += __shfl_xor_sync(0xffffffffu, csum[a][j], 8);
          csum[a][j] += __shfl_xor_sync(0xffffffffu, csum[a][j], 16);
        }
      if (lane < 8) {
#pragma unroll
        for (int a = 0; a < NATOM; ++a) {
          float4* dst = reinterpret_cast<float4*>(sm->lsum[sw] + a * 64 + lane * 8);
          dst[0] = make_float4(csum[a][0], csum[a][1], csum[a][2], csum[a][3]);
          dst[1] = make_float4(csum[a][4], csum[a][5], csum[a][6], csum[a][7]);
        }
      }
    }
    if (!*(volatile int*)&sm->abort && group_sync() &&
        mbar_spin(bar(O_DONE), (n_tiles - 1) & 1, &sm->abort, p.dev_status)) {
      tc_fence_after();
      const bool direct = nsplit == 1;
      const float o_mul = (KV8 && !has_draft) ? p.v_scale : 1.0f;   // a quantised context tile: the V scale
      const size_t part0 = (size_t)s * bd.total_nodes * kHq;
      uint8_t* gbase = reinterpret_cast<uint8_t*>(direct ? p.out : p.o_part + part0 * kDim);
      if (quarter * 32 < rows) {   // warp-uniform: the tensor-memory loads are collective
        const int q = row;
        const bool mine = q < rows;
        const float lq = mine ? sm->lsum[0][q] + sm->lsum[1][q] + sm->lsum[2][q] + sm->lsum[3][q] : 0.f;
        const float inv = lq > 0.f ? __fdividef(o_mul, lq) : 0.f;   // no visible key in this split: 0
        // The warp's 32 rows are staged in the idle K tile (16 KB per warp): the
        // 16-byte chunk ch of the lane's row at chunk ch ^ lane of its 512-byte
        // slot, so that both the per-lane writes and the per-row reads below
        // are free of bank conflicts.  Each row then leaves as one coalesced
        // 512-byte warp store instead of 32 scattered 16-byte ones.
        uint8_t* wst = sK + quarter * (32 * 512);
        const uint32_t t_row = tmem + lane_addr + kColO;
        // 128 dims per wait: each tensor-memory round trip costs hundreds of cycles
#pragma unroll 1
        for (int c = 0; c < kDim; c += 128) {
          float v[8][16];
#pragma unroll
          for (int k = 0; k < 8; ++k) tmem_ld16(t_row + c + 16 * k, v[k]);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const __nv_bfloat162 h = __floats2bfloat162_rn(v[k][2 * e] * inv, v[k][2 * e + 1] * inv);
              w[e] = *reinterpret_cast<const uint32_t*>(&h);
            }
            const int ch = (c + 16 * k) / 8;   // 16-byte chunk of the row (8 dims)
            *reinterpret_cast<uint4*>(wst + lane * 512 + ((ch ^ lane) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(wst + lane * 512 + (((ch + 1) ^ lane) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
        __syncwarp();
        // eight rows per round, their loads issued before any store; the last
        // round repeats the final row (the same bytes to the same place)
        const int nrow = min(32, rows - quarter * 32);
        const int my_out = mine ? sm->outrow[q] : 0;
#pragma unroll 1
        for (int r0 = 0; r0 < nrow; r0 += 8) {
          uint4 val[8];
          int orow[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int r = min(r0 + u, nrow - 1);
            val[u] = *reinterpret_cast<const uint4*>(wst + r * 512 + ((lane ^ r) << 4));
            orow[u] = __shfl_sync(0xffffffffu, my_out, r);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(gbase + ((size_t)orow[u] << 9) + (lane << 4)) = val[u];
        }
      }
      // log-sum-exp of query column sw * 32 + lane (base 2 for the merge)
      for (int q = sw * 32 + lane; q < rows; q += 128) {
        const float lq = sm->lsum[0][q] + sm->lsum[1][q] + sm->lsum[2][q] + sm->lsum[3][q];
        const float lse2 = sm->m[q] + fast_log2(lq);
        if (direct) {
          if (p.lse != nullptr) p.lse[sm->outrow[q]] = lse2 * kLn2;
        } else {
          p.lse_part[part0 + sm->outrow[q]] = lse2;
        }
      }
    }
  }

  tc_fence_before();
  }  // compute warps
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(sm->tmem));
  }
}


// ---------------------------------------------------------------- host side

// The driver's tensor-map encoder, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

template <int NQ, bool WIN, bool KV8>
cudaError_t launch_nq(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p, const BatchDesc& bd,
                      int hpc, int hparts, cudaStream_t st) {
  const size_t smem = tc_smem_bytes(NQ);
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<NQ, WIN, KV8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_splits * kHkv * hparts, bd.batch);
  cfg.blockDim = dim3(KV8 ? kThreads8 : kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_tc_kernel<NQ, WIN, KV8>, mk, mv, p, bd, hpc, hparts);
}

// Dispatch over the compiled query-column widths (attn_tc16.cu: bf16 caches, attn_tc8.cu: e4m3).
template <bool KV8>
cudaError_t launch_tc_kind(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p, const BatchDesc& bd,
                           cudaStream_t st) {
  const TcPlan pl = tc_plan(bd.max_nodes);
  const bool win = p.window > 0;
  switch (pl.nq) {
    case 32: return win ? launch_nq<32, true, KV8>(mk, mv, p, bd, pl.hpc, pl.hparts, st)
                        : launch_nq<32, false, KV8>(mk, mv, p, bd, pl.hpc, pl.hparts, st);
    case 48: return win ? launch_nq<48, true, KV8>(mk, mv, p, bd, pl.hpc, pl.hparts, st)
                        : launch_nq<48, false, KV8>(mk, mv, p, bd, pl.hpc, pl.hparts, st);
    case 64: return win ? launch_nq<64, true, KV8>(mk, mv, p, bd, pl.hpc, pl.hparts, st)
                        : launch_nq<64, false, KV8>(mk, mv, p, bd, pl.hpc, pl.hparts, st);
    case 80: return win ? launch_nq<80, true, KV8>(mk, mv, p, bd, pl.hpc, pl.hparts, st)
                        : launch_nq<80, false, KV8>(mk, mv, p, bd, pl.hpc, pl.hparts, st);
    case 96: return win ? launch_nq<96, true, KV8>(mk, mv, p, bd, pl.hpc, pl.hparts, st)
                        : launch_nq<96, false, KV8>(mk, mv, p, bd, pl.hpc, pl.hparts, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace sdv
