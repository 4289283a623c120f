// Split-KV verify attention over bf16 pages, one CTA per (split, KV head):
// every query head of the KV group in one tile, V streamed through a page
// ring, accumulators in tensor memory (tcgen05).
//
// What it computes is the tree/causal-masked grouped-query attention of the
// verify step: for sequence b, draft node j and query head h, softmax
// attention (scale 1/16) of q[j][h] over every context token of KV head h/6
// plus the draft nodes on j's root path.  Sources, by page title:
// «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍» (为什么我们要做这个测试:
// 24 Q / 4 KV heads, head dim 256; 关键突破: the tree mask follows each node's
// parent chain) and «Qwen3.8-27B投机解码实测：从14到159 tok/s的性能断点地图» (§2, §4:
// 16-token pages from one pool; §5.3: bottom-right causal mask of a chain).
//
// Layout of the work.  A CTA owns (split s, KV head g, head part c, sequence
// b).  The hpc query heads of the part (6 whenever 6 * N <= 144, i.e. trees
// of up to 24 nodes) times the N draft nodes form NQ (multiple of 16, <= 144)
// query columns, so each context page is read by one CTA only.  Per 128-token
// tile:
//   S^T[128 tok][NQ]      = K_tile[128 tok][256] . Q^T          (K-major A and B)
//   O^T[256 dim][NQ]     += V_tile^T[256][128 tok] . P^T[128 tok][NQ]
//                           (two M = 128 halves of the dims; MN-major A and B)
// In tensor memory: S^T in columns [0, NQ), O^T in [NQ, 3 NQ) (dims 0-127, then
// 128-255; one dim per lane).
//
// Shared memory.  Q^T (NQ x 512 B) stays for the whole CTA.  K is one 64 KB
// tile, loaded as eight 8 KB page boxes (contiguous in the cache) and released
// as soon as QK has read it.  V pages (8 KB each) go through a ring of at least
// a whole tile, released page by page as PV consumes them (a page is one
// 16-token K-step of the PV product).  P^T holds half a tile: token rows 0-63
// are written, multiplied (pages 0-3), then replaced by rows 64-127 (pages
// 4-7); its 64-column atoms use the 128-byte swizzle, and for NQ = 144 a
// 16-column tail the 32-byte swizzle.  Halving P^T is what leaves room for the
// whole-tile V ring at NQ = 144.
//
// Warp roles (256 threads): warp 0 streams K, warp 6 streams V; warp 1
// allocates tensor memory and one lane issues the QK products, warp 7 one lane
// the PV products, each blocking on exactly the barrier it needs next; warps
// 2-5 (one per tensor-memory lane quarter: thread = token row) run the online
// softmax (running per-column maxima raised, with O and l rescaled, only when
// a score exceeds them by more than 2^8) and write P^T, then in the epilogue
// (thread = one dim of every query column) normalise and store the output
// rows.  Every mbarrier wait is bounded; on expiry the kernel reports
// SD_DEV_TIMEOUT and winds down.
#pragma once

#include <cstddef>
#include <cstring>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace sdv {
namespace {

constexpr int kT = kTileTokens;        // tokens per tile
constexpr int kRingThreads = 256;
constexpr int kRWarpK = 0, kRWarpQK = 1, kRWarpV = 6, kRWarpPV = 7;
constexpr int kComputeThreads = 192;   // warps 1-5 and 7 (they stage Q^T)
constexpr int kKTileB = kT / 8 * kGroupB;   // the K tile: 16 groups of 8 rows x 4 dim blocks (64 KB)
constexpr int kPRows = kT / 2;         // P^T holds half a tile: token rows 0-63, then 64-127
constexpr int kSmemMax = 232448;       // 227 KB of dynamic shared memory per CTA
constexpr int kMaxStage = kRingMaxNQ + 2 * kMaxNodes;   // staging rows: Q^T + the draft block's K and V
constexpr int kMaxBars = 44;
constexpr float kThresh = 8.0f;        // base-2 growth of a maximum tolerated without rescaling
constexpr float kNoMax = -1.0e30f;     // the running maximum before any visible score

// Per-column state and barriers (COLS = query columns padded to 32).
template <int COLS>
struct RSmall {
  float m[COLS];          // running maximum of each query column (base-2 score units)
  float alpha[COLS];      // rescale factor of the current tile; 1/l of each column in the epilogue
  int outrow[COLS];       // output row (node row * 24 + head) of each query column (-1: padding)
  int lo_col[COLS];       // sliding window: oldest context position each query column sees
  float red[4][COLS];     // per softmax warp: column maxima of a tile; column sums in the epilogue
  uint64_t bar[kMaxBars];
  unsigned long long anc[kMaxNodes];   // bit r of anc[n]: draft node r is node n or one of its ancestors
  int par[kMaxNodes];
  int depth[kMaxNodes];
  int flag[2][4];
  uint32_t tmem;
  int abort;
};

template <int NQ>
struct Ring {
  static constexpr int NG = (NQ + 31) / 32;               // 32-column groups
  static constexpr int kCols = NG * 32;
  // P^T: 64-column atoms with the 128-byte swizzle, or (NQ > 128) 16-column
  // atoms with the 32-byte swizzle, so that one product with N = NQ reads it.
  static constexpr bool kSW32 = NQ > 128;
  static constexpr int kPAtom = kSW32 ? kPRows * 32 : kPRows * 128;   // bytes per atom
  static constexpr int kPA = kSW32 ? NQ / 16 : (NQ + 63) / 64;         // atoms
  static constexpr int kQB = NQ * 512;                     // Q^T: 4 blocks of NQ rows x 128 B
  static constexpr int kPB = kPA * kPAtom;
  static constexpr int kFixed = kQB + kPB + (int)sizeof(RSmall<kCols>);
  static constexpr int kBudget = kSmemMax - kFixed - kKTileB;
  static constexpr int RV0 = kBudget / kPageB;
  static constexpr int RV = RV0 >= 12 ? 12 : RV0 / 4 * 4;   // V pages: ring slots of four pages (half a tile)
  static constexpr int RVH = RV / 4;
  static constexpr int kNumBars = 2 * RVH + 12;
  static constexpr size_t kSmem = (size_t)kQB + (size_t)kKTileB + (size_t)RV * kPageB + kPB + sizeof(RSmall<kCols>);
  static_assert(RV >= 8, "the V ring holds at least a whole tile");
  static_assert(kNumBars <= kMaxBars, "barrier array too small");
  static_assert(kSmem <= (size_t)kSmemMax, "shared memory over 227 KB");
  static_assert(kPB >= kMaxStage * 16, "the staging table lives in the P^T region");
  static_assert(3 * NQ <= 512, "tensor memory holds S^T and both halves of O^T");
};

// WIN: compiled with the sliding-window paths (band masks, depths).
template <int NQ, bool WIN>
__global__ void __launch_bounds__(kRingThreads, 1)
attn_ring_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const AttnParams p, const BatchDesc bd, const int hpc, const int hparts) {
  using R = Ring<NQ>;
  constexpr int NG = R::NG, RV = R::RV, RVH = R::RVH;
  constexpr int kHalfB = 4 * kPageB;   // one V ring slot: four pages
  constexpr bool SW32 = R::kSW32;
  constexpr int kPAtomB = R::kPAtom;
  // column sums: 64-column atoms (a lane: 8 columns of each), or 16-column atoms (a lane: up to three)
  constexpr int NCS = SW32 ? 3 : R::kPA;
  constexpr uint32_t kColS = 0, kColO = NQ;   // tensor-memory columns: S^T, then O^T (two halves of NQ)
  // Barriers: V half-slot full / empty, then the tile-level ones.  CSUM_A / CSUM_B:
  // the warps of a half tile have read their P^T rows back (column sums).
  constexpr int B_VF = 0, B_VE = RVH;
  constexpr int K_FULL = 2 * RVH, K_EMPTY = K_FULL + 1, S_FULL = K_FULL + 2, S_FREE = K_FULL + 3,
                P_FULL_A = K_FULL + 4, O_HALF = K_FULL + 5, P_FULL_B = K_FULL + 6, O_DONE = K_FULL + 7,
                CSUM_A = K_FULL + 8, CSUM_B = K_FULL + 9, GROUP = K_FULL + 10;
  // No static shared memory: the dynamic window starts on a 1024-byte boundary
  // (the 128-byte swizzle atoms need it).
  extern __shared__ __align__(1024) uint8_t dyn_smem[];
  uint8_t* sQ = dyn_smem;
  uint8_t* sK = sQ + R::kQB;
  uint8_t* sV = sK + kKTileB;
  uint8_t* sP = sV + RV * kPageB;
  using Sm = RSmall<R::kCols>;
  Sm* sm = reinterpret_cast<Sm*>(sP + R::kPB);
  // The staging table of the prologue (row source, destination, block stride)
  // borrows the P^T region, which the softmax first writes after it.
  const __nv_bfloat16** rsrc = reinterpret_cast<const __nv_bfloat16**>(sP);
  uint32_t* rdst = reinterpret_cast<uint32_t*>(sP + 8 * kMaxStage);
  uint32_t* rblk = rdst + kMaxStage;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool producer = warp == kRWarpK || warp == kRWarpV;
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
  // the context lengths, the page table nor the context pages) a context CTA's
  // producers read those and issue their first tile's loads first, then wait;
  // its compute warps wait before they read Q or the parents, so the outputs
  // and the workspace are written only after the wait.  The draft CTA always
  // waits here.  Then the merge kernel's blocks may be scheduled (they wait for
  // this grid to finish before reading).
  const bool early = p.ctx_stable != 0 && s != 0;
  if (smem_u32(dyn_smem) & 1023u) {  // not expected; refuse rather than mis-swizzle
    if (threadIdx.x == 0) report_dep(p.dev_status, SD_DEV_TIMEOUT);
    return;
  }
  // The draft CTA (split 0) runs to the end in every case: it takes its tensor
  // memory before the wait (no global memory involved).
  if (s == 0 && warp == kRWarpQK) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&sm->tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (producer && lane == 0)
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(warp == kRWarpV ? &tm_v : &tm_k))
                 : "memory");
  if (!early) asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Split 0 attends to the draft block alone; split s >= 1 to context tokens
  // [base + (s - 1) * chunk, base + s * chunk).  The producers fetch their first
  // tile's page ids beside the context length (any entry of the row is in bounds).
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
  // valid token rows of tile i (the draft tile: the block's nodes)
  auto tile_valid = [&](int i) { return has_draft ? n_nodes : min(kT, ctx_end - (ctx_begin + i * kT)); };

  // ---------------------------------------------------------------- prologue
  if (tid == 0) {
    for (int i = 0; i < R::kNumBars; ++i) {
      const uint32_t cnt = (i == S_FREE || i == P_FULL_A || i == GROUP) ? 4u
                           : (i == P_FULL_B || i == CSUM_A || i == CSUM_B) ? 2u : 1u;
      mbar_init(smem_u32(&sm->bar[i]), cnt);
    }
    sm->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int q = tid; q < R::kCols; q += kRingThreads) {
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
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };

  // Staging of the operands that do not come by TMA, by `nthr` threads (index
  // t): Q^T (K-major, block-major; column q = node * hpc + head-in-part, zeros
  // past `rows`) and, in the draft CTA, the draft block: K rows into the K tile
  // and V rows into the first V slots (both group-major; node t = token row t).  A row table (source, destination, block
  // stride) is built first, then one pass of 16-byte copies with up to 12
  // loads in flight per thread; the last round repeats the final chunk instead
  // of branching, so the unrolled copies stay independent.
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
      rsrc[r] = src;
      rdst[r] = dst;
      rblk[r] = blk;
    }
    if (all_warps) __syncthreads();
    else asm volatile("bar.sync 3, 192;" ::: "memory");   // the compute warps
    constexpr int U = 12;
    const int tasks = n_stage * 32;
    for (int t0 = t; t0 - t < tasks; t0 += nthr * U) {
      uint4 v[U];
      uint32_t d[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int task = min(t0 + u * nthr, tasks - 1);
        const int r = task >> 5, cc = task & 31;
        const __nv_bfloat16* src = rsrc[r];
        const uint32_t off = rdst[r];
        v[u] = src != nullptr ? __ldg(reinterpret_cast<const uint4*>(src) + cc) : make_uint4(0, 0, 0, 0);
        d[u] = off + (cc >> 3) * rblk[r] + (((cc & 7) ^ ((off >> 7) & 7)) << 4);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) *reinterpret_cast<uint4*>(dyn_smem + d[u]) = v[u];
    }
  };
  if (has_draft) {
    // The draft CTA has no TMA work: all warps stage its operands.  V rows from
    // the block's end to the next 16-row boundary are zeroed (the draft tile's
    // PV product stops there; P^T is 0 on them, but 0 times stale shared
    // memory could be NaN).  K rows past the block are masked.
    stage_operands(tid, kRingThreads, true);
    const int v_end = (n_nodes + 15) & ~15;
    for (int i = tid; i < (v_end - n_nodes) * 32; i += kRingThreads)
      *reinterpret_cast<uint4*>(sV + kv_off(n_nodes + (i >> 5), i & 31)) = make_uint4(0, 0, 0, 0);
    fence_async_smem();   // plain stores above, read by the tensor core
    __syncthreads();
  }

  if (producer) {
    // ------------------------------------------------------------ producers (K: warp 0, V: warp 6)
    const bool is_k = warp == kRWarpK;
    const int n_ctx = has_draft ? 0 : n_tiles;
    const __nv_bfloat16* cache = is_k ? p.k_cache : p.v_cache;
    int page_next = page0;   // lane l < 8: page id of page l of the coming tile, fetched a tile ahead
    int fills = 0;           // K tiles, or V half tiles, issued so far (V half f goes to ring slot f % RVH)
    bool ok = true;
    for (int i = 0; i < n_ctx && ok; ++i) {
      const int t0 = ctx_begin + i * kT;
      const int valid = min(kT, ctx_end - t0);
      int page = (lane < 8 && lane * kPage < valid) ? page_next : -1;
      if (lane < 8 && i + 1 < n_ctx && lane * kPage < ctx_end - (t0 + kT))
        page_next = p.page_table[(size_t)b * p.max_pages + (((t0 + kT) >> 4) + lane)];
      bool bad = false;
      if (lane < 8 && lane * kPage < valid && (page < 0 || page >= p.num_pool_pages)) {
        if (is_k) report_dep(p.dev_status, SD_DEV_BAD_PAGE);
        page = -1;
        bad = true;
      }
      if (is_k) {
        // K: the whole tile, one 8 KB box per page.  Pages past the context are
        // not loaded (their rows are masked); pages with an id out of range
        // are zeros.
        // every lane waits (a lone waiting lane while the rest of the warp sits
        // at a warp-wide step resumed about 0.7 us after the phase completed)
        ok = mbar_wait(bar(K_EMPTY), (uint32_t)(i & 1) ^ 1u, &sm->abort, p.dev_status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint32_t tma_mask = __ballot_sync(0xffffffffu, lane < 8 && page >= 0);
        const uint32_t zero_mask = __ballot_sync(0xffffffffu, bad);
        if (zero_mask != 0u) {
          for (uint32_t zm = zero_mask; zm != 0u; zm &= zm - 1u) {
            const int pi = __ffs(zm) - 1;
            for (int e = lane; e < kPageB / 16; e += 32)
              *reinterpret_cast<uint4*>(sK + pi * kPageB + e * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_expect_tx(bar(K_FULL), (uint32_t)__popc(tma_mask) * (uint32_t)kPageB);
        __syncwarp();
        if ((tma_mask >> lane) & 1u)
          tma_load_page(smem_u32(sK + lane * kPageB), &tm_k, (page * kHkv + g) * 2, bar(K_FULL));
        ++fills;
      } else {
        // V: the tile's pages up to the last valid token, in two halves of up
        // to four pages (0-3, 4-7).  A half takes one ring slot of four pages
        // with one full and one empty barrier: it is issued once PV has
        // consumed the slot's previous half, and PV waits for it once.  A page
        // goes by TMA when it is in range and all its 16 tokens are valid
        // (the half's lanes issue their boxes together, as one warp
        // instruction); otherwise the warp copies it with plain loads first,
        // zero past the context (P is 0 there, but 0 times stale data could be
        // NaN).
        const int npg = (valid + kPage - 1) / kPage;
        const bool full = lane < npg && page >= 0 && (lane + 1) * kPage <= valid;
        for (int grp = 0; grp < 2 && grp * 4 < npg && ok; ++grp) {
          const int hs = fills % RVH;
          ok = mbar_wait(bar(B_VE + hs), ((uint32_t)(fills / RVH) & 1u) ^ 1u, &sm->abort, p.dev_status);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          uint8_t* slot = sV + hs * kHalfB;
          const bool mine = lane >= 4 * grp && lane < 4 * grp + 4 && lane < npg;
          for (uint32_t part = __ballot_sync(0xffffffffu, mine && !full); part != 0u; part &= part - 1u) {
            const int j = __ffs(part) - 1;
            const int pg = __shfl_sync(0xffffffffu, page, j);
            stage_rows(slot + (j - 4 * grp) * kPageB, 0, kPage, [&](int r) -> const __nv_bfloat16* {
              return (pg >= 0 && j * kPage + r < valid) ? cache + (((size_t)pg * kHkv + g) * kPage + r) * kDim
                                                        : nullptr;
            }, lane, 32);
          }
          fence_async_smem();
          const uint32_t tma_n = (uint32_t)__popc(__ballot_sync(0xffffffffu, mine && full));
          __syncwarp();
          if (lane == 0) mbar_expect_tx(bar(B_VF + hs), tma_n * (uint32_t)kPageB);   // the half's one arrival
          __syncwarp();
          if (mine && full)
            tma_load_page(smem_u32(slot + (lane - 4 * grp) * kPageB), &tm_v, (page * kHkv + g) * 2, bar(B_VF + hs));
          __syncwarp();
          ++fills;
        }
        if (!ok) break;
      }
      // early context loads: the later slots free up only as the compute warps (which wait) progress
      if (early && i == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
      if (__shfl_sync(0xffffffffu, *(volatile int*)&sm->abort, 0)) break;
    }
    // After an abort no copy may still be landing when the CTA ends: wait,
    // bounded, for the last fill of every slot.
    if (lane == 0 && *(volatile int*)&sm->abort) {
      const int nslots = is_k ? 1 : RVH;
      for (int j = 0; j < nslots && j < fills; ++j) {
        const int last = j + (fills - 1 - j) / nslots * nslots;   // the last fill of slot j
        const uint32_t parity = (uint32_t)(last / nslots) & 1u;
        const long long t0 = clock64();
        while (!mbar_test(bar(is_k ? K_FULL : B_VF + j), parity) && clock64() - t0 < kWaitCycles) {
        }
      }
    }
  } else {
  // ---------------------------------------------------------------- compute warps (1-5, 7)
  // While the producers fetch the first tiles, these six warps stage Q^T and
  // allocate tensor memory.
  {
    const int ct = warp == kRWarpPV ? 160 + lane : tid - 32;
    if (early) {
      // tensor memory first (no global memory), then the wait for the previous kernel
      if (warp == kRWarpQK) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&sm->tmem)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      if (W > 0)
        for (int j = ct; j < n_nodes; j += kComputeThreads) sm->par[j] = p.parents[q0 + j];
    }
    if (!has_draft) stage_operands(ct, kComputeThreads, false);
    if (W > 0) {
      // oldest visible context position of each query column: L + depth(node) - W + 1
      // (padding columns take the root's; an invalid parent chain stops the walk)
      const float inv_hpc = 1.0f / (float)hpc;
      for (int q = ct; q < R::kCols; q += kComputeThreads) {
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
    if (warp == kRWarpQK && !early && s != 0) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&sm->tmem)));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    fence_async_smem();
    tc_fence_before();
    asm volatile("bar.sync 1, 192;" ::: "memory");   // the compute warps, all arrive unconditionally
    tc_fence_after();
  }
  const uint32_t tmem = sm->tmem;
  if (warp == kRWarpQK) {
    // ------------------------------------------------------------ QK issuer
    // QK of tile i once its K tile has landed and the softmax has read S^T of tile i - 1.
    if (lane == 0) {
      constexpr uint32_t kIdQK = f16_idesc(128, NQ, 0, 0);
      const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK);
      for (int i = 0; i < n_tiles; ++i) {
        if (i > 0 && !mbar_wait(bar(S_FREE), (uint32_t)(i - 1) & 1u, &sm->abort, p.dev_status)) break;
        if (!has_draft && !mbar_wait(bar(K_FULL), (uint32_t)i & 1u, &sm->abort, p.dev_status)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kDim / 16; ++kk) {
          // A = K, K-major: 8-row groups 4 KB apart, 64-dim blocks 1 KB apart, 32 bytes per 16-dim step;
          // B = Q^T, K-major, block-major: 64-dim blocks NQ * 128 B apart, 8-row groups 1 KB apart
          const uint32_t off = (kk & 3) * 32;
          umma(tmem + kColS, sw128_desc(k_addr + (kk >> 2) * 1024 + off, 16, kGroupB),
               sw128_desc(q_addr + (kk >> 2) * NQ * 128 + off, 16, 1024), kIdQK, kk > 0 ? 1u : 0u);
        }
        if (!has_draft) umma_commit(bar(K_EMPTY));
        umma_commit(bar(S_FULL));
      }
    }
  } else if (warp == kRWarpPV) {
    // ------------------------------------------------------------ PV issuer
    // PV of tile i, one page (16 tokens) at a time, in two halves: pages 0-3
    // once P^T holds token rows 0-63 (P_FULL_A) and the half's V slot has
    // landed, then pages 4-7 once the softmax has replaced them by rows 64-127
    // (P_FULL_B).
    if (lane == 0) {
      constexpr uint32_t kIdPV = f16_idesc(128, NQ, 1, 1);
      const uint32_t v_addr = smem_u32(sV), p_addr = smem_u32(sP);
      int fills = 0;   // V halves consumed so far (half f in ring slot f % RVH)
      bool ok = true;
      for (int i = 0; i < n_tiles && ok; ++i) {
        const int npg = (tile_valid(i) + kPage - 1) / kPage;
        for (int half = 0; half < 2 && ok; ++half) {
          ok = mbar_wait(bar(half ? P_FULL_B : P_FULL_A), (uint32_t)i & 1u, &sm->abort, p.dev_status);
          if (!ok) break;
          const int nh = min(4, npg - 4 * half);   // pages of this half (none: an empty second half)
          const int hs = fills % RVH;
          if (nh > 0 && !has_draft) {
            ok = mbar_wait(bar(B_VF + hs), (uint32_t)(fills / RVH) & 1u, &sm->abort, p.dev_status);
            if (!ok) break;
          }
          tc_fence_after();
          for (int jj = 0; jj < nh; ++jj) {
            const uint32_t va = has_draft ? v_addr + (uint32_t)(4 * half + jj) * kPageB
                                          : v_addr + (uint32_t)hs * kHalfB + (uint32_t)jj * kPageB;
            const uint32_t acc = (i > 0 || half > 0 || jj > 0) ? 1u : 0u;
            const uint32_t prow = (uint32_t)jj * 16;   // the page's first row in the half tile
#pragma unroll
            for (int mb = 0; mb < 2; ++mb) {
              // A = V^T, dims mb*128.., MN-major: 64-dim atoms 1 KB apart, 8-token groups 4 KB apart;
              // B = P^T rows of the page, MN-major: column atoms kPAtomB apart, 8-token groups one atom row group apart
              const uint64_t a = sw128_desc(va + mb * 2048, 1024, kGroupB);
              const uint64_t bd = SW32 ? sw32_desc(p_addr + prow * 32, kPAtomB, 256)
                                       : sw128_desc(p_addr + prow * 128, kPAtomB, 1024);
              umma(tmem + kColO + mb * NQ, a, bd, kIdPV, acc);
            }
          }
          if (nh > 0 && !has_draft) {
            umma_commit(bar(B_VE + hs));
            ++fills;
          }
          if (!ok) break;
          umma_commit(bar(half ? O_DONE : O_HALF));
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int sw = warp - 2;                 // 0..3
    const int quarter = warp & 3;            // tensor-memory lane quarter of this warp
    const int row = quarter * 32 + lane;     // token row of S^T; dim (mod 128) of O^T in the epilogue
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + kColS;
    int gphase = 0;
    // Barrier of the four softmax warps on an mbarrier, so that it is bounded too.
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
    // Column sums of P from the bf16 tile this warp wrote (the same rounded
    // weights the PV product multiplies V with); each read is conflict-free.
    //  64-column atoms: csum[a][j] is column 64a + 8(L%8) + j, summed over the
    //    warp's token rows L/8 + 4k (k < 8);
    //  16-column atoms: csum[m][j] is column 16(L/8 + 4m) + 8(L%2) + j, summed
    //    over rows (L%8)/2 + 4k (k < 8) (a quarter warp reads four rows of one atom).
    // The lanes and the four warps are added in the epilogue.
    float csum[NCS][8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int a = 0; a < NCS; ++a) csum[a][j] = 0.f;
    auto csum_col = [&](int a) -> int {   // first column of csum[a] for this lane (>= NQ: none)
      return SW32 ? 16 * ((lane >> 3) + 4 * a) + 8 * (lane & 1) : 64 * a + 8 * (lane & 7);
    };
    // Draft CTA: the tree masks.  Node `row` walks its root path (its ancestor
    // set), then, after the group barrier, gathers its descendant set: bit n
    // set when node n has `row` on its root path (itself included).
    unsigned long long my_desc = 0ull;
    bool masks_ok = true;
    if (has_draft) {
      if (row < n_nodes) {
        unsigned long long a = 1ull << row;
        int d = 0;
        bool okp = row == 0 ? sm->par[0] == -1 : true;
        for (int u = row; okp && u > 0; ++d) {
          const int pu = sm->par[u];
          okp = pu >= 0 && pu < u;
          if (okp) a |= 1ull << pu;
          u = pu;
        }
        if (!okp) { report(p.dev_status, SD_DEV_BAD_PARENTS); a = 1ull << row; d = 0; }
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
    uint32_t pk[NQ / 2];   // this token row's bf16 P, column pairs
    for (int i = 0; i < n_tiles && masks_ok; ++i) {
      if (!mbar_spin(bar(S_FULL), (uint32_t)i & 1u, &sm->abort, p.dev_status)) break;
      tc_fence_after();
      const int t0 = ctx_begin + i * kT;
      const int valid = tile_valid(i);
      // Visibility of this thread's token row, one bit per column of each
      // 32-column group: context rows before `valid` see every query column;
      // in the draft tile, node `row` is seen by the columns of its
      // descendants (itself included; padding columns see the root only).
      uint32_t vis[NG];
#pragma unroll
      for (int gq = 0; gq < NG; ++gq) {
        const int ncol = min(32, NQ - gq * 32);
        vis[gq] = (!has_draft && row < valid) ? (ncol >= 32 ? 0xffffffffu : ((1u << ncol) - 1u)) : 0u;
      }
      if (!has_draft && W > 0 && t0 < L - W + 1 + kMaxNodes) {
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
      if (has_draft) {
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
      // Scores of group g32 of this thread's token row (32 columns, 16 for a
      // tail group), base 2, masked to -inf.
      auto load_scores = [&](int g32, float (&v)[32]) {
        float a[16], cc[16];
        const bool second = g32 * 32 + 16 < NQ;
        tmem_ld16(s_addr + g32 * 32, a);
        if (second) tmem_ld16(s_addr + g32 * 32 + 16, cc);
        tmem_wait_ld();
        const uint32_t vm = vis_of(vis, g32);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float raw = e < 16 ? a[e] : (second ? cc[e - 16] : 0.f);
          v[e] = ((vm >> e) & 1u) ? raw * kScaleLog2 : -INFINITY;
        }
      };
      // P = exp2(s - m) of group g32 into the packed row; returns the largest s - m.
      auto make_p = [&](int g32, const float (&v)[32]) -> float {
        float mm[32];
        load_cols(sm->m, g32 * 32, mm);
        float dm = -INFINITY;
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          if (g32 * 32 + e < NQ) {
            const float d0 = v[e] - mm[e], d1 = v[e + 1] - mm[e + 1];
            dm = fmaxf(dm, fmaxf(d0, d1));
            const __nv_bfloat162 h = __floats2bfloat162_rn(fast_exp2(d0), fast_exp2(d1));
            pk[(g32 * 32 + e) / 2] = *reinterpret_cast<const uint32_t*>(&h);
          }
        }
        return dm;
      };
      // Fast pass (every tile after the first, and the first one of a plain
      // context split): P with the running maxima, and whether any score
      // exceeds its column's maximum by more than 2^8.  A context tile outside
      // a window's band has no per-element mask (a token row is visible to
      // every column or to none), so its scores go straight from tensor memory
      // into exp2(s * scale - m), 64 columns per tensor-memory wait.
      bool slow = true;
      const bool plain = !has_draft && !(W > 0 && t0 < L - W + 1 + kMaxNodes);
      if (i == 0 && plain) {
        // The running maxima start at token row 0's scores (every column sees
        // that token).  Any score more than 2^8 above them takes the exact
        // path below, as in a later tile, so this only saves the three-pass
        // maximum search of the first tile in the common case.
        if (quarter == 0) {
#pragma unroll 1
          for (int c0 = 0; c0 < NQ / 16; ++c0) {
            float a[16];
            tmem_ld16(s_addr + c0 * 16, a);
            tmem_wait_ld();
            if (lane == 0) {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                reinterpret_cast<float4*>(sm->m + c0 * 16)[k] =
                    make_float4(a[4 * k] * kScaleLog2, a[4 * k + 1] * kScaleLog2, a[4 * k + 2] * kScaleLog2,
                                a[4 * k + 3] * kScaleLog2);
            }
          }
        }
        if (!group_sync()) break;
      }
      if (i > 0 || plain) {
        float dmax = -INFINITY;
        if (plain) {
          constexpr int NC = NQ / 16;   // 16-column chunks
#pragma unroll
          for (int c0 = 0; c0 < NC; c0 += 4) {
            float a[4][16];
#pragma unroll
            for (int c = 0; c < 4; ++c)
              if (c0 + c < NC) tmem_ld16(s_addr + (c0 + c) * 16, a[c]);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              if (c0 + c < NC) {
                const int col = (c0 + c) * 16;
                float mm[16];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const float4 m4 = reinterpret_cast<const float4*>(sm->m + col)[k];
                  mm[4 * k] = m4.x; mm[4 * k + 1] = m4.y; mm[4 * k + 2] = m4.z; mm[4 * k + 3] = m4.w;
                }
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                  const float d0 = fmaf(a[c][e], kScaleLog2, -mm[e]);
                  const float d1 = fmaf(a[c][e + 1], kScaleLog2, -mm[e + 1]);
                  dmax = fmaxf(dmax, fmaxf(d0, d1));
                  const __nv_bfloat162 h = __floats2bfloat162_rn(fast_exp2(d0), fast_exp2(d1));
                  pk[(col + e) / 2] = *reinterpret_cast<const uint32_t*>(&h);
                }
              }
            }
          }
          if (row >= valid) {   // past the context: no weight (whatever the stale scores were)
#pragma unroll
            for (int k = 0; k < NQ / 2; ++k) pk[k] = 0u;
            dmax = -INFINITY;
          }
        } else {
#pragma unroll
          for (int g32 = 0; g32 < NG; ++g32) {
            float v[32];
            load_scores(g32, v);
            dmax = fmaxf(dmax, make_p(g32, v));
          }
        }
        if (lane == 0) sm->flag[i & 1][sw] = 0;
        __syncwarp();
        if (__any_sync(0xffffffffu, dmax > kThresh) && lane == 0) sm->flag[i & 1][sw] = 1;
        if (!group_sync()) break;
        slow = (sm->flag[i & 1][0] | sm->flag[i & 1][1] | sm->flag[i & 1][2] | sm->flag[i & 1][3]) != 0;
      }
      if (slow) {
        // exact column maxima of this tile, new running maxima and rescale factors
#pragma unroll 1
        for (int g32 = 0; g32 < NG; ++g32) {
          float v[32];
          load_scores(g32, v);
          sm->red[sw][g32 * 32 + lane] = transpose_max32(v, lane);
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
        for (int g32 = 0; g32 < NG; ++g32) {
          float v[32];
          load_scores(g32, v);
          make_p(g32, v);
        }
      }
      // S^T is read: the next tile's QK may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(S_FREE));
      // P^T and O belong to the previous tile's PV until it has finished
      if (i > 0 && !mbar_spin(bar(O_DONE), (uint32_t)(i - 1) & 1u, &sm->abort, p.dev_status)) break;
      tc_fence_after();
      if (slow && i > 0) {
        // rescale what O^T and the column sums hold to the new maxima: this
        // thread's dim (both halves) across every query column
#pragma unroll
        for (int a = 0; a < NCS; ++a) {
          const int c0 = csum_col(a);
          if (c0 < NQ) {
            const float4 f0 = reinterpret_cast<const float4*>(sm->alpha + c0)[0];
            const float4 f1 = reinterpret_cast<const float4*>(sm->alpha + c0)[1];
            csum[a][0] *= f0.x; csum[a][1] *= f0.y; csum[a][2] *= f0.z; csum[a][3] *= f0.w;
            csum[a][4] *= f1.x; csum[a][5] *= f1.y; csum[a][6] *= f1.z; csum[a][7] *= f1.w;
          }
        }
#pragma unroll 1
        for (int mb = 0; mb < 2; ++mb) {
#pragma unroll 1
          for (int q = 0; q < NQ; q += 16) {
            float v[16];
            const uint32_t ad = tmem + lane_addr + kColO + mb * NQ + q;
            tmem_ld16(ad, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] *= sm->alpha[q + e];
            tmem_st16(ad, v);
          }
        }
        tmem_wait_st();
      }
      // P^T holds half a tile: the warps of token rows 0-63 (lane quarters 0
      // and 1) write theirs first; the warps of rows 64-127 signal that their
      // rescale (if any) is done, wait until the PV product and the first
      // warps' column sums have read rows 0-63, then write theirs into the same
      // rows of P^T.  The next tile's first warps wait in turn for the PV
      // product and these warps' column sums.
      const bool second_half = quarter >= 2;
      const int hr = row & (kPRows - 1);   // row within the half tile
      if (second_half) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(P_FULL_A));
        if (!mbar_spin(bar(O_HALF), (uint32_t)i & 1u, &sm->abort, p.dev_status)) break;
        if (!mbar_spin(bar(CSUM_A), (uint32_t)i & 1u, &sm->abort, p.dev_status)) break;
      } else if (i > 0) {
        if (!mbar_spin(bar(CSUM_B), (uint32_t)(i - 1) & 1u, &sm->abort, p.dev_status)) break;
      }
      // P^T row of this token, 16 bytes (8 columns) at a time
#pragma unroll
      for (int ch = 0; ch < NQ / 8; ++ch) {
        const uint4 w = make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        const uint32_t off = SW32 ? (uint32_t)((ch >> 1) * kPAtomB + hr * 32 + (((ch & 1) ^ ((hr >> 2) & 1)) << 4))
                                  : (uint32_t)((ch >> 3) * kPAtomB) + p_off(hr, ch & 7);
        *reinterpret_cast<uint4*>(sP + off) = w;
      }
      tc_fence_before();
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(second_half ? P_FULL_B : P_FULL_A));
      // Column sums of this tile's P from the rows this warp just wrote (the
      // same bf16 weights the PV product multiplies V with), while PV runs.
#pragma unroll
      for (int a = 0; a < NCS; ++a) {
        if (csum_col(a) < NQ) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            uint32_t off;
            if (SW32) {
              const int r = (quarter & 1) * 32 + ((lane & 7) >> 1) + 4 * k;
              off = (uint32_t)(((lane >> 3) + 4 * a) * kPAtomB + r * 32 + (((lane & 1) ^ ((r >> 2) & 1)) << 4));
            } else {
              const int r = (quarter & 1) * 32 + (lane >> 3) + 4 * k;
              off = (uint32_t)(a * kPAtomB) + p_off(r, lane & 7);
            }
            const uint4 pv = *reinterpret_cast<const uint4*>(sP + off);
            const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pw[e]));
              csum[a][2 * e] += f.x;
              csum[a][2 * e + 1] += f.y;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(second_half ? CSUM_B : CSUM_A));
    }

    // ------------------------------------------------------------ epilogue
    // Column sums l: the lanes with the same columns, then the four warps
    // (through red[], free now).  Thread `row` then holds dim `row` (and
    // 128 + row) of every query column in its tensor-memory lane; it scales by
    // 1/l and adjacent lanes pair their dims, so that each 4-byte store writes
    // two dims of one output row (64 bytes per row per store instruction).
    bool ok_epi = !*(volatile int*)&sm->abort;
    if (ok_epi) {
      // lanes holding the same columns: L/8 for 64-column atoms, (L%8)/2 for 16-column atoms
#pragma unroll
      for (int a = 0; a < NCS; ++a)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          csum[a][j] += __shfl_xor_sync(0xffffffffu, csum[a][j], SW32 ? 2 : 8);
          csum[a][j] += __shfl_xor_sync(0xffffffffu, csum[a][j], SW32 ? 4 : 16);
        }
      // red[] may still be read by another warp's last max reduction: barrier first
      ok_epi = group_sync();
      if (ok_epi) {
        if (SW32 ? (lane & 6) == 0 : lane < 8) {
#pragma unroll
          for (int a = 0; a < NCS; ++a) {
            const int c0 = csum_col(a);
            if (c0 < NQ) {
              float4* dst = reinterpret_cast<float4*>(&sm->red[sw][c0]);
              dst[0] = make_float4(csum[a][0], csum[a][1], csum[a][2], csum[a][3]);
              dst[1] = make_float4(csum[a][4], csum[a][5], csum[a][6], csum[a][7]);
            }
          }
        }
        ok_epi = group_sync();
      }
    }
    if (ok_epi && mbar_spin(bar(O_DONE), (uint32_t)(n_tiles - 1) & 1u, &sm->abort, p.dev_status)) {
      tc_fence_after();
      const bool direct = nsplit == 1;
      const size_t part0 = (size_t)s * bd.total_nodes * kHq;
      // 1/l and the log-sum-exp of each query column (base 2 for the merge); a
      // column with no visible key in this split gives 0 and -inf
      for (int q = sw * 32 + lane; q < NQ; q += 128) {
        const float lq = sm->red[0][q] + sm->red[1][q] + sm->red[2][q] + sm->red[3][q];
        sm->alpha[q] = lq > 0.f ? 1.0f / lq : 0.f;
        if (q < rows) {
          const float lse2 = sm->m[q] + fast_log2(lq);
          if (direct) {
            if (p.lse != nullptr) p.lse[sm->outrow[q]] = lse2 * kLn2;
          } else {
            p.lse_part[part0 + sm->outrow[q]] = lse2;
          }
        }
      }
      if (group_sync()) {
        uint8_t* gbase = reinterpret_cast<uint8_t*>(direct ? p.out : p.o_part + part0 * kDim);
        const bool odd = (lane & 1) != 0;
        const int dpair = (row & ~1) * 2;   // byte offset of this lane pair's two dims
        const int nq16 = (rows + 15) / 16;
#pragma unroll 1
        for (int mb = 0; mb < 2; ++mb) {
#pragma unroll 1
          for (int q16 = 0; q16 < nq16; ++q16) {
            const int qb = q16 * 16;
            float v[16];
            tmem_ld16(tmem + lane_addr + kColO + mb * NQ + qb, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float ev = v[2 * k] * sm->alpha[qb + 2 * k];
              const float od = v[2 * k + 1] * sm->alpha[qb + 2 * k + 1];
              // even lanes keep the even column and take the odd lane's dim of it; odd lanes the reverse
              const float recv = __shfl_xor_sync(0xffffffffu, odd ? ev : od, 1);
              const float lo = odd ? recv : ev, hi = odd ? od : recv;
              const int q = qb + 2 * k + (odd ? 1 : 0);
              if (q < rows) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
                *reinterpret_cast<uint32_t*>(gbase + ((size_t)sm->outrow[q] << 9) + mb * 256 + dpair) =
                    *reinterpret_cast<const uint32_t*>(&h);
              }
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  }  // compute warps
  __syncthreads();
  if (warp == kRWarpQK) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(sm->tmem));
  }
}

}  // namespace
}  // namespace sdv
