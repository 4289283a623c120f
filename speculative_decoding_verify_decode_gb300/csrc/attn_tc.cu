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
// b): hpc query heads of group g (6, 3, 2 or 1, so that hpc * N <= 112)
// times the sequence's N draft nodes form NQ (multiple of 16) query columns.
// Tokens are the MMA's M dimension ("swap-AB"), so a 128-token K/V tile
// serves every query column at once:
//   S^T[128 tok][NQ]   = K_tile[128 tok][256]  . Q^T          (K-major A and B)
//   O^T[256 dim][NQ]  += V_tile^T[256][128 tok] . P^T[128][NQ]  (MN-major A and B)
// S^T (double-buffered) and O^T live in tensor memory: 4 * NQ <= 448 of the
// 512 columns.  When a sequence needs several CTAs for its query heads (hpc
// < 6), the CTAs of one split are adjacent in launch order and read the same
// pages while they are still in L2.
//
// Warp roles (192 threads): warp 0 streams K/V pages with TMA (16 tokens x
// 64 dims per box, 128-byte swizzle), warp 1 allocates tensor memory and one
// lane issues every tcgen05.mma, warps 2-5 (one per tensor-memory lane
// quarter, thread = token row) run the online softmax: masking, a running
// per-column maximum that is only raised (and O^T rescaled) when a score
// exceeds it by more than 2^8, exp2, column sums by a warp transpose-reduce,
// and the bf16 P^T tile for the PV product.  Every wait on an mbarrier is
// bounded; on expiry the kernel reports SD_DEV_TIMEOUT and winds down.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace sdv {
namespace {

constexpr int kT = 128;                 // tokens per tile
constexpr int kRegionB = kT * 128;      // one 64-dim block of a K/V tile: 16 KB
constexpr int kTileB = 4 * kRegionB;    // 64 KB
constexpr int kThreads = 192;
constexpr float kThresh = 8.0f;         // base-2 growth of the max tolerated without rescaling
constexpr long long kWaitCycles = 2000000000LL;  // about a second at GB300 clocks

enum Bar { K_FULL, K_EMPTY, V_FULL, V_EMPTY, S_FULL0, S_FULL1, S_FREE0, S_FREE1, P_FULL, O_DONE, GROUP, NUM_BARS };

struct Small {
  uint64_t bar[NUM_BARS];
  uint64_t anc[kMaxNodes];
  float m[kTcMaxNQ];
  float alpha[kTcMaxNQ];
  float red[4][kTcMaxNQ];
  int colnode[kTcMaxNQ];
  int flag[2][4];
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------ mbarrier / TMA

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false (and the CTA's abort flag set) if the phase never completes.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, Small* sm, int* status) {
  if (mbar_try(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (clock64() - t0 > kWaitCycles || *(volatile int*)&sm->abort) {
      sm->abort = 1;
      report(status, SD_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// ------------------------------------------------------------ tcgen05

// Shared-memory matrix descriptor, 128-byte swizzle: start, leading and
// stride byte offsets (16-byte units), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: bf16 x bf16 -> f32, M x N, operand majors.
__host__ __device__ constexpr uint32_t f16_idesc(int m, int n, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 16 consecutive 32-bit columns -> 16 registers per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }


// Byte offset of 16-byte chunk cc (0..7) of row r inside a 128-byte-swizzled
// block whose rows are 128 bytes apart (8-row groups 1024 bytes apart).
__device__ __forceinline__ uint32_t sw_off(int r, int cc) {
  return (uint32_t)(r * 128 + ((cc ^ (r & 7)) << 4));
}

// Copy one 512-byte row (256 bf16) into a K-major tile of `rows_per_block`
// rows per 64-dim block, or zero it when src is null.  One lane moves 16 B.
__device__ __forceinline__ void put_row_chunk(uint8_t* base, int rows_per_block, int r, int c,
                                              const __nv_bfloat16* src) {
  uint4 v = make_uint4(0, 0, 0, 0);
  if (src != nullptr) v = *reinterpret_cast<const uint4*>(src + c * 8);
  *reinterpret_cast<uint4*>(base + (c >> 3) * rows_per_block * 128 + sw_off(r, c & 7)) = v;
}

// Reduce 32 values per lane across the warp so that lane L ends with the
// sum (or max) over all lanes of value L (transpose-reduce, 31 shuffles).
template <bool kMax>
__device__ __forceinline__ float transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool up = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, half);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

template <int NQ>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const AttnParams p, const BatchDesc bd, const int hpc, const int hparts) {
  constexpr int NG = (NQ + 31) / 32;          // 32-column groups
  constexpr int NATOM = (NQ + 63) / 64;       // 64-column atoms of the P^T tile
  constexpr int kQB = NQ * 512;               // Q^T: 4 blocks of NQ rows x 128 B
  extern __shared__ uint8_t dyn_smem[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sK = sQ + kQB;
  uint8_t* sV = sK + kTileB;
  uint8_t* sP = sV + kTileB;
  Small* sm = reinterpret_cast<Small*>(sP + NATOM * kRegionB);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bid = blockIdx.x;
  const int c = bid % hparts;
  const int g = (bid / hparts) % kHkv;
  const int s = bid / (hparts * kHkv);
  const int b = blockIdx.y;
  const int q0 = bd.q_indptr[b];
  const int n_nodes = bd.q_indptr[b + 1] - q0;
  const int rows = hpc * n_nodes;
  if (c * hpc >= kGroup) return;
  int L = p.ctx_lens[b];
  if (L < 0 || L > p.max_pages * kPage) {
    if (s == 0 && c == 0 && g == 0 && tid == 0) report(p.dev_status, SD_DEV_BAD_CTX);
    L = L < 0 ? 0 : p.max_pages * kPage;
  }
  const int nsplit = active_splits(L, p.chunk);
  if (s >= nsplit) return;
  const int ctx_begin = s * p.chunk;
  const int ctx_end = min(L, ctx_begin + p.chunk);
  const bool has_draft = (s == 0);
  const int n_ctx_tiles = ctx_end > ctx_begin ? (ctx_end - ctx_begin + kT - 1) / kT : 0;
  const int n_tiles = n_ctx_tiles + (has_draft ? 1 : 0);
  const int head0 = g * kGroup + c * hpc;

  // ---------------------------------------------------------------- prologue
  if (tid == 0) {
    for (int i = 0; i < NUM_BARS; ++i) {
      const uint32_t cnt = (i == S_FREE0 || i == S_FREE1 || i == P_FULL || i == GROUP) ? 4u : 1u;
      mbar_init(smem_u32(&sm->bar[i]), cnt);
    }
    sm->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int q = tid; q < NQ; q += kThreads) {
    sm->m[q] = -INFINITY;
    sm->colnode[q] = q < rows ? q / hpc : -1;
  }
  if (has_draft && tid < n_nodes) {
    // ancestor bitmask of node tid (bit i: i is tid or an ancestor of tid)
    uint64_t mask = 1ull << tid;
    bool ok = true;
    if (tid == 0) {
      ok = p.parents[q0] == -1;
    } else {
      int u = tid;
      while (u > 0) {
        const int pu = p.parents[q0 + u];
        if (pu < 0 || pu >= u) { ok = false; break; }
        mask |= 1ull << pu;
        u = pu;
      }
    }
    if (!ok) { report(p.dev_status, SD_DEV_BAD_PARENTS); mask = 1ull << tid; }
    sm->anc[tid] = mask;
  }
  // Q^T (K-major): column q = node * hpc + head-in-part; zero columns past `rows`.
  for (int task = tid; task < NQ * 32; task += kThreads) {
    const int q = task >> 5, ch = task & 31;
    const __nv_bfloat16* src = nullptr;
    if (q < rows) src = p.q + ((size_t)(q0 + q / hpc) * kHq + head0 + q % hpc) * kDim;
    put_row_chunk(sQ, NQ, q, ch, src);
  }
  if (has_draft) {  // the draft block is tile 0 of split 0: node t is token row t
    for (int task = tid; task < kT * 32; task += kThreads) {
      const int t = task >> 5, ch = task & 31;
      const bool valid = t < n_nodes;
      const size_t off = ((size_t)(q0 + (valid ? t : 0)) * kHkv + g) * kDim;
      put_row_chunk(sK, kT, t, ch, valid ? p.k_new + off : nullptr);
      put_row_chunk(sV, kT, t, ch, valid ? p.v_new + off : nullptr);
    }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&sm->tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem;
  const uint32_t bars = smem_u32(&sm->bar[0]);
  auto bar = [&](int i) { return bars + 8u * i; };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int ek = 0, ev = 0;
    const int first = has_draft ? 1 : 0;
    const uint32_t init_full = has_draft ? 1u : 0u;
    for (int i = first; i < n_tiles; ++i) {
      const int t0 = ctx_begin + (i - first) * kT;
      const int valid = min(kT, ctx_end - t0);
      int page = -1;
      if (lane < 8 && lane * kPage < valid) {
        page = p.page_table[(size_t)b * p.max_pages + ((t0 >> 4) + lane)];
        if (page < 0 || page >= p.num_pool_pages) { report(p.dev_status, SD_DEV_BAD_PAGE); page = -1; }
      }
      // a page goes by TMA when it is in range and all 16 of its tokens are valid
      const bool page_full = page >= 0 && (lane + 1) * kPage <= valid;
      const uint32_t tma_mask = __ballot_sync(0xffffffffu, lane < 8 && page_full);
      for (int kv = 0; kv < 2; ++kv) {
        uint8_t* dst = kv == 0 ? sK : sV;
        const int e = kv == 0 ? ek++ : ev++;
        const uint32_t parity = (uint32_t)(e & 1) ^ init_full ^ 1u;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(bar(kv == 0 ? K_EMPTY : V_EMPTY), parity, sm, p.dev_status);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        // pages that are partial, missing or out of range: plain copies, zero past the context
        for (int pi = 0; pi < 8; ++pi) {
          if (tma_mask & (1u << pi)) continue;
          const int pg = __shfl_sync(0xffffffffu, page, pi);
          const __nv_bfloat16* cache = kv == 0 ? p.k_cache : p.v_cache;
          for (int task = lane; task < kPage * 32; task += 32) {
            const int slot = task >> 5, ch = task & 31;
            const int tok = pi * kPage + slot;
            const __nv_bfloat16* src = nullptr;
            if (pg >= 0 && tok < valid) src = cache + (((size_t)pg * kHkv + g) * kPage + slot) * kDim;
            put_row_chunk(dst, kT, tok, ch, src);
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0)
          mbar_expect_tx(bar(kv == 0 ? K_FULL : V_FULL), (uint32_t)__popc(tma_mask) * (kPage * 512));
        // issue the TMA boxes (page ids live in lanes 0..7)
        for (int pi = 0; pi < 8; ++pi) {
          const int pg = __shfl_sync(0xffffffffu, page, pi);
          if (lane == 0 && (tma_mask & (1u << pi))) {
            const CUtensorMap* map = kv == 0 ? &tm_k : &tm_v;
            const int y = (pg * kHkv + g) * kPage;
#pragma unroll
            for (int blk = 0; blk < 4; ++blk)
              tma_load_2d(smem_u32(dst + blk * kRegionB + pi * kPage * 128), map, blk * 64, y,
                          bar(kv == 0 ? K_FULL : V_FULL));
          }
        }
      }
      if (__shfl_sync(0xffffffffu, sm->abort, 0)) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescQK = f16_idesc(128, NQ, 0, 0);
      constexpr uint32_t kIdescPV = f16_idesc(128, NQ, 1, 1);
      const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV), p_addr = smem_u32(sP);
      int kf = 0, vf = 0, pf = 0;
      int sfree[2] = {0, 0};
      auto pv = [&](int t) -> bool {
        if (!mbar_wait(bar(P_FULL), pf & 1, sm, p.dev_status)) return false;
        ++pf;
        if (!(has_draft && t == 0)) {
          if (!mbar_wait(bar(V_FULL), vf & 1, sm, p.dev_status)) return false;
          ++vf;
        }
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int j = 0; j < kT / 16; ++j) {
            // A = V^T rows 128h.., MN-major: 64-dim atoms 16 KB apart, 8-token groups 1 KB apart
            const uint64_t a = sw128_desc(v_addr + 2 * h * kRegionB + j * 2048, kRegionB, 1024);
            // B = P^T, MN-major: 64-column atoms 16 KB apart, 8-token groups 1 KB apart
            const uint64_t bd_ = sw128_desc(p_addr + j * 2048, kRegionB, 1024);
            umma(tmem + 2 * NQ + h * NQ, a, bd_, kIdescPV, (t > 0 || j > 0) ? 1u : 0u);
          }
        }
        umma_commit(bar(V_EMPTY));
        umma_commit(bar(O_DONE));
        return true;
      };
      bool ok = true;
      for (int i = 0; i < n_tiles && ok; ++i) {
        const int sb = i & 1;
        if (!(has_draft && i == 0)) {
          if (!mbar_wait(bar(K_FULL), kf & 1, sm, p.dev_status)) break;
          ++kf;
        }
        if (i >= 2) {
          if (!mbar_wait(bar(S_FREE0 + sb), sfree[sb] & 1, sm, p.dev_status)) break;
          ++sfree[sb];
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kDim / 16; ++kk) {
          // K-major: 64-dim blocks, 32 bytes per 16-element step, 8-row groups 1 KB apart
          const uint64_t a = sw128_desc(k_addr + (kk >> 2) * kRegionB + (kk & 3) * 32, 16, 1024);
          const uint64_t bq = sw128_desc(q_addr + (kk >> 2) * NQ * 128 + (kk & 3) * 32, 16, 1024);
          umma(tmem + sb * NQ, a, bq, kIdescQK, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(S_FULL0 + sb));
        umma_commit(bar(K_EMPTY));
        if (i >= 1) ok = pv(i - 1);
      }
      if (ok && !sm->abort && n_tiles > 0) pv(n_tiles - 1);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int sw = warp - 2;                 // 0..3
    const int quarter = warp & 3;            // tensor-memory lane quarter of this warp
    const int row = quarter * 32 + lane;     // token row of S^T / dim row of O^T
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    // Barrier of the four softmax warps on an mbarrier, so that it is bounded too.
    int gphase = 0;
    auto group_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(GROUP));
      return mbar_wait(bar(GROUP), (uint32_t)(gphase++ & 1), sm, p.dev_status);
    };
    float lcol[NG];
#pragma unroll
    for (int i = 0; i < NG; ++i) lcol[i] = 0.f;
    for (int i = 0; i < n_tiles; ++i) {
      const int sb = i & 1;
      if (!mbar_wait(bar(S_FULL0 + sb), (i >> 1) & 1, sm, p.dev_status)) break;
      tc_fence_after();
      float sv[NG * 32];
#pragma unroll
      for (int c16 = 0; c16 < NQ / 16; ++c16) {
        float v[16];
        tmem_ld16(tmem + lane_addr + sb * NQ + c16 * 16, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) sv[c16 * 16 + e] = v[e];
      }
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(S_FREE0 + sb));

      // mask, scale, and check whether any score outgrows its column maximum
      const bool draft_tile = has_draft && i == 0;
      const int t0 = ctx_begin + (i - (has_draft ? 1 : 0)) * kT;
      const int valid = draft_tile ? n_nodes : min(kT, ctx_end - t0);
      bool over = false;
#pragma unroll
      for (int q = 0; q < NG * 32; ++q) {
        float x = -INFINITY;
        if (q < NQ) {
          bool vis = row < valid;
          if (draft_tile) {
            const int node = sm->colnode[q];
            vis = node >= 0 ? (row < n_nodes && ((sm->anc[node] >> row) & 1ull)) : row == 0;
          }
          if (vis) x = sv[q] * kScaleLog2;
          over |= x - sm->m[q] > kThresh;
        }
        sv[q] = x;
      }
      if (lane == 0) sm->flag[i & 1][sw] = 0;
      __syncwarp();
      if (__any_sync(0xffffffffu, over) && lane == 0) sm->flag[i & 1][sw] = 1;
      if (!group_sync()) break;
      const bool slow = (sm->flag[i & 1][0] | sm->flag[i & 1][1] | sm->flag[i & 1][2] | sm->flag[i & 1][3]) != 0;
      bool pv_waited = false;
      if (slow) {
        // exact column maxima of this tile, new running maxima and rescale factors
#pragma unroll
        for (int gq = 0; gq < NG; ++gq) {
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = sv[gq * 32 + e];
          const float mx = transpose_reduce32<true>(v, lane);
          if (gq * 32 + lane < NQ) sm->red[sw][gq * 32 + lane] = mx;
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
        for (int gq = 0; gq < NG; ++gq)
          if (gq * 32 + lane < NQ) lcol[gq] *= sm->alpha[gq * 32 + lane];
        if (i > 0) {
          // O^T holds PV of earlier tiles: wait for the last one, then rescale its columns
          if (!mbar_wait(bar(O_DONE), (i - 1) & 1, sm, p.dev_status)) break;
          pv_waited = true;
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int c16 = 0; c16 < NQ / 16; ++c16) {
              float v[16];
              const uint32_t a = tmem + lane_addr + 2 * NQ + h * NQ + c16 * 16;
              tmem_ld16(a, v);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] *= sm->alpha[c16 * 16 + e];
              tmem_st16(a, v);
            }
          }
          tmem_wait_st();
        }
      }
      // P = exp2(s - m): column sums, then the bf16 P^T row of this token
#pragma unroll
      for (int q = 0; q < NG * 32; ++q) sv[q] = q < NQ ? fast_exp2(sv[q] - sm->m[q]) : 0.f;
#pragma unroll
      for (int gq = 0; gq < NG; ++gq) {
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = sv[gq * 32 + e];
        lcol[gq] += transpose_reduce32<false>(v, lane);
      }
      if (i > 0 && !pv_waited) {
        if (!mbar_wait(bar(O_DONE), (i - 1) & 1, sm, p.dev_status)) break;
      }
#pragma unroll
      for (int ch = 0; ch < NQ / 8; ++ch) {
        uint4 v;
        __nv_bfloat162 h0 = __floats2bfloat162_rn(sv[ch * 8 + 0], sv[ch * 8 + 1]);
        __nv_bfloat162 h1 = __floats2bfloat162_rn(sv[ch * 8 + 2], sv[ch * 8 + 3]);
        __nv_bfloat162 h2 = __floats2bfloat162_rn(sv[ch * 8 + 4], sv[ch * 8 + 5]);
        __nv_bfloat162 h3 = __floats2bfloat162_rn(sv[ch * 8 + 6], sv[ch * 8 + 7]);
        v.x = *reinterpret_cast<uint32_t*>(&h0);
        v.y = *reinterpret_cast<uint32_t*>(&h1);
        v.z = *reinterpret_cast<uint32_t*>(&h2);
        v.w = *reinterpret_cast<uint32_t*>(&h3);
        // MN-major P^T: atom ch/8 (64 columns), token row `row`, 16-byte chunk ch%8
        *reinterpret_cast<uint4*>(sP + (ch >> 3) * kRegionB + sw_off(row, ch & 7)) = v;
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(P_FULL));
    }

    // ------------------------------------------------------------ epilogue
    // (every wait is bounded, so warps that disagree after an abort cannot hang)
    if (!*(volatile int*)&sm->abort) {
#pragma unroll
      for (int gq = 0; gq < NG; ++gq)
        if (gq * 32 + lane < NQ) sm->red[sw][gq * 32 + lane] = lcol[gq];
      bool done = group_sync();
      for (int q = sw * 32 + lane; q < NQ; q += 128)
        sm->alpha[q] = sm->red[0][q] + sm->red[1][q] + sm->red[2][q] + sm->red[3][q];  // column sums
      done = group_sync() && done;
      done = done && mbar_wait(bar(O_DONE), (n_tiles - 1) & 1, sm, p.dev_status);
      tc_fence_after();
      if (done) {
        const bool direct = nsplit == 1;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int c16 = 0; c16 < NQ / 16; ++c16) {
            float v[16];
            tmem_ld16(tmem + lane_addr + 2 * NQ + h * NQ + c16 * 16, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int q = c16 * 16 + e;
              if (q >= rows) continue;
              const int r = q0 + q / hpc;
              const int head = head0 + q % hpc;
              const float o = v[e] / sm->alpha[q];
              const int d = h * 128 + row;
              if (direct) p.out[((size_t)r * kHq + head) * kDim + d] = __float2bfloat16_rn(o);
              else p.o_part[(((size_t)s * bd.total_nodes + r) * kHq + head) * kDim + d] = o;
            }
          }
        }
        for (int q = sw * 32 + lane; q < rows; q += 128) {
          const int r = q0 + q / hpc;
          const int head = head0 + q % hpc;
          const float lse2 = sm->m[q] + fast_log2(sm->alpha[q]);
          if (direct) {
            if (p.lse != nullptr) p.lse[(size_t)r * kHq + head] = lse2 * kLn2;
          } else {
            p.lse_part[((size_t)s * bd.total_nodes + r) * kHq + head] = lse2;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
}

// ---------------------------------------------------------------- host side

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

// [pool pages * 4 heads * 16 slots] rows of 256 bf16; boxes of 16 rows x 64 dims, 128-byte swizzle.
bool cache_map(CUtensorMap* map, const void* cache, int pool_pages) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)pool_pages * kHkv * kPage};
  cuuint64_t strides[1] = {(cuuint64_t)kDim * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kPage};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NQ>
cudaError_t launch_nq(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p, const BatchDesc& bd,
                      int hpc, int hparts, cudaStream_t st) {
  const size_t smem = tc_smem_bytes(NQ);
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_splits * kHkv * hparts, bd.batch);
  attn_tc_kernel<NQ><<<grid, kThreads, smem, st>>>(mk, mv, p, bd, hpc, hparts);
  return cudaGetLastError();
}

}  // namespace

size_t tc_smem_bytes(int nq) {
  const int natom = (nq + 63) / 64;
  return 1024 + (size_t)nq * 512 + 2 * (size_t)kTileB + (size_t)natom * kRegionB + sizeof(Small);
}

TcPlan tc_plan(int max_nodes) {
  TcPlan pl;
  const int opts[4] = {6, 3, 2, 1};
  pl.hpc = 1;
  for (int h : opts) {
    if (h * max_nodes <= kTcMaxNQ) { pl.hpc = h; break; }
  }
  pl.hparts = (kGroup + pl.hpc - 1) / pl.hpc;
  pl.nq = (pl.hpc * max_nodes + 15) / 16 * 16;
  if (pl.nq < 32) pl.nq = 32;
  return pl;
}

int attn_tc_tile() { return kT; }

cudaError_t launch_attn_tc(const AttnParams& p, const BatchDesc& bd, cudaStream_t st) {
  CUtensorMap mk, mv;
  if (!cache_map(&mk, p.k_cache, p.num_pool_pages) || !cache_map(&mv, p.v_cache, p.num_pool_pages))
    return cudaErrorInvalidValue;
  const TcPlan pl = tc_plan(bd.max_nodes);
  cudaError_t e;
  switch (pl.nq) {
    case 32: e = launch_nq<32>(mk, mv, p, bd, pl.hpc, pl.hparts, st); break;
    case 48: e = launch_nq<48>(mk, mv, p, bd, pl.hpc, pl.hparts, st); break;
    case 64: e = launch_nq<64>(mk, mv, p, bd, pl.hpc, pl.hparts, st); break;
    case 80: e = launch_nq<80>(mk, mv, p, bd, pl.hpc, pl.hparts, st); break;
    case 96: e = launch_nq<96>(mk, mv, p, bd, pl.hpc, pl.hparts, st); break;
    case 112: e = launch_nq<112>(mk, mv, p, bd, pl.hpc, pl.hparts, st); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess || p.num_splits == 1) return e;
  return launch_attn_merge(p, bd, st);
}

}  // namespace sdv
