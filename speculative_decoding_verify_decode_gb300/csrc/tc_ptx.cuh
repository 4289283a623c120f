// Inline-PTX building blocks of the tcgen05 / TMA kernels: mbarriers with
// bounded waits, TMA box loads of the paged cache, shared-memory matrix and
// instruction descriptors, tcgen05.mma / commit / ld / st, and small warp
// helpers.  Internal to the library.
#pragma once

#include <cstdint>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace sdv {
namespace {

constexpr long long kWaitCycles = 2000000000LL;  // about a second at GB300 clocks
// Shared-memory image of K/V rows (256 bf16 each): 8-row groups of four 64-dim
// blocks (1 KB each: 8 rows x 128 B, 128-byte swizzle).
constexpr int kGroupB = 4096;           // 8 token rows x 4 dim blocks x 128 B
constexpr int kPageB = 2 * kGroupB;     // one page of one KV head: 16 rows x 256 dims

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
// Test a phase; the waiting thread is suspended in hardware (up to about
// 10 ms, or until the phase completes) instead of spinning on issue slots.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(10000000u)
      : "memory");
  return ok != 0;
}
// Non-blocking test of a phase.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false (and the CTA's abort flag set) if the phase never completes.
// Status bits from a thread that may not have waited for the previous kernel
// yet (context loads issued before the wait): wait first, so that the bit
// cannot be lost to a predecessor that resets the status word.  A no-op wait
// once the predecessor has finished.
__device__ __forceinline__ void report_dep(int* status, int bits) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  report(status, bits);
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* abort, int* status) {
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (clock64() - t0 > kWaitCycles || *(volatile int*)abort) {
      *abort = 1;
      report_dep(status, SD_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}
// Bounded spin on a phase (no suspension): the softmax warps have nothing
// else to do while they wait, and a spin sees the phase flip soonest.
__device__ __forceinline__ bool mbar_spin(uint32_t bar, uint32_t parity, int* abort, int* status) {
  const long long t0 = clock64();
  while (!mbar_test(bar, parity)) {
    if (clock64() - t0 > kWaitCycles || *(volatile int*)abort) {
      *abort = 1;
      report_dep(status, SD_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// L2 policy for data read once (the context pages): its lines are the first
// to be evicted, so streaming the cache does not push the kernels' code, the
// page tables, the queries and the split partials out of L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// One page of one KV head (8 KB) into shared memory: the 4-D box of the
// cache map at outer coordinate w, x = y = z = 0, read with the evict-first policy.
__device__ __forceinline__ void tma_load_page(uint32_t dst, const CUtensorMap* map, int w, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %2, %2, %3}], [%4], %5;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(w), "r"(bar), "l"(l2_evict_first())
      : "memory");
}

// ------------------------------------------------------------ tcgen05

// Shared-memory matrix descriptor, 128-byte swizzle: start, leading and
// stride byte offsets (16-byte units), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// The same with the 32-byte swizzle (16-byte chunk bit 0 XOR address bit 7).
__device__ __forceinline__ uint64_t sw32_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (6ull << 61);
}
// Instruction descriptor of kind::f16: bf16 x bf16 (or f16 x f16) -> f32, M x N, operand majors.
__host__ __device__ constexpr uint32_t f16_idesc(int m, int n, int a_mn, int b_mn, bool bf16 = true) {
  return (1u << 4) | (bf16 ? (1u << 7) | (1u << 10) : 0u) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
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


// Byte offset of 16-byte chunk c (0..31) of token row r in a group-major
// K/V tile: 8-row group r/8 (4 KB), 64-dim block c/8 (1 KB), row r%8,
// swizzled chunk (c%8) ^ (r%8).  A page's 16 rows are 8 contiguous KB.
__device__ __forceinline__ uint32_t kv_off(int r, int c) {
  return (uint32_t)((r >> 3) * kGroupB + (c >> 3) * 1024 + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4));
}
// Byte offset of 16-byte chunk cc (0..7) of token row r in the P^T tile
// (MN-major: 64-column atoms of 128 rows x 128 B, 128-byte swizzle).
__device__ __forceinline__ uint32_t p_off(int r, int cc) {
  return (uint32_t)(r * 128 + ((cc ^ (r & 7)) << 4));
}

// Copy `nrows` rows of 256 bf16 into rows r0.. of a group-major K/V tile
// (row r's source is src_of(r), or zeros when that is null).  `nthreads`
// threads starting at `t` share the work; each keeps 8 independent 16-byte
// loads in flight.
template <typename SrcFn>
__device__ __forceinline__ void stage_rows(uint8_t* base, int r0, int nrows, SrcFn src_of, int t, int nthreads) {
  constexpr int U = 8;
  const int tasks = nrows * 32;
  for (int t0 = t; t0 < tasks; t0 += nthreads * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int task = t0 + u * nthreads;
      v[u] = make_uint4(0, 0, 0, 0);
      if (task < tasks) {
        const __nv_bfloat16* src = src_of(task >> 5);
        if (src != nullptr) v[u] = __ldg(reinterpret_cast<const uint4*>(src) + (task & 31));
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int task = t0 + u * nthreads;
      if (task < tasks) *reinterpret_cast<uint4*>(base + kv_off(r0 + (task >> 5), task & 31)) = v[u];
    }
  }
}

// Bits [start, start + len) of a 32-bit word (clipped to the word).
__device__ __forceinline__ uint32_t bit_range(int start, int len) {
  const int a = max(start, 0), e = min(start + len, 32);
  if (e <= a) return 0u;
  const uint32_t upto = e >= 32 ? 0xffffffffu : ((1u << e) - 1u);
  return upto & ~((1u << a) - 1u);
}

// Element g of a small per-thread array, by a select chain rather than a
// dynamically indexed (local-memory) access.
template <int N>
__device__ __forceinline__ uint32_t vis_of(const uint32_t (&a)[N], int g) {
  uint32_t r = a[0];
#pragma unroll
  for (int k = 1; k < N; ++k) r = (g == k) ? a[k] : r;
  return r;
}

// Reduce 32 values per lane across the warp so that lane L ends with the
// maximum over all lanes of value L (transpose-reduce, 31 shuffles).
__device__ __forceinline__ float transpose_max32(float (&v)[32], int lane) {
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool up = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, half));
    }
  }
  return v[0];
}

}  // namespace
}  // namespace sdv
