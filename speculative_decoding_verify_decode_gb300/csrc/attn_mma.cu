// Split-KV verify attention on the warp-level tensor-core path (mma.sync
// m16n8k16, bf16 in, fp32 accumulate), plus the log-sum-exp merge of splits.
//
// What it computes: for sequence b, draft node j and query head h, softmax
// attention (scale 1/16) of q[j][h] over every context token of KV head h/6
// and over the draft nodes on j's root path — the tree mask of
// «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍» (关键突破: each node
// follows its parent chain) which, for a chain, is the bottom-right-aligned
// causal mask of «Qwen3.8-27B投机解码实测：从14到159 tok/s的性能断点地图» (§5.3).
// The paged cache (16-token pages from one pool, same page §2 and §4) is read
// through the page table.
//
// Work split: one CTA per (split s, KV head g, row block, sequence b).  The
// query rows of a CTA are the 6 heads of group g times the sequence's draft
// nodes (row m = node * 6 + head-in-group), so every K/V tile staged in
// shared memory is used by all of them.  Split 0 also handles the draft
// block as one extra masked tile.  Each CTA keeps an online softmax; a split
// writes its normalised partial output and base-2 log-sum-exp, and the merge
// kernel combines them.  A sequence with a single active split is written
// directly in bf16.
#include "common.cuh"
#include "kernels.h"

namespace sdv {
namespace {

constexpr int kTile = 64;        // KV tokens per pipeline stage
constexpr int kRowB = kDim * 2;  // bytes of one 256-wide bf16 row

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Byte offset of 16-byte chunk c of row `row` in a [rows][256] bf16 tile,
// XOR-swizzled so that 8 consecutive rows of one chunk hit 8 bank groups.
__device__ __forceinline__ uint32_t swz(int row, int c) {
  return static_cast<uint32_t>(row * kRowB + ((c ^ (row & 7)) << 4));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int sz = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Ancestor bitmask of every node of one sequence (bit i of anc[j] set when i
// is j or one of its ancestors).  Invalid parent arrays are reported and
// reduced to "self only" masks, so nothing is read out of range.
__device__ void build_ancestors(const int* parents, int q0, int n, uint64_t* anc, int* status) {
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    uint64_t mask = 1ull << j;
    bool ok = true;
    if (j == 0) {
      ok = parents[q0] == -1;
    } else {
      int u = j;
      while (u > 0) {  // parents strictly decrease, so at most j steps
        const int pu = parents[q0 + u];
        if (pu < 0 || pu >= u) { ok = false; break; }
        mask |= 1ull << pu;
        u = pu;
      }
    }
    if (!ok) { report(status, SD_DEV_BAD_PARENTS); mask = 1ull << j; }
    anc[j] = mask;
  }
}

template <int NW>
__global__ void __launch_bounds__(NW * 32, 1)
attn_split_mma_kernel(const AttnParams p, const BatchDesc bd) {
  constexpr int R = 16 * NW;          // query rows per CTA
  constexpr int NT = NW * 32;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t s_anc[kMaxNodes];

  const int s = blockIdx.x;
  const int g = blockIdx.y % kHkv;
  const int row0 = (blockIdx.y / kHkv) * R;
  const int b = blockIdx.z;
  const int q0 = bd.q_indptr[b];
  const int n_nodes = bd.q_indptr[b + 1] - q0;
  const int M = n_nodes * kGroup;
  if (row0 >= M) return;

  int L = p.ctx_lens[b];
  if (L < 0 || L > p.max_pages * kPage) {
    if (s == 0 && threadIdx.x == 0 && blockIdx.y == 0) report(p.dev_status, SD_DEV_BAD_CTX);
    L = L < 0 ? 0 : p.max_pages * kPage;
  }
  const int nsplit = active_splits(L, p.chunk);
  if (s >= nsplit) return;
  const int ctx_begin = s * p.chunk;
  const int ctx_end = min(L, ctx_begin + p.chunk);
  const bool has_draft = (s == 0);
  const int n_ctx_tiles = ctx_end > ctx_begin ? (ctx_end - ctx_begin + kTile - 1) / kTile : 0;
  const int n_tiles = n_ctx_tiles + (has_draft ? 1 : 0);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + R * kRowB;  // stage st: K at st*2*T, V at st*2*T + T
  constexpr int kTileB = kTile * kRowB;

  if (has_draft) build_ancestors(p.parents, q0, n_nodes, s_anc, p.dev_status);

  // Q rows of this CTA (zero rows past M).
  for (int task = tid; task < R * 32; task += NT) {
    const int r = task >> 5, c = task & 31;
    const int m = row0 + r;
    const bool valid = m < M;
    const int node = valid ? m / kGroup : 0;
    const int head = g * kGroup + (valid ? m % kGroup : 0);
    const __nv_bfloat16* src = p.q + ((size_t)(q0 + node) * kHq + head) * kDim + c * 8;
    cp_async16(smem_u32(sQ) + swz(r, c), src, valid);
  }

  auto load_tile = [&](int it, int st) {
    const uint32_t kb = smem_u32(sKV) + st * 2 * kTileB;
    const uint32_t vb = kb + kTileB;
    if (has_draft && it == 0) {
      for (int task = tid; task < kTile * 32; task += NT) {
        const int r = task >> 5, c = task & 31;
        const bool valid = r < n_nodes;
        const size_t off = ((size_t)(q0 + (valid ? r : 0)) * kHkv + g) * kDim + c * 8;
        cp_async16(kb + swz(r, c), p.k_new + off, valid);
        cp_async16(vb + swz(r, c), p.v_new + off, valid);
      }
    } else {
      const int t0 = ctx_begin + (it - (has_draft ? 1 : 0)) * kTile;
      for (int task = tid; task < kTile * 32; task += NT) {
        const int r = task >> 5, c = task & 31;
        const int pos = t0 + r;
        bool valid = pos < ctx_end;
        int page = 0;
        if (valid) {
          page = p.page_table[(size_t)b * p.max_pages + (pos >> 4)];
          if (page < 0 || page >= p.num_pool_pages) {
            if (c == 0) report(p.dev_status, SD_DEV_BAD_PAGE);
            valid = false;
            page = 0;
          }
        }
        const size_t off = (((size_t)page * kHkv + g) * kPage + (pos & 15)) * kDim + c * 8;
        cp_async16(kb + swz(r, c), p.k_cache + off, valid);
        cp_async16(vb + swz(r, c), p.v_cache + off, valid);
      }
    }
    cp_async_commit();
  };

  float o[32][4];
#pragma unroll
  for (int i = 0; i < 32; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};

  load_tile(0, 0);  // the Q copies join the first group
  for (int it = 0; it < n_tiles; ++it) {
    if (it + 1 < n_tiles) load_tile(it + 1, (it + 1) & 1);
    else cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    const uint32_t kb = smem_u32(sKV) + (it & 1) * 2 * kTileB;
    const uint32_t vb = kb + kTileB;
    const bool draft_tile = has_draft && it == 0;
    const int t0 = draft_tile ? 0 : ctx_begin + (it - (has_draft ? 1 : 0)) * kTile;

    // S = Q K^T for this warp's 16 rows x 64 tokens.
    float sacc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      uint32_t a[4];
      ldsm_x4(a, smem_u32(sQ) + swz(warp * 16 + (lane & 15), kk * 2 + (lane >> 4)));
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t bb[4];
        ldsm_x4(bb, kb + swz(np * 16 + (lane & 7) + ((lane >> 4) << 3), kk * 2 + ((lane >> 3) & 1)));
        mma16816(sacc[2 * np], a, bb[0], bb[1]);
        mma16816(sacc[2 * np + 1], a, bb[2], bb[3]);
      }
    }

    // Mask, online softmax (base 2).
    float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int rl = warp * 16 + (lane >> 2) + ((e >> 1) << 3);
        const int col = n * 8 + ((lane & 3) << 1) + (e & 1);
        bool vis;
        if (draft_tile) {
          const int node = (row0 + rl) / kGroup;
          vis = col < n_nodes && (node < n_nodes ? ((s_anc[node] >> col) & 1ull) != 0 : col == 0);
        } else {
          vis = t0 + col < ctx_end;
        }
        const float x = vis ? sacc[n][e] * kScaleLog2 : -INFINITY;
        sacc[n][e] = x;
        mt[e >> 1] = fmaxf(mt[e >> 1], x);
      }
    }
    float alpha[2], mu[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], 1));
      mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], 2));
      const float mn = fmaxf(m_run[h], mt[h]);
      mu[h] = mn == -INFINITY ? 0.f : mn;
      alpha[h] = fast_exp2(m_run[h] - mu[h]);
      m_run[h] = mn;
      l_run[h] *= alpha[h];
    }
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pv = fast_exp2(sacc[n][e] - mu[e >> 1]);
        sacc[n][e] = pv;
        l_run[e >> 1] += pv;
      }
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      o[i][0] *= alpha[0]; o[i][1] *= alpha[0];
      o[i][2] *= alpha[1]; o[i][3] *= alpha[1];
    }

    // O += P V.
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t a[4];
      a[0] = pack_bf16(sacc[2 * kk][0], sacc[2 * kk][1]);
      a[1] = pack_bf16(sacc[2 * kk][2], sacc[2 * kk][3]);
      a[2] = pack_bf16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
      a[3] = pack_bf16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < 16; ++dp) {
        uint32_t bb[4];
        ldsm_x4_t(bb, vb + swz(kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3), dp * 2 + (lane >> 4)));
        mma16816(o[2 * dp], a, bb[0], bb[1]);
        mma16816(o[2 * dp + 1], a, bb[2], bb[3]);
      }
    }
    __syncthreads();  // this stage is refilled by the next iteration's load
  }
  cp_async_wait<0>();

  // Epilogue: finish the row sums and write.
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int m = row0 + warp * 16 + (lane >> 2) + h * 8;
    if (m >= M) continue;
    const int r = q0 + m / kGroup;
    const int head = g * kGroup + m % kGroup;
    const float inv = 1.f / l_run[h];
    const float lse2 = m_run[h] + fast_log2(l_run[h]);
    if (nsplit == 1) {
      __nv_bfloat16* dst = p.out + ((size_t)r * kHq + head) * kDim;
#pragma unroll
      for (int dt = 0; dt < 32; ++dt) {
        const int d = dt * 8 + ((lane & 3) << 1);
        *reinterpret_cast<__nv_bfloat162*>(dst + d) =
            __floats2bfloat162_rn(o[dt][2 * h] * inv, o[dt][2 * h + 1] * inv);
      }
      if (p.lse != nullptr && (lane & 3) == 0) p.lse[(size_t)r * kHq + head] = lse2 * kLn2;
    } else {
      float* dst = p.o_part + (((size_t)s * bd.total_nodes + r) * kHq + head) * kDim;
#pragma unroll
      for (int dt = 0; dt < 32; ++dt) {
        const int d = dt * 8 + ((lane & 3) << 1);
        *reinterpret_cast<float2*>(dst + d) = make_float2(o[dt][2 * h] * inv, o[dt][2 * h + 1] * inv);
      }
      if ((lane & 3) == 0) p.lse_part[((size_t)s * bd.total_nodes + r) * kHq + head] = lse2;
    }
  }
}

template <int NW>
cudaError_t launch_split(const AttnParams& p, const BatchDesc& bd, cudaStream_t st) {
  constexpr int R = 16 * NW;
  const size_t smem = (size_t)R * kRowB + 4 * (size_t)kTile * kRowB;
  cudaError_t e = cudaFuncSetAttribute(attn_split_mma_kernel<NW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int row_blocks = (bd.max_nodes * kGroup + R - 1) / R;
  dim3 grid(p.num_splits, kHkv * row_blocks, bd.batch);
  attn_split_mma_kernel<NW><<<grid, NW * 32, smem, st>>>(p, bd);
  return cudaGetLastError();
}

}  // namespace

int attn_mma_tile() { return kTile; }

int attn_mma_ctas_per_split(const BatchDesc& bd) {
  const int M = bd.max_nodes * kGroup;
  const int R = M <= 32 ? 32 : (M <= 64 ? 64 : 144);
  return bd.batch * kHkv * ((M + R - 1) / R);
}

cudaError_t launch_attn_mma(const AttnParams& p, const BatchDesc& bd, cudaStream_t st) {
  const int M = bd.max_nodes * kGroup;
  cudaError_t e;
  if (M <= 32) e = launch_split<2>(p, bd, st);
  else if (M <= 64) e = launch_split<4>(p, bd, st);
  else e = launch_split<9>(p, bd, st);
  if (e != cudaSuccess || p.num_splits == 1) return e;
  return launch_attn_merge(p, bd, st);
}

}  // namespace sdv
