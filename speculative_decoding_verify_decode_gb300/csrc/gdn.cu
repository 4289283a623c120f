// Tree-aware Gated DeltaNet verify for the hybrid model's linear-attention
// layers: the short causal convolution along each node's parent chain, the
// gated delta rule over the draft tree, and persist-on-accept of the
// recurrent and convolution states.  Source: «如何在单张 RTX 3090 上让
// Qwen3.5-27B token 生成速度提升 6 倍» (为什么我们要做这个测试: 48 of 64 layers are
// Gated DeltaNet with a recurrent state cache; 关键突破: tree-aware delta-net
// and convolution kernels, siblings gathering their windows along the parent
// chain, the accepted state written in place).
//
// Per value head the state S (d_v rows x d_k) follows
//   S_j = alpha_j S_p + beta_j (v_j - alpha_j S_p k_j) k_j^T,  o_j = S_j q_j,
// with p the parent of node j (the cached state for the root), alpha = exp(g),
// k and q L2-normalised and q scaled by 1/sqrt(d_k).  Unrolled along a root
// path this is S_j = gamma_j S_0 + sum_{m on the path} (gamma_j / gamma_m) u_m k_m^T
// with gamma the product of alpha along the path and
//   u_j = beta_j (v_j - gamma_j S_0 k_j - sum_{m above j} (gamma_j / gamma_m) (k_m . k_j) u_m),
// a triangular system over the ancestor sets.  Every row of S evolves on its
// own, so a CTA owns 32 rows of one head's state: it reads them once
// (the dominant bytes), forms S_0 k_j and S_0 q_j for every node, the node-pair
// dot products under the ancestor mask, solves for its rows of u in node
// order and writes o.  The ratios are exp(G_j - G_m) of log-decays G, so long
// paths of strong decay never divide by an underflowed gamma.  u, G and the
// normalised keys go to a per-layer tree cache, from which the commit rebuilds
// the accepted node's state without ever storing every node's.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace sdv {
namespace {

constexpr int kD = kGdnDim;        // d_k = d_v
constexpr int kRows = 32;          // state rows per CTA
constexpr int kPad = kD + 1;       // padded state row in shared memory (no bank conflicts across rows)
constexpr int kGdnThreads = 256;

struct GdnSmem {
  // sizes for n nodes, laid out by gdn_smem_bytes
  static size_t bytes(int n) {
    return sizeof(float) * ((size_t)kRows * kPad + 2 * (size_t)n * kD + (size_t)n * kRows * 4 +
                            2 * (size_t)n * n + 4 * (size_t)n) +
           sizeof(unsigned long long) * n + sizeof(int) * n;
  }
};

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

__global__ void __launch_bounds__(kGdnThreads) gdn_tree_kernel(const GdnParams p, const BatchDesc bd) {
  extern __shared__ __align__(16) float smem[];
  const int b = blockIdx.y;
  const int rb = blockIdx.x % (kD / kRows);
  const int h = blockIdx.x / (kD / kRows);
  const int hk = h / (p.hv / p.hk);
  const int q0 = bd.q_indptr[b];
  const int n = bd.q_indptr[b + 1] - q0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  float* s0 = smem;                              // [32][kPad]
  float* kh = s0 + kRows * kPad;                 // [n][128] normalised keys
  float* qh = kh + n * kD;                       // [n][128] normalised, scaled queries
  float* vv = qh + n * kD;                       // [n][32] this block's value rows
  float* W = vv + n * kRows;                     // [n][32] S_0 k_j
  float* Z = W + n * kRows;                      // [n][32] S_0 q_j
  float* U = Z + n * kRows;                      // [n][32]
  float* A = U + n * kRows;                      // [n][n] beta_j e^{G_j - G_m} (k_m . k_j), m above j
  float* C = A + n * n;                          // [n][n] e^{G_j - G_m} (k_m . q_j), m on j's path
  float* G = C + n * n;                          // [n] log gamma
  float* beta = G + n;                           // [n]
  float* gg = beta + n;                          // [n] g
  float* pad_ = gg + n;                          // [n] (keeps the 8-byte arrays aligned)
  unsigned long long* anc = reinterpret_cast<unsigned long long*>(pad_ + n);   // [n] path bits, j included
  int* par = reinterpret_cast<int*>(anc + n);

  // ---- tree: parents, gates, ancestor sets and log-decays (thread j walks its root path)
  for (int j = tid; j < n; j += kGdnThreads) {
    int pj = p.parents[q0 + j];
    if ((j == 0 && pj != -1) || (j > 0 && (pj < 0 || pj >= j))) {
      report(p.dev_status, SD_DEV_BAD_PARENTS);
      pj = j == 0 ? -1 : j - 1;   // a chain stands in for a broken tree (the output is unspecified)
    }
    par[j] = pj;
    gg[j] = p.g[(size_t)(q0 + j) * p.hv + h];
    beta[j] = p.beta[(size_t)(q0 + j) * p.hv + h];
  }
  __syncthreads();
  for (int j = tid; j < n; j += kGdnThreads) {
    unsigned long long a = 0ull;
    float lg = 0.f;
    for (int u = j; u >= 0; u = par[u]) {
      a |= 1ull << u;
      lg += gg[u];
    }
    anc[j] = a;
    G[j] = lg;
  }
  // ---- normalised keys and queries of the key head (a warp per node), this block's value rows
  const float qscale = rsqrtf((float)kD);
  for (int j = warp; j < n; j += kGdnThreads / 32) {
    const __nv_bfloat16* kr = p.k + ((size_t)(q0 + j) * p.hk + hk) * kD;
    const __nv_bfloat16* qr = p.q + ((size_t)(q0 + j) * p.hk + hk) * kD;
    float kv4[4], qv4[4], sk = 0.f, sq = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      kv4[e] = bf2f(kr[lane + 32 * e]);
      qv4[e] = bf2f(qr[lane + 32 * e]);
      sk += kv4[e] * kv4[e];
      sq += qv4[e] * qv4[e];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
    }
    const float ik = sk > 0.f ? rsqrtf(sk) : 0.f, iq = sq > 0.f ? rsqrtf(sq) * qscale : 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      kh[j * kD + lane + 32 * e] = kv4[e] * ik;
      qh[j * kD + lane + 32 * e] = qv4[e] * iq;
    }
  }
  for (int i = tid; i < n * kRows; i += kGdnThreads) {
    const int j = i / kRows, r = i % kRows;
    vv[i] = bf2f(p.v[((size_t)(q0 + j) * p.hv + h) * kD + rb * kRows + r]);
  }
  // ---- this block's 32 state rows (16 KB contiguous), float4 loads
  {
    const float4* src = reinterpret_cast<const float4*>(p.state + (((size_t)b * p.hv + h) * kD + rb * kRows) * kD);
    for (int i = tid; i < kRows * kD / 4; i += kGdnThreads) {
      const float4 x = __ldg(src + i);
      const int r = (i * 4) / kD, c = (i * 4) % kD;
      float* d = s0 + r * kPad + c;
      d[0] = x.x; d[1] = x.y; d[2] = x.z; d[3] = x.w;
    }
  }
  __syncthreads();
  // ---- W[j][r] = S_0[r] . k_j and Z[j][r] = S_0[r] . q_j: lane = row, warps over nodes
  for (int j = warp; j < n; j += kGdnThreads / 32) {
    float aw = 0.f, az = 0.f;
    const float* sr = s0 + lane * kPad;
#pragma unroll 8
    for (int c = 0; c < kD; ++c) {
      const float s = sr[c];
      aw = fmaf(s, kh[j * kD + c], aw);
      az = fmaf(s, qh[j * kD + c], az);
    }
    W[j * kRows + lane] = aw;
    Z[j * kRows + lane] = az;
  }
  // ---- pair coefficients under the ancestor mask (dot products start at a rotated dim: no conflicts)
  for (int i = tid; i < n * n; i += kGdnThreads) {
    const int j = i / n, m = i % n;
    float a = 0.f, c = 0.f;
    if ((anc[j] >> m) & 1ull) {
      float dk = 0.f, dq = 0.f;
      for (int t = 0; t < kD; ++t) {
        const int e = (t + i) & (kD - 1);
        const float km = kh[m * kD + e];
        dk = fmaf(km, kh[j * kD + e], dk);
        dq = fmaf(km, qh[j * kD + e], dq);
      }
      const float ratio = __expf(G[j] - G[m]);
      if (m != j) a = beta[j] * ratio * dk;
      c = ratio * dq;
    }
    A[i] = a;
    C[i] = c;
  }
  __syncthreads();
  // ---- u in node order (a node's ancestors come first): one warp, lane = row
  if (warp == 0) {
    for (int j = 0; j < n; ++j) {
      float acc = beta[j] * (vv[j * kRows + lane] - __expf(G[j]) * W[j * kRows + lane]);
      unsigned long long a = anc[j] & ~(1ull << j);
      while (a != 0ull) {
        const int m = __ffsll((long long)a) - 1;
        a &= a - 1ull;
        acc = fmaf(-A[j * n + m], U[m * kRows + lane], acc);
      }
      U[j * kRows + lane] = acc;
      __syncwarp();
    }
  }
  __syncthreads();
  // ---- outputs, u, log-decays and normalised keys
  for (int i = tid; i < n * kRows; i += kGdnThreads) {
    const int j = i / kRows, r = i % kRows;
    float acc = __expf(G[j]) * Z[j * kRows + r];
    unsigned long long a = anc[j];
    while (a != 0ull) {
      const int m = __ffsll((long long)a) - 1;
      a &= a - 1ull;
      acc = fmaf(C[j * n + m], U[m * kRows + r], acc);
    }
    const size_t row = (size_t)(q0 + j) * p.hv + h;
    p.out[row * kD + rb * kRows + r] = __float2bfloat16_rn(acc);
    p.cache_u[row * kD + rb * kRows + r] = U[i];
  }
  if (rb == 0)
    for (int j = tid; j < n; j += kGdnThreads) p.cache_g[(size_t)(q0 + j) * p.hv + h] = G[j];
  if (rb == 0 && h % (p.hv / p.hk) == 0)
    for (int i = tid; i < n * kD; i += kGdnThreads)
      p.cache_k[((size_t)(q0 + i / kD) * p.hk + hk) * kD + i % kD] = kh[i];
}

// Persist-on-accept of the recurrent state, every layer in one launch:
// S <- gamma_last S + sum over the accepted path of (gamma_last / gamma_m) u_m k_m^T,
// 32 rows of one head per CTA, in place.
__global__ void __launch_bounds__(kGdnThreads) gdn_commit_kernel(const GdnCommitParams p, const BatchDesc bd) {
  __shared__ float ks[kMaxNodes][kD];      // normalised keys of the path (32 KB)
  __shared__ float us[kMaxNodes][kRows];   // this block's u rows of the path
  __shared__ float wt[kMaxNodes];          // e^{G_last - G_m}
  __shared__ int bad;
  const int layer = blockIdx.z, b = blockIdx.y;
  const int rb = blockIdx.x % (kD / kRows), h = blockIdx.x / (kD / kRows);
  const int hk = h / (p.hv / p.hk);
  const int q0 = bd.q_indptr[b];
  const int n = bd.q_indptr[b + 1] - q0;
  const int a = p.accept_len[b];
  const int tid = threadIdx.x;
  if (tid == 0) bad = (a < 1 || a > n || a > p.max_path) ? 1 : 0;
  __syncthreads();
  if (!bad && tid < a) {
    const int node = p.path[(size_t)b * p.max_path + tid];
    if (node < 0 || node >= n || (tid == 0 && node != 0)) atomicOr(&bad, 1);
  }
  __syncthreads();
  if (bad) {
    if (tid == 0 && layer == 0 && h == 0 && rb == 0) report(p.dev_status, SD_DEV_BAD_ACCEPT);
    return;
  }
  const float* cu = p.cache_u[layer];
  const float* cg = p.cache_g[layer];
  const float* ck = p.cache_k[layer];
  const int last = p.path[(size_t)b * p.max_path + a - 1];
  const float g_last = cg[(size_t)(q0 + last) * p.hv + h];
  for (int i = tid; i < a * kD; i += kGdnThreads) {
    const int m = p.path[(size_t)b * p.max_path + i / kD];
    ks[i / kD][i % kD] = ck[((size_t)(q0 + m) * p.hk + hk) * kD + i % kD];
  }
  for (int i = tid; i < a * kRows; i += kGdnThreads) {
    const int m = p.path[(size_t)b * p.max_path + i / kRows];
    us[i / kRows][i % kRows] = cu[((size_t)(q0 + m) * p.hv + h) * kD + rb * kRows + i % kRows];
  }
  for (int i = tid; i < a; i += kGdnThreads) {
    const int m = p.path[(size_t)b * p.max_path + i];
    wt[i] = __expf(g_last - cg[(size_t)(q0 + m) * p.hv + h]);
  }
  __syncthreads();
  const float gamma = __expf(g_last);
  float* st = p.state[layer] + (((size_t)b * p.hv + h) * kD + rb * kRows) * kD;
  for (int i = tid; i < kRows * kD; i += kGdnThreads) {
    const int r = i / kD, c = i % kD;
    float acc = gamma * st[i];
    for (int m = 0; m < a; ++m) acc = fmaf(wt[m] * us[m][r], ks[m][c], acc);
    st[i] = acc;
  }
}

// Persist of the convolution state: the last three inputs of (old state, accepted nodes' inputs).
__global__ void __launch_bounds__(256) conv_commit_kernel(const GdnCommitParams p, const BatchDesc bd) {
  const int layer = blockIdx.z, b = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const int q0 = bd.q_indptr[b];
  const int n = bd.q_indptr[b + 1] - q0;
  const int a = p.accept_len[b];
  if (c >= p.channels || a < 1 || a > n || a > p.max_path) return;   // the state kernel reports it
  __nv_bfloat16* st = p.conv_state[layer] + ((size_t)b * p.channels + c) * 3;
  const __nv_bfloat16* x = p.x[layer];
  __nv_bfloat16 seq[3];
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const int from_path = a - 3 + i;      // index into the accepted path, or into the old state if < 0
    if (from_path >= 0) {
      const int node = p.path[(size_t)b * p.max_path + from_path];
      if (node < 0 || node >= n) return;
      seq[i] = x[(size_t)(q0 + node) * p.channels + c];
    } else {
      seq[i] = st[3 + from_path];
    }
  }
#pragma unroll
  for (int i = 0; i < 3; ++i) st[i] = seq[i];
}

// Causal 4-tap depthwise convolution + SiLU along each node's parent chain.
// Block: 256 channels of one sequence, every node.
__global__ void __launch_bounds__(256) conv_tree_kernel(const ConvTreeParams p, const BatchDesc bd) {
  __shared__ int par[kMaxNodes];
  const int b = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const int q0 = bd.q_indptr[b];
  const int n = bd.q_indptr[b + 1] - q0;
  if (threadIdx.x < n) {
    const int j = threadIdx.x;
    int pj = p.parents[q0 + j];
    if ((j == 0 && pj != -1) || (j > 0 && (pj < 0 || pj >= j))) {
      if (blockIdx.x == 0) report(p.dev_status, SD_DEV_BAD_PARENTS);
      pj = j == 0 ? -1 : j - 1;
    }
    par[j] = pj;
  }
  __syncthreads();
  if (c >= p.channels) return;
  const float4 w = reinterpret_cast<const float4*>(p.weight)[c];   // w.w multiplies the node's own input
  const __nv_bfloat16* cs = p.conv_state + ((size_t)b * p.channels + c) * 3;
  const float s0 = bf2f(cs[0]), s1 = bf2f(cs[1]), s2 = bf2f(cs[2]);
  for (int j = 0; j < n; ++j) {
    float x[4];   // newest first
    int u = j, t = 0;
    for (; t < 4 && u >= 0; ++t, u = par[u]) x[t] = bf2f(p.x[(size_t)(q0 + u) * p.channels + c]);
    const float st[3] = {s2, s1, s0};
    for (int k = 0; t < 4; ++t, ++k) x[t] = st[k];
    const float acc = w.w * x[0] + w.z * x[1] + w.y * x[2] + w.x * x[3];
    p.y[(size_t)(q0 + j) * p.channels + c] = __float2bfloat16_rn(acc / (1.0f + __expf(-acc)));
  }
}

}  // namespace

size_t gdn_smem_bytes(int max_nodes) { return GdnSmem::bytes(max_nodes); }

cudaError_t launch_gdn_tree(const GdnParams& p, const BatchDesc& bd, cudaStream_t st) {
  const size_t smem = GdnSmem::bytes(bd.max_nodes);
  cudaError_t e = cudaFuncSetAttribute(gdn_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  gdn_tree_kernel<<<dim3(p.hv * (kD / kRows), bd.batch), kGdnThreads, smem, st>>>(p, bd);
  return cudaGetLastError();
}

cudaError_t launch_gdn_commit(const GdnCommitParams& p, const BatchDesc& bd, cudaStream_t st) {
  gdn_commit_kernel<<<dim3(p.hv * (kD / kRows), bd.batch, p.num_layers), kGdnThreads, 0, st>>>(p, bd);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.channels == 0) return e;
  conv_commit_kernel<<<dim3((p.channels + 255) / 256, bd.batch, p.num_layers), 256, 0, st>>>(p, bd);
  return cudaGetLastError();
}

cudaError_t launch_conv_tree(const ConvTreeParams& p, const BatchDesc& bd, cudaStream_t st) {
  conv_tree_kernel<<<dim3((p.channels + 255) / 256, bd.batch), 256, 0, st>>>(p, bd);
  return cudaGetLastError();
}

}  // namespace sdv
