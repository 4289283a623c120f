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
constexpr int kCommitRows = 32;    // state rows per commit CTA
constexpr int kLd = kD + 4;        // padded row (state, keys, queries): 8 consecutive rows read as float4 hit
                                   // 8 distinct 16-byte bank groups
constexpr int kGdnThreads = 256;

size_t gdn_tree_smem(int n, int kRows) {
  return sizeof(float) * ((size_t)kRows * kLd + 2 * (size_t)n * kLd + (size_t)(4 * n + 1) * kRows +
                          2 * (size_t)n * (n + 1) + 4 * (size_t)n) +
         (size_t)n * kMaxNodes + sizeof(int) * (3 * (size_t)n + 1);
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Two 128-element dot products sharing their first row: (a . b, a . c), each row read once (float4 loads).
__device__ __forceinline__ float2 dot128x2(const float* a, const float* b, const float* c) {
  const float4* a4 = reinterpret_cast<const float4*>(a);
  const float4* b4 = reinterpret_cast<const float4*>(b);
  const float4* c4 = reinterpret_cast<const float4*>(c);
  float s0 = 0.f, s1 = 0.f, t0 = 0.f, t1 = 0.f;
#pragma unroll 8
  for (int t = 0; t < kD / 4; ++t) {
    const float4 x = a4[t], y = b4[t], z = c4[t];
    s0 = fmaf(x.x, y.x, fmaf(x.y, y.y, s0));
    s1 = fmaf(x.z, y.z, fmaf(x.w, y.w, s1));
    t0 = fmaf(x.x, z.x, fmaf(x.y, z.y, t0));
    t1 = fmaf(x.z, z.z, fmaf(x.w, z.w, t1));
  }
  return make_float2(s0 + s1, t0 + t1);
}


// ROWS state rows per CTA: 16 when the batch is small (more CTAs), 64 when it is large (the fixed chain of
// phases is paid once per 64 rows).
template <int kRows>
__global__ void __launch_bounds__(kGdnThreads) gdn_tree_kernel(const GdnParams p, const BatchDesc bd) {
  extern __shared__ __align__(16) float smem[];
  const int b = blockIdx.y;
  const int rb = blockIdx.x % (kD / kRows);
  const int h = blockIdx.x / (kD / kRows);
  const int hk = h / (p.hv / p.hk);
  const int q0 = bd.q_indptr[b];
  const int n = bd.q_indptr[b + 1] - q0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  float* s0 = smem;                              // [16][kLd] this block's state rows
  float* kh = s0 + kRows * kLd;                  // [n][kLd] normalised keys
  float* qh = kh + n * kLd;                      // [n][kLd] normalised, scaled queries
  float* vv = qh + n * kLd;                      // [n][16] this block's value rows
  float* W = vv + n * kRows;                     // [n][16] S_0 k_j
  float* Z = W + n * kRows;                      // [n][16] S_0 q_j
  float* U = Z + n * kRows;                      // [n + 1][16]; row n stays zero (padding of the sums)
  float* A = U + (n + 1) * kRows;                // [n][n + 1] beta_j e^{G_j - G_m} (k_m . k_j), m above j
  float* C = A + n * (n + 1);                    // [n][n + 1] e^{G_j - G_m} (k_m . q_j), m on j's path
  float* G = C + n * (n + 1);                    // [n] log of the path's decay product
  float* beta = G + n;
  float* gg = beta + n;
  float* eg = gg + n;                            // [n] e^{G_j}
  int* par = reinterpret_cast<int*>(eg + n);     // [n]
  int* depth = par + n;                          // [n] proper ancestors of j
  int* poff = depth + n;                         // [n + 1] offsets of each node's (node, path member) pairs
  uint8_t* alist = reinterpret_cast<uint8_t*>(poff + n + 1);   // [n][64] proper ancestors, padded with n

  // ---- every global load of the CTA, before any barrier
  {
    const float4* src = reinterpret_cast<const float4*>(p.state + (((size_t)b * p.hv + h) * kD + rb * kRows) * kD);
    for (int i = tid; i < kRows * kD / 4; i += kGdnThreads) {
      const int r = (i * 4) / kD, c = (i * 4) % kD;
      *reinterpret_cast<float4*>(s0 + r * kLd + c) = __ldg(src + i);
    }
    for (int i = tid; i < n * kRows; i += kGdnThreads) {
      const int j = i / kRows, r = i % kRows;
      vv[i] = bf2f(p.v[((size_t)(q0 + j) * p.hv + h) * kD + rb * kRows + r]);
    }
    if (tid < kRows) U[n * kRows + tid] = 0.f;
    for (int j = tid; j < n; j += kGdnThreads) {
      int pj = p.parents[q0 + j];
      if ((j == 0 && pj != -1) || (j > 0 && (pj < 0 || pj >= j))) {
        if (rb == 0 && h == 0) report(p.dev_status, SD_DEV_BAD_PARENTS);
        pj = j == 0 ? -1 : j - 1;   // a chain stands in for a broken tree (the output is unspecified)
      }
      par[j] = pj;
      gg[j] = p.g[(size_t)(q0 + j) * p.hv + h];
      beta[j] = p.beta[(size_t)(q0 + j) * p.hv + h];
    }
    // normalised keys and queries of the key head, a warp per node
    const float qscale = rsqrtf((float)kD);
    for (int j = warp; j < n; j += kGdnThreads / 32) {
      const __nv_bfloat16* kr = p.k + ((size_t)(q0 + j) * p.hk + hk) * kD;
      const __nv_bfloat16* qr = p.q + ((size_t)(q0 + j) * p.hk + hk) * kD;
      float kv4[4], qv4[4], sk = 0.f, sq = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kv4[e] = bf2f(kr[lane + 32 * e]);
        qv4[e] = bf2f(qr[lane + 32 * e]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sk = fmaf(kv4[e], kv4[e], sk);
        sq = fmaf(qv4[e], qv4[e], sq);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
      }
      const float ik = sk > 0.f ? rsqrtf(sk) : 0.f, iq = sq > 0.f ? rsqrtf(sq) * qscale : 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kh[j * kLd + lane + 32 * e] = kv4[e] * ik;
        qh[j * kLd + lane + 32 * e] = qv4[e] * iq;
      }
    }
  }
  __syncthreads();
  // ---- root paths (thread j): ancestor list, depth, log-decay; S_0 k_j and S_0 q_j (thread = (row, node))
  for (int j = tid; j < n; j += kGdnThreads) {
    float lg = gg[j];
    int d = 0;
    for (int u = par[j]; u >= 0; u = par[u]) {
      alist[j * kMaxNodes + d++] = (uint8_t)u;
      lg += gg[u];
    }
    for (int e = d; e < ((d + 3) & ~3); ++e) alist[j * kMaxNodes + e] = (uint8_t)n;   // padding: the zero row
    depth[j] = d;
    G[j] = lg;
    eg[j] = __expf(lg);
  }
  __syncthreads();
  if (tid < 32) {   // offsets of the compacted (node, path member) pairs: node j owns depth[j] + 1 of them
    int run = 0;
    for (int j0 = 0; j0 < n; j0 += 32) {
      const int j = j0 + tid;
      const int cnt = j < n ? depth[j] + 1 : 0;
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (tid >= off) incl += o;
      }
      if (j < n) poff[j] = run + incl - cnt;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (tid == 0) poff[n] = run;
  }
  // S_0 k_j and S_0 q_j: one thread per (node, row), the row read once for both products
  for (int i = tid; i < n * kRows; i += kGdnThreads) {
    const int j = i / kRows, r = i % kRows;
    const float2 wz = dot128x2(s0 + r * kLd, kh + j * kLd, qh + j * kLd);
    W[i] = wz.x;
    Z[i] = wz.y;
  }
  __syncthreads();
  // ---- pair coefficients along each node's path (row j, column = ancestor index; column n = padding 0),
  // one thread per (node, path member) pair
  for (int i = tid; i < poff[n]; i += kGdnThreads) {
    int lo = 0, hi = n - 1;   // node j with poff[j] <= i < poff[j + 1]
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (poff[mid] <= i) lo = mid; else hi = mid - 1;
    }
    const int j = lo, e = i - poff[j];
    const int d = depth[j];
    const int m = e < d ? alist[j * kMaxNodes + e] : j;   // the ancestors, then j itself
    const float ratio = __expf(G[j] - G[m]);
    const float2 kq = dot128x2(kh + m * kLd, kh + j * kLd, qh + j * kLd);
    if (m != j) A[j * (n + 1) + m] = beta[j] * ratio * kq.x;
    C[j * (n + 1) + m] = ratio * kq.y;
    if (e == 0) {
      A[j * (n + 1) + n] = 0.f;
      C[j * (n + 1) + n] = 0.f;
    }
  }
  __syncthreads();
  // ---- u in node order (a node's ancestors come first): thread = row, four ancestors per round
  if (tid < kRows) {
    const int r = tid;
    for (int j = 0; j < n; ++j) {
      float acc = beta[j] * (vv[j * kRows + r] - eg[j] * W[j * kRows + r]);
      const uint8_t* al = alist + j * kMaxNodes;
      const float* aj = A + j * (n + 1);
      const int d = depth[j];
      for (int e = 0; e < d; e += 4) {
        const int m0 = al[e], m1 = al[e + 1], m2 = al[e + 2], m3 = al[e + 3];
        const float a0 = aj[m0], a1 = aj[m1], a2 = aj[m2], a3 = aj[m3];
        const float u0 = U[m0 * kRows + r], u1 = U[m1 * kRows + r];
        const float u2 = U[m2 * kRows + r], u3 = U[m3 * kRows + r];
        acc = fmaf(-a0, u0, acc);
        acc = fmaf(-a1, u1, acc);
        acc = fmaf(-a2, u2, acc);
        acc = fmaf(-a3, u3, acc);
      }
      U[j * kRows + r] = acc;
    }
  }
  __syncthreads();
  // ---- outputs, u, log-decays and normalised keys
  for (int i = tid; i < n * kRows; i += kGdnThreads) {
    const int j = i / kRows, r = i % kRows;
    const float* cj = C + j * (n + 1);
    const uint8_t* al = alist + j * kMaxNodes;
    float acc = fmaf(cj[j], U[i], eg[j] * Z[i]);
    const int d = depth[j];
    for (int e = 0; e < d; e += 4) {
      const int m0 = al[e], m1 = al[e + 1], m2 = al[e + 2], m3 = al[e + 3];
      acc = fmaf(cj[m0], U[m0 * kRows + r], acc);
      acc = fmaf(cj[m1], U[m1 * kRows + r], acc);
      acc = fmaf(cj[m2], U[m2 * kRows + r], acc);
      acc = fmaf(cj[m3], U[m3 * kRows + r], acc);
    }
    const size_t row = (size_t)(q0 + j) * p.hv + h;
    p.out[row * kD + rb * kRows + r] = __float2bfloat16_rn(acc);
    p.cache_u[row * kD + rb * kRows + r] = U[i];
  }
  if (rb == 0)
    for (int j = tid; j < n; j += kGdnThreads) p.cache_g[(size_t)(q0 + j) * p.hv + h] = G[j];
  if (rb == 0 && h % (p.hv / p.hk) == 0)
    for (int i = tid; i < n * kD; i += kGdnThreads)
      p.cache_k[((size_t)(q0 + i / kD) * p.hk + hk) * kD + i % kD] = kh[(i / kD) * kLd + i % kD];
}

// Persist-on-accept of the recurrent state, every layer in one launch:
// S <- gamma_last S + sum over the accepted path of (gamma_last / gamma_m) u_m k_m^T,
// 32 rows of one head per CTA, in place.
__global__ void __launch_bounds__(kGdnThreads) gdn_commit_kernel(const GdnCommitParams p, const BatchDesc bd) {
  __shared__ __align__(16) float ks[kMaxNodes][kD];   // normalised keys of the path (32 KB)
  __shared__ float us[kMaxNodes][kCommitRows];   // this block's u rows of the path
  __shared__ float wt[kMaxNodes];          // e^{G_last - G_m}
  __shared__ int bad;
  const int layer = blockIdx.z, b = blockIdx.y;
  const int rb = blockIdx.x % (kD / kCommitRows), h = blockIdx.x / (kD / kCommitRows);
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
  for (int i = tid; i < a * kCommitRows; i += kGdnThreads) {
    const int m = p.path[(size_t)b * p.max_path + i / kCommitRows];
    us[i / kCommitRows][i % kCommitRows] = cu[((size_t)(q0 + m) * p.hv + h) * kD + rb * kCommitRows + i % kCommitRows];
  }
  for (int i = tid; i < a; i += kGdnThreads) {
    const int m = p.path[(size_t)b * p.max_path + i];
    wt[i] = __expf(g_last - cg[(size_t)(q0 + m) * p.hv + h]);
  }
  __syncthreads();
  const float gamma = __expf(g_last);
  // four consecutive columns per thread: 16-byte loads and stores of the state
  float4* st = reinterpret_cast<float4*>(p.state[layer] + (((size_t)b * p.hv + h) * kD + rb * kCommitRows) * kD);
  for (int i = tid; i < kCommitRows * kD / 4; i += kGdnThreads) {
    const int r = (i * 4) / kD, c = (i * 4) % kD;
    float4 acc = st[i];
    acc.x *= gamma; acc.y *= gamma; acc.z *= gamma; acc.w *= gamma;
    for (int m = 0; m < a; ++m) {
      const float wu = wt[m] * us[m][r];
      const float4 k4 = *reinterpret_cast<const float4*>(&ks[m][c]);
      acc.x = fmaf(wu, k4.x, acc.x);
      acc.y = fmaf(wu, k4.y, acc.y);
      acc.z = fmaf(wu, k4.z, acc.z);
      acc.w = fmaf(wu, k4.w, acc.w);
    }
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
// Block: 256 channels of one node (grid y = node row); the node's sequence
// is found in the batch's row offsets and its parents are read once into
// shared memory, so each thread issues its four window loads at once.
__global__ void __launch_bounds__(256) conv_tree_kernel(const ConvTreeParams p, const BatchDesc bd) {
  __shared__ int par[kMaxNodes];
  const int row = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  int lo = 0, hi = bd.batch;   // sequence b with q_indptr[b] <= row < q_indptr[b + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (bd.q_indptr[mid] <= row) lo = mid; else hi = mid;
  }
  const int b = lo;
  const int q0 = bd.q_indptr[b];
  const int n = bd.q_indptr[b + 1] - q0;
  const int j = row - q0;
  if (threadIdx.x < n) {
    const int t = threadIdx.x;
    int pt = p.parents[q0 + t];
    if ((t == 0 && pt != -1) || (t > 0 && (pt < 0 || pt >= t))) {
      if (blockIdx.x == 0 && t == j) report(p.dev_status, SD_DEV_BAD_PARENTS);
      pt = t == 0 ? -1 : t - 1;
    }
    par[t] = pt;
  }
  __syncthreads();
  if (c >= p.channels) return;
  // window, newest first: the node, its parent, ... then the cached inputs (newest first)
  int src[4];
  int u = j, t = 0;
  for (; t < 4 && u >= 0; ++t, u = par[u]) src[t] = u;
  const int on_tree = t;
  const float4 w = reinterpret_cast<const float4*>(p.weight)[c];   // w.w multiplies the node's own input
  const __nv_bfloat16* cs = p.conv_state + ((size_t)b * p.channels + c) * 3;
  float x[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    x[k] = k < on_tree ? bf2f(p.x[(size_t)(q0 + src[k]) * p.channels + c]) : bf2f(cs[2 - (k - on_tree)]);
  const float acc = w.w * x[0] + w.z * x[1] + w.y * x[2] + w.x * x[3];
  p.y[(size_t)row * p.channels + c] = __float2bfloat16_rn(acc / (1.0f + __expf(-acc)));
}

}  // namespace

size_t gdn_smem_bytes(int max_nodes) { return gdn_tree_smem(max_nodes, 64); }

template <int kRows>
cudaError_t launch_gdn_rows(const GdnParams& p, const BatchDesc& bd, cudaStream_t st) {
  const size_t smem = gdn_tree_smem(bd.max_nodes, kRows);
  cudaError_t e =
      cudaFuncSetAttribute(gdn_tree_kernel<kRows>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  gdn_tree_kernel<kRows><<<dim3(p.hv * (kD / kRows), bd.batch), kGdnThreads, smem, st>>>(p, bd);
  return cudaGetLastError();
}

cudaError_t launch_gdn_tree(const GdnParams& p, const BatchDesc& bd, cudaStream_t st) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 152;
  // 16-row CTAs while they fit in about four per SM, else 64-row CTAs
  const long long ctas16 = (long long)bd.batch * p.hv * (kD / 16);
  return ctas16 <= 4LL * sms ? launch_gdn_rows<16>(p, bd, st) : launch_gdn_rows<64>(p, bd, st);
}

cudaError_t launch_gdn_commit(const GdnCommitParams& p, const BatchDesc& bd, cudaStream_t st) {
  gdn_commit_kernel<<<dim3(p.hv * (kD / kCommitRows), bd.batch, p.num_layers), kGdnThreads, 0, st>>>(p, bd);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.channels == 0) return e;
  conv_commit_kernel<<<dim3((p.channels + 255) / 256, bd.batch, p.num_layers), 256, 0, st>>>(p, bd);
  return cudaGetLastError();
}

cudaError_t launch_conv_tree(const ConvTreeParams& p, const BatchDesc& bd, cudaStream_t st) {
  conv_tree_kernel<<<dim3((p.channels + 255) / 256, bd.total_nodes), 256, 0, st>>>(p, bd);
  return cudaGetLastError();
}

}  // namespace sdv
