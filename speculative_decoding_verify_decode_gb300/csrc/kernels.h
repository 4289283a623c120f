// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace sdv {

// Verify attention on tcgen05 tiles with TMA-staged pages (+ merge when num_splits > 1).
struct TcPlan {
  int hpc;      // query heads of a KV group handled by one CTA: 6, 3, 2 or 1
  int hparts;   // CTAs per (split, KV head): ceil(6 / hpc)
  int nq;       // query columns per CTA: hpc x max nodes rounded up to 16 (>= 32)
};
// bf16 caches: the ring-buffered kernel (attn_ring_kernel.cuh), up to 144 query columns per CTA.
constexpr int kRingMaxNQ = 144;
// The bf16 page tensor map both bf16 kernels load through (one 8 KB page of one KV head per box).
bool bf16_page_map(CUtensorMap* map, const void* cache, int pool_pages);
TcPlan ring_plan(int max_nodes);
cudaError_t launch_attn_ring(const AttnParams& p, const BatchDesc& bd, cudaStream_t st);
// its sliding-window instances (attn_ring_win.cu)
cudaError_t launch_ring_window(const CUtensorMap& mk, const CUtensorMap& mv, const AttnParams& p,
                               const BatchDesc& bd, const TcPlan& pl, cudaStream_t st);
// attn_tc_kernel.cuh, up to 96 query columns per CTA: e4m3 caches (p.k_cache8 / p.v_cache8 with
// p.k_scale / p.v_scale, attn_tc8.cu), and bf16 caches when every context split is a single tile
// (attn_tc16.cu).
constexpr int kTcMaxNQ = 96;
TcPlan tc_plan(int max_nodes);
size_t tc_smem_bytes(int nq);
cudaError_t launch_attn_tc8(const AttnParams& p, const BatchDesc& bd, cudaStream_t st);
cudaError_t launch_attn_tc16(const AttnParams& p, const BatchDesc& bd, cudaStream_t st);

// Host-side validation of a verify-attention shape (the status sd_verify_attn returns for it).
sd_status verify_shape_status(const sd_shape* s);

// Log-sum-exp merge of the split partials into the bf16 output.
cudaError_t launch_attn_merge(const AttnParams& p, const BatchDesc& bd, cudaStream_t st);

// Argmax + greedy path selection.
struct AcceptParams {
  const float* logits;
  const int* parents;
  const int* draft_tokens;
  int* accept_len;
  int* path;
  int* out_tokens;
  int* target_tokens;   // nullable
  int* dev_status;      // nullable
  void* partial;        // [total_nodes][chunks] (value, index) pairs
  int vocab;
  int chunks;           // row chunks of kAcceptChunk logits
  int max_path;
};
constexpr int kAcceptChunk = 4096;
cudaError_t launch_accept(const AcceptParams& p, const BatchDesc& bd, cudaStream_t st);

// Sampling-based verify: per-chunk softmax statistics, then one CTA per sequence walking its tree.
constexpr int kSampleTile = 4096;        // logits per tile of the statistics pass and of the inverse-CDF search
constexpr int kSampleMaxTiles = 512;    // vocabulary <= 512 x 4096 = 2048 x 1024
struct SampleParams {
  const float* logits;        // [sumN][V] target logits
  const float* draft_probs;   // [sumN][V] draft distribution at each node (its children were drawn from it)
  const int* parents;
  const int* draft_tokens;
  const float* r_accept;      // [sumN] uniforms of the nodes' acceptance tests
  const float* r_sample;      // [sumN] uniforms of a bonus drawn at the node
  int* accept_len;
  int* path;
  int* out_tokens;
  int* dev_status;            // nullable
  void* partial;              // [sumN][chunks] (max, sum) pairs per 1024-logit tile
  float* resid;               // [sumN][chunks] per tile: sum of max(0, p - q) (the first residual)
  int vocab;
  int chunks;
  int max_path;
  float inv_t;                // 1 / temperature
};
cudaError_t launch_sample_accept(const SampleParams& p, const BatchDesc& bd, cudaStream_t st);

// Commit of accepted K/V for all layers.
struct CommitParams {
  void* k_cache[kMaxLayers];
  void* v_cache[kMaxLayers];
  const void* k_new[kMaxLayers];
  const void* v_new[kMaxLayers];
  const int* page_table;
  const int* ctx_lens;
  int* new_ctx_lens;    // nullable
  const int* accept_len;
  const int* path;
  int* dev_status;      // nullable
  int max_path;
  int max_pages;
  int num_pool_pages;
  int num_layers;
  int fp8;                       // caches hold e4m3 codes: rows are quantised on the way in
  float k_inv[kMaxLayers];       // fp32 reciprocals of the per-layer K / V scales (fp8 only)
  float v_inv[kMaxLayers];
};
cudaError_t launch_commit(const CommitParams& p, const BatchDesc& bd, cudaStream_t st);

// Draft-tree construction: per-position top-K of the draft logits, then a best-first tree.
constexpr int kDdTopKMax = 8;      // candidates per position
constexpr int kDdChunk = 4096;     // logits per chunk of the top-K pass (16 per thread)
struct DdtreeParams {
  const float* logits;       // [batch][positions][vocab]
  const int* root_tokens;    // [batch]
  int* parents;              // [batch][1 + budget]
  int* tokens;               // [batch][1 + budget]
  float* scores;             // [batch][1 + budget], nullable
  int* dev_status;           // nullable
  float* part_v;             // [batch * positions][chunks][8] chunk top-8 values
  int* part_i;               // [batch * positions][chunks][8] and their token ids
  float* part_ms;            // [batch * positions][chunks][2] (max, sum of exp(x - max))
  int batch, positions, vocab, topk, budget, chunks;
};
size_t ddtree_smem_bytes(int chunks);
cudaError_t launch_ddtree(const DdtreeParams& p, cudaStream_t st);

// Tree Gated DeltaNet (hybrid layers): tree convolution, gated delta rule over the tree, persist-on-accept.
constexpr int kGdnDim = 128;       // d_k = d_v
struct GdnParams {
  const __nv_bfloat16* q;    // [sumN][hk][128]
  const __nv_bfloat16* k;    // [sumN][hk][128]
  const __nv_bfloat16* v;    // [sumN][hv][128]
  const float* g;            // [sumN][hv] log decay
  const float* beta;         // [sumN][hv]
  const float* state;        // [B][hv][128 rows][128]
  const int* parents;
  __nv_bfloat16* out;        // [sumN][hv][128]
  float* cache_u;            // [sumN][hv][128]
  float* cache_g;            // [sumN][hv] log of the path's decay product
  float* cache_k;            // [sumN][hk][128] normalised keys
  int* dev_status;
  int hk, hv;
};
struct GdnCommitParams {
  float* state[kMaxLayers];
  const float* cache_u[kMaxLayers];
  const float* cache_g[kMaxLayers];
  const float* cache_k[kMaxLayers];
  __nv_bfloat16* conv_state[kMaxLayers];   // [B][channels][3]
  const __nv_bfloat16* x[kMaxLayers];      // [sumN][channels]
  const int* accept_len;
  const int* path;
  int* dev_status;
  int max_path, num_layers, hk, hv, channels;
};
struct ConvTreeParams {
  const __nv_bfloat16* x;           // [sumN][channels]
  const float* weight;              // [channels][4]
  const __nv_bfloat16* conv_state;  // [B][channels][3], oldest first
  const int* parents;
  __nv_bfloat16* y;                 // [sumN][channels]
  int* dev_status;
  int channels;
};
size_t gdn_smem_bytes(int max_nodes);
cudaError_t launch_gdn_tree(const GdnParams& p, const BatchDesc& bd, cudaStream_t st);
cudaError_t launch_gdn_commit(const GdnCommitParams& p, const BatchDesc& bd, cudaStream_t st);
cudaError_t launch_conv_tree(const ConvTreeParams& p, const BatchDesc& bd, cudaStream_t st);

}  // namespace sdv
