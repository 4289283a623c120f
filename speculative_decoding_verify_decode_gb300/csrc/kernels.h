// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include "common.cuh"

namespace sdv {

// Verify attention on mma.sync tiles: split kernel (+ merge when num_splits > 1).
int attn_mma_tile();
int attn_mma_ctas_per_split(const BatchDesc& bd);
cudaError_t launch_attn_mma(const AttnParams& p, const BatchDesc& bd, cudaStream_t st);

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
};
cudaError_t launch_commit(const CommitParams& p, const BatchDesc& bd, cudaStream_t st);

}  // namespace sdv
