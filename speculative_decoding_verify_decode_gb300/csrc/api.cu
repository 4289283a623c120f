// C-ABI entry points (declared in include/sd_verify.h): host-side argument
// checks, workspace layout, split-KV sizing, and the kernel launches.  Nothing
// here allocates device memory or synchronises; every launch goes on the
// caller's stream.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/sd_gdn.h"
#include "common.cuh"
#include "kernels.h"

using namespace sdv;

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

sd_status fill_batch(int batch, const int* indptr, BatchDesc* bd) {
  if (batch < 1 || batch > kMaxBatch || indptr == nullptr) return SD_ERR_INVALID_ARG;
  if (indptr[0] != 0) return SD_ERR_INVALID_ARG;
  bd->batch = batch;
  bd->max_nodes = 0;
  for (int b = 0; b <= batch; ++b) bd->q_indptr[b] = indptr[b];
  for (int b = 0; b < batch; ++b) {
    const int n = indptr[b + 1] - indptr[b];
    if (n < 1) return SD_ERR_INVALID_ARG;
    if (n > kMaxNodes) return SD_ERR_UNSUPPORTED;
    if (n > bd->max_nodes) bd->max_nodes = n;
  }
  bd->total_nodes = indptr[batch];
  return SD_OK;
}

sd_status check_shape(const sd_shape* s, BatchDesc* bd) {
  if (s == nullptr) return SD_ERR_INVALID_ARG;
  if (s->num_q_heads != kHq || s->num_kv_heads != kHkv || s->head_dim != kDim || s->page_size != kPage)
    return SD_ERR_UNSUPPORTED;
  if (s->max_pages_per_seq < 1 || s->num_pool_pages < 1 || s->num_splits < 0 || s->window < 0)
    return SD_ERR_INVALID_ARG;
  if ((long long)s->max_pages_per_seq * kPage > (1LL << 30)) return SD_ERR_UNSUPPORTED;
  return fill_batch(s->batch, s->q_indptr_h, bd);
}

int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
    cudaGetLastError();  // no device here: size for a 152-SM part
    return 152;
  }
  return sms;
}

struct SplitPlan {
  int chunk;     // context tokens per context split
  int nsplit;    // splits in the grid: the draft split + the context splits
};

// Context tokens per context split, for a kernel that runs `hparts` CTAs per
// (split, sequence, KV head).  Every split CTA (one per SM) pays a fixed set-up
// and epilogue, so a single sequence gets one wave of CTAs, each with an equal
// share of the 128-token tiles; a batch, whose context lengths are not known on
// the host, is cut for two waves of the worst case (every sequence full), which
// keeps the last wave short when the lengths are ragged.  num_splits > 0 fixes
// the number of context chunks per (sequence, KV head) instead.
SplitPlan plan_splits(const sd_shape* s, const BatchDesc& bd, int hparts) {
  const int tile = kTileTokens;
  long long max_ctx = (long long)s->max_pages_per_seq * kPage;
  // with a window only the tiles from window_base on are read: at most W - 1 positions plus the
  // rounding to a tile boundary
  if (s->window > 0 && (long long)s->window + 2 * tile < max_ctx) max_ctx = (long long)s->window + 2 * tile;
  const long long max_tiles = (max_ctx + tile - 1) / tile;
  long long chunk;
  if (s->num_splits > 0) {
    chunk = (max_ctx + s->num_splits - 1) / s->num_splits;
  } else {
    const long long streams = (long long)bd.batch * kHkv * hparts;
    const long long waves = bd.batch > 1 ? 2 : 1;
    long long slots = waves * device_sm_count() - streams;    // the draft CTAs take one slot per stream
    if (slots < streams) slots = streams;
    const long long per_cta = (streams * max_tiles + slots - 1) / slots;
    chunk = (per_cta < 1 ? 1 : per_cta) * tile;
  }
  chunk = (chunk + tile - 1) / tile * tile;
  if (chunk < tile) chunk = tile;
  const long long n = 1 + (max_ctx + chunk - 1) / chunk;   // the draft split + the context chunks
  return SplitPlan{(int)chunk, (int)n};
}

// The plan of each cache kind: bf16 caches run the ring kernel's plan, e4m3 caches the converter kernel's.
SplitPlan plan_for(const sd_shape* s, const BatchDesc& bd, bool fp8) {
  return plan_splits(s, bd, fp8 ? tc_plan(bd.max_nodes).hparts : ring_plan(bd.max_nodes).hparts);
}

// bf16 caches: when every context split is a single tile and attn_tc_kernel cuts the query heads the
// same way (so the grid, the plan and the workspace are the ring kernel's), the layer is a latency
// chain and attn_tc_kernel's shorter one wins; otherwise the ring kernel streams the tiles.
bool short_bf16(const SplitPlan& pl, const BatchDesc& bd) {
  return pl.chunk == kTileTokens && tc_plan(bd.max_nodes).hparts == ring_plan(bd.max_nodes).hparts &&
         tc_plan(bd.max_nodes).hpc * bd.max_nodes <= kTcMaxNQ;
}

size_t attn_workspace(const SplitPlan& pl, const BatchDesc& bd) {
  if (pl.nsplit <= 1) return 0;
  const size_t rows = (size_t)pl.nsplit * bd.total_nodes * kHq;
  return align_up(rows * kDim * sizeof(__nv_bfloat16)) + align_up(rows * sizeof(float));
}

sd_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SD_OK : SD_ERR_CUDA; }

// The kernels move bf16 rows with 16-byte vector accesses.
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A per-tensor scale of an e4m3 cache: positive, finite, with a finite fp32 reciprocal.
bool scale_ok(float s) { return std::isfinite(s) && s > 0.f && std::isfinite(1.0f / s); }

sd_status check_gdn_shape(const sd_gdn_shape* s, BatchDesc* bd) {
  if (s == nullptr) return SD_ERR_INVALID_ARG;
  if (s->head_dim != kGdnDim) return SD_ERR_UNSUPPORTED;
  if (s->num_k_heads < 1 || s->num_v_heads < s->num_k_heads || s->num_v_heads % s->num_k_heads != 0)
    return SD_ERR_INVALID_ARG;
  if (s->num_v_heads > 256) return SD_ERR_UNSUPPORTED;
  return fill_batch(s->batch, s->q_indptr_h, bd);
}

// Tree cache of one layer: u [sumN][H_v][128], log decay [sumN][H_v], normalised keys [sumN][H_k][128] (fp32).
struct GdnCacheLayout {
  size_t u, g, k, total;
};
GdnCacheLayout gdn_cache_layout(const sd_gdn_shape* s, const BatchDesc& bd) {
  GdnCacheLayout l;
  const size_t n = (size_t)bd.total_nodes;
  l.u = 0;
  l.g = align_up(n * s->num_v_heads * kGdnDim * sizeof(float));
  l.k = l.g + align_up(n * s->num_v_heads * sizeof(float));
  l.total = l.k + align_up(n * s->num_k_heads * kGdnDim * sizeof(float));
  return l;
}

// sd_verify_attn and sd_verify_attn_fp8: checks, split plan, parameter block, launch.
sd_status verify_attn(const sd_shape* shape, const void* q, const void* k_cache, const void* v_cache,
                      const void* k_new, const void* v_new, const int* page_table, const int* ctx_lens,
                      const int* parents, void* out, float* lse, void* workspace, size_t ws_bytes, int* dev_status,
                      void* stream, bool fp8, float k_scale, float v_scale) {
  BatchDesc bd;
  sd_status st = check_shape(shape, &bd);
  if (st != SD_OK) return st;
  if (!q || !k_cache || !v_cache || !k_new || !v_new || !page_table || !ctx_lens || !parents || !out)
    return SD_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new) ||
      !aligned16(out) || (workspace != nullptr && !aligned16(workspace)))
    return SD_ERR_INVALID_ARG;
  if (fp8 && (!scale_ok(k_scale) || !scale_ok(v_scale))) return SD_ERR_INVALID_ARG;
  const SplitPlan pl = plan_for(shape, bd, fp8);
  const size_t need = attn_workspace(pl, bd);
  if (need > 0 && (workspace == nullptr || ws_bytes < need)) return SD_ERR_WORKSPACE;

  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const __nv_bfloat16*>(q);
  if (fp8) {
    p.k_cache8 = static_cast<const uint8_t*>(k_cache);
    p.v_cache8 = static_cast<const uint8_t*>(v_cache);
    p.k_scale = k_scale;
    p.v_scale = v_scale;
  } else {
    p.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
    p.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  }
  p.k_new = static_cast<const __nv_bfloat16*>(k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(v_new);
  p.page_table = page_table;
  p.ctx_lens = ctx_lens;
  p.parents = parents;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.dev_status = dev_status;
  p.max_pages = shape->max_pages_per_seq;
  p.num_pool_pages = shape->num_pool_pages;
  p.chunk = pl.chunk;
  p.num_splits = pl.nsplit;
  p.window = shape->window;
  p.ctx_stable = shape->ctx_stable != 0;
  if (need > 0) {
    const size_t rows = (size_t)pl.nsplit * bd.total_nodes * kHq;
    p.o_part = static_cast<__nv_bfloat16*>(workspace);
    p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + align_up(rows * kDim * sizeof(__nv_bfloat16)));
  }
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (fp8) return cuda_status(launch_attn_tc8(p, bd, cs));
  return cuda_status(short_bf16(pl, bd) ? launch_attn_tc16(p, bd, cs) : launch_attn_ring(p, bd, cs));
}

// sd_kv_commit and sd_kv_commit_fp8.
sd_status kv_commit(const sd_shape* shape, int num_layers, void* const* k_cache_layers, void* const* v_cache_layers,
                    const float* k_scales, const float* v_scales, const void* const* k_new_layers,
                    const void* const* v_new_layers, const int* page_table, const int* ctx_lens, int* new_ctx_lens,
                    const int* accept_len, const int* path, int max_path, int* dev_status, void* stream, bool fp8) {
  BatchDesc bd;
  sd_status st = check_shape(shape, &bd);
  if (st != SD_OK) return st;
  if (num_layers < 1) return SD_ERR_INVALID_ARG;
  if (num_layers > kMaxLayers) return SD_ERR_UNSUPPORTED;
  if (!k_cache_layers || !v_cache_layers || !k_new_layers || !v_new_layers || !page_table || !ctx_lens ||
      !accept_len || !path || max_path < 1)
    return SD_ERR_INVALID_ARG;
  if (fp8 && (!k_scales || !v_scales)) return SD_ERR_INVALID_ARG;
  if (new_ctx_lens != nullptr && new_ctx_lens == ctx_lens) return SD_ERR_INVALID_ARG;
  CommitParams p;
  std::memset(&p, 0, sizeof(p));
  for (int l = 0; l < num_layers; ++l) {
    if (!k_cache_layers[l] || !v_cache_layers[l] || !k_new_layers[l] || !v_new_layers[l])
      return SD_ERR_INVALID_ARG;
    if (!aligned16(k_cache_layers[l]) || !aligned16(v_cache_layers[l]) || !aligned16(k_new_layers[l]) ||
        !aligned16(v_new_layers[l]))
      return SD_ERR_INVALID_ARG;
    if (fp8) {
      if (!scale_ok(k_scales[l]) || !scale_ok(v_scales[l])) return SD_ERR_INVALID_ARG;
      p.k_inv[l] = 1.0f / k_scales[l];
      p.v_inv[l] = 1.0f / v_scales[l];
    }
    p.k_cache[l] = k_cache_layers[l];
    p.v_cache[l] = v_cache_layers[l];
    p.k_new[l] = k_new_layers[l];
    p.v_new[l] = v_new_layers[l];
  }
  p.fp8 = fp8 ? 1 : 0;
  p.page_table = page_table;
  p.ctx_lens = ctx_lens;
  p.new_ctx_lens = new_ctx_lens;
  p.accept_len = accept_len;
  p.path = path;
  p.dev_status = dev_status;
  p.max_path = max_path;
  p.max_pages = shape->max_pages_per_seq;
  p.num_pool_pages = shape->num_pool_pages;
  p.num_layers = num_layers;
  return cuda_status(launch_commit(p, bd, static_cast<cudaStream_t>(stream)));
}

}  // namespace

sd_status sdv::verify_shape_status(const sd_shape* s) {
  BatchDesc bd;
  return check_shape(s, &bd);
}

extern "C" {

const char* sd_status_string(sd_status s) {
  switch (s) {
    case SD_OK: return "ok";
    case SD_ERR_INVALID_ARG: return "invalid argument";
    case SD_ERR_UNSUPPORTED: return "unsupported shape";
    case SD_ERR_CUDA: return "CUDA error";
    case SD_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

size_t sd_verify_attn_workspace_size(const sd_shape* shape) {
  BatchDesc bd;
  if (check_shape(shape, &bd) != SD_OK) return 0;
  // one size serves both cache kinds (sd_verify_attn and sd_verify_attn_fp8 share the query)
  const size_t a = attn_workspace(plan_for(shape, bd, false), bd), b = attn_workspace(plan_for(shape, bd, true), bd);
  return a > b ? a : b;
}

sd_status sd_verify_attn(const sd_shape* shape, const void* q, const void* k_cache, const void* v_cache,
                         const void* k_new, const void* v_new, const int* page_table, const int* ctx_lens,
                         const int* parents, void* out, float* lse, void* workspace, size_t ws_bytes,
                         int* dev_status, void* stream) {
  return verify_attn(shape, q, k_cache, v_cache, k_new, v_new, page_table, ctx_lens, parents, out, lse, workspace,
                     ws_bytes, dev_status, stream, false, 1.f, 1.f);
}

sd_status sd_verify_attn_fp8(const sd_shape* shape, const void* q, const void* k_cache, const void* v_cache,
                             float k_scale, float v_scale, const void* k_new, const void* v_new,
                             const int* page_table, const int* ctx_lens, const int* parents, void* out, float* lse,
                             void* workspace, size_t ws_bytes, int* dev_status, void* stream) {
  return verify_attn(shape, q, k_cache, v_cache, k_new, v_new, page_table, ctx_lens, parents, out, lse, workspace,
                     ws_bytes, dev_status, stream, true, k_scale, v_scale);
}

size_t sd_accept_workspace_size(int batch, const int* q_indptr_h, int vocab) {
  BatchDesc bd;
  if (fill_batch(batch, q_indptr_h, &bd) != SD_OK || vocab < 1) return 0;
  const size_t chunks = ((size_t)vocab + kAcceptChunk - 1) / kAcceptChunk;
  return align_up((size_t)bd.total_nodes * chunks * 8);
}

sd_status sd_accept(int batch, const int* q_indptr_h, int vocab, const float* logits, const int* parents,
                    const int* draft_tokens, int* accept_len, int* path, int* out_tokens, int* target_tokens,
                    int max_path, void* workspace, size_t ws_bytes, int* dev_status, void* stream) {
  BatchDesc bd;
  sd_status st = fill_batch(batch, q_indptr_h, &bd);
  if (st != SD_OK) return st;
  if (vocab < 1 || max_path < 1 || !logits || !parents || !draft_tokens || !accept_len || !path || !out_tokens)
    return SD_ERR_INVALID_ARG;
  const size_t need = sd_accept_workspace_size(batch, q_indptr_h, vocab);
  if (workspace == nullptr || ws_bytes < need) return SD_ERR_WORKSPACE;
  AcceptParams p;
  p.logits = logits;
  p.parents = parents;
  p.draft_tokens = draft_tokens;
  p.accept_len = accept_len;
  p.path = path;
  p.out_tokens = out_tokens;
  p.target_tokens = target_tokens;
  p.dev_status = dev_status;
  p.partial = workspace;
  p.vocab = vocab;
  p.chunks = (vocab + kAcceptChunk - 1) / kAcceptChunk;
  p.max_path = max_path;
  return cuda_status(launch_accept(p, bd, static_cast<cudaStream_t>(stream)));
}

sd_status sd_kv_commit(const sd_shape* shape, int num_layers, void* const* k_cache_layers,
                       void* const* v_cache_layers, const void* const* k_new_layers,
                       const void* const* v_new_layers, const int* page_table, const int* ctx_lens,
                       int* new_ctx_lens, const int* accept_len, const int* path, int max_path,
                       int* dev_status, void* stream) {
  return kv_commit(shape, num_layers, k_cache_layers, v_cache_layers, nullptr, nullptr, k_new_layers, v_new_layers,
                   page_table, ctx_lens, new_ctx_lens, accept_len, path, max_path, dev_status, stream, false);
}

sd_status sd_kv_commit_fp8(const sd_shape* shape, int num_layers, void* const* k_cache_layers,
                           void* const* v_cache_layers, const float* k_scales, const float* v_scales,
                           const void* const* k_new_layers, const void* const* v_new_layers,
                           const int* page_table, const int* ctx_lens, int* new_ctx_lens, const int* accept_len,
                           const int* path, int max_path, int* dev_status, void* stream) {
  return kv_commit(shape, num_layers, k_cache_layers, v_cache_layers, k_scales, v_scales, k_new_layers,
                   v_new_layers, page_table, ctx_lens, new_ctx_lens, accept_len, path, max_path, dev_status, stream,
                   true);
}

size_t sd_sample_accept_workspace_size(int batch, const int* q_indptr_h, int vocab) {
  BatchDesc bd;
  if (fill_batch(batch, q_indptr_h, &bd) != SD_OK || vocab < 1) return 0;
  const size_t chunks = ((size_t)vocab + kSampleTile - 1) / kSampleTile;
  return align_up((size_t)bd.total_nodes * chunks * 8) + align_up((size_t)bd.total_nodes * chunks * 4);
}

sd_status sd_sample_accept(int batch, const int* q_indptr_h, int vocab, float temperature, const float* logits,
                           const float* draft_probs, const int* parents, const int* draft_tokens,
                           const float* r_accept, const float* r_sample, int* accept_len, int* path,
                           int* out_tokens, int max_path, void* workspace, size_t ws_bytes, int* dev_status,
                           void* stream) {
  BatchDesc bd;
  sd_status st = fill_batch(batch, q_indptr_h, &bd);
  if (st != SD_OK) return st;
  if (vocab < 1 || max_path < 1 || !logits || !draft_probs || !parents || !draft_tokens || !r_accept ||
      !r_sample || !accept_len || !path || !out_tokens)
    return SD_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !std::isfinite(temperature) || !std::isfinite(1.0f / temperature))
    return SD_ERR_INVALID_ARG;
  if ((long long)vocab > (long long)kSampleMaxTiles * kSampleTile) return SD_ERR_UNSUPPORTED;
  const size_t need = sd_sample_accept_workspace_size(batch, q_indptr_h, vocab);
  if (workspace == nullptr || ws_bytes < need || !aligned16(workspace)) return SD_ERR_WORKSPACE;
  SampleParams p;
  p.logits = logits;
  p.draft_probs = draft_probs;
  p.parents = parents;
  p.draft_tokens = draft_tokens;
  p.r_accept = r_accept;
  p.r_sample = r_sample;
  p.accept_len = accept_len;
  p.path = path;
  p.out_tokens = out_tokens;
  p.dev_status = dev_status;
  p.partial = workspace;
  p.vocab = vocab;
  p.chunks = (vocab + kSampleTile - 1) / kSampleTile;
  p.resid = reinterpret_cast<float*>(static_cast<char*>(workspace) + align_up((size_t)bd.total_nodes * p.chunks * 8));
  p.max_path = max_path;
  p.inv_t = 1.0f / temperature;
  return cuda_status(launch_sample_accept(p, bd, static_cast<cudaStream_t>(stream)));
}

size_t sd_gdn_tree_cache_size(const sd_gdn_shape* shape) {
  BatchDesc bd;
  if (check_gdn_shape(shape, &bd) != SD_OK) return 0;
  return gdn_cache_layout(shape, bd).total;
}

sd_status sd_gdn_conv_tree(int batch, const int* q_indptr_h, int channels, const void* x, const float* weight,
                           const void* conv_state, const int* parents, void* y, int* dev_status, void* stream) {
  BatchDesc bd;
  sd_status st = fill_batch(batch, q_indptr_h, &bd);
  if (st != SD_OK) return st;
  if (channels < 1 || !x || !weight || !conv_state || !parents || !y) return SD_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(weight) || !aligned16(y)) return SD_ERR_INVALID_ARG;
  ConvTreeParams p;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.weight = weight;
  p.conv_state = static_cast<const __nv_bfloat16*>(conv_state);
  p.parents = parents;
  p.y = static_cast<__nv_bfloat16*>(y);
  p.dev_status = dev_status;
  p.channels = channels;
  return cuda_status(launch_conv_tree(p, bd, static_cast<cudaStream_t>(stream)));
}

sd_status sd_gdn_tree(const sd_gdn_shape* shape, const void* q, const void* k, const void* v, const float* g,
                      const float* beta, const float* state, const int* parents, void* out, void* tree_cache,
                      size_t cache_bytes, int* dev_status, void* stream) {
  BatchDesc bd;
  sd_status st = check_gdn_shape(shape, &bd);
  if (st != SD_OK) return st;
  if (!q || !k || !v || !g || !beta || !state || !parents || !out) return SD_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(state) || !aligned16(out))
    return SD_ERR_INVALID_ARG;
  const GdnCacheLayout l = gdn_cache_layout(shape, bd);
  if (tree_cache == nullptr || cache_bytes < l.total || !aligned16(tree_cache)) return SD_ERR_WORKSPACE;
  GdnParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.g = g;
  p.beta = beta;
  p.state = state;
  p.parents = parents;
  p.out = static_cast<__nv_bfloat16*>(out);
  char* c = static_cast<char*>(tree_cache);
  p.cache_u = reinterpret_cast<float*>(c + l.u);
  p.cache_g = reinterpret_cast<float*>(c + l.g);
  p.cache_k = reinterpret_cast<float*>(c + l.k);
  p.dev_status = dev_status;
  p.hk = shape->num_k_heads;
  p.hv = shape->num_v_heads;
  return cuda_status(launch_gdn_tree(p, bd, static_cast<cudaStream_t>(stream)));
}

sd_status sd_gdn_commit(const sd_gdn_shape* shape, int num_layers, float* const* state_layers,
                        const void* const* tree_cache_layers, int channels, void* const* conv_state_layers,
                        const void* const* x_layers, const int* accept_len, const int* path, int max_path,
                        int* dev_status, void* stream) {
  BatchDesc bd;
  sd_status st = check_gdn_shape(shape, &bd);
  if (st != SD_OK) return st;
  if (num_layers < 1 || channels < 0 || max_path < 1 || !state_layers || !tree_cache_layers || !accept_len || !path)
    return SD_ERR_INVALID_ARG;
  if (num_layers > kMaxLayers) return SD_ERR_UNSUPPORTED;
  if (channels > 0 && (!conv_state_layers || !x_layers)) return SD_ERR_INVALID_ARG;
  const GdnCacheLayout l = gdn_cache_layout(shape, bd);
  GdnCommitParams p;
  std::memset(&p, 0, sizeof(p));
  for (int i = 0; i < num_layers; ++i) {
    if (!state_layers[i] || !tree_cache_layers[i] || !aligned16(state_layers[i]) || !aligned16(tree_cache_layers[i]))
      return SD_ERR_INVALID_ARG;
    const char* c = static_cast<const char*>(tree_cache_layers[i]);
    p.state[i] = state_layers[i];
    p.cache_u[i] = reinterpret_cast<const float*>(c + l.u);
    p.cache_g[i] = reinterpret_cast<const float*>(c + l.g);
    p.cache_k[i] = reinterpret_cast<const float*>(c + l.k);
    if (channels > 0) {
      if (!conv_state_layers[i] || !x_layers[i]) return SD_ERR_INVALID_ARG;
      p.conv_state[i] = static_cast<__nv_bfloat16*>(conv_state_layers[i]);
      p.x[i] = static_cast<const __nv_bfloat16*>(x_layers[i]);
    }
  }
  p.accept_len = accept_len;
  p.path = path;
  p.dev_status = dev_status;
  p.max_path = max_path;
  p.num_layers = num_layers;
  p.hk = shape->num_k_heads;
  p.hv = shape->num_v_heads;
  p.channels = channels;
  return cuda_status(launch_gdn_commit(p, bd, static_cast<cudaStream_t>(stream)));
}

size_t sd_ddtree_workspace_size(int batch, int positions, int vocab, int topk) {
  if (batch < 1 || batch > kMaxBatch || positions < 1 || positions > kMaxNodes || topk < 1 ||
      topk > kDdTopKMax || vocab < topk)
    return 0;
  const size_t rows = (size_t)batch * positions;
  const size_t chunks = ((size_t)vocab + kDdChunk - 1) / kDdChunk;
  return align_up(rows * chunks * kDdTopKMax * sizeof(float)) + align_up(rows * chunks * kDdTopKMax * sizeof(int)) +
         align_up(rows * chunks * 2 * sizeof(float));
}

sd_status sd_ddtree_build(int batch, int positions, int vocab, int topk, int budget, const float* draft_logits,
                          const int* root_tokens, int* parents, int* tokens, float* scores, void* workspace,
                          size_t ws_bytes, int* dev_status, void* stream) {
  if (batch < 1 || positions < 1 || topk < 1 || budget < 1 || vocab < 1) return SD_ERR_INVALID_ARG;
  if (batch > kMaxBatch || positions > kMaxNodes || topk > kDdTopKMax || budget > kMaxNodes - 1)
    return SD_ERR_UNSUPPORTED;
  if (vocab < topk || !draft_logits || !root_tokens || !parents || !tokens) return SD_ERR_INVALID_ARG;
  const size_t need = sd_ddtree_workspace_size(batch, positions, vocab, topk);
  if (workspace == nullptr || ws_bytes < need || !aligned16(workspace)) return SD_ERR_WORKSPACE;
  if ((vocab % 4 == 0) && !aligned16(draft_logits)) return SD_ERR_INVALID_ARG;
  const int chunks = (vocab + kDdChunk - 1) / kDdChunk;
  if (ddtree_smem_bytes(chunks) > 200 * 1024) return SD_ERR_UNSUPPORTED;
  DdtreeParams p;
  std::memset(&p, 0, sizeof(p));
  const size_t rows = (size_t)batch * positions;
  char* ws = static_cast<char*>(workspace);
  p.logits = draft_logits;
  p.root_tokens = root_tokens;
  p.parents = parents;
  p.tokens = tokens;
  p.scores = scores;
  p.dev_status = dev_status;
  p.part_v = reinterpret_cast<float*>(ws);
  p.part_i = reinterpret_cast<int*>(ws + align_up(rows * chunks * kDdTopKMax * sizeof(float)));
  p.part_ms = reinterpret_cast<float*>(ws + align_up(rows * chunks * kDdTopKMax * sizeof(float)) +
                                       align_up(rows * chunks * kDdTopKMax * sizeof(int)));
  p.batch = batch;
  p.positions = positions;
  p.vocab = vocab;
  p.topk = topk;
  p.budget = budget;
  p.chunks = chunks;
  return cuda_status(launch_ddtree(p, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
