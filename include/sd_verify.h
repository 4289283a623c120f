/*
 * sd_verify.h — C ABI of the speculative-decoding verify step (sm_103a).
 *
 * One verify step of greedy speculative decoding, as the pages describe it:
 * the target model scores a whole draft block (a chain, or a DDTree-style
 * token tree) in one forward pass, keeps the longest draft prefix that
 * matches its own greedy choices, emits one bonus token, and appends the
 * accepted tokens' K/V to the cache.  Sources, by page title:
 *
 *  [S5] «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍»
 *       (blog.xiaohack.org/246393): 为什么我们要做这个测试 (24 Q heads, 4 KV
 *       heads, head dim 256; one full-attention layer in four); 架构设计
 *       (greedy verify, draft block 16); 从自回归到 DDTree (accept length, tree
 *       budget); 关键突破 (tree mask along the parent chain; logits buffer of
 *       vocab x (budget + 1); a persist kernel writing accepted state in place).
 *  [S1] «Qwen3.8-27B投机解码实测：从14到159 tok/s的性能断点地图»
 *       (xdnf.cn/news/337238): §2 (paged KV cache, 16 tokens per page; the
 *       verify stream reads the cache sequentially), §4 (all verify slots take
 *       pages from one physical pool), §5.3 (the causal mask of a multi-token
 *       draft).
 *  [S3] «Qwen3.8-27B 部署技术报告» (FlintyLemming): chain drafts of 4 and 8,
 *       temperature 0.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is DEVICE memory owned by the caller, except where
 *    a parameter says "host".  The library never allocates, frees or
 *    synchronises; scratch space is the caller's `workspace`, sized by the
 *    matching *_workspace_size query.  Calls are asynchronous and ordered on
 *    `stream` (a cudaStream_t passed as void*; NULL = the legacy default
 *    stream), so a whole step can be captured into one CUDA graph.
 *  - bf16 tensors (q, caches, k_new/v_new, out) and workspaces must start on a
 *    16-byte boundary (SD_ERR_INVALID_ARG otherwise).
 *  - Geometry is fixed: 24 query heads, 4 KV heads, head_dim 256, 16-token
 *    pages.  Query head h reads KV head h / 6.  bf16 tensors are raw 16-bit
 *    bf16 values (uint16 storage is fine).
 *  - A batch holds B sequences.  Sequence b owns draft nodes
 *    q_indptr[b] .. q_indptr[b+1]-1 (host array, B+1 entries); its node count
 *    N_b = q_indptr[b+1]-q_indptr[b] must be 1..64.  Node 0 of a sequence is
 *    the root: the last token already emitted, whose K/V is not cached yet.
 *    parents[] holds per-sequence local ids: parents[root] = -1 and
 *    0 <= parents[j] < j otherwise (a chain of N nodes is -1, 0, 1, .., N-2).
 *  - The KV cache of one layer is [num_pool_pages][4][16][256] bf16
 *    (page-major, then KV head, then slot, then dim).  page_table is
 *    [B][max_pages_per_seq] int32; context token p of sequence b lives in
 *    page page_table[b][p / 16], slot p % 16.  ctx_lens[b] (device int32) is
 *    the committed context length L_b >= 0.
 *  - Errors: problems visible on the host (geometry, N_b out of range, null
 *    pointers, workspace too small, batch too large) return a status at once
 *    and launch nothing.  Problems only visible on the device (a parent array
 *    out of order, a page id outside the pool, a context longer than the page
 *    table, an accept result out of range, NaN logits) OR a bit into
 *    *dev_status (nullable; the caller zeroes it and reads it when it likes);
 *    the kernel then skips the offending accesses (it never traps), and the
 *    affected outputs are unspecified.  CUDA launch errors return SD_ERR_CUDA.
 */
#ifndef SD_VERIFY_H_
#define SD_VERIFY_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SD_OK = 0,
  SD_ERR_INVALID_ARG = 1,  /* a host-checkable argument is wrong */
  SD_ERR_UNSUPPORTED = 2,  /* geometry other than 24/4/256/16, or too many nodes/sequences */
  SD_ERR_CUDA = 3,         /* a CUDA call or launch failed */
  SD_ERR_WORKSPACE = 4     /* workspace pointer null or smaller than the size query */
} sd_status;

/* Bits OR-ed into *dev_status by the kernels. */
#define SD_DEV_BAD_PARENTS   1   /* parents[root] != -1 or parents[j] outside [0, j) */
#define SD_DEV_BAD_PAGE      2   /* a page id needed for a read or write is outside [0, num_pool_pages) */
#define SD_DEV_BAD_CTX       4   /* ctx_lens[b] < 0, or ctx + nodes beyond max_pages_per_seq pages */
#define SD_DEV_BAD_ACCEPT    8   /* accept_len / path out of range at commit time */
#define SD_DEV_NAN_LOGITS   16   /* a logits row holds NaN (argmax of such a row is unspecified) */
#define SD_DEV_PATH_OVERFLOW 32  /* accept length larger than max_path */
#define SD_DEV_TIMEOUT      64   /* an internal pipeline wait expired (about 1 s); outputs unspecified */

#define SD_MAX_BATCH 256
#define SD_MAX_NODES 64
#define SD_MAX_LAYERS 64

/* Shape of one verify batch.  All fields are host values. */
typedef struct sd_shape {
  int batch;                 /* B, 1..SD_MAX_BATCH */
  const int* q_indptr_h;     /* host [B+1], q_indptr_h[0] = 0, N_b in 1..64 */
  int num_q_heads;           /* must be 24 */
  int num_kv_heads;          /* must be 4 */
  int head_dim;              /* must be 256 */
  int page_size;             /* must be 16 */
  int max_pages_per_seq;     /* columns of page_table, >= 1 */
  int num_pool_pages;        /* pages in each layer's cache pool, >= 1 */
  int num_splits;            /* split-KV chunks per (sequence, KV head); 0 = choose automatically */
  int window;                /* sliding window W >= 1: node j (position L + depth(j)) attends only to keys at
                                positions > L + depth(j) - W, its W most recent ones (own key included);
                                0 = the whole context.  Source: «如何在单张 RTX 3090 上让 Qwen3.5-27B token
                                生成速度提升 6 倍», 补充测试 (attention over the most recent 2,048 positions). */
  int ctx_stable;            /* sd_verify_attn / sd_verify_attn_fp8 only; other calls ignore it.  Nonzero: the
                                caller guarantees that the kernel issued just before this call on its stream
                                writes none of ctx_lens, page_table and the pool pages holding positions
                                [0, L_b) — true for every layer of a step after the first, whose predecessor
                                is the previous layer's attention.  The context CTAs then read those and start
                                their cache loads before they wait for that kernel to finish (programmatic
                                dependent launch); q, k_new, v_new, parents, the outputs and the workspace are
                                still touched only after the wait.  0: everything waits (always safe, e.g.
                                for the first layer after the previous step's commit). */
} sd_shape;

/* Human-readable name of a status code (static string). */
const char* sd_status_string(sd_status s);

/* Bytes of workspace sd_verify_attn needs for this shape (0 on a bad shape). */
size_t sd_verify_attn_workspace_size(const sd_shape* shape);

/*
 * sd_verify_attn — tree/causal-masked grouped-query attention of ONE layer.
 *
 * For sequence b, node j and query head h, the output is softmax attention
 * (scale 1/16 = 1/sqrt(256)) of q[j][h] over the keys of KV head h/6:
 *   all L_b context tokens of the paged cache, then the draft nodes i on j's
 *   root path (root .. j, i.e. i = j or i an ancestor of j), whose K/V come
 *   from k_new / v_new.
 * For a chain this is the bottom-right-aligned causal mask ([S1] §5.3); for
 * a tree each node follows its own parent chain ([S5] 关键突破).  The context
 * is split into chunks processed in parallel (split-KV); partial results are
 * merged with their log-sum-exp weights.
 *
 *   q          bf16 [sumN][24][256]            queries (post-RoPE)
 *   k_cache    bf16 [num_pool_pages][4][16][256] this layer's K pool (read only)
 *   v_cache    bf16 same layout                 this layer's V pool (read only)
 *   k_new      bf16 [sumN][4][256]              K of the draft nodes (not yet cached)
 *   v_new      bf16 [sumN][4][256]
 *   page_table int32 [B][max_pages_per_seq]
 *   ctx_lens   int32 [B]
 *   parents    int32 [sumN]                      per-sequence local parent ids
 *   out        bf16 [sumN][24][256]            attention output (written)
 *   lse        fp32 [sumN][24] or NULL          natural-log sum of exp(scores) (written)
 *   workspace  device scratch of >= sd_verify_attn_workspace_size(shape) bytes
 *   dev_status int32 device word or NULL
 */
sd_status sd_verify_attn(const sd_shape* shape, const void* q, const void* k_cache,
                         const void* v_cache, const void* k_new, const void* v_new,
                         const int* page_table, const int* ctx_lens, const int* parents,
                         void* out, float* lse, void* workspace, size_t ws_bytes,
                         int* dev_status, void* stream);

/*
 * sd_verify_attn_fp8 — sd_verify_attn over a quantised (e4m3) KV cache.
 *
 * The quantised KV cache of «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度
 * 提升 6 倍» (24 GB 显存上的 128K 上下文: the cache is stored quantised, written
 * once through a quantiser and read quantised by the verify attention), with
 * FP8 e4m3 codes in place of the page's Q4_0 blocks: one byte per value, half
 * the bytes of bf16.  Code c of the K (V) pool stands for decode(c) * k_scale
 * (v_scale), decode being the e4m3 value (1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits; subnormals m * 2^-9; 0x7F / 0xFF are NaN; largest 448).
 * Everything else is sd_verify_attn: the same masks, split plan, workspace
 * size (sd_verify_attn_workspace_size) and outputs.  The draft nodes' own
 * K/V (k_new, v_new) are not cached yet and stay bf16.
 *
 *   k_cache, v_cache  uint8 e4m3 codes [num_pool_pages][4][16][256] (read only), 16-byte aligned
 *   k_scale, v_scale  host fp32: positive, finite, with a finite reciprocal (else SD_ERR_INVALID_ARG)
 *   other arguments   as for sd_verify_attn
 * Queries and the draft block are taken to f16 inside the kernel: values
 * beyond the f16 range (|x| > 65504) give an unspecified output.
 */
sd_status sd_verify_attn_fp8(const sd_shape* shape, const void* q, const void* k_cache,
                             const void* v_cache, float k_scale, float v_scale, const void* k_new,
                             const void* v_new, const int* page_table, const int* ctx_lens,
                             const int* parents, void* out, float* lse, void* workspace,
                             size_t ws_bytes, int* dev_status, void* stream);

/*
 * sd_verify_attn_noalloc — sd_verify_attn for callers that cannot allocate
 * device memory (the pages have no counterpart: this is a library entry point,
 * not part of the method).
 *
 * Some callers cannot make or hold a device allocation where they call us:
 * a plugin running inside another runtime whose device memory belongs to that
 * runtime's pool, or a decode loop on a path where allocating (and the
 * synchronisation it may cause) is not allowed.  This entry point takes the
 * same inputs and outputs as sd_verify_attn but no workspace: the split
 * partials go to a scratch array of SD_NOALLOC_SCRATCH_BYTES that the library
 * keeps in device memory.  It calls no allocating routine.
 *
 *  - The array is device memory of the library's module, which the CUDA
 *    runtime loads lazily: the first call on a device loads it and reserves
 *    the array then (and can fail with SD_ERR_CUDA when the device has no
 *    room); the device keeps it until the process exits.  Later calls
 *    allocate nothing.  Make the first call early and before any stream
 *    capture.
 *  - The first call in a CUDA context (normally the device's primary context,
 *    i.e. once per device) looks up the array's address with that context
 *    current and keeps it under the context's unique id; another context, or
 *    the new context after a device reset, does its own lookup.
 *  - Every call in a context shares the one array and it keeps the last call's
 *    contents (nothing in it needs to start at zero).  Calls that may overlap
 *    on the GPU — on unordered streams or from several threads — race on it.
 *  - A shape that sd_verify_attn would reject returns the same status; a shape
 *    whose scratch need (sd_verify_attn_workspace_size) exceeds
 *    SD_NOALLOC_SCRATCH_BYTES is rejected with SD_ERR_WORKSPACE before any
 *    launch.  Other arguments and errors are as for sd_verify_attn.
 */
#define SD_NOALLOC_SCRATCH_BYTES (16u << 20)
sd_status sd_verify_attn_noalloc(const sd_shape* shape, const void* q, const void* k_cache,
                                 const void* v_cache, const void* k_new, const void* v_new,
                                 const int* page_table, const int* ctx_lens, const int* parents,
                                 void* out, float* lse, int* dev_status, void* stream);

/* Bytes of workspace sd_accept needs (0 on bad arguments). */
size_t sd_accept_workspace_size(int batch, const int* q_indptr_h, int vocab);

/*
 * sd_accept — greedy verification of every sequence's draft block.
 *
 * First t[r] = argmax_v logits[r][v] for every node row r (the smallest index
 * on ties; -0.0 == +0.0).  logits hold one row per node, root included, i.e.
 * budget + 1 rows per sequence ([S5] 关键突破).  Then, per sequence, node j
 * is accepted when its parent is accepted (the root always is) and
 * draft_tokens[j] == t[parent[j]] ([S5] 架构设计: greedy verify).  The chosen
 * path is the longest accepted root path (ties: the lexicographically
 * smallest sequence of node ids); its length in nodes, root included, is the
 * accept length A (1 <= A <= depth + 1; [S5] 从自回归到 DDTree).  The emitted
 * tokens are the accepted drafts followed by the bonus token t[last node].
 *
 *   vocab          V >= 1
 *   logits         fp32 [sumN][V]
 *   parents        int32 [sumN]
 *   draft_tokens   int32 [sumN]  (the root's entry is ignored)
 *   accept_len     int32 [B]                 A_b (written)
 *   path           int32 [B][max_path]       node ids of the path, -1 after A_b (written)
 *   out_tokens     int32 [B][max_path]       emitted tokens, -1 after A_b (written)
 *   target_tokens  int32 [sumN] or NULL      t[] (written)
 *   max_path       >= 1; an A_b above it sets SD_DEV_PATH_OVERFLOW and is clipped
 */
sd_status sd_accept(int batch, const int* q_indptr_h, int vocab, const float* logits,
                    const int* parents, const int* draft_tokens, int* accept_len, int* path,
                    int* out_tokens, int* target_tokens, int max_path, void* workspace,
                    size_t ws_bytes, int* dev_status, void* stream);

/* Bytes of workspace sd_sample_accept needs (0 on bad arguments). */
size_t sd_sample_accept_workspace_size(int batch, const int* q_indptr_h, int vocab);

/*
 * sd_sample_accept — sampling-based verification (temperature T > 0) of every
 * sequence's draft block, in place of sd_accept's greedy rule.
 *
 * The pages verify greedily and name sampling as future work ([S5] 补充测试 and
 * 关键突破; [S3] runs at temperature 0) without an acceptance rule; this is
 * standard speculative sampling with the multi-candidate rule for trees:
 *   p_u = softmax(logits_u / T); the children of node u were drawn from the
 *   draft distribution q_u = draft_probs[u]; they are tried in increasing node
 *   order, child c with token x being accepted when r_accept[c] * q_u(x) <
 *   p(x) (so with probability min(1, p(x) / q_u(x))); after a rejection p
 *   becomes max(0, p - q_u), renormalised; the walk descends into an accepted
 *   child; when every child of the current node is rejected, or it is a leaf,
 *   the bonus token is the smallest v with sum_{w <= v} p(w) > r_sample[u] *
 *   sum(p).  The emitted sequence is distributed as sampling from the target.
 * Outputs follow sd_accept (accept length with the root counted, the path's
 * node ids, the accepted drafts followed by the bonus token, -1 after A_b).
 * Decisions are taken in fp32; a draft token outside [0, vocab) is never
 * accepted.
 *
 *   vocab          V, 1..2048 * 1024
 *   temperature    host float > 0 (finite)
 *   logits         fp32 [sumN][V]
 *   draft_probs    fp32 [sumN][V]   q at each node (rows of leaves are not read)
 *   parents, draft_tokens   int32 [sumN]
 *   r_accept, r_sample      fp32 [sumN], uniforms in [0, 1) (caller-drawn)
 *   accept_len, path, out_tokens, max_path   as for sd_accept
 */
sd_status sd_sample_accept(int batch, const int* q_indptr_h, int vocab, float temperature, const float* logits,
                           const float* draft_probs, const int* parents, const int* draft_tokens,
                           const float* r_accept, const float* r_sample, int* accept_len, int* path,
                           int* out_tokens, int max_path, void* workspace, size_t ws_bytes, int* dev_status,
                           void* stream);

/*
 * sd_kv_commit — append the accepted nodes' K/V to the cache, all layers in
 * one launch.  For every layer, sequence b and i < accept_len[b], node
 * path[b][i] is copied (bytes unchanged, all 4 KV heads, K and V) to context
 * position ctx_lens[b] + i.  Rejected nodes are never written ([S5] 关键突破:
 * accepted state is written in place instead of being copied around).
 * new_ctx_lens[b] = ctx_lens[b] + accept_len[b].
 *
 *   num_layers                 1..SD_MAX_LAYERS
 *   k_cache_layers / v_cache_layers   HOST arrays of num_layers device pointers (caches, written)
 *   k_new_layers / v_new_layers       HOST arrays of num_layers device pointers, bf16 [sumN][4][256]
 *   page_table, ctx_lens       as for sd_verify_attn; the pages for positions
 *                              ctx .. ctx + A - 1 must already be in the table
 *   new_ctx_lens               int32 [B] or NULL; must not alias ctx_lens
 *   accept_len, path           as written by sd_accept (path row stride = max_path)
 */
sd_status sd_kv_commit(const sd_shape* shape, int num_layers, void* const* k_cache_layers,
                       void* const* v_cache_layers, const void* const* k_new_layers,
                       const void* const* v_new_layers, const int* page_table,
                       const int* ctx_lens, int* new_ctx_lens, const int* accept_len,
                       const int* path, int max_path, int* dev_status, void* stream);

/*
 * sd_kv_commit_fp8 — sd_kv_commit into e4m3 caches: quantise on commit.
 *
 * The accepted rows are quantised once, on the way into the cache (the
 * write-time quantiser of «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升
 * 6 倍», 24 GB 显存上的 128K 上下文): for layer l each bf16 value x of K (V)
 * becomes code e4m3(x * r), r = 1 / k_scales[l] (v_scales[l]) rounded to fp32,
 * the product rounded to fp32, then to the nearest e4m3 value with ties to
 * the even code; finite values beyond +-448 (and infinities) saturate to
 * +-448; NaN gives a NaN code.  Everything else is sd_kv_commit.
 *
 *   k_cache_layers / v_cache_layers   HOST arrays of device pointers to uint8 caches
 *                                     [num_pool_pages][4][16][256] (written)
 *   k_scales / v_scales               HOST fp32 arrays [num_layers]; each positive, finite,
 *                                     with a finite reciprocal (else SD_ERR_INVALID_ARG)
 */
sd_status sd_kv_commit_fp8(const sd_shape* shape, int num_layers, void* const* k_cache_layers,
                           void* const* v_cache_layers, const float* k_scales, const float* v_scales,
                           const void* const* k_new_layers, const void* const* v_new_layers,
                           const int* page_table, const int* ctx_lens, int* new_ctx_lens,
                           const int* accept_len, const int* path, int max_path, int* dev_status,
                           void* stream);

/*
 * sd_ddtree_build — the draft tree the verify step checks, built from the
 * draft model's logits for a block of `positions` positions
 * («如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍», 从自回归到 DDTree:
 * a draft block of 16 positions becomes a token tree of `budget` nodes;
 * 关键突破: per-position top-K (32 -> 8), chain pre-seed).
 *
 * Per position d, the candidates are the topk tokens with the largest draft
 * logits (ties: the smaller token id first), scored by log-probability
 * logit - log(sum(exp(logits of the position))).  A node at depth d >= 1 holds
 * a candidate of position d - 1 and scores the sum of the log-probabilities on
 * its root path.  The rank-0 chain is inserted first, down to depth
 * min(positions, budget); then, until the tree has 1 + budget nodes, the best
 * of the candidates "first child (rank 0, one position deeper) of an inserted
 * node" and "next sibling (rank + 1, same parent) of an inserted node" is
 * inserted (ties: the candidate created first).  Node 0 is the root with
 * token root_tokens[b]; nodes are numbered in insertion order, so
 * parents[j] < j and the outputs feed sd_verify_attn / sd_accept directly
 * (q_indptr = b * (1 + budget)).
 *
 *   batch                      1..SD_MAX_BATCH
 *   positions                  1..SD_MAX_NODES
 *   vocab                      >= topk
 *   topk                       1..8
 *   budget                     1..SD_MAX_NODES - 1 (non-root nodes)
 *   draft_logits               fp32 [batch][positions][vocab]
 *   root_tokens                int32 [batch]
 *   parents, tokens            int32 [batch][1 + budget], written; entries past the available
 *                              candidates are -1
 *   scores                     fp32 [batch][1 + budget] or NULL (path log-probabilities)
 *   workspace                  >= sd_ddtree_workspace_size bytes, 16-byte aligned
 * Errors: bad sizes or null pointers -> SD_ERR_INVALID_ARG / SD_ERR_UNSUPPORTED
 * before any launch; NaN logits -> SD_DEV_NAN_LOGITS in *dev_status (the tree
 * is then unspecified).
 */
size_t sd_ddtree_workspace_size(int batch, int positions, int vocab, int topk);
sd_status sd_ddtree_build(int batch, int positions, int vocab, int topk, int budget,
                          const float* draft_logits, const int* root_tokens, int* parents, int* tokens,
                          float* scores, void* workspace, size_t ws_bytes, int* dev_status,
                          void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SD_VERIFY_H_ */
