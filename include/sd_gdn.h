/*
 * sd_gdn.h — C ABI of the tree-aware Gated DeltaNet verify (sm_103a).
 *
 * The target model of «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍»
 * is hybrid: 为什么我们要做这个测试 states that 48 of its 64 layers are Gated
 * DeltaNet layers with a recurrent (SSM) state cache besides the KV cache, and
 * 关键突破 lists the tree-aware kernels that verify a draft tree through them:
 * a delta-net kernel that writes the accepted state in place (persist), and a
 * short convolution in which every node gathers its window along its own
 * parent chain.  The page gives no formulas; this library computes the
 * published Gated DeltaNet rule along each node's parent chain:
 *
 *   per value head h (key head h / (H_v / H_k)), state S (128 x 128, rows =
 *   value dims), node j with parent p (the cached state for the root):
 *     S_j = exp(g_j) S_p + beta_j (v_j - exp(g_j) S_p k_j) k_j^T,   o_j = S_j q_j,
 *   k and q L2-normalised per head (a zero vector stays zero), q scaled by
 *   1/sqrt(128);
 *   convolution: y_j = silu(sum_i w[i] x_{t-3+i}) per channel, where x_{t-1},
 *   x_{t-2}, x_{t-3} are the inputs of j's parent, grandparent, ... and, past
 *   the root, the cached convolution state (the last three committed inputs);
 *   persist: after the step accepts path p_0 .. p_{A-1} (sd_accept), the
 *   state becomes S_{p_{A-1}} and the convolution state the last three inputs
 *   of (old state, x_{p_0}, .., x_{p_{A-1}}).
 *
 * Conventions are those of sd_verify.h (device pointers owned by the caller,
 * no allocation, no synchronisation, asynchronous on `stream`, host-checkable
 * errors returned before any launch, device-only problems OR-ed into
 * *dev_status).  Batches are described by the host q_indptr of sd_verify.h:
 * sequence b owns nodes q_indptr[b] .. q_indptr[b+1]-1 (1..64 nodes), and
 * parents[] holds local ids (parents[root] = -1, 0 <= parents[j] < j).
 * bf16 tensors, fp32 tensors and the tree cache must start on 16 bytes.
 */
#ifndef SD_GDN_H_
#define SD_GDN_H_

#include <stddef.h>

#include "sd_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct sd_gdn_shape {
  int batch;                 /* B, 1..SD_MAX_BATCH */
  const int* q_indptr_h;     /* host [B+1], q_indptr_h[0] = 0, N_b in 1..64 */
  int num_k_heads;           /* H_k >= 1 */
  int num_v_heads;           /* H_v, a multiple of H_k, at most 256 */
  int head_dim;              /* must be 128 (d_k = d_v) */
} sd_gdn_shape;

/* Bytes of one layer's tree cache (written by sd_gdn_tree, read by
 * sd_gdn_commit): per node, the value-head vectors u, the log decay of its
 * root path, and the normalised keys.  0 on a bad shape. */
size_t sd_gdn_tree_cache_size(const sd_gdn_shape* shape);

/*
 * sd_gdn_conv_tree — the short convolution of one layer over the draft tree.
 *
 *   channels     C >= 1 (the convolved q, k and v channels of the layer)
 *   x            bf16 [sumN][C]   inputs of the draft nodes
 *   weight       fp32 [C][4]      taps; weight[c][3] multiplies the node's own input
 *   conv_state   bf16 [B][C][3]   the last three committed inputs, oldest first (read only)
 *   parents      int32 [sumN]
 *   y            bf16 [sumN][C]   silu of the convolution (written)
 */
sd_status sd_gdn_conv_tree(int batch, const int* q_indptr_h, int channels, const void* x, const float* weight,
                           const void* conv_state, const int* parents, void* y, int* dev_status, void* stream);

/*
 * sd_gdn_tree — the gated delta rule of one layer over the draft tree.
 *
 *   q, k         bf16 [sumN][H_k][128]
 *   v            bf16 [sumN][H_v][128]
 *   g            fp32 [sumN][H_v]   log decay (g <= 0; alpha = exp(g))
 *   beta         fp32 [sumN][H_v]   write strength in [0, 1]
 *   state        fp32 [B][H_v][128][128]   cached state before the step (read only)
 *   parents      int32 [sumN]
 *   out          bf16 [sumN][H_v][128]     o_j (written)
 *   tree_cache   >= sd_gdn_tree_cache_size bytes, this layer's (written; keep it for sd_gdn_commit)
 */
sd_status sd_gdn_tree(const sd_gdn_shape* shape, const void* q, const void* k, const void* v, const float* g,
                      const float* beta, const float* state, const int* parents, void* out, void* tree_cache,
                      size_t cache_bytes, int* dev_status, void* stream);

/*
 * sd_gdn_commit — persist-on-accept for every Gated DeltaNet layer in one
 * launch: state_layers[l] becomes the state of the last accepted node (rebuilt
 * from that layer's tree cache), and, when channels > 0, conv_state_layers[l]
 * the last three inputs of (old state, accepted nodes' x_layers[l] rows).
 *
 *   num_layers                  1..SD_MAX_LAYERS
 *   state_layers                HOST array of device pointers, fp32 [B][H_v][128][128] (updated in place)
 *   tree_cache_layers           HOST array of device pointers (as written by sd_gdn_tree)
 *   channels                    C of the convolution, or 0 to leave the convolution states alone
 *   conv_state_layers, x_layers HOST arrays of device pointers (bf16 [B][C][3] updated; bf16 [sumN][C]),
 *                               NULL when channels = 0
 *   accept_len, path, max_path  as written by sd_accept
 * An accept result out of range sets SD_DEV_BAD_ACCEPT and leaves that sequence's states untouched.
 */
sd_status sd_gdn_commit(const sd_gdn_shape* shape, int num_layers, float* const* state_layers,
                        const void* const* tree_cache_layers, int channels, void* const* conv_state_layers,
                        const void* const* x_layers, const int* accept_len, const int* path, int max_path,
                        int* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SD_GDN_H_ */
