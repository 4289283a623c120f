// Shared constants, parameter blocks and small device helpers of the verify
// kernels.  Internal to the library (the public interface is sd_verify.h).
#pragma once

#include <utility>

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/sd_verify.h"

namespace sdv {

constexpr int kHq = 24;          // query heads
constexpr int kHkv = 4;          // KV heads
constexpr int kGroup = kHq / kHkv;
constexpr int kDim = 256;        // head_dim
constexpr int kPage = 16;        // tokens per KV page
constexpr int kTileTokens = 128; // context tokens per attention tile (the MMA's M)
constexpr int kMaxNodes = SD_MAX_NODES;
constexpr int kMaxBatch = SD_MAX_BATCH;
constexpr int kMaxLayers = SD_MAX_LAYERS;

// log2(e) / sqrt(256): scores are kept in base 2 so exp becomes ex2.
constexpr float kScaleLog2 = 1.4426950408889634f / 16.0f;
constexpr float kLn2 = 0.6931471805599453f;

// Per-call batch description passed by value to every kernel.
struct BatchDesc {
  int batch;
  int total_nodes;
  int max_nodes;
  int q_indptr[kMaxBatch + 1];
};

// Attention launch parameters (one layer).
struct AttnParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_cache;
  const __nv_bfloat16* v_cache;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const int* page_table;
  const int* ctx_lens;
  const int* parents;
  __nv_bfloat16* out;
  float* lse;            // nullable
  __nv_bfloat16* o_part; // [num_splits][total_nodes][24][256] normalised partial outputs
  float* lse_part;       // [num_splits][total_nodes][24]  (base-2 log-sum-exp)
  int* dev_status;       // nullable
  int max_pages;
  int num_pool_pages;
  int chunk;             // context tokens per split (multiple of the kernel's tile)
  int num_splits;
  int window;            // sliding window (0: the whole context)
  int ctx_stable;        // context CTAs may read the table and cache pages before the wait on the previous kernel
  // e4m3 caches (the quantised path): code c of K / V stands for decode(c) * k_scale / v_scale
  const uint8_t* k_cache8;
  const uint8_t* v_cache8;
  float k_scale;
  float v_scale;
};

// Programmatic dependent launch of a kernel whose first statement is
// pdl_wait(): it may be scheduled while the previous kernel in the stream
// runs, and reads or writes nothing before that kernel has finished.
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
// Wait for the previous kernel in the stream (and see its writes), then let
// the next one be scheduled.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void report(int* status, int bits) {
  if (status != nullptr) atomicOr(status, bits);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// First context position a sequence's splits cover: 0 for full attention;
// with a window W, the root's oldest visible position L - W + 1, rounded down
// to a multiple of `tile` (the splits start on tile boundaries).
__host__ __device__ __forceinline__ int window_base(int L, int window, int tile) {
  if (window <= 0) return 0;
  const int first = L - window + 1;
  return first <= 0 ? 0 : first / tile * tile;
}

// Number of active splits of a sequence with context length L: split 0
// attends to the draft block alone and splits 1.. to consecutive chunks of
// `chunk` context tokens from window_base on, so a sequence without
// (visible) context has one split.
__host__ __device__ __forceinline__ int active_splits(int L, int window, int tile, int chunk) {
  const int span = L - window_base(L, window, tile);
  return 1 + (span > 0 ? (span + chunk - 1) / chunk : 0);
}

}  // namespace sdv
