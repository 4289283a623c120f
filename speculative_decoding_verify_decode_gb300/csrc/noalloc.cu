// sd_verify_attn_noalloc: verify attention for callers that cannot allocate
// device memory.  It runs the same kernels as sd_verify_attn, with the split
// partials kept in a fixed scratch array that lives in this file instead of a
// caller-provided workspace.
//
// Who needs it: code that must not allocate device memory at the point where
// it calls us -- for example a plugin inside another runtime whose device
// memory is owned by that runtime's pool, or a decode loop on a real-time
// path where an allocation (and the synchronisation it can cause) is not
// allowed.  Such callers still own every input and output buffer; only the
// scratch space moves into the library.
//
// Costs and rules:
//  - every GPU that loads the library holds kNoallocScratchBytes of device
//    memory for this array until the process exits;
//  - the first call on each device looks up the array's device address
//    (cudaGetSymbolAddress, with that device current) and caches it; make that
//    first call before any stream capture;
//  - all calls share the one array, so calls that can overlap on the GPU
//    (different streams without ordering, or several threads) race on it;
//  - the array keeps the previous call's contents; nothing in it has to start
//    at zero, because each split writes its partial before the merge reads it;
//  - a shape whose scratch need exceeds the array is rejected with
//    SD_ERR_WORKSPACE before anything is launched.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kNoallocScratchBytes = SD_NOALLOC_SCRATCH_BYTES;
static_assert(kNoallocScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (looked up once).
sd_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return SD_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SD_OK;
}

}  // namespace

extern "C" sd_status sd_verify_attn_noalloc(const sd_shape* shape, const void* q, const void* k_cache,
                                            const void* v_cache, const void* k_new, const void* v_new,
                                            const int* page_table, const int* ctx_lens, const int* parents,
                                            void* out, float* lse, int* dev_status, void* stream) {
  const size_t need = sd_verify_attn_workspace_size(shape);
  if (shape == nullptr) return SD_ERR_INVALID_ARG;
  if (need > kNoallocScratchBytes) return SD_ERR_WORKSPACE;
  void* scratch = nullptr;
  const sd_status st = scratch_for_current_device(&scratch);
  if (st != SD_OK) return st;
  return sd_verify_attn(shape, q, k_cache, v_cache, k_new, v_new, page_table, ctx_lens, parents, out, lse, scratch,
                        kNoallocScratchBytes, dev_status, stream);
}
