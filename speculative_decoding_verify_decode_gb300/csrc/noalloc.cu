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
//  - the array takes kNoallocScratchBytes of device memory on every device
//    where it is used, until the process exits.  The CUDA runtime loads this
//    file's module lazily: the first call on a device (with that device
//    current) loads it and reserves the array then, so that first call can
//    fail with SD_ERR_CUDA when the device is out of memory.  Make it early,
//    and before any stream capture; later calls allocate nothing;
//  - set-up: the first call in a CUDA context (normally the device's primary
//    context, so once per device) looks up the array's device address with
//    cudaGetSymbolAddress, that context current, and keeps it under the
//    context's unique id.  A context created after a device reset, or a
//    non-primary context, has another id and gets its own lookup, never a
//    stale address;
//  - all calls in one context share the one array, so calls that can overlap
//    on the GPU (different streams without ordering, or several threads) race
//    on it;
//  - the array keeps the previous call's contents; nothing in it has to start
//    at zero, because each split writes its partial before the merge reads it;
//  - a shape whose scratch need exceeds the array is rejected with
//    SD_ERR_WORKSPACE before anything is launched; an invalid shape returns
//    the status sd_verify_attn gives it.
#include <cuda.h>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kNoallocScratchBytes = SD_NOALLOC_SCRATCH_BYTES;
static_assert(kNoallocScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// The array's address per context, keyed by the driver's unique context id.
constexpr int kMaxContexts = 64;
struct ScratchEntry {
  unsigned long long ctx_id;
  void* ptr;
};
ScratchEntry g_entries[kMaxContexts];
int g_num_entries = 0;
std::mutex g_scratch_mutex;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}

// Unique id of the calling thread's current context (the runtime makes the
// device's primary context current when there is none yet).
sd_status current_context_id(unsigned long long* id) {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (get_current == nullptr || get_id == nullptr) return SD_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return SD_ERR_CUDA;
  if (ctx == nullptr) {
    // no context yet: setting the current device again initialises its primary context and makes it current
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) {
      cudaGetLastError();
      return SD_ERR_CUDA;
    }
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return SD_ERR_CUDA;
  }
  return get_id(ctx, id) == CUDA_SUCCESS ? SD_OK : SD_ERR_CUDA;
}

// The scratch array's device address in the current context (set up once per context).
sd_status scratch_for_current_context(void** out) {
  unsigned long long id = 0;
  const sd_status st = current_context_id(&id);
  if (st != SD_OK) return st;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  for (int i = 0; i < g_num_entries; ++i)
    if (g_entries[i].ctx_id == id) {
      *out = g_entries[i].ptr;
      return SD_OK;
    }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return SD_ERR_CUDA;
  }
  if (g_num_entries < kMaxContexts) g_entries[g_num_entries++] = ScratchEntry{id, p};
  *out = p;
  return SD_OK;
}

}  // namespace

extern "C" sd_status sd_verify_attn_noalloc(const sd_shape* shape, const void* q, const void* k_cache,
                                            const void* v_cache, const void* k_new, const void* v_new,
                                            const int* page_table, const int* ctx_lens, const int* parents,
                                            void* out, float* lse, int* dev_status, void* stream) {
  const sd_status shape_ok = sdv::verify_shape_status(shape);
  if (shape_ok != SD_OK) return shape_ok;
  if (sd_verify_attn_workspace_size(shape) > kNoallocScratchBytes) return SD_ERR_WORKSPACE;
  void* scratch = nullptr;
  const sd_status st = scratch_for_current_context(&scratch);
  if (st != SD_OK) return st;
  return sd_verify_attn(shape, q, k_cache, v_cache, k_new, v_new, page_table, ctx_lens, parents, out, lse, scratch,
                        kNoallocScratchBytes, dev_status, stream);
}
