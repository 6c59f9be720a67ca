// gt_tree_attn_noalloc: the tree attention of gt_tree_attn with its scratch in a fixed
// array that this library owns, so that the caller allocates nothing.
//
// The scratch is one file-scope device array of GT_ATTN_NOALLOC_SCRATCH_BYTES. Each device
// gets its own copy of it when the library's module is loaded there. Under lazy module
// loading (the CUDA default) that happens on the first use of any kernel of this library on
// the device; under CUDA_MODULE_LOADING=EAGER it happens when a context is created. Either
// way every device that loads the module holds the 32 MiB until the process exits, whether
// or not this entry point is ever called.
//
// Its device address is looked up with that device current, on the first call made in each
// context, and cached with the context's id: after cudaDeviceReset the next call sees a new
// context and looks the address up again instead of passing a dead one.
#include <atomic>
#include <mutex>
#include <stdio.h>

#include "gt_internal.cuh"

namespace gt {

static __device__ __align__(256) unsigned char g_attn_scratch[GT_ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int NOALLOC_MAX_DEVICES = 64;
struct ScratchRecord {
  uint64_t ctx = 0;  // current_context_id() of the context the address belongs to
  uintptr_t addr = 0;
};
static ScratchRecord g_scratch[NOALLOC_MAX_DEVICES];
static std::mutex g_scratch_mu;

// Device address of this context's copy of the scratch array (0 on failure, with the
// detail recorded for gt_last_error).
static uintptr_t scratch_address() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    launch_status(e, "gt_tree_attn_noalloc: cudaGetDevice");
    return 0;
  }
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) {
    note_message("gt_tree_attn_noalloc: device ordinal above 63");
    return 0;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const uint64_t ctx = current_context_id();
  if (ctx != 0 && g_scratch[dev].ctx == ctx) return g_scratch[dev].addr;
  void *ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_attn_scratch);
  if (e != cudaSuccess) {
    launch_status(e, "gt_tree_attn_noalloc: cudaGetSymbolAddress(scratch)");
    return 0;
  }
  if (!ptr) {
    note_message("gt_tree_attn_noalloc: cudaGetSymbolAddress(scratch) gave a null address");
    return 0;
  }
  // the look-up creates the context when there was none: key the record on it
  g_scratch[dev].ctx = current_context_id();
  g_scratch[dev].addr = reinterpret_cast<uintptr_t>(ptr);
  return g_scratch[dev].addr;
}

}  // namespace gt

using namespace gt;

GT_API int gt_tree_attn_noalloc(const void *Q, const void *K, const void *V,
                                const uint64_t *mask, const int32_t *prefix_len,
                                const int32_t *n_nodes, int B, int N, int Hq, int Hkv, int d,
                                int Lcap, int dtype, float scale, void *O, int32_t *err,
                                gt_stream_t stream) {
  GT_TRACE("gt_tree_attn_noalloc");
  const size_t need = gt_tree_attn_workspace(B, N, Hq, Hkv, d, Lcap);
  if (need == 0) {  // an invalid shape: gt_tree_attn reports which error, launching nothing
    return gt_tree_attn(Q, K, V, mask, prefix_len, n_nodes, B, N, Hq, Hkv, d, Lcap, dtype,
                        scale, O, nullptr, 0, err, stream);
  }
  if (need > (size_t)GT_ATTN_NOALLOC_SCRATCH_BYTES) {
    char msg[160];
    snprintf(msg, sizeof(msg),
             "gt_tree_attn_noalloc: this shape needs %zu bytes of scratch, the static array "
             "holds %zu",
             need, (size_t)GT_ATTN_NOALLOC_SCRATCH_BYTES);
    note_message(msg);
    return GT_ERR_SHAPE;
  }
  const uintptr_t a = scratch_address();
  if (!a) return GT_ERR_CUDA;
  return gt_tree_attn(Q, K, V, mask, prefix_len, n_nodes, B, N, Hq, Hkv, d, Lcap, dtype, scale,
                      O, reinterpret_cast<void *>(a), (size_t)GT_ATTN_NOALLOC_SCRATCH_BYTES, err,
                      stream);
}
