// Internal helpers shared by the sm_103a kernels of libgt.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include <nvtx3/nvToolsExt.h>

#include "gt.h"

#define GT_API extern "C" __attribute__((visibility("default")))

// Checked builds (compiled with -DGT_CHECK=1 into libgt_check.so) add device-side checks of
// what the method assumes of its inputs but the kernels do not need for memory safety. A
// failed check writes its code into *err, as any data error does, and the kernel carries
// on; nothing traps.
#ifndef GT_CHECK
#define GT_CHECK 0
#endif

namespace gt {

// A named NVTX range over one C-ABI call on the calling host thread, so that profilers
// attribute the kernels the call launches to it (ncu --nvtx --nvtx-include "gt_tree_attn/").
// Without a tool attached a push or pop is a call through an unset hook.
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};
#define GT_TRACE(name) ::gt::NvtxRange gt_trace_range_(name)

// First device-side error wins; later ones are dropped.
__device__ __forceinline__ void set_err(int32_t *err, int code) {
  if (err != nullptr) atomicCAS(reinterpret_cast<int *>(err), 0, code);
}

// A check of checked builds: reports `code` when cond is false; compiled out otherwise.
#define GT_CHECKED(cond, err, code)                      \
  do {                                                   \
    if (GT_CHECK && !(cond)) ::gt::set_err((err), (code)); \
  } while (0)

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Programmatic dependent launch. Every libgt kernel is launched with programmatic stream
// serialisation: it lets the next kernel of the stream start launching at once, then waits
// until all earlier work of the stream has completed and its memory is visible. Called
// before a kernel's first global-memory access, it keeps stream order for every read and
// write while the launch latency of consecutive kernels overlaps.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Records a host-side failure detail for gt_last_error() (thread-local).
void note_error(const char *what, cudaError_t e);
// Records a complete host-side message for gt_last_error() (thread-local).
void note_message(const char *msg);

static inline int launch_status(cudaError_t e, const char *what = "kernel launch") {
  if (e != cudaSuccess) {
    note_error(what, e);
    (void)cudaGetLastError();  // clear a non-sticky launch error
    return GT_ERR_CUDA;
  }
  return GT_OK;
}

// Identity of the calling thread's current CUDA context (cuCtxGetId: unique over the
// process's lifetime, so the context that replaces one destroyed by cudaDeviceReset gets a
// new value), or 0 when there is none yet or it cannot be read. Per-device caches of state
// that lives in a context (function attributes, symbol addresses) are keyed on it.
uint64_t current_context_id();

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the current device.
// The runtime keeps the attribute per context, so each call site remembers, per device, the
// context it set the limit in and the largest limit set there (a static SmemAttr: one word
// per device, context id in the high 40 bits, bytes in the low 24); repeated calls in the
// same context then cost no attribute call.
struct SmemAttr {
  std::atomic<uint64_t> state[64];  // zero-initialised when declared static
};
template <typename Kernel>
static inline int ensure_smem(Kernel kernel, int bytes, SmemAttr &a, const char *what) {
  int dev = 0;
  const cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess) return launch_status(ge, "cudaGetDevice");
  const bool cached = dev >= 0 && dev < 64;
  const uint64_t ctx = current_context_id();
  const bool keyed = ctx != 0 && ctx < (1ull << 40);
  if (cached && keyed) {
    const uint64_t st = a.state[dev].load(std::memory_order_relaxed);
    if ((st >> 24) == ctx && (int)(st & 0xFFFFFFu) >= bytes) return GT_OK;
  }
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return launch_status(e, what);
  // the attribute call created the context if there was none: key the record on it
  const uint64_t ctx_now = current_context_id();
  if (cached && ctx_now != 0 && ctx_now < (1ull << 40) && bytes < (1 << 24)) {
    const uint64_t want = (ctx_now << 24) | (uint64_t)bytes;
    uint64_t cur = a.state[dev].load(std::memory_order_relaxed);
    // keep the larger limit of the same context; a record of another context is replaced
    while (!((cur >> 24) == ctx_now && (cur & 0xFFFFFFu) >= (uint64_t)bytes) &&
           !a.state[dev].compare_exchange_weak(cur, want)) {
    }
  }
  return GT_OK;
}

// Barrier over the first nthreads threads of the block (named barrier 1; nthreads a
// multiple of 32), or over the whole block when nthreads is 0.
__device__ __forceinline__ void sync_threads_n(int nthreads) {
  if (nthreads == 0)
    __syncthreads();
  else
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Exclusive prefix count of `flag` over the threads of a block (flags by thread index), or
// over its first nthreads threads (see sync_threads_n). `warp_tot` is shared scratch of 32
// ints. Returns the prefix; *total receives the sum.
__device__ __forceinline__ int block_excl_count(bool flag, int *warp_tot, int *total,
                                                int nthreads = 0) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = ((nthreads ? nthreads : (int)blockDim.x) + 31) >> 5;
  unsigned bal = __ballot_sync(0xffffffffu, flag);
  int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) warp_tot[warp] = __popc(bal);
  sync_threads_n(nthreads);
  int off = 0, tot = 0;
  for (int w = 0; w < nwarps; ++w) {
    int c = warp_tot[w];
    off += (w < warp) ? c : 0;
    tot += c;
  }
  sync_threads_n(nthreads);
  *total = tot;
  return off + in_warp;
}

// Order-preserving 32-bit key of a float for "larger is better" comparisons:
// +0.0 and -0.0 map to the same key, every NaN maps to 1 (below -inf), 0 is unused
// by any float and marks an empty slot.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7fffffffu) > 0x7f800000u) return 1u;
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

}  // namespace gt
