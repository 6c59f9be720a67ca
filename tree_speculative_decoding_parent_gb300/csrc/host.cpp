// Host-side helpers of libgt: stage budget, default retrieval template, status strings,
// and an external event record for timing inside captured CUDA graphs.
//
// Source: "浙江大学、阿里巴巴联手破解AI推理瓶颈" §二 (prune stages 0/1/5 keep 8/24/40 draft nodes
// and refill 52/36/20 of 60 slots from the successor table; the template is asymmetric:
// higher-ranked successors get more children and go deeper).
#include <cuda.h>
#include <cuda_runtime.h>

#include <stdio.h>

#include <atomic>

#include <queue>
#include <map>
#include <tuple>
#include <vector>

#include "gt.h"
#include "gt_internal.cuh"


GT_API int gt_stage_budget(int stage, int slots, int32_t *draft, int32_t *retrieved) {
  if (!draft || !retrieved || slots < 1) return GT_ERR_ARG;
  if (stage == -1) {
    *draft = slots;
    *retrieved = 0;
    return GT_OK;
  }
  if (slots != 60) return GT_ERR_ARG;
  switch (stage) {
    case 0: *draft = 8; *retrieved = 52; return GT_OK;
    case 1: *draft = 24; *retrieved = 36; return GT_OK;
    case 5: *draft = 40; *retrieved = 20; return GT_OK;
    default: return GT_ERR_ARG;
  }
}

// Best-first selection over successor-rank paths. A candidate is (weight, depth, path);
// weight = prod(rank + 2) grows strictly along a path, so parents are always chosen
// before their children and every prefix of the output is ancestor-closed.
GT_API int gt_default_template(int T, int k, int max_depth, int32_t *tpar, int32_t *trank) {
  if (T < 0 || k < 1 || max_depth < 1 || (T > 0 && (!tpar || !trank))) return GT_ERR_ARG;
  using Cand = std::tuple<long long, int, std::vector<int>>;
  std::priority_queue<Cand, std::vector<Cand>, std::greater<Cand>> heap;
  for (int r = 0; r < k; ++r) heap.push(Cand(r + 2, 1, std::vector<int>{r}));
  std::map<std::vector<int>, int> index;
  int t = 0;
  while (t < T && !heap.empty()) {
    Cand c = heap.top();
    heap.pop();
    const long long w = std::get<0>(c);
    const int dep = std::get<1>(c);
    const std::vector<int> &path = std::get<2>(c);
    index[path] = t;
    if (dep > 1) {
      std::vector<int> up(path.begin(), path.end() - 1);
      tpar[t] = index[up];
    } else {
      tpar[t] = -1;
    }
    trank[t] = path.back();
    ++t;
    if (dep < max_depth && w <= (1ll << 40)) {
      for (int r = 0; r < k; ++r) {
        std::vector<int> np = path;
        np.push_back(r);
        heap.push(Cand(w * (r + 2), dep + 1, np));
      }
    }
  }
  return t == T ? GT_OK : GT_ERR_SHAPE;
}

GT_API const char *gt_status_string(int status) {
  switch (status) {
    case GT_OK: return "ok";
    case GT_ERR_ARG: return "invalid argument";
    case GT_ERR_SHAPE: return "unsupported shape";
    case GT_ERR_CUDA: return "CUDA launch or driver error";
    case GT_ERR_TREE: return "malformed tree or id out of range";
    case GT_ERR_NONMONOTONE: return "cumulative score exceeds its parent's (or NaN)";
    case GT_ERR_TIMEOUT: return "bounded device wait timed out";
    case GT_ERR_RANGE: return "device-side count exceeds its buffer";
    default: return "unknown status";
  }
}

GT_API int gt_event_record_external(void *event, gt_stream_t stream) {
  if (!event) return GT_ERR_ARG;
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing((cudaStream_t)stream, &st) != cudaSuccess) return GT_ERR_CUDA;
  const unsigned flags = st == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0u;
  return cudaEventRecordWithFlags((cudaEvent_t)event, (cudaStream_t)stream, flags) == cudaSuccess
             ? GT_OK
             : GT_ERR_CUDA;
}

namespace gt {

namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);
std::atomic<void *> g_ctx_get_current{nullptr}, g_ctx_get_id{nullptr};

void *driver_entry(const char *name, unsigned version, std::atomic<void *> &slot) {
  void *f = slot.load(std::memory_order_acquire);
  if (f) return f;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  slot.store(f, std::memory_order_release);  // every racing caller finds the same pointer
  return f;
}
}  // namespace

uint64_t current_context_id() {
  auto get_cur = reinterpret_cast<CtxGetCurrentFn>(
      driver_entry("cuCtxGetCurrent", 4000, g_ctx_get_current));
  auto get_id = reinterpret_cast<CtxGetIdFn>(driver_entry("cuCtxGetId", 12000, g_ctx_get_id));
  if (!get_cur || !get_id) return 0;
  CUcontext ctx = nullptr;
  if (get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return (uint64_t)id + 1;  // 0 stays "no context"
}

static thread_local char last_error[256];
void note_error(const char *what, cudaError_t e) {
  snprintf(last_error, sizeof(last_error), "%s: %s", what,
           e == cudaSuccess ? "failed" : cudaGetErrorString(e));
}
void note_message(const char *msg) { snprintf(last_error, sizeof(last_error), "%s", msg); }
}  // namespace gt

GT_API const char *gt_last_error(void) { return gt::last_error; }
