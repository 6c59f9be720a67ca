// Host-side helpers of libgt: stage budget, default retrieval template, successor-table
// files, status strings, and an external event record for timing inside captured CUDA graphs.
//
// Source: "浙江大学、阿里巴巴联手破解AI推理瓶颈" §二 (prune stages 0/1/5 keep 8/24/40 draft nodes
// and refill 52/36/20 of 60 slots from the successor table; the template is asymmetric:
// higher-ranked successors get more children and go deeper).
#include <cuda.h>
#include <cuda_runtime.h>

#include <stdio.h>
#include <string.h>

#include <atomic>
#include <map>
#include <queue>
#include <string>
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

// ------------------------------------------------------------------------------------
// Successor-table persistence ([Graft] §六: the table warmed up in earlier runs is a prior
// that carries over to later ones). File layout, little-endian:
//   [0, 8)   magic "GTSUCC" 0x00 0x01 (format 1)
//   [8, 12)  uint32 V        [12, 16) uint32 k        [16, 24) uint64 payload bytes = 4 V k
//   [24, 28) uint32 CRC-32 of the payload   [28, 32) uint32 CRC-32 of bytes [0, 28)
//   [32, ..) the table, int32 [V][k] row-major
// CRC-32 is the IEEE 802.3 checksum (reflected polynomial 0xEDB88320, initial value and final
// XOR 0xFFFFFFFF), computed bit by bit from its definition.
// ------------------------------------------------------------------------------------
namespace {
constexpr unsigned char SUCC_MAGIC[8] = {'G', 'T', 'S', 'U', 'C', 'C', 0, 1};
constexpr size_t SUCC_HDR = 32;

uint32_t crc32_update(uint32_t crc, const unsigned char *p, size_t n) {
  for (size_t i = 0; i < n; ++i) {
    crc ^= p[i];
    for (int b = 0; b < 8; ++b) crc = (crc >> 1) ^ (0xEDB88320u & (0u - (crc & 1u)));
  }
  return crc;
}
uint32_t crc32_of(const unsigned char *p, size_t n) {
  return crc32_update(0xFFFFFFFFu, p, n) ^ 0xFFFFFFFFu;
}
void put_u32(unsigned char *p, uint32_t v) {
  for (int i = 0; i < 4; ++i) p[i] = (unsigned char)(v >> (8 * i));
}
void put_u64(unsigned char *p, uint64_t v) {
  for (int i = 0; i < 8; ++i) p[i] = (unsigned char)(v >> (8 * i));
}
uint32_t get_u32(const unsigned char *p) {
  uint32_t v = 0;
  for (int i = 0; i < 4; ++i) v |= (uint32_t)p[i] << (8 * i);
  return v;
}
uint64_t get_u64(const unsigned char *p) {
  uint64_t v = 0;
  for (int i = 0; i < 8; ++i) v |= (uint64_t)p[i] << (8 * i);
  return v;
}
// The table as little-endian bytes (int32 two's complement), independent of the host order.
std::vector<unsigned char> table_bytes(const int32_t *t, size_t n) {
  std::vector<unsigned char> out(4 * n);
  for (size_t i = 0; i < n; ++i) put_u32(&out[4 * i], (uint32_t)t[i]);
  return out;
}

// Reads and validates the header; on success *V, *k and *crc hold its fields.
int read_header(FILE *f, uint32_t *V, uint32_t *k, uint32_t *crc) {
  unsigned char h[SUCC_HDR];
  if (fread(h, 1, SUCC_HDR, f) != SUCC_HDR) return GT_ERR_IO;
  if (memcmp(h, SUCC_MAGIC, 8) != 0 || get_u32(h + 28) != crc32_of(h, 28)) return GT_ERR_CORRUPT;
  *V = get_u32(h + 8);
  *k = get_u32(h + 12);
  if (*V < 1 || *k < 1 || *V > 0x7FFFFFFFu || *k > 0x7FFFFFFFu ||
      get_u64(h + 16) != 4ull * (uint64_t)*V * (uint64_t)*k)
    return GT_ERR_CORRUPT;
  *crc = get_u32(h + 24);
  return GT_OK;
}
}  // namespace

GT_API int gt_succ_save(const char *path, const int32_t *table, int V, int k) {
  if (!path || !table || V < 1 || k < 1) return GT_ERR_ARG;
  const size_t n = (size_t)V * (size_t)k;
  for (size_t i = 0; i < n; ++i)
    if (table[i] < -1 || table[i] >= V) return GT_ERR_ARG;
  const std::vector<unsigned char> body = table_bytes(table, n);
  unsigned char h[SUCC_HDR];
  memcpy(h, SUCC_MAGIC, 8);
  put_u32(h + 8, (uint32_t)V);
  put_u32(h + 12, (uint32_t)k);
  put_u64(h + 16, 4ull * n);
  put_u32(h + 24, crc32_of(body.data(), body.size()));
  put_u32(h + 28, crc32_of(h, 28));
  // written under a temporary name and renamed, so the path never names a partial file
  std::string tmp = std::string(path) + ".tmp";
  FILE *f = fopen(tmp.c_str(), "wb");
  if (!f) return GT_ERR_IO;
  bool ok = fwrite(h, 1, SUCC_HDR, f) == SUCC_HDR && fwrite(body.data(), 1, body.size(), f) == body.size();
  ok = (fclose(f) == 0) && ok;
  if (!ok || rename(tmp.c_str(), path) != 0) {
    remove(tmp.c_str());
    return GT_ERR_IO;
  }
  return GT_OK;
}

GT_API int gt_succ_file_shape(const char *path, int32_t *V, int32_t *k) {
  if (!path || !V || !k) return GT_ERR_ARG;
  FILE *f = fopen(path, "rb");
  if (!f) return GT_ERR_IO;
  uint32_t v = 0, kk = 0, crc = 0;
  const int rc = read_header(f, &v, &kk, &crc);
  fclose(f);
  if (rc != GT_OK) return rc;
  *V = (int32_t)v;
  *k = (int32_t)kk;
  return GT_OK;
}

GT_API int gt_succ_load(const char *path, int32_t *table, int V, int k) {
  if (!path || !table || V < 1 || k < 1) return GT_ERR_ARG;
  FILE *f = fopen(path, "rb");
  if (!f) return GT_ERR_IO;
  uint32_t fv = 0, fk = 0, crc = 0;
  int rc = read_header(f, &fv, &fk, &crc);
  if (rc == GT_OK && (fv != (uint32_t)V || fk != (uint32_t)k)) rc = GT_ERR_SHAPE;
  const size_t n = (size_t)V * (size_t)k;
  std::vector<unsigned char> body;
  if (rc == GT_OK) {
    body.resize(4 * n);
    unsigned char extra;
    if (fread(body.data(), 1, body.size(), f) != body.size() || fread(&extra, 1, 1, f) != 0)
      rc = GT_ERR_IO;  // shorter or longer than the header says
  }
  fclose(f);
  if (rc != GT_OK) return rc;
  if (crc32_of(body.data(), body.size()) != crc) return GT_ERR_CORRUPT;
  for (size_t i = 0; i < n; ++i) {
    const int32_t e = (int32_t)get_u32(&body[4 * i]);
    if (e < -1 || e >= V) return GT_ERR_CORRUPT;
  }
  // the caller's table changes only once the whole file has been checked
  for (size_t i = 0; i < n; ++i) table[i] = (int32_t)get_u32(&body[4 * i]);
  return GT_OK;
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
    case GT_ERR_IO: return "file cannot be opened, read or written, or has the wrong length";
    case GT_ERR_CORRUPT: return "file magic, checksum or contents invalid";
    case GT_ERR_VALUE: return "NaN where a number is required (checked build)";
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
