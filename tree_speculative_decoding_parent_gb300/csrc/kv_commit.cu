// KV commit: compaction of the accepted path's cache rows.
//
// Sources: "TreeGraft 精读：多起草器共嫁接一棵草稿树，让投机解码跨越快与好的单选题" §一 (keep the
// agreeing prefix of the draft, drop everything after the first error) and
// "浙江大学、阿里巴巴联手破解AI推理瓶颈" §二 third gear (the verified tokens join the context).
//
// After the greedy walk, row kv_dst[b][j] = P_b + j of every KV head must hold the row
// that was at kv_src[b][j] = P_b + path[j], j = 0..acc_len[b]. The path's node indices grow
// with depth and path[j] >= j, so a destination of one copy can be the source of an
// earlier one (path = 0, 2, 3: row P+2 is read for j = 1 and written for j = 2). One CTA
// per (KV head, request) therefore reads every source row of the path into shared memory
// before it writes the first destination, first for K, then for V.
#include "gt_internal.cuh"
#include "launch.cuh"

namespace gt {

constexpr int KVC_THREADS = 256;
constexpr int KVC_MAX_N = 64;        // path rows per request
constexpr int KVC_MAX_ROW = 1024;    // bytes per cache row (d * element size)
constexpr int KVC_BATCH = 8;         // 16-byte chunks per thread in flight

__global__ void __launch_bounds__(KVC_THREADS)
kv_commit_kernel(uint8_t *__restrict__ K, uint8_t *__restrict__ V,
                 const int32_t *__restrict__ kv_src, const int32_t *__restrict__ kv_dst,
                 const int32_t *__restrict__ acc_len, int N, int Hkv, int Lcap, int row_bytes,
                 int32_t *err) {
  pdl_enter();
  extern __shared__ uint4 s_rows[];  // [acc_len + 1][row_bytes / 16]
  __shared__ int s_src[KVC_MAX_N], s_dst[KVC_MAX_N];
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int L = acc_len[b];
  const bool len_ok = L >= 0 && L < N;
  bool bad = !len_ok;
  if (len_ok && tid <= L) {
    const int s = kv_src[(size_t)b * N + tid], d = kv_dst[(size_t)b * N + tid];
    bad = s < 0 || s >= Lcap || d < 0 || d >= Lcap;
    s_src[tid] = s;
    s_dst[tid] = d;
  }
  if (__syncthreads_or(bad)) {  // this request keeps its cache as it was
    if (tid == 0 && h == 0) set_err(err, GT_ERR_RANGE);
    return;
  }
  const int chunks = row_bytes / 16, total = (L + 1) * chunks;
  const size_t plane = ((size_t)b * Hkv + h) * (size_t)Lcap * row_bytes;
  for (int pass = 0; pass < 2; ++pass) {
    uint8_t *X = (pass == 0 ? K : V) + plane;
    // every load of a thread's batch is issued before the first shared-memory store
    for (int e0 = tid; e0 < total; e0 += KVC_THREADS * KVC_BATCH) {
      uint4 v[KVC_BATCH];
#pragma unroll
      for (int u = 0; u < KVC_BATCH; ++u) {
        const int e = e0 + u * KVC_THREADS;
        if (e < total) {
          const int j = e / chunks, c = e - j * chunks;
          v[u] = *reinterpret_cast<const uint4 *>(X + (size_t)s_src[j] * row_bytes + c * 16);
        }
      }
#pragma unroll
      for (int u = 0; u < KVC_BATCH; ++u) {
        const int e = e0 + u * KVC_THREADS;
        if (e < total) s_rows[e] = v[u];
      }
    }
    __syncthreads();  // every source row of this pass is read before any row is written
    for (int e = tid; e < total; e += KVC_THREADS) {
      const int j = e / chunks, c = e - j * chunks;
      *reinterpret_cast<uint4 *>(X + (size_t)s_dst[j] * row_bytes + c * 16) = s_rows[e];
    }
    __syncthreads();  // the staging rows are reused by the next pass
  }
}

}  // namespace gt

using namespace gt;

GT_API int gt_kv_commit(void *K, void *V, const int32_t *kv_src, const int32_t *kv_dst,
                        const int32_t *acc_len, int B, int N, int Hkv, int d, int Lcap,
                        int dtype, int32_t *err, gt_stream_t stream) {
  GT_TRACE("gt_kv_commit");
  if (B < 0 || N < 1 || Hkv < 1 || d < 1 || Lcap < 1) return GT_ERR_ARG;
  if (dtype != GT_F32 && dtype != GT_BF16) return GT_ERR_ARG;
  const int es = dtype == GT_F32 ? 4 : 2;
  const long long row_bytes = (long long)d * es;
  if (N > KVC_MAX_N || row_bytes > KVC_MAX_ROW || row_bytes % 16 != 0 || Hkv > 65535)
    return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (B > 65535) return GT_ERR_SHAPE;
  if (!K || !V || !kv_src || !kv_dst || !acc_len) return GT_ERR_ARG;
  if (((uintptr_t)K | (uintptr_t)V) & 15) return GT_ERR_ARG;
  const size_t smem = (size_t)N * row_bytes;
  static SmemAttr attr;  // up to 64 KB of staged rows
  const int rc = ensure_smem(kv_commit_kernel, (int)((size_t)KVC_MAX_N * KVC_MAX_ROW), attr,
                             "cudaFuncSetAttribute(kv_commit_kernel)");
  if (rc != GT_OK) return rc;
  return launch(kv_commit_kernel, dim3(Hkv, B), dim3(KVC_THREADS), smem, (cudaStream_t)stream,
                (uint8_t *)K, (uint8_t *)V, kv_src, kv_dst, acc_len, N, Hkv, Lcap,
                (int)row_bytes, err);
}
