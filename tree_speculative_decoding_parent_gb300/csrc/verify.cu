// a5 top-k / argmax over the vocabulary, a6 greedy path walk + commit indices,
// a7 successor-table update.
//
// Sources: "浙江大学、阿里巴巴联手破解AI推理瓶颈" §二 third gear (one parallel verify of the
// flattened tree; the row of every verified position is rewritten with the target's most
// likely next tokens) and §六 (accepted and rejected positions both update the table);
// "TreeGraft 精读：多起草器共嫁接一棵草稿树，让投机解码跨越快与好的单选题" §一 (accept the agreeing
// prefix, roll back at the first error) and §五 (greedy decoding, temperature 0).
//
// Top-k design (HBM-bound: rows * V * 4 bytes, read once):
//   - a thread-block cluster of CL CTAs shares one row; each CTA streams a contiguous
//     1/CL of the row with 128-bit evict-first loads, so the 60-960 rows of a step fill
//     all 152 SMs;
//   - every thread keeps a sorted top-KK list in registers; an element enters only if its
//     order key beats the list's last key (one compare on the common path);
//   - lists merge warp -> CTA by KK rounds of a warp-wide max over 64-bit keys
//     (order key, inverted index), then CTA -> cluster through distributed shared
//     memory into the leader CTA, which writes the row's result.
#include <cooperative_groups.h>
#include <math.h>

#include "gt_internal.cuh"
#include "launch.cuh"

namespace cg = cooperative_groups;

namespace gt {

constexpr int TOPK_THREADS = 256;
constexpr int TOPK_CLUSTER = 8;

__device__ __forceinline__ uint64_t pack_key(uint32_t key, int idx) {
  return ((uint64_t)key << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)idx);
}
__device__ __forceinline__ int unpack_idx(uint64_t p) {
  return (int)(0xFFFFFFFFu - (uint32_t)(p & 0xFFFFFFFFull));
}

// Insert (nk, ni) into a list sorted by key descending. Callers scan indices in
// increasing order, so on equal keys the new element (larger index) goes below.
template <int KK>
__device__ __forceinline__ void list_insert(uint32_t (&key)[KK], int (&idx)[KK], uint32_t nk,
                                            int ni) {
#pragma unroll
  for (int j = KK - 1; j >= 0; --j) {
    if (nk > key[j]) {
      if (j > 0 && nk > key[j - 1]) {
        key[j] = key[j - 1];
        idx[j] = idx[j - 1];
      } else {
        key[j] = nk;
        idx[j] = ni;
      }
    }
  }
}

template <int KK>
__device__ __forceinline__ void consider(uint32_t (&key)[KK], int (&idx)[KK], float f, int i) {
  const uint32_t kx = order_key(f);
  if (kx > key[KK - 1]) list_insert<KK>(key, idx, kx, i);
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// KK rounds of a warp-wide max over each lane's list head; lane r returns the r-th best.
template <int KK>
__device__ __forceinline__ uint64_t warp_merge_lists(uint32_t (&key)[KK], int (&idx)[KK]) {
  const int lane = threadIdx.x & 31;
  uint64_t out = 0;
#pragma unroll
  for (int r = 0; r < KK; ++r) {
    const uint64_t my = pack_key(key[0], idx[0]);
    const uint64_t best = warp_max_u64(my);
    if (best != 0 && my == best) {
#pragma unroll
      for (int j = 0; j < KK - 1; ++j) {
        key[j] = key[j + 1];
        idx[j] = idx[j + 1];
      }
      key[KK - 1] = 0u;
      idx[KK - 1] = -1;
    }
    if (lane == r) out = best;
  }
  return out;
}

// KK rounds over NC unsorted candidates per lane; lane r returns the r-th best.
template <int KK, int NC>
__device__ __forceinline__ uint64_t warp_merge_cands(uint64_t (&c)[NC]) {
  const int lane = threadIdx.x & 31;
  uint64_t out = 0;
#pragma unroll
  for (int r = 0; r < KK; ++r) {
    uint64_t my = c[0];
#pragma unroll
    for (int j = 1; j < NC; ++j) my = c[j] > my ? c[j] : my;
    const uint64_t best = warp_max_u64(my);
    if (best != 0) {
#pragma unroll
      for (int j = 0; j < NC; ++j)
        if (c[j] == best) c[j] = 0;
    }
    if (lane == r) out = best;
  }
  return out;
}

template <int KK, int CL>
__global__ void __launch_bounds__(TOPK_THREADS)
topk_cluster_kernel(const float *__restrict__ logits, int row0, int V, int k,
                    int32_t *__restrict__ ids, float *__restrict__ vals) {
  constexpr int NW = TOPK_THREADS / 32;
  __shared__ uint64_t s_warp[NW * KK];
  __shared__ uint64_t s_clus[CL * KK];
  cg::cluster_group cluster = cg::this_cluster();
  // Every CTA of the cluster must be running before the leader's shared memory is
  // written remotely; arrive now, wait just before that write.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");

  const int crank = (int)cluster.block_rank();
  const int row = row0 + blockIdx.y;
  const float *x = logits + (size_t)row * V;
  uint32_t key[KK];
  int idx[KK];
#pragma unroll
  for (int j = 0; j < KK; ++j) {
    key[j] = 0u;
    idx[j] = -1;
  }
  const int tid = threadIdx.x;
  const bool vec = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  if (vec) {
    const int V4 = V >> 2;
    const int b4 = (int)((long long)V4 * crank / CL), e4 = (int)((long long)V4 * (crank + 1) / CL);
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    int i = b4 + tid;
    for (; i + 3 * TOPK_THREADS < e4; i += 4 * TOPK_THREADS) {
      const float4 a = __ldcs(x4 + i);
      const float4 b = __ldcs(x4 + i + TOPK_THREADS);
      const float4 c = __ldcs(x4 + i + 2 * TOPK_THREADS);
      const float4 d = __ldcs(x4 + i + 3 * TOPK_THREADS);
      int base = 4 * i;
      consider<KK>(key, idx, a.x, base), consider<KK>(key, idx, a.y, base + 1);
      consider<KK>(key, idx, a.z, base + 2), consider<KK>(key, idx, a.w, base + 3);
      base += 4 * TOPK_THREADS;
      consider<KK>(key, idx, b.x, base), consider<KK>(key, idx, b.y, base + 1);
      consider<KK>(key, idx, b.z, base + 2), consider<KK>(key, idx, b.w, base + 3);
      base += 4 * TOPK_THREADS;
      consider<KK>(key, idx, c.x, base), consider<KK>(key, idx, c.y, base + 1);
      consider<KK>(key, idx, c.z, base + 2), consider<KK>(key, idx, c.w, base + 3);
      base += 4 * TOPK_THREADS;
      consider<KK>(key, idx, d.x, base), consider<KK>(key, idx, d.y, base + 1);
      consider<KK>(key, idx, d.z, base + 2), consider<KK>(key, idx, d.w, base + 3);
    }
    for (; i < e4; i += TOPK_THREADS) {
      const float4 a = __ldcs(x4 + i);
      const int base = 4 * i;
      consider<KK>(key, idx, a.x, base), consider<KK>(key, idx, a.y, base + 1);
      consider<KK>(key, idx, a.z, base + 2), consider<KK>(key, idx, a.w, base + 3);
    }
  } else {
    const int b = (int)((long long)V * crank / CL), e = (int)((long long)V * (crank + 1) / CL);
    for (int i = b + tid; i < e; i += TOPK_THREADS) consider<KK>(key, idx, __ldcs(x + i), i);
  }

  // warp -> CTA
  const int lane = tid & 31, warp = tid >> 5;
  const uint64_t wbest = warp_merge_lists<KK>(key, idx);
  if (lane < KK) s_warp[warp * KK + lane] = wbest;
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
  if (warp == 0) {
    constexpr int NC = (NW * KK + 31) / 32;
    uint64_t c[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int q = lane + 32 * j;
      c[j] = q < NW * KK ? s_warp[q] : 0ull;
    }
    const uint64_t cbest = warp_merge_cands<KK, NC>(c);
    uint64_t *leader = cluster.map_shared_rank(s_clus, 0);
    if (lane < KK) leader[crank * KK + lane] = cbest;
  }
  cluster.sync();
  if (crank == 0 && warp == 0) {
    constexpr int NC = (CL * KK + 31) / 32;
    uint64_t c[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int q = lane + 32 * j;
      c[j] = q < CL * KK ? s_clus[q] : 0ull;
    }
    const uint64_t best = warp_merge_cands<KK, NC>(c);
    if (lane < k) {
      const int id = best ? unpack_idx(best) : -1;
      ids[(size_t)row * k + lane] = id;
      vals[(size_t)row * k + lane] = id >= 0 ? x[id] : __int_as_float(0x7fc00000);
    }
  }
}

static int topk_launch(const float *logits, int rows, int V, int k, int32_t *ids, float *vals,
                       cudaStream_t s) {
  for (int r0 = 0; r0 < rows; r0 += 65535) {
    const int nr = min(65535, rows - r0);
    int rc;
    if (k <= 8)
      rc = launch_cluster(topk_cluster_kernel<8, TOPK_CLUSTER>, dim3(TOPK_CLUSTER, nr),
                          dim3(TOPK_THREADS), dim3(TOPK_CLUSTER, 1, 1), 0, s, logits, r0, V, k,
                          ids, vals);
    else
      rc = launch_cluster(topk_cluster_kernel<16, TOPK_CLUSTER>, dim3(TOPK_CLUSTER, nr),
                          dim3(TOPK_THREADS), dim3(TOPK_CLUSTER, 1, 1), 0, s, logits, r0, V, k,
                          ids, vals);
    if (rc != GT_OK) return rc;
  }
  return GT_OK;
}

// ------------------------------------------------------------------------------------
// a6: greedy walk. Thread v walks its root path checking tokens[u] == argmax[parent[u]]
// on each edge; the deepest accepted node (ties: smaller index) wins a block max over
// (depth << 16 | ~v).
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
walk_kernel(const int32_t *__restrict__ tokens, const int32_t *__restrict__ parent,
            const int32_t *__restrict__ n_nodes, const int32_t *__restrict__ prefix_len, int N,
            int k, const int32_t *__restrict__ topk_id, int32_t *__restrict__ acc_len,
            int32_t *__restrict__ path, int32_t *__restrict__ out_tok,
            int32_t *__restrict__ kv_src, int32_t *__restrict__ kv_dst, int32_t *err) {
  extern __shared__ int s_w[];
  int *s_par = s_w, *s_tok = s_w + N, *s_am = s_w + 2 * N, *s_path = s_w + 3 * N;
  __shared__ uint32_t s_best[32];
  __shared__ int s_bad;
  const int b = blockIdx.x, v = threadIdx.x;
  const size_t row0 = (size_t)b * N;
  const int n = n_nodes[b], P = prefix_len[b];
  if (v == 0) s_bad = 0;
  int code = (n < 1 || n > N) ? GT_ERR_RANGE : 0;
  if (!code && v < n) {
    const int p = parent[row0 + v];
    s_par[v] = p;
    s_tok[v] = tokens[row0 + v];
    s_am[v] = topk_id[(row0 + v) * k];
    if (v == 0 ? (p != -1) : (p < 0 || p >= v)) code = GT_ERR_TREE;
  }
  __syncthreads();
  if (code) atomicCAS(&s_bad, 0, code);
  __syncthreads();
  const int bad = s_bad;
  int L = 0, vstar = 0;
  if (!bad) {
    uint32_t key = 0u;
    if (v < n) {
      bool acc = true;
      int d = 0;
      for (int u = v; u != 0; u = s_par[u]) {
        acc = acc && (s_tok[u] == s_am[s_par[u]]);
        ++d;
      }
      if (acc) key = ((uint32_t)d << 16) | (0xFFFFu - (uint32_t)v);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
    if ((v & 31) == 0) s_best[v >> 5] = key;
    __syncthreads();
    uint32_t best = 0u;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) best = max(best, s_best[w]);
    L = (int)(best >> 16);
    vstar = (int)(0xFFFFu - (best & 0xFFFFu));
    if (v <= L) {
      int u = vstar;
      for (int s = 0; s < L - v; ++s) u = s_par[u];
      s_path[v] = u;
    }
    __syncthreads();
  } else if (v == 0) {
    set_err(err, bad);
  }
  if (v < N) {
    const bool on = !bad && v <= L;
    path[row0 + v] = on ? s_path[v] : -1;
    kv_src[row0 + v] = on ? P + s_path[v] : -1;
    kv_dst[row0 + v] = on ? P + v : -1;
  }
  for (int j = v; j < N + 1; j += blockDim.x) {
    int t = -1;
    if (!bad && j < L) t = s_tok[s_path[j + 1]];
    else if (!bad && j == L) t = s_am[vstar];
    out_tok[(size_t)b * (N + 1) + j] = t;
  }
  if (v == 0) acc_len[b] = bad ? 0 : L;
}

// ------------------------------------------------------------------------------------
// a7: table update. Candidate i = b*N + v writes row tokens[i] iff no later valid
// candidate carries the same token; winners own distinct rows, so plain stores suffice.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
update_kernel(int32_t *__restrict__ table, int V, int k, const int32_t *__restrict__ tokens,
              const int32_t *__restrict__ topk_id, const int32_t *__restrict__ n_nodes, int N,
              int total, int32_t *err) {
  extern __shared__ int s_tok[];  // [total]
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    const int b = i / N, v = i - b * N;
    const int n = n_nodes[b];
    int t = -1;
    if (n < 0 || n > N) {
      if (v == 0) set_err(err, GT_ERR_RANGE);
    } else if (v < n) {
      t = tokens[i];
      if (t < 0 || t >= V) {
        set_err(err, GT_ERR_TREE);
        t = -1;
      }
    }
    s_tok[i] = t;
  }
  __syncthreads();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int t = s_tok[i];
  if (t < 0) return;
  for (int j = i + 1; j < total; ++j)
    if (s_tok[j] == t) return;
  const int32_t *src = topk_id + (size_t)i * k;
  int32_t *dst = table + (size_t)t * k;
  for (int c = 0; c < k; ++c) dst[c] = src[c];
}

}  // namespace gt

using namespace gt;

GT_API int gt_vocab_topk(const float *logits, int rows, int V, int k, int32_t *ids,
                         float *vals, gt_stream_t stream) {
  if (rows < 0 || V < 1 || k < 1) return GT_ERR_ARG;
  if (k > 16 || k > V) return GT_ERR_SHAPE;
  if (rows == 0) return GT_OK;
  if (!logits || !ids || !vals) return GT_ERR_ARG;
  return topk_launch(logits, rows, V, k, ids, vals, (cudaStream_t)stream);
}

GT_API int gt_verify_greedy(const float *logits, const int32_t *tokens, const int32_t *parent,
                            const int32_t *n_nodes, const int32_t *prefix_len, int B, int N,
                            int V, int k, int32_t *topk_id, float *topk_val, int32_t *acc_len,
                            int32_t *path, int32_t *out_tok, int32_t *kv_src, int32_t *kv_dst,
                            int32_t *err, gt_stream_t stream) {
  if (B < 0 || N < 1 || V < 1 || k < 1) return GT_ERR_ARG;
  if (N > 1024 || k > 16 || k > V) return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (!logits || !tokens || !parent || !n_nodes || !prefix_len || !topk_id || !topk_val ||
      !acc_len || !path || !out_tok || !kv_src || !kv_dst)
    return GT_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int rc = topk_launch(logits, B * N, V, k, topk_id, topk_val, s);
  if (rc != GT_OK) return rc;
  const int threads = (N + 31) / 32 * 32;
  return launch(walk_kernel, dim3(B), dim3(threads), 4 * sizeof(int) * (size_t)N, s, tokens,
                parent, n_nodes, prefix_len, N, k, topk_id, acc_len, path, out_tok, kv_src,
                kv_dst, err);
}

GT_API int gt_succ_update(int32_t *table, int V, int k, const int32_t *tokens,
                          const int32_t *topk_id, const int32_t *n_nodes, int B, int N,
                          int32_t *err, gt_stream_t stream) {
  if (B < 0 || N < 1 || V < 1 || k < 1) return GT_ERR_ARG;
  const long long total = (long long)B * N;
  if (total > 16384) return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (!table || !tokens || !topk_id || !n_nodes) return GT_ERR_ARG;
  const size_t smem = sizeof(int) * (size_t)total;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(update_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return launch_status(e);
  }
  const int blocks = (int)((total + 255) / 256);
  return launch(update_kernel, dim3(blocks), dim3(256), smem, (cudaStream_t)stream, table, V, k,
                tokens, topk_id, n_nodes, N, (int)total, err);
}
