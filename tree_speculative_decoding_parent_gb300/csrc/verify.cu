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
//   - a thread-block cluster of CL CTAs shares one row; each CTA takes a contiguous 1/CL of
//     it, so the 60-960 rows of a step fill the GPU in one wave. Each thread streams its
//     part in chunks of PER float4 with the next chunk's loads in flight (evict-first);
//   - threshold: from the first chunk, the KK-th largest of the CTA's lane maxima (warp
//     bitonic sorts); KK distinct elements lie at or above it, so nothing below reaches the
//     CTA's top-KK. Elements not below it (ties and NaN included) are appended to a shared
//     buffer; for ordinary logits that is a few dozen per CTA;
//   - one warp merges the buffer by KK rounds of a warp argmax built from two redux.sync
//     reductions (order key, then lowest index); the CTA results meet in the cluster
//     leader's shared memory (DSMEM) for the same merge;
//   - a buffer overflow (massive ties) redoes the CTA's part with exact per-thread sorted
//     lists, so the threshold never decides correctness; rows whose length or alignment
//     rules out 16-byte loads take that path too.
#include <math.h>

#include "gt_internal.cuh"
#include "launch.cuh"
#include "sample.cuh"
#include "topk_common.cuh"

namespace gt {

template <int KK, int CL>
__global__ void __launch_bounds__(TOPK_THREADS)
topk_cluster_kernel(const float *__restrict__ logits, int row0, int V, int k,
                    int32_t *__restrict__ ids, float *__restrict__ vals, int32_t *err) {
  pdl_enter();
  bool nan_seen = false;  // checked builds: a NaN logit is reported as GT_ERR_VALUE
  constexpr int NW = TOPK_THREADS / 32;
  constexpr int CH = TOPK_PER * TOPK_THREADS;  // float4 per chunk of the CTA
  __shared__ uint64_t s_cand[TOPK_CAP];        // candidates, then scratch of the merges
  __shared__ uint64_t s_top[KK];               // the CTA's top-KK
  __shared__ uint64_t s_clus[CL * KK];
  __shared__ uint32_t s_lmax[NW * KK];         // each warp's KK largest lane maxima
  __shared__ uint32_t s_thr;
  __shared__ int s_cnt;
  cg::cluster_group cluster = cg::this_cluster();
  // Every CTA of the cluster must be running before the leader's shared memory is
  // written remotely; arrive now, wait just before that write.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");

  const int crank = (int)cluster.block_rank();
  const int row = row0 + blockIdx.y;
  const float *x = logits + (size_t)row * V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_cnt = 0;

  const bool vec = ((V & 3) == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  if (vec) {
    const int V4 = V >> 2;
    const int b4 = (int)((long long)V4 * crank / CL), e4 = (int)((long long)V4 * (crank + 1) / CL);
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    float4 a[TOPK_PER], nx[TOPK_PER];
#pragma unroll
    for (int u = 0; u < TOPK_PER; ++u) {
      const int q = b4 + tid + u * TOPK_THREADS;
      a[u] = q < e4 ? __ldcs(x4 + q) : ninf;
    }
    float thr = -INFINITY;
    for (int c0 = b4; c0 < e4; c0 += CH) {
      // the next chunk's loads are in flight while this chunk is examined
#pragma unroll
      for (int u = 0; u < TOPK_PER; ++u) {
        const int q = c0 + CH + tid + u * TOPK_THREADS;
        nx[u] = q < e4 ? __ldcs(x4 + q) : ninf;
      }
      if (c0 == b4) {
        // threshold: the KK-th largest of the CTA's lane maxima over the first chunk; KK
        // distinct elements lie at or above it, so nothing below reaches the CTA's top-KK
        uint32_t km = 0u;
#pragma unroll
        for (int u = 0; u < TOPK_PER; ++u)
          if (c0 + tid + u * TOPK_THREADS < e4)
            km = max(km, max(max(order_key(a[u].x), order_key(a[u].y)),
                             max(order_key(a[u].z), order_key(a[u].w))));
        const uint32_t sorted = warp_sorted_desc(km);
        if (lane < KK) s_lmax[warp * KK + lane] = sorted;
        __syncthreads();
        if (warp == 0) {
          constexpr int NC = (NW * KK + 31) / 32;
          uint32_t v = 0u;
          // each lane keeps the max of its NC values, then the KK-th largest over lanes is a
          // lower bound of the KK-th largest of all NW*KK values (each lane's max is one
          // distinct value)
#pragma unroll
          for (int j = 0; j < NC; ++j) {
            const int q = lane + 32 * j;
            if (q < NW * KK) v = max(v, s_lmax[q]);
          }
          const uint32_t kth = __shfl_sync(0xffffffffu, warp_sorted_desc(v), KK - 1);
          if (lane == 0) s_thr = kth;
        }
        __syncthreads();
        thr = key_floor(s_thr);
      }
#pragma unroll
      for (int u = 0; u < TOPK_PER; ++u) {
        const int q = c0 + tid + u * TOPK_THREADS;
        const float e[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (GT_CHECK && q < e4) nan_seen |= e[c] != e[c];
          if (q < e4 && !(e[c] < thr)) {
            const int pos = atomicAdd(&s_cnt, 1);
            if (pos < TOPK_CAP) s_cand[pos] = pack_key(order_key(e[c]), 4 * q + c);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < TOPK_PER; ++u) a[u] = nx[u];
    }
    __syncthreads();
    const int cnt = s_cnt;
    if (cnt > TOPK_CAP) {
      __syncthreads();  // the buffer is reused as scratch
      topk_exact<KK>(x, 4 * b4, 4 * e4, s_cand, s_top);
    } else {
      select_candidates<KK>(cnt, s_cand, s_top);
    }
  } else {
    const int b = (int)((long long)V * crank / CL), e = (int)((long long)V * (crank + 1) / CL);
    topk_exact<KK>(x, b, e, s_cand, s_top);
    if (GT_CHECK)
      for (int i = b + tid; i < e; i += TOPK_THREADS) nan_seen |= x[i] != x[i];
  }
  GT_CHECKED(!nan_seen, err, GT_ERR_VALUE);

  // CTA -> cluster leader (every CTA of the cluster is running after the wait)
  asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
  send_to_leader<KK>(cluster, crank, s_top, s_clus);
  cluster.sync();
  leader_write<KK, CL>(crank, s_clus, x, row, k, ids, vals);
}

template <int KK, int CL>
static int topk_launch_cl(const float *logits, int r0, int nr, int V, int k, int32_t *ids,
                          float *vals, int32_t *err, cudaStream_t s) {
  return launch_cluster(topk_cluster_kernel<KK, CL>, dim3(CL, nr), dim3(TOPK_THREADS),
                        dim3(CL, 1, 1), 0, s, logits, r0, V, k, ids, vals, err);
}

template <int KK>
static int topk_launch_k(const float *logits, int r0, int nr, int V, int k, int32_t *ids,
                         float *vals, int cl, int32_t *err, cudaStream_t s) {
  switch (cl) {
    case 2: return topk_launch_cl<KK, 2>(logits, r0, nr, V, k, ids, vals, err, s);
    case 4: return topk_launch_cl<KK, 4>(logits, r0, nr, V, k, ids, vals, err, s);
    default: return topk_launch_cl<KK, TOPK_CLUSTER>(logits, r0, nr, V, k, ids, vals, err, s);
  }
}

// err: the device error word of the calling entry point (NULL for gt_vocab_topk, which has
// none); only checked builds write to it.
static int topk_launch(const float *logits, int rows, int V, int k, int32_t *ids, float *vals,
                       int32_t *err, cudaStream_t s) {
  // CTAs per row: enough that the rows fill the GPU with about four CTAs per SM, and at
  // least two. Each split costs one more merge per row, while a whole-row CTA takes its
  // threshold from too small a first chunk of a long row and overflows its candidate
  // buffer (measured at 960 rows of 151,936: 2 CTAs 103 us, 8 CTAs 117 us, 1 CTA 256 us).
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    sms = 148;
  }
  int cl = 2;
  while (cl < TOPK_CLUSTER && (long long)rows * cl < 4ll * sms) cl *= 2;
  for (int r0 = 0; r0 < rows; r0 += 65535) {
    const int nr = min(65535, rows - r0);
    const int rc = k <= 8 ? topk_launch_k<8>(logits, r0, nr, V, k, ids, vals, cl, err, s)
                          : topk_launch_k<16>(logits, r0, nr, V, k, ids, vals, cl, err, s);
    if (rc != GT_OK) return rc;
  }
  return GT_OK;
}

// ------------------------------------------------------------------------------------
// a6: greedy walk. Thread v walks its root path checking tokens[u] == argmax[parent[u]]
// on each edge; the deepest accepted node (ties: smaller index) wins a block max over
// (depth << 16 | ~v).
// ------------------------------------------------------------------------------------
// With one target draw per node (T > 0) the walk enters only the first child carrying the
// draw: a later sibling with the same token as an earlier one can never be entered, so its
// token is replaced by -1 (draws are never negative). Every thread of the block calls this.
__device__ __forceinline__ void shadow_duplicates(const int *s_par, int *s_tok, int n, int v,
                                                  int nthreads = 0) {
  bool shadowed = false;
  if (v < n && v > 0)
    for (int w = 1; w < v && !shadowed; ++w)
      shadowed = s_par[w] == s_par[v] && s_tok[w] == s_tok[v];
  sync_threads_n(nthreads);
  if (shadowed) s_tok[v] = -1;
  sync_threads_n(nthreads);
}

__global__ void __launch_bounds__(1024)
walk_kernel(const int32_t *__restrict__ tokens, const int32_t *__restrict__ parent,
            const int32_t *__restrict__ n_nodes, const int32_t *__restrict__ prefix_len, int N,
            int V, int k, const int32_t *__restrict__ topk_id, const int32_t *__restrict__ sample,
            int32_t *__restrict__ acc_len, int32_t *__restrict__ path,
            int32_t *__restrict__ out_tok, int32_t *__restrict__ kv_src,
            int32_t *__restrict__ kv_dst, int32_t *err) {
  pdl_enter();
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
    s_am[v] = sample ? sample[row0 + v] : topk_id[(row0 + v) * k];
    if (v == 0 ? (p != -1) : (p < 0 || p >= v)) code = GT_ERR_TREE;
    // checked builds: every verified token is a vocabulary id (the walk itself only compares)
    if (GT_CHECK && (s_tok[v] < 0 || s_tok[v] >= V)) code = GT_ERR_TREE;
  }
  __syncthreads();
  if (code) atomicCAS(&s_bad, 0, code);
  __syncthreads();
  const int bad = s_bad;
  int L = 0, vstar = 0;
  if (!bad) {
    if (sample) shadow_duplicates(s_par, s_tok, n, v);
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
  pdl_enter();
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

// ------------------------------------------------------------------------------------
// a6 + a7 fused: CTA b walks request b's tree (as walk_kernel) and then writes the table
// rows its verified nodes win (as update_kernel: the largest linear index b*N + v of a
// token wins). Every CTA stages the tokens of all requests in shared memory for that test
// and, when it fits, hashes them (open addressing, token -> largest index) so that the
// test is one lookup per node instead of a scan of every later node.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
walk_update_kernel(const int32_t *__restrict__ tokens, const int32_t *__restrict__ parent,
                   const int32_t *__restrict__ n_nodes, const int32_t *__restrict__ prefix_len,
                   int B, int N, int k, const int32_t *__restrict__ topk_id,
                   const int32_t *__restrict__ sample, int32_t *__restrict__ acc_len, int32_t *__restrict__ path,
                   int32_t *__restrict__ out_tok, int32_t *__restrict__ kv_src,
                   int32_t *__restrict__ kv_dst, int32_t *__restrict__ table, int V, int hs,
                   int32_t *err) {
  pdl_enter();
  extern __shared__ int s_w[];
  int *s_par = s_w, *s_tok = s_w + N, *s_am = s_w + 2 * N, *s_path = s_w + 3 * N;
  int *s_all = s_w + 4 * N;  // [B*N] verified tokens of every request (-1: none)
  int *s_hk = s_all + B * N, *s_hv = s_hk + hs;  // [hs] hash keys (tokens) and last indices
  for (int i = threadIdx.x; i < hs; i += blockDim.x) s_hk[i] = s_hv[i] = -1;
  __shared__ uint32_t s_best[32];
  __shared__ int s_bad;
  const int b = blockIdx.x, v = threadIdx.x;
  const int total = B * N;
  const size_t row0 = (size_t)b * N;
  // node v's own reads are in bounds for any v < N: they are issued together with the
  // node count, not after it, and the node's top-k row waits in registers for the table
  int p_v = -1, tok_v = -1, am_v = -1;
  int krow[16];
  if (v < N) {
    p_v = parent[row0 + v];
    tok_v = tokens[row0 + v];
    am_v = sample ? sample[row0 + v] : topk_id[(row0 + v) * k];
#pragma unroll
    for (int c = 0; c < 16; ++c) krow[c] = c < k ? topk_id[(row0 + v) * k + c] : -1;
  }
  const int n = n_nodes[b], P = prefix_len[b];
  if (v == 0) s_bad = 0;
  for (int i = v; i < total; i += blockDim.x) {
    const int bb = i / N, vv = i - bb * N;
    const int nn = n_nodes[bb];
    int t = -1;
    if (nn >= 0 && nn <= N && vv < nn) {
      t = tokens[i];
      if (t < 0 || t >= V) {
        if (bb == b) set_err(err, GT_ERR_TREE);
        t = -1;
      }
    } else if ((nn < 0 || nn > N) && vv == 0 && bb == b) {
      set_err(err, GT_ERR_RANGE);
    }
    s_all[i] = t;
  }
  int code = (n < 1 || n > N) ? GT_ERR_RANGE : 0;
  if (!code && v < n) {
    const int p = p_v;
    s_par[v] = p;
    s_tok[v] = tok_v;
    s_am[v] = am_v;
    if (v == 0 ? (p != -1) : (p < 0 || p >= v)) code = GT_ERR_TREE;
    if (GT_CHECK && (tok_v < 0 || tok_v >= V)) code = GT_ERR_TREE;
  }
  __syncthreads();
  if (code) atomicCAS(&s_bad, 0, code);
  __syncthreads();
  const int bad = s_bad;
  int L = 0, vstar = 0;
  if (!bad) {
    if (sample) shadow_duplicates(s_par, s_tok, n, v);
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
  // table rows won by this request's verified nodes
  auto slot0 = [&](int t) { return (int)(((uint32_t)t * 2654435761u) & (uint32_t)(hs - 1)); };
  if (hs > 0) {  // hs is a power of two above B*N, so every probe sequence ends
    for (int i = v; i < total; i += blockDim.x) {
      const int t = s_all[i];
      if (t < 0) continue;
      for (int h = slot0(t);; h = (h + 1) & (hs - 1)) {
        const int prev = atomicCAS(&s_hk[h], -1, t);
        if (prev == -1 || prev == t) {
          atomicMax(&s_hv[h], i);
          break;
        }
      }
    }
    __syncthreads();
  }
  for (int vv = v; vv < N; vv += blockDim.x) {
    const int i = b * N + vv;
    const int t = s_all[i];
    if (t < 0) continue;
    bool last = true;
    if (hs > 0) {
      int h = slot0(t);
      while (s_hk[h] != t) h = (h + 1) & (hs - 1);
      last = s_hv[h] == i;
    } else {
      for (int j = i + 1; j < total; ++j)
        if (s_all[j] == t) {
          last = false;
          break;
        }
    }
    if (!last) continue;
    int32_t *dst = table + (size_t)t * k;
    if (vv == v) {  // the launch gives every node its own thread (blockDim >= N)
#pragma unroll
      for (int c = 0; c < 16; ++c)
        if (c < k) dst[c] = krow[c];
    } else {
      const int32_t *src = topk_id + (size_t)i * k;
      for (int c = 0; c < k; ++c) dst[c] = src[c];
    }
  }
}

// walk_update_kernel with the two halves of its work on separate warps, concurrently: the
// first nw threads (a thread per node) walk the tree and write the path, the tokens and the
// commit indices, synchronising on named barrier 1; the next nu threads stage every
// request's verified tokens, hash them and write this request's table rows, on named
// barrier 2. The table rows depend on every node's tokens and top-k, not on the walk, so
// neither half waits for the other. Same results and error codes as walk_update_kernel.
__global__ void __launch_bounds__(1024, 1)
walk_update_split_kernel(const int32_t *__restrict__ tokens, const int32_t *__restrict__ parent,
                         const int32_t *__restrict__ n_nodes,
                         const int32_t *__restrict__ prefix_len, int B, int N, int k,
                         const int32_t *__restrict__ topk_id, const int32_t *__restrict__ sample,
                         int32_t *__restrict__ acc_len, int32_t *__restrict__ path,
                         int32_t *__restrict__ out_tok, int32_t *__restrict__ kv_src,
                         int32_t *__restrict__ kv_dst, int32_t *__restrict__ table, int V, int hs,
                         int nw, int32_t *err) {
  pdl_enter();
  extern __shared__ int s_w[];
  int *s_par = s_w, *s_tok = s_w + N, *s_am = s_w + 2 * N, *s_path = s_w + 3 * N;
  int *s_all = s_w + 4 * N;  // [B*N] verified tokens of every request (-1: none)
  int *s_hk = s_all + B * N, *s_hv = s_hk + hs;  // [hs] hash keys (tokens) and last indices
  __shared__ uint32_t s_best[32];
  __shared__ int s_bad;
  const int b = blockIdx.x, total = B * N;
  const size_t row0 = (size_t)b * N;
  if ((int)threadIdx.x < nw) {
    // ----------------------------------------------------------------------- the walk
    const int v = threadIdx.x;
    int p_v = -1, tok_v = -1, am_v = -1;
    if (v < N) {
      p_v = parent[row0 + v];
      tok_v = tokens[row0 + v];
      am_v = sample ? sample[row0 + v] : topk_id[(row0 + v) * k];
    }
    const int n = n_nodes[b], P = prefix_len[b];
    if (v == 0) s_bad = 0;
    int code = (n < 1 || n > N) ? GT_ERR_RANGE : 0;
    if (!code && v < n) {
      const int p = p_v;
      s_par[v] = p;
      s_tok[v] = tok_v;
      s_am[v] = am_v;
      if (v == 0 ? (p != -1) : (p < 0 || p >= v)) code = GT_ERR_TREE;
      if (GT_CHECK && (tok_v < 0 || tok_v >= V)) code = GT_ERR_TREE;
    }
    sync_threads_n(nw);
    if (code) atomicCAS(&s_bad, 0, code);
    sync_threads_n(nw);
    const int bad = s_bad;
    int L = 0, vstar = 0;
    if (!bad) {
      if (sample) shadow_duplicates(s_par, s_tok, n, v, nw);
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
      sync_threads_n(nw);
      uint32_t best = 0u;
      for (int w = 0; w < (nw >> 5); ++w) best = max(best, s_best[w]);
      L = (int)(best >> 16);
      vstar = (int)(0xFFFFu - (best & 0xFFFFu));
      if (v <= L) {
        int u = vstar;
        for (int s = 0; s < L - v; ++s) u = s_par[u];
        s_path[v] = u;
      }
      sync_threads_n(nw);
    } else if (v == 0) {
      set_err(err, bad);
    }
    if (v < N) {
      const bool on = !bad && v <= L;
      path[row0 + v] = on ? s_path[v] : -1;
      kv_src[row0 + v] = on ? P + s_path[v] : -1;
      kv_dst[row0 + v] = on ? P + v : -1;
    }
    for (int j = v; j < N + 1; j += nw) {
      int t = -1;
      if (!bad && j < L) t = s_tok[s_path[j + 1]];
      else if (!bad && j == L) t = s_am[vstar];
      out_tok[(size_t)b * (N + 1) + j] = t;
    }
    if (v == 0) acc_len[b] = bad ? 0 : L;
    return;
  }
  // ------------------------------------------------------------ the successor-table rows
  const int u = threadIdx.x - nw, nu = (int)blockDim.x - nw;
  // this thread's node's top-k row waits in registers for its table row
  int krow[16];
  if (u < N) {
#pragma unroll
    for (int c = 0; c < 16; ++c) krow[c] = c < k ? topk_id[(row0 + u) * k + c] : -1;
  }
  for (int i = u; i < hs; i += nu) s_hk[i] = s_hv[i] = -1;
  for (int i = u; i < total; i += nu) {
    const int bb = i / N, vv = i - bb * N;
    const int nn = n_nodes[bb];
    int t = -1;
    if (nn >= 0 && nn <= N && vv < nn) {
      t = tokens[i];
      if (t < 0 || t >= V) {
        if (bb == b) set_err(err, GT_ERR_TREE);
        t = -1;
      }
    } else if ((nn < 0 || nn > N) && vv == 0 && bb == b) {
      set_err(err, GT_ERR_RANGE);
    }
    s_all[i] = t;
  }
  asm volatile("bar.sync 2, %0;" ::"r"(nu) : "memory");
  auto slot0 = [&](int t) { return (int)(((uint32_t)t * 2654435761u) & (uint32_t)(hs - 1)); };
  if (hs > 0) {  // hs is a power of two above B*N, so every probe sequence ends
    for (int i = u; i < total; i += nu) {
      const int t = s_all[i];
      if (t < 0) continue;
      for (int h = slot0(t);; h = (h + 1) & (hs - 1)) {
        const int prev = atomicCAS(&s_hk[h], -1, t);
        if (prev == -1 || prev == t) {
          atomicMax(&s_hv[h], i);
          break;
        }
      }
    }
    asm volatile("bar.sync 2, %0;" ::"r"(nu) : "memory");
  }
  for (int vv = u; vv < N; vv += nu) {
    const int i = b * N + vv;
    const int t = s_all[i];
    if (t < 0) continue;
    bool last = true;
    if (hs > 0) {
      int h = slot0(t);
      while (s_hk[h] != t) h = (h + 1) & (hs - 1);
      last = s_hv[h] == i;
    } else {
      for (int j = i + 1; j < total; ++j)
        if (s_all[j] == t) {
          last = false;
          break;
        }
    }
    if (!last) continue;
    int32_t *dst = table + (size_t)t * k;
    if (vv == u) {
#pragma unroll
      for (int c = 0; c < 16; ++c)
        if (c < k) dst[c] = krow[c];
    } else {
      const int32_t *src = topk_id + (size_t)i * k;
      for (int c = 0; c < k; ++c) dst[c] = src[c];
    }
  }
}

}  // namespace gt

using namespace gt;

GT_API int gt_vocab_topk(const float *logits, int rows, int V, int k, int32_t *ids,
                         float *vals, gt_stream_t stream) {
  GT_TRACE("gt_vocab_topk");
  if (rows < 0 || V < 1 || k < 1) return GT_ERR_ARG;
  if (k > 16 || k > V) return GT_ERR_SHAPE;
  if (rows == 0) return GT_OK;
  if (!logits || !ids || !vals) return GT_ERR_ARG;
  return topk_launch(logits, rows, V, k, ids, vals, nullptr, (cudaStream_t)stream);
}

GT_API int gt_verify_greedy(const float *logits, const int32_t *tokens, const int32_t *parent,
                            const int32_t *n_nodes, const int32_t *prefix_len, int B, int N,
                            int V, int k, int32_t *topk_id, float *topk_val, int32_t *acc_len,
                            int32_t *path, int32_t *out_tok, int32_t *kv_src, int32_t *kv_dst,
                            int32_t *err, gt_stream_t stream) {
  GT_TRACE("gt_verify_greedy");
  if (B < 0 || N < 1 || V < 1 || k < 1) return GT_ERR_ARG;
  if (N > 1024 || k > 16 || k > V) return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (!logits || !tokens || !parent || !n_nodes || !prefix_len || !topk_id || !topk_val ||
      !acc_len || !path || !out_tok || !kv_src || !kv_dst)
    return GT_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int rc = topk_launch(logits, B * N, V, k, topk_id, topk_val, err, s);
  if (rc != GT_OK) return rc;
  const int threads = (N + 31) / 32 * 32;
  return launch(walk_kernel, dim3(B), dim3(threads), 4 * sizeof(int) * (size_t)N, s, tokens,
                parent, n_nodes, prefix_len, N, V, k, topk_id, (const int32_t *)nullptr, acc_len,
                path, out_tok, kv_src, kv_dst, err);
}

GT_API int gt_succ_update(int32_t *table, int V, int k, const int32_t *tokens,
                          const int32_t *topk_id, const int32_t *n_nodes, int B, int N,
                          int32_t *err, gt_stream_t stream) {
  GT_TRACE("gt_succ_update");
  if (B < 0 || N < 1 || V < 1 || k < 1) return GT_ERR_ARG;
  const long long total = (long long)B * N;
  if (total > 16384) return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (!table || !tokens || !topk_id || !n_nodes) return GT_ERR_ARG;
  const size_t smem = sizeof(int) * (size_t)total;
  if (smem > 48 * 1024) {
    static SmemAttr attr;
    const int rc = ensure_smem(update_kernel, (int)smem, attr, "cudaFuncSetAttribute(update_kernel)");
    if (rc != GT_OK) return rc;
  }
  const int blocks = (int)((total + 255) / 256);
  return launch(update_kernel, dim3(blocks), dim3(256), smem, (cudaStream_t)stream, table, V, k,
                tokens, topk_id, n_nodes, N, (int)total, err);
}

// walk + table update of a5-a7 once the top-k (and, at T > 0, the draws) are in memory
static int walk_update_launch(const int32_t *tokens, const int32_t *parent,
                              const int32_t *n_nodes, const int32_t *prefix_len, int B, int N,
                              int V, int k, const int32_t *topk_id, const int32_t *sample,
                              int32_t *acc_len, int32_t *path, int32_t *out_tok, int32_t *kv_src,
                              int32_t *kv_dst, int32_t *table, int32_t *err, cudaStream_t s) {
  // a thread per node for the walk; up to 512 threads so that the B*N verified tokens every
  // CTA stages and hashes take a few load rounds instead of B rounds
  const int threads = (max(N, min(B * N, 512)) + 31) / 32 * 32;
  // the walk and the table rows on separate warps when both fit in one block
  const int nw = (N + 31) / 32 * 32, nu = (min(B * N, 512) + 31) / 32 * 32;
  size_t smem = sizeof(int) * (4 * (size_t)N + (size_t)B * N);
  // the token hash: a power of two at least twice B*N, when it fits (else the scan)
  int hs = 1;
  while (hs < 2 * B * N) hs *= 2;
  if (smem + 2 * sizeof(int) * (size_t)hs > 160 * 1024)
    hs = 0;
  smem += 2 * sizeof(int) * (size_t)hs;
  if (nw + nu <= 1024) {
    if (smem > 48 * 1024) {
      static SmemAttr attr;
      const int rc = ensure_smem(walk_update_split_kernel, (int)smem, attr,
                                 "cudaFuncSetAttribute(walk_update_split_kernel)");
      if (rc != GT_OK) return rc;
    }
    return launch(walk_update_split_kernel, dim3(B), dim3(nw + nu), smem, s, tokens, parent,
                  n_nodes, prefix_len, B, N, k, topk_id, sample, acc_len, path, out_tok, kv_src,
                  kv_dst, table, V, hs, nw, err);
  }
  if (smem > 48 * 1024) {
    static SmemAttr attr;
    const int rc = ensure_smem(walk_update_kernel, (int)smem, attr,
                               "cudaFuncSetAttribute(walk_update_kernel)");
    if (rc != GT_OK) return rc;
  }
  return launch(walk_update_kernel, dim3(B), dim3(threads), smem, s, tokens, parent, n_nodes,
                prefix_len, B, N, k, topk_id, sample, acc_len, path, out_tok, kv_src, kv_dst,
                table, V, hs, err);
}

GT_API int gt_verify_commit(const float *logits, const int32_t *tokens, const int32_t *parent,
                            const int32_t *n_nodes, const int32_t *prefix_len, int B, int N, int V,
                            int k, int32_t *topk_id, float *topk_val, int32_t *acc_len,
                            int32_t *path, int32_t *out_tok, int32_t *kv_src, int32_t *kv_dst,
                            int32_t *table, int32_t *err, gt_stream_t stream) {
  GT_TRACE("gt_verify_commit");
  if (B < 0 || N < 1 || V < 1 || k < 1) return GT_ERR_ARG;
  if (N > 1024 || k > 16 || k > V || (long long)B * N > 16384) return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (!logits || !tokens || !parent || !n_nodes || !prefix_len || !topk_id || !topk_val ||
      !acc_len || !path || !out_tok || !kv_src || !kv_dst || !table)
    return GT_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int rc = topk_launch(logits, B * N, V, k, topk_id, topk_val, err, s);
  if (rc != GT_OK) return rc;
  return walk_update_launch(tokens, parent, n_nodes, prefix_len, B, N, V, k, topk_id, nullptr,
                            acc_len, path, out_tok, kv_src, kv_dst, table, err, s);
}

GT_API int gt_vocab_sample(const float *logits, int rows, int V, float temperature,
                           uint64_t seed, uint64_t step, int32_t *sample, gt_stream_t stream) {
  GT_TRACE("gt_vocab_sample");
  if (rows < 0 || V < 1) return GT_ERR_ARG;
  if (rows == 0) return GT_OK;
  if (!logits || !sample) return GT_ERR_ARG;
  return sample_launch(logits, rows, V, temperature, seed, step, sample, (cudaStream_t)stream);
}

GT_API int gt_verify_sample(const float *logits, const int32_t *tokens, const int32_t *parent,
                            const int32_t *n_nodes, const int32_t *prefix_len, int B, int N,
                            int V, float temperature, uint64_t seed, uint64_t step,
                            int32_t *sample, int32_t *acc_len, int32_t *path, int32_t *out_tok,
                            int32_t *kv_src, int32_t *kv_dst, int32_t *err, gt_stream_t stream) {
  GT_TRACE("gt_verify_sample");
  if (B < 0 || N < 1 || V < 1) return GT_ERR_ARG;
  if (N > 1024 || (long long)B * N > 16384) return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (!logits || !tokens || !parent || !n_nodes || !prefix_len || !sample || !acc_len ||
      !path || !out_tok || !kv_src || !kv_dst)
    return GT_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int rc = sample_launch(logits, B * N, V, temperature, seed, step, sample, s);
  if (rc != GT_OK) return rc;
  const int threads = (N + 31) / 32 * 32;
  return launch(walk_kernel, dim3(B), dim3(threads), 4 * sizeof(int) * (size_t)N, s, tokens,
                parent, n_nodes, prefix_len, N, V, 1, (const int32_t *)nullptr,
                (const int32_t *)sample, acc_len, path, out_tok, kv_src, kv_dst, err);
}

GT_API int gt_verify_sample_commit(const float *logits, const int32_t *tokens,
                                   const int32_t *parent, const int32_t *n_nodes,
                                   const int32_t *prefix_len, int B, int N, int V, int k,
                                   float temperature, uint64_t seed, uint64_t step,
                                   int32_t *topk_id, float *topk_val, int32_t *sample,
                                   int32_t *acc_len, int32_t *path, int32_t *out_tok,
                                   int32_t *kv_src, int32_t *kv_dst, int32_t *table, int32_t *err,
                                   gt_stream_t stream) {
  GT_TRACE("gt_verify_sample_commit");
  if (B < 0 || N < 1 || V < 1 || k < 1) return GT_ERR_ARG;
  if (N > 1024 || k > 16 || k > V || (long long)B * N > 16384) return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (!logits || !tokens || !parent || !n_nodes || !prefix_len || !topk_id || !topk_val ||
      !sample || !acc_len || !path || !out_tok || !kv_src || !kv_dst || !table)
    return GT_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  // the draws and the top-k of the unscaled logits in one pass over the logits
  const int rc = sample_launch(logits, B * N, V, temperature, seed, step, sample, s, k, topk_id,
                               topk_val, err);
  if (rc != GT_OK) return rc;
  return walk_update_launch(tokens, parent, n_nodes, prefix_len, B, N, V, k, topk_id, sample,
                            acc_len, path, out_tok, kv_src, kv_dst, table, err, s);
}
