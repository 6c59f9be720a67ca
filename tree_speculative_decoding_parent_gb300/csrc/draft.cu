// Drafting side of a tree step: frontier selection, the n-gram drafter, the
// non-destructive attach.
//
// Sources: "TreeGraft 精读：多起草器共嫁接一棵草稿树，让投机解码跨越快与好的单选题" §一 (a
// training-free n-gram small drafter and a neural mid drafter grow one shared tree), §三
// (each step takes the top-W frontier of a candidate pool by cumulative path score and
// hangs the top-m children of every frontier node), §四 Where (the mid drafter's pool is
// every node it has not visited; the small drafter's pool is the newest nodes), §四 How
// (children are attached without overwriting existing nodes), §七 item 6 (the n-gram
// drafter drafts from the target's top-m cache of prefill and a context n-gram index).
//
// One CTA per request in every kernel: a tree holds at most 1024 nodes and a step adds
// W * m children, so the work is latency-bound except the n-gram scan, which reads the
// request's history once (L * 4 bytes) and compares each position with the W keys.
#include "gt_internal.cuh"
#include "launch.cuh"
#include "prune_select.cuh"

namespace gt {

constexpr int DRAFT_MAX_W = 64;    // frontier nodes per step
constexpr int DRAFT_MAX_M = 32;    // children per frontier node
constexpr int DRAFT_MAX_Q = 8;     // longest n-gram key
constexpr int NGRAM_THREADS = 512;

// ------------------------------------------------------------------------------------
// Frontier: the top-W nodes of the pool by (score desc, index asc), NaN last. Pool: nodes
// [pool_lo[b], n) when pool_lo is given, else the nodes with visited[b][v] == 0, after
// which every node v < n is marked visited. Thread v holds node v.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
frontier_kernel(const float *__restrict__ score, const int32_t *__restrict__ n_nodes, int Nmax,
                const int32_t *__restrict__ pool_lo, uint8_t *__restrict__ visited, int W,
                int32_t *__restrict__ frontier, int32_t *__restrict__ n_frontier, int32_t *err) {
  pdl_enter();
  __shared__ int s_hist[256], s_sel[3], warp_tot[32];
  __shared__ uint32_t s_key[DRAFT_MAX_W];
  __shared__ int s_idx[DRAFT_MAX_W];
  const int b = blockIdx.x, v = threadIdx.x;
  const size_t row0 = (size_t)b * Nmax;
  const int n = n_nodes[b];
  const bool ok = n >= 1 && n <= Nmax;
  if (!ok && v == 0) set_err(err, GT_ERR_RANGE);
  bool in_pool = false;
  if (ok && v < n) in_pool = pool_lo ? v >= pool_lo[b] : visited[row0 + v] == 0;
  const uint32_t key = in_pool ? order_key(score[row0 + v]) : 0u;
  const bool keep = topk_keys_keep(key, W, s_hist, s_sel, warp_tot);
  int cnt;
  const int slot = block_excl_count(keep, warp_tot, &cnt);
  if (keep) {
    s_key[slot] = key;
    s_idx[slot] = v;
  }
  __syncthreads();
  if (keep) {  // place in frontier order: larger key first, then smaller index
    int r = 0;
    for (int s = 0; s < cnt; ++s)
      r += s_key[s] > key || (s_key[s] == key && s_idx[s] < v);
    frontier[(size_t)b * W + r] = v;
  }
  for (int w = cnt + v; w < W; w += blockDim.x) frontier[(size_t)b * W + w] = -1;
  if (v == 0) n_frontier[b] = cnt;
  if (ok && !pool_lo && v < n) visited[row0 + v] = 1;
}

// ------------------------------------------------------------------------------------
// n-gram drafter. Key of frontier node f: the tokens of the root-to-f path preceded by
// the history, read backwards (key[0] = token(f)), at most q_max long. Position i of the
// history matches to length ell(i) = the number of leading key tokens equal to
// H[i], H[i-1], ...; the drafter takes the largest ell, then the largest i (the longest
// key with a match, at its most recent position), and copies the top-m cache row i.
// The scan is split over a grid of (history chunk, request) CTAs: each compares its
// positions with every key's first token, walks back only on a hit, and merges its best
// (ell << 32 | i) per key into the caller's match array with one global atomic max.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(NGRAM_THREADS)
ngram_scan_kernel(const int32_t *__restrict__ hist, const int32_t *__restrict__ hist_len, int Lh,
                  int chunk, const int32_t *__restrict__ parent,
                  const int32_t *__restrict__ tokens, const int32_t *__restrict__ n_nodes,
                  int Nmax, const int32_t *__restrict__ frontier,
                  const int32_t *__restrict__ n_frontier, int W, int q_max,
                  unsigned long long *__restrict__ best_out, int32_t *err) {
  pdl_enter();
  __shared__ int s_key[DRAFT_MAX_W][DRAFT_MAX_Q];
  __shared__ int s_klen[DRAFT_MAX_W];
  __shared__ unsigned long long s_best[DRAFT_MAX_W];
  const int b = blockIdx.y, tid = threadIdx.x;
  const bool report = blockIdx.x == 0;  // one CTA per request reports data errors
  const size_t row0 = (size_t)b * Nmax;
  const int32_t *H = hist + (size_t)b * Lh;
  const int n = n_nodes[b], L = hist_len[b], nf = n_frontier[b];
  const bool ok = n >= 1 && n <= Nmax && L >= 0 && L <= Lh && nf >= 0 && nf <= W;
  if (!ok && tid == 0 && report) set_err(err, GT_ERR_RANGE);
  const int nk = ok ? nf : 0;
  const int i0 = blockIdx.x * chunk, i1 = min(L, i0 + chunk);
  if (i0 >= i1 && !report) return;  // no positions of this request in this chunk
  if (tid < nk) {
    int t = 0;
    const int f = frontier[(size_t)b * W + tid];
    if (f < 0 || f >= n) {
      if (report) set_err(err, GT_ERR_RANGE);
    } else {
      // the path from f up to the root (at most q_max steps; parents precede children)
      for (int u = f; u != -1 && t < q_max; ++t) {
        s_key[tid][t] = tokens[row0 + u];
        const int p = parent[row0 + u];
        if (p >= u || p < -1) {
          if (report) set_err(err, GT_ERR_TREE);
          t = 0;
          break;
        }
        u = p;
      }
      if (t > 0)  // then the history, newest first
        for (int h = L - 1; t < q_max && h >= 0; --h) s_key[tid][t++] = H[h];
    }
    s_klen[tid] = t;
    s_best[tid] = 0ull;
  }
  __syncthreads();
  for (int i = i0 + tid; i < i1; i += NGRAM_THREADS) {
    const int h0 = H[i];
    for (int w = 0; w < nk; ++w) {
      if (s_klen[w] == 0 || h0 != s_key[w][0]) continue;
      int ell = 1;
      while (ell < s_klen[w] && ell <= i && H[i - ell] == s_key[w][ell]) ++ell;
      atomicMax(&s_best[w], ((unsigned long long)ell << 32) | (unsigned)i);
    }
  }
  __syncthreads();
  if (tid < nk && s_best[tid] != 0ull) atomicMax(&best_out[(size_t)b * W + tid], s_best[tid]);
}

// The children: row `pos` of the top-m cache for every key with a match; the match array
// becomes (position, length), position -1 without a match.
__global__ void __launch_bounds__(256)
ngram_children_kernel(int Lh, const int32_t *__restrict__ cache_id,
                      const float *__restrict__ cache_p, int m,
                      const int32_t *__restrict__ n_frontier, int W,
                      int32_t *__restrict__ child_id, float *__restrict__ child_p,
                      int32_t *__restrict__ match) {
  pdl_enter();
  const int b = blockIdx.x;
  const int nf = n_frontier[b];
  const int nk = (nf >= 0 && nf <= W) ? nf : 0;
  const unsigned long long *best = reinterpret_cast<const unsigned long long *>(match);
  for (int e = threadIdx.x; e < W * m; e += blockDim.x) {
    const int w = e / m, c = e - w * m;
    const unsigned long long bw = w < nk ? best[(size_t)b * W + w] : 0ull;
    const int ell = (int)(bw >> 32), pos = (int)(bw & 0xFFFFFFFFull);
    const size_t src = ((size_t)b * Lh + pos) * m + c;
    child_id[(size_t)b * W * m + e] = ell ? cache_id[src] : -1;
    child_p[(size_t)b * W * m + e] = ell ? cache_p[src] : 0.0f;
  }
  __syncthreads();  // every read of the packed bests is done before they are rewritten
  for (int w = threadIdx.x; w < W; w += blockDim.x) {
    const unsigned long long bw = w < nk ? best[(size_t)b * W + w] : 0ull;
    const int ell = (int)(bw >> 32);
    match[((size_t)b * W + w) * 2] = ell ? (int)(bw & 0xFFFFFFFFull) : -1;
    match[((size_t)b * W + w) * 2 + 1] = ell;
  }
}

// ------------------------------------------------------------------------------------
// Non-destructive attach. Thread e = w * m + c holds child c of frontier node w; the
// valid children (id >= 0) take the slots n, n+1, ... in (w, c) order up to Nmax, with
// score fl(score(f) * p). Existing nodes are only read.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
attach_kernel(int32_t *__restrict__ parent, int32_t *__restrict__ tokens, float *__restrict__ score,
              int32_t *__restrict__ n_nodes, int Nmax, const int32_t *__restrict__ frontier,
              const int32_t *__restrict__ n_frontier, int W, const int32_t *__restrict__ child_id,
              const float *__restrict__ child_p, int m, int V, int32_t *__restrict__ first_new,
              int32_t *err) {
  pdl_enter();
  __shared__ int warp_tot[32];
  const int b = blockIdx.x, e = threadIdx.x;
  const size_t row0 = (size_t)b * Nmax;
  const int n = n_nodes[b], nf = n_frontier[b];
  int code = (n < 1 || n > Nmax || nf < 0 || nf > W) ? GT_ERR_RANGE : 0;
  int f = -1, id = -1;
  float p = 0.0f;
  if (!code && e < nf * m) {
    const int w = e / m;
    f = frontier[(size_t)b * W + w];
    id = child_id[(size_t)b * W * m + e];
    p = child_p[(size_t)b * W * m + e];
    if (f < 0 || f >= n) code = GT_ERR_RANGE;
    else if (id < -1 || id >= V) code = GT_ERR_TREE;
  }
  if (__syncthreads_or(code)) {  // this request keeps its tree
    if (code) set_err(err, code);
    if (e == 0 && n >= 1 && n <= Nmax) first_new[b] = n;
    return;
  }
  const bool valid = id >= 0;
  int total;
  const int slot = block_excl_count(valid, warp_tot, &total);
  const int dst = n + slot;
  if (valid && dst < Nmax) {
    parent[row0 + dst] = f;
    tokens[row0 + dst] = id;
    score[row0 + dst] = __fmul_rn(score[row0 + f], p);
  }
  const int n_new = min(Nmax, n + total);
  for (int j = n_new + e; j < Nmax; j += blockDim.x) {
    parent[row0 + j] = tokens[row0 + j] = -1;
    score[row0 + j] = 0.0f;
  }
  if (e == 0) {
    n_nodes[b] = n_new;
    first_new[b] = n;
  }
}

}  // namespace gt

using namespace gt;

GT_API int gt_frontier_select(const float *score, const int32_t *n_nodes, int B, int Nmax,
                              const int32_t *pool_lo, uint8_t *visited, int W, int32_t *frontier,
                              int32_t *n_frontier, int32_t *err, gt_stream_t stream) {
  GT_TRACE("gt_frontier_select");
  if (B < 0 || Nmax < 1 || W < 1) return GT_ERR_ARG;
  if (Nmax > 1024 || W > DRAFT_MAX_W) return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (!score || !n_nodes || !frontier || !n_frontier || (!pool_lo == !visited)) return GT_ERR_ARG;
  return launch(frontier_kernel, dim3(B), dim3((Nmax + 31) / 32 * 32), 0, (cudaStream_t)stream,
                score, n_nodes, Nmax, pool_lo, visited, W, frontier, n_frontier, err);
}

GT_API int gt_ngram_draft(const int32_t *hist, const int32_t *hist_len, int B, int Lh,
                          const int32_t *cache_id, const float *cache_p, int m,
                          const int32_t *parent, const int32_t *tokens, const int32_t *n_nodes,
                          int Nmax, const int32_t *frontier, const int32_t *n_frontier, int W,
                          int q_max, int32_t *child_id, float *child_p, int32_t *match,
                          int32_t *err, gt_stream_t stream) {
  GT_TRACE("gt_ngram_draft");
  if (B < 0 || Lh < 0 || m < 1 || Nmax < 1 || W < 1 || q_max < 1) return GT_ERR_ARG;
  if (Nmax > 1024 || W > DRAFT_MAX_W || m > DRAFT_MAX_M || q_max > DRAFT_MAX_Q || B > 65535)
    return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (!hist_len || !parent || !tokens || !n_nodes || !frontier || !n_frontier || !child_id ||
      !child_p || !match || ((uintptr_t)match & 7) ||
      (Lh > 0 && (!hist || !cache_id || !cache_p)))
    return GT_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  // the match array holds each key's packed best (length << 32 | position) during the scan
  cudaError_t e = cudaMemsetAsync(match, 0, sizeof(int32_t) * 2 * (size_t)B * W, s);
  if (e != cudaSuccess) return launch_status(e, "cudaMemsetAsync(match)");
  // history chunks per request: enough CTAs for about two per SM, each at least 1024
  // positions long
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    sms = 148;
  }
  const int want = max(1, (2 * sms + B - 1) / B);
  const int C = max(1, min(want, (Lh + 1023) / 1024));
  const int chunk = max(1, (Lh + C - 1) / C);
  int rc = launch(ngram_scan_kernel, dim3(C, B), dim3(NGRAM_THREADS), 0, s, hist, hist_len, Lh,
                  chunk, parent, tokens, n_nodes, Nmax, frontier, n_frontier, W, q_max,
                  reinterpret_cast<unsigned long long *>(match), err);
  if (rc != GT_OK) return rc;
  return launch(ngram_children_kernel, dim3(B), dim3(256), 0, s, Lh, cache_id, cache_p, m,
                n_frontier, W, child_id, child_p, match);
}

GT_API int gt_tree_attach(int32_t *parent, int32_t *tokens, float *score, int32_t *n_nodes,
                          int B, int Nmax, const int32_t *frontier, const int32_t *n_frontier,
                          int W, const int32_t *child_id, const float *child_p, int m, int V,
                          int32_t *first_new, int32_t *err, gt_stream_t stream) {
  GT_TRACE("gt_tree_attach");
  if (B < 0 || Nmax < 1 || W < 1 || m < 1 || V < 1) return GT_ERR_ARG;
  if (Nmax > 1024 || W > DRAFT_MAX_W || m > DRAFT_MAX_M || W * m > 1024) return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (!parent || !tokens || !score || !n_nodes || !frontier || !n_frontier || !child_id ||
      !child_p || !first_new)
    return GT_ERR_ARG;
  return launch(attach_kernel, dim3(B), dim3((W * m + 31) / 32 * 32), 0, (cudaStream_t)stream,
                parent, tokens, score, n_nodes, Nmax, frontier, n_frontier, W, child_id, child_p,
                m, V, first_new, err);
}
