// a1 prune, a2 graft, a3 mask: the small per-request tree kernels.
//
// One CTA per request, one thread per node (or template node). These steps move a few
// KB per request and are latency-bound; the kernels keep every dependent access in
// shared memory and finish in a handful of barriers.
//
// Sources: "TreeGraft 精读：多起草器共嫁接一棵草稿树，让投机解码跨越快与好的单选题" §三 and
// §四 How (cumulative path score, global prune to Bver); "浙江大学、阿里巴巴联手破解AI推理瓶颈"
// §二 (successor-table retrieval by a template into the freed slots; flatten, tree
// position ids and mask) and §四 (static per-request slot count in batched serving).
#include <math.h>

#include "gt_internal.cuh"
#include "prune_select.cuh"
#include "launch.cuh"

namespace gt {

// ------------------------------------------------------------------------------------
// a1: prune. Rank of non-root node v = number of eligible nodes better than v in the
// order (score desc, index asc); keep v iff rank < keep-1 (the root takes one slot). The
// kept set is found without ranking every node: topk_keys_keep selects it in O(n).
// With scores non-increasing from parent to child (checked), the kept set is
// ancestor-closed, so a prefix count over kept flags renumbers it in index order.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
prune_kernel(const float *__restrict__ score, const int32_t *__restrict__ parent,
             const int32_t *__restrict__ tokens, const int32_t *__restrict__ n_in, int Nin,
             const int32_t *__restrict__ keep, const float *__restrict__ thresh, int Nout,
             int32_t *__restrict__ out_parent, int32_t *__restrict__ out_tokens,
             float *__restrict__ out_score, int32_t *__restrict__ out_old,
             int32_t *__restrict__ n_out, int32_t *err) {
  pdl_enter();
  extern __shared__ float s_score[];           // [Nin4] scores, then s_new [Nin]
  const int Nin4 = (Nin + 3) & ~3;
  int *s_new = reinterpret_cast<int *>(s_score + Nin4);  // [Nin]
  __shared__ int warp_tot[32];
  __shared__ int s_hist[256], s_sel[3];
  __shared__ int s_bad;
  const int b = blockIdx.x, v = threadIdx.x;
  const size_t in0 = (size_t)b * Nin, out0 = (size_t)b * Nout;
  const int n = n_in ? n_in[b] : Nin;
  const int kb = keep[b];
  if (v == 0) s_bad = 0;
  int code = (n < 1 || n > Nin) ? GT_ERR_RANGE : 0;
  int p = -1;
  float s = 0.f;
  if (!code && v < n) {
    p = parent[in0 + v];
    s = score[in0 + v];
    s_score[v] = s;
  }
  __syncthreads();
  if (!code && v < n) {
    if (v == 0) {
      if (p != -1) code = GT_ERR_TREE;
    } else if (p < 0 || p >= v) {
      code = GT_ERR_TREE;
    } else {
      const float ps = (p == 0) ? INFINITY : s_score[p];
      if (!(s <= ps)) code = GT_ERR_NONMONOTONE;
    }
  }
  const int ke = min(kb, n);
  if (!code && (kb < 1 || ke > Nout)) code = GT_ERR_RANGE;
  if (code) atomicCAS(&s_bad, 0, code);
  __syncthreads();
  const int bad = s_bad;
  if (bad) {
    if (v == 0) {
      set_err(err, bad);
      n_out[b] = 0;
    }
    for (int j = v; j < Nout; j += blockDim.x) {
      out_parent[out0 + j] = -1;
      out_tokens[out0 + j] = -1;
      if (out_score) out_score[out0 + j] = 0.f;
      if (out_old) out_old[out0 + j] = -1;
    }
    return;
  }
  const float th = thresh ? thresh[b] : -INFINITY;
  // the root is always kept; the other nodes compete for the remaining ke - 1 slots
  const bool cand = v > 0 && v < n && s >= th;
  const bool sel = topk_keys_keep(cand ? order_key(s) : 0u, ke - 1, s_hist, s_sel, warp_tot);
  const bool kept = (v == 0) || sel;
  int total;
  const int newi = block_excl_count(kept, warp_tot, &total);
  if (v < n) s_new[v] = kept ? newi : -1;
  __syncthreads();
  if (kept) {
    const size_t o = out0 + newi;
    out_parent[o] = (v == 0) ? -1 : s_new[p];
    out_tokens[o] = tokens[in0 + v];
    if (out_score) out_score[o] = s;
    if (out_old) out_old[o] = v;
  }
  for (int j = total + v; j < Nout; j += blockDim.x) {
    out_parent[out0 + j] = -1;
    out_tokens[out0 + j] = -1;
    if (out_score) out_score[out0 + j] = 0.f;
    if (out_old) out_old[out0 + j] = -1;
  }
  if (v == 0) n_out[b] = total;
}

// ------------------------------------------------------------------------------------
// a2: graft. Template nodes are resolved level by level (a node's token needs its
// template parent's token), then survivors are compacted by a prefix count. The retrieved
// tree hangs from the anchor node: the root, or (Graft-TAIL) the last kept node.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
graft_kernel(int32_t *__restrict__ parent, int32_t *__restrict__ tokens,
             int32_t *__restrict__ n_nodes, int Nmax, const int32_t *__restrict__ tpar,
             const int32_t *__restrict__ trank, int T, const int32_t *__restrict__ R,
             const int32_t *__restrict__ anchor, const int32_t *__restrict__ table, int V,
             int k, int32_t *err) {
  pdl_enter();
  extern __shared__ int s_i32[];
  int *s_par = s_i32;           // [T]
  int *s_tok = s_i32 + T;       // [T]
  int *s_new = s_i32 + 2 * T;   // [T]
  __shared__ int warp_tot[32];
  __shared__ int s_bad, s_maxd;
  const int b = blockIdx.x, t = threadIdx.x;
  const size_t row0 = (size_t)b * Nmax;
  const int n = n_nodes[b];
  if (t == 0) {
    s_bad = 0;
    s_maxd = 0;
  }
  int code = (n < 1 || n > Nmax) ? GT_ERR_RANGE : 0;
  int a = 0;  // anchor node of the retrieved tree
  if (!code && anchor) {
    a = anchor[b] == -1 ? n - 1 : anchor[b];
    if (a < 0 || a >= n) code = GT_ERR_RANGE;
  }
  const int root_tok = code ? -1 : tokens[row0 + a];
  if (!code && (root_tok < 0 || root_tok >= V)) code = GT_ERR_TREE;
  const int r = code ? 0 : max(0, min(min(R[b], Nmax - n), T));
  const bool active = t < r;
  int tp = -1, rk = 0;
  if (active) {
    tp = tpar[t];
    rk = trank[t];
    if (tp < -1 || tp >= t || rk < 0 || rk >= k) code = GT_ERR_TREE;
    s_par[t] = tp;
  }
  __syncthreads();
  if (code) atomicCAS(&s_bad, 0, code);
  __syncthreads();
  const int bad = s_bad;
  if (bad) {
    if (t == 0) set_err(err, bad);
    if (n >= 1 && n <= Nmax)  // kept tree stays valid: no graft, pad the free slots
      for (int j = n + t; j < Nmax; j += blockDim.x) parent[row0 + j] = tokens[row0 + j] = -1;
    return;
  }
  // every template parent precedes its child (checked above), so the walks end
  int dep = 0;
  if (active) {
    for (int u = t; u != -1; u = s_par[u]) ++dep;
    atomicMax(&s_maxd, dep);
  }
  __syncthreads();
  const int maxd = s_maxd;
  for (int L = 1; L <= maxd; ++L) {
    if (active && dep == L) {
      const int ptok = (tp == -1) ? root_tok : s_tok[tp];
      int tok = -1;
      if (ptok >= 0) {
        tok = table[(size_t)ptok * k + rk];
        if (tok < -1 || tok >= V) {
          set_err(err, GT_ERR_TREE);
          tok = -1;
        }
      }
      s_tok[t] = tok;
    }
    __syncthreads();
  }
  const bool alive = active && s_tok[t] >= 0;
  int cnt;
  const int newi = block_excl_count(alive, warp_tot, &cnt);
  if (active) s_new[t] = newi;
  __syncthreads();
  if (alive) {
    const size_t o = row0 + n + newi;
    parent[o] = (tp == -1) ? a : n + s_new[tp];
    tokens[o] = s_tok[t];
  }
  for (int j = n + cnt + t; j < Nmax; j += blockDim.x) parent[row0 + j] = tokens[row0 + j] = -1;
  if (t == 0) n_nodes[b] = n + cnt;
}

// ------------------------------------------------------------------------------------
// a3: mask + position ids. Thread v walks its own root path once (ancestors have
// decreasing indices, so mask words are visited from high to low and flushed in order).
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
mask_kernel(const int32_t *__restrict__ parent, const int32_t *__restrict__ n_nodes,
            const int32_t *__restrict__ prefix_len, int N, int W, int32_t *__restrict__ depth,
            int32_t *__restrict__ pos, uint64_t *__restrict__ mask, int32_t *err) {
  pdl_enter();
  extern __shared__ int s_par[];  // [N]
  __shared__ int s_bad;
  const int b = blockIdx.x, v = threadIdx.x;
  const size_t row0 = (size_t)b * N;
  const int n = n_nodes[b];
  const int P = prefix_len[b];
  if (v == 0) s_bad = 0;
  int code = (n < 1 || n > N) ? GT_ERR_RANGE : 0;
  if (!code && v < n) {
    const int p = parent[row0 + v];
    s_par[v] = p;
    if (v == 0 ? (p != -1) : (p < 0 || p >= v)) code = GT_ERR_TREE;
  }
  __syncthreads();
  if (code) atomicCAS(&s_bad, 0, code);
  __syncthreads();
  const int bad = s_bad;
  if (bad && v == 0) set_err(err, bad);
  if (v >= N) return;
  uint64_t *mrow = mask + (row0 + v) * W;
  if (bad || v >= n) {
    for (int w = 0; w < W; ++w) mrow[w] = 0ull;
    depth[row0 + v] = -1;
    pos[row0 + v] = -1;
    return;
  }
  int d = 0, cur = v >> 6;
  uint64_t word = 0ull;
  for (int w = W - 1; w > cur; --w) mrow[w] = 0ull;
  for (int u = v;; u = s_par[u]) {
    const int wu = u >> 6;
    while (wu < cur) {  // leaving word `cur`: flush it and zero-fill the gap
      mrow[cur] = word;
      word = 0ull;
      --cur;
    }
    word |= 1ull << (u & 63);
    if (u == 0) break;
    ++d;
  }
  mrow[cur] = word;
  for (int w = cur - 1; w >= 0; --w) mrow[w] = 0ull;
  depth[row0 + v] = d;
  pos[row0 + v] = P + d;
}

}  // namespace gt

using namespace gt;

static int round32(int x) { return (x + 31) / 32 * 32; }

GT_API int gt_prune_topB(const float *score, const int32_t *parent, const int32_t *tokens,
                         const int32_t *n_in, int B, int Nin, const int32_t *keep,
                         const float *thresh, int Nout, int32_t *out_parent,
                         int32_t *out_tokens, float *out_score, int32_t *out_old_idx,
                         int32_t *n_out, int32_t *err, gt_stream_t stream) {
  GT_TRACE("gt_prune_topB");
  if (B < 0 || Nin < 1 || Nout < 1) return GT_ERR_ARG;
  if (Nin > 1024) return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (!score || !parent || !tokens || !keep || !out_parent || !out_tokens || !n_out)
    return GT_ERR_ARG;
  const size_t smem = sizeof(int) * ((size_t)((Nin + 3) & ~3) + (size_t)Nin);
  return launch(prune_kernel, dim3(B), dim3(round32(Nin)), smem, (cudaStream_t)stream, score,
                parent, tokens, n_in, Nin, keep, thresh, Nout, out_parent, out_tokens,
                out_score, out_old_idx, n_out, err);
}

GT_API int gt_graft_expand(int32_t *parent, int32_t *tokens, int32_t *n_nodes, int B,
                           int Nmax, const int32_t *tpar, const int32_t *trank, int T,
                           const int32_t *R, const int32_t *anchor, const int32_t *table, int V,
                           int k, int32_t *err, gt_stream_t stream) {
  GT_TRACE("gt_graft_expand");
  if (B < 0 || Nmax < 1 || T < 0 || V < 1 || k < 1) return GT_ERR_ARG;
  if (T > 1024) return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (!parent || !tokens || !n_nodes || !R || !table || (T > 0 && (!tpar || !trank)))
    return GT_ERR_ARG;
  const int Tb = T > 0 ? T : 1;
  const size_t smem = 3 * sizeof(int) * (size_t)Tb;
  return launch(graft_kernel, dim3(B), dim3(round32(Tb)), smem, (cudaStream_t)stream, parent,
                tokens, n_nodes, Nmax, tpar, trank, T, R, anchor, table, V, k, err);
}

GT_API int gt_tree_mask(const int32_t *parent, const int32_t *n_nodes,
                        const int32_t *prefix_len, int B, int N, int32_t *depth, int32_t *pos,
                        uint64_t *mask, int32_t *err, gt_stream_t stream) {
  GT_TRACE("gt_tree_mask");
  if (B < 0 || N < 1) return GT_ERR_ARG;
  if (N > 1024) return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (!parent || !n_nodes || !prefix_len || !depth || !pos || !mask) return GT_ERR_ARG;
  const int W = (N + 63) / 64;
  return launch(mask_kernel, dim3(B), dim3(round32(N)), sizeof(int) * (size_t)N,
                (cudaStream_t)stream, parent, n_nodes, prefix_len, N, W, depth, pos, mask, err);
}
