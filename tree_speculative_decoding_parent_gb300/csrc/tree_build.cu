// a1 + a2 + a3 fused: prune, graft and mask of one request in one CTA.
//
// The same computation as gt_prune_topB (with Nout = N) -> gt_graft_expand (Nmax = N) ->
// gt_tree_mask, with identical outputs and error codes, but the tree stays in shared
// memory between the three phases: one launch and one round trip to global memory for the
// inputs instead of three launches and a chain of dependent reads and writes.
//
// Sources: "TreeGraft 精读：多起草器共嫁接一棵草稿树，让投机解码跨越快与好的单选题" §三, §四 How
// (cumulative path score, global prune to Bver); "浙江大学、阿里巴巴联手破解AI推理瓶颈" §二
// (successor-table retrieval by a template into the freed slots; flatten, tree position ids
// and mask) and §四 (static slot count per request in batched serving).
#include <limits.h>
#include <math.h>

#include "gt_internal.cuh"
#include "prune_select.cuh"
#include "launch.cuh"

namespace gt {

__global__ void __launch_bounds__(1024, 1)
tree_build_kernel(const float *__restrict__ score, const int32_t *__restrict__ parent_in,
                  const int32_t *__restrict__ tokens_in, const int32_t *__restrict__ n_in,
                  int Nin, const int32_t *__restrict__ keep, const float *__restrict__ thresh,
                  const int32_t *__restrict__ tpar, const int32_t *__restrict__ trank, int T,
                  const int32_t *__restrict__ R, const int32_t *__restrict__ anchor,
                  const int32_t *__restrict__ table, int V, int k,
                  const int32_t *__restrict__ prefix_len, int N, int W,
                  int32_t *__restrict__ parent, int32_t *__restrict__ tokens,
                  float *__restrict__ out_score, int32_t *__restrict__ out_old,
                  int32_t *__restrict__ n_nodes, int32_t *__restrict__ depth,
                  int32_t *__restrict__ pos, uint64_t *__restrict__ mask, int32_t *err,
                  int gw) {
  pdl_enter();
  extern __shared__ int s_dyn[];
  const int Nin4 = (Nin + 3) & ~3;
  float *s_score = reinterpret_cast<float *>(s_dyn);  // [Nin4]
  int *s_new = s_dyn + Nin4;                          // [Nin]
  int *s_par = s_new + Nin;                           // [N] tree being built
  int *s_tok = s_par + N;                             // [N]
  const int Tb = T > 0 ? T : 1;
  int *s_tpar = s_tok + N;                            // [Tb]
  int *s_ttok = s_tpar + Tb;                          // [Tb]
  int *s_tnew = s_ttok + Tb;                          // [Tb]
  int *s_tflag = s_tnew + Tb;                         // [Tb] graft warp: bad template / entry
  int *s_tdep = s_tflag + Tb;                         // [Tb] graft warp: template depth
  __shared__ int warp_tot[32];
  __shared__ int s_hist[256], s_sel[3];
  __shared__ int s_bad, s_maxd, s_n;
  __shared__ int s_gtot, s_fbad, s_grmax;  // graft warp: retrieved count, first bad template node
  const int b = blockIdx.x, t = threadIdx.x;
  // gw: the block's last warp retrieves the graft (one dependent table read per template
  // level) while the others prune; the prune then synchronises only its own np threads
  const int np = gw ? (int)blockDim.x - 32 : 0;
  const bool graft_warp = gw && t >= np;
  const size_t in0 = (size_t)b * Nin, row0 = (size_t)b * N;
  const int n = n_in ? n_in[b] : Nin;
  const int kb = keep[b];
  const int P = prefix_len[b];
  if (t == 0) {
    s_bad = 0;
    s_maxd = 0;
  }

  // ---------------------------------------------------------------- phase A: prune
  int code = (n < 1 || n > Nin) ? GT_ERR_RANGE : 0;
  int p = -1, tok = -1;
  float s = 0.f;
  int nk = 0;
  // every global read of the prune and of the graft set-up is issued here, before the
  // first barrier, so that none of them waits for a phase before it
  const float th = thresh ? thresh[b] : -INFINITY;
  const int anchor_b = anchor ? anchor[b] : 0;
  const int R_b = R[b];
  const int tpar_t = t < T ? tpar[t] : -1;
  const int trank_t = t < T ? trank[t] : 0;
  if (graft_warp) {
    // --------------------------------------------- concurrent graft retrieval (one warp)
    // Template nodes t' < min(R, T, N - nk) fit, nk the kept count. Without a threshold
    // the prune keeps exactly min(keep, n) nodes (every non-root node competes: a NaN
    // score fails the monotonicity check); with one, at least the root. Every node up to
    // that bound is retrieved now, and only the nodes that fit count (errors included).
    const int lane = t - np;
    const int nk_min = thresh ? 1 : max(1, min(kb, n));
    const int rmax = max(0, min(min(R_b, T), N - nk_min));
    const int rt = tokens_in[in0];  // the root's token: the graft hangs from the root
    const int rtok = (rt >= 0 && rt < V) ? rt : -1;
    // a retrieved entry outside [-1, V) is bad: flagged (reported after the prune if the node
    // fits) and retrieved as -1
    auto publish = [&](int u, int tk) {
      if (tk < -1 || tk >= V) {
        s_tflag[u] |= 2;
        tk = -1;
      }
      s_ttok[u] = tk;
    };
    constexpr int GPL = 2;  // template nodes per lane held in registers (rmax <= 64)
    if (rmax <= 32 * GPL) {
      // lane holds nodes u = lane + 32 j; every read of a level leaves at once, and level 1
      // (children of the root, which need only the root's row) as soon as the template
      // entries are in, before the depths are known
      int tpv[GPL], rkv[GPL], tkv[GPL], dv[GPL];
#pragma unroll
      for (int j = 0; j < GPL; ++j) {
        const int u = lane + 32 * j;
        tpv[j] = u < rmax ? tpar[u] : -1;
        rkv[j] = u < rmax ? trank[u] : 0;
      }
#pragma unroll
      for (int j = 0; j < GPL; ++j) {
        const int u = lane + 32 * j;
        tkv[j] = -1;
        if (u < rmax) {
          const int tp = tpv[j], rk = rkv[j];
          const bool badt = tp < -1 || tp >= u || rk < 0 || rk >= k;
          s_tpar[u] = tp;
          s_tflag[u] = badt ? 1 : 0;
          if (!badt && tp == -1 && rtok >= 0) tkv[j] = table[(size_t)rtok * k + rk];
        }
      }
#pragma unroll
      for (int j = 0; j < GPL; ++j) {
        const int u = lane + 32 * j;
        if (u < rmax) publish(u, tkv[j]);
      }
      __syncwarp();
      // parents precede children, so a chain of valid nodes ends at the root; a node with a
      // bad entry on its chain is never retrieved
      int maxd = 0;
#pragma unroll
      for (int j = 0; j < GPL; ++j) {
        const int u = lane + 32 * j;
        int d = 0;
        if (u < rmax)
          for (int v = u; v != -1; v = s_tpar[v]) {
            if (s_tflag[v] & 1) {
              d = 0;
              break;
            }
            ++d;
          }
        dv[j] = d;
        maxd = max(maxd, d);
      }
      maxd = (int)__reduce_max_sync(0xffffffffu, (unsigned)maxd);
      for (int L = 2; L <= maxd; ++L) {
        bool at[GPL];
#pragma unroll
        for (int j = 0; j < GPL; ++j) {
          at[j] = dv[j] == L;
          tkv[j] = -1;
          if (at[j]) {
            const int ptok = s_ttok[tpv[j]];
            if (ptok >= 0) tkv[j] = table[(size_t)ptok * k + rkv[j]];
          }
        }
#pragma unroll
        for (int j = 0; j < GPL; ++j)
          if (at[j]) publish(lane + 32 * j, tkv[j]);
        __syncwarp();
      }
    } else {
      for (int u = lane; u < rmax; u += 32) {
        const int tp = tpar[u], rk = trank[u];
        s_tpar[u] = tp;
        s_tnew[u] = rk;  // the rank, until the placement reuses the array
        s_tflag[u] = (tp < -1 || tp >= u || rk < 0 || rk >= k) ? 1 : 0;
        s_ttok[u] = -1;
      }
      __syncwarp();
      int maxd = 0;
      for (int u = lane; u < rmax; u += 32) {
        int d = 0;
        for (int v = u; v != -1; v = s_tpar[v]) {
          if (s_tflag[v] & 1) {
            d = 0;
            break;
          }
          ++d;
        }
        s_tdep[u] = d;
        maxd = max(maxd, d);
      }
      maxd = (int)__reduce_max_sync(0xffffffffu, (unsigned)maxd);
      __syncwarp();
      for (int L = 1; L <= maxd; ++L) {
        for (int u = lane; u < rmax; u += 32) {
          if (s_tdep[u] != L) continue;
          const int tp = s_tpar[u];
          const int ptok = tp == -1 ? rtok : s_ttok[tp];
          publish(u, ptok >= 0 ? table[(size_t)ptok * k + s_tnew[u]] : -1);
        }
        __syncwarp();
      }
    }
    // for the placement after the join: the exclusive prefix counts of the retrieved nodes
    // (s_tnew, no longer the ranks), their total, and the first node with a bad template
    // entry; the fitting count r <= rmax, so prefixes up to r are the ones the join needs
    int base = 0, fb = INT_MAX;
    for (int u0 = 0; u0 < rmax; u0 += 32) {
      const int u = u0 + lane;
      const bool got = u < rmax && s_ttok[u] >= 0;
      const unsigned ba = __ballot_sync(0xffffffffu, got);
      const unsigned bb = __ballot_sync(0xffffffffu, u < rmax && (s_tflag[u] & 1));
      if (u < rmax) s_tnew[u] = base + __popc(ba & ((1u << lane) - 1u));
      base += __popc(ba);
      if (bb && fb == INT_MAX) fb = u0 + __ffs(bb) - 1;
    }
    if (lane == 0) {
      s_gtot = base;
      s_fbad = fb;
      s_grmax = rmax;
    }
  } else {
  if (!code && t < n) {
    p = parent_in[in0 + t];
    s = score[in0 + t];
    tok = tokens_in[in0 + t];
    s_score[t] = s;
  }
  sync_threads_n(np);
  if (!code && t < n) {
    if (t == 0) {
      if (p != -1) code = GT_ERR_TREE;
    } else if (p < 0 || p >= t) {
      code = GT_ERR_TREE;
    } else {
      const float ps = (p == 0) ? INFINITY : s_score[p];
      if (!(s <= ps)) code = GT_ERR_NONMONOTONE;
    }
  }
  const int ke = min(kb, n);
  if (!code && (kb < 1 || ke > N)) code = GT_ERR_RANGE;
  if (code) atomicCAS(&s_bad, 0, code);
  sync_threads_n(np);
  if (!s_bad) {
  // the root is always kept; the other nodes compete for the remaining ke - 1 slots
  const bool cand = t > 0 && t < n && s >= th;
  const bool sel = topk_keys_keep(cand ? order_key(s) : 0u, ke - 1, s_hist, s_sel, warp_tot,
                                  np);
  const bool kept = (t == 0) || sel;
  const int newi = block_excl_count(kept, warp_tot, &nk, np);
  if (t < n) s_new[t] = kept ? newi : -1;
  sync_threads_n(np);
  if (kept) {
    s_par[newi] = (t == 0) ? -1 : s_new[p];
    s_tok[newi] = tok;
    if (out_score) out_score[row0 + newi] = s;
    if (out_old) out_old[row0 + newi] = t;
  }
  for (int j = nk + t; j < N; j += (gw ? np : (int)blockDim.x)) {
    if (out_score) out_score[row0 + j] = 0.f;
    if (out_old) out_old[row0 + j] = -1;
  }
  if (gw && t == 0) s_n = nk;  // for the graft warp, which did not count the kept nodes
  }
  }
  // the prune's tree and (gw) the retrieved tokens are complete for every thread here
  __syncthreads();
  if (gw) nk = s_n;
  const int bad = s_bad;
  if (bad) {  // as the separate calls: nothing kept, every row padded
    if (t == 0) {
      set_err(err, bad);
      n_nodes[b] = 0;
    }
    for (int j = t; j < N; j += blockDim.x) {
      parent[row0 + j] = tokens[row0 + j] = -1;
      if (out_score) out_score[row0 + j] = 0.f;
      if (out_old) out_old[row0 + j] = -1;
      depth[row0 + j] = pos[row0 + j] = -1;
      for (int w = 0; w < W; ++w) mask[(row0 + j) * W + w] = 0ull;
    }
    return;
  }

  // ---------------------------------------------------------------- phase B: graft
  int nf_gw = 0;  // graft warp mode: the final count, the same in every thread
  if (gw) {
    // The graft warp retrieved, flagged and counted every template node that can fit; the
    // r = min(R, N - nk, T) that do fit hang from the root. A bad root token, or a bad
    // template entry among them, keeps the pruned tree alone (as the separate calls do);
    // otherwise a bad table entry among them is reported. Every thread decides alike.
    const int root_tok = s_tok[0];
    const int r = max(0, min(min(R_b, N - nk), T));
    int n_final = nk;
    if (root_tok < 0 || root_tok >= V || s_fbad < r) {
      if (t == 0) set_err(err, GT_ERR_TREE);
    } else {
      if (t < r && (s_tflag[t] & 2)) set_err(err, GT_ERR_TREE);
      if (t < r && s_ttok[t] >= 0) {
        const int gi = s_tnew[t];
        s_par[nk + gi] = (tpar_t == -1) ? 0 : nk + s_tnew[tpar_t];
        s_tok[nk + gi] = s_ttok[t];
      }
      n_final = nk + (r < s_grmax ? s_tnew[r] : s_gtot);
    }
    // kept in a register: a slower thread may still be reading the kept count from s_n
    nf_gw = n_final;
  } else {
  // the retrieved tree hangs from the anchor: the root, or (Graft-TAIL) the last kept node
  int a = 0;
  code = 0;
  if (anchor) {
    a = anchor_b == -1 ? nk - 1 : anchor_b;
    if (a < 0 || a >= nk) {
      code = GT_ERR_RANGE;
      a = 0;
    }
  }
  const int root_tok = s_tok[a];
  if (!code && (root_tok < 0 || root_tok >= V)) code = GT_ERR_TREE;
  const int r = code ? 0 : max(0, min(min(R_b, N - nk), T));
  const bool active = t < r;
  int tp = -1, rk = 0;
  if (active) {
    tp = tpar_t;
    rk = trank_t;
    if (tp < -1 || tp >= t || rk < 0 || rk >= k) code = GT_ERR_TREE;
    s_tpar[t] = tp;
  }
  if (code) atomicCAS(&s_bad, 0, code);
  __syncthreads();
  int n_final = nk;
  if (s_bad) {  // the kept tree stays; no graft
    if (t == 0) set_err(err, s_bad);
  } else {
    int dep = 0;
    if (active) {
      for (int u = t; u != -1; u = s_tpar[u]) ++dep;
      atomicMax(&s_maxd, dep);
    }
    __syncthreads();
    const int maxd = s_maxd;
    for (int L = 1; L <= maxd; ++L) {
      if (active && dep == L) {
        const int ptok = (tp == -1) ? root_tok : s_ttok[tp];
        int tok = -1;
        if (ptok >= 0) {
          tok = table[(size_t)ptok * k + rk];
          if (tok < -1 || tok >= V) {
            set_err(err, GT_ERR_TREE);
            tok = -1;
          }
        }
        s_ttok[t] = tok;
      }
      __syncthreads();
    }
  }
  if (!s_bad) {
    const bool alive = active && s_ttok[t] >= 0;
    int cnt;
    const int gi = block_excl_count(alive, warp_tot, &cnt);
    if (active) s_tnew[t] = gi;
    __syncthreads();
    if (alive) {
      s_par[nk + gi] = (tp == -1) ? a : nk + s_tnew[tp];
      s_tok[nk + gi] = s_ttok[t];
    }
    n_final = nk + cnt;
  }
  if (t == 0) s_n = n_final;
  }
  __syncthreads();

  // ---------------------------------------------------------------- phase C: mask
  const int nf = gw ? nf_gw : s_n;
  for (int v = t; v < N; v += blockDim.x) {
    const size_t o = row0 + v;
    uint64_t *mrow = mask + o * W;
    if (v >= nf) {
      parent[o] = tokens[o] = -1;
      depth[o] = pos[o] = -1;
      for (int w = 0; w < W; ++w) mrow[w] = 0ull;
      continue;
    }
    parent[o] = s_par[v];
    tokens[o] = s_tok[v];
    int d = 0, cur = v >> 6;
    uint64_t word = 0ull;
    for (int w = W - 1; w > cur; --w) mrow[w] = 0ull;
    for (int u = v;; u = s_par[u]) {
      const int wu = u >> 6;
      while (wu < cur) {
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
    depth[o] = d;
    pos[o] = P + d;
  }
  if (t == 0) n_nodes[b] = nf;
}

}  // namespace gt

using namespace gt;

GT_API int gt_tree_build(const float *score, const int32_t *parent_in, const int32_t *tokens_in,
                         const int32_t *n_in, int B, int Nin, const int32_t *keep,
                         const float *thresh, const int32_t *tpar, const int32_t *trank, int T,
                         const int32_t *R, const int32_t *anchor, const int32_t *table, int V,
                         int k,
                         const int32_t *prefix_len, int N, int32_t *parent, int32_t *tokens,
                         float *out_score, int32_t *out_old_idx, int32_t *n_nodes,
                         int32_t *depth, int32_t *pos, uint64_t *mask, int32_t *err,
                         gt_stream_t stream) {
  GT_TRACE("gt_tree_build");
  if (B < 0 || Nin < 1 || N < 1 || T < 0 || V < 1 || k < 1) return GT_ERR_ARG;
  if (Nin > 1024 || N > 1024 || T > 1024) return GT_ERR_SHAPE;
  if (B == 0) return GT_OK;
  if (!score || !parent_in || !tokens_in || !keep || !R || !table || !prefix_len || !parent ||
      !tokens || !n_nodes || !depth || !pos || !mask || (T > 0 && (!tpar || !trank)))
    return GT_ERR_ARG;
  const int W = (N + 63) / 64;
  const int Tb = T > 0 ? T : 1;
  int threads = (max(max(Nin, N), Tb) + 31) / 32 * 32;
  // a graft hung from the root does not depend on the prune: one more warp retrieves it
  // meanwhile (a Graft-TAIL anchor is only known once the prune is done)
  const int gw = (T > 0 && !anchor && threads + 32 <= 1024) ? 1 : 0;
  threads += 32 * gw;
  const size_t smem = sizeof(int) * ((size_t)((Nin + 3) & ~3) + Nin + 2 * (size_t)N + 5 * (size_t)Tb);
  return launch(tree_build_kernel, dim3(B), dim3(threads), smem, (cudaStream_t)stream, score,
                parent_in, tokens_in, n_in, Nin, keep, thresh, tpar, trank, T, R, anchor, table, V, k,
                prefix_len, N, W, parent, tokens, out_score, out_old_idx, n_nodes, depth, pos,
                mask, err, gw);
}
