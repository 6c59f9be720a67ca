"""Plain CPU oracle of the verify-and-graft step of tree speculative decoding.

Test infrastructure. It is slow on purpose and follows the pages' definitions step by
step, in numpy and pure Python, in float64 wherever there is arithmetic. It shares no
code with the CUDA path and never imports it.

Sources (page title, then section):
  [Graft]     "浙江大学、阿里巴巴联手破解AI推理瓶颈" (write-up of the Graft paper),
              §二 (the three gears: calibrated pruning, retrieval graft from the GPU
              successor table with a stage-adaptive template and the 8/24/40 + 52/36/20
              split of 60 slots, flatten + tree positions + mask + one parallel verify,
              online table update from every verified position), §三 (monotonicity of
              tree verification, the grafted tree is a superset of the pruned tree),
              §四 (batched serving keeps a fixed slot count per request and swaps
              low-confidence draft nodes for retrieved ones), §六 (online update uses
              accepted and rejected positions alike).
  [TreeGraft] "TreeGraft 精读：多起草器共嫁接一棵草稿树，让投机解码跨越快与好的单选题",
              §一 (accept the correct tokens, roll back from the first error),
              §三 (cumulative path score = product of edge scores; global prune to the
              verification budget Bver; tree-attention verification), §四 How
              (non-destructive graft, then one global prune to Bver = 63), §五 (temperature
              0, D=5, W=10, m=10, Bver=63).

Readings where the pages are silent:
  * node 0 is the root (the current token); it counts among the N verified slots;
  * prune keeps the root plus the best nodes by (score desc, index asc); scores must
    not increase from parent to child (products of probabilities), otherwise the
    input is rejected;
  * the retrieved tree is rooted at the tree root; template node t has a template
    parent (-1 = root) and a successor rank; an empty table entry (-1) drops the node
    and its template descendants; survivors are appended in template order;
  * the table row of every verified node's token is replaced by the target's top-k
    ids at that node; when several nodes share a token the last one in (request,
    node) order wins;
  * top-k order is (value desc, index asc), +0.0 equals -0.0, NaN ranks below -inf;
  * the accepted node is the deepest accepted node, ties to the smaller index.

Parity pins live in tests/ (brute force, closed forms, library routines, invariants).
"""
from __future__ import annotations

import heapq
import math
from typing import Optional, Sequence

import numpy as np


class OracleError(ValueError):
    """Invalid input to the oracle."""


class TreeError(OracleError):
    """Parent array is not a rooted tree in topological order, or an id is out of range."""


class NonMonotoneError(OracleError):
    """A node's cumulative score exceeds its parent's (or is NaN)."""


# --------------------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------------------


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bits (uint16) -> float64: the bf16 value is the top half of an fp32."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def _check_tree(parent: Sequence[int], n: int) -> None:
    """Root at index 0, every other node's parent has a smaller index."""
    if n < 1:
        raise TreeError("a tree has at least its root")
    if int(parent[0]) != -1:
        raise TreeError("parent[0] must be -1 (node 0 is the root)")
    for v in range(1, n):
        p = int(parent[v])
        if not 0 <= p < v:
            raise TreeError(f"parent[{v}]={p} is not in [0,{v})")


def _children(parent: Sequence[int], n: int):
    ch = [[] for _ in range(n)]
    for v in range(1, n):
        ch[int(parent[v])].append(v)
    return ch


def stage_budget(stage: Optional[int], slots: int = 60):
    """Draft / retrieved slot split per prune stage ([Graft] §二): a prune triggered at
    depth 0, 1 or 5 keeps 8, 24 or 40 draft nodes and refills 52, 36 or 20 slots from
    the table; with no prune every slot stays with the drafter."""
    table = {0: (8, 52), 1: (24, 36), 5: (40, 20)}
    if stage is None:
        return slots, 0
    if stage not in table:
        raise OracleError("prune stages are 0, 1 and 5")
    return table[stage]


# --------------------------------------------------------------------------------------
# a1: prune to the verification budget
# --------------------------------------------------------------------------------------


def prune_topB(score, parent, tokens, n_in: int, keep: int, thresh: Optional[float] = None):
    """Keep the root and the best nodes by cumulative score ([TreeGraft] §三, §四 How;
    [Graft] §四 for the threshold form used by static batched trees).

    Best-first expansion: start from the root, repeatedly take the frontier node with the
    largest score (smaller index first on ties) and add its children to the frontier,
    until ``keep`` nodes are held or (with ``thresh``) the best frontier score is below
    the threshold. Kept nodes are renumbered in ascending old index.

    Returns (parent, tokens, score, old_idx) lists of the kept tree.
    """
    _check_tree(parent, n_in)
    for v in range(1, n_in):
        p = int(parent[v])
        ps = math.inf if p == 0 else float(score[p])
        if not float(score[v]) <= ps:
            raise NonMonotoneError(f"score[{v}] > score[parent] or NaN")
    keep = min(int(keep), n_in)
    if keep < 1:
        raise OracleError("keep must be >= 1 (the root is always kept)")
    ch = _children(parent, n_in)
    kept = {0}
    heap = [(-float(score[c]), c) for c in ch[0]]
    heapq.heapify(heap)
    while len(kept) < keep and heap:
        neg, v = heapq.heappop(heap)
        if thresh is not None and -neg < float(thresh):
            break
        kept.add(v)
        for c in ch[v]:
            heapq.heappush(heap, (-float(score[c]), c))
    old = sorted(kept)
    new_of = {o: i for i, o in enumerate(old)}
    out_parent = [-1 if o == 0 else new_of[int(parent[o])] for o in old]
    out_tokens = [int(tokens[o]) for o in old]
    out_score = [np.float32(score[o]) for o in old]
    return out_parent, out_tokens, out_score, old


# --------------------------------------------------------------------------------------
# a2: graft retrieved nodes into the freed slots
# --------------------------------------------------------------------------------------


def graft_expand(parent, tokens, n_kept: int, tpar, trank, R: int, table, Nmax: int,
                 anchor: int = 0):
    """Refill freed slots from the successor table ([Graft] §二, second gear; §七 for the
    tail graft of block drafts, Graft-TAIL).

    The retrieved tree hangs from the anchor node: the tree root (the current token) by
    default; for Graft-TAIL the last kept node of the pruned draft chain (anchor = -1
    means node n_kept - 1). Template node t
    (t = 0 .. R'-1 with R' = min(R, Nmax - n_kept, T)) has template parent tpar[t]
    (-1 = the anchor) and successor rank trank[t]; its token is row ``token(parent)`` of the
    table at column ``trank[t]``. An empty entry (-1) drops the node, and with it every
    template descendant. Survivors are appended after the kept nodes in template order.

    Returns (parent, tokens, n) of length Nmax, padded with -1.
    """
    V, k = np.asarray(table).shape
    T = len(tpar)
    out_p = [int(x) for x in parent[:n_kept]]
    out_t = [int(x) for x in tokens[:n_kept]]
    for t in out_t:
        if not 0 <= t < V:
            raise TreeError("token out of range")
    a = n_kept - 1 if int(anchor) == -1 else int(anchor)
    if not 0 <= a < n_kept:
        raise OracleError("graft anchor outside the kept tree")
    r = max(0, min(int(R), Nmax - n_kept, T))
    node_of = {}
    for t in range(r):
        tp, rank = int(tpar[t]), int(trank[t])
        if not -1 <= tp < t or not 0 <= rank < k:
            raise TreeError("template parent must precede its child; rank < k")
        if tp == -1:
            pnode = a
        elif tp in node_of:
            pnode = node_of[tp]
        else:
            continue  # template parent was dropped
        tok = int(table[out_t[pnode]][rank])
        if tok == -1:
            continue
        if not 0 <= tok < V:
            raise TreeError("table entry out of range")
        node_of[t] = len(out_p)
        out_p.append(pnode)
        out_t.append(tok)
    n = len(out_p)
    out_p += [-1] * (Nmax - n)
    out_t += [-1] * (Nmax - n)
    return out_p, out_t, n


# --------------------------------------------------------------------------------------
# a3: ancestor mask and tree position ids
# --------------------------------------------------------------------------------------


def tree_mask(parent, n: int, prefix_len: int, N: int):
    """Flattened-tree mask and positions ([Graft] §二, third gear).

    For each node i, walk parent pointers from i to the root and set bit j of row i for
    every node j visited (i itself included). depth = number of steps to the root;
    position id = prefix_len + depth. Rows >= n are 0 (mask) and -1 (depth, position).
    Returns (depth[N], pos[N], mask[N][ceil(N/64)] uint64).
    """
    _check_tree(parent, n)
    W = (N + 63) // 64
    mask = np.zeros((N, W), dtype=np.uint64)
    depth = np.full(N, -1, dtype=np.int64)
    pos = np.full(N, -1, dtype=np.int64)
    for i in range(n):
        j, d = i, 0
        while True:
            mask[i, j // 64] |= np.uint64(1) << np.uint64(j % 64)
            if j == 0:
                break
            j = int(parent[j])
            d += 1
        depth[i] = d
        pos[i] = prefix_len + d
    return depth, pos, mask


def _is_ancestor_or_self(parent, j: int, i: int) -> bool:
    while True:
        if i == j:
            return True
        if i == 0:
            return False
        i = int(parent[i])


# --------------------------------------------------------------------------------------
# a4: tree attention
# --------------------------------------------------------------------------------------


def tree_attn(Q, K, Vv, parent, n: int, prefix_len: int, scale: float):
    """Tree-masked GQA attention of one request, in float64 ([Graft] §二 third gear;
    [TreeGraft] §三 tree-attention verification).

    Q: [N][Hq][d]; K, Vv: [Hkv][Lcap][d] (float arrays, already decoded). Query node i,
    head h attends the prefix keys 0..prefix_len-1 and the tree keys prefix_len + u for
    every tree node u that is an ancestor of i or i itself (explicit parent walk), with
    KV head h // (Hq/Hkv). Softmax of scale * q.k with the row max subtracted.
    Returns O [n][Hq][d] float64.
    """
    _check_tree(parent, n)
    Hq, d = Q.shape[1], Q.shape[2]
    Hkv = K.shape[0]
    if Hq % Hkv:
        raise OracleError("Hq must be a multiple of Hkv")
    g = Hq // Hkv
    P = int(prefix_len)
    L = P + n
    allowed = np.ones((n, L), dtype=bool)
    for i in range(n):
        for u in range(n):
            allowed[i, P + u] = _is_ancestor_or_self(parent, u, i)
    O = np.zeros((n, Hq, d), dtype=np.float64)
    for h in range(Hq):
        kvh = h // g
        keys = np.asarray(K[kvh, :L], dtype=np.float64)
        vals = np.asarray(Vv[kvh, :L], dtype=np.float64)
        q = np.asarray(Q[:n, h], dtype=np.float64)
        s = (q @ keys.T) * float(scale)
        s = np.where(allowed, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        O[:, h] = (e @ vals) / e.sum(axis=1, keepdims=True)
    return O


# --------------------------------------------------------------------------------------
# a5: vocab-wide top-k (argmax = entry 0)
# --------------------------------------------------------------------------------------


def vocab_topk(row, k: int):
    """The k largest logits of one row by full sort ([Graft] §二: table rows hold the
    target's k most likely next tokens; [TreeGraft] §五: greedy, temperature 0).

    Order: non-NaN before NaN, then value descending (+0.0 equals -0.0), then index
    ascending. Returns (ids int32[k], values float32[k]).
    """
    v = np.asarray(row, dtype=np.float32)
    isn = np.isnan(v)
    val = np.where(isn, 0.0, v.astype(np.float64))
    order = np.lexsort((np.arange(v.size), -val, isn))
    top = order[:k]
    return top.astype(np.int32), v[top]


# --------------------------------------------------------------------------------------
# a6: longest accepted path and commit indices
# --------------------------------------------------------------------------------------


def verify_greedy(tokens, parent, n: int, argmax, prefix_len: int):
    """Greedy tree verification of one request ([Graft] §二 third gear; [TreeGraft] §一, §三).

    A node is accepted when every edge on its root path carries the token the target
    predicts at the edge's upper end (tokens[c] == argmax[parent[c]]). Recursive DFS from
    the root explores accepted children in index order and keeps the deepest node (ties:
    smaller index). The committed tokens are the path's draft tokens plus the target's
    token at the last accepted node (the bonus); the accepted nodes' KV rows move from
    prefix_len + path[j] to prefix_len + j.

    Returns dict(acc_len, path, out_tok, kv_src, kv_dst) (lists).
    """
    _check_tree(parent, n)
    ch = _children(parent, n)
    best = [0, 0]  # depth, node

    def dfs(u: int, d: int) -> None:
        if d > best[0] or (d == best[0] and u < best[1]):
            best[0], best[1] = d, u
        for c in ch[u]:
            if int(tokens[c]) == int(argmax[u]):
                dfs(c, d + 1)

    dfs(0, 0)
    path = []
    u = best[1]
    while True:
        path.append(u)
        if u == 0:
            break
        u = int(parent[u])
    path.reverse()
    L = len(path) - 1
    out_tok = [int(tokens[path[j]]) for j in range(1, L + 1)] + [int(argmax[path[-1]])]
    P = int(prefix_len)
    return dict(acc_len=L, path=path, out_tok=out_tok,
                kv_src=[P + p for p in path], kv_dst=[P + j for j in range(L + 1)])


# --------------------------------------------------------------------------------------
# a7: successor-table update
# --------------------------------------------------------------------------------------


def succ_update(table, tokens, topk_id, n_nodes):
    """Online table update ([Graft] §二 third gear, §六 second level).

    For request b = 0..B-1 and node v = 0..n_b-1 in that order (accepted or rejected),
    row tokens[b][v] of the table becomes the target's top-k ids at (b, v). A later
    write to the same row replaces an earlier one. Returns the updated copy.
    """
    t = np.array(table, dtype=np.int32, copy=True)
    V, k = t.shape
    for b in range(len(n_nodes)):
        for v in range(int(n_nodes[b])):
            tok = int(tokens[b][v])
            if not 0 <= tok < V:
                raise TreeError("token out of range")
            t[tok, :] = np.asarray(topk_id[b][v][:k], dtype=np.int32)
    return t


# --------------------------------------------------------------------------------------
# KV commit: compaction of the accepted path's cache rows
# --------------------------------------------------------------------------------------


def kv_commit(K, Vc, kv_src, kv_dst, acc_len):
    """Move the accepted path's K/V rows to the committed positions ([TreeGraft] §一: keep
    the agreeing prefix, drop the rest; [Graft] §二 third gear: the verified tokens join the
    context).

    For every request b and j = 0..acc_len[b], row kv_dst[b][j] of every KV head ends up
    holding what row kv_src[b][j] held before the commit; no other row changes. Written as
    its definition: every source row is read from the unchanged cache, then written.
    K, Vc: [B][Hkv][Lcap][d]; kv_src, kv_dst: [B][>= acc_len + 1]. Returns new copies.
    """
    K = np.array(K, copy=True)
    Vc = np.array(Vc, copy=True)
    B, _, Lcap, _ = K.shape
    K0, V0 = K.copy(), Vc.copy()
    for b in range(B):
        L = int(acc_len[b])
        if L < 0 or L + 1 > len(kv_src[b]):
            raise OracleError("accepted length outside the path buffer")
        src = [int(x) for x in kv_src[b][:L + 1]]
        dst = [int(x) for x in kv_dst[b][:L + 1]]
        if any(not 0 <= x < Lcap for x in src + dst):
            raise OracleError("cache row outside the cache")
        for j in range(L + 1):
            K[b, :, dst[j]] = K0[b, :, src[j]]
            Vc[b, :, dst[j]] = V0[b, :, src[j]]
    return K, Vc


# --------------------------------------------------------------------------------------
# whole step
# --------------------------------------------------------------------------------------


def step_tree_phase(parent_in, tokens_in, score_in, n_in, keep, thresh, tpar, trank, R, table,
                    prefix_len, N: int, anchor=None):
    """a1 + a2 + a3 for every request: prune, graft (at anchor[b], default the root),
    mask. Returns a dict of arrays."""
    B = len(keep)
    W = (N + 63) // 64
    out = dict(parent=np.full((B, N), -1, np.int32), tokens=np.full((B, N), -1, np.int32),
               n_kept=np.zeros(B, np.int32), n_nodes=np.zeros(B, np.int32),
               old_idx=np.full((B, N), -1, np.int32), score=np.zeros((B, N), np.float32),
               depth=np.full((B, N), -1, np.int64), pos=np.full((B, N), -1, np.int64),
               mask=np.zeros((B, N, W), np.uint64))
    for b in range(B):
        th = None if thresh is None else float(thresh[b])
        p, t, s, o = prune_topB(score_in[b], parent_in[b], tokens_in[b], int(n_in[b]),
                                int(keep[b]), th)
        nk = len(p)
        if nk > N:
            raise OracleError("kept tree exceeds the slot count")
        out["n_kept"][b] = nk
        out["old_idx"][b, :nk] = o
        out["score"][b, :nk] = s
        gp, gt, n = graft_expand(p, t, nk, tpar, trank, int(R[b]), table, N,
                                 0 if anchor is None else int(anchor[b]))
        out["parent"][b], out["tokens"][b], out["n_nodes"][b] = gp, gt, n
        d, ps, m = tree_mask(gp, n, int(prefix_len[b]), N)
        out["depth"][b], out["pos"][b], out["mask"][b] = d, ps, m
    return out


def step_verify_phase(tree, logits, table, prefix_len, k: int, rows=None):
    """a5 + a6 + a7 given the final trees and the target logits [B][N][V]."""
    B, N, V = logits.shape
    topk_id = np.full((B, N, k), -1, np.int32)
    topk_val = np.zeros((B, N, k), np.float32)
    for b in range(B):
        for v in range(N):
            topk_id[b, v], topk_val[b, v] = vocab_topk(logits[b, v], k)
    res = dict(topk_id=topk_id, topk_val=topk_val, acc_len=np.zeros(B, np.int32),
               path=np.full((B, N), -1, np.int32), out_tok=np.full((B, N + 1), -1, np.int32),
               kv_src=np.full((B, N), -1, np.int32), kv_dst=np.full((B, N), -1, np.int32))
    for b in range(B):
        n = int(tree["n_nodes"][b])
        r = verify_greedy(tree["tokens"][b], tree["parent"][b], n, topk_id[b, :, 0],
                          int(prefix_len[b]))
        L = r["acc_len"]
        res["acc_len"][b] = L
        res["path"][b, :L + 1] = r["path"]
        res["out_tok"][b, :L + 1] = r["out_tok"]
        res["kv_src"][b, :L + 1] = r["kv_src"]
        res["kv_dst"][b, :L + 1] = r["kv_dst"]
    res["table"] = succ_update(table, tree["tokens"], topk_id, tree["n_nodes"])
    return res
