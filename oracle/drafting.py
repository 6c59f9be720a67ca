"""CPU oracle of the drafting side of a tree step: frontier selection, the n-gram drafter
and the non-destructive attach (test infrastructure).

Like the rest of ``oracle/``, this module is slow on purpose, shares no code with the CUDA
path and is imported only by the tests, the package smoke check and the benchmark's CPU
leg.

Sources (page title, then section):
  [TreeGraft] "TreeGraft 精读：多起草器共嫁接一棵草稿树，让投机解码跨越快与好的单选题",
              §一 (a training-free n-gram small drafter and a pre-trained mid drafter grow
              one shared tree), §三 (each step picks the top-W frontier from a candidate
              pool by the cumulative path score s(v), the product of edge scores, and hangs
              the top-m children of every frontier node), §四 Where (the mid drafter's pool
              is every tree node it has not visited yet, and the pool joins the visited set
              after its step; the small drafter's pool is the newest nodes), §四 How (new
              children are attached without overwriting any existing node), §七 item 6 (the
              n-gram drafter drafts from the target's top-m cache produced at prefill and a
              context n-gram index).

Readings where the pages are silent:
  * Frontier: the top-W pool nodes by (score desc, index asc; NaN last, as in the prune).
    The small drafter's pool is
    the nodes added by the previous step, [first_new, n); the mid drafter's pool is every
    node not yet visited, and afterwards every node of the tree counts as visited.
  * Attach: children are appended after the existing nodes, frontier by frontier in
    frontier order and within a frontier node in child order; a child's score is
    fl(s(f) * p) in float32; an empty child (id -1) is skipped; growth stops at the
    capacity Nmax. Existing nodes never change; duplicate siblings are kept.
  * n-gram drafter: the history H[0..L) holds the committed tokens before the tree root;
    the key of frontier node f is the last q tokens of H followed by the tokens of the
    root-to-f path. The index finds the most recent position i (largest i, q-1 <= i < L)
    with H[i-q+1..i] equal to the key, trying q = q_max first and backing off to q = 1.
    The children are the top-m cache entry of that position: the target's m most likely
    tokens for position i+1 and their probabilities, as produced at prefill (cache row i).
    No match at any q: no children.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .step import OracleError


def frontier_select(score, n: int, W: int, pool_lo: Optional[int] = None,
                    visited: Optional[Sequence[int]] = None):
    """Top-W frontier of one request ([TreeGraft] §三, §四 Where).

    Exactly one of ``pool_lo`` (small drafter: pool = nodes pool_lo .. n-1) and ``visited``
    (mid drafter: pool = nodes with visited[v] == 0) is given. Returns (frontier list,
    new visited list or None); with ``visited`` every node v < n is visited afterwards.
    """
    if (pool_lo is None) == (visited is None):
        raise OracleError("give exactly one of pool_lo and visited")
    if pool_lo is not None:
        pool = list(range(max(0, int(pool_lo)), n))
    else:
        pool = [v for v in range(n) if not visited[v]]
    def key(v):  # score descending, NaN last, +0.0 equal to -0.0, then index ascending
        x = float(np.float32(score[v]))
        return (x != x, 0.0 if x != x else -x, v)

    order = sorted(pool, key=key)
    front = order[:W]
    new_visited = None
    if visited is not None:
        new_visited = [1 if v < n else int(visited[v]) for v in range(len(visited))]
    return front, new_visited


def _path_tokens(parent, tokens, f: int):
    path = []
    u = f
    while u != -1:
        path.append(int(tokens[u]))
        u = int(parent[u])
    path.reverse()
    return path


def ngram_children(hist: Sequence[int], L: int, cache_id, cache_p, parent, tokens, f: int,
                   q_max: int, m: int):
    """Children of frontier node f proposed by the n-gram drafter ([TreeGraft] §一, §七).

    Returns (ids [m], probs [m], matched position i or -1, matched order q or 0); ids are -1
    past the end of the cache entry or when nothing matches.
    """
    seq = [int(t) for t in hist[:L]] + _path_tokens(parent, tokens, f)
    ids = np.full(m, -1, np.int32)
    probs = np.zeros(m, np.float32)
    for q in range(q_max, 0, -1):
        if q > len(seq):
            continue
        key = seq[len(seq) - q:]
        for i in range(L - 1, q - 2, -1):  # most recent first
            if [int(t) for t in hist[i - q + 1:i + 1]] == key:
                ids[:] = np.asarray(cache_id[i][:m], np.int32)
                probs[:] = np.asarray(cache_p[i][:m], np.float32)
                return ids, probs, i, q
    return ids, probs, -1, 0


def tree_attach(parent, tokens, score, n: int, Nmax: int, frontier, child_id, child_p):
    """Non-destructive attach ([TreeGraft] §四 How): the children of every frontier node
    are appended after the existing nodes; existing nodes never change.

    Returns new (parent, tokens, score) lists of length Nmax (-1 / -1 / 0 padded), the new
    node count, and the first new index (the previous n).
    """
    par = [int(x) for x in parent[:Nmax]] + [-1] * max(0, Nmax - len(parent))
    tok = [int(x) for x in tokens[:Nmax]] + [-1] * max(0, Nmax - len(tokens))
    sc = [np.float32(x) for x in score[:Nmax]] + [np.float32(0)] * max(0, Nmax - len(score))
    nn = n
    for w, f in enumerate(frontier):
        for c in range(len(child_id[w])):
            cid = int(child_id[w][c])
            if cid < 0 or nn >= Nmax:
                continue
            par[nn], tok[nn] = int(f), cid
            sc[nn] = np.float32(np.float32(score[f]) * np.float32(child_p[w][c]))
            nn += 1
    for v in range(nn, Nmax):
        par[v], tok[v], sc[v] = -1, -1, np.float32(0)
    return par, tok, np.asarray(sc, np.float32), nn, n
