"""Pins of the drafting oracle (oracle/drafting.py): a hand-worked example, a library
selection routine, an independently written tree generator and a brute-force longest
match."""
import heapq
import math

import numpy as np

from conftest import golden
from oracle.drafting import frontier_select, ngram_children, tree_attach
from workload.synth import _edge_probs, _top_children, treegraft_tree


def _cache(L, m):
    ids = np.array([[100 * (c + 1) + i for c in range(m)] for i in range(L)], np.int32)
    p = np.tile(np.float32([0.5, 0.25, 0.125, 0.0625][:m]), (L, 1))
    return ids, p


def test_hand_example_children_and_attach():
    g = golden("ngram_small.json")
    H, m = g["hist"], g["m"]
    ids, p = _cache(len(H), m)
    for f, want in g["expect_children"].items():
        got_ids, got_p, pos, q = ngram_children(H, len(H), ids, p, g["parent"], g["tokens"],
                                                int(f), g["q_max"], m)
        assert (pos, q) == (want["pos"], want["q"]) and got_ids.tolist() == want["ids"]
    a = g["attach"]
    kids = [ngram_children(H, len(H), ids, p, g["parent"], g["tokens"], f, g["q_max"], m)
            for f in a["frontier"]]
    par, tok, sc, n, first = tree_attach(g["parent"], g["tokens"], np.float32(g["score"]), 5,
                                         a["Nmax"], a["frontier"], [k[0] for k in kids],
                                         [k[1] for k in kids])
    assert par == a["parent"] and tok == a["tokens"] and (n, first) == (a["n"], a["first_new"])
    assert np.array_equal(sc, np.float32(a["score"]))


def test_frontier_matches_library_selection():
    rng = np.random.default_rng(0)
    for _ in range(200):
        n = int(rng.integers(1, 80))
        score = np.float32(rng.choice([0.5, 0.25, 0.125, 0.1], size=n))  # many ties
        W = int(rng.integers(1, 12))
        lo = int(rng.integers(0, n))
        front, _ = frontier_select(score, n, W, pool_lo=lo)
        assert front == heapq.nsmallest(W, range(lo, n), key=lambda v: (-score[v], v))
        vis = rng.integers(0, 2, size=100).tolist()
        front, nv = frontier_select(score, n, W, visited=vis)
        pool = [v for v in range(n) if not vis[v]]
        assert front == heapq.nsmallest(W, pool, key=lambda v: (-score[v], v))
        assert nv[:n] == [1] * n and nv[n:] == vis[n:]


def _better(score, u: int, v: int) -> bool:
    """The frontier's order rule written out case by case: a number beats NaN; between two
    numbers the larger wins (+0.0 and -0.0 are equal numbers) and a tie goes to the smaller
    index; between two NaN the smaller index wins."""
    a, b = float(np.float32(score[u])), float(np.float32(score[v]))
    a_nan, b_nan = math.isnan(a), math.isnan(b)
    if a_nan != b_nan:
        return b_nan
    if not a_nan and a != b:
        return a > b
    return u < v


def _brute_frontier(score, pool, W):
    """Frontier by counting, for each pool node, the pool nodes that beat it (its rank);
    the nodes of rank < W, listed by rank."""
    rank = {v: sum(_better(score, u, v) for u in pool if u != v) for v in pool}
    return sorted((v for v in pool if rank[v] < W), key=lambda v: rank[v])


def test_frontier_order_with_nan_signed_zeros_and_infinities():
    """Hand example of the rule: +inf, 1.0, the two 0.5 by index, -0.0 and +0.0 by index
    (equal numbers), then the NaN by index."""
    nan, inf = float("nan"), float("inf")
    score = np.float32([1.0, nan, 0.5, -0.0, 0.0, nan, inf, 0.5, -inf])
    assert frontier_select(score, 9, 5, pool_lo=0)[0] == [6, 0, 2, 7, 3]
    assert frontier_select(score, 9, 9, pool_lo=0)[0] == [6, 0, 2, 7, 3, 4, 8, 1, 5]
    assert frontier_select(score, 9, 3, pool_lo=4)[0] == [6, 7, 4]
    vis = [1, 0, 1, 0, 0, 1, 1, 0, 0]
    assert frontier_select(score, 9, 4, visited=vis)[0] == [7, 3, 4, 8]


def test_frontier_matches_pairwise_brute_force_on_special_values():
    rng = np.random.default_rng(7)
    specials = np.float32([float("nan"), -float("nan"), 0.0, -0.0, float("inf"),
                           -float("inf"), 0.5, 0.5, 1e-30, -1e-30])
    for _ in range(300):
        n = int(rng.integers(1, 40))
        score = np.where(rng.random(n) < 0.6, rng.choice(specials, size=n),
                         np.float32(rng.integers(-3, 4, size=n) / 4)).astype(np.float32)
        W = int(rng.integers(1, 12))
        lo = int(rng.integers(0, n))
        assert frontier_select(score, n, W, pool_lo=lo)[0] == \
            _brute_frontier(score, list(range(lo, n)), W)
        vis = rng.integers(0, 2, size=n).tolist()
        assert frontier_select(score, n, W, visited=vis)[0] == \
            _brute_frontier(score, [v for v in range(n) if not vis[v]], W)


def test_replays_the_two_drafter_tree_generator():
    """frontier_select + tree_attach with the generator's own drafter draws rebuild the
    tree that workload.treegraft_tree grows (written separately, as an input generator)."""
    V, D, W, m, n_max, schedule = 3000, 5, 10, 10, 256, (1, 0, 1, 0, 1)
    for seed in range(3):
        ss = np.random.SeedSequence(seed).spawn(2)
        want = treegraft_tree(np.random.Generator(np.random.PCG64(ss[0])),
                              np.random.Generator(np.random.PCG64(ss[1])), V, D, W, m,
                              schedule, n_max)
        rs = np.random.Generator(np.random.PCG64(ss[0]))
        rm = np.random.Generator(np.random.PCG64(ss[1]))
        parent, tokens, score = [-1], [int(rs.integers(V))], np.float32([1.0])
        n, first_new, visited = 1, 0, [0] * n_max
        for k in range(D):
            if n >= n_max:
                break
            mid = bool(schedule[k])
            if mid:
                front, visited = frontier_select(score, n, W, visited=visited)
            else:
                front, _ = frontier_select(score, n, W, pool_lo=first_new)
            cid, cp = [], []
            for f in front:
                p = _edge_probs(rm if mid else rs, V)
                top = _top_children(p, m)
                cid.append(top.astype(np.int32))
                cp.append(p[top])
            parent, tokens, score, n2, first_new = tree_attach(parent, tokens, score, n, n_max,
                                                               front, cid, cp)
            n = n2
        assert n == len(want[0])
        assert parent[:n] == want[0].tolist() and tokens[:n] == want[1].tolist()
        assert np.array_equal(score[:n], want[2])


def test_children_equal_longest_then_latest_match_by_brute_force():
    rng = np.random.default_rng(7)
    for trial in range(60):
        L = int(rng.integers(1, 60))
        H = rng.integers(0, 4, size=L).tolist()  # small alphabet: many repeats
        ids, p = _cache(L, 3)
        n = int(rng.integers(1, 9))
        parent = [-1] + [int(rng.integers(0, v)) for v in range(1, n)]
        tokens = rng.integers(0, 4, size=n).tolist()
        q_max = int(rng.integers(1, 5))
        for f in range(n):
            path = []
            u = f
            while u != -1:
                path.append(tokens[u])
                u = parent[u]
            seq = H + path[::-1]
            best = (0, -1)  # (matched length, position): longest first, then latest
            for i in range(L):
                ell = 0
                while (ell < q_max and ell <= i and ell < len(seq)
                       and H[i - ell] == seq[len(seq) - 1 - ell]):
                    ell += 1
                if ell > 0 and (ell, i) > best:
                    best = (ell, i)
            got_ids, _, pos, q = ngram_children(H, L, ids, p, parent, tokens, f, q_max, 3)
            assert (q, pos) == (best[0], best[1] if best[0] else -1)
            if pos >= 0:
                assert got_ids.tolist() == ids[pos].tolist()
            else:
                assert got_ids.tolist() == [-1, -1, -1]


def test_attach_keeps_existing_nodes_and_respects_capacity():
    rng = np.random.default_rng(9)
    for _ in range(100):
        n = int(rng.integers(1, 30))
        Nmax = n + int(rng.integers(0, 40))
        parent = [-1] + [int(rng.integers(0, v)) for v in range(1, n)]
        tokens = rng.integers(0, 50, size=n).tolist()
        score = np.float32(rng.random(n))
        W = int(rng.integers(0, 6))
        front = rng.choice(n, size=min(W, n), replace=False).tolist()
        cid = rng.integers(-1, 50, size=(len(front), 4)).astype(np.int32)
        cp = np.float32(rng.random((len(front), 4)))
        par, tok, sc, n2, first = tree_attach(parent, tokens, score, n, Nmax, front, cid, cp)
        assert first == n and par[:n] == parent and tok[:n] == tokens
        assert np.array_equal(sc[:n], score)
        assert n2 == min(Nmax, n + int((cid >= 0).sum()))
        for v in range(n, n2):
            assert 0 <= par[v] < n and np.float32(sc[v]) <= score[par[v]]
        assert all(x == -1 for x in par[n2:]) and all(x == -1 for x in tok[n2:])
