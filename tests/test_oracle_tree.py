"""Pins for the oracle's tree steps: mask, prune, graft, walk, table update.

Every check compares the oracle with something other than itself: page-fixed numbers,
hand-worked fixtures, brute force over all small trees, or invariants the pages state.
"""
import itertools
import random

import numpy as np
import pytest

import oracle
from conftest import golden


def all_trees(n):
    """Every parent array of n nodes in topological order (parent[v] < v)."""
    for choice in itertools.product(*[range(v) for v in range(1, n)]):
        yield [-1] + list(choice)


def closure(parent):
    """Ancestor-or-self relation by boolean matrix closure (no parent walk)."""
    n = len(parent)
    A = np.zeros((n, n), dtype=bool)
    for i in range(1, n):
        A[i, parent[i]] = True
    R = np.eye(n, dtype=bool) | A
    while True:
        R2 = R | ((R.astype(np.int64) @ R.astype(np.int64)) > 0)
        if (R2 == R).all():
            return R
        R = R2


# ------------------------------------------------------------------------------- budgets


def test_stage_budget_matches_page():
    g = golden("budgets.json")
    for st, (d, r) in g["stages"].items():
        assert oracle.stage_budget(int(st), g["slots"]) == (d, r)
        assert d + r == g["slots"]
    assert oracle.stage_budget(None, g["slots"]) == tuple(g["no_prune"])
    with pytest.raises(oracle.OracleError):
        oracle.stage_budget(3)


# ---------------------------------------------------------------------------------- mask


def test_mask_hand_example():
    g = golden("hand_tree7.json")
    depth, pos, mask = oracle.tree_mask(g["parent"], 7, g["prefix_len"], 7)
    assert depth.tolist() == g["depth"]
    assert pos.tolist() == g["pos"]
    assert mask[:, 0].astype(np.int64).tolist() == g["mask"]


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7])
def test_mask_brute_force_all_trees(n):
    N = n + 2  # padded rows
    for parent in all_trees(n):
        depth, pos, mask = oracle.tree_mask(parent, n, 5, N)
        R = closure(parent)
        for i in range(n):
            bits = [(int(mask[i, 0]) >> j) & 1 for j in range(N)]
            assert bits[:n] == R[i].astype(int).tolist()
            assert not any(bits[n:])
            assert depth[i] == R[i].sum() - 1
            assert pos[i] == 5 + depth[i]
        assert (mask[n:] == 0).all() and (depth[n:] == -1).all() and (pos[n:] == -1).all()


def test_mask_chain_is_lower_triangular_and_star():
    n = 64
    chain = [-1] + list(range(n - 1))
    _, _, m = oracle.tree_mask(chain, n, 0, n)
    for i in range(n):
        assert int(m[i, 0]) == (1 << (i + 1)) - 1 if i < 63 else int(m[i, 0]) == (1 << 64) - 1
    star = [-1] + [0] * (n - 1)
    d, _, m = oracle.tree_mask(star, n, 0, n)
    assert all(int(m[i, 0]) == (1 | (1 << i)) for i in range(n))
    assert d.tolist() == [0] + [1] * (n - 1)


def test_mask_multiword():
    n = 130
    chain = [-1] + list(range(n - 1))
    _, _, m = oracle.tree_mask(chain, n, 0, n)
    assert m.shape == (130, 3)
    row = m[129]
    assert int(row[0]) == (1 << 64) - 1 and int(row[1]) == (1 << 64) - 1 and int(row[2]) == 3


def test_mask_rejects_bad_trees():
    with pytest.raises(oracle.TreeError):
        oracle.tree_mask([0, 0], 2, 0, 2)
    with pytest.raises(oracle.TreeError):
        oracle.tree_mask([-1, 1], 2, 0, 2)
    with pytest.raises(oracle.TreeError):
        oracle.tree_mask([-1, 0, 3, 0], 4, 0, 4)


# --------------------------------------------------------------------------------- prune


def test_prune_hand_example():
    g = golden("prune_small.json")
    for c in g["cases"]:
        p, t, s, o = oracle.prune_topB(np.float32(g["score"]), g["parent"], g["tokens"], 6,
                                       c["keep"], c.get("thresh"))
        assert o == c["old_idx"]
        assert p == c["parent"]
        assert t == [g["tokens"][i] for i in o]


def _dyadic_tree(rng, n):
    parent = [-1] + [rng.randrange(v) for v in range(1, n)]
    score = [1.0]
    for v in range(1, n):
        # child = parent * (j/8), exact in binary; ties are frequent on purpose
        score.append(score[parent[v]] * rng.choice([0.125, 0.25, 0.5, 0.75, 1.0]))
    return parent, np.float32(score)


def test_prune_brute_force_max_sum_closed_set():
    rng = random.Random(7)
    for _ in range(300):
        n = rng.randint(1, 8)
        parent, score = _dyadic_tree(rng, n)
        R = closure(parent)
        for keep in range(1, n + 1):
            _, _, _, got = oracle.prune_topB(score, parent, list(range(n)), n, keep)
            best, best_sets = -1.0, []
            for sub in itertools.combinations(range(1, n), keep - 1):
                s = (0,) + sub
                if not all(set(np.nonzero(R[v])[0]) <= set(s) for v in s):
                    continue
                tot = sum(float(score[v]) for v in s[1:])
                if tot > best:
                    best, best_sets = tot, [s]
                elif tot == best:
                    best_sets.append(s)
            assert tuple(got) in best_sets
            # among equal-sum sets, the (score desc, index asc) order decides
            order = sorted(range(1, n), key=lambda v: (-float(score[v]), v))
            assert set(got) == {0, *order[:keep - 1]}


def test_prune_threshold_is_filtered_topk():
    rng = random.Random(11)
    for _ in range(200):
        n = rng.randint(2, 12)
        parent, score = _dyadic_tree(rng, n)
        th = rng.choice([0.0, 0.1, 0.3, 0.5, 0.9])
        keep = rng.randint(1, n)
        _, _, _, got = oracle.prune_topB(score, parent, list(range(n)), n, keep, th)
        order = [v for v in sorted(range(1, n), key=lambda v: (-float(score[v]), v))
                 if float(score[v]) >= th]
        assert set(got) == {0, *order[:keep - 1]}


def test_prune_chain_and_errors():
    n = 10
    chain = [-1] + list(range(n - 1))
    sc = np.float32([0.9 ** i for i in range(n)])
    p, _, _, o = oracle.prune_topB(sc, chain, list(range(n)), n, 4)
    assert o == [0, 1, 2, 3] and p == [-1, 0, 1, 2]
    bad = sc.copy()
    bad[5] = 2.0
    with pytest.raises(oracle.NonMonotoneError):
        oracle.prune_topB(bad, chain, list(range(n)), n, 4)
    bad[5] = np.nan
    with pytest.raises(oracle.NonMonotoneError):
        oracle.prune_topB(bad, chain, list(range(n)), n, 4)
    with pytest.raises(oracle.TreeError):
        oracle.prune_topB(sc, [-1, 0, 5] + list(range(2, n - 1)), list(range(n)), n, 4)


# --------------------------------------------------------------------------------- graft


def test_graft_hand_example():
    g = golden("graft_small.json")
    table = np.asarray(g["table"], np.int32)
    for c in g["cases"]:
        p, t, n = oracle.graft_expand(g["kept_parent"], g["kept_tokens"], 3, g["tpar"],
                                      g["trank"], c["R"], table, c["Nmax"])
        assert (p, t, n) == (c["parent"], c["tokens"], c["n"])


def _walk_len(parent, tokens, n, f):
    argmax = [f[t] for t in tokens[:n]]
    return oracle.verify_greedy(tokens, parent, n, argmax, 0)["acc_len"]


def test_graft_properties_and_superset_acceptance():
    """Each grafted token is table[token(parent)][rank]; the kept tree is untouched
    (superset, Graft write-up §三), so acceptance never drops when slots are refilled."""
    rng = np.random.default_rng(3)
    V, k = 12, 4
    from workload import default_template
    tpar, trank = default_template(40, k)
    for _ in range(200):
        table = rng.integers(-1, V, size=(V, k)).astype(np.int32)
        f = rng.integers(0, V, size=V)            # bigram target: argmax is f[token]
        nk = int(rng.integers(1, 8))
        parent = [-1] + [int(rng.integers(0, v)) for v in range(1, nk)]
        tokens = [int(x) for x in rng.integers(0, V, size=nk)]
        R = int(rng.integers(0, 41))
        Nmax = nk + int(rng.integers(0, 45))
        gp, gt, n = oracle.graft_expand(parent, tokens, nk, tpar, trank, R, table, Nmax)
        assert gp[:nk] == parent and gt[:nk] == tokens
        assert n <= min(Nmax, nk + R)
        for v in range(nk, n):
            assert 0 <= gp[v] < v
            assert gt[v] != -1
            assert gt[v] in table[gt[gp[v]]].tolist()
        assert gp[n:] == [-1] * (Nmax - n) and gt[n:] == [-1] * (Nmax - n)
        assert _walk_len(gp, gt, n, f) >= _walk_len(parent, tokens, nk, f)


def test_graft_full_table_fills_budget():
    g = golden("budgets.json")
    from workload import default_template
    V, k = 50, 8
    table = (np.arange(V * k).reshape(V, k) % V).astype(np.int32)
    tpar, trank = default_template(52, k)
    for d, r in g["stages"].values():
        parent = [-1] + list(range(d - 1))
        tokens = list(range(d))
        gp, gt, n = oracle.graft_expand(parent, tokens, d, tpar, trank, r, table, g["slots"])
        assert n == g["slots"]


# ---------------------------------------------------------------------------------- walk


def test_walk_hand_example():
    g = golden("hand_tree7.json")
    r = oracle.verify_greedy(g["tokens"], g["parent"], 7, g["argmax"], g["prefix_len"])
    for key in ("acc_len", "path", "out_tok", "kv_src", "kv_dst"):
        assert r[key] == g[key], key


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6])
def test_walk_brute_force_all_trees(n):
    rng = random.Random(n)
    for parent in all_trees(n):
        for _ in range(3):
            tokens = [rng.randrange(3) for _ in range(n)]
            argmax = [rng.randrange(3) for _ in range(n)]
            acc = []
            for v in range(n):
                u, ok = v, True
                while u != 0:
                    ok &= tokens[u] == argmax[parent[u]]
                    u = parent[u]
                acc.append(ok)
            depth = [int(closure(parent)[v].sum()) - 1 for v in range(n)]
            best = min((v for v in range(n) if acc[v]), key=lambda v: (-depth[v], v))
            r = oracle.verify_greedy(tokens, parent, n, argmax, 3)
            assert r["path"][-1] == best and r["acc_len"] == depth[best]
            path = r["path"]
            assert path[0] == 0 and all(parent[path[j + 1]] == path[j] for j in range(len(path) - 1))
            assert r["out_tok"] == [tokens[p] for p in path[1:]] + [argmax[best]]
            assert r["kv_src"] == [3 + p for p in path]
            assert r["kv_dst"] == [3 + j for j in range(len(path))]


def test_walk_lossless_vs_sequential_greedy():
    """Accepted tokens + bonus equal plain greedy decoding under a bigram target
    (Graft write-up §二: verification keeps the target's output unchanged)."""
    rng = np.random.default_rng(5)
    for _ in range(300):
        V = int(rng.integers(2, 6))
        f = rng.integers(0, V, size=V)
        n = int(rng.integers(1, 30))
        parent = [-1] + [int(rng.integers(0, v)) for v in range(1, n)]
        tokens = [int(x) for x in rng.integers(0, V, size=n)]
        r = oracle.verify_greedy(tokens, parent, n, [int(f[t]) for t in tokens], 0)
        seq, x = [], tokens[0]
        for _j in range(r["acc_len"] + 1):
            x = int(f[x])
            seq.append(x)
        assert r["out_tok"] == seq


def test_walk_monotone_under_superset():
    """Adding nodes never shortens the accepted prefix (Graft write-up §三)."""
    rng = np.random.default_rng(9)
    for _ in range(300):
        V = 3
        f = rng.integers(0, V, size=V)
        n = int(rng.integers(1, 15))
        parent = [-1] + [int(rng.integers(0, v)) for v in range(1, n)]
        tokens = [int(x) for x in rng.integers(0, V, size=n)]
        L0 = _walk_len(parent, tokens, n, f)
        for _add in range(10):
            parent.append(int(rng.integers(0, len(parent))))
            tokens.append(int(rng.integers(0, V)))
            L1 = _walk_len(parent, tokens, len(parent), f)
            assert L1 >= L0
            L0 = L1


# -------------------------------------------------------------------------------- update


def test_update_hand_example():
    g = golden("update_small.json")
    t = oracle.succ_update(np.asarray(g["table"]), g["tokens"], g["topk_id"], g["n_nodes"])
    assert t.tolist() == g["expected"]


def test_update_last_writer_and_untouched_rows():
    rng = np.random.default_rng(2)
    V, k, B, N = 40, 8, 3, 20
    table = rng.integers(0, V, size=(V, k)).astype(np.int32)
    tokens = rng.integers(0, V, size=(B, N))
    topk = rng.integers(0, V, size=(B, N, k))
    n = rng.integers(0, N + 1, size=B)
    t = oracle.succ_update(table, tokens, topk, n)
    writers = {}
    for b in range(B):
        for v in range(int(n[b])):
            writers[int(tokens[b, v])] = (b, v)
    for row in range(V):
        if row in writers:
            b, v = writers[row]
            assert t[row].tolist() == topk[b, v].tolist()
        else:
            assert t[row].tolist() == table[row].tolist()


def test_graft_at_anchor_tail_of_a_chain():
    # Graft-TAIL: a 5-node chain kept, the retrieved nodes hang from its last node
    table = np.array([[1, 2], [3, 4], [0, 1], [4, 0], [2, 3]], np.int32)  # V = 5, k = 2
    parent = [-1, 0, 1, 2, 3, -1, -1, -1, -1, -1]
    tokens = [0, 1, 3, 4, 2, -1, -1, -1, -1, -1]
    tpar, trank = [-1, -1, 0], [0, 1, 0]
    p, t, n = oracle.graft_expand(parent, tokens, 5, tpar, trank, 3, table, 10, anchor=-1)
    # anchor = node 4 (token 2): children table[2] = (0, 1); grandchild table[0][0] = 1
    assert n == 8
    assert p[:8] == [-1, 0, 1, 2, 3, 4, 4, 5]
    assert t[:8] == [0, 1, 3, 4, 2, 0, 1, 1]
    # an explicit anchor inside the kept tree, and the default (root) unchanged
    p2, t2, n2 = oracle.graft_expand(parent, tokens, 5, tpar, trank, 3, table, 10, anchor=2)
    assert p2[5:8] == [2, 2, 5] and t2[5:8] == [4, 0, 2]
    assert oracle.graft_expand(parent, tokens, 5, tpar, trank, 3, table, 10, anchor=0) == \
        oracle.graft_expand(parent, tokens, 5, tpar, trank, 3, table, 10)
    with pytest.raises(oracle.OracleError):
        oracle.graft_expand(parent, tokens, 5, tpar, trank, 3, table, 10, anchor=5)
