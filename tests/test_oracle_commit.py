"""Pins of the oracle's KV commit (compaction of the accepted path's cache rows): a hand
example, the in-place sequential reading, the chain identity and input checks."""
import numpy as np
import pytest

import oracle


def _cache(B, H, L, d, seed=0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((B, H, L, d)), rng.standard_normal((B, H, L, d))


def test_kv_commit_hand_example():
    # one request, two KV heads, cache of 8 rows; row r of head h holds (10h + r, -r)
    K = np.array([[[[10 * h + r, -r] for r in range(8)] for h in range(2)]], dtype=np.float64)
    V = -K
    # prefix P = 2, accepted path 0 -> 2 -> 3: rows 2, 4, 5 move to rows 2, 3, 4
    Kn, Vn = oracle.kv_commit(K, V, [[2, 4, 5]], [[2, 3, 4]], [2])
    expect_rows = [0, 1, 2, 4, 5, 5, 6, 7]  # row 5 keeps its value, it is not a destination
    for h in range(2):
        assert Kn[0, h, :, 0].tolist() == [10 * h + r for r in expect_rows]
        assert Kn[0, h, :, 1].tolist() == [-r for r in expect_rows]
    assert np.array_equal(Vn, -Kn)


def _random_walk(rng, n, P):
    parent = [-1] + [int(rng.integers(0, v)) for v in range(1, n)]
    tokens = rng.integers(0, 5, size=n)
    argmax = rng.integers(0, 5, size=n)
    return oracle.verify_greedy(tokens, parent, n, argmax, P)


def test_kv_commit_equals_in_place_copies_in_path_order():
    # the path's nodes increase with depth and path[j] >= j, so copying row by row in place,
    # j = 0, 1, ..., never overwrites a row that a later copy still reads
    rng = np.random.default_rng(1)
    for trial in range(200):
        B, H, d, N = 3, 2, 4, 24
        P = [int(x) for x in rng.integers(0, 20, size=B)]
        walks = [_random_walk(rng, int(rng.integers(1, N + 1)), P[b]) for b in range(B)]
        Lcap = max(P) + N
        K, V = _cache(B, H, Lcap, d, seed=trial)
        src = [w["kv_src"] for w in walks]
        dst = [w["kv_dst"] for w in walks]
        L = [w["acc_len"] for w in walks]
        Kn, Vn = oracle.kv_commit(K, V, src, dst, L)
        Ks, Vs = K.copy(), V.copy()
        for b in range(B):
            for j in range(L[b] + 1):
                Ks[b, :, dst[b][j]] = Ks[b, :, src[b][j]]
                Vs[b, :, dst[b][j]] = Vs[b, :, src[b][j]]
        assert np.array_equal(Kn, Ks) and np.array_equal(Vn, Vs)
        # rows outside [P, P + L] are untouched
        for b in range(B):
            keep = np.ones(Lcap, bool)
            keep[P[b]:P[b] + L[b] + 1] = False
            assert np.array_equal(Kn[b][:, keep], K[b][:, keep])


def test_kv_commit_chain_is_identity():
    K, V = _cache(2, 3, 40, 8)
    L = [5, 0]
    src = [[10 + j for j in range(6)], [7]]
    dst = [[10 + j for j in range(6)], [7]]
    Kn, Vn = oracle.kv_commit(K, V, src, dst, L)
    assert np.array_equal(Kn, K) and np.array_equal(Vn, V)


def test_kv_commit_rejects_rows_outside_the_cache():
    K, V = _cache(1, 1, 10, 2)
    with pytest.raises(oracle.OracleError):
        oracle.kv_commit(K, V, [[3, 12]], [[3, 4]], [1])
    with pytest.raises(oracle.OracleError):
        oracle.kv_commit(K, V, [[3]], [[3]], [1])  # acc_len beyond the path buffer
