"""Pins for the oracle's floating-point steps: tree attention and vocab top-k.

Attention is checked against torch's scaled_dot_product_attention in float64 on the CPU
(a different routine from the oracle's numpy softmax) with a mask from brute-force
ancestor closure, against causal attention for a chain tree and against plain decode
attention for a one-node tree. Top-k is checked against torch.topk on tie-free rows and
against a brute-force Python sort on rows full of ties, signed zeros, NaN and infinities.
"""
import random

import numpy as np
import pytest
import torch

import oracle
from test_oracle_tree import closure


def _sdpa(Q, K, V, allowed, scale, g):
    q = torch.from_numpy(Q).permute(1, 0, 2)[None]                 # [1,Hq,n,d]
    k = torch.from_numpy(K).repeat_interleave(g, dim=0)[None]      # [1,Hq,L,d]
    v = torch.from_numpy(V).repeat_interleave(g, dim=0)[None]
    m = torch.from_numpy(allowed)[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 2), (12, 4)])
def test_attn_matches_sdpa_random_trees(Hq, Hkv):
    rng = np.random.default_rng(Hq * 10 + Hkv)
    d, g = 16, Hq // Hkv
    for _ in range(6):
        n = int(rng.integers(1, 20))
        P = int(rng.integers(0, 40))
        parent = [-1] + [int(rng.integers(0, v)) for v in range(1, n)]
        L = P + n
        Q = rng.standard_normal((n, Hq, d))
        K = rng.standard_normal((Hkv, L + 7, d))
        V = rng.standard_normal((Hkv, L + 7, d))
        scale = float(np.float32(1 / np.sqrt(d)))
        O = oracle.tree_attn(Q, K, V, parent, n, P, scale)
        allowed = np.ones((n, L), bool)
        allowed[:, P:] = closure(parent)
        ref = _sdpa(Q, K[:, :L], V[:, :L], allowed, scale, g)
        np.testing.assert_allclose(O, ref, rtol=1e-12, atol=1e-12)


def test_attn_chain_is_causal_and_single_node_is_decode():
    rng = np.random.default_rng(1)
    Hq, Hkv, d, P, n = 4, 2, 32, 25, 9
    Q = rng.standard_normal((n, Hq, d))
    K = rng.standard_normal((Hkv, P + n, d))
    V = rng.standard_normal((Hkv, P + n, d))
    chain = [-1] + list(range(n - 1))
    O = oracle.tree_attn(Q, K, V, chain, n, P, 0.125)
    # causal attention over the full sequence, queries at positions P..P+n-1
    qf = torch.zeros(1, Hq, P + n, d, dtype=torch.float64)
    qf[0, :, P:] = torch.from_numpy(Q).permute(1, 0, 2)
    kf = torch.from_numpy(K).repeat_interleave(2, dim=0)[None]
    vf = torch.from_numpy(V).repeat_interleave(2, dim=0)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf, is_causal=True, scale=0.125)
    np.testing.assert_allclose(O, ref[0, :, P:].permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)
    # one node: plain decode attention over all P+1 keys
    O1 = oracle.tree_attn(Q[:1], K, V, [-1], 1, P, 0.125)
    for h in range(Hq):
        s = (K[h // 2, :P + 1] @ Q[0, h]) * 0.125
        w = np.exp(s - s.max())
        w /= w.sum()
        np.testing.assert_allclose(O1[0, h], w @ V[h // 2, :P + 1], rtol=1e-12, atol=1e-12)


def test_attn_equal_keys_average_visible_values():
    rng = np.random.default_rng(4)
    Hq, Hkv, d, P, n = 2, 1, 8, 6, 5
    parent = [-1, 0, 0, 1, 3]
    Q = rng.standard_normal((n, Hq, d))
    K = np.ones((Hkv, P + n, d))
    V = rng.standard_normal((Hkv, P + n, d))
    O = oracle.tree_attn(Q, K, V, parent, n, P, 0.3)
    R = closure(parent)
    for i in range(n):
        vis = list(range(P)) + [P + u for u in range(n) if R[i, u]]
        np.testing.assert_allclose(O[i, 0], V[0, vis].mean(axis=0), rtol=1e-12)


def test_bf16_decode():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x8000, 0x7F80, 0x4049, 0x0001], np.uint16)
    v = oracle.bf16_to_f64(bits)
    assert v[0] == 1.0 and v[1] == -1.0 and v[2] == 0.0 and np.signbit(v[3])
    assert np.isinf(v[4]) and v[5] == 3.140625
    assert v[6] == 2.0 ** -133  # smallest bf16 subnormal


def test_topk_matches_torch_on_distinct_values():
    rng = np.random.default_rng(0)
    for V in (1, 7, 100, 5000):
        for _ in range(5):
            row = rng.permutation(V).astype(np.float32) * np.float32(0.37) - np.float32(V / 5)
            k = min(8, V)
            ids, vals = oracle.vocab_topk(row, k)
            tv, ti = torch.topk(torch.from_numpy(row), k)
            assert ids.tolist() == ti.tolist()
            assert vals.tolist() == tv.tolist()


def test_topk_brute_force_with_ties_zeros_nan_inf():
    rng = random.Random(3)
    pool = [0.0, -0.0, 1.0, -1.0, 2.5, float("inf"), float("-inf"), float("nan"), 1e-30, -1e-30]
    for _ in range(500):
        V = rng.randint(1, 40)
        row = np.float32([rng.choice(pool) for _ in range(V)])
        k = rng.randint(1, 16)
        ids, vals = oracle.vocab_topk(row, min(k, V))
        key = lambda i: (bool(np.isnan(row[i])), 0.0 if np.isnan(row[i]) else -float(row[i]), i)
        ref = sorted(range(V), key=key)[:min(k, V)]
        assert ids.tolist() == ref
        assert np.array_equal(vals.view(np.uint32), row[ref].view(np.uint32))


def test_topk_closed_forms():
    V = 1000
    ids, _ = oracle.vocab_topk(np.arange(V, dtype=np.float32), 8)
    assert ids.tolist() == list(range(V - 1, V - 9, -1))
    ids, _ = oracle.vocab_topk(np.full(V, 3.0, np.float32), 8)
    assert ids.tolist() == list(range(8))
    row = np.zeros(V, np.float32)
    row[::2] = -0.0
    ids, _ = oracle.vocab_topk(row, 5)
    assert ids.tolist() == [0, 1, 2, 3, 4]
