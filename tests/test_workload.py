"""Sanity of the seeded input generator (shapes, tree validity, reproducibility)."""
import numpy as np
import torch

from workload import (CONFIGS, bf16_bits_to_f32, bigram_table, default_template,
                      f32_to_bf16_bits, make_scenario, stream_table)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32),
                        np.float32([0.0, -0.0, 1e-40, -3e38, np.inf, -np.inf])])
    ours = f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(bf16_bits_to_f32(ours), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_template_is_ancestor_closed_and_asymmetric():
    tpar, trank = default_template(52, 8)
    assert len(tpar) == 52
    for t in range(52):
        assert -1 <= tpar[t] < t and 0 <= trank[t] < 8
    # subtree sizes of the root's children shrink with rank
    size = np.ones(52, int)
    for t in range(51, -1, -1):
        if tpar[t] >= 0:
            size[tpar[t]] += size[t]
    roots = [t for t in range(52) if tpar[t] == -1]
    sizes = [size[t] for t in sorted(roots, key=lambda t: trank[t])]
    assert sizes == sorted(sizes, reverse=True) and sizes[0] > sizes[-1]
    # prefixes serve every refill size
    for R in (20, 36, 52):
        p, r = default_template(R, 8)
        assert np.array_equal(p, tpar[:R]) and np.array_equal(r, trank[:R])


def test_tables_in_range_and_distinct_rows():
    rng = np.random.default_rng(1)
    for t in (bigram_table(rng, 5000, 8), stream_table(rng, 5000, 8, length=50000)):
        assert t.shape == (5000, 8) and t.min() >= 0 and t.max() < 5000
        assert all(len(set(row)) == 8 for row in t[:2000].tolist())


def test_scenarios_small_are_valid_and_reproducible():
    for cid in CONFIGS:
        s = make_scenario(cid, V=3000, P=(100, 300) if cid == 4 else 200, B=3 if cid == 4 else None,
                          stream_len=20000)
        s2 = make_scenario(cid, V=3000, P=(100, 300) if cid == 4 else 200, B=3 if cid == 4 else None,
                           stream_len=20000)
        assert np.array_equal(s.parent_in, s2.parent_in) and np.array_equal(s.table, s2.table)
        assert np.array_equal(s.Q, s2.Q)
        for b in range(s.B):
            p, sc = s.parent_in[b], s.score_in[b]
            assert p[0] == -1 and all(0 <= p[v] < v for v in range(1, s.Nin))
            assert all(sc[v] <= sc[p[v]] for v in range(1, s.Nin))
        assert s.Q.shape == (s.B, s.N, s.Hq, s.d)
        assert s.K.shape == (s.B, s.Hkv, s.Lcap, s.d)
    assert make_scenario(1, V=3000, P=100).Nin == 411
    assert make_scenario(5, V=3000, P=100).Nin == 256
    assert make_scenario(4, V=3000, P=(100, 200), B=2).Nin == 60


def test_block_draft_is_a_chain_with_falling_scores():
    s = make_scenario(6, V=3000, P=100, B=4, stream_len=20000)
    assert s.Nin == 17 and s.N == 17 and s.anchor.tolist() == [-1] * 4
    for b in range(s.B):
        assert s.parent_in[b].tolist() == list(range(-1, 16))
        assert np.all(np.diff(s.score_in[b].astype(np.float64)) < 0)
        # the threshold lies strictly inside the chain's score range
        assert s.score_in[b, -1] < s.thresh[b] < s.score_in[b, 1]
