"""Pins of the T > 0 verification oracle (oracle/sampling.py) to published vectors,
closed forms, exact distributions and the independently pinned greedy walk."""
import itertools

import numpy as np
import pytest

import oracle
from conftest import golden
from oracle.sampling import (argmax_first, gumbel_scores, log_f32, noise_words, philox4x32_10,
                             step_verify_sampled, uniform_f32, verify_sampled, vocab_sample)


def test_philox_known_answers():
    for vec in golden("philox_kat.json")["vectors"]:
        c = [int(x, 16) for x in vec["ctr"]]
        k = [int(x, 16) for x in vec["key"]]
        out = philox4x32_10(*[np.array([x]) for x in c], *k)
        assert [int(w[0]) for w in out] == [int(x, 16) for x in vec["out"]]


def test_noise_words_are_uniform_and_independent():
    x = noise_words(200003, np.arange(4), seed=8, step=2).astype(np.uint64)
    n = x.size
    # the top byte and the low 24 bits come from different Philox blocks: each uniform
    for part, bins in ((x >> np.uint64(24), 256), ((x >> np.uint64(8)) & np.uint64(0xFF), 256),
                       (x & np.uint64(0xFF), 256)):
        cnt = np.bincount(part.astype(np.int64).ravel(), minlength=bins)
        chi2 = ((cnt - n / bins) ** 2 / (n / bins)).sum()
        assert chi2 < bins + 6 * np.sqrt(2 * bins)  # mean bins - 1, sd sqrt(2 (bins - 1))
    u = x.astype(np.float64) / 2.0 ** 32
    for a, b in ((u[:, :-1], u[:, 1:]), (u[:, :-16], u[:, 16:]), (u[:-1], u[1:])):
        assert abs(np.corrcoef(a.ravel(), b.ravel())[0, 1]) < 5 / np.sqrt(a.size)
    top, low = (x >> np.uint64(24)).astype(np.float64), (x & np.uint64(0xFFFFFF)).astype(np.float64)
    assert abs(np.corrcoef(top.ravel(), low.ravel())[0, 1]) < 5 / np.sqrt(n)
    # the candidate byte (255) marks exactly the words of U >= 255/256
    assert np.array_equal(x >= np.uint64(0xFF000000), (x >> np.uint64(24)) == 255)


def test_uniform_grid_and_ends():
    x = np.array([0, 1 << 9, 0xFFFFFFFF, 0x80000000], np.uint32)
    u = uniform_f32(x)
    assert u.dtype == np.float32
    assert u.tolist() == [2.0 ** -24, 3 * 2.0 ** -24, 1 - 2.0 ** -24, 0.5 + 2.0 ** -24]
    r = np.random.default_rng(0).integers(0, 1 << 32, size=100000, dtype=np.uint64)
    u = uniform_f32(r.astype(np.uint32)).astype(np.float64)
    assert np.all((u > 0) & (u < 1))
    assert np.all(np.mod(u * 2.0 ** 24, 2.0) == 1.0)  # odd multiples of 2^-24


def test_log_f32_error_bound_and_exact_points():
    x = np.float32(np.exp(np.linspace(np.log(2.0 ** -30), np.log(1e6), 300001)))
    x = np.concatenate([x, np.float32(1 - np.arange(1, 2000) * 2.0 ** -24),
                        np.float32(1 + np.arange(1, 2000) * 2.0 ** -23)])
    got = log_f32(x).astype(np.float64)
    ref = np.log(x.astype(np.float64))
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 3 * ulp + 1e-45)
    # powers of two: the series vanishes, e * float32(ln 2) remains
    for e in range(-24, 20):
        assert log_f32(np.float32([2.0 ** e]))[0] == np.float32(e) * np.float32(np.log(2.0))
    assert log_f32(np.float32([1.0]))[0] == 0.0


def test_gumbel_noise_moments():
    # G = -log(-log U): mean = Euler's constant, variance = pi^2 / 6 (standard Gumbel)
    z = np.zeros((50, 20000), np.float32)
    g = gumbel_scores(z, np.arange(50), 1.0, seed=99, step=3).astype(np.float64).ravel()
    n = g.size
    assert abs(g.mean() - np.euler_gamma) < 5 * np.sqrt(np.pi ** 2 / 6 / n)
    assert abs(g.var() - np.pi ** 2 / 6) < 0.02
    # CDF exp(-exp(-x)) at a few points
    for x in (-1.0, 0.0, 1.0, 3.0):
        p = np.exp(-np.exp(-x))
        assert abs((g <= x).mean() - p) < 5 * np.sqrt(p * (1 - p) / n)


@pytest.mark.parametrize("T", [0.5, 1.0, 2.0])
def test_gumbel_max_draws_follow_softmax(T):
    z0 = np.float32([0.1, 1.0, -0.5, 2.0, 0.0, -3.0])
    M = 200000
    s = vocab_sample(np.tile(z0, (M, 1)), np.arange(M), T, seed=1234, step=77)
    freq = np.bincount(s, minlength=z0.size) / M
    w = np.exp(z0.astype(np.float64) / T)
    p = w / w.sum()
    assert np.all(np.abs(freq - p) <= 5 * np.sqrt(p * (1 - p) / M) + 1e-12)


def test_draws_depend_on_row_step_and_seed_words():
    z = np.zeros((4, 4096), np.float32)
    base = vocab_sample(z, np.arange(4), 1.0, seed=1, step=1)
    assert len(set(base.tolist())) == 4  # rows differ
    for kw in (dict(seed=1 + (1 << 32), step=1), dict(seed=1, step=1 + (1 << 32)),
               dict(seed=2, step=1), dict(seed=1, step=2)):
        assert not np.array_equal(vocab_sample(z, np.arange(4), 1.0, **kw), base)
    assert np.array_equal(vocab_sample(z, np.arange(4), 1.0, seed=1, step=1), base)


def test_low_temperature_is_argmax_and_order_rules():
    rng = np.random.default_rng(5)
    z = rng.permutation(np.arange(3000, dtype=np.float32) * np.float32(0.05))[None, :]
    z = np.repeat(z, 8, axis=0)
    # score gaps of at least 0.05 / 1e-3 = 50 exceed the Gumbel range [-2.9, 16.7]
    s = vocab_sample(z, np.arange(8), 1e-3, seed=3, step=0)
    assert np.all(s == np.argmax(z[0]))
    # NaN ranks below -inf; +0 equals -0 (first index wins); equal maxima: first index
    sc = np.float32([[np.nan, -np.inf, -1.0], [np.nan, np.nan, np.nan], [-0.0, 0.0, -1.0],
                     [2.0, 5.0, 5.0], [np.inf, np.nan, np.inf]])
    assert argmax_first(sc).tolist() == [2, 0, 0, 1, 0]


def _all_trees(n):
    for par in itertools.product(*[range(v) for v in range(1, n)]):
        yield [-1] + list(par)


def test_sampled_walk_equals_greedy_walk_when_draws_are_argmaxes():
    # distinct sibling tokens: one draw per node equal to the argmax makes the sampled walk
    # the greedy walk (the greedy oracle is pinned by brute force elsewhere)
    rng = np.random.default_rng(11)
    for n in range(1, 7):
        for parent in _all_trees(n):
            tokens = [int(rng.integers(0, 3))]
            for v in range(1, n):
                used = {tokens[c] for c in range(1, v) if parent[c] == parent[v]}
                tokens.append(min(set(range(n + 1)) - used) if rng.random() < 0.5
                              else int(rng.choice(sorted(set(range(n + 1)) - used))))
            draw = [int(rng.integers(0, n + 1)) for _ in range(n)]
            a = verify_sampled(tokens, parent, n, draw, 10)
            b = oracle.verify_greedy(tokens, parent, n, draw, 10)
            assert a == b


def test_sampled_walk_takes_the_first_duplicate_sibling():
    parent = [-1, 0, 0, 1, 2, 4]
    tokens = [9, 4, 4, 7, 7, 3]  # nodes 1 and 2 both carry token 4; node 2 has the deeper subtree
    r = verify_sampled(tokens, parent, 6, [4, 7, 7, 0, 3, 0], 100)
    assert r["path"] == [0, 1, 3] and r["out_tok"] == [4, 7, 0]
    assert r["kv_src"] == [100, 101, 103] and r["kv_dst"] == [100, 101, 102]


def test_sampled_verification_is_lossless():
    """The emitted tokens follow the target's own conditionals: the first token ~ p(.|root),
    and given an accepted first token a, the second ~ p(.|a); a duplicate sibling that
    the first-child rule shadows is never entered."""
    V, T = 4, 0.8
    rng = np.random.default_rng(21)
    ctx_logits = {(): rng.standard_normal(V), (0,): rng.standard_normal(V),
                  (1,): rng.standard_normal(V), (0, 2): rng.standard_normal(V),
                  (0, 0): rng.standard_normal(V)}
    # root children: token 0 (node 1), token 1 (node 2), token 0 again (node 3, shadowed);
    # under node 1: tokens 2 (node 4) and 0 (node 5)
    parent = [-1, 0, 0, 0, 1, 1]
    tokens = [3, 0, 1, 0, 2, 0]
    ctx = [(), (0,), (1,), (0,), (0, 2), (0, 0)]
    n, M = len(parent), 120000
    logits = np.stack([np.float32(ctx_logits[c]) for c in ctx])
    rows = np.arange(M * n)
    draws = vocab_sample(np.tile(logits, (M, 1)), rows, T, seed=2024, step=5).reshape(M, n)
    first, second = np.zeros(M, int), np.full(M, -1)
    for i in range(M):
        r = verify_sampled(tokens, parent, n, draws[i], 0)
        assert 3 not in r["path"]
        first[i] = r["out_tok"][0]
        if len(r["out_tok"]) > 1:
            second[i] = r["out_tok"][1]

    def p(c):
        w = np.exp(np.float32(ctx_logits[c]).astype(np.float64) / T)
        return w / w.sum()

    def close(samples, probs):
        f = np.bincount(samples, minlength=V) / len(samples)
        return np.all(np.abs(f - probs) <= 5 * np.sqrt(probs * (1 - probs) / len(samples)))

    assert close(first, p(()))
    for a in (0, 1):  # tokens with a child at the root: a second token is always emitted
        sel = second[first == a]
        assert np.all(sel >= 0) and close(sel, p((a,)))
    assert np.all(second[(first == 2) | (first == 3)] == -1)


def test_step_at_temperature_keeps_the_greedy_table_update():
    from workload import make_scenario
    scn = make_scenario(2, V=700, P=64, stream_len=5000)
    tree = oracle.step_tree_phase(scn.parent_in, scn.tokens_in, scn.score_in, [scn.Nin] * scn.B,
                                  scn.keep, scn.thresh, scn.tpar, scn.trank, scn.R, scn.table,
                                  scn.prefix_len, scn.N)
    logits = scn.logits(tree["parent"], tree["tokens"], tree["n_nodes"])
    g = oracle.step_verify_phase(tree, logits, scn.table, scn.prefix_len, scn.k)
    s = step_verify_sampled(tree, logits, scn.table, scn.prefix_len, scn.k, 0.7, 9, 4)
    assert np.array_equal(s["table"], g["table"]) and np.array_equal(s["topk_id"], g["topk_id"])
    assert s["acc_len"][0] == len(verify_sampled(tree["tokens"][0], tree["parent"][0],
                                                 int(tree["n_nodes"][0]), s["sample"][0],
                                                 0)["path"]) - 1
