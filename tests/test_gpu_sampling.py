"""GPU parity of verification at temperature T > 0: the draws, the sampled walk and the
table update through the C ABI against the oracle, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from oracle.sampling import step_verify_sampled, verify_sampled, vocab_sample
from parity_util import device_inputs, np_, oracle_tree, shape_of
from tree_speculative_decoding_parent_gb300 import gt
from tree_speculative_decoding_parent_gb300.step import (StepBuffers, run_tree_build,
                                                         run_verify_sample_commit)
from workload import make_scenario

pytestmark = pytest.mark.gpu

SEEDS = [(0, 0), (12345, 7), ((1 << 40) + 3, (1 << 33) + 11), (0xFFFFFFFFFFFFFFFF, 0xFFFFFFFF)]


def _gpu_sample(z: np.ndarray, T: float, seed: int, step: int) -> np.ndarray:
    rows, V = z.shape
    dz = torch.from_numpy(np.ascontiguousarray(z)).cuda()
    out = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
    gt.gt_vocab_sample(dz, rows, V, T, seed, step, out)
    torch.cuda.synchronize()
    return np_(out)


@pytest.mark.parametrize("V", [4099, 32000, 151936])
def test_vocab_sample_matches_oracle(V):
    rng = np.random.default_rng(V)
    rows = 70 if V < 100000 else 12
    z = (rng.standard_normal((rows, V)) * rng.uniform(0.5, 4.0, size=(rows, 1))).astype(np.float32)
    for T, (seed, step) in zip([1.0, 0.55, 1.7, 1.0], SEEDS):
        got = _gpu_sample(z, T, seed, step)
        want = vocab_sample(z, np.arange(rows), T, seed, step)
        assert np.array_equal(got, want), (T, seed, step, np.flatnonzero(got != want))


def test_vocab_sample_special_values_and_unaligned_rows():
    V = 1000
    rng = np.random.default_rng(3)
    z = rng.standard_normal((9, V)).astype(np.float32)
    z[0, ::3] = np.nan                    # NaN entries never win over numbers
    z[1, :] = np.nan                      # a row of NaN only: index 0
    z[2, :] = -np.inf                     # all -inf: index 0 (every score is -inf)
    z[3, 17] = np.inf                     # +inf wins
    z[4, [5, 600]] = np.inf               # two +inf: the lower index
    z[5, :] = 0.0                         # a flat row: a uniform draw
    z[6, ::2] = -0.0
    z[7, :] = 3e38                        # z / T overflows to +inf at T = 0.5: index 0
    z[8, :] = rng.standard_normal(V).astype(np.float32) * 1e-30
    for T in (1.0, 0.5):
        assert np.array_equal(_gpu_sample(z, T, 77, 5), vocab_sample(z, np.arange(9), T, 77, 5))
    # rows that start off a 16-byte boundary take the element-wise load path
    zz = rng.standard_normal((5 * 4096 + 1,)).astype(np.float32)
    dz = torch.from_numpy(zz).cuda()[1:]
    out = torch.empty(5, dtype=torch.int32, device="cuda")
    gt.gt_vocab_sample(dz, 5, 4096, 0.9, 4, 8, out)
    torch.cuda.synchronize()
    want = vocab_sample(zz[1:].reshape(5, 4096), np.arange(5), 0.9, 4, 8)
    assert np.array_equal(np_(out), want)


def test_vocab_sample_rejects_bad_temperatures():
    z = torch.zeros((2, 64), device="cuda")
    out = torch.empty(2, dtype=torch.int32, device="cuda")
    for T in (0.0, -1.0, float("inf"), float("nan"), 1e-39):
        with pytest.raises(gt.GTError) as e:
            gt.gt_vocab_sample(z, 2, 64, T, 1, 1, out)
        assert e.value.status == gt.GT_ERR_ARG


def _tree_and_logits(scn):
    tree = oracle_tree(scn)
    logits = scn.logits(tree["parent"], tree["tokens"], tree["n_nodes"])
    return tree, logits


SMALL = {1: dict(), 2: dict(V=5000, P=700), 3: dict(V=4099, P=1333, stream_len=50000),
         4: dict(V=4096, P=(200, 900), B=5, stream_len=50000), 5: dict(V=5003, P=611),
         6: dict(V=4099, P=500, B=4, stream_len=50000)}


@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5, 6])
def test_verify_sample_commit_matches_oracle(cid):
    scn = make_scenario(cid, **SMALL[cid])
    tree, logits = _tree_and_logits(scn)
    for T, (seed, step) in ((1.0, (99, 3)), (0.6, ((1 << 35) + 5, (1 << 32) + 1))):
        buf = StepBuffers(shape_of(scn))
        inp = device_inputs(scn, logits)
        run_tree_build(buf, inp)
        run_verify_sample_commit(buf, inp, T, seed, step)
        torch.cuda.synchronize()
        assert int(buf.err.item()) == 0
        want = step_verify_sampled(tree, logits, scn.table, scn.prefix_len, scn.k, T, seed, step)
        assert np.array_equal(np_(buf.sample), want["sample"])
        assert np.array_equal(np_(buf.topk_id), want["topk_id"])
        assert np.array_equal(np_(buf.topk_val).view(np.uint32), want["topk_val"].view(np.uint32))
        for key in ("acc_len", "path", "out_tok", "kv_src", "kv_dst"):
            assert np.array_equal(np_(getattr(buf, key)), want[key]), key
        assert np.array_equal(np_(inp["table"]), want["table"])


def test_verify_sample_full_size_and_walk_only_call():
    scn = make_scenario(3)
    tree, logits = _tree_and_logits(scn)
    buf = StepBuffers(shape_of(scn))
    inp = device_inputs(scn, logits)
    run_tree_build(buf, inp)
    s = buf.shape
    gt.gt_verify_sample(inp["logits"], buf.tokens, buf.parent, buf.n_nodes, inp["prefix_len"],
                        s.B, s.N, s.V, 1.0, 2024, 9, buf.sample, buf.acc_len, buf.path,
                        buf.out_tok, buf.kv_src, buf.kv_dst, buf.err)
    torch.cuda.synchronize()
    assert int(buf.err.item()) == 0
    want = step_verify_sampled(tree, logits, scn.table, scn.prefix_len, scn.k, 1.0, 2024, 9)
    assert np.array_equal(np_(buf.sample), want["sample"])
    for key in ("acc_len", "path", "out_tok", "kv_src", "kv_dst"):
        assert np.array_equal(np_(getattr(buf, key)), want[key]), key


def test_sampled_walk_enters_the_first_duplicate_sibling():
    # nodes 1 and 3 both carry token 4 under the root; node 3 has the longer subtree.
    # Low temperature and planted peaks make every draw the planted token.
    B, N, V = 2, 8, 64
    parent = np.array([[-1, 0, 0, 0, 3, 4, 1, -1], [-1, 0, 1, 1, 2, 2, 4, 5]], np.int32)
    tokens = np.array([[9, 4, 5, 4, 7, 8, 6, -1], [9, 1, 2, 2, 3, 3, 5, 6]], np.int32)
    n = np.array([7, 8], np.int32)
    peak = np.array([[4, 6, 0, 7, 8, 1, 2, 0], [1, 2, 3, 5, 5, 6, 7, 9]])
    logits = np.zeros((B, N, V), np.float32)
    for b in range(B):
        logits[b, np.arange(N), peak[b]] = 40.0
    prefix = np.array([30, 50], np.int32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    sample = torch.empty((B, N), dtype=torch.int32, device="cuda")
    outs = {k: torch.empty((B, N + (k == "out_tok")), dtype=torch.int32, device="cuda")
            for k in ("path", "out_tok", "kv_src", "kv_dst")}
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gt.gt_verify_sample(t(logits), t(tokens), t(parent), t(n), t(prefix), B, N, V, 0.25, 1, 1,
                        sample, acc, outs["path"], outs["out_tok"], outs["kv_src"],
                        outs["kv_dst"], err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(np_(sample), peak)
    for b in range(B):
        r = verify_sampled(tokens[b], parent[b], int(n[b]), peak[b], int(prefix[b]))
        L = r["acc_len"]
        assert int(acc[b]) == L
        assert np_(outs["path"])[b, :L + 1].tolist() == r["path"]
        assert np_(outs["out_tok"])[b, :L + 2].tolist() == r["out_tok"] + [-1]
        assert np_(outs["kv_src"])[b, :L + 1].tolist() == r["kv_src"]
    # request 0: root draw 4 -> node 1 (first duplicate), whose draw 6 -> node 6; bonus 2
    assert np_(outs["path"])[0, :3].tolist() == [0, 1, 6]
    # request 1: two duplicate pairs (2, 3) and (4, 5): path 0 -> 1 -> 2 -> 4 -> 6
    assert np_(outs["path"])[1, :5].tolist() == [0, 1, 2, 4, 6]


def test_vocab_sample_long_rows_overflow_the_candidate_queue():
    # 305 rows give one CTA per row; a row of 420,000 logits holds ~1,640 candidates, more
    # than a CTA queues, so the CTA rescans its row exactly. Sampled rows against the oracle.
    rows, V = 305, 420000
    g = torch.Generator(device="cuda").manual_seed(5)
    dz = torch.randn((rows, V), device="cuda", generator=g)
    out = torch.empty(rows, dtype=torch.int32, device="cuda")
    gt.gt_vocab_sample(dz, rows, V, 1.3, 31, 2, out)
    torch.cuda.synchronize()
    pick = np.array([0, 1, 150, 304])
    z = dz[torch.from_numpy(pick).cuda()].cpu().numpy()
    assert np.array_equal(np_(out)[pick], vocab_sample(z, pick, 1.3, 31, 2))


@pytest.mark.parametrize("V", [37, 4099, 20000])
def test_sampled_commit_topk_special_values_and_ties(V):
    """The top-k that gt_verify_sample_commit forms in its sampling pass, against the oracle's
    top-k on rows of ties, +-0, +-inf, NaN, and rows of one repeated value (every element a
    candidate: the exact per-thread-list path), on aligned and unaligned rows."""
    import oracle
    rng = np.random.default_rng(V)
    B, N, k = 2, 33, 8
    pool = np.float32([0.0, -0.0, 1.0, -1.0, 2.5, np.inf, -np.inf, np.nan, 1e-30, -1e-30])
    logits = pool[rng.integers(0, len(pool), size=(B, N, V))].astype(np.float32)
    logits[0, 3, :] = 1.5          # one repeated value
    logits[1, 7, :] = -0.0
    logits[1, 8, :] = rng.standard_normal(V).astype(np.float32)
    parent = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    tokens = rng.integers(0, V, size=(B, N)).astype(np.int32)
    n = np.full(B, N, np.int32)
    P = np.zeros(B, np.int32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    ids = torch.empty((B, N, k), dtype=torch.int32, device="cuda")
    vals = torch.empty((B, N, k), dtype=torch.float32, device="cuda")
    outs = [torch.empty((B, N), dtype=torch.int32, device="cuda") for _ in range(4)]
    out_tok = torch.empty((B, N + 1), dtype=torch.int32, device="cuda")
    sample = torch.empty((B, N), dtype=torch.int32, device="cuda")
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    table = t(np.full((V, k), -1, np.int32))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gt.gt_verify_sample_commit(t(logits), t(tokens), t(parent), t(n), t(P), B, N, V, k, 0.9, 5, 2,
                               ids, vals, sample, acc, outs[0], out_tok, outs[1], outs[2], table,
                               err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    gi, gv = np_(ids), np_(vals)
    for b in range(B):
        for v in range(N):
            wi, wv = oracle.vocab_topk(logits[b, v], k)
            assert gi[b, v].tolist() == list(wi), (b, v)
            assert np.array_equal(gv[b, v].view(np.uint32), np.float32(wv).view(np.uint32)), (b, v)
