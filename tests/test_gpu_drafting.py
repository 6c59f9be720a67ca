"""GPU parity of the drafting calls (frontier selection, n-gram drafter, attach) through the
C ABI against the oracle, step by step, bit for bit."""
import numpy as np
import pytest
import torch

from oracle.drafting import frontier_select, ngram_children, tree_attach
from tree_speculative_decoding_parent_gb300 import gt
from workload import make_draft_scenario

pytestmark = pytest.mark.gpu


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _np(x):
    return x.detach().cpu().numpy()


class OracleTrees:
    def __init__(self, ds):
        B, N = len(ds.root), ds.Nmax
        self.ds = ds
        self.parent = [[-1] * N for _ in range(B)]
        self.tokens = [[int(ds.root[b])] + [-1] * (N - 1) for b in range(B)]
        self.score = [np.float32([1.0] + [0.0] * (N - 1)) for _ in range(B)]
        self.n = [1] * B
        self.first_new = [0] * B
        self.visited = [[0] * N for _ in range(B)]

    def step(self, mid: bool):
        ds, out = self.ds, []
        for b in range(len(self.n)):
            if mid:
                front, self.visited[b] = frontier_select(self.score[b], self.n[b], ds.W,
                                                         visited=self.visited[b])
            else:
                front, _ = frontier_select(self.score[b], self.n[b], ds.W,
                                           pool_lo=self.first_new[b])
            kids = [ngram_children(ds.hist[b], int(ds.hist_len[b]), ds.cache_id[b], ds.cache_p[b],
                                   self.parent[b], self.tokens[b], f, ds.q_max, ds.m)
                    for f in front]
            par, tok, sc, n2, first = tree_attach(self.parent[b], self.tokens[b], self.score[b],
                                                  self.n[b], ds.Nmax, front,
                                                  [k[0] for k in kids], [k[1] for k in kids])
            self.parent[b], self.tokens[b], self.score[b] = par, tok, sc
            self.n[b], self.first_new[b] = n2, first
            out.append((front, kids))
        return out


class GpuTrees:
    def __init__(self, ds):
        B, N = len(ds.root), ds.Nmax
        self.ds, self.B = ds, B
        par = np.full((B, N), -1, np.int32)
        tok = np.full((B, N), -1, np.int32)
        tok[:, 0] = ds.root
        sc = np.zeros((B, N), np.float32)
        sc[:, 0] = 1.0
        self.parent, self.tokens, self.score = _t(par), _t(tok), _t(sc)
        self.n = _t(np.ones(B, np.int32))
        self.first_new = _t(np.zeros(B, np.int32))
        self.visited = torch.zeros((B, N), dtype=torch.uint8, device="cuda")
        self.hist, self.hist_len = _t(ds.hist), _t(ds.hist_len)
        self.cache_id, self.cache_p = _t(ds.cache_id), _t(ds.cache_p)
        self.frontier = torch.empty((B, ds.W), dtype=torch.int32, device="cuda")
        self.n_frontier = torch.empty(B, dtype=torch.int32, device="cuda")
        self.child_id = torch.empty((B, ds.W, ds.m), dtype=torch.int32, device="cuda")
        self.child_p = torch.empty((B, ds.W, ds.m), dtype=torch.float32, device="cuda")
        self.match = torch.empty((B, ds.W, 2), dtype=torch.int32, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step(self, mid: bool):
        ds, B, N = self.ds, self.B, self.ds.Nmax
        gt.gt_frontier_select(self.score, self.n, B, N, None if mid else self.first_new,
                              self.visited if mid else None, ds.W, self.frontier,
                              self.n_frontier, self.err)
        gt.gt_ngram_draft(self.hist, self.hist_len, B, ds.hist.shape[1], self.cache_id,
                          self.cache_p, ds.m, self.parent, self.tokens, self.n, N, self.frontier,
                          self.n_frontier, ds.W, ds.q_max, self.child_id, self.child_p,
                          self.match, self.err)
        gt.gt_tree_attach(self.parent, self.tokens, self.score, self.n, B, N, self.frontier,
                          self.n_frontier, ds.W, self.child_id, self.child_p, ds.m, ds.V,
                          self.first_new, self.err)
        torch.cuda.synchronize()


def _grow_and_compare(ds, schedule):
    o, g = OracleTrees(ds), GpuTrees(ds)
    for mid in schedule:
        want = o.step(bool(mid))
        g.step(bool(mid))
        assert int(g.err.item()) == 0
        fr, nf = _np(g.frontier), _np(g.n_frontier)
        cid, cp, mt = _np(g.child_id), _np(g.child_p), _np(g.match)
        for b, (front, kids) in enumerate(want):
            assert nf[b] == len(front) and fr[b, :nf[b]].tolist() == front
            assert np.all(fr[b, nf[b]:] == -1)
            for w, (ids, probs, pos, q) in enumerate(kids):
                assert cid[b, w].tolist() == ids.tolist(), (b, w)
                assert np.array_equal(cp[b, w].view(np.uint32), probs.view(np.uint32))
                assert mt[b, w].tolist() == [pos, q]
        assert _np(g.n).tolist() == o.n and _np(g.first_new).tolist() == o.first_new
        assert _np(g.parent).tolist() == o.parent and _np(g.tokens).tolist() == o.tokens
        assert np.array_equal(_np(g.score).view(np.uint32), np.stack(o.score).view(np.uint32))
        if any(schedule):
            assert _np(g.visited).astype(int).tolist() == o.visited
    return o


def test_ngram_steps_match_oracle():
    ds = make_draft_scenario(B=3, L=4096, V=5000, seed=11)
    o = _grow_and_compare(ds, [0, 1, 0, 1, 0])
    assert min(o.n) > 50  # the tree did grow


def test_ngram_small_vocab_long_keys_and_capacity():
    ds = make_draft_scenario(B=2, L=3000, V=50, m=4, W=16, q_max=8, Nmax=128, seed=3)
    o = _grow_and_compare(ds, [0, 0, 1, 0, 1, 0])
    assert max(o.n) == 128  # growth stopped at the capacity


def test_ngram_ragged_and_empty_histories():
    ds = make_draft_scenario(B=3, L=2000, V=300, seed=5)
    ds.hist_len[1] = 777
    ds.hist_len[2] = 0  # nothing to match: no children, the tree stays the root
    o = _grow_and_compare(ds, [0, 1, 0])
    assert o.n[2] == 1


def test_drafting_errors_are_reported():
    ds = make_draft_scenario(B=2, L=500, V=300, seed=2)
    g = GpuTrees(ds)
    g.step(False)
    g.frontier[1, 0] = 999  # not a node of request 1
    g.n_frontier[1] = 1
    gt.gt_tree_attach(g.parent, g.tokens, g.score, g.n, 2, ds.Nmax, g.frontier, g.n_frontier,
                      ds.W, g.child_id, g.child_p, ds.m, ds.V, g.first_new, g.err)
    torch.cuda.synchronize()
    assert int(g.err.item()) == gt.GT_ERR_RANGE
    with pytest.raises(gt.GTError):  # both pools given
        gt.gt_frontier_select(g.score, g.n, 2, ds.Nmax, g.first_new, g.visited, ds.W,
                              g.frontier, g.n_frontier, g.err)


@pytest.mark.parametrize("mid", [False, True])
def test_frontier_with_nan_signed_zeros_infinities_and_ties(mid):
    """gt_frontier_select against the oracle on pools full of the values whose order the
    rule fixes: NaN last (by index), +0.0 equal to -0.0, +-inf, ties to the smaller index."""
    rng = np.random.default_rng(17 + mid)
    B, N, W = 6, 1024, 64
    specials = np.float32([float("nan"), -float("nan"), 0.0, -0.0, float("inf"),
                           -float("inf"), 0.5, 0.25, 1e-30])
    n = np.array([1, 5, 64, 300, 1000, 1024], np.int32)
    score = np.where(rng.random((B, N)) < 0.5, rng.choice(specials, size=(B, N)),
                     np.float32(rng.integers(-2, 3, size=(B, N)) / 8)).astype(np.float32)
    lo = np.array([0, 2, 10, 0, 900, 1023], np.int32)
    nfr = torch.empty(B, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for Wc in (1, 10, W):
        fr = torch.empty((B, Wc), dtype=torch.int32, device="cuda")  # [B][W] of this call
        vis = rng.integers(0, 2, size=(B, N)).astype(np.uint8)  # a fresh unvisited pool
        dvis = _t(vis)
        gt.gt_frontier_select(_t(score), _t(n), B, N, None if mid else _t(lo),
                              dvis if mid else None, Wc, fr, nfr, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got, gn = _np(fr), _np(nfr)
        for b in range(B):
            if mid:
                want, new_vis = frontier_select(score[b], int(n[b]), Wc, visited=vis[b].tolist())
            else:
                want, new_vis = frontier_select(score[b], int(n[b]), Wc, pool_lo=int(lo[b]))
            assert gn[b] == len(want) and got[b, :gn[b]].tolist() == want, (b, Wc)
            assert np.all(got[b, gn[b]:Wc] == -1)
            if mid:
                assert _np(dvis)[b].tolist() == new_vis
