"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the same seeded
inputs. Indices, trees, masks, top-k, paths, commit indices and the table are compared
bit for bit; attention to the max-abs tolerance of its input precision."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import (TOL, attn_max_err, compare_tree, compare_verify, device_inputs, np_,
                         oracle_tree, run_gpu_step, shape_of)
from tree_speculative_decoding_parent_gb300 import gt
from tree_speculative_decoding_parent_gb300.step import (StepBuffers, run_step, run_tree_build,
                                                         run_tree_phase)
from workload import make_scenario

pytestmark = pytest.mark.gpu

# Reduced vocabularies and prefixes (several KV tiles plus a ragged tail; vocab sizes that
# do and do not divide by 4), with the trees and budgets of each workload unchanged.
SMALL = {
    1: dict(),                                                   # config 1 is small already
    2: dict(V=5000, P=700),
    3: dict(V=4099, P=1333, stream_len=50000),
    4: dict(V=4096, P=(200, 900), B=5, stream_len=50000),
    5: dict(V=5003, P=611),
}


def _full_check(scn, reqs=None, fused=True):
    tree = oracle_tree(scn)
    logits = scn.logits(tree["parent"], tree["tokens"], tree["n_nodes"])
    buf, inp = run_gpu_step(scn, logits, fused=fused)
    assert int(buf.err.item()) == 0
    compare_tree(buf, tree)
    res = oracle.step_verify_phase(tree, logits, scn.table, scn.prefix_len, scn.k)
    compare_verify(buf, res, inp["table"])
    err = attn_max_err(buf, scn, tree, reqs)
    assert err <= TOL[scn.dtype], err
    return buf, tree


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "separate"])
@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5])
def test_step_parity_small(cid, fused):
    _full_check(make_scenario(cid, **SMALL[cid]), fused=fused)


def test_step_parity_nan_kv_tail_and_zero_prefix():
    # cache rows past each request's length hold NaN: they must never reach the result
    _full_check(make_scenario(2, V=5000, P=300, kv_fill="nan"))
    _full_check(make_scenario(1, V=3000, P=0, kv_fill="nan"))
    _full_check(make_scenario(4, V=4096, P=(0, 200), B=3, stream_len=20000, kv_fill="nan"))


def test_step_parity_root_only_trees():
    # keep = 1 and no graft: every tree is its root alone (one query row per head, an empty
    # path, the bonus token only)
    for cid, kw in ((2, dict(V=5000, P=300)), (4, dict(V=4096, P=(0, 200), B=3, stream_len=20000))):
        scn = make_scenario(cid, **kw)
        scn.keep[:] = 1
        scn.R[:] = 0
        if scn.thresh is not None:
            scn.thresh[:] = np.float32(np.inf)
        buf, tree = _full_check(scn)
        assert (np_(buf.n_nodes) == 1).all() and (np_(buf.acc_len) == 0).all()


@pytest.mark.parametrize("cid", [2, 3, 5])
def test_step_parity_full_size(cid):
    _full_check(make_scenario(cid))


def test_step_parity_full_size_batched():
    """Workload 4 at full size: 16 requests, attention compared on every one of them."""
    scn = make_scenario(4)
    _full_check(scn)


def test_repeated_steps_keep_parity():
    """Three steps in a row on the evolving table (each graft reads the last update)."""
    scn = make_scenario(3, V=4099, P=500, stream_len=30000)
    buf = StepBuffers(shape_of(scn))
    table = scn.table.copy()
    for _ in range(3):
        scn.table = table
        tree = oracle_tree(scn)
        logits = scn.logits(tree["parent"], tree["tokens"], tree["n_nodes"])
        inp = device_inputs(scn, logits)
        run_step(buf, inp, scale=scn.scale)
        torch.cuda.synchronize()
        compare_tree(buf, tree)
        res = oracle.step_verify_phase(tree, logits, table, scn.prefix_len, scn.k)
        compare_verify(buf, res, inp["table"])
        table = res["table"]


# ------------------------------------------------------------------------ single kernels


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_vocab_topk_ties_zeros_nan():
    rng = np.random.default_rng(0)
    pool = np.float32([0.0, -0.0, 1.0, -1.0, 2.5, np.inf, -np.inf, np.nan, 1e-30, -1e-30])
    for V, rows, k in ((37, 50, 8), (1000, 20, 16), (4096, 9, 5), (131, 70, 1), (8, 3, 8)):
        x = pool[rng.integers(0, len(pool), size=(rows, V))]
        ids = torch.empty((rows, k), dtype=torch.int32, device="cuda")
        vals = torch.empty((rows, k), dtype=torch.float32, device="cuda")
        gt.gt_vocab_topk(_t(x), rows, V, k, ids, vals)
        torch.cuda.synchronize()
        for r in range(rows):
            ri, rv = oracle.vocab_topk(x[r], k)
            assert np_(ids[r]).tolist() == ri.tolist()
            assert np.array_equal(np_(vals[r]).view(np.uint32), rv.view(np.uint32))


def test_vocab_topk_random_large():
    rng = np.random.default_rng(1)
    for V in (151936, 128256, 32000, 99991):
        x = rng.standard_normal((6, V), dtype=np.float32)
        x[2, 1000:1010] = 9.0  # ties at the top
        ids = torch.empty((6, 8), dtype=torch.int32, device="cuda")
        vals = torch.empty((6, 8), dtype=torch.float32, device="cuda")
        gt.gt_vocab_topk(_t(x), 6, V, 8, ids, vals)
        torch.cuda.synchronize()
        for r in range(6):
            assert np_(ids[r]).tolist() == oracle.vocab_topk(x[r], 8)[0].tolist()


def test_succ_update_duplicates():
    rng = np.random.default_rng(2)
    V, k, B, N = 50, 8, 7, 60
    table = rng.integers(0, V, size=(V, k)).astype(np.int32)
    tokens = rng.integers(0, 12, size=(B, N)).astype(np.int32)   # many shared rows
    topk = rng.integers(0, V, size=(B, N, k)).astype(np.int32)
    n = rng.integers(0, N + 1, size=B).astype(np.int32)
    dt = _t(table)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gt.gt_succ_update(dt, V, k, _t(tokens), _t(topk), _t(n), B, N, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(np_(dt), oracle.succ_update(table, tokens, topk, n))


def test_graft_with_empty_entries():
    rng = np.random.default_rng(3)
    from workload import default_template
    V, k, B, Nmax = 40, 8, 6, 60
    tpar, trank = default_template(52, k)
    for trial in range(5):
        table = rng.integers(-1, V, size=(V, k)).astype(np.int32)
        table[rng.random((V, k)) < 0.3] = -1
        nk = rng.integers(1, 20, size=B).astype(np.int32)
        parent = np.full((B, Nmax), -1, np.int32)
        tokens = np.full((B, Nmax), -1, np.int32)
        for b in range(B):
            parent[b, 1:nk[b]] = [rng.integers(0, v) for v in range(1, nk[b])]
            tokens[b, :nk[b]] = rng.integers(0, V, size=nk[b])
        R = rng.integers(0, 60, size=B).astype(np.int32)
        dp, dtk, dn = _t(parent), _t(tokens), _t(nk)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        gt.gt_graft_expand(dp, dtk, dn, B, Nmax, _t(tpar), _t(trank), 52, _t(R), None, _t(table), V, k,
                           err)
        torch.cuda.synchronize()
        assert err.item() == 0
        for b in range(B):
            p, t, n = oracle.graft_expand(parent[b], tokens[b], int(nk[b]), tpar, trank, int(R[b]),
                                          table, Nmax)
            assert np_(dn)[b] == n
            assert np_(dp)[b].tolist() == p and np_(dtk)[b].tolist() == t


def test_graft_at_anchors_and_bad_anchor():
    """Graft-TAIL: the retrieved tree hangs from anchor[b] (-1 = the last kept node)."""
    rng = np.random.default_rng(13)
    from workload import default_template
    V, k, B, Nmax = 50, 8, 8, 60
    tpar, trank = default_template(52, k)
    for trial in range(4):
        table = rng.integers(0, V, size=(V, k)).astype(np.int32)
        table[rng.random((V, k)) < 0.2] = -1
        nk = rng.integers(1, 24, size=B).astype(np.int32)
        parent = np.full((B, Nmax), -1, np.int32)
        tokens = np.full((B, Nmax), -1, np.int32)
        for b in range(B):
            parent[b, 1:nk[b]] = [rng.integers(0, v) for v in range(1, nk[b])]
            tokens[b, :nk[b]] = rng.integers(0, V, size=nk[b])
        anchor = np.array([-1, 0] + [int(rng.integers(0, nk[b])) for b in range(2, B)], np.int32)
        bad = trial % 2 == 1
        if bad:  # request 3 names a node past its kept tree: it keeps its tree, no graft
            anchor[3] = nk[3]
        R = rng.integers(0, 60, size=B).astype(np.int32)
        dp, dtk, dn = _t(parent), _t(tokens), _t(nk)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        gt.gt_graft_expand(dp, dtk, dn, B, Nmax, _t(tpar), _t(trank), 52, _t(R), _t(anchor),
                           _t(table), V, k, err)
        torch.cuda.synchronize()
        assert err.item() == (gt.GT_ERR_RANGE if bad else 0)
        for b in range(B):
            if bad and b == 3:
                p, t, n = oracle.graft_expand(parent[b], tokens[b], int(nk[b]), tpar, trank, 0,
                                              table, Nmax)
            else:
                p, t, n = oracle.graft_expand(parent[b], tokens[b], int(nk[b]), tpar, trank,
                                              int(R[b]), table, Nmax, int(anchor[b]))
            assert np_(dn)[b] == n
            assert np_(dp)[b].tolist() == p and np_(dtk)[b].tolist() == t


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "separate"])
def test_step_parity_dflash_tail(fused):
    """A 16-token block draft: threshold prune to a prefix, graft at the prefix's tail."""
    scn = make_scenario(6, V=4099, P=777, B=6, stream_len=50000)
    buf, tree = _full_check(scn, fused=fused)
    for b in range(scn.B):
        nk, n = int(tree["n_kept"][b]), int(tree["n_nodes"][b])
        assert tree["parent"][b][:nk].tolist() == list(range(-1, nk - 1))  # a kept prefix
        assert all(tree["parent"][b][v] >= nk - 1 for v in range(nk, n))  # below the tail
    assert len(set(tree["n_kept"].tolist())) > 1  # the thresholds keep prefixes of several lengths


def test_step_parity_dflash_tail_full_size():
    _full_check(make_scenario(6))


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "separate"])
def test_tree_phase_bad_anchor_keeps_the_pruned_tree(fused):
    scn = make_scenario(6, V=3001, P=200, B=3, stream_len=20000)
    nk = oracle_tree(scn)["n_kept"]
    scn.anchor = np.array([-1, nk[1], 0], np.int32)  # request 1: one past its kept tree
    shape = shape_of(scn)
    buf = StepBuffers(shape)
    inp = device_inputs(scn, np.zeros((scn.B, scn.N, scn.V), np.float32))
    (run_tree_build if fused else run_tree_phase)(buf, inp)
    torch.cuda.synchronize()
    assert int(buf.err.item()) == gt.GT_ERR_RANGE
    R = scn.R.copy()
    R[1] = 0
    want = oracle.step_tree_phase(scn.parent_in, scn.tokens_in, scn.score_in, [scn.Nin] * scn.B,
                                  scn.keep, scn.thresh, scn.tpar, scn.trank, R, scn.table,
                                  scn.prefix_len, scn.N, anchor=np.array([-1, 0, 0], np.int32))
    compare_tree(buf, want)


def test_prune_ties_and_threshold():
    rng = np.random.default_rng(4)
    B, Nin, Nout = 9, 300, 64
    parent = np.full((B, Nin), -1, np.int32)
    score = np.zeros((B, Nin), np.float32)
    for b in range(B):
        parent[b, 1:] = [rng.integers(max(0, v - 20), v) for v in range(1, Nin)]
        s = [1.0]
        for v in range(1, Nin):
            s.append(s[parent[b, v]] * rng.choice([0.25, 0.5, 0.75, 1.0]))
        score[b] = s
    tokens = rng.integers(0, 1000, size=(B, Nin)).astype(np.int32)
    keep = rng.integers(1, Nout + 1, size=B).astype(np.int32)
    thresh = np.float32(rng.choice([0.0, 0.01, 0.1, 0.5], size=B))
    outs = [torch.empty((B, Nout), dtype=dt, device="cuda")
            for dt in (torch.int32, torch.int32, torch.float32, torch.int32)]
    n_out = torch.empty(B, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gt.gt_prune_topB(_t(score), _t(parent), _t(tokens), None, B, Nin, _t(keep), _t(thresh), Nout,
                     *outs, n_out, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    for b in range(B):
        p, t, s, o = oracle.prune_topB(score[b], parent[b], tokens[b], Nin, int(keep[b]),
                                       float(thresh[b]))
        m = len(p)
        assert np_(n_out)[b] == m
        assert np_(outs[0])[b, :m].tolist() == p and np_(outs[3])[b, :m].tolist() == o
        assert np_(outs[1])[b, :m].tolist() == t
        assert (np_(outs[0])[b, m:] == -1).all()


def test_device_errors_are_reported():
    scn = make_scenario(1, V=3000, P=64)
    tree = oracle_tree(scn)
    logits = scn.logits(tree["parent"], tree["tokens"], tree["n_nodes"])
    for fused in (True, False):
        # a node whose score exceeds its parent's
        bad = make_scenario(1, V=3000, P=64)
        bad.score_in[0, 200] = 2.0
        buf, _ = run_gpu_step(bad, logits, fused=fused)
        assert buf.err.item() == gt.GT_ERR_NONMONOTONE
        assert buf.n_nodes.item() == 0 and (np_(buf.parent) == -1).all()
        # a parent index that is not smaller than the child's
        bad = make_scenario(1, V=3000, P=64)
        bad.parent_in[0, 17] = 300
        buf, _ = run_gpu_step(bad, logits, fused=fused)
        assert buf.err.item() == gt.GT_ERR_TREE
    # a prefix that does not fit in the cache
    buf = StepBuffers(shape_of(scn))
    inp = device_inputs(scn, logits)
    inp["prefix_len"] = torch.tensor([scn.Lcap], dtype=torch.int32, device="cuda")
    run_step(buf, inp, scale=scn.scale)
    torch.cuda.synchronize()
    assert buf.err.item() == gt.GT_ERR_RANGE
    # host-visible errors raise without launching
    with pytest.raises(gt.GTError):
        gt.gt_vocab_topk(inp["logits"], 1, scn.V, 17, buf.topk_id, buf.topk_val)


# ------------------------------------------------------------------------------ KV commit


def _bits(x: torch.Tensor) -> np.ndarray:
    """Raw element bits of a device tensor (bf16 -> uint16, fp32 -> uint32)."""
    if x.dtype == torch.bfloat16:
        return np_(x.view(torch.int16)).view(np.uint16)
    return np_(x).view(np.uint32)


def _host_bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint16) if a.dtype == np.uint16 else np.ascontiguousarray(a, np.float32).view(np.uint32)


@pytest.mark.parametrize("cid", [1, 2])
def test_kv_commit_after_step(cid):
    scn = make_scenario(cid, **SMALL[cid])
    tree = oracle_tree(scn)
    logits = scn.logits(tree["parent"], tree["tokens"], tree["n_nodes"])
    buf, inp = run_gpu_step(scn, logits)
    res = oracle.step_verify_phase(tree, logits, scn.table, scn.prefix_len, scn.k)
    s = shape_of(scn)
    gt.gt_kv_commit(inp["K"], inp["V"], buf.kv_src, buf.kv_dst, buf.acc_len, s.B, s.N, s.Hkv,
                    s.d, s.Lcap, s.dtype, buf.err)
    torch.cuda.synchronize()
    assert buf.err.item() == 0
    Ke, Ve = oracle.kv_commit(scn.K, scn.Vc, res["kv_src"], res["kv_dst"], res["acc_len"])
    assert np.array_equal(_bits(inp["K"]), _host_bits(Ke))
    assert np.array_equal(_bits(inp["V"]), _host_bits(Ve))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_kv_commit_random_paths_and_bad_requests(dtype):
    rng = np.random.default_rng(11)
    B, Hkv, N, d, Lcap = 9, 3, 64, 128, 300
    P = rng.integers(0, Lcap - N, size=B).astype(np.int32)
    L = rng.integers(0, N, size=B).astype(np.int32)
    L[0] = N - 1                                   # the longest path the buffers hold
    src = np.full((B, N), -1, np.int32)
    dst = np.full((B, N), -1, np.int32)
    for b in range(B):
        # a root path of an N-node tree: node indices increase, path[j] >= j, and
        # consecutive nodes are often adjacent, so destinations overlap later sources
        nodes = np.sort(rng.choice(np.arange(1, N), size=L[b], replace=False))
        path = np.concatenate([[0], nodes])
        src[b, :L[b] + 1] = P[b] + path
        dst[b, :L[b] + 1] = P[b] + np.arange(L[b] + 1)
    bad = [3, 6]
    L[3] = N                                       # accepted length past the path buffer
    src[6, 1] = Lcap + 5                           # a row outside the cache
    x = rng.standard_normal((2, B, Hkv, Lcap, d)).astype(np.float32)
    if dtype == "bf16":
        from workload import f32_to_bf16_bits
        host = [f32_to_bf16_bits(x[0]), f32_to_bf16_bits(x[1])]
        dev = [torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).cuda() for h in host]
    else:
        host = [x[0], x[1]]
        dev = [torch.from_numpy(h.copy()).cuda() for h in host]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gt.gt_kv_commit(dev[0], dev[1], _t(src), _t(dst), _t(L), B, N, Hkv, d, Lcap,
                    gt.GT_BF16 if dtype == "bf16" else gt.GT_F32, err)
    torch.cuda.synchronize()
    assert err.item() == gt.GT_ERR_RANGE
    good = [b for b in range(B) if b not in bad]
    Ke, Ve = oracle.kv_commit(host[0][good], host[1][good], src[good], dst[good], L[good])
    for got, want, orig in ((dev[0], Ke, host[0]), (dev[1], Ve, host[1])):
        g_bits = _bits(got)
        assert np.array_equal(g_bits[good], _host_bits(want))
        assert np.array_equal(g_bits[bad], _host_bits(orig[bad]))   # bad requests untouched


# ------------------------------------------------------------------ attention edge shapes


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_tree_attn_edge_shapes(dtype):
    """Random trees through gt_tree_attn alone, masks from the oracle: a full 64-node mask
    word, single-node trees, zero prefixes, prefixes on and next to 128-key tile edges,
    8 query heads per KV head (512 query rows of one KV head), and more segments than one
    wave of clusters (both schedule paths), and clusters of two, three and four CTAs."""
    from workload import f32_to_bf16_bits
    rng = np.random.default_rng(21)
    cases = [  # B, N, Hq, Hkv, prefixes, nodes per request (None: N)
        (1, 64, 8, 8, [0], None),
        (2, 1, 32, 8, [0, 5], None),
        (3, 64, 16, 2, [127, 128, 129], [64, 33, 1]),
        (2, 40, 4, 4, [1000, 255], [40, 17]),
        # 160 segments: the block-wide schedule
        (20, 9, 16, 8, rng.integers(0, 700, size=20).tolist(), rng.integers(1, 10, size=20).tolist()),
        # 96 segments over 38 clusters of 4 CTAs: the one-warp schedule in several waves
        (12, 49, 64, 8, rng.integers(0, 900, size=12).tolist(), rng.integers(1, 50, size=12).tolist()),
        # three-CTA clusters (257..384 rows), whose third CTA loads nothing and receives every
        # tile by multicast: ragged trees over two requests, and one segment cut into
        # one-tile pieces
        (2, 33, 64, 8, [130, 7], [33, 20]),
        (1, 24, 16, 1, [3000], None),
    ]
    for B, N, Hq, Hkv, P, nn in cases:
        d = 128
        n = np.array(nn if nn else [N] * B, np.int32)
        P = np.array(P, np.int32)
        Lcap = int((P + N).max() + 64) // 64 * 64
        parent = np.full((B, N), -1, np.int32)
        for b in range(B):
            parent[b, 1:n[b]] = [rng.integers(0, v) for v in range(1, n[b])]
        mask = np.zeros((B, N, 1), np.uint64)
        for b in range(B):
            _, _, mask[b] = oracle.tree_mask(parent[b], int(n[b]), int(P[b]), N)
        Q = rng.standard_normal((B, N, Hq, d), dtype=np.float32)
        K = rng.standard_normal((B, Hkv, Lcap, d), dtype=np.float32)
        Vv = rng.standard_normal((B, Hkv, Lcap, d), dtype=np.float32)
        for b in range(B):  # cache rows past each request's length must never be read
            K[b, :, P[b] + n[b]:] = np.nan
            Vv[b, :, P[b] + n[b]:] = np.nan
        if dtype == "bf16":
            hq, hk, hv = (f32_to_bf16_bits(x) for x in (Q, K, Vv))
            dev = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda() for x in (hq, hk, hv)]
            dec = oracle.bf16_to_f64
            O = torch.empty((B, N, Hq, d), dtype=torch.bfloat16, device="cuda")
            gdt = gt.GT_BF16
        else:
            hq, hk, hv = Q, K, Vv
            dev = [_t(x) for x in (Q, K, Vv)]
            dec = lambda a: np.asarray(a, np.float64)  # noqa: E731
            O = torch.empty((B, N, Hq, d), dtype=torch.float32, device="cuda")
            gdt = gt.GT_F32
        wsb = gt.gt_tree_attn_workspace(B, N, Hq, Hkv, d, Lcap)
        ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        scale = 1.0 / np.sqrt(d)
        gt.gt_tree_attn(dev[0], dev[1], dev[2], _t(mask), _t(P), _t(n), B, N, Hq, Hkv, d, Lcap,
                        gdt, scale, O, ws, wsb, err)
        torch.cuda.synchronize()
        assert err.item() == 0
        got = O.float().cpu().numpy().astype(np.float64)
        for b in range(B):
            L = int(P[b] + n[b])
            ref = oracle.tree_attn(dec(hq[b]), dec(hk[b][:, :L]), dec(hv[b][:, :L]), parent[b],
                                   int(n[b]), int(P[b]), scale)
            e = float(np.abs(got[b, :n[b]] - ref).max())
            assert e <= TOL[dtype], (B, N, Hq, Hkv, b, e)
            assert np.all(got[b, n[b]:] == 0.0)


def test_tree_attn_two_cta_cluster_shapes():
    """bf16 shapes with 129..256 query rows per KV head (two-CTA clusters sharing every
    K/V tile by multicast): prefixes on and next to tile edges, a one-node tree whose
    second CTA has no rows, zero prefixes (the tail tile is the only tile), a single
    segment cut into one-tile pieces, and more segments than one wave (long pieces that
    wrap the ring). Cache rows past each request hold NaN."""
    from workload import f32_to_bf16_bits
    rng = np.random.default_rng(33)
    cases = [  # B, N, Hq, Hkv, prefixes, nodes per request (None: N)
        (3, 60, 32, 8, [127, 128, 129], [60, 33, 1]),
        (2, 64, 8, 2, [0, 3], None),
        (1, 17, 8, 1, [4000], None),
        (16, 40, 16, 4, rng.integers(1000, 5000, size=16).tolist(),
         rng.integers(1, 41, size=16).tolist()),
        (24, 33, 32, 8, rng.integers(0, 3500, size=24).tolist(),
         rng.integers(1, 34, size=24).tolist()),
    ]
    for B, N, Hq, Hkv, P, nn in cases:
        assert 128 < (Hq // Hkv) * N <= 256
        d = 128
        n = np.array(nn if nn else [N] * B, np.int32)
        P = np.array(P, np.int32)
        Lcap = int((P + N).max() + 64) // 64 * 64
        parent = np.full((B, N), -1, np.int32)
        for b in range(B):
            parent[b, 1:n[b]] = [rng.integers(0, v) for v in range(1, n[b])]
        mask = np.zeros((B, N, 1), np.uint64)
        for b in range(B):
            _, _, mask[b] = oracle.tree_mask(parent[b], int(n[b]), int(P[b]), N)
        Q = rng.standard_normal((B, N, Hq, d), dtype=np.float32)
        K = rng.standard_normal((B, Hkv, Lcap, d), dtype=np.float32)
        Vv = rng.standard_normal((B, Hkv, Lcap, d), dtype=np.float32)
        for b in range(B):
            K[b, :, P[b] + n[b]:] = np.nan
            Vv[b, :, P[b] + n[b]:] = np.nan
        hq, hk, hv = (f32_to_bf16_bits(x) for x in (Q, K, Vv))
        dev = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda() for x in (hq, hk, hv)]
        O = torch.empty((B, N, Hq, d), dtype=torch.bfloat16, device="cuda")
        wsb = gt.gt_tree_attn_workspace(B, N, Hq, Hkv, d, Lcap)
        ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        scale = 1.0 / np.sqrt(d)
        refs = []
        for b in range(B):
            L = int(P[b] + n[b])
            refs.append(oracle.tree_attn(oracle.bf16_to_f64(hq[b]), oracle.bf16_to_f64(hk[b][:, :L]),
                                         oracle.bf16_to_f64(hv[b][:, :L]), parent[b], int(n[b]),
                                         int(P[b]), scale))
        # twice on one workspace (the second call finds what the first left there) and into
        # an output filled with NaN: every output element is written
        for _ in range(2):
            O.fill_(float("nan"))
            gt.gt_tree_attn(dev[0], dev[1], dev[2], _t(mask), _t(P), _t(n), B, N, Hq, Hkv, d,
                            Lcap, gt.GT_BF16, scale, O, ws, wsb, err)
            torch.cuda.synchronize()
            assert err.item() == 0
            got = O.float().cpu().numpy().astype(np.float64)
            for b in range(B):
                e = float(np.abs(got[b, :n[b]] - refs[b]).max())
                assert e <= TOL["bf16"], (B, N, Hq, Hkv, b, e)
                assert np.all(got[b, n[b]:] == 0.0)


def test_tree_attn_more_segments_than_clusters():
    """Launches with as many segments as resident clusters or more (pieces in several
    waves, longest first): requests of very unequal length (the long one's segments cut
    into several pieces, merged by the combine, the short ones' single pieces stored
    directly), and invalid requests among valid ones (their rows zero, GT_ERR_RANGE
    reported)."""
    rng = np.random.default_rng(57)
    cases = [  # B, N, Hq, Hkv, prefixes, nodes per request, expected error
        (5, 60, 64, 8, [8000, 100, 100, 100, 100], [60, 7, 1, 30, 60], 0),
        (6, 60, 64, 8, [300, 300, 4000, 300, 0, 2000], [60, 0, 60, 61, 5, 60], gt.GT_ERR_RANGE),
        (40, 20, 16, 4, rng.integers(0, 3000, size=40).tolist(),
         rng.integers(1, 21, size=40).tolist(), 0),
        # two-CTA clusters, one-warp schedule: 32 requests (pieces ordered by length) and
        # 40 requests (more than 32: pieces in segment order)
        (32, 40, 16, 4, rng.integers(0, 4000, size=32).tolist(),
         rng.integers(1, 41, size=32).tolist(), 0),
        (40, 20, 16, 2, rng.integers(0, 3000, size=40).tolist(),
         rng.integers(1, 21, size=40).tolist(), 0),
    ]
    for B, N, Hq, Hkv, P, nn, want in cases:
        valid = [1 <= v <= N for v in nn]
        a, refs, n = _random_attn_case(rng, B, N, Hq, Hkv, P,
                                        [v if ok else 1 for v, ok in zip(nn, valid)], "bf16")
        a["n"] = _t(np.array(nn, np.int32))
        wsb = gt.gt_tree_attn_workspace(B, N, Hq, Hkv, 128, a["Lcap"])
        ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        gt.gt_tree_attn(a["Q"], a["K"], a["V"], a["mask"], a["P"], a["n"], B, N, Hq, Hkv, 128,
                        a["Lcap"], a["dt"], a["scale"], a["O"], ws, wsb, err)
        torch.cuda.synchronize()
        assert err.item() == want, (B, N, Hq, Hkv, err.item())
        got = a["O"].float().cpu().numpy().astype(np.float64)
        for b in range(B):
            if not valid[b]:
                assert np.all(got[b] == 0.0), (B, b)
                continue
            e = float(np.abs(got[b, :n[b]] - refs[b]).max())
            assert e <= TOL["bf16"], (B, N, Hq, Hkv, b, e)
            assert np.all(got[b, n[b]:] == 0.0)


def _random_attn_case(rng, B, N, Hq, Hkv, P, nn, dtype):
    """Random trees and NaN-tailed caches for gt_tree_attn alone; returns the device
    arguments and the oracle's output per request."""
    from workload import f32_to_bf16_bits
    d = 128
    n = np.array(nn if nn else [N] * B, np.int32)
    P = np.array(P, np.int32)
    Lcap = int((P + N).max() + 64) // 64 * 64
    parent = np.full((B, N), -1, np.int32)
    for b in range(B):
        parent[b, 1:n[b]] = [rng.integers(0, v) for v in range(1, n[b])]
    mask = np.zeros((B, N, 1), np.uint64)
    for b in range(B):
        _, _, mask[b] = oracle.tree_mask(parent[b], int(n[b]), int(P[b]), N)
    Q = rng.standard_normal((B, N, Hq, d), dtype=np.float32)
    K = rng.standard_normal((B, Hkv, Lcap, d), dtype=np.float32)
    Vv = rng.standard_normal((B, Hkv, Lcap, d), dtype=np.float32)
    for b in range(B):
        K[b, :, P[b] + n[b]:] = np.nan
        Vv[b, :, P[b] + n[b]:] = np.nan
    if dtype == "bf16":
        hq, hk, hv = (f32_to_bf16_bits(x) for x in (Q, K, Vv))
        dev = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda() for x in (hq, hk, hv)]
        dec, odt, gdt = oracle.bf16_to_f64, torch.bfloat16, gt.GT_BF16
    else:
        hq, hk, hv = Q, K, Vv
        dev = [_t(x) for x in (Q, K, Vv)]
        dec, odt, gdt = (lambda a: np.asarray(a, np.float64)), torch.float32, gt.GT_F32
    scale = 1.0 / np.sqrt(d)
    refs = []
    for b in range(B):
        L = int(P[b] + n[b])
        refs.append(oracle.tree_attn(dec(hq[b]), dec(hk[b][:, :L]), dec(hv[b][:, :L]), parent[b],
                                     int(n[b]), int(P[b]), scale))
    args = dict(Q=dev[0], K=dev[1], V=dev[2], mask=_t(mask), P=_t(P), n=_t(n), B=B, N=N, Hq=Hq,
                Hkv=Hkv, d=d, Lcap=Lcap, dt=gdt, scale=scale,
                O=torch.full((B, N, Hq, d), float("nan"), dtype=odt, device="cuda"))
    return args, refs, n


def _check_attn_out(a, refs, n, dtype, tag):
    got = a["O"].float().cpu().numpy().astype(np.float64)
    for b in range(a["B"]):
        e = float(np.abs(got[b, :n[b]] - refs[b]).max())
        assert e <= TOL[dtype], (tag, b, e)
        assert np.all(got[b, n[b]:] == 0.0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_tree_attn_gqa_ratios_not_dividing_128(dtype):
    """Query heads per KV head of 3, 5, 6, 7 and 12: a node's heads straddle the 128-row
    M-tiles of the tcgen05 kernel (bf16), in clusters of two, three and four CTAs."""
    rng = np.random.default_rng(41)
    cases = [  # B, N, Hq, Hkv, prefixes, nodes per request (None: N)
        (2, 60, 24, 8, [500, 129], [60, 31]),      # g = 3, 180 rows
        (2, 50, 40, 8, [128, 1], [50, 9]),         # g = 5, 250 rows
        (1, 64, 6, 1, [300], None),                # g = 6, 384 rows
        (1, 64, 7, 1, [700], None),                # g = 7, 448 rows
        (3, 20, 36, 3, [1000, 2, 64], [20, 1, 13]),  # g = 12, 240 rows
        (2, 42, 12, 1, [260, 0], [42, 5]),         # g = 12, 504 rows
    ]
    for B, N, Hq, Hkv, P, nn in cases:
        a, refs, n = _random_attn_case(rng, B, N, Hq, Hkv, P, nn, dtype)
        wsb = gt.gt_tree_attn_workspace(B, N, Hq, Hkv, 128, a["Lcap"])
        ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        gt.gt_tree_attn(a["Q"], a["K"], a["V"], a["mask"], a["P"], a["n"], B, N, Hq, Hkv, 128,
                        a["Lcap"], a["dt"], a["scale"], a["O"], ws, wsb, err)
        torch.cuda.synchronize()
        assert err.item() == 0
        _check_attn_out(a, refs, n, dtype, (B, N, Hq, Hkv))


def test_tree_attn_refuses_memory_of_other_places():
    """Q, K, V and O must be device memory of the current device: host-pinned and pageable
    host arrays are refused on the host with GT_ERR_ARG and nothing is launched (the output
    and the error word keep their contents)."""
    rng = np.random.default_rng(5)
    a, refs, n = _random_attn_case(rng, 1, 20, 8, 2, [300], None, "bf16")
    wsb = gt.gt_tree_attn_workspace(1, 20, 8, 2, 128, a["Lcap"])
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # host arrays go in as raw addresses (the binding itself takes CUDA tensors only)
    pinned_K = a["K"].cpu().pin_memory()
    pageable_V = a["V"].cpu()
    pinned_O = a["O"].cpu().pin_memory()
    sentinel = a["O"].clone()
    for name, q, k, v, o in (("K", a["Q"], pinned_K.data_ptr(), a["V"], a["O"]),
                             ("V", a["Q"], a["K"], pageable_V.data_ptr(), a["O"]),
                             ("O", a["Q"], a["K"], a["V"], pinned_O.data_ptr())):
        with pytest.raises(gt.GTError) as ei:
            gt.gt_tree_attn(q, k, v, a["mask"], a["P"], a["n"], 1, 20, 8, 2, 128, a["Lcap"],
                            gt.GT_BF16, a["scale"], o, ws, wsb, err)
        assert ei.value.status == gt.GT_ERR_ARG
        assert name in gt.last_error() and "not device memory" in gt.last_error()
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(a["O"].isnan(), sentinel.isnan())  # untouched: still all NaN
    # the same call on device memory runs and matches the oracle
    gt.gt_tree_attn(a["Q"], a["K"], a["V"], a["mask"], a["P"], a["n"], 1, 20, 8, 2, 128,
                    a["Lcap"], gt.GT_BF16, a["scale"], a["O"], ws, wsb, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    _check_attn_out(a, refs, n, "bf16", "device memory")


@pytest.mark.parametrize("R", [60, 180])
def test_tree_build_grafts_large_templates(R):
    """The fused tree build retrieves the graft on its extra warp while the prune runs; with
    60 template nodes a lane holds up to two of them in registers, with 180 the warp loops
    over them.
    Random draft trees (monotone scores), empty table entries, a root-only request; the
    result against the oracle's prune -> graft -> mask. Then out-of-range table entries
    report GT_ERR_TREE and are retrieved as empty; a bad template entry among a request's
    fitting nodes, or a bad root token, reports GT_ERR_TREE and keeps that request's pruned
    tree alone, while a bad entry past a request's fitting nodes leaves its graft as it is."""
    from workload import default_template
    rng = np.random.default_rng(R)
    V, k, B, Nin, N = 300, 8, 3, 256, 200
    tpar, trank = default_template(R, k)
    table = rng.integers(0, V, size=(V, k)).astype(np.int32)
    table[rng.random((V, k)) < 0.25] = -1
    parent_in = np.full((B, Nin), -1, np.int32)
    tokens_in = rng.integers(0, V, size=(B, Nin)).astype(np.int32)
    score_in = np.ones((B, Nin), np.float32)
    for b in range(B):
        for v in range(1, Nin):
            p = int(rng.integers(0, v))
            parent_in[b, v] = p
            score_in[b, v] = np.float32(score_in[b, p] * rng.uniform(0.3, 0.99))
    keep = np.array([10, 20, 1], np.int32)
    Rv = np.array([R, R - 7, R], np.int32)
    prefix = np.array([100, 0, 5000], np.int32)
    W = (N + 63) // 64

    def run(tab, trk=trank, toks=tokens_in):
        outs = dict(parent=torch.empty((B, N), dtype=torch.int32, device="cuda"),
                    tokens=torch.empty((B, N), dtype=torch.int32, device="cuda"),
                    score=torch.empty((B, N), dtype=torch.float32, device="cuda"),
                    old_idx=torch.empty((B, N), dtype=torch.int32, device="cuda"),
                    n_nodes=torch.empty((B,), dtype=torch.int32, device="cuda"),
                    depth=torch.empty((B, N), dtype=torch.int32, device="cuda"),
                    pos=torch.empty((B, N), dtype=torch.int32, device="cuda"),
                    mask=torch.empty((B, N, W), dtype=torch.int64, device="cuda"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        gt.gt_tree_build(_t(score_in), _t(parent_in), _t(toks), None, B, Nin, _t(keep), None,
                         _t(tpar), _t(trk), R, _t(Rv), None, _t(tab), V, k, _t(prefix), N,
                         outs["parent"], outs["tokens"], outs["score"], outs["old_idx"],
                         outs["n_nodes"], outs["depth"], outs["pos"], outs["mask"], err)
        torch.cuda.synchronize()
        return type("Out", (), outs), int(err.item())

    got, err = run(table)
    assert err == 0
    want = oracle.step_tree_phase(parent_in, tokens_in, score_in, [Nin] * B, keep, None, tpar,
                                  trank, Rv, table, prefix, N)
    compare_tree(got, want)
    assert int(np_(got.n_nodes)[0]) > 10 + R // 4  # the graft did fill slots
    # out-of-range entries: reported, and retrieved as empty (the oracle's -1)
    bad = table.copy()
    hit = rng.random((V, k)) < 0.05
    bad[hit] = V + 3
    got, err = run(bad)
    assert err == gt.GT_ERR_TREE
    clean = bad.copy()
    clean[hit] = -1
    want = oracle.step_tree_phase(parent_in, tokens_in, score_in, [Nin] * B, keep, None, tpar,
                                  trank, Rv, clean, prefix, N)
    compare_tree(got, want)
    # bad template entries: inside every request's fitting nodes, then past request 1's
    for u_bad, graft in ((5, [0, 0, 0]), (R - 1, [0, R - 7, 0])):
        trk = np.array(trank, np.int32).copy()
        trk[u_bad] = k  # a rank outside the table row
        got, err = run(table, trk=trk)
        assert err == gt.GT_ERR_TREE, u_bad
        want = oracle.step_tree_phase(parent_in, tokens_in, score_in, [Nin] * B, keep, None, tpar,
                                      trank, np.array(graft, np.int32), table, prefix, N)
        compare_tree(got, want)
    # a root token outside the vocabulary: request 1 keeps its pruned tree alone
    toks = tokens_in.copy()
    toks[1, 0] = V + 1
    got, err = run(table, toks=toks)
    assert err == gt.GT_ERR_TREE
    # (the oracle refuses the bad token outright: its trees with the clean token and no graft
    # for request 1, whose root token is copied as given)
    want = oracle.step_tree_phase(parent_in, tokens_in, score_in, [Nin] * B, keep, None, tpar,
                                  trank, np.array([R, 0, R], np.int32), table, prefix, N)
    want["tokens"][1, 0] = V + 1
    compare_tree(got, want)


def _select_stop(scores, K):
    """Where the radix select of the prune settles for the given candidate scores (host model
    of its stop rule, used only to check that the cases below reach every stop): the pass
    (1-4) after which the K-th largest key's digit bucket is taken whole, 5 when the final
    tie count decides, 0 when no selection is needed."""
    b = np.asarray(scores, np.float32).view(np.uint32).astype(np.uint64)
    b = np.where(b == 0x80000000, 0, b)
    key = np.where(b & 0x80000000, ~b & 0xFFFFFFFF, b | 0x80000000)
    if K <= 0 or len(key) <= K:
        return 0
    prefix, kr = 0, K
    for p, shift in enumerate((24, 16, 8, 0), 1):
        sel = key if p == 1 else key[(key >> (shift + 8)) == (prefix >> (shift + 8))]
        digits = (sel >> shift) & 255
        acc = 0
        for d in range(255, -1, -1):
            c = int((digits == d).sum())
            if acc + c >= kr:
                prefix |= d << shift
                kr -= acc
                if c == kr:
                    return p
                break
            acc += c
    return 5


def test_prune_select_stops_at_every_pass():
    """Keys built so that the prune's radix select settles after each of its four passes or
    only through the final tie count, for K from 1 to 200: star trees (every node a child of
    the root, so any scores are monotone), gt_prune_topB and the fused gt_tree_build against
    the oracle's best-first prune."""
    rng = np.random.default_rng(21)
    Nin, Nout = 400, 256
    n = Nin - 1
    families = {
        "spread": lambda: np.float32(10.0 ** rng.uniform(-30, 30, n)),
        "one_octave": lambda: np.float32(1.0 + rng.random(n)),
        "shared_16_bits": lambda: np.float32(1.0 + rng.integers(0, 4096, n) * 2.0 ** -20),
        "shared_24_bits": lambda: np.float32(1.0 + rng.integers(0, 128, n) * 2.0 ** -23),
        "ties": lambda: np.float32(rng.choice([0.5, 0.25, 0.125], n)),
    }
    cases = []
    for name, gen in families.items():
        for K in (1, 7, 23, 62, 200):
            cases.append((name, K, gen()))
    stops = {_select_stop(s, K - 1) for _, K, s in cases}
    assert {1, 2, 3, 4, 5} <= stops, stops
    B = len(cases)
    parent = np.zeros((B, Nin), np.int32)
    parent[:, 0] = -1
    score = np.ones((B, Nin), np.float32)
    for b, (_, _, s) in enumerate(cases):
        score[b, 1:] = s
    tokens = rng.integers(0, 1000, size=(B, Nin)).astype(np.int32)
    keep = np.array([K for _, K, _ in cases], np.int32)
    outs = [torch.empty((B, Nout), dtype=dt, device="cuda")
            for dt in (torch.int32, torch.int32, torch.float32, torch.int32)]
    n_out = torch.empty(B, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gt.gt_prune_topB(_t(score), _t(parent), _t(tokens), None, B, Nin, _t(keep), None, Nout, *outs,
                     n_out, err)
    # the fused build with no template: prune, then mask
    W = (Nout + 63) // 64
    f = dict(parent=torch.empty((B, Nout), dtype=torch.int32, device="cuda"),
             tokens=torch.empty((B, Nout), dtype=torch.int32, device="cuda"),
             score=torch.empty((B, Nout), dtype=torch.float32, device="cuda"),
             old_idx=torch.empty((B, Nout), dtype=torch.int32, device="cuda"),
             n_nodes=torch.empty((B,), dtype=torch.int32, device="cuda"),
             depth=torch.empty((B, Nout), dtype=torch.int32, device="cuda"),
             pos=torch.empty((B, Nout), dtype=torch.int32, device="cuda"),
             mask=torch.empty((B, Nout, W), dtype=torch.int64, device="cuda"))
    table = np.zeros((1000, 8), np.int32)
    gt.gt_tree_build(_t(score), _t(parent), _t(tokens), None, B, Nin, _t(keep), None, None, None, 0,
                     _t(np.zeros(B, np.int32)), None, _t(table), 1000, 8,
                     _t(np.zeros(B, np.int32)), Nout, f["parent"], f["tokens"], f["score"],
                     f["old_idx"], f["n_nodes"], f["depth"], f["pos"], f["mask"], err)
    torch.cuda.synchronize()
    assert err.item() == 0
    for b, (name, K, _) in enumerate(cases):
        p, t, s, o = oracle.prune_topB(score[b], parent[b], tokens[b], Nin, K)
        m = len(p)
        for got_n, got_p, got_o in ((n_out, outs[0], outs[3]), (f["n_nodes"], f["parent"], f["old_idx"])):
            assert np_(got_n)[b] == m, (name, K)
            assert np_(got_o)[b, :m].tolist() == o, (name, K)
            assert np_(got_p)[b, :m].tolist() == p, (name, K)


@pytest.mark.parametrize("fused_sampler", [False, True], ids=["topk", "draws+topk"])
def test_vocab_topk_candidate_counts_of_every_selection_tier(fused_sampler):
    """Rows of 151,936 logits, each CTA's part (8 per row) holding c copies of 5.0, a value no
    other element reaches: the CTA's threshold is 5.0 and its candidates are those c copies,
    so c picks the selection tier (ranked up to 128, warp rounds over 8 or 16 candidates per
    lane up to 256 or 512, the exact per-thread lists beyond). The top-k (the 8 lowest
    indices holding 5.0) against the oracle, from gt_vocab_topk and from the sampler's pass
    of gt_verify_sample_commit."""
    rng = np.random.default_rng(31)
    V, k, CL = 151936, 8, 8
    counts = [40, 100, 128, 129, 200, 256, 257, 400, 512, 513, 700]
    rows = len(counts)
    x = (rng.standard_normal((rows, V)) * 0.5).astype(np.float32)
    V4 = V // 4
    for r, c in enumerate(counts):
        for part in range(CL):
            b, e = 4 * (V4 * part // CL), 4 * (V4 * (part + 1) // CL)
            x[r, rng.choice(np.arange(b, e), size=c, replace=False)] = 5.0
    ids = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
    vals = torch.empty((rows, k), dtype=torch.float32, device="cuda")
    if not fused_sampler:
        gt.gt_vocab_topk(_t(x), rows, V, k, ids, vals)
    else:
        # one request of `rows` nodes (a chain), the draws at T = 1.0 beside the top-k
        B, N = 1, rows
        parent = np.arange(-1, N - 1, dtype=np.int32)[None]
        tokens = rng.integers(0, V, size=(B, N)).astype(np.int32)
        outs = [torch.empty((B, N), dtype=torch.int32, device="cuda") for _ in range(4)]
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        gt.gt_verify_sample_commit(_t(x[None]), _t(tokens), _t(parent),
                                   _t(np.array([N], np.int32)), _t(np.zeros(1, np.int32)), B, N,
                                   V, k, 1.0, 3, 1, ids, vals,
                                   torch.empty((B, N), dtype=torch.int32, device="cuda"),
                                   torch.empty((B,), dtype=torch.int32, device="cuda"), outs[0],
                                   torch.empty((B, N + 1), dtype=torch.int32, device="cuda"),
                                   outs[1], outs[2], _t(np.full((V, k), -1, np.int32)), err)
    torch.cuda.synchronize()
    gi, gv = np_(ids), np_(vals)
    for r in range(rows):
        wi, wv = oracle.vocab_topk(x[r], k)
        assert gi[r].tolist() == wi.tolist(), counts[r]
        assert np.array_equal(gv[r].view(np.uint32), wv.view(np.uint32)), counts[r]
