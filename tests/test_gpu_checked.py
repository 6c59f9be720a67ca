"""The checked flavour of the library (libgt_check.so, -DGT_CHECK=1) and guard bands around
every output buffer of the default library.

A checked build reports inputs the method excludes but the kernels tolerate (a verified token
outside the vocabulary, a NaN logit, a mask row without its own node) through the error word,
without trapping; the default build runs the same inputs without a report. Guard bands of a
known byte pattern before and after every output buffer must survive a whole step (both step
forms, T > 0, the KV commit): no kernel writes outside its outputs."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import device_inputs, np_, oracle_tree, shape_of
from tree_speculative_decoding_parent_gb300 import build, gt
from tree_speculative_decoding_parent_gb300.step import (StepBuffers, run_kv_commit, run_step,
                                                         run_tree_build)
from workload import make_scenario

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def chk():
    build.build(check=True)
    return gt.load_checked()


def _ptr(x):
    return None if x is None else (x if isinstance(x, int) else x.data_ptr())


def _call(lib, name, *args):
    stream = torch.cuda.current_stream().cuda_stream
    return getattr(lib, name)(*[_ptr(a) if (a is None or torch.is_tensor(a)) else a
                                for a in args], stream)


def _verify(lib, buf, inp, s, tokens, logits, err):
    return _call(lib, "gt_verify_greedy", logits, tokens, buf.parent, buf.n_nodes,
                 inp["prefix_len"], s.B, s.N, s.V, s.k, buf.topk_id, buf.topk_val, buf.acc_len,
                 buf.path, buf.out_tok, buf.kv_src, buf.kv_dst, err)


def test_checked_build_reports_out_of_range_token(chk):
    scn = make_scenario(2, V=3000, P=300)
    tree = oracle_tree(scn)
    logits = scn.logits(tree["parent"], tree["tokens"], tree["n_nodes"])
    s = shape_of(scn)
    buf = StepBuffers(s)
    inp = device_inputs(scn, logits)
    run_tree_build(buf, inp)
    torch.cuda.synchronize()
    bad = buf.tokens.clone()
    bad[0, 5] = scn.V  # one past the vocabulary
    for lib, want in ((gt.load(), gt.GT_OK), (chk, gt.GT_ERR_TREE)):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _verify(lib, buf, inp, s, bad, inp["logits"], err) == gt.GT_OK
        torch.cuda.synchronize()
        assert int(err.item()) == want
    # the default build treats the token as one that matches no argmax: as the oracle does
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _verify(gt.load(), buf, inp, s, bad, inp["logits"], err)
    torch.cuda.synchronize()
    n = int(tree["n_nodes"][0])
    am = np.array([oracle.vocab_topk(logits[0, v], 1)[0][0] for v in range(s.N)], np.int32)
    r = oracle.verify_greedy(np_(bad)[0], tree["parent"][0], n, am, int(scn.prefix_len[0]))
    L = r["acc_len"]
    assert int(np_(buf.acc_len)[0]) == L
    for key in ("path", "out_tok", "kv_src", "kv_dst"):
        assert np_(getattr(buf, key))[0, :L + 1].tolist() == list(r[key]), key


def test_checked_build_reports_nan_logit_and_bad_mask_row(chk):
    scn = make_scenario(2, V=3000, P=300)
    tree = oracle_tree(scn)
    logits = scn.logits(tree["parent"], tree["tokens"], tree["n_nodes"])
    s = shape_of(scn)
    buf = StepBuffers(s)
    inp = device_inputs(scn, logits)
    run_tree_build(buf, inp)
    torch.cuda.synchronize()
    nan_logits = inp["logits"].clone()
    nan_logits[0, 3, 1234] = float("nan")
    for lib, want in ((gt.load(), gt.GT_OK), (chk, gt.GT_ERR_VALUE)):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        _verify(lib, buf, inp, s, buf.tokens, nan_logits, err)
        torch.cuda.synchronize()
        assert int(err.item()) == want
    mask = buf.mask.clone()
    mask[0, 7] &= ~(1 << 7)  # row 7 without its own node
    ws = torch.zeros(buf.ws_bytes, dtype=torch.uint8, device="cuda")
    for lib, want in ((gt.load(), gt.GT_OK), (chk, gt.GT_ERR_TREE)):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _call(lib, "gt_tree_attn", inp["Q"], inp["K"], inp["V"], mask, inp["prefix_len"],
                     buf.n_nodes, s.B, s.N, s.Hq, s.Hkv, s.d, s.Lcap, s.dtype, scn.scale,
                     buf.O, ws, buf.ws_bytes, err) == gt.GT_OK
        torch.cuda.synchronize()
        assert int(err.item()) == want


GUARD = 4096          # bytes before and after every buffer
PATTERN = 0xA5


def _guarded_like(t: torch.Tensor):
    nbytes = t.numel() * t.element_size()
    raw = torch.full((nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=t.device)
    view = raw[GUARD:GUARD + nbytes].view(t.dtype).view(t.shape)
    view.copy_(t)
    return raw, view


def _guards_intact(raw: torch.Tensor) -> bool:
    return bool((raw[:GUARD] == PATTERN).all()) and bool((raw[-GUARD:] == PATTERN).all())


OUTPUTS = ("parent", "tokens", "score", "old_idx", "n_nodes", "depth", "pos", "mask", "O",
           "topk_id", "topk_val", "sample", "acc_len", "path", "out_tok", "kv_src", "kv_dst",
           "err", "ws")


@pytest.mark.parametrize("cid,kw", [(2, dict(V=4099, P=700)),
                                    (4, dict(V=4096, P=(200, 900), B=5, stream_len=50000)),
                                    (1, dict())])
def test_outputs_stay_inside_their_buffers(cid, kw):
    scn = make_scenario(cid, kv_fill="nan", **kw)
    tree = oracle_tree(scn)
    logits = scn.logits(tree["parent"], tree["tokens"], tree["n_nodes"])
    buf = StepBuffers(shape_of(scn))
    inp = device_inputs(scn, logits)
    raws = []
    for name in OUTPUTS:
        raw, view = _guarded_like(getattr(buf, name))
        setattr(buf, name, view)
        raws.append((name, raw))
    for name in ("table", "K", "V"):  # written in place by the update and the KV commit
        raw, view = _guarded_like(inp[name])
        inp[name] = view
        raws.append((name, raw))
    buf.err.zero_()
    for fused in (True, False):
        run_step(buf, inp, scale=scn.scale, fused=fused)
    run_step(buf, inp, scale=scn.scale, temperature=0.7, seed=3, step=1)
    run_kv_commit(buf, inp)
    torch.cuda.synchronize()
    assert int(buf.err.item()) == 0
    for name, raw in raws:
        assert _guards_intact(raw), name
