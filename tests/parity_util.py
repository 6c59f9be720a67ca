"""Shared helpers of the GPU parity tests: move a scenario to the device, run the CUDA step
through the C ABI, run the oracle on the same inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from tree_speculative_decoding_parent_gb300 import gt
from tree_speculative_decoding_parent_gb300.step import StepBuffers, StepShape, run_step

TOL = {"f32": 1e-5, "bf16": 2e-2}  # max-abs attention error vs the float64 oracle


def _bf16_tensor(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def shape_of(scn) -> StepShape:
    return StepShape(B=scn.B, Nin=scn.Nin, N=scn.N, V=scn.V, k=scn.k, Hq=scn.Hq, Hkv=scn.Hkv,
                     d=scn.d, Lcap=scn.Lcap, T=len(scn.tpar),
                     dtype=gt.GT_BF16 if scn.dtype == "bf16" else gt.GT_F32)


def device_inputs(scn, logits: np.ndarray, dev="cuda") -> dict:
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    d = dict(score_in=t(scn.score_in), parent_in=t(scn.parent_in), tokens_in=t(scn.tokens_in),
             keep=t(scn.keep), R=t(scn.R), table=t(scn.table), prefix_len=t(scn.prefix_len),
             logits=t(logits))
    if scn.thresh is not None:
        d["thresh"] = t(scn.thresh)
    if scn.anchor is not None:
        d["anchor"] = t(scn.anchor)
    if len(scn.tpar):
        d["tpar"], d["trank"] = t(scn.tpar), t(scn.trank)
    if scn.dtype == "bf16":
        d["Q"], d["K"], d["V"] = (_bf16_tensor(x).to(dev) for x in (scn.Q, scn.K, scn.Vc))
    else:
        d["Q"], d["K"], d["V"] = t(scn.Q), t(scn.K), t(scn.Vc)
    return d


def oracle_tree(scn) -> dict:
    return oracle.step_tree_phase(scn.parent_in, scn.tokens_in, scn.score_in, [scn.Nin] * scn.B,
                                  scn.keep, scn.thresh, scn.tpar, scn.trank, scn.R, scn.table,
                                  scn.prefix_len, scn.N, anchor=scn.anchor)


def decode(x: np.ndarray, dtype: str) -> np.ndarray:
    return oracle.bf16_to_f64(x) if dtype == "bf16" else np.asarray(x, np.float64)


def oracle_attn(scn, tree: dict, b: int) -> np.ndarray:
    n, P = int(tree["n_nodes"][b]), int(scn.prefix_len[b])
    L = P + n
    return oracle.tree_attn(decode(scn.Q[b], scn.dtype), decode(scn.K[b][:, :L], scn.dtype),
                            decode(scn.Vc[b][:, :L], scn.dtype), tree["parent"][b], n, P,
                            scn.scale)


def run_gpu_step(scn, logits: np.ndarray, fused: bool = True):
    buf = StepBuffers(shape_of(scn))
    inp = device_inputs(scn, logits)
    run_step(buf, inp, scale=scn.scale, fused=fused)
    torch.cuda.synchronize()
    return buf, inp


def np_(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().numpy()


def compare_tree(buf, tree):
    n = np_(buf.n_nodes)
    assert np.array_equal(n, tree["n_nodes"]), (n, tree["n_nodes"])
    assert np.array_equal(np_(buf.parent), tree["parent"])
    assert np.array_equal(np_(buf.tokens), tree["tokens"])
    B, N = tree["parent"].shape
    old = np_(buf.old_idx)
    sc = np_(buf.score)
    for b in range(B):
        nk = int(tree["n_kept"][b])
        assert np.array_equal(old[b, :nk], tree["old_idx"][b, :nk])
        assert np.array_equal(sc[b, :nk].view(np.uint32), tree["score"][b, :nk].view(np.uint32))
    assert np.array_equal(np_(buf.depth), tree["depth"])
    assert np.array_equal(np_(buf.pos), tree["pos"])
    assert np.array_equal(np_(buf.mask).view(np.uint64), tree["mask"])


def compare_verify(buf, res, table_after):
    assert np.array_equal(np_(buf.topk_id), res["topk_id"])
    assert np.array_equal(np_(buf.topk_val).view(np.uint32), res["topk_val"].view(np.uint32))
    for key in ("acc_len", "path", "out_tok", "kv_src", "kv_dst"):
        assert np.array_equal(np_(getattr(buf, key)), res[key]), key
    assert np.array_equal(np_(table_after), res["table"])


def attn_max_err(buf, scn, tree, reqs=None) -> float:
    O = buf.O.float().cpu().numpy().astype(np.float64)
    worst = 0.0
    for b in (range(scn.B) if reqs is None else reqs):
        n = int(tree["n_nodes"][b])
        ref = oracle_attn(scn, tree, b)
        worst = max(worst, float(np.abs(O[b, :n] - ref).max()))
        assert np.all(O[b, n:] == 0.0)
    return worst
