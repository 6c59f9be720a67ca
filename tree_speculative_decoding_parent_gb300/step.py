"""One verify-and-graft step through the C ABI, with its device buffers.

``StepBuffers`` owns (through torch) every output and scratch buffer of the step for a
fixed shape; ``run_step`` issues, on one stream and without host synchronisation, either
the fused form (default: 5 kernel launches)
  a1+a2+a3 gt_tree_build -> a4 gt_tree_attn -> a5+a6+a7 gt_verify_commit
or the separate calls
  a1 gt_prune_topB -> a2 gt_graft_expand (when the template is non-empty)
  -> a3 gt_tree_mask -> a4 gt_tree_attn -> a5+a6 gt_verify_greedy -> a7 gt_succ_update.
Both give identical results. Every step of the computation runs in libgt's kernels; this
module only allocates and passes pointers.
"""
from __future__ import annotations

import dataclasses

import torch

from . import gt


@dataclasses.dataclass
class StepShape:
    B: int
    Nin: int
    N: int
    V: int
    k: int
    Hq: int
    Hkv: int
    d: int
    Lcap: int
    T: int
    dtype: int  # gt.GT_F32 or gt.GT_BF16

    @property
    def W(self) -> int:
        return (self.N + 63) // 64


class StepBuffers:
    """Outputs and scratch of one step (device memory, allocated once)."""

    def __init__(self, shape: StepShape, device="cuda"):
        s, i32 = shape, torch.int32
        self.shape = s
        dev = torch.device(device)
        self.parent = torch.empty((s.B, s.N), dtype=i32, device=dev)
        self.tokens = torch.empty((s.B, s.N), dtype=i32, device=dev)
        self.score = torch.empty((s.B, s.N), dtype=torch.float32, device=dev)
        self.old_idx = torch.empty((s.B, s.N), dtype=i32, device=dev)
        self.n_nodes = torch.empty((s.B,), dtype=i32, device=dev)
        self.depth = torch.empty((s.B, s.N), dtype=i32, device=dev)
        self.pos = torch.empty((s.B, s.N), dtype=i32, device=dev)
        self.mask = torch.empty((s.B, s.N, s.W), dtype=torch.int64, device=dev)
        odt = torch.float32 if s.dtype == gt.GT_F32 else torch.bfloat16
        self.O = torch.empty((s.B, s.N, s.Hq, s.d), dtype=odt, device=dev)
        self.topk_id = torch.empty((s.B, s.N, s.k), dtype=i32, device=dev)
        self.topk_val = torch.empty((s.B, s.N, s.k), dtype=torch.float32, device=dev)
        self.sample = torch.empty((s.B, s.N), dtype=i32, device=dev)  # draws at T > 0
        self.acc_len = torch.empty((s.B,), dtype=i32, device=dev)
        self.path = torch.empty((s.B, s.N), dtype=i32, device=dev)
        self.out_tok = torch.empty((s.B, s.N + 1), dtype=i32, device=dev)
        self.kv_src = torch.empty((s.B, s.N), dtype=i32, device=dev)
        self.kv_dst = torch.empty((s.B, s.N), dtype=i32, device=dev)
        self.err = torch.zeros((1,), dtype=i32, device=dev)
        self.ws_bytes = gt.gt_tree_attn_workspace(s.B, s.N, s.Hq, s.Hkv, s.d, s.Lcap)
        if self.ws_bytes == 0:
            raise gt.GTError("gt_tree_attn_workspace", gt.GT_ERR_SHAPE)
        self.ws = torch.empty((self.ws_bytes,), dtype=torch.uint8, device=dev)


def run_tree_phase(buf: StepBuffers, inp: dict, stream=None):
    """a1 prune, a2 graft, a3 mask."""
    s = buf.shape
    gt.gt_prune_topB(inp["score_in"], inp["parent_in"], inp["tokens_in"], inp.get("n_in"), s.B,
                     s.Nin, inp["keep"], inp.get("thresh"), s.N, buf.parent, buf.tokens,
                     buf.score, buf.old_idx, buf.n_nodes, buf.err, stream)
    if s.T > 0:
        gt.gt_graft_expand(buf.parent, buf.tokens, buf.n_nodes, s.B, s.N, inp["tpar"],
                           inp["trank"], s.T, inp["R"], inp.get("anchor"), inp["table"], s.V, s.k,
                           buf.err, stream)
    gt.gt_tree_mask(buf.parent, buf.n_nodes, inp["prefix_len"], s.B, s.N, buf.depth, buf.pos,
                    buf.mask, buf.err, stream)


def run_verify_phase(buf: StepBuffers, inp: dict, stream=None, scale=None):
    """a4 attention, a5+a6 verify, a7 table update."""
    s = buf.shape
    if scale is None:
        scale = 1.0 / (s.d ** 0.5)
    gt.gt_tree_attn(inp["Q"], inp["K"], inp["V"], buf.mask, inp["prefix_len"], buf.n_nodes, s.B,
                    s.N, s.Hq, s.Hkv, s.d, s.Lcap, s.dtype, scale, buf.O, buf.ws, buf.ws_bytes,
                    buf.err, stream)
    gt.gt_verify_greedy(inp["logits"], buf.tokens, buf.parent, buf.n_nodes, inp["prefix_len"],
                        s.B, s.N, s.V, s.k, buf.topk_id, buf.topk_val, buf.acc_len, buf.path,
                        buf.out_tok, buf.kv_src, buf.kv_dst, buf.err, stream)
    gt.gt_succ_update(inp["table"], s.V, s.k, buf.tokens, buf.topk_id, buf.n_nodes, s.B, s.N,
                      buf.err, stream)


def run_tree_build(buf: StepBuffers, inp: dict, stream=None):
    """a1+a2+a3 in one launch."""
    s = buf.shape
    gt.gt_tree_build(inp["score_in"], inp["parent_in"], inp["tokens_in"], inp.get("n_in"), s.B,
                     s.Nin, inp["keep"], inp.get("thresh"), inp.get("tpar"), inp.get("trank"),
                     s.T, inp["R"], inp.get("anchor"), inp["table"], s.V, s.k, inp["prefix_len"],
                     s.N, buf.parent,
                     buf.tokens, buf.score, buf.old_idx, buf.n_nodes, buf.depth, buf.pos,
                     buf.mask, buf.err, stream)


def run_attn(buf: StepBuffers, inp: dict, stream=None, scale=None):
    """a4."""
    s = buf.shape
    if scale is None:
        scale = 1.0 / (s.d ** 0.5)
    gt.gt_tree_attn(inp["Q"], inp["K"], inp["V"], buf.mask, inp["prefix_len"], buf.n_nodes, s.B,
                    s.N, s.Hq, s.Hkv, s.d, s.Lcap, s.dtype, scale, buf.O, buf.ws, buf.ws_bytes,
                    buf.err, stream)


def run_verify_commit(buf: StepBuffers, inp: dict, stream=None):
    """a5+a6+a7: top-k launch, then one walk + table-update launch."""
    s = buf.shape
    gt.gt_verify_commit(inp["logits"], buf.tokens, buf.parent, buf.n_nodes, inp["prefix_len"],
                        s.B, s.N, s.V, s.k, buf.topk_id, buf.topk_val, buf.acc_len, buf.path,
                        buf.out_tok, buf.kv_src, buf.kv_dst, inp["table"], buf.err, stream)


def run_verify_sample_commit(buf: StepBuffers, inp: dict, temperature: float, seed: int,
                             step: int, stream=None):
    """a5+a6+a7 at temperature T > 0: per-node draws, top-k, sampled walk + table update."""
    s = buf.shape
    gt.gt_verify_sample_commit(inp["logits"], buf.tokens, buf.parent, buf.n_nodes,
                               inp["prefix_len"], s.B, s.N, s.V, s.k, temperature, seed, step,
                               buf.topk_id, buf.topk_val, buf.sample, buf.acc_len, buf.path,
                               buf.out_tok, buf.kv_src, buf.kv_dst, inp["table"], buf.err, stream)


def run_kv_commit(buf: StepBuffers, inp: dict, stream=None):
    """Move the accepted path's K/V rows to their committed positions (in place)."""
    s = buf.shape
    gt.gt_kv_commit(inp["K"], inp["V"], buf.kv_src, buf.kv_dst, buf.acc_len, s.B, s.N, s.Hkv,
                    s.d, s.Lcap, s.dtype, buf.err, stream)


def run_step(buf: StepBuffers, inp: dict, stream=None, scale=None, fused: bool = True,
             temperature: float = 0.0, seed: int = 0, step: int = 0):
    """The whole verify-and-graft step (a1..a7) on one stream, no host synchronisation.
    temperature > 0 verifies by one target draw per node (seed, step pick the draws)."""
    if temperature > 0:
        run_tree_build(buf, inp, stream)
        run_attn(buf, inp, stream, scale)
        run_verify_sample_commit(buf, inp, temperature, seed, step, stream)
    elif fused:
        run_tree_build(buf, inp, stream)
        run_attn(buf, inp, stream, scale)
        run_verify_commit(buf, inp, stream)
    else:
        run_tree_phase(buf, inp, stream)
        run_verify_phase(buf, inp, stream, scale)
