"""gt_tree_attn_noalloc (attention with the library's static scratch) against gt_tree_attn
with a caller workspace and against the oracle, on the same trees and caches: two calls in a
row must each match within the attention tolerance. The file name sorts last so that the
static scratch is also exercised after every other GPU test has run in the same process."""
import numpy as np
import pytest
import torch

from parity_util import TOL, device_inputs, np_, oracle_attn, oracle_tree, shape_of
from tree_speculative_decoding_parent_gb300 import gt
from tree_speculative_decoding_parent_gb300.step import StepBuffers, run_attn, run_tree_build
from workload import make_scenario

pytestmark = pytest.mark.gpu

CASES = {
    "qwen3-8b-small-bf16": (3, dict(V=4099, P=1333, stream_len=50000)),
    "tiny-eagle-fp32": (1, dict()),
    "llama3.1-8b-small-bf16-nan-tail": (2, dict(V=5000, P=700, kv_fill="nan")),
    "qwen3-8b-P32768-bf16": (3, dict()),
}


def _noalloc(buf, inp, s, scale, O):
    gt.gt_tree_attn_noalloc(inp["Q"], inp["K"], inp["V"], buf.mask, inp["prefix_len"],
                            buf.n_nodes, s.B, s.N, s.Hq, s.Hkv, s.d, s.Lcap, s.dtype, scale, O,
                            buf.err)


@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_matches_workspace_entry_point(case):
    cid, kw = CASES[case]
    scn = make_scenario(cid, **kw)
    tree = oracle_tree(scn)
    logits = scn.logits(tree["parent"], tree["tokens"], tree["n_nodes"])
    s = shape_of(scn)
    assert gt.gt_tree_attn_workspace(s.B, s.N, s.Hq, s.Hkv, s.d, s.Lcap) <= \
        gt.GT_ATTN_NOALLOC_SCRATCH_BYTES
    buf = StepBuffers(s)
    inp = device_inputs(scn, logits)
    run_tree_build(buf, inp)
    run_attn(buf, inp, scale=scn.scale)
    torch.cuda.synchronize()
    assert buf.err.item() == 0
    ref = buf.O.float().cpu().numpy()
    n = np_(buf.n_nodes)
    want = [oracle_attn(scn, tree, b) for b in range(s.B)]
    for _ in range(2):
        O = torch.full_like(buf.O, float("nan"))
        _noalloc(buf, inp, s, scn.scale, O)
        torch.cuda.synchronize()
        assert buf.err.item() == 0
        got = O.float().cpu().numpy()
        for b in range(s.B):
            nb = int(n[b])
            assert np.all(got[b, nb:] == 0.0)
            err = float(np.abs(got[b, :nb].astype(np.float64) - ref[b, :nb]).max())
            assert err <= TOL[scn.dtype], (case, b, err)
            err = float(np.abs(got[b, :nb].astype(np.float64) - want[b]).max())
            assert err <= TOL[scn.dtype], (case, "oracle", b, err)


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    # B = 16 requests, 8 KV heads, 8 query heads per KV head, 60 nodes: about 73 MB of
    # scratch, more than the static array holds; refused on the host, nothing launched
    B, N, Hq, Hkv, d, Lcap = 16, 60, 64, 8, 128, 8256
    need = gt.gt_tree_attn_workspace(B, N, Hq, Hkv, d, Lcap)
    assert need > gt.GT_ATTN_NOALLOC_SCRATCH_BYTES
    with pytest.raises(gt.GTError) as ei:
        gt.gt_tree_attn_noalloc(None, None, None, None, None, None, B, N, Hq, Hkv, d, Lcap,
                                gt.GT_BF16, 0.088, None, None)
    assert ei.value.status == gt.GT_ERR_SHAPE
    assert str(need) in gt.last_error()
