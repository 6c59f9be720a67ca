"""Failure detection on the GPU without a fault: a bounded wait on a barrier that nothing
arrives on ends with GT_ERR_TIMEOUT after its limit, and the context stays usable."""
import numpy as np
import pytest
import torch

from parity_util import TOL, attn_max_err, compare_tree, oracle_tree, run_gpu_step
from tree_speculative_decoding_parent_gb300 import gt
from workload import make_scenario

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_the_context_survives():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    gt.gt_selftest_wait_timeout(5_000_000, err, waited)  # 5 ms
    torch.cuda.synchronize()
    assert int(err.item()) == gt.GT_ERR_TIMEOUT
    assert 5_000_000 <= int(waited.item()) < 500_000_000
    # the same context still runs a step and matches the oracle
    scn = make_scenario(2, V=3000, P=300)
    tree = oracle_tree(scn)
    logits = scn.logits(tree["parent"], tree["tokens"], tree["n_nodes"])
    buf, _ = run_gpu_step(scn, logits)
    assert int(buf.err.item()) == 0
    compare_tree(buf, tree)
    assert attn_max_err(buf, scn, tree) <= TOL[scn.dtype]
    _ = np
