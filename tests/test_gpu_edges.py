"""GPU edge cases of the row-level calls: tiny and odd vocabularies for the draws and the
top-k, and degenerate drafting shapes, each against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle.sampling import vocab_sample
from tree_speculative_decoding_parent_gb300 import gt
from workload import make_draft_scenario

pytestmark = pytest.mark.gpu


def _np(x):
    return x.detach().cpu().numpy()


@pytest.mark.parametrize("V", [1, 3, 15, 16, 17, 33])
def test_draws_and_topk_on_tiny_vocabularies(V):
    rng = np.random.default_rng(V)
    rows = 37
    z = rng.standard_normal((rows, V)).astype(np.float32)
    z[0] = 0.0  # a flat row
    dz = torch.from_numpy(z).cuda()
    out = torch.full((rows,), -9, dtype=torch.int32, device="cuda")
    gt.gt_vocab_sample(dz, rows, V, 0.9, 123, 4, out)
    k = min(V, 4)
    ids = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    vals = torch.empty((rows, k), dtype=torch.float32, device="cuda")
    gt.gt_vocab_topk(dz, rows, V, k, ids, vals)
    torch.cuda.synchronize()
    assert np.array_equal(_np(out), vocab_sample(z, np.arange(rows), 0.9, 123, 4))
    for r in range(rows):
        wi, wv = oracle.vocab_topk(z[r], k)
        assert _np(ids)[r].tolist() == wi.tolist()
        assert np.array_equal(_np(vals)[r].view(np.uint32), wv.view(np.uint32))


def test_drafting_degenerate_shapes():
    from test_gpu_drafting import _grow_and_compare
    for kw in (dict(W=1, m=1, q_max=1, Nmax=37), dict(W=3, m=2, q_max=2, Nmax=33),
               dict(W=64, m=16, q_max=8, Nmax=1024)):
        ds = make_draft_scenario(B=2, L=900, V=97, seed=kw["W"], **kw)
        _grow_and_compare(ds, [0, 1, 0, 1])
