"""CPU oracle of the verify-and-graft step (test infrastructure, not product code).

Only the tests, the smoke check of the package entry module and the CPU-baseline leg
of the benchmark may import this package. The product path never calls it and has
no CPU fallback.
"""
from .step import (  # noqa: F401
    OracleError,
    NonMonotoneError,
    TreeError,
    bf16_to_f64,
    graft_expand,
    kv_commit,
    prune_topB,
    stage_budget,
    step_tree_phase,
    step_verify_phase,
    succ_update,
    tree_attn,
    tree_mask,
    verify_greedy,
    vocab_topk,
)
from .sampling import (  # noqa: F401
    philox4x32_10,
    step_verify_sampled,
    verify_sampled,
    vocab_sample,
)
from .drafting import (  # noqa: F401
    frontier_select,
    ngram_children,
    tree_attach,
)
