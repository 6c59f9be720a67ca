"""Seeded synthetic inputs for the verify-and-graft step (shared by both sides)."""
from .synth import (  # noqa: F401
    CONFIGS,
    Scenario,
    bf16_bits_to_f32,
    bigram_table,
    default_template,
    dflash_chain,
    eagle_tree,
    f32_to_bf16_bits,
    make_scenario,
    DraftScenario,
    make_draft_scenario,
    topm_cache,
    plant_logits,
    static_tree_widths,
    stream_table,
    treegraft_tree,
)
