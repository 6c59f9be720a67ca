"""The C-ABI library builds, loads without a GPU and exports every declared entry point;
host helpers agree with the pages and with the input generator."""
import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT, golden

HEADER = os.path.join(ROOT, "include", "gt.h")


@pytest.fixture(scope="module")
def lib():
    from tree_speculative_decoding_parent_gb300 import build, gt
    build.build()
    return gt


def declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(gt_[A-Za-z0-9_]+)\s*\(", txt)))


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(so, n), n
    assert set(names) == set(lib.exported_symbols())


def test_stage_budget_matches_page(lib):
    g = golden("budgets.json")
    for st, (d, r) in g["stages"].items():
        assert lib.gt_stage_budget(int(st), g["slots"]) == (d, r)
    assert lib.gt_stage_budget(-1, 60) == tuple(g["no_prune"])
    with pytest.raises(lib.GTError):
        lib.gt_stage_budget(2, 60)


def test_default_template_matches_generator(lib):
    from workload import default_template
    for T in (0, 1, 20, 36, 52, 200):
        tp, tr = lib.gt_default_template(T, 8, 8)
        wp, wr = default_template(T, 8, 8)
        assert np.array_equal(tp, wp) and np.array_equal(tr, wr)


def test_status_strings_and_arg_errors(lib):
    assert lib.status_string(0) == "ok"
    assert "parent" in lib.status_string(lib.GT_ERR_NONMONOTONE)
    # host-visible argument errors are reported without touching the GPU
    so = lib.load()
    assert so.gt_tree_attn_workspace(1, 60, 32, 8, 64, 100) == 0          # d != 128
    assert so.gt_tree_attn_workspace(1, 65, 32, 8, 128, 100) == 0         # N > 64
    assert so.gt_vocab_topk(None, 4, 10, 17, None, None, None) == lib.GT_ERR_SHAPE
    assert so.gt_prune_topB(None, None, None, None, 1, 2000, None, None, 60, None, None, None,
                            None, None, None, None) == lib.GT_ERR_SHAPE
    assert so.gt_prune_topB(None, None, None, None, 0, 10, None, None, 60, None, None, None,
                            None, None, None, None) == lib.GT_OK


def test_sampling_and_drafting_calls_validate_arguments_without_gpu(lib):
    so = lib.load()
    P = 4096  # a stand-in address: these calls must return before any CUDA work
    ARG, SHAPE, OK = lib.GT_ERR_ARG, lib.GT_ERR_SHAPE, lib.GT_OK
    for T in (0.0, -1.0, float("inf"), float("nan"), 1e-39):
        assert so.gt_vocab_sample(P, 2, 100, T, 1, 1, P, None) == ARG
    assert so.gt_vocab_sample(None, 0, 100, 1.0, 1, 1, None, None) == OK
    assert so.gt_vocab_sample(P, 2, 0, 1.0, 1, 1, P, None) == ARG
    assert so.gt_verify_sample(P, P, P, P, P, 1, 2000, 10, 1.0, 1, 1, P, P, P, P, P, P, P,
                               None) == SHAPE
    assert so.gt_verify_sample(None, None, None, None, None, 0, 60, 10, 1.0, 1, 1, None, None,
                               None, None, None, None, None, None) == OK
    assert so.gt_verify_sample_commit(P, P, P, P, P, 1, 60, 100, 17, 1.0, 1, 1, P, P, P, P, P, P,
                                      P, P, P, P, None) == SHAPE
    # drafting: frontier width, both pools, key length, match alignment, children per CTA
    assert so.gt_frontier_select(P, P, 1, 256, P, None, 65, P, P, P, None) == SHAPE
    assert so.gt_frontier_select(P, P, 1, 256, P, P, 10, P, P, P, None) == ARG
    assert so.gt_frontier_select(P, P, 1, 256, None, None, 10, P, P, P, None) == ARG
    assert so.gt_ngram_draft(P, P, 1, 100, P, P, 10, P, P, P, 256, P, P, 10, 9, P, P, P, P,
                             None) == SHAPE
    assert so.gt_ngram_draft(P, P, 1, 100, P, P, 10, P, P, P, 256, P, P, 10, 4, P, P, P + 4, P,
                             None) == ARG
    assert so.gt_ngram_draft(P, P, 1, 100, P, P, 10, P, P, P, 256, P, P, 10, 4, P, P, None, P,
                             None) == ARG
    assert so.gt_tree_attach(P, P, P, P, 1, 256, P, P, 64, P, P, 32, 100, P, P, None) == SHAPE
    assert so.gt_tree_attach(P, P, P, P, 1, 256, P, P, 10, P, P, 10, 0, P, P, None) == ARG
    # KV commit: rows must be whole 16-byte chunks
    assert so.gt_kv_commit(P, P, P, P, P, 1, 8, 8, 100, 1000, lib.GT_BF16, P, None) == SHAPE


def test_wait_selftest_rejects_bad_limits_without_gpu(lib):
    so = lib.load()
    for ns in (0, -5, 2_000_000_000):
        assert so.gt_selftest_wait_timeout(ns, 4096, None, None) == lib.GT_ERR_ARG
    assert so.gt_selftest_wait_timeout(1000, None, None, None) == lib.GT_ERR_ARG
