"""ctypes binding of libgt (include/gt.h): same names, argument marshalling only.

Device arguments take CUDA torch tensors (or raw integer device addresses); ``None``
passes a null pointer. ``stream`` takes a torch.cuda.Stream, a raw cudaStream_t integer,
or None for torch's current stream. A nonzero status raises GTError. There is no CPU
path: the library must be built (``build()``) and a CUDA device present.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgt.so")

GT_OK, GT_ERR_ARG, GT_ERR_SHAPE, GT_ERR_CUDA = 0, -1, -2, -3
GT_ERR_TREE, GT_ERR_NONMONOTONE, GT_ERR_TIMEOUT, GT_ERR_RANGE = -4, -5, -6, -7
GT_ERR_IO, GT_ERR_CORRUPT, GT_ERR_VALUE = -8, -9, -10
GT_F32, GT_BF16 = 0, 1
GT_ATTN_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024  # size of the static scratch in libgt

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_u64 = ctypes.c_uint64
_SIGS = {
    "gt_prune_topB": (_i, [_vp, _vp, _vp, _vp, _i, _i, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp,
                           _vp, _vp]),
    "gt_graft_expand": (_i, [_vp, _vp, _vp, _i, _i, _vp, _vp, _i, _vp, _vp, _vp, _i, _i, _vp,
                             _vp]),
    "gt_tree_mask": (_i, [_vp, _vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp]),
    "gt_tree_attn_workspace": (_sz, [_i, _i, _i, _i, _i, _i]),
    "gt_tree_attn": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp,
                          _vp, _sz, _vp, _vp]),
    "gt_tree_attn_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f,
                                  _vp, _vp, _vp]),
    "gt_vocab_topk": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp]),
    "gt_kv_commit": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp]),
    "gt_verify_greedy": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp,
                              _vp, _vp, _vp, _vp]),
    "gt_succ_update": (_i, [_vp, _i, _i, _vp, _vp, _vp, _i, _i, _vp, _vp]),
    "gt_tree_build": (_i, [_vp, _vp, _vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _i,
                           _i, _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "gt_verify_commit": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp,
                              _vp, _vp, _vp, _vp, _vp]),
    "gt_vocab_sample": (_i, [_vp, _i, _i, _f, _u64, _u64, _vp, _vp]),
    "gt_verify_sample": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _f, _u64, _u64, _vp, _vp, _vp,
                              _vp, _vp, _vp, _vp, _vp]),
    "gt_verify_sample_commit": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _u64, _u64,
                                     _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "gt_frontier_select": (_i, [_vp, _vp, _i, _i, _vp, _vp, _i, _vp, _vp, _vp, _vp]),
    "gt_ngram_draft": (_i, [_vp, _vp, _i, _i, _vp, _vp, _i, _vp, _vp, _vp, _i, _vp, _vp, _i, _i,
                            _vp, _vp, _vp, _vp, _vp]),
    "gt_tree_attach": (_i, [_vp, _vp, _vp, _vp, _i, _i, _vp, _vp, _i, _vp, _vp, _i, _i, _vp, _vp,
                            _vp]),
    "gt_selftest_wait_timeout": (_i, [ctypes.c_int64, _vp, _vp, _vp]),
    "gt_succ_save": (_i, [ctypes.c_char_p, _vp, _i, _i]),
    "gt_succ_file_shape": (_i, [ctypes.c_char_p, _vp, _vp]),
    "gt_succ_load": (_i, [ctypes.c_char_p, _vp, _i, _i]),
    "gt_stage_budget": (_i, [_i, _i, _vp, _vp]),
    "gt_default_template": (_i, [_i, _i, _i, _vp, _vp]),
    "gt_status_string": (ctypes.c_char_p, [_i]),
    "gt_last_error": (ctypes.c_char_p, []),
    "gt_event_record_external": (_i, [_vp, _vp]),
}

_lib = None


class GTError(RuntimeError):
    def __init__(self, name: str, status: int):
        detail = last_error() if status == GT_ERR_CUDA else ""
        super().__init__(f"{name}: {status_string(status)} ({status})"
                         + (f" [{detail}]" if detail else ""))
        self.status = status


def _open(path: str) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "tree_speculative_decoding_parent_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load() -> ctypes.CDLL:
    """Load libgt.so (built in-tree); raises if it has not been built."""
    global _lib
    if _lib is None:
        _lib = _open(LIB_PATH)
    return _lib


_lib_check = None


def load_checked() -> ctypes.CDLL:
    """Load the checked flavour libgt_check.so (extra device-side input checks reported in
    the error word; built by ``build.build(check=True)``): the same entry points with the
    same signatures, called directly on the returned handle."""
    global _lib_check
    if _lib_check is None:
        _lib_check = _open(os.path.join(_HERE, "libgt_check.so"))
    return _lib_check


def exported_symbols():
    return list(_SIGS)


def status_string(status: int) -> str:
    return load().gt_status_string(int(status)).decode()


def last_error() -> str:
    return (load().gt_last_error() or b"").decode()


def _p(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_cuda:
            raise ValueError("libgt takes CUDA tensors (there is no CPU path)")
        if not x.is_contiguous():
            raise ValueError("libgt takes contiguous tensors")
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x)} as a device pointer")


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name, rc):
    if rc != GT_OK:
        raise GTError(name, rc)


def gt_prune_topB(score, parent, tokens, n_in, B, Nin, keep, thresh, Nout, out_parent,
                  out_tokens, out_score, out_old_idx, n_out, err, stream=None):
    _check("gt_prune_topB", load().gt_prune_topB(
        _p(score), _p(parent), _p(tokens), _p(n_in), B, Nin, _p(keep), _p(thresh), Nout,
        _p(out_parent), _p(out_tokens), _p(out_score), _p(out_old_idx), _p(n_out), _p(err),
        _s(stream)))


def gt_graft_expand(parent, tokens, n_nodes, B, Nmax, tpar, trank, T, R, anchor, table, V, k,
                    err, stream=None):
    _check("gt_graft_expand", load().gt_graft_expand(
        _p(parent), _p(tokens), _p(n_nodes), B, Nmax, _p(tpar), _p(trank), T, _p(R), _p(anchor),
        _p(table), V, k, _p(err), _s(stream)))


def gt_tree_mask(parent, n_nodes, prefix_len, B, N, depth, pos, mask, err, stream=None):
    _check("gt_tree_mask", load().gt_tree_mask(
        _p(parent), _p(n_nodes), _p(prefix_len), B, N, _p(depth), _p(pos), _p(mask), _p(err),
        _s(stream)))


def gt_tree_attn_workspace(B, N, Hq, Hkv, d, Lcap) -> int:
    return int(load().gt_tree_attn_workspace(B, N, Hq, Hkv, d, Lcap))


def gt_tree_attn(Q, K, V, mask, prefix_len, n_nodes, B, N, Hq, Hkv, d, Lcap, dtype, scale, O,
                 workspace, ws_bytes, err, stream=None):
    _check("gt_tree_attn", load().gt_tree_attn(
        _p(Q), _p(K), _p(V), _p(mask), _p(prefix_len), _p(n_nodes), B, N, Hq, Hkv, d, Lcap,
        dtype, float(scale), _p(O), _p(workspace), int(ws_bytes), _p(err), _s(stream)))


def gt_tree_attn_noalloc(Q, K, V, mask, prefix_len, n_nodes, B, N, Hq, Hkv, d, Lcap, dtype,
                         scale, O, err, stream=None):
    _check("gt_tree_attn_noalloc", load().gt_tree_attn_noalloc(
        _p(Q), _p(K), _p(V), _p(mask), _p(prefix_len), _p(n_nodes), B, N, Hq, Hkv, d, Lcap,
        dtype, float(scale), _p(O), _p(err), _s(stream)))


def gt_kv_commit(K, V, kv_src, kv_dst, acc_len, B, N, Hkv, d, Lcap, dtype, err, stream=None):
    _check("gt_kv_commit", load().gt_kv_commit(
        _p(K), _p(V), _p(kv_src), _p(kv_dst), _p(acc_len), B, N, Hkv, d, Lcap, dtype, _p(err),
        _s(stream)))


def gt_vocab_topk(logits, rows, V, k, ids, vals, stream=None):
    _check("gt_vocab_topk", load().gt_vocab_topk(_p(logits), rows, V, k, _p(ids), _p(vals),
                                                 _s(stream)))


def gt_verify_greedy(logits, tokens, parent, n_nodes, prefix_len, B, N, V, k, topk_id,
                     topk_val, acc_len, path, out_tok, kv_src, kv_dst, err, stream=None):
    _check("gt_verify_greedy", load().gt_verify_greedy(
        _p(logits), _p(tokens), _p(parent), _p(n_nodes), _p(prefix_len), B, N, V, k,
        _p(topk_id), _p(topk_val), _p(acc_len), _p(path), _p(out_tok), _p(kv_src), _p(kv_dst),
        _p(err), _s(stream)))


def gt_succ_update(table, V, k, tokens, topk_id, n_nodes, B, N, err, stream=None):
    _check("gt_succ_update", load().gt_succ_update(
        _p(table), V, k, _p(tokens), _p(topk_id), _p(n_nodes), B, N, _p(err), _s(stream)))


def gt_tree_build(score, parent_in, tokens_in, n_in, B, Nin, keep, thresh, tpar, trank, T, R,
                  anchor, table, V, k, prefix_len, N, parent, tokens, out_score, out_old_idx,
                  n_nodes, depth, pos, mask, err, stream=None):
    _check("gt_tree_build", load().gt_tree_build(
        _p(score), _p(parent_in), _p(tokens_in), _p(n_in), B, Nin, _p(keep), _p(thresh),
        _p(tpar), _p(trank), T, _p(R), _p(anchor), _p(table), V, k, _p(prefix_len), N, _p(parent),
        _p(tokens), _p(out_score), _p(out_old_idx), _p(n_nodes), _p(depth), _p(pos), _p(mask),
        _p(err), _s(stream)))


def gt_verify_commit(logits, tokens, parent, n_nodes, prefix_len, B, N, V, k, topk_id, topk_val,
                     acc_len, path, out_tok, kv_src, kv_dst, table, err, stream=None):
    _check("gt_verify_commit", load().gt_verify_commit(
        _p(logits), _p(tokens), _p(parent), _p(n_nodes), _p(prefix_len), B, N, V, k, _p(topk_id),
        _p(topk_val), _p(acc_len), _p(path), _p(out_tok), _p(kv_src), _p(kv_dst), _p(table),
        _p(err), _s(stream)))


def gt_vocab_sample(logits, rows, V, temperature, seed, step, sample, stream=None):
    _check("gt_vocab_sample", load().gt_vocab_sample(
        _p(logits), rows, V, temperature, seed, step, _p(sample), _s(stream)))


def gt_verify_sample(logits, tokens, parent, n_nodes, prefix_len, B, N, V, temperature, seed,
                     step, sample, acc_len, path, out_tok, kv_src, kv_dst, err, stream=None):
    _check("gt_verify_sample", load().gt_verify_sample(
        _p(logits), _p(tokens), _p(parent), _p(n_nodes), _p(prefix_len), B, N, V, temperature,
        seed, step, _p(sample), _p(acc_len), _p(path), _p(out_tok), _p(kv_src), _p(kv_dst),
        _p(err), _s(stream)))


def gt_verify_sample_commit(logits, tokens, parent, n_nodes, prefix_len, B, N, V, k,
                            temperature, seed, step, topk_id, topk_val, sample, acc_len, path,
                            out_tok, kv_src, kv_dst, table, err, stream=None):
    _check("gt_verify_sample_commit", load().gt_verify_sample_commit(
        _p(logits), _p(tokens), _p(parent), _p(n_nodes), _p(prefix_len), B, N, V, k,
        temperature, seed, step, _p(topk_id), _p(topk_val), _p(sample), _p(acc_len), _p(path),
        _p(out_tok), _p(kv_src), _p(kv_dst), _p(table), _p(err), _s(stream)))


def gt_frontier_select(score, n_nodes, B, Nmax, pool_lo, visited, W, frontier, n_frontier, err,
                       stream=None):
    _check("gt_frontier_select", load().gt_frontier_select(
        _p(score), _p(n_nodes), B, Nmax, _p(pool_lo), _p(visited), W, _p(frontier),
        _p(n_frontier), _p(err), _s(stream)))


def gt_ngram_draft(hist, hist_len, B, Lh, cache_id, cache_p, m, parent, tokens, n_nodes, Nmax,
                   frontier, n_frontier, W, q_max, child_id, child_p, match, err, stream=None):
    _check("gt_ngram_draft", load().gt_ngram_draft(
        _p(hist), _p(hist_len), B, Lh, _p(cache_id), _p(cache_p), m, _p(parent), _p(tokens),
        _p(n_nodes), Nmax, _p(frontier), _p(n_frontier), W, q_max, _p(child_id), _p(child_p),
        _p(match), _p(err), _s(stream)))


def gt_tree_attach(parent, tokens, score, n_nodes, B, Nmax, frontier, n_frontier, W, child_id,
                   child_p, m, V, first_new, err, stream=None):
    _check("gt_tree_attach", load().gt_tree_attach(
        _p(parent), _p(tokens), _p(score), _p(n_nodes), B, Nmax, _p(frontier), _p(n_frontier), W,
        _p(child_id), _p(child_p), m, V, _p(first_new), _p(err), _s(stream)))


def gt_selftest_wait_timeout(limit_ns, err, waited_ns=None, stream=None):
    _check("gt_selftest_wait_timeout", load().gt_selftest_wait_timeout(
        int(limit_ns), _p(err), _p(waited_ns), _s(stream)))


def gt_succ_save(path: str, table) -> None:
    """Write a successor table (host int32 [V][k]; a torch tensor is copied to the host) to
    path."""
    import numpy as np
    t = table.detach().cpu().numpy() if hasattr(table, "detach") else table
    t = np.ascontiguousarray(t, dtype=np.int32)
    V, k = t.shape
    _check("gt_succ_save", load().gt_succ_save(os.fsencode(path), t.ctypes.data, V, k))


def gt_succ_file_shape(path: str):
    V, k = ctypes.c_int32(), ctypes.c_int32()
    _check("gt_succ_file_shape", load().gt_succ_file_shape(os.fsencode(path), ctypes.byref(V),
                                                           ctypes.byref(k)))
    return V.value, k.value


def gt_succ_load(path: str, V: int = None, k: int = None):
    """Read a successor table file; returns a host int32 [V][k] array (V, k: the expected
    shape, else the file's)."""
    import numpy as np
    if V is None or k is None:
        V, k = gt_succ_file_shape(path)
    t = np.empty((V, k), np.int32)
    _check("gt_succ_load", load().gt_succ_load(os.fsencode(path), t.ctypes.data, V, k))
    return t


def gt_stage_budget(stage: int, slots: int = 60):
    d, r = ctypes.c_int32(), ctypes.c_int32()
    _check("gt_stage_budget", load().gt_stage_budget(stage, slots, ctypes.byref(d),
                                                     ctypes.byref(r)))
    return d.value, r.value


def gt_default_template(T: int, k: int = 8, max_depth: int = 8):
    import numpy as np
    tpar = np.zeros(max(T, 1), np.int32)
    trank = np.zeros(max(T, 1), np.int32)
    _check("gt_default_template", load().gt_default_template(
        T, k, max_depth, tpar.ctypes.data, trank.ctypes.data))
    return tpar[:T], trank[:T]


def gt_event_record_external(event, stream=None):
    _check("gt_event_record_external",
           load().gt_event_record_external(event.cuda_event, _s(stream)))
