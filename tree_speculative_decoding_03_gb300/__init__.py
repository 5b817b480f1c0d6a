"""Python binding of libtsv: the GB300 target-side verification step of tree-based
speculative decoding (tree-masked paged attention, rejection-sampling tree walk,
KV-cache compaction of the accepted path).

Argument marshalling only: every step runs in the library's CUDA kernels.  Torch
tensors supply device memory and the current CUDA stream.  There is no CPU
fallback: if the library is not built, or the device cannot run it, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
HEADER = os.path.join(os.path.dirname(HERE), "include", "tsv.h")

TSV_OK, TSV_ERR_ARG, TSV_ERR_UNSUPPORTED, TSV_ERR_CUDA = 0, 1, 2, 3
TSV_BF16, TSV_F32 = 0, 1
# device-side data error bits in seq_err (include/tsv.h)
TSV_DERR_PARENT, TSV_DERR_BLOCK, TSV_DERR_CAPACITY, TSV_DERR_TOKEN, TSV_DERR_NONFINITE, TSV_DERR_TIMEOUT = 1, 2, 4, 8, 16, 32
TSV_DERR_INTERNAL = 64  # checked test build only
DERR_PARENT, DERR_BLOCK, DERR_CAPACITY, DERR_TOKEN, DERR_NONFINITE = 1, 2, 4, 8, 16

_libs = {}           # loaded libraries by build variant (None = the product build)
_variant = None      # the variant load() returns by default (tests switch it)


class TsvError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"libtsv status {status}: {msg}")
        self.status = status


def lib_path(variant=None) -> str:
    from .builder import lib_path as _p
    return _p(variant)


def build(verbose: bool = False, variant=None) -> str:
    """Builds the library: the product build, or a test build ("checked": device-side
    index checks; "hooks": short bounded waits and a stall switch)."""
    from .builder import build_library
    return build_library(verbose=verbose, variant=variant)


def use_variant(variant=None):
    """Makes load() -- and so every call of this module -- use a test build (None: the
    product build).  For tests only."""
    global _variant
    _variant = variant


def load(variant=None):
    """Loads the in-tree libtsv.so (raises if it has not been built)."""
    v = _variant if variant is None else variant
    if v in _libs:
        return _libs[v]
    path = lib_path(v)
    if not os.path.exists(path):
        raise RuntimeError(f"libtsv.so not built at {path}; run build() first")
    lib = ctypes.CDLL(path)
    P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.tsv_last_error.restype = ctypes.c_char_p
    lib.tsv_last_error.argtypes = []
    lib.tsv_attn_workspace_size.restype = sz
    lib.tsv_attn_workspace_size.argtypes = [i32] * 8
    lib.tsv_tree_verify_attn.restype = i32
    lib.tsv_tree_verify_attn.argtypes = [P] * 7 + [i32] * 8 + [f32, i32, P, sz, P, P]
    lib.tsv_tree_verify_attn_append.restype = i32
    lib.tsv_tree_verify_attn_append.argtypes = [P] * 9 + [i32] * 8 + [f32, i32, P, sz, P, P]
    lib.tsv_tree_reject_sample.restype = i32
    lib.tsv_tree_reject_sample.argtypes = [P, P, P, P, P, P, f32, i32, i32, i32, P, P, P, P, P, P]
    lib.tsv_tree_verify_attn_noalloc.restype = i32
    lib.tsv_tree_verify_attn_noalloc.argtypes = [P] * 7 + [i32] * 8 + [f32, i32, P, P]
    lib.tsv_noalloc_scratch_bytes.restype = sz
    lib.tsv_noalloc_scratch_bytes.argtypes = []
    lib.tsv_kv_compact_accepted.restype = i32
    lib.tsv_kv_compact_accepted.argtypes = [P] * 7 + [i32] * 8 + [P, P]
    lib.tsv_tree_reject_sample_ex.restype = i32
    lib.tsv_tree_reject_sample_ex.argtypes = [P, P, P, P, P, P, f32, P, i32, i32, i32, P, P, P, P, P, P]
    lib.tsv_tree_reject_sample_compact_ex.restype = i32
    lib.tsv_tree_reject_sample_compact_ex.argtypes = ([P, P, P, P, P, P, f32, P, i32, i32, i32, P, P, P, P, P] +
                                                      [P] * 5 + [i32] * 6 + [P, P])
    lib.tsv_tree_reject_sample_compact.restype = i32
    lib.tsv_tree_reject_sample_compact.argtypes = ([P, P, P, P, P, P, f32, i32, i32, i32, P, P, P, P, P] + [P] * 5 +
                                                   [i32] * 6 + [P, P])
    f64 = ctypes.c_double
    lib.tsv_sequoia_values.restype = i32
    lib.tsv_sequoia_values.argtypes = [P, i32, i32, i32, P]
    lib.tsv_sequoia_tree.restype = i32
    lib.tsv_sequoia_tree.argtypes = [P, i32, i32, i32, P, P]
    lib.tsv_sequoia_plan.restype = i32
    lib.tsv_sequoia_plan.argtypes = [P, i32, i32, i32, P, f64, P, P, P]
    lib.tsv_sequoia_accept_counts.restype = i32
    lib.tsv_sequoia_accept_counts.argtypes = [P, P, P, i32, i32, i32, P, P]
    if hasattr(lib, "tsv_test_set_stall"):  # the "hooks" test build only
        lib.tsv_test_set_stall.restype = i32
        lib.tsv_test_set_stall.argtypes = [i32]
    _libs[v] = lib
    return lib


def header_symbols() -> list:
    """Entry points declared in include/tsv.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(tsv_[a-z0-9_]+)\s*\(", text)))


def _check(status: int):
    if status != TSV_OK:
        raise TsvError(status, load().tsv_last_error().decode())


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return TSV_BF16
    if t.dtype == torch.float32:
        return TSV_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def attn_workspace_size(B, N, Hq, Hkv, D, block_size, max_blocks, dtype_code) -> int:
    return int(load().tsv_attn_workspace_size(B, N, Hq, Hkv, D, block_size, max_blocks, dtype_code))


def tree_verify_attn(q, k_cache, v_cache, block_table, seq_lens, parent, out, scale: float,
                     workspace=None, seq_err=None, stream=None):
    """out[b,n,h,:] = tree-masked attention of q[b,n,h,:] over the paged cache
    (see include/tsv.h).  q/out [B,N,Hq,D]; caches [num_blocks,bs,Hkv,D]."""
    _contig(q, k_cache, v_cache, block_table, seq_lens, parent, out, workspace, seq_err)
    B, N, Hq, D = q.shape
    num_blocks, bs, Hkv, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().tsv_tree_verify_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), _ptr(parent), _ptr(out),
        B, N, Hq, Hkv, D, bs, block_table.shape[1], num_blocks, float(scale), _dtype_code(q),
        _ptr(workspace), ws_bytes, _ptr(seq_err), _stream(stream)))


def tree_verify_attn_append(q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, parent, out, scale: float,
                            workspace=None, seq_err=None, stream=None):
    """tree_verify_attn that first writes the tree's K/V rows (k_new / v_new
    [B,N,Hkv,D]) into the cache at logical slots seq_lens[b] + j (see include/tsv.h)."""
    _contig(q, k_new, v_new, k_cache, v_cache, block_table, seq_lens, parent, out, workspace, seq_err)
    B, N, Hq, D = q.shape
    num_blocks, bs, Hkv, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().tsv_tree_verify_attn_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
        _ptr(parent), _ptr(out), B, N, Hq, Hkv, D, bs, block_table.shape[1], num_blocks, float(scale),
        _dtype_code(q), _ptr(workspace), ws_bytes, _ptr(seq_err), _stream(stream)))


def tree_verify_attn_noalloc(q, k_cache, v_cache, block_table, seq_lens, parent, out, scale: float,
                             seq_err, stream=None):
    """tree_verify_attn for callers that cannot allocate: the split-K scratch is the
    library's own fixed device array (see include/tsv.h; calls must not overlap)."""
    _contig(q, k_cache, v_cache, block_table, seq_lens, parent, out, seq_err)
    B, N, Hq, D = q.shape
    num_blocks, bs, Hkv, _ = k_cache.shape
    _check(load().tsv_tree_verify_attn_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), _ptr(parent), _ptr(out),
        B, N, Hq, Hkv, D, bs, block_table.shape[1], num_blocks, float(scale), _dtype_code(q),
        _ptr(seq_err), _stream(stream)))


class WalkOptions(ctypes.Structure):
    """tsv_walk_options (include/tsv.h)."""
    _fields_ = [("with_replacement", ctypes.c_int), ("logits_dtype", ctypes.c_int), ("top_k", ctypes.c_int),
                ("top_p", ctypes.c_float)]


def _walk_options(target_logits, with_replacement, top_k, top_p):
    return WalkOptions(1 if with_replacement else 0, _dtype_code(target_logits), int(top_k), float(top_p))


def tree_reject_sample(target_logits, draft_probs, draft_tokens, parent, u_accept, u_bonus,
                       temperature: float, accepted_nodes, accept_len, bonus_token, out_tokens, seq_err,
                       stream=None, with_replacement=False, top_k=0, top_p=1.0):
    """Rejection-sampling walk of the draft tree (see include/tsv.h).  target_logits may
    be float32 or bfloat16; with_replacement, top_k and top_p select the variants of
    tsv_walk_options."""
    _contig(target_logits, draft_probs, draft_tokens, parent, u_accept, u_bonus, accepted_nodes, accept_len,
            bonus_token, out_tokens, seq_err)
    B, N, V = target_logits.shape
    opts = _walk_options(target_logits, with_replacement, top_k, top_p)
    _check(load().tsv_tree_reject_sample_ex(
        _ptr(target_logits), _ptr(draft_probs), _ptr(draft_tokens), _ptr(parent), _ptr(u_accept), _ptr(u_bonus),
        float(temperature), ctypes.byref(opts), B, N, V, _ptr(accepted_nodes), _ptr(accept_len), _ptr(bonus_token),
        _ptr(out_tokens), _ptr(seq_err), _stream(stream)))


def tree_reject_sample_compact(target_logits, draft_probs, draft_tokens, parent, u_accept, u_bonus,
                               temperature: float, accepted_nodes, accept_len, bonus_token, out_tokens, seq_err,
                               k_cache, v_cache, block_table, seq_lens, new_seq_lens, compact_err, stream=None,
                               with_replacement=False, top_k=0, top_p=1.0):
    """The walk and the KV-cache rewrite of its accepted path in one launch (see include/tsv.h)."""
    _contig(target_logits, draft_probs, draft_tokens, parent, u_accept, u_bonus, accepted_nodes, accept_len,
            bonus_token, out_tokens, seq_err, k_cache, v_cache, block_table, seq_lens, new_seq_lens, compact_err)
    B, N, V = target_logits.shape
    num_blocks, bs, Hkv, D = k_cache.shape
    opts = _walk_options(target_logits, with_replacement, top_k, top_p)
    _check(load().tsv_tree_reject_sample_compact_ex(
        _ptr(target_logits), _ptr(draft_probs), _ptr(draft_tokens), _ptr(parent), _ptr(u_accept), _ptr(u_bonus),
        float(temperature), ctypes.byref(opts), B, N, V, _ptr(accepted_nodes), _ptr(accept_len), _ptr(bonus_token),
        _ptr(out_tokens), _ptr(seq_err), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
        _ptr(new_seq_lens), Hkv, D, bs, block_table.shape[1], num_blocks, _dtype_code(k_cache), _ptr(compact_err),
        _stream(stream)))


def kv_compact_accepted(k_cache, v_cache, block_table, seq_lens, accepted_nodes, accept_len, new_seq_lens,
                        seq_err, stream=None):
    """Moves the accepted path's K/V rows into contiguous slots (see include/tsv.h)."""
    _contig(k_cache, v_cache, block_table, seq_lens, accepted_nodes, accept_len, new_seq_lens, seq_err)
    num_blocks, bs, Hkv, D = k_cache.shape
    B, N = accepted_nodes.shape
    _check(load().tsv_kv_compact_accepted(
        _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens), _ptr(accepted_nodes), _ptr(accept_len),
        _ptr(new_seq_lens), B, N, Hkv, D, bs, block_table.shape[1], num_blocks, _dtype_code(k_cache),
        _ptr(seq_err), _stream(stream)))


# ----------------------------------------------------------------------------- tree construction
# Host-side calls (numpy arrays, no GPU): the draft-tree shape with the largest expected
# number of generated tokens per step, and the hardware-aware choice of size and depth
# (see include/tsv.h for the acceptance model).

def _f64(a):
    import numpy as np
    return np.ascontiguousarray(a, dtype=np.float64)


def sequoia_values(accept, n_max: int, d_max: int):
    """[n_max + 1, d_max + 1] array: best expected tokens per step of an n-node tree of
    depth <= d (-inf where no tree exists)."""
    import numpy as np
    acc = _f64(accept)
    out = np.empty((n_max + 1, d_max + 1), np.float64)
    _check(load().tsv_sequoia_values(acc.ctypes.data, len(acc), n_max, d_max, out.ctypes.data))
    return out


def sequoia_tree(accept, n: int, max_depth: int):
    """(parent[n] int32 in breadth-first order with siblings by rank, expected tokens)."""
    import numpy as np
    acc = _f64(accept)
    parent = np.empty(n, np.int32)
    e = ctypes.c_double()
    _check(load().tsv_sequoia_tree(acc.ctypes.data, len(acc), n, max_depth, parent.ctypes.data, ctypes.byref(e)))
    return parent, e.value


def sequoia_plan(accept, n_max: int, d_max: int, t_verify, t_draft: float):
    """(n, d, speedup) maximising E_best(n, d) * t_verify[1] / (t_verify[n] + d * t_draft);
    t_verify[n] for n = 0..n_max (entry 0 is not read)."""
    acc, tv = _f64(accept), _f64(t_verify)
    if len(tv) < n_max + 1:
        raise ValueError("t_verify needs n_max + 1 entries")
    nb, db, sp = ctypes.c_int(), ctypes.c_int(), ctypes.c_double()
    _check(load().tsv_sequoia_plan(acc.ctypes.data, len(acc), n_max, d_max, tv.ctypes.data, float(t_draft),
                                   ctypes.byref(nb), ctypes.byref(db), ctypes.byref(sp)))
    return nb.value, db.value, sp.value


def sequoia_accept_counts(parent, accepted_nodes, accept_len, K: int, reached=None, accepted=None):
    """Adds the positional acceptance counts of one step's walk outputs (host arrays) to
    `reached` / `accepted` (int64 [K], new zero arrays if None) and returns them;
    accepted / reached estimates the acceptance vector the planner takes."""
    import numpy as np
    par = np.ascontiguousarray(parent, np.int32)
    nodes = np.ascontiguousarray(accepted_nodes, np.int32)
    lens = np.ascontiguousarray(accept_len, np.int32)
    B, N = par.shape
    if nodes.shape != (B, N) or lens.shape != (B,):
        raise ValueError("accepted_nodes must be [B, N] and accept_len [B] like parent")
    reached = np.zeros(K, np.int64) if reached is None else reached
    accepted = np.zeros(K, np.int64) if accepted is None else accepted
    for a in (reached, accepted):
        if a.dtype != np.int64 or a.shape != (K,) or not a.flags.c_contiguous:
            raise ValueError("count arrays must be contiguous int64 [K]")
    _check(load().tsv_sequoia_accept_counts(par.ctypes.data, nodes.ctypes.data, lens.ctypes.data, B, N, K,
                                            reached.ctypes.data, accepted.ctypes.data))
    return reached, accepted
