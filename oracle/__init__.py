"""CPU oracle for the tree-verification step -- TEST INFRASTRUCTURE ONLY.

Wraps `tsv_oracle.c` (plain single-threaded C, fp64 accumulation) with ctypes.
Only the tests, the smoke check and the benchmark's CPU-baseline leg use it; the
CUDA library never imports, links or calls it.  It shares no code with the
library: the only common module is the seeded input generator (`workloads`),
which draws inputs and holds none of the method's arithmetic.

`build()` compiles the C file with gcc (no fast-math, no FP contraction, so x86
and Arm hosts give identical results).  `mutant=k` builds a copy with planted
mistake k, used only to show that the pins catch it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tsv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")

ERR_PARENT, ERR_BLOCK, ERR_CAPACITY, ERR_TOKEN, ERR_NONFINITE = 1, 2, 4, 8, 16
DTYPE_CODE = {"bf16": 0, "f32": 1}

_libs: dict = {}


def build(mutant: int = 0) -> str:
    os.makedirs(_BUILD, exist_ok=True)
    out = os.path.join(_BUILD, f"libtsv_oracle{'' if mutant == 0 else f'_mutant{mutant}'}.so")
    if not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                               "-shared", "-fPIC", f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, out)
    return out


def _lib(mutant: int = 0):
    if mutant not in _libs:
        lib = ctypes.CDLL(build(mutant))
        P = ctypes.c_void_p
        i32, f64, f32, i64 = ctypes.c_int, ctypes.c_double, ctypes.c_float, ctypes.c_int64
        lib.oracle_tree_verify_attn.argtypes = [P, P, P, i32, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                                i32, f64, P, i64, P, P]
        lib.oracle_tree_verify_attn.restype = i32
        lib.oracle_tree_reject_sample.argtypes = [P, P, P, P, P, P, f32, i32, i32, i32, P, P, P, P, P, P, P, i32, i32,
                                                  f64, i32]
        lib.oracle_tree_reject_sample.restype = i32
        lib.oracle_kv_compact_accepted.argtypes = [P, P, i32, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                                   i32, P]
        lib.oracle_kv_compact_accepted.restype = i32
        _libs[mutant] = lib
    return _libs[mutant]


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def tree_verify_attn(inp: dict, rows: Optional[np.ndarray] = None, *, mutant: int = 0):
    """fp64 tree-masked attention.  rows: flattened (b*N+n)*Hq+h ids (None = all).
    Returns (out [nrows, D] float64, seq_err [B] int32)."""
    B, N, Hq, Hkv, D = inp["B"], inp["N"], inp["Hq"], inp["Hkv"], inp["D"]
    el = np.float32 if inp["dtype"] == "f32" else np.uint16
    q, k, v = _c(inp["q"], el), _c(inp["k_cache"], el), _c(inp["v_cache"], el)
    bt = _c(inp["block_table"], np.int32)
    sl = _c(inp["seq_lens"], np.int32)
    par = _c(inp["parent"], np.int32)
    if rows is not None:
        rows = _c(rows, np.int64)
        nrows = len(rows)
    else:
        nrows = B * N * Hq
    out = np.empty((nrows, D), dtype=np.float64)
    err = np.zeros(B, dtype=np.int32)
    rc = _lib(mutant).oracle_tree_verify_attn(
        _ptr(q), _ptr(k), _ptr(v), DTYPE_CODE[inp["dtype"]], _ptr(bt), _ptr(sl), _ptr(par),
        B, N, Hq, Hkv, D, inp["block_size"], bt.shape[1], inp["num_blocks"], float(inp["scale"]),
        _ptr(rows), nrows, _ptr(out), _ptr(err))
    if rc != 0:
        raise ValueError("oracle_tree_verify_attn: bad arguments")
    return out, err


def tree_reject_sample(inp: dict, *, temperature: Optional[float] = None, mutant: int = 0,
                       replacement: bool = False, top_k: int = 0, top_p: float = 1.0) -> dict:
    """Literal sequential rejection-sampling walk in fp64.  Returns a dict with
    accepted_nodes [B,N], accept_len [B], bonus_token [B], out_tokens [B,N],
    ratio [B,N] (tried children; NaN otherwise), bonus_cdf [B,2], err [B].
    replacement=True: the walk for siblings drafted independently from q (q kept
    after a rejection); the default is the without-replacement walk.  top_k / top_p
    filter the target distribution p (top_k 0 and top_p 1: no filter).  target_logits
    may be float32 or bfloat16 bit patterns (uint16), which are decoded exactly."""
    B, N, V = inp["B"], inp["N"], inp["V"]
    T = float(inp["T"] if temperature is None else temperature)
    bf16_logits = inp["target_logits"].dtype == np.uint16  # bfloat16 bit patterns
    logits = _c(inp["target_logits"], np.uint16 if bf16_logits else np.float32)
    probs = None if inp.get("draft_probs") is None else _c(inp["draft_probs"], np.float32)
    tok = _c(inp["draft_tokens"], np.int32)
    par = _c(inp["parent"], np.int32)
    ua = _c(inp["u_accept"], np.float32)
    ub = _c(inp["u_bonus"], np.float32)
    r = dict(accepted_nodes=np.empty((B, N), np.int32), accept_len=np.empty(B, np.int32),
             bonus_token=np.empty(B, np.int32), out_tokens=np.empty((B, N), np.int32),
             ratio=np.empty((B, N), np.float64), bonus_cdf=np.empty((B, 2), np.float64),
             err=np.empty(B, np.int32))
    rc = _lib(mutant).oracle_tree_reject_sample(
        _ptr(logits), _ptr(probs), _ptr(tok), _ptr(par), _ptr(ua), _ptr(ub), T, B, N, V,
        _ptr(r["accepted_nodes"]), _ptr(r["accept_len"]), _ptr(r["bonus_token"]), _ptr(r["out_tokens"]),
        _ptr(r["ratio"]), _ptr(r["bonus_cdf"]), _ptr(r["err"]), 1 if replacement else 0, int(top_k),
        float(np.float32(top_p)),  # the threshold as the library's float argument holds it
        DTYPE_CODE["bf16" if bf16_logits else "f32"])
    if rc != 0:
        raise ValueError("oracle_tree_reject_sample: bad arguments")
    return r


def kv_compact_accepted(inp: dict, accepted_nodes: np.ndarray, accept_len: np.ndarray, *,
                        mutant: int = 0, inplace: bool = False):
    """Array-copy compaction, on copies of the caches unless `inplace` (then the
    given C-contiguous arrays are modified).  Returns (k_cache, v_cache,
    new_seq_lens, err)."""
    B, N = inp["B"], inp["N"]
    el = np.float32 if inp["dtype"] == "f32" else np.uint16
    if inplace:
        k, v = inp["k_cache"], inp["v_cache"]
        assert k.dtype == el and v.dtype == el and k.flags.c_contiguous and v.flags.c_contiguous
    else:
        k = np.array(inp["k_cache"], dtype=el, copy=True, order="C")
        v = np.array(inp["v_cache"], dtype=el, copy=True, order="C")
    bt = _c(inp["block_table"], np.int32)
    sl = _c(inp["seq_lens"], np.int32)
    an = _c(accepted_nodes, np.int32)
    al = _c(accept_len, np.int32)
    new_len = np.empty(B, np.int32)
    err = np.empty(B, np.int32)
    rc = _lib(mutant).oracle_kv_compact_accepted(
        _ptr(k), _ptr(v), DTYPE_CODE[inp["dtype"]], _ptr(bt), _ptr(sl), _ptr(an), _ptr(al), _ptr(new_len),
        B, N, inp["Hkv"], inp["D"], inp["block_size"], bt.shape[1], inp["num_blocks"], _ptr(err))
    if rc != 0:
        raise ValueError("oracle_kv_compact_accepted: bad arguments")
    return k, v, new_len, err
