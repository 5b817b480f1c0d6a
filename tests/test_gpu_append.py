"""GPU tests of tsv_tree_verify_attn_append: the attention call that first writes the
tree's own K/V rows into the paged cache (sglang report, "Tree-based Speculative
Decoding (EAGLE) Implementation Summary": selective KV update for the tree tokens).

The tree rows of a generated batch are taken out of its cache as k_new / v_new and
their slots overwritten with other data; after the call the cache must be byte for
byte the original, the output bit for bit what tsv_tree_verify_attn gives on the
original cache, and within the attention tolerance of the fp64 oracle.  Sequences
whose block ids fail the checks get no rows written and NaN outputs."""
import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_03_gb300 as tsv
import workloads as W
from gpu_util import dev, device_inputs, run_attn

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-4}


def _tree_rows(inp):
    """k_new, v_new [B, N, Hkv, D] from the cache slots L_b .. L_b + N - 1."""
    B, N, bs = inp["B"], inp["N"], inp["block_size"]
    kn = np.empty((B, N) + inp["k_cache"].shape[2:], inp["k_cache"].dtype)
    vn = np.empty_like(kn)
    for b in range(B):
        L = int(inp["seq_lens"][b])
        for j in range(N):
            t = L + j
            blk = inp["block_table"][b, t // bs]
            kn[b, j] = inp["k_cache"][blk, t % bs]
            vn[b, j] = inp["v_cache"][blk, t % bs]
    return kn, vn


def _scramble_tree_slots(inp, rng):
    """A copy of the caches whose tree slots hold other data (finite values)."""
    k, v = inp["k_cache"].copy(), inp["v_cache"].copy()
    bs = inp["block_size"]
    for b in range(inp["B"]):
        L = int(inp["seq_lens"][b])
        if L < 0:
            continue
        for j in range(inp["N"]):
            t = L + j
            if t // bs >= inp["block_table"].shape[1]:
                continue
            blk = inp["block_table"][b, t // bs]
            if 0 <= blk < inp["num_blocks"]:
                k[blk, t % bs] = k[blk, (t + 1) % bs][::-1]
                v[blk, t % bs] = v[blk, (t + 3) % bs]
    return k, v


def _run_append(inp, k_scr, v_scr):
    bf = inp["dtype"] == "bf16"
    el = torch.bfloat16 if bf else None

    def kv(x):
        return dev(x.view(np.int16) if bf else x, el)

    d = device_inputs(inp, verify=False)
    d["k_cache"], d["v_cache"] = kv(k_scr), kv(v_scr)
    kn, vn = _tree_rows(inp)
    B, N, Hq, D = d["q"].shape
    out = torch.empty_like(d["q"])
    code = tsv.TSV_BF16 if bf else tsv.TSV_F32
    ws_bytes = tsv.attn_workspace_size(B, N, Hq, inp["Hkv"], D, inp["block_size"], inp["max_blocks"], code)
    ws = torch.empty(max(16, ws_bytes), dtype=torch.uint8, device="cuda")
    err = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    tsv.tree_verify_attn_append(d["q"], kv(kn), kv(vn), d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                d["parent"], out, inp["scale"], workspace=ws if ws_bytes else None, seq_err=err)
    torch.cuda.synchronize()
    host = lambda t: t.cpu().view(torch.uint8).numpy()
    got = out.float().cpu().numpy().reshape(B * N * Hq, D).astype(np.float64)
    return got, err.cpu().numpy(), host(d["k_cache"]), host(d["v_cache"])


def _check(inp, full_rows=True, seed=0):
    rng = np.random.default_rng(seed)
    k_scr, v_scr = _scramble_tree_slots(inp, rng)
    got, err, kc, vc = _run_append(inp, k_scr, v_scr)
    # the cache now holds the tree rows again, everything else untouched
    assert np.array_equal(kc.reshape(-1), np.ascontiguousarray(inp["k_cache"]).view(np.uint8).reshape(-1))
    assert np.array_equal(vc.reshape(-1), np.ascontiguousarray(inp["v_cache"]).view(np.uint8).reshape(-1))
    want_lib, err_lib = run_attn(inp)  # the plain call on the original cache
    assert np.array_equal(err, err_lib)
    ok = ~np.isnan(want_lib).any(axis=1)
    assert np.array_equal(np.isnan(got).any(axis=1), ~ok)
    assert np.array_equal(got[ok], want_lib[ok]), "append call differs from the call on the appended cache"
    if full_rows:
        want, oerr = oracle.tree_verify_attn(inp)
    else:
        rows = np.unique(np.concatenate([rng.integers(0, got.shape[0], 40), [0, got.shape[0] - 1]]))
        want, oerr = oracle.tree_verify_attn(inp, rows)
        got = got[rows]
    assert np.array_equal(err, oerr)
    m = ~np.isnan(want).any(axis=1)
    assert np.abs(got[m] - want[m]).max() <= TOL[inp["dtype"]]


def test_tiny_fp32():
    _check(W.generate(W.CONFIGS[0]))


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("f32", 128)])
def test_random_trees_ragged_prefixes(dtype, D):
    w = W.CONFIGS[3].replace(B=5, Hq=16, Hkv=4, D=D, dtype=dtype, prefix=(0, 1500), N=37, depth=6, V=64, seed=88)
    _check(W.generate(w))


def test_flagged_sequences_get_no_rows():
    w = W.CONFIGS[3].replace(B=6, Hq=16, Hkv=4, prefix=(100, 900), N=30, depth=6, V=64, seed=13)
    inp = W.generate(w)
    inp["block_table"] = inp["block_table"].copy()
    inp["block_table"][2, 0] = -4          # bad block id: nothing written, NaN rows
    inp["parent"] = inp["parent"].copy()
    inp["parent"][4, 3] = 9                # not a tree: rows written, NaN outputs
    rng = np.random.default_rng(1)
    k_scr, v_scr = _scramble_tree_slots(inp, rng)
    got, err, kc, vc = _run_append(inp, k_scr, v_scr)
    assert err[2] & tsv.TSV_DERR_BLOCK and err[4] & tsv.TSV_DERR_PARENT
    B, N, Hq = inp["B"], inp["N"], inp["Hq"]
    rows = got.reshape(B, N * Hq, -1)
    assert np.isnan(rows[2]).all() and np.isnan(rows[4]).all()
    assert not np.isnan(rows[[0, 1, 3, 5]]).any()
    # sequence 2's slots keep the scrambled data; every other sequence has its rows back
    want_k = np.ascontiguousarray(inp["k_cache"]).copy()
    bs = inp["block_size"]
    L = int(inp["seq_lens"][2])
    for j in range(N):
        t = L + j
        blk = inp["block_table"][2, t // bs]
        if 0 <= blk < inp["num_blocks"]:
            want_k[blk, t % bs] = k_scr[blk, t % bs]
    assert np.array_equal(kc.reshape(-1), want_k.view(np.uint8).reshape(-1))


@pytest.mark.parametrize("cfg", [2, 3])
def test_full_size(cfg):
    _check(W.generate(W.CONFIGS[cfg]), full_rows=False, seed=cfg)
