"""The checked test build (-DTSV_CHECKED): every global access the kernels make
through a computed index is first compared with its buffer's extent, and an index
outside it sets TSV_DERR_INTERNAL instead of reading or writing.  This stands in for
a memory sanitizer: tiny cases of every call (N <= 15, V <= 16 and a few more
shapes), on edge inputs, must give the oracle's results with that bit never set."""
import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_03_gb300 as tsv
import workloads as W
from gpu_util import compare_decisions, device_inputs, run_attn, run_compact, run_verify

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def checked_lib():
    tsv.build(variant="checked")
    tsv.use_variant("checked")
    yield tsv.load("checked")
    tsv.use_variant(None)


def _no_internal(err):
    assert not (np.asarray(err) & tsv.TSV_DERR_INTERNAL).any(), err


@pytest.mark.parametrize("dtype,D,N,tree,prefix", [
    ("f32", 64, 15, "binary", (0, 40)), ("bf16", 64, 15, "random", (0, 300)), ("bf16", 128, 7, "chain", (1, 129)),
    ("bf16", 128, 1, "chain", (0, 17)), ("bf16", 128, 64, "random", (100, 700))])
def test_attention(dtype, D, N, tree, prefix):
    w = W.CONFIGS[3].replace(B=3, Hq=8, Hkv=2, D=D, dtype=dtype, prefix=prefix, N=N, tree=tree, depth=6, V=16,
                             seed=3 + N)
    inp = W.generate(w)
    got, err = run_attn(inp)
    _no_internal(err)
    want, oerr = oracle.tree_verify_attn(inp)
    assert np.array_equal(err, oerr)
    assert np.abs(got - want).max() <= (2e-2 if dtype == "bf16" else 1e-4)


@pytest.mark.parametrize("T", [0.0, 0.6, 1.0])
@pytest.mark.parametrize("opts", [{}, {"with_replacement": True}, {"top_k": 3}, {"top_p": 0.7}])
def test_walk(T, opts):
    w = W.CONFIGS[3].replace(B=32, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=15, depth=4, V=16, T=T, seed=8,
                             siblings="independent" if opts.get("with_replacement") else "without")
    inp = W.generate(w, temperature=T)
    g = run_verify(inp, temperature=T, **opts)
    _no_internal(g["err"])
    o = oracle.tree_reject_sample(inp, temperature=T, replacement=opts.get("with_replacement", False),
                                  top_k=opts.get("top_k", 0), top_p=opts.get("top_p", 1.0))
    exempt, fails = compare_decisions(inp, g, o, T)
    assert not fails, fails


def test_compaction_and_fused_walk():
    w = W.CONFIGS[3].replace(B=8, Hq=4, Hkv=2, D=64, prefix=(0, 100), N=15, depth=5, V=16, T=1.0, seed=12)
    inp = W.generate(w)
    o = oracle.tree_reject_sample(inp)
    gk, gv, gl, ge = run_compact(inp, o["accepted_nodes"], o["accept_len"])
    _no_internal(ge)
    ok_, ov, ol, oe = oracle.kv_compact_accepted(inp, o["accepted_nodes"], o["accept_len"])
    assert np.array_equal(gk.view(np.uint8), ok_.view(np.uint8)) and np.array_equal(gl, ol)
    d = device_inputs(inp)
    B, N = inp["B"], inp["N"]
    i32 = dict(dtype=torch.int32, device="cuda")
    an, ot = torch.empty(B, N, **i32), torch.empty(B, N, **i32)
    al, bt, err, nl, cerr = (torch.empty(B, **i32) for _ in range(5))
    tsv.tree_reject_sample_compact(d["target_logits"], d["draft_probs"], d["draft_tokens"], d["parent"],
                                   d["u_accept"], d["u_bonus"], 1.0, an, al, bt, ot, err, d["k_cache"],
                                   d["v_cache"], d["block_table"], d["seq_lens"], nl, cerr)
    torch.cuda.synchronize()
    _no_internal(err.cpu().numpy())
    _no_internal(cerr.cpu().numpy())
    assert np.array_equal(an.cpu().numpy(), o["accepted_nodes"]) and np.array_equal(nl.cpu().numpy(), ol)
