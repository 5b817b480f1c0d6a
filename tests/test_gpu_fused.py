"""tsv_tree_reject_sample_compact (the walk with the KV-cache rewrite in its tail) must
give exactly what tsv_tree_reject_sample followed by tsv_kv_compact_accepted gives:
decisions, tokens, error codes, new lengths and both caches byte for byte — including
sequences the walk flags (left untouched) and sequences whose rewrite fails."""
import numpy as np
import pytest
import torch

import tree_speculative_decoding_03_gb300 as tsv
import workloads as W
from gpu_util import device_inputs

pytestmark = pytest.mark.gpu


def _run(inp, fused, T):
    d = device_inputs(inp, attn=True, verify=True)
    B, N, V = d["target_logits"].shape
    i32 = dict(dtype=torch.int32, device="cuda")
    an, ot = torch.full((B, N), -9, **i32), torch.full((B, N), -9, **i32)
    al, bt, err = torch.full((B,), -9, **i32), torch.full((B,), -9, **i32), torch.full((B,), -9, **i32)
    nl, cerr = torch.full((B,), -9, **i32), torch.full((B,), -9, **i32)
    walk = (d["target_logits"], d["draft_probs"], d["draft_tokens"], d["parent"], d["u_accept"], d["u_bonus"], T,
            an, al, bt, ot, err)
    if fused:
        tsv.tree_reject_sample_compact(*walk, d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], nl, cerr)
    else:
        tsv.tree_reject_sample(*walk)
        tsv.kv_compact_accepted(d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], an, al, nl, cerr)
    torch.cuda.synchronize()
    host = lambda t: t.cpu().view(torch.uint8).numpy()  # bytes: the caches hold NaN past each sequence's slots
    return dict(an=an.cpu().numpy(), al=al.cpu().numpy(), bt=bt.cpu().numpy(), ot=ot.cpu().numpy(),
                err=err.cpu().numpy(), nl=nl.cpu().numpy(), cerr=cerr.cpu().numpy(), k=host(d["k_cache"]),
                v=host(d["v_cache"]))


def _same(inp, T=None):
    T = inp["T"] if T is None else T
    a, b = _run(inp, False, T), _run(inp, True, T)
    for key in a:
        assert np.array_equal(a[key], b[key]), key
    return a


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_chain_matches_the_two_calls(T):
    inp = W.generate(W.CONFIGS[1].replace(B=4, prefix=(100, 700), V=5000, seed=21), temperature=T)
    r = _same(inp, T)
    assert (r["cerr"] == 0).all() and (r["nl"] == inp["seq_lens"] + 1 + r["al"]).all()


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64)])
def test_trees_with_flagged_sequences(dtype, D):
    w = W.CONFIGS[3].replace(B=12, Hq=8, Hkv=2, D=D, dtype=dtype, prefix=(0, 900), N=48, depth=8, V=3001, T=0.6,
                             seed=33)
    inp = W.generate(w)
    inp["parent"] = inp["parent"].copy()
    inp["parent"][2, 5] = 7          # not a tree: the walk flags it, the rewrite leaves it alone
    inp["block_table"] = inp["block_table"].copy()
    inp["block_table"][6, 0] = -3    # the walk runs, the rewrite reports a bad block id
    r = _same(inp)
    assert r["al"][2] == -1 and r["cerr"][2] == 0 and r["nl"][2] == inp["seq_lens"][2]
    assert r["cerr"][6] == tsv.TSV_DERR_BLOCK and r["nl"][6] == inp["seq_lens"][6]


def _against_oracle(inp, T=None):
    """The fused call against the oracle: its walk decisions against the oracle's walk
    (bit-exact up to counted near ties), then the caches, new lengths and rewrite errors
    against the oracle's array copy applied to the path the walk took."""
    import oracle
    from gpu_util import compare_decisions

    T = inp["T"] if T is None else T
    r = _run(inp, True, T)
    o = oracle.tree_reject_sample(inp, temperature=T)
    g = dict(accepted_nodes=r["an"], accept_len=r["al"], bonus_token=r["bt"], out_tokens=r["ot"], err=r["err"])
    exempt, fails = compare_decisions(inp, g, o, T)
    B = inp["B"]
    msg = f"{exempt} of {B} sequences exempt as near ties; {len(fails)} mismatches: {fails[:5]}"
    assert not fails, msg
    assert exempt <= 0.05 * B + 1, msg
    print(msg)
    ok_, ov, ol, oe = oracle.kv_compact_accepted(inp, r["an"], r["al"])
    assert np.array_equal(r["cerr"], oe), (r["cerr"], oe)
    assert np.array_equal(r["nl"], ol), (r["nl"], ol)
    assert np.array_equal(r["k"].reshape(-1), ok_.reshape(-1).view(np.uint8)), "K cache differs from the oracle's"
    assert np.array_equal(r["v"].reshape(-1), ov.reshape(-1).view(np.uint8)), "V cache differs from the oracle's"
    return r, o, exempt


@pytest.mark.parametrize("T", [0.0, 0.6, 1.0])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64)])
def test_random_trees_against_the_oracle(T, dtype, D):
    w = W.CONFIGS[3].replace(B=20, Hq=8, Hkv=2, D=D, dtype=dtype, prefix=(0, 700), N=40, depth=7, V=3001, T=T,
                             seed=60 + int(10 * T) + D)
    _against_oracle(W.generate(w, temperature=T), T)


@pytest.mark.parametrize("cfg,T", [(1, 0.0), (1, 1.0), (2, None), (3, None), (4, None)])
def test_full_size_against_the_oracle(cfg, T):
    """The call the benchmark times, on the full workloads it times."""
    inp = W.generate(W.CONFIGS[cfg], temperature=T)
    r, o, _ = _against_oracle(inp, T)
    if cfg == 4:  # the p == q sequences accept every draft down to a leaf
        assert all(o["accept_len"][b] >= 1 for b in inp["pq_seqs"])
