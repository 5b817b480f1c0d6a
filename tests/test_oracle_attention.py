"""Pins for the oracle's tree-masked attention (CPU only).

Each pin ties the oracle to something other than itself:
  * a chain-shaped tree equals ordinary causal attention over prefix + chain
    (statistical-learning-notes "Speculative Decoding", section "Draft Token
    Validation": causal masks let the K drafts be scored in one parallel pass),
    checked against torch's scaled_dot_product_attention in float64;
  * every tree node's output equals attention over its own root-to-node path,
    brute-forced per node with the same library routine (sglang report, "What is
    Tree-Attention?": a tree node attends only to its ancestors);
  * invariants: physical block placement does not matter; heads of one GQA group
    with equal queries give equal outputs; a single visible key returns its value.
The planted-mistake builds of the oracle (no self-attention; interleaved heads)
must fail the pins above.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from workloads import bf16_bits_to_f32

TINY = W.CONFIGS[0]


def _logical_kv(inp, b, upto):
    """[upto, Hkv, D] float64 logical-order K and V of sequence b (library gather)."""
    bs = inp["block_size"]
    t = np.arange(upto)
    phys = inp["block_table"][b, t // bs].astype(np.int64) * bs + t % bs
    def dec(c):
        flat = c.reshape(-1, inp["Hkv"], inp["D"])[phys]
        return (bf16_bits_to_f32(flat) if inp["dtype"] == "bf16" else flat).astype(np.float64)
    return dec(inp["k_cache"]), dec(inp["v_cache"])


def _q64(inp):
    q = inp["q"]
    return (bf16_bits_to_f32(q) if inp["dtype"] == "bf16" else q).astype(np.float64)


def _sdpa(q, k, v, mask, scale):
    """torch SDPA in float64. q [H, M, D]; k, v [H, S, D]; mask [M, S] bool (True = visible)."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=torch.from_numpy(mask), scale=scale).numpy()


def _expand_heads(x, G):
    return np.repeat(x, G, axis=1)  # [S, Hkv, D] -> [S, Hq, D] grouped


def _chain_inputs(dtype, L=37, N=9, Hq=8, Hkv=2, D=32, B=2, seed=5):
    w = TINY.replace(B=B, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype, prefix=(L, L), tree="chain", N=N, V=16, seed=seed)
    return W.generate(w)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mutant", [0, 3, 4])
def test_chain_equals_causal_attention(oracle_mod, dtype, mutant):
    inp = _chain_inputs(dtype)
    B, N, Hq, Hkv, D = inp["B"], inp["N"], inp["Hq"], inp["Hkv"], inp["D"]
    out, err = oracle_mod.tree_verify_attn(inp, mutant=mutant)
    assert not err.any()
    out = out.reshape(B, N, Hq, D)
    q = _q64(inp)
    worst = 0.0
    for b in range(B):
        L = int(inp["seq_lens"][b])
        k, v = _logical_kv(inp, b, L + N)
        k, v = _expand_heads(k, Hq // Hkv), _expand_heads(v, Hq // Hkv)
        # causal over prefix + chain: query n sees slots [0, L + n]
        mask = np.arange(L + N)[None, :] <= (L + np.arange(N))[:, None]
        ref = _sdpa(q[b].transpose(1, 0, 2), k.transpose(1, 0, 2), v.transpose(1, 0, 2), mask, inp["scale"])
        worst = max(worst, float(np.nan_to_num(np.abs(out[b] - ref.transpose(1, 0, 2)), nan=np.inf).max()))
    if mutant == 0:
        assert worst < 1e-12
    else:
        assert worst > 1e-3


@pytest.mark.parametrize("mutant", [0, 3, 4])
def test_each_node_equals_attention_over_its_path(oracle_mod, mutant):
    rng = np.random.default_rng(11)
    worst = 0.0
    for trial in range(6):
        N = int(rng.integers(2, 16))
        w = TINY.replace(B=2, Hq=6, Hkv=3, D=16, prefix=(int(rng.integers(0, 40)),) * 2, tree="random",
                         depth=int(rng.integers(1, 6)), N=N, V=16, seed=100 + trial,
                         dtype=["f32", "bf16"][trial % 2])
        inp = W.generate(w)
        B, Hq, Hkv, D = inp["B"], inp["Hq"], inp["Hkv"], inp["D"]
        out, err = oracle_mod.tree_verify_attn(inp, mutant=mutant)
        assert not err.any()
        out = out.reshape(B, N, Hq, D)
        q = _q64(inp)
        for b in range(B):
            L = int(inp["seq_lens"][b])
            k, v = _logical_kv(inp, b, L + N)
            for n in range(N):
                path = []
                a = n
                while a >= 0:
                    path.append(a)
                    a = int(inp["parent"][b, a])
                keys = list(range(L)) + [L + j for j in sorted(path)]
                kk = _expand_heads(k[keys], Hq // Hkv).transpose(1, 0, 2)
                vv = _expand_heads(v[keys], Hq // Hkv).transpose(1, 0, 2)
                ref = _sdpa(q[b, n][:, None, :], kk, vv, np.ones((1, len(keys)), bool), inp["scale"])[:, 0]
                worst = max(worst, float(np.nan_to_num(np.abs(out[b, n] - ref), nan=np.inf).max()))
    if mutant == 0:
        assert worst < 1e-12
    else:
        assert worst > 1e-3


def test_block_placement_does_not_matter(oracle_mod):
    inp = W.generate(TINY.replace(B=3, prefix=(10, 70), seed=7))
    out1, _ = oracle_mod.tree_verify_attn(inp)
    # move every physical block to a new place and rewrite the table accordingly
    perm = np.random.default_rng(3).permutation(inp["num_blocks"])
    inv = np.argsort(perm)
    moved = dict(inp)
    moved["k_cache"] = inp["k_cache"][perm]
    moved["v_cache"] = inp["v_cache"][perm]
    bt = inp["block_table"].copy()
    bt[bt >= 0] = inv[bt[bt >= 0]]
    moved["block_table"] = bt
    out2, _ = oracle_mod.tree_verify_attn(moved)
    assert np.array_equal(out1, out2)


def test_gqa_group_heads_with_equal_queries_agree(oracle_mod):
    inp = W.generate(TINY.replace(B=1, Hq=8, Hkv=2, seed=9))
    q = inp["q"].copy()
    q[:, :, 1] = q[:, :, 0]  # heads 0 and 1 share kv head 0
    q[:, :, 5] = q[:, :, 4]  # heads 4 and 5 share kv head 1
    inp["q"] = q
    out, _ = oracle_mod.tree_verify_attn(inp)
    out = out.reshape(1, inp["N"], 8, inp["D"])
    assert np.array_equal(out[:, :, 0], out[:, :, 1])
    assert np.array_equal(out[:, :, 4], out[:, :, 5])
    assert not np.allclose(out[:, :, 0], out[:, :, 4])


def test_single_visible_key_returns_its_value(oracle_mod):
    # empty prefix: the root sees only itself
    inp = W.generate(TINY.replace(B=2, prefix=(0, 0), seed=13))
    out, _ = oracle_mod.tree_verify_attn(inp)
    out = out.reshape(2, inp["N"], inp["Hq"], inp["D"])
    for b in range(2):
        _, v = _logical_kv(inp, b, 1)
        for h in range(inp["Hq"]):
            assert np.array_equal(out[b, 0, h], v[0, h // (inp["Hq"] // inp["Hkv"])])


def test_uniform_scores_average_values(oracle_mod):
    # all-zero queries make every visible key equally likely: out = mean of visible values
    inp = W.generate(TINY.replace(B=1, prefix=(20, 20), N=3, tree="chain", seed=17))
    inp["q"] = np.zeros_like(inp["q"])
    out, _ = oracle_mod.tree_verify_attn(inp)
    out = out.reshape(1, 3, inp["Hq"], inp["D"])
    _, v = _logical_kv(inp, 0, 23)
    for n in range(3):
        ref = v[:21 + n].mean(axis=0)  # prefix + root..n
        assert np.allclose(out[0, n, ::4], ref, atol=1e-13)


def test_sampled_rows_match_full_evaluation(oracle_mod):
    inp = W.generate(TINY.replace(B=2, seed=19))
    full, _ = oracle_mod.tree_verify_attn(inp)
    rows = np.array([0, 5, 77, full.shape[0] - 1], dtype=np.int64)
    part, _ = oracle_mod.tree_verify_attn(inp, rows)
    assert np.array_equal(part, full[rows])


def test_error_bits(oracle_mod):
    inp = W.generate(TINY.replace(B=4, seed=23))
    bad = dict(inp)
    par = inp["parent"].copy()
    par[0, 3] = 5  # parent after child
    bad["parent"] = par
    bt = inp["block_table"].copy()
    bt[1, 2] = inp["num_blocks"]  # block id out of range
    bad["block_table"] = bt
    sl = inp["seq_lens"].copy()
    sl[2] = inp["block_table"].shape[1] * 16  # no room for the tree
    bad["seq_lens"] = sl
    out, err = oracle_mod.tree_verify_attn(bad)
    assert list(err) == [oracle_mod.ERR_PARENT, oracle_mod.ERR_BLOCK, oracle_mod.ERR_CAPACITY, 0]
    out = out.reshape(4, -1)
    assert np.isnan(out[:3]).all() and np.isfinite(out[3]).all()
    assert math.isclose(inp["scale"], 1 / 8)
