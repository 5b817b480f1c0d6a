"""Pins for the oracle's KV-cache compaction (CPU only).

The sglang report ("Tree-based Speculative Decoding (EAGLE) Implementation
Summary"; "Issue: Speculative Decoding on vLLM") says the KV cache must be
rewritten for the accepted indices, and the SGLang page ("Speculative Decoding",
prefix match) that rejected tokens' KV is evicted.  Pins, checked through a
logical-order view of the paged cache built with numpy fancy indexing:
  * after compaction, logical slot L + j holds the pre-call bytes of slot
    L + path[j] for j = 1..A, including paths whose sources overlap destinations;
  * every other slot keeps its bytes; the new length is L + 1 + A;
  * a chain accepted in full is the identity; a sequence marked failed is untouched.
A planted off-by-one must fail.
"""
import numpy as np
import pytest

import workloads as W


def _logical(inp, cache, b, upto):
    bs = inp["block_size"]
    t = np.arange(upto)
    phys = inp["block_table"][b, t // bs].astype(np.int64) * bs + t % bs
    return cache.reshape(-1, inp["Hkv"], inp["D"])[phys]


def _random_paths(rng, parent, B):
    N = parent.shape[1]
    nodes = np.full((B, N), -1, np.int32)
    lens = np.zeros(B, np.int32)
    for b in range(B):
        path = [0]
        while True:
            kids = [c for c in range(N) if parent[b, c] == path[-1]]
            if not kids or rng.random() < 0.2:
                break
            path.append(int(rng.choice(kids)))
        nodes[b, :len(path)] = path
        lens[b] = len(path) - 1
    return nodes, lens


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mutant", [0, 6])
def test_path_rows_move_to_contiguous_slots(oracle_mod, dtype, mutant):
    w = W.CONFIGS[3].replace(B=6, Hq=4, Hkv=2, D=16, prefix=(5, 60), N=24, depth=8, V=32, dtype=dtype, seed=31)
    inp = W.generate(w)
    rng = np.random.default_rng(0)
    nodes, lens = _random_paths(rng, inp["parent"], inp["B"])
    # force one overlapping path: 0 -> 2 -> 5 style (sources overlap destinations)
    nodes[0] = -1
    nodes[0, :3] = [0, 1, 2]
    lens[0] = 2
    k, v, new_len, err = oracle_mod.kv_compact_accepted(inp, nodes, lens, mutant=mutant)
    assert not err.any()
    ok = True
    for b in range(inp["B"]):
        L, A, N = int(inp["seq_lens"][b]), int(lens[b]), inp["N"]
        ok &= new_len[b] == L + 1 + A
        for old, new in ((inp["k_cache"], k), (inp["v_cache"], v)):
            before = _logical(inp, old, b, L + N)
            after = _logical(inp, new, b, L + N)
            want = before.copy()
            want[L + 1:L + 1 + A] = before[L + nodes[b, 1:A + 1]]
            ok &= np.array_equal(want.view(np.uint8), after.view(np.uint8))
    # blocks nobody references are untouched (all blocks are referenced here)
    assert ok == (mutant == 0)


def test_overlap_path_0_2_5(oracle_mod):
    w = W.CONFIGS[0].replace(B=1, D=8, Hkv=2, Hq=2, prefix=(3, 3), tree="chain", N=8, V=4, seed=2)
    inp = W.generate(w)
    parent = np.array([[-1, 0, 0, 1, 1, 2, 2, 3]], np.int32)
    inp["parent"] = parent
    nodes = np.array([[0, 2, 5, -1, -1, -1, -1, -1]], np.int32)
    k, v, new_len, err = oracle_mod.kv_compact_accepted(inp, nodes, np.array([2], np.int32))
    before = _logical(inp, inp["k_cache"], 0, 11)
    after = _logical(inp, k, 0, 11)
    assert np.array_equal(after[4], before[5]) and np.array_equal(after[5], before[8])
    assert np.array_equal(after[:4], before[:4]) and np.array_equal(after[6:], before[6:])
    assert new_len[0] == 6 and err[0] == 0


def test_full_chain_accept_is_identity_and_failed_sequence_untouched(oracle_mod):
    w = W.CONFIGS[1].replace(B=2, Hq=4, Hkv=2, D=16, prefix=(40, 40), V=8, seed=3)
    inp = W.generate(w)
    nodes = np.array([np.arange(6), np.full(6, -1)], np.int32)
    lens = np.array([5, -1], np.int32)
    k, v, new_len, err = oracle_mod.kv_compact_accepted(inp, nodes, lens)
    assert np.array_equal(k.view(np.uint8), inp["k_cache"].view(np.uint8))
    assert np.array_equal(v.view(np.uint8), inp["v_cache"].view(np.uint8))
    assert list(new_len) == [46, 40] and not err.any()


def test_bad_path_and_block_errors(oracle_mod):
    w = W.CONFIGS[1].replace(B=3, Hq=4, Hkv=2, D=16, prefix=(40, 40), V=8, seed=4)
    inp = W.generate(w)
    nodes = np.array([[0, 2, 1, -1, -1, -1], [1, 2, -1, -1, -1, -1], [0, 1, 2, -1, -1, -1]], np.int32)
    lens = np.array([2, 1, 2], np.int32)
    bt = inp["block_table"].copy()
    bt[2, 2] = -5
    inp["block_table"] = bt
    k, v, new_len, err = oracle_mod.kv_compact_accepted(inp, nodes, lens)
    assert list(err) == [1, 1, 2]
    assert list(new_len) == [40, 40, 40]
    assert np.array_equal(k.view(np.uint8), inp["k_cache"].view(np.uint8))
