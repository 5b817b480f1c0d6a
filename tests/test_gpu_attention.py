"""GPU parity of tsv_tree_verify_attn against the fp64 oracle.

Tolerances: max |gpu - oracle| <= 2e-2 for bf16 inputs/outputs, <= 1e-4 for fp32
(the stated bounds of the verification step).  Small cases are compared on every
row; the full-size workloads, in the launch configuration the benchmark times, on
rows stratified over the work layout (every unit, row group and M tile)."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import run_attn

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-4}


def _check_all_rows(inp):
    got, gerr = run_attn(inp)
    want, oerr = oracle.tree_verify_attn(inp)
    assert np.array_equal(gerr, oerr)
    ok = ~np.isnan(want).any(axis=1)
    assert np.isnan(got[~ok]).all()
    err = np.abs(got[ok] - want[ok]).max() if ok.any() else 0.0
    assert err <= TOL[inp["dtype"]], err
    return err


def test_tiny_binary_tree_fp32_all_rows():
    _check_all_rows(W.generate(W.CONFIGS[0]))


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("f32", 128)])
def test_ragged_prefixes_random_trees(dtype, D):
    # prefixes spanning several key tiles and chunks with a ragged tail; 148 query rows per kv head
    w = W.CONFIGS[3].replace(B=3, Hq=16, Hkv=4, D=D, dtype=dtype, prefix=(1, 1500), N=37, depth=6, V=64, seed=77)
    _check_all_rows(W.generate(w))


@pytest.mark.parametrize("N,tree,prefix", [(1, "chain", (0, 0)), (6, "chain", (0, 40)), (128, "random", (300, 700)),
                                           (64, "random", (2048, 2048)), (15, "binary", (4095, 4097))])
def test_edge_shapes(N, tree, prefix):
    w = W.CONFIGS[2].replace(B=2, Hq=8, Hkv=2, N=N, tree=tree, depth=10 if tree == "random" else 0,
                             prefix=prefix, V=256, seed=5 + N)
    _check_all_rows(W.generate(w))


def test_gqa_8_and_block_size_32():
    w = W.CONFIGS[4].replace(B=2, Hq=16, Hkv=2, prefix=(100, 900), N=20, V=300, block_size=32, seed=8)
    _check_all_rows(W.generate(w))


def test_bad_sequences_are_poisoned_and_flagged():
    inp = W.generate(W.CONFIGS[1].replace(B=4, Hq=8, Hkv=2, prefix=(300, 300), V=64, seed=3))
    inp["parent"] = inp["parent"].copy()
    inp["parent"][0, 2] = 3
    inp["block_table"] = inp["block_table"].copy()
    inp["block_table"][1, 5] = inp["num_blocks"] + 10
    inp["seq_lens"] = inp["seq_lens"].copy()
    inp["seq_lens"][2] = -1
    _check_all_rows(inp)


def test_many_units_two_row_groups_flagged_in_the_middle():
    # 12 sequences of mixed lengths (empty prefixes included) cut across CTAs; 320 rows
    # per kv head = a full and a partial row group; two flagged sequences mid-batch
    w = W.CONFIGS[3].replace(B=12, Hq=32, Hkv=4, N=40, depth=6, prefix=(0, 2600), V=64, seed=91)
    inp = W.generate(w)
    inp["seq_lens"] = inp["seq_lens"].copy()
    inp["seq_lens"][3] = 0
    inp["seq_lens"][5] = -7
    inp["block_table"] = inp["block_table"].copy()
    inp["block_table"][8, 0] = -1
    _check_all_rows(inp)


def _unit_rows(inp, rng):
    """Rows to compare at full size, stratified over the work layout: in every (sequence,
    kv head) unit, the first and last row of every 128-row M tile and one random row of
    each, so every unit, row group and M tile boundary -- and with them every stream-K
    split and merge -- is checked.  Flat row id = (b*N + n)*Hq + h, unit row r = n*G + j."""
    B, N, Hq, Hkv = inp["B"], inp["N"], inp["Hq"], inp["Hkv"]
    G = Hq // Hkv
    R = N * G
    picks = []
    for t0 in range(0, R, 128):
        t1 = min(R, t0 + 128) - 1
        picks.append(np.array([t0, t1]))
        picks.append(rng.integers(t0, t1 + 1, 1))
    unit_rows = np.unique(np.concatenate(picks))
    b, g, r = np.meshgrid(np.arange(B), np.arange(Hkv), unit_rows, indexing="ij")
    n, j = r // G, r % G
    return np.unique(((b * N + n) * Hq + g * G + j).ravel())


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_full_size_sampled_rows(cfg):
    inp = W.generate(W.CONFIGS[cfg])
    got, gerr = run_attn(inp)
    assert not gerr.any()
    assert np.isfinite(got).all()
    rows = _unit_rows(inp, np.random.default_rng(cfg))
    assert len(rows) >= inp["B"] * inp["Hkv"] * 3
    want, _ = oracle.tree_verify_attn(inp, rows)
    err = np.abs(got[rows] - want).max()
    assert err <= TOL[inp["dtype"]], err
