"""Host-side logic of bench.py: algorithmic byte counts and the replica aggregation
(max over ranks) with world_size 2 over gloo."""
import os

import numpy as np
import torch.multiprocessing as mp

import bench
import workloads as W


def test_algorithmic_bytes():
    inp = W.generate(W.CONFIGS[1].replace(B=2, V=64))
    # K and V of 2054 slots x 8 heads x 128 dims x 2 bytes, both sequences; Q in and O out
    assert bench.attn_bytes(inp, append=False) == 2 * 2054 * 8 * 128 * 2 * 2 + 2 * 2 * 6 * 32 * 128 * 2
    # the fused append also reads the tree's new K/V rows and writes them into the cache
    assert bench.attn_bytes(inp) - bench.attn_bytes(inp, append=False) == 2 * 2 * 2 * 6 * 8 * 128 * 2
    an = np.array([[0, 1, 2, -1, -1, -1], [0, -1, -1, -1, -1, -1]])
    al = np.array([2, 0])
    # seq 0 visits 3 nodes; first children accepted at 0 and 1; node 2 rejects its child -> draft row read
    # seq 1 visits the root and rejects its only child -> draft row read
    assert bench.verify_bytes(inp, an, al) == (3 + 1 + 1 + 1) * 64 * 4
    assert bench.compact_bytes(inp, al) == 2 * 8 * 128 * 2 * 2 * 2


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    secs = [0.5, 2.0][rank]
    out[rank] = bench.whole_job_rate(100.0, secs, world)
    dist.destroy_process_group()


def test_replica_rate_uses_slowest_rank():
    mgr = mp.Manager()
    out = mgr.dict()
    port = 29500 + os.getpid() % 1000
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1] == 2 * 100.0 / 2.0


def test_attention_flops():
    inp = W.generate(W.CONFIGS[1].replace(B=2, V=64))
    assert bench.attn_flops(inp) == 2 * 4 * 6 * 32 * 128 * (2048 + 6)


def test_parity_summary_counts_identical_exempt_and_mismatched():
    import oracle
    inp = W.generate(W.CONFIGS[3].replace(B=6, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=20, depth=5, V=300, seed=5))
    o = oracle.tree_reject_sample(inp)
    g = {k: v.copy() for k, v in o.items()}
    # seq 1: a different bonus with u_bonus moved onto the oracle's CDF boundary -> exempt near tie
    lo, hi = o["bonus_cdf"][1]
    inp["u_bonus"] = inp["u_bonus"].copy()
    inp["u_bonus"][1] = np.float32(hi)
    g["bonus_token"][1] += 1
    # seq 2: a different bonus far from any boundary -> mismatched
    inp["u_bonus"][2] = np.float32(0.5 * (o["bonus_cdf"][2][0] + o["bonus_cdf"][2][1]))
    g["bonus_token"][2] += 1
    rows = np.array([0, 3])
    want = np.zeros((2, 64))
    got = np.zeros((inp["B"] * inp["N"] * inp["Hq"], 64))
    got[3, 5] = 0.01
    p = bench.parity_summary(inp, g, o, rows, want, got)
    assert (p["identical"], p["exempt_near_ties"], p["mismatched"]) == (4, 1, 1)
    assert p["attn_max_abs_err"] == 0.01 and not p["ok"]


def test_tree_rows_are_the_cache_slots_after_each_prefix():
    inp = W.generate(W.CONFIGS[3].replace(B=3, Hq=4, Hkv=2, D=64, prefix=(5, 70), N=9, depth=4, V=32, seed=2))
    kn, vn = bench.tree_rows(inp)
    bs = inp["block_size"]
    for b in range(3):
        for j in range(9):
            t = int(inp["seq_lens"][b]) + j
            blk = inp["block_table"][b, t // bs]
            assert np.array_equal(kn[b, j], inp["k_cache"][blk, t % bs])
            assert np.array_equal(vn[b, j], inp["v_cache"][blk, t % bs])
