"""The seeded input generator: tree shapes and layouts of the five workloads."""
import numpy as np

import workloads as W


def _levels(parent):
    d = np.zeros(len(parent), int)
    for i in range(1, len(parent)):
        assert 0 <= parent[i] < i
        d[i] = d[parent[i]] + 1
    return np.bincount(d)


def test_tree_shapes():
    assert list(_levels(W.binary_tree(15))) == [1, 2, 4, 8]
    assert list(_levels(W.chain_tree(6))) == [1] * 6
    assert list(_levels(W.topk_tree((4, 3, 2, 2, 1, 1), 60))) == [1, 4, 7, 9, 13, 13, 13]
    rng = np.random.default_rng(0)
    for N, depth in ((128, 10), (64, 8)):
        for _ in range(20):
            lv = _levels(W.random_tree(rng, N, depth))
            assert lv.sum() == N and len(lv) - 1 == depth


def test_generator_is_deterministic_and_paged():
    w = W.CONFIGS[4].replace(B=5, Hq=8, Hkv=2, D=16, V=64, prefix=(3, 90))
    a, b = W.generate(w), W.generate(w)
    for k in ("parent", "seq_lens", "block_table", "q", "k_cache", "target_logits", "draft_tokens", "u_accept"):
        assert np.array_equal(a[k], b[k])
    bt = a["block_table"]
    used = bt[bt >= 0]
    assert len(np.unique(used)) == len(used) == a["num_blocks"]  # every block owned exactly once
    for s in range(5):
        need = -(-(int(a["seq_lens"][s]) + w.N) // 16)
        assert (bt[s, :need] >= 0).all() and (bt[s, need:] == -1).all()
    assert len(a["pq_seqs"]) == 0 or np.array_equal(a["target_logits"][a["pq_seqs"]],
                                                     2 * (a["target_logits"][a["pq_seqs"]] / 2))
    # siblings are distinct tokens (drafted without replacement)
    for s in range(5):
        for i in range(w.N):
            kids = np.nonzero(a["parent"][s] == i)[0]
            assert len(set(a["draft_tokens"][s, kids])) == len(kids)
