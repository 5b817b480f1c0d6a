"""The library's tree construction (host-side C ABI, no GPU) against the oracle:
the value table element by element, trees that are valid for the walk and attain the
best value, and the hardware-aware choice of size and depth."""
import time

import numpy as np
import pytest

import tree_speculative_decoding_03_gb300 as tsv
from oracle import sequoia as sq

ACCEPTS = {
    "geometric3": [0.6, 0.2, 0.1],
    "power_law16": list(0.92 * np.arange(1, 17) ** -1.3 / np.sum(np.arange(1, 17) ** -1.3)),
    "gap": [0.5, 0.0, 0.3],
    "single": [0.7],
    "dirichlet10": list(0.97 * np.random.default_rng(8).dirichlet(np.ones(10))),
}


@pytest.fixture(scope="module", autouse=True)
def lib():
    tsv.build()
    return tsv.load()


def _same(a, b):
    fin = np.isfinite(b)
    return np.array_equal(np.isfinite(a), fin) and np.all(a[~fin] == b[~fin]) and \
        np.allclose(a[fin], b[fin], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("name", sorted(ACCEPTS))
def test_value_table_matches_oracle(name):
    acc = ACCEPTS[name]
    for n_max, d_max in [(1, 0), (9, 9), (128, 12)]:
        assert _same(tsv.sequoia_values(acc, n_max, d_max), sq.dp_values(acc, n_max, d_max)), (n_max, d_max)


def _valid_for_walk(parent, n, max_depth):
    assert len(parent) == n and parent[0] == -1
    assert all(0 <= parent[i] < i for i in range(1, n))
    # breadth-first: parents appear in non-decreasing order, so siblings are contiguous and
    # a node's children have increasing indices (the walk tries them in index order)
    assert all(parent[i - 1] <= parent[i] for i in range(2, n))
    assert sq.tree_depth(parent) <= max_depth


@pytest.mark.parametrize("name", sorted(ACCEPTS))
def test_tree_is_valid_and_attains_the_best_value(name):
    acc = ACCEPTS[name]
    F = sq.dp_values(acc, 128, 16)
    for n, d in [(1, 0), (1, 3), (2, 1), (8, 3), (9, 2), (30, 5), (64, 8), (128, 10), (128, 16)]:
        parent, e = tsv.sequoia_tree(acc, n, d)
        _valid_for_walk(list(parent), n, d)
        assert e == pytest.approx(F[n, d], rel=1e-12)
        assert sq.tree_value(parent, acc) == pytest.approx(F[n, d], rel=1e-12)
    # depth past n - 1 changes nothing
    p1, e1 = tsv.sequoia_tree(acc, 12, 11)
    p2, e2 = tsv.sequoia_tree(acc, 12, 100)
    assert e1 == e2 and np.array_equal(p1, p2)


def test_tree_small_cases_against_brute_force():
    acc = ACCEPTS["geometric3"]
    for n in range(1, 9):
        for d in range(1 if n > 1 else 0, n):
            parent, e = tsv.sequoia_tree(acc, n, d)
            assert e == pytest.approx(sq.best_value_brute(n, d, acc), rel=1e-12)
            assert list(parent) in sq.ordered_trees(n, d)


def test_plan_matches_oracle():
    rng = np.random.default_rng(3)
    for name in sorted(ACCEPTS):
        acc = ACCEPTS[name]
        for n_max, d_max in [(16, 6), (64, 10)]:
            # verification time that grows with the tree once it is large (memory- then compute-bound)
            tv = np.array([0.0] + [1.0 + 0.002 * n + 4e-5 * n * n for n in range(1, n_max + 1)])
            t_draft = float(rng.uniform(0.02, 0.2))
            assert tsv.sequoia_plan(acc, n_max, d_max, tv, t_draft)[:2] == sq.plan(acc, n_max, d_max, tv, t_draft)[:2]
            s_lib = tsv.sequoia_plan(acc, n_max, d_max, tv, t_draft)[2]
            assert s_lib == pytest.approx(sq.plan(acc, n_max, d_max, tv, t_draft)[2], rel=1e-12)


def test_argument_errors():
    acc = [0.5, 0.3]
    bad = [([0.5, 0.6], 8, 3), ([-0.1], 8, 3), ([np.nan], 8, 3), (acc, 0, 3), (acc, 129, 3), (acc, 8, -1)]
    for a, n, d in bad:
        with pytest.raises(tsv.TsvError) as e:
            tsv.sequoia_values(a, n, d)
        assert e.value.status == tsv.TSV_ERR_ARG
    with pytest.raises(tsv.TsvError):
        tsv.sequoia_tree(acc, 5, 0)  # five nodes do not fit in depth 0
    with pytest.raises(tsv.TsvError):
        tsv.sequoia_plan(acc, 4, 2, [0.0, 1.0, 1.0, 0.0, 1.0], 0.1)  # t_verify[3] = 0
    with pytest.raises(tsv.TsvError):
        tsv.sequoia_plan(acc, 4, 2, [0.0, 1.0, 1.0, 1.0, 1.0], -0.1)


def test_largest_problem_runs_in_well_under_a_second():
    acc = list(0.95 * np.arange(1, 128) ** -1.2 / np.sum(np.arange(1, 128) ** -1.2))
    t0 = time.perf_counter()
    v = tsv.sequoia_values(acc, 128, 127)
    dt = time.perf_counter() - t0
    print(f"tree construction, n_max 128, depth 127, 127 ranks: {dt * 1e3:.1f} ms")
    assert np.all(np.isfinite(v[1:, 1:])) and dt < 5.0


def test_accept_counts_hand_case():
    # root has children 1, 2 (ranks 1, 2); node 1 has 3, 4; node 2 has 5.  Path 0 -> 2 -> 5.
    parent = np.array([[-1, 0, 0, 1, 1, 2]], np.int32)
    nodes = np.array([[0, 2, 5, -1, -1, -1]], np.int32)
    reached, accepted = tsv.sequoia_accept_counts(parent, nodes, np.array([2], np.int32), K=2)
    assert list(reached) == [2, 1] and list(accepted) == [1, 1]
    assert [list(x) for x in sq.accept_counts(parent, nodes, [2], 2)] == [[2, 1], [1, 1]]


def test_accept_counts_match_oracle_on_walk_outputs():
    import oracle
    import workloads as W
    w = W.CONFIGS[3].replace(B=48, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=40, depth=6, V=800, T=1.0, seed=17)
    inp = W.generate(w)
    o = oracle.tree_reject_sample(inp)
    inp2 = dict(inp)
    inp2["parent"] = inp["parent"].copy()
    inp2["parent"][3, 5] = 7  # a bad tree: the walk flags it (accept_len -1) and the counts skip it
    o2 = oracle.tree_reject_sample(inp2)
    assert o2["accept_len"][3] == -1
    for K in (1, 4, 12):
        r, a = tsv.sequoia_accept_counts(inp["parent"], o["accepted_nodes"], o["accept_len"], K)
        r0, a0 = sq.accept_counts(inp["parent"], o["accepted_nodes"], o["accept_len"], K)
        assert np.array_equal(r, r0) and np.array_equal(a, a0) and r.sum() > 0
        # accumulation over two steps
        r2, a2 = tsv.sequoia_accept_counts(inp2["parent"], o2["accepted_nodes"], o2["accept_len"], K,
                                           reached=r.copy(), accepted=a.copy())
        r1, a1 = sq.accept_counts(inp2["parent"], o2["accepted_nodes"], o2["accept_len"], K)
        assert np.array_equal(r2, r + r1) and np.array_equal(a2, a + a1)


def test_accept_counts_reject_inconsistent_inputs():
    parent = np.array([[-1, 0, 0, 1]], np.int32)
    with pytest.raises(tsv.TsvError):  # 3 is not a child of 2
        tsv.sequoia_accept_counts(parent, np.array([[0, 2, 3, -1]], np.int32), np.array([2], np.int32), 2)
    with pytest.raises(tsv.TsvError):  # parent[2] = 2 is not a tree
        tsv.sequoia_accept_counts(np.array([[-1, 0, 2, 1]], np.int32), np.array([[0, 1, -1, -1]], np.int32),
                                  np.array([1], np.int32), 2)
