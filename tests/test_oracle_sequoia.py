"""Pins of the tree-construction oracle (oracle/sequoia.py) to things other than
itself: brute force over every ordered tree, closed forms, and a Monte-Carlo run of
the walk whose expected length the objective claims to be."""
import numpy as np
import pytest

from oracle import sequoia as sq

ACCEPTS = {
    "geometric3": [0.6, 0.2, 0.1],
    "flat5": [0.3, 0.25, 0.2, 0.1, 0.05],
    "power_law8": list(0.9 * np.arange(1, 9) ** -1.5 / np.sum(np.arange(1, 9) ** -1.5)),
    "gap": [0.5, 0.0, 0.3],
    "single": [0.7],
    "sure": [1.0],
    "dirichlet6": list(0.95 * np.random.default_rng(5).dirichlet(np.ones(6))),
}


@pytest.mark.parametrize("name", sorted(ACCEPTS))
def test_dp_equals_brute_force_over_all_trees(name):
    acc = ACCEPTS[name]
    n_max, d_max = 9, 9
    F = sq.dp_values(acc, n_max, d_max)
    for n in range(1, n_max + 1):
        for d in range(0, d_max + 1):
            brute = sq.best_value_brute(n, d, acc)
            assert F[n, d] == pytest.approx(brute, rel=1e-12, abs=1e-12) or (F[n, d] == brute == -np.inf), (n, d)


def test_tree_counts_are_catalan():
    # ordered trees with n nodes: Catalan(n - 1); the brute force sees all of them
    catalan = [1, 1, 2, 5, 14, 42, 132, 429, 1430]
    for n in range(1, 10):
        assert len(sq.ordered_trees(n, n)) == catalan[n - 1]
    assert len(sq.ordered_trees(4, 1)) == 1  # the star
    assert len(sq.ordered_trees(3, 0)) == 0


def test_closed_forms():
    n_max, d_max = 40, 45
    # one rank: the best tree is the rank-1 chain as deep as allowed (the other nodes
    # are never-accepted leaves): sum of p^j for j = 0..min(d, n - 1)
    p = 0.7
    F = sq.dp_values([p], n_max, d_max)
    for n in range(1, n_max + 1):
        for d in range(1, d_max + 1):
            h = min(d, n - 1)
            assert F[n, d] == pytest.approx((1 - p ** (h + 1)) / (1 - p), rel=1e-12)
    # depth 1: the star, 1 + sum of the first n - 1 acceptance probabilities
    acc = ACCEPTS["flat5"]
    F = sq.dp_values(acc, 12, 3)
    for n in range(1, 13):
        assert F[n, 1] == pytest.approx(1 + sum(acc[:n - 1]), rel=1e-12)
    # certain acceptance of the first draft: 1 + min(d, n - 1)
    F = sq.dp_values([1.0], 20, 25)
    for n in range(1, 21):
        for d in range(1, 26):
            assert F[n, d] == 1 + min(d, n - 1)
    # no tree of more than one node at depth 0
    assert np.all(F[2:, 0] == -np.inf) and np.all(F[1, :] == 1)


def test_values_grow_with_size_and_depth():
    F = sq.dp_values(ACCEPTS["power_law8"], 64, 10)
    assert np.all(np.diff(F[1:, 1:], axis=0) >= -1e-12)
    assert np.all(np.diff(F[2:, :], axis=1) >= -1e-12)


@pytest.mark.parametrize("parent", [[-1, 0, 0, 0, 1, 1, 2, 4], [-1, 0, 1, 2, 3], [-1, 0, 0, 0, 0, 0]])
def test_tree_value_is_the_expected_walk_length(parent):
    acc = ACCEPTS["geometric3"]
    rng = np.random.default_rng(11)
    x = sq.simulate_walk(parent, acc, 200_000, rng)
    e = sq.tree_value(parent, acc)
    assert abs(x.mean() - e) < 5 * x.std() / np.sqrt(len(x)), (x.mean(), e)


def test_plan_by_definition():
    acc = ACCEPTS["power_law8"]
    tv = [0.0] + [1.0 + 0.004 * n + 1e-4 * n * n for n in range(1, 33)]
    n, d, s = sq.plan(acc, 32, 8, tv, 0.08)
    F = sq.dp_values(acc, 32, 8)
    grid = [(F[a, b] * tv[1] / (tv[a] + b * 0.08), a, b) for a in range(1, 33) for b in range(9) if F[a, b] > -np.inf]
    assert max(grid)[0] == pytest.approx(s, rel=1e-15)
    assert F[n, d] * tv[1] / (tv[n] + d * 0.08) == s
    # free drafts and flat verification cost: the largest tree wins, at the smallest
    # depth that reaches its best value
    n, d, _ = sq.plan(acc, 16, 6, [0.0] + [1.0] * 16, 0.0)
    F = sq.dp_values(acc, 16, 6)
    assert n == 16 and F[16, d] == F[16].max() and np.all(F[16, :d] < F[16, d])


def test_accept_counts_recover_the_acceptance_vector():
    # walks simulated under a known positional model on a tree where every rank up to 4
    # occurs: accepted / reached estimates accept[k] (binomial, 5 sigma)
    acc = [0.45, 0.2, 0.1, 0.05]
    parent = [-1, 0, 0, 0, 0, 1, 1, 1, 1, 2, 2, 2, 5, 5, 5, 5]
    rng = np.random.default_rng(7)
    nodes, lens = sq.simulate_paths(parent, acc, 15_000, rng)
    reached, accepted = sq.accept_counts([parent] * len(lens), nodes, lens, 4)
    for k in range(4):
        p_hat = accepted[k] / reached[k]
        sigma = np.sqrt(acc[k] * (1 - acc[k]) / reached[k])
        assert abs(p_hat - acc[k]) < 5 * sigma, (k, p_hat, acc[k])
