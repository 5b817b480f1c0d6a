"""Oracle for the draft-tree construction -- TEST INFRASTRUCTURE ONLY.

Only the tests use it; the library never imports or calls it, and it shares no code
with the library's tree construction (`csrc/sequoia_tree.cpp`).

What it follows.  Sequoia summary, sections "Scalable Speculative Decoding" and
"Dynamic Programming": the tree of speculated tokens gets an optimal shape found by
dynamic programming; figure of forward-pass time against input length: the tree size
is chosen from the trade between draft time and verification time.  The pages give
neither the objective nor the recurrence, so the oracle takes the plainest reading
that the rest of the pages supports:

* positional acceptance: accept[k] is the probability that the (k+1)-th drafted
  sibling is the one the walk accepts at a node it has reached (the walk tries the
  children in draft order and accepts at most one; siblings past the vector's end are
  never accepted);
* the objective is the expected number of tokens one verification step generates,
  accepted drafts plus the bonus: E(tree) = sum over nodes of P(walk reaches node),
  with P(root) = 1 and P(child of rank r) = P(parent) * accept[r - 1];
* hardware-aware choice: speedup(n, d) = E_best(n, d) * t_verify[1] /
  (t_verify[n] + d * t_draft), one draft forward per tree level.

Functions, and what pins them (tests/test_oracle_sequoia.py):
  tree_value      the definition of E, written out; pinned by a Monte-Carlo run of
                  the walk it describes and by closed forms (chains, stars);
  ordered_trees   every ordered tree of n nodes and depth <= d (brute force, n <= 10);
  best_value_brute  max of tree_value over ordered_trees: the definition of E_best;
  dp_values       the recurrence, stated plainly; pinned to best_value_brute for every
                  n <= 9 and to closed forms at larger n;
  plan            argmax of the speedup over the dp values, by its definition;
  accept_counts   the positional acceptance counts of walk outputs, by their
                  definition; pinned by recovering a known acceptance vector from
                  simulated walks.
"""
from __future__ import annotations

from functools import lru_cache
from typing import List, Sequence

import numpy as np


def _acc(accept: Sequence[float], rank: int) -> float:
    """Acceptance probability of the sibling of the given rank (1-based)."""
    return float(accept[rank - 1]) if rank <= len(accept) else 0.0


def tree_value(parent: Sequence[int], accept: Sequence[float]) -> float:
    """E(tree): sum over nodes of the probability that the walk reaches them.  Nodes are
    listed with parent[i] < i; a node's rank is 1 + the number of earlier siblings."""
    n = len(parent)
    reach = [0.0] * n
    seen_children = [0] * n
    total = 0.0
    for v in range(n):
        if v == 0:
            reach[v] = 1.0
        else:
            p = int(parent[v])
            seen_children[p] += 1
            reach[v] = reach[p] * _acc(accept, seen_children[p])
        total += reach[v]
    return total


def tree_depth(parent: Sequence[int]) -> int:
    depth = [0] * len(parent)
    for v in range(1, len(parent)):
        depth[v] = depth[int(parent[v])] + 1
    return max(depth)


@lru_cache(maxsize=None)
def _forests(m: int, d: int) -> tuple:
    """Every ordered sequence of trees with m nodes in total, each of depth <= d (a tree
    is the tuple of its children's trees)."""
    if m == 0:
        return ((),)
    out = []
    for a in range(1, m + 1):
        for t in _trees(a, d):
            for rest in _forests(m - a, d):
                out.append((t,) + rest)
    return tuple(out)


@lru_cache(maxsize=None)
def _trees(n: int, d: int) -> tuple:
    if n == 1:
        return ((),)
    if d <= 0:
        return ()
    return tuple(_forests(n - 1, d - 1))


def _to_parent(tree) -> List[int]:
    """Breadth-first numbering, children in their order."""
    parent = [-1]
    queue = [(tree, 0)]
    h = 0
    while h < len(queue):
        t, idx = queue[h]
        h += 1
        for c in t:
            parent.append(idx)
            queue.append((c, len(parent) - 1))
    return parent


def ordered_trees(n: int, max_depth: int) -> List[List[int]]:
    """All ordered trees of n nodes and depth <= max_depth, as parent arrays."""
    return [_to_parent(t) for t in _trees(n, max_depth)]


def best_value_brute(n: int, max_depth: int, accept: Sequence[float]) -> float:
    trees = ordered_trees(n, max_depth)
    return max((tree_value(p, accept) for p in trees), default=-np.inf)


def dp_values(accept: Sequence[float], n_max: int, d_max: int) -> np.ndarray:
    """E_best(n, d) for n = 0..n_max, d = 0..d_max (row 0 is 0; -inf where no tree
    exists).  F(1, d) = 1; F(n > 1, 0) = -inf; for d >= 1, F(n, d) = 1 + G_d(1, n - 1)
    where G_d(r, m) is the best value of m nodes hung below a node as children of rank
    r, r + 1, ...: G_d(r, 0) = 0, G_d(K + 1, m) = 0 (never-accepted leaves), and
    G_d(r, m) = max over a in 1..m with F(a, d - 1) > -inf of
    accept[r-1] * F(a, d - 1) + G_d(r + 1, m - a)."""
    K = len(accept)
    F = np.full((n_max + 1, d_max + 1), -np.inf)
    F[0, :] = 0.0
    F[1, :] = 1.0
    for d in range(1, d_max + 1):
        G = np.zeros(n_max)  # G_d(K + 1, m) for m = 0..n_max-1
        for r in range(K, 0, -1):
            Gr = np.zeros(n_max)
            for m in range(1, n_max):
                a = np.arange(1, m + 1)
                a = a[F[a, d - 1] > -np.inf]  # subtree sizes that fit in depth d - 1
                cand = float(accept[r - 1]) * F[a, d - 1] + G[m - a]
                Gr[m] = cand.max()
            G = Gr
        for n in range(2, n_max + 1):
            F[n, d] = 1.0 + G[n - 1]
    return F


def plan(accept: Sequence[float], n_max: int, d_max: int, t_verify: Sequence[float], t_draft: float):
    """(n, d, speedup) maximising E_best(n, d) t_verify[1] / (t_verify[n] + d t_draft);
    ties to the smaller n, then the smaller d."""
    F = dp_values(accept, n_max, d_max)
    best = (-np.inf, 1, 0)
    for n in range(1, n_max + 1):
        for d in range(0, d_max + 1):
            if F[n, d] == -np.inf:
                continue
            s = F[n, d] * t_verify[1] / (t_verify[n] + d * t_draft)
            if s > best[0]:
                best = (s, n, d)
    return best[1], best[2], best[0]


def simulate_walk(parent: Sequence[int], accept: Sequence[float], trials: int, rng: np.random.Generator) -> np.ndarray:
    """Generated tokens per step (accepted drafts + 1) of `trials` walks: at a reached
    node the accepted rank is drawn from accept (none with the remaining mass); the walk
    moves to the child of that rank if the node has one, else it stops."""
    n = len(parent)
    kids: List[List[int]] = [[] for _ in range(n)]
    for v in range(1, n):
        kids[int(parent[v])].append(v)
    probs = np.append(np.asarray(accept, np.float64), max(0.0, 1.0 - float(np.sum(accept))))
    out = np.ones(trials, np.int64)
    node = np.zeros(trials, np.int64)
    alive = np.ones(trials, bool)
    while alive.any():
        idx = np.flatnonzero(alive)
        rank = rng.choice(len(probs), size=len(idx), p=probs / probs.sum()) + 1  # 1-based; len(probs) = none
        nxt = np.full(len(idx), -1)
        for j, (v, r) in enumerate(zip(node[idx], rank)):
            if r <= len(accept) and r <= len(kids[v]):
                nxt[j] = kids[v][r - 1]
        moved = nxt >= 0
        out[idx[moved]] += 1
        node[idx[moved]] = nxt[moved]
        alive[idx[~moved]] = False
    return out


def accept_counts(parent, accepted_nodes, accept_len, K: int):
    """For every reached node (on an accepted path) with c children: reached[k] += 1 for
    ranks k + 1 <= min(c, K); accepted[r - 1] += 1 when the path goes on to the child of
    rank r <= K.  Sequences with accept_len < 0 are skipped."""
    reached = np.zeros(K, np.int64)
    accepted = np.zeros(K, np.int64)
    for b in range(len(accept_len)):
        A = int(accept_len[b])
        if A < 0:
            continue
        par = [int(x) for x in parent[b]]
        kids = [[] for _ in par]
        for c in range(1, len(par)):
            kids[par[c]].append(c)
        path = [int(x) for x in accepted_nodes[b][:A + 1]]
        for j, v in enumerate(path):
            for k in range(min(len(kids[v]), K)):
                reached[k] += 1
            if j < A:
                r = kids[v].index(path[j + 1]) + 1
                if r <= K:
                    accepted[r - 1] += 1
    return reached, accepted


def simulate_paths(parent, accept: Sequence[float], trials: int, rng: np.random.Generator):
    """Accepted paths (accepted_nodes rows padded with -1, accept_len) of `trials` walks
    on one tree under the positional model, for the estimator's pin."""
    n = len(parent)
    kids: List[List[int]] = [[] for _ in range(n)]
    for v in range(1, n):
        kids[int(parent[v])].append(v)
    probs = np.append(np.asarray(accept, np.float64), max(0.0, 1.0 - float(np.sum(accept))))
    probs = probs / probs.sum()
    nodes = np.full((trials, n), -1, np.int32)
    lens = np.zeros(trials, np.int32)
    for t in range(trials):
        v, path = 0, [0]
        while True:
            r = int(rng.choice(len(probs), p=probs)) + 1
            if r > len(accept) or r > len(kids[v]):
                break
            v = kids[v][r - 1]
            path.append(v)
        nodes[t, :len(path)] = path
        lens[t] = len(path) - 1
    return nodes, lens
