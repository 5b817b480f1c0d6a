"""Pins for the oracle's rejection-sampling tree walk (CPU only).

  * hand-worked cases (tests/golden/verifier_hand.json) computed from the rules of
    statistical-learning-notes ch.07 "Speculative Decoding", section "Draft Token
    Validation", and the Sequoia summary, section "Robust Sampling";
  * losslessness: the emitted tokens follow the target distribution (vLLM PR
    #2188 "Feature list": rejection sampling guarantees the target model's
    distribution) -- chi-square over 10^6 seeded trials on a 16-token vocabulary,
    for a chain, for siblings drafted without replacement, and at T = 0.6, on the
    first token and on the second token given the first;
  * p == q accepts every draft (SGLang "SpeculativeDecoding", case "Full Match");
  * T = 0 reduces to greedy argmax matching, checked against an independent walk;
  * no match returns exactly one target token, and the page's prefix-match example
    ("and it's so hot" vs "and it's very warm") keeps the first two drafts.
Planted mistakes (residual left unnormalised, residual skipped) and the walk for
independent drafts applied to siblings drafted without replacement must fail the
chi-square pin.  The walk for siblings drafted independently from q (with
replacement, q kept after a rejection -- the SpecInfer variant the Sequoia summary
compares against) passes it on such drafts, where the without-replacement walk fails.
"""
import json
import os

import numpy as np
import pytest
from scipy import stats

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "verifier_hand.json")


def _softmax64(x, T):
    z = np.asarray(x, np.float64) / T
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def _inp(logits, probs, tokens, parent, ua, ub, T):
    logits = np.ascontiguousarray(logits, np.float32)
    B, N, V = logits.shape
    return dict(B=B, N=N, V=V, T=T, target_logits=logits,
                draft_probs=None if probs is None else np.ascontiguousarray(probs, np.float32),
                draft_tokens=np.ascontiguousarray(tokens, np.int32),
                parent=np.ascontiguousarray(parent, np.int32),
                u_accept=np.ascontiguousarray(ua, np.float32), u_bonus=np.ascontiguousarray(ub, np.float32))


# ----------------------------------------------------------------------------- hand-worked

def _golden_cases():
    g = json.load(open(GOLDEN))
    for c in g["cases"]:
        yield g, c


@pytest.mark.parametrize("case", [c["name"] for _, c in _golden_cases()])
def test_hand_worked_cases(oracle_mod, case):
    g, c = next((g, c) for g, c in _golden_cases() if c["name"] == case)
    V, parent = g["V"], np.array(g["parent"])
    N = len(parent)
    logits = np.log(np.array(g["probs_target"], np.float64))[None]
    probs = np.array(g["draft_probs"], np.float64)
    for k, row in c.get("draft_probs_override", {}).items():
        probs[int(k)] = row
    r = oracle_mod.tree_reject_sample(_inp(logits, probs[None], [c["tokens"]], parent[None],
                                           [c["u_accept"]], [c["u_bonus"]], c["T"]))
    assert r["err"][0] == 0
    assert list(r["accepted_nodes"][0]) == c["accepted_nodes"]
    assert r["accept_len"][0] == c["accept_len"]
    assert r["bonus_token"][0] == c["bonus_token"]
    assert list(r["out_tokens"][0]) == c["out_tokens"]
    for j, want in enumerate(c["ratio"]):
        got = r["ratio"][0, j]
        if want is None:
            assert np.isnan(got)
        elif want == "inf":
            assert np.isinf(got)
        else:
            assert abs(got - want) < 1e-6, (j, got, want)
    assert V == 3 and N == 4


# ----------------------------------------------------------------------------- losslessness

def _markov_trials(rng, n, parent, V, T, tgt_table, drf_table, x0, iid=False):
    """n independent verification trials of one tree topology.  The target and
    draft distributions after a node depend only on that node's token (a Markov
    target), so the emitted chain must follow softmax(tgt_table[x] / T).  Siblings
    are drafted without replacement (Gumbel top-k), or independently if iid."""
    N = len(parent)
    kids = [[] for _ in range(N)]
    for c in range(1, N):
        kids[parent[c]].append(c)
    tok = np.empty((n, N), np.int64)
    tok[:, 0] = x0
    for i in range(N):
        if not kids[i]:
            continue
        q = drf_table[tok[:, i]].astype(np.float64)
        if iid:
            cdf = np.cumsum(q, axis=1)
            u = rng.random((n, len(kids[i]))) * cdf[:, -1:]
            tok[:, kids[i]] = np.minimum((u[:, :, None] >= cdf[:, None, :]).sum(axis=2), V - 1)
            continue
        with np.errstate(divide="ignore"):
            key = np.log(q) + rng.gumbel(size=q.shape)
        top = np.argsort(-key, axis=1, kind="stable")[:, :len(kids[i])]
        tok[:, kids[i]] = top
    logits = tgt_table[tok]
    probs = drf_table[tok]
    ua = rng.random((n, N), dtype=np.float32)
    ub = rng.random(n, dtype=np.float32)
    return _inp(logits, probs, tok, np.tile(parent, (n, 1)), ua, ub, T)


def _chi2_pvalues(oracle_mod, parent, T, trials=1_000_000, chunk=200_000, seed=0, mutant=0, V=16, iid=False,
                  replacement=False):
    rng = np.random.default_rng(seed)
    tgt_table = rng.normal(0.0, 1.0, (V, V)).astype(np.float32)
    drf_logits = tgt_table + rng.normal(0.0, 0.8, (V, V)).astype(np.float32)
    drf_table = _softmax64(drf_logits, T).astype(np.float32)
    x0 = 3
    first = np.zeros(V, np.int64)
    pair = np.zeros((V, V), np.int64)
    for s in range(0, trials, chunk):
        inp = _markov_trials(rng, min(chunk, trials - s), np.array(parent), V, T, tgt_table, drf_table, x0, iid=iid)
        r = oracle_mod.tree_reject_sample(inp, mutant=mutant, replacement=replacement)
        assert not r["err"].any()
        ot = r["out_tokens"]
        if (ot[:, 0] < 0).any():  # no token emitted at all: not a distribution over the vocab
            return 0.0, 0.0, first
        first += np.bincount(ot[:, 0], minlength=V)
        two = r["accept_len"] >= 1
        np.add.at(pair, (ot[two, 0], ot[two, 1]), 1)
    p_first = _softmax64(tgt_table[x0], T)
    p1 = stats.chisquare(first, p_first * first.sum()).pvalue
    stat, dof = 0.0, 0
    p_next = _softmax64(tgt_table, T)
    for x in range(V):
        m = pair[x].sum()
        if m >= 200:
            stat += stats.chisquare(pair[x], p_next[x] * m).statistic
            dof += V - 1
    p2 = stats.chi2.sf(stat, dof) if dof else 1.0
    return p1, p2, first


CHAIN = [-1, 0, 1, 2]
SIBLINGS = [-1, 0, 0, 0, 1, 1, 2, 2, 3, 3]  # 3 siblings drafted without replacement, depth 2


@pytest.mark.parametrize("parent,T", [(CHAIN, 1.0), (SIBLINGS, 1.0), (SIBLINGS, 0.6)],
                         ids=["chain_T1", "siblings_T1", "siblings_T0.6"])
def test_output_follows_target_distribution(oracle_mod, parent, T):
    p1, p2, first = _chi2_pvalues(oracle_mod, parent, T)
    assert first.sum() == 1_000_000
    assert p1 > 1e-3, p1
    assert p2 > 1e-3, p2


@pytest.mark.parametrize("mutant", [2, 5])
def test_planted_sampler_mistakes_fail_chi_square(oracle_mod, mutant):
    p1, p2, _ = _chi2_pvalues(oracle_mod, SIBLINGS, 1.0, trials=400_000, mutant=mutant)
    assert min(p1, p2) < 1e-6, (p1, p2)


def test_walk_must_match_how_siblings_were_drafted(oracle_mod):
    # drafted without replacement: keeping q after a rejection is a mistake
    p1, p2, _ = _chi2_pvalues(oracle_mod, SIBLINGS, 1.0, trials=400_000, replacement=True)
    assert min(p1, p2) < 1e-6, (p1, p2)
    # drafted independently from q: zeroing the rejected token in q is the mistake
    p1, p2, _ = _chi2_pvalues(oracle_mod, SIBLINGS, 1.0, trials=400_000, iid=True)
    assert min(p1, p2) < 1e-6, (p1, p2)


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_with_replacement_walk_is_lossless_on_independent_drafts(oracle_mod, T):
    p1, p2, first = _chi2_pvalues(oracle_mod, SIBLINGS, T, iid=True, replacement=True)
    assert first.sum() == 1_000_000
    assert p1 > 1e-3, p1
    assert p2 > 1e-3, p2


# ----------------------------------------------------------------------------- special cases

def test_p_equals_q_accepts_every_draft(oracle_mod):
    rng = np.random.default_rng(1)
    B, V, T = 64, 500, 0.8
    for parent in (np.arange(-1, 7), W.binary_tree(15), W.topk_tree((4, 3, 2, 2, 1, 1), 60)):
        N = len(parent)
        logits = rng.normal(0, 2, (B, N, V)).astype(np.float32)
        probs = _softmax64(logits, T).astype(np.float32)
        tok = rng.integers(0, V, (B, N))
        ua = (rng.random((B, N)) * 0.999).astype(np.float32)  # keep u away from the ratio 1 +- 1e-7
        ub = rng.random(B).astype(np.float32)
        r = oracle_mod.tree_reject_sample(_inp(logits, probs, tok, np.tile(parent, (B, 1)), ua, ub, T))
        # the first child of every visited node is accepted: follow first children
        path = [0]
        while True:
            kids = [c for c in range(N) if parent[c] == path[-1]]
            if not kids:
                break
            path.append(kids[0])
        assert (r["accept_len"] == len(path) - 1).all()
        assert (r["accepted_nodes"][:, :len(path)] == path).all()
        # bonus: inverse CDF of the leaf's target distribution (numpy searchsorted)
        leaf_p = _softmax64(logits[:, path[-1]], T)
        want = np.array([np.searchsorted(np.cumsum(leaf_p[b]), ub[b], side="right") for b in range(B)])
        assert (r["bonus_token"] == want).all()


def _greedy_walk(logits, tok, parent):
    N = len(parent)
    node, path = 0, [0]
    while True:
        best = int(np.argmax(logits[node]))
        nxt = next((c for c in range(node + 1, N) if parent[c] == node and tok[c] == best), None)
        if nxt is None:
            return path, best
        path.append(nxt)
        node = nxt


def test_temperature_zero_is_greedy_matching(oracle_mod):
    rng = np.random.default_rng(2)
    B, V = 200, 12
    parent = W.random_tree(np.random.default_rng(5), 20, 6)
    N = len(parent)
    logits = rng.integers(-3, 4, (B, N, V)).astype(np.float32)  # many ties: lowest index wins
    tok = rng.integers(0, V, (B, N))
    r = oracle_mod.tree_reject_sample(_inp(logits, None, tok, np.tile(parent, (B, 1)),
                                           np.zeros((B, N)), np.zeros(B), 0.0))
    accepted_something = 0
    for b in range(B):
        path, bonus = _greedy_walk(logits[b], tok[b], parent)
        assert list(r["accepted_nodes"][b, :len(path)]) == path
        assert r["accept_len"][b] == len(path) - 1
        assert r["bonus_token"][b] == bonus
        accepted_something += len(path) > 1
    assert accepted_something > 20


def test_no_match_and_prefix_match_examples(oracle_mod):
    # drafts "and it's so hot" (ids 10 11 12 13) vs target "and it's very warm" (10 11 20 21)
    V = 32
    parent = np.arange(-1, 4)
    logits = np.zeros((1, 5, V), np.float32)
    for node, best in enumerate([10, 11, 20, 21, 22]):
        logits[0, node, best] = 5.0
    tok = np.array([[1, 10, 11, 12, 13]])
    r = oracle_mod.tree_reject_sample(_inp(logits, None, tok, parent[None], np.zeros((1, 5)), [0.0], 0.0))
    assert r["accept_len"][0] == 2
    assert list(r["out_tokens"][0]) == [10, 11, 20, -1, -1]
    # no match: exactly one token, from the target
    tok2 = np.array([[1, 9, 11, 12, 13]])
    r = oracle_mod.tree_reject_sample(_inp(logits, None, tok2, parent[None], np.zeros((1, 5)), [0.0], 0.0))
    assert r["accept_len"][0] == 0 and list(r["out_tokens"][0]) == [10, -1, -1, -1, -1]
    # full match: every draft plus one more
    tok3 = np.array([[1, 10, 11, 20, 21]])
    r = oracle_mod.tree_reject_sample(_inp(logits, None, tok3, parent[None], np.zeros((1, 5)), [0.0], 0.0))
    assert r["accept_len"][0] == 4 and list(r["out_tokens"][0]) == [10, 11, 20, 21, 22]


def test_error_bits(oracle_mod):
    rng = np.random.default_rng(4)
    B, N, V = 5, 7, 50
    parent = np.tile(W.binary_tree(N), (B, 1))
    logits = rng.normal(0, 1, (B, N, V)).astype(np.float32)
    probs = _softmax64(logits + 0.3, 1.0).astype(np.float32)
    tok = rng.integers(0, V, (B, N))
    B = 7
    parent = np.tile(W.binary_tree(N), (B, 1))
    logits = rng.normal(0, 1, (B, N, V)).astype(np.float32)
    probs = _softmax64(logits + 0.3, 1.0).astype(np.float32)
    tok = rng.integers(0, V, (B, N))
    ua = rng.random((B, N))
    parent[0, 4] = 4        # bad tree
    tok[1, 1] = V           # token out of range (child 1 of the root is always tried)
    logits[2, 0, 17] = np.nan  # the root row is always visited
    probs[3, 0, tok[3, 1]] = np.inf  # the drafted token's q is read when child 1 is tried
    # a non-finite draft row matters only once a residual is formed: sequence 4 rejects
    # child 1 at the root (p(x) ~ 0), sequence 5 accepts it (p(x) ~ 1)
    logits[4, 0, tok[4, 1]] = -30.0
    probs[4, 0, (tok[4, 1] + 1) % V] = np.nan
    logits[5, 0, tok[5, 1]] = 30.0
    ua[5, 1] = 0.5
    probs[5, 0, (tok[5, 1] + 1) % V] = np.nan
    r = oracle_mod.tree_reject_sample(_inp(logits, probs, tok, parent, ua, rng.random(B), 1.0))
    assert list(r["err"]) == [1, 8, 16, 16, 16, 0, 0]
    assert list(r["accept_len"][:5]) == [-1] * 5 and (r["accept_len"][5:] >= 0).all()
    assert (r["out_tokens"][:5] == -1).all() and (r["bonus_token"][:5] == -1).all()


# ----------------------------------------------------------------------------- top-k / top-p

def _filtered(p, top_k, top_p):
    """The filtered target distribution, built directly: stable descending order."""
    order = np.lexsort((np.arange(len(p)), -p))
    keep = len(p) if top_k <= 0 else min(top_k, len(p))
    if top_p < 1.0:
        cum = np.cumsum(p[order[:keep]])
        keep = int(np.searchsorted(cum, top_p, side="left")) + 1
        keep = min(keep, len(cum))
    out = np.zeros_like(p)
    out[order[:keep]] = p[order[:keep]] / p[order[:keep]].sum()
    return out


def test_no_filter_is_the_plain_walk(oracle_mod):
    w = W.CONFIGS[3].replace(B=32, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=30, depth=6, V=500, T=1.0, seed=41)
    inp = W.generate(w)
    a = oracle_mod.tree_reject_sample(inp)
    b = oracle_mod.tree_reject_sample(inp, top_k=0, top_p=1.0)
    for key in ("accepted_nodes", "accept_len", "bonus_token", "out_tokens", "err"):
        assert np.array_equal(a[key], b[key])


def test_top1_reduces_to_greedy(oracle_mod):
    # only the argmax keeps mass: a child is accepted iff it is the argmax (its q > 0
    # makes the ratio >= 1 > u), and the bonus is the argmax -- the T = 0 walk
    w = W.CONFIGS[3].replace(B=48, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=25, depth=5, V=300, T=1.0, seed=43)
    inp = W.generate(w)
    a = oracle_mod.tree_reject_sample(inp, top_k=1)
    g = oracle_mod.tree_reject_sample(inp, temperature=0.0)
    for key in ("accepted_nodes", "accept_len", "bonus_token", "out_tokens"):
        assert np.array_equal(a[key], g[key]), key


@pytest.mark.parametrize("top_k,top_p", [(0, 0.8), (5, 1.0), (6, 0.6)])
def test_filtered_output_follows_filtered_target(oracle_mod, top_k, top_p):
    V, T, x0 = 16, 1.0, 3
    rng = np.random.default_rng(17)
    tgt_table = rng.normal(0.0, 1.0, (V, V)).astype(np.float32)
    drf_logits = tgt_table + rng.normal(0.0, 0.8, (V, V)).astype(np.float32)
    # the drafter samples from its own filtered distribution
    drf_table = np.stack([_filtered(r, top_k, top_p) for r in _softmax64(drf_logits, T)]).astype(np.float32)
    counts = np.zeros(V, np.int64)
    for _ in range(3):
        inp = _markov_trials(rng, 200_000, np.array(SIBLINGS), V, T, tgt_table, drf_table, x0)
        r = oracle_mod.tree_reject_sample(inp, top_k=top_k, top_p=top_p)
        assert not r["err"].any()
        counts += np.bincount(r["out_tokens"][:, 0], minlength=V)
    want = _filtered(_softmax64(tgt_table[x0], T), top_k, top_p)
    assert np.all(counts[want == 0] == 0)
    m = want > 0
    assert stats.chisquare(counts[m], want[m] * counts.sum()).pvalue > 1e-3


# ----------------------------------------------------------------------------- top of the unit interval

@pytest.mark.parametrize("logits,u,want", [
    ([0.0, 0.0, -1000.0, -1000.0], 1.0, 1),                  # p = [1/2, 1/2, 0, 0] exactly: u = 1 passes every boundary
    ([0.0, 0.0, 0.0, -1000.0], 1.0, 2),                      # p = [1/3, 1/3, 1/3, 0]: the last token with mass
    ([0.0, 0.0, -1000.0, -1000.0], float("nan"), 1),         # no boundary lies above NaN either
    ([0.0, 0.0, -1000.0, -1000.0], np.nextafter(np.float32(1), np.float32(0)), 1),  # u < 1: the ordinary draw
    ([0.0, 0.0, -1000.0, -1000.0], 0.5, 1),                  # u on the boundary sum_{v<=0} p = 1/2: strict '<'
    ([0.0, 0.0, -1000.0, -1000.0], 0.49999997, 0),
])
def test_bonus_draw_at_the_top_of_the_unit_interval(oracle_mod, logits, u, want):
    """Inverse CDF (statistical-learning-notes ch.07, "Draft Token Validation": a fully
    accepted run draws one more token from the next-token distribution): the smallest
    t with u < sum_{v<=t} p(v).  A u at or past the top of [0, 1) -- which a caller may
    pass, and fp rounding of the sums could in principle reach -- passes every
    boundary; the draw is then the inverse CDF's limit, the last token with p > 0
    (never a token of zero probability).  exp(-1000) is 0 in fp64, so the p rows here
    are exact."""
    inp = _inp(np.array([[logits]]), np.full((1, 1, 4), 0.25), [[0]], [[-1]], [[0.0]], [u], 1.0)
    r = oracle_mod.tree_reject_sample(inp)
    assert r["err"][0] == 0 and r["accept_len"][0] == 0
    assert r["bonus_token"][0] == want
    assert list(r["out_tokens"][0]) == [want]


# ----------------------------------------------------------------------------- bf16 target logits

@pytest.mark.parametrize("T", [0.0, 0.6, 1.0])
def test_bf16_logits_walk_is_the_walk_on_their_exact_decode(oracle_mod, T):
    """bf16 target logits (vLLM PR #2188, "Usage": the target model's output dtype) carry
    the top 16 bits of a float32; the walk on them must be the walk on those floats,
    decoded here independently of the oracle (bits << 16, reinterpreted).  A decode that
    converts the 16-bit pattern as an integer (planted mistake 7) fails."""
    w = W.CONFIGS[3].replace(B=40, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=24, depth=6, V=700, T=T, seed=77)
    inp = W.generate(w, temperature=T)
    bits = W.f32_to_bf16_bits(inp["target_logits"])
    dec = (bits.astype(np.uint32) << 16).view(np.float32)
    a = oracle_mod.tree_reject_sample(dict(inp, target_logits=bits))
    b = oracle_mod.tree_reject_sample(dict(inp, target_logits=dec))
    for key in ("accepted_nodes", "accept_len", "bonus_token", "out_tokens", "err"):
        assert np.array_equal(a[key], b[key]), key
    m = oracle_mod.tree_reject_sample(dict(inp, target_logits=bits), mutant=7)
    assert not all(np.array_equal(m[k], b[k]) for k in ("accepted_nodes", "bonus_token"))
