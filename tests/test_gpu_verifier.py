"""GPU parity of tsv_tree_reject_sample against the oracle's literal walk.

Accepted paths, accept lengths, bonus tokens and output tokens must be identical,
except sequences whose first differing decision is a near tie (|u - p/q| < 1e-6,
or u_bonus within 1e-6 of a CDF boundary); those are counted and printed.  The
GPU sampler is also held to the same chi-square losslessness test as the oracle."""
import json
import os

import numpy as np
import pytest
import torch
from scipy import stats

import oracle
import workloads as W
from gpu_util import compare_decisions, run_verify

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(__file__)


def _check(inp, T=None, max_exempt_frac=0.05):
    T = inp["T"] if T is None else T
    g = run_verify(inp, temperature=T)
    o = oracle.tree_reject_sample(inp, temperature=T)
    exempt, fails = compare_decisions(inp, g, o, T)
    assert not fails, fails[:5]
    assert exempt <= max_exempt_frac * len(o["accept_len"]) + 1
    print(f"exempt near-tie sequences: {exempt} of {len(o['accept_len'])}")
    return g, o


def test_tiny_config():
    _check(W.generate(W.CONFIGS[0]))


@pytest.mark.parametrize("T", [0.0, 0.6, 1.0])
@pytest.mark.parametrize("V", [1000, 3001, 32000])
def test_random_trees(T, V):
    w = W.CONFIGS[3].replace(B=64, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=40, depth=7, V=V, T=T, seed=V + int(10 * T))
    _check(W.generate(w, temperature=T))


def test_hand_worked_cases_on_gpu():
    g = json.load(open(os.path.join(HERE, "golden", "verifier_hand.json")))
    for c in g["cases"]:
        probs = np.array(g["draft_probs"], np.float64)
        for k, row in c.get("draft_probs_override", {}).items():
            probs[int(k)] = row
        inp = dict(B=1, N=4, V=3, T=c["T"], target_logits=np.log(np.array(g["probs_target"]))[None].astype(np.float32),
                   draft_probs=probs[None].astype(np.float32), draft_tokens=np.array([c["tokens"]], np.int32),
                   parent=np.array([g["parent"]], np.int32), u_accept=np.array([c["u_accept"]], np.float32),
                   u_bonus=np.array([c["u_bonus"]], np.float32))
        r = run_verify(inp)
        assert list(r["accepted_nodes"][0]) == c["accepted_nodes"], c["name"]
        assert r["bonus_token"][0] == c["bonus_token"], c["name"]
        assert list(r["out_tokens"][0]) == c["out_tokens"], c["name"]


def test_p_equals_q_full_accept_and_errors():
    w = W.CONFIGS[2].replace(B=16, Hq=4, Hkv=1, D=64, prefix=(0, 0), V=5000, seed=9)
    inp = W.generate(w)
    inp["target_logits"] = (np.log(inp["draft_probs"].astype(np.float64))).astype(np.float32)
    inp["u_accept"] = (inp["u_accept"] * 0.999).astype(np.float32)
    g, o = _check(inp)
    assert (o["accept_len"] == 6).all()
    # errors: token out of range, non-finite row, bad tree
    inp["draft_tokens"] = inp["draft_tokens"].copy()
    inp["draft_tokens"][1, 1] = 5000
    inp["target_logits"] = inp["target_logits"].copy()
    inp["target_logits"][2, 0, 7] = np.inf
    inp["parent"] = inp["parent"].copy()
    inp["parent"][3, 0] = 0
    _check(inp)


@pytest.mark.parametrize("T", [0.0, 0.6, 1.0])
@pytest.mark.parametrize("V", [3001, 32000])
@pytest.mark.parametrize("N,tree", [(1, "chain"), (2, "chain"), (6, "chain"), (8, "random")])
def test_small_trees(T, V, N, tree):
    """Small trees down to the root alone and one-child chains, unaligned and aligned
    vocabularies: decisions identical to the oracle's walk."""
    w = W.CONFIGS[3].replace(B=64, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=N, depth=4, tree=tree, V=V, T=T,
                             seed=V + 10 * N + int(10 * T))
    _check(W.generate(w, temperature=T))


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_small_tree_errors_only_on_visited_rows(T):
    """A non-finite logit is an error only in a row the walk visits."""
    w = W.CONFIGS[1].replace(B=8, Hq=4, Hkv=1, D=64, prefix=(0, 0), V=5000, seed=21)
    inp = W.generate(w, temperature=T)
    inp["target_logits"] = (np.log(inp["draft_probs"].astype(np.float64))).astype(np.float32)
    inp["u_accept"] = (inp["u_accept"] * 0.999).astype(np.float32)
    inp["draft_tokens"] = inp["draft_tokens"].copy()
    inp["draft_tokens"][1, 3] = 5000                   # token out of range
    inp["target_logits"][2, 0, 7] = np.inf             # root row: always visited
    inp["target_logits"][3, 4, 11] = np.nan            # node 4: visited at T = 1 (p == q accepts)
    inp["target_logits"][5, 0, inp["draft_tokens"][5, 1]] = -60.0  # child 1 rejected at the root ...
    inp["target_logits"][5, 3, 11] = np.inf            # ... so node 3's row is never visited
    g, o = _check(inp, T)
    assert o["err"][5] == 0 and g["err"][5] == 0
    assert o["err"][2] != 0


def _markov(n, parent, V, T, rng, tgt, drf, x0):
    N = len(parent)
    kids = [[] for _ in range(N)]
    for c in range(1, N):
        kids[parent[c]].append(c)
    tok = np.empty((n, N), np.int64)
    tok[:, 0] = x0
    for i in range(N):
        if kids[i]:
            q = drf[tok[:, i]].astype(np.float64)
            with np.errstate(divide="ignore"):
                key = np.log(q) + rng.gumbel(size=q.shape)
            tok[:, kids[i]] = np.argsort(-key, axis=1, kind="stable")[:, :len(kids[i])]
    return dict(B=n, N=N, V=V, T=T, target_logits=np.ascontiguousarray(tgt[tok], np.float32),
                draft_probs=np.ascontiguousarray(drf[tok], np.float32), draft_tokens=tok.astype(np.int32),
                parent=np.tile(np.array(parent, np.int32), (n, 1)),
                u_accept=rng.random((n, N), dtype=np.float32), u_bonus=rng.random(n, dtype=np.float32))


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_chi_square_losslessness_on_gpu(T):
    V, parent, x0 = 16, [-1, 0, 0, 0, 1, 1, 2, 2, 3, 3], 3
    rng = np.random.default_rng(123)
    tgt = rng.normal(0, 1, (V, V)).astype(np.float32)
    z = (tgt + rng.normal(0, 0.8, (V, V))) / T
    drf = np.exp(z - z.max(1, keepdims=True))
    drf = (drf / drf.sum(1, keepdims=True)).astype(np.float32)
    counts = np.zeros(V, np.int64)
    exempt_total = 0
    for _ in range(5):
        inp = _markov(200_000, parent, V, T, rng, tgt, drf, x0)
        g = run_verify(inp)
        o = oracle.tree_reject_sample(inp)
        exempt, fails = compare_decisions(inp, g, o, T)
        assert not fails, fails[:5]
        exempt_total += exempt
        counts += np.bincount(g["out_tokens"][:, 0], minlength=V)
    zt = tgt[x0].astype(np.float64) / T
    p = np.exp(zt - zt.max())
    p /= p.sum()
    assert stats.chisquare(counts, p * counts.sum()).pvalue > 1e-3
    print("exempt near ties:", exempt_total)


@pytest.mark.parametrize("cfg,T", [(1, 0.0), (1, 1.0), (2, None), (3, None), (4, None)])
def test_full_size(cfg, T):
    inp = W.generate(W.CONFIGS[cfg], temperature=T)
    _check(inp, T)


def test_bonus_draw_at_the_top_of_the_unit_interval_on_gpu():
    """u_bonus at or past 1 (and NaN) gives the last token with p > 0, as the oracle
    does; compared exactly (no near-tie exemption applies to this rule)."""
    w = W.CONFIGS[1].replace(B=16, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=4, V=5000, seed=71)
    inp = W.generate(w)
    inp["target_logits"] = inp["target_logits"].copy()
    inp["target_logits"][:, :, 4900:] = -1000.0        # no mass on the last 100 tokens
    inp["target_logits"][1::2, :, 4000:4900] = -1000.0  # odd sequences: none past token 3999 either
    inp["u_bonus"] = inp["u_bonus"].copy()
    inp["u_bonus"][0::3] = 1.0
    inp["u_bonus"][1::3] = np.nan
    for T in (1.0, 0.6):
        g = run_verify(inp, temperature=T)
        o = oracle.tree_reject_sample(inp, temperature=T)
        top = ~(inp["u_bonus"] < 1.0)
        assert top.sum() >= 10
        for key in ("accepted_nodes", "accept_len", "bonus_token", "out_tokens", "err"):
            assert np.array_equal(g[key][top], o[key][top]), key
        assert (o["bonus_token"][top] < np.where(np.arange(16)[top] % 2 == 1, 4000, 4900)).all()
        exempt, fails = compare_decisions(
            {k: (v[~top] if isinstance(v, np.ndarray) and v.shape[:1] == (16,) else v) for k, v in inp.items()},
            {k: v[~top] for k, v in g.items()}, {k: v[~top] for k, v in o.items()}, T)
        assert not fails, fails
