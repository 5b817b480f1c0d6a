"""GPU parity of the walk's variants (tsv_walk_options) against the oracle's modes.

  * with_replacement = 1 (the SpecInfer verification that the Sequoia summary's figure
    of rejection rates compares against, "More on figures"): siblings drafted
    independently from q; q kept after a rejection.  Decisions identical to the
    oracle's with-replacement walk (up to counted near ties), and on a 16-token
    vocabulary the first emitted token follows the target distribution (chi-square,
    10^6 trials on independent drafts).
  * bf16 target logits: decisions identical to the oracle's walk on the same bf16
    logits, from small unaligned vocabularies to the full serving mix.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
import workloads as W
from gpu_util import compare_decisions, run_verify

pytestmark = pytest.mark.gpu


def _check(inp, T, replacement=False, max_exempt_frac=0.05):
    g = run_verify(inp, temperature=T, with_replacement=replacement)
    o = oracle.tree_reject_sample(inp, temperature=T, replacement=replacement)
    exempt, fails = compare_decisions(inp, g, o, T)
    B = len(o["accept_len"])
    msg = f"{exempt} of {B} sequences exempt as near ties; {len(fails)} mismatches: {fails[:5]}"
    assert not fails, msg
    assert exempt <= max_exempt_frac * B + 1, msg
    print(msg)
    return g, o


@pytest.mark.parametrize("T", [0.0, 0.6, 1.0])
@pytest.mark.parametrize("V", [3001, 32000])
def test_with_replacement_matches_the_oracle(T, V):
    w = W.CONFIGS[3].replace(B=64, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=40, depth=6, V=V, T=T, siblings="independent",
                             seed=500 + V + int(10 * T))
    inp = W.generate(w, temperature=T)
    g, o = _check(inp, T, replacement=True)
    if T > 0:  # the drafts repeat tokens among siblings, which only this walk handles as drafted
        dup = sum(len(set(inp["draft_tokens"][b, inp["parent"][b] == i])) < (inp["parent"][b] == i).sum()
                  for b in range(inp["B"]) for i in range(inp["N"]))
        assert dup > 0


def test_with_replacement_differs_from_the_default_walk():
    """The two walks are different functions: on the same independent drafts their
    decisions differ for some sequences (each matches its own oracle mode)."""
    w = W.CONFIGS[3].replace(B=64, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=40, depth=6, V=64, T=1.0,
                             siblings="independent", seed=911)
    inp = W.generate(w)
    a = run_verify(inp, with_replacement=True)
    b = run_verify(inp, with_replacement=False)
    assert not np.array_equal(a["out_tokens"], b["out_tokens"])
    _check(inp, 1.0, replacement=False)


def _iid_trials(n, parent, V, T, rng, tgt, drf, x0):
    N = len(parent)
    kids = [[] for _ in range(N)]
    for c in range(1, N):
        kids[parent[c]].append(c)
    tok = np.empty((n, N), np.int64)
    tok[:, 0] = x0
    for i in range(N):
        if kids[i]:
            cdf = np.cumsum(drf[tok[:, i]].astype(np.float64), axis=1)
            u = rng.random((n, len(kids[i]))) * cdf[:, -1:]
            tok[:, kids[i]] = np.minimum((u[:, :, None] >= cdf[:, None, :]).sum(axis=2), V - 1)
    return dict(B=n, N=N, V=V, T=T, target_logits=np.ascontiguousarray(tgt[tok], np.float32),
                draft_probs=np.ascontiguousarray(drf[tok], np.float32), draft_tokens=tok.astype(np.int32),
                parent=np.tile(np.array(parent, np.int32), (n, 1)),
                u_accept=rng.random((n, N), dtype=np.float32), u_bonus=rng.random(n, dtype=np.float32))


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_with_replacement_is_lossless_on_independent_drafts_on_gpu(T):
    V, parent, x0 = 16, [-1, 0, 0, 0, 1, 1, 2, 2, 3, 3], 3
    rng = np.random.default_rng(321)
    tgt = rng.normal(0, 1, (V, V)).astype(np.float32)
    z = (tgt + rng.normal(0, 0.8, (V, V))) / T
    drf = np.exp(z - z.max(1, keepdims=True))
    drf = (drf / drf.sum(1, keepdims=True)).astype(np.float32)
    counts = np.zeros(V, np.int64)
    exempt_total = 0
    for _ in range(5):
        inp = _iid_trials(200_000, parent, V, T, rng, tgt, drf, x0)
        g = run_verify(inp, with_replacement=True)
        o = oracle.tree_reject_sample(inp, replacement=True)
        exempt, fails = compare_decisions(inp, g, o, T)
        assert not fails, fails[:5]
        exempt_total += exempt
        counts += np.bincount(g["out_tokens"][:, 0], minlength=V)
    zt = tgt[x0].astype(np.float64) / T
    p = np.exp(zt - zt.max())
    p /= p.sum()
    pv = stats.chisquare(counts, p * counts.sum()).pvalue
    assert pv > 1e-3, (pv, exempt_total)
    print("exempt near ties:", exempt_total)


def _bf16(inp):
    return dict(inp, target_logits=W.f32_to_bf16_bits(inp["target_logits"]))


@pytest.mark.parametrize("T", [0.0, 0.6, 1.0])
@pytest.mark.parametrize("V", [1000, 3001, 32000])
def test_bf16_logits_match_the_oracle(T, V):
    w = W.CONFIGS[3].replace(B=64, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=40, depth=7, V=V, T=T, seed=700 + V + int(10 * T))
    _check(_bf16(W.generate(w, temperature=T)), T)


def test_bf16_logits_with_replacement():
    w = W.CONFIGS[3].replace(B=48, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=30, depth=5, V=5000, T=1.0,
                             siblings="independent", seed=811)
    _check(_bf16(W.generate(w)), 1.0, replacement=True)


def test_bf16_logits_full_serving_mix():
    inp = W.generate(W.CONFIGS[4])
    g, o = _check(_bf16(inp), inp["T"])
    assert all(o["accept_len"][b] >= 1 for b in inp["pq_seqs"])
