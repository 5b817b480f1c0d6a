"""GPU parity of the top-k / top-p filtered walk (tsv_walk_options top_k, top_p) with
the oracle's filter_top mode (Sequoia summary, "More on tables": robustness to top-p
sampling).  At every visited node the target p is restricted to its first entries in
order of decreasing p (ties to the lower index) until top_k of them, or a mass of
top_p, is reached, then renormalised.

Pins on the GPU, as on the oracle: decisions identical to the oracle's filtered walk
(up to counted near ties), including boundaries inside a run of equal logits; top-1
reduces to the greedy walk; on a 16-token vocabulary with drafts from the drafter's
own filtered distribution the first emitted token follows the filtered target
(chi-square, 6 x 10^5 trials), and never falls outside its support."""
import numpy as np
import pytest
from scipy import stats

import oracle
import workloads as W
from gpu_util import compare_decisions, run_verify

pytestmark = pytest.mark.gpu


def _check(inp, T, top_k, top_p, max_exempt_frac=0.05):
    g = run_verify(inp, temperature=T, top_k=top_k, top_p=top_p)
    o = oracle.tree_reject_sample(inp, temperature=T, top_k=top_k, top_p=top_p)
    exempt, fails = compare_decisions(inp, g, o, T)
    B = len(o["accept_len"])
    msg = f"top_k={top_k} top_p={top_p}: {exempt} of {B} exempt near ties; {len(fails)} mismatches: {fails[:5]}"
    assert not fails, msg
    assert exempt <= max_exempt_frac * B + 1, msg
    print(msg)
    return g, o


@pytest.mark.parametrize("top_k,top_p", [(5, 1.0), (50, 1.0), (0, 0.8), (0, 0.95), (20, 0.9)])
@pytest.mark.parametrize("T,V", [(1.0, 3001), (0.6, 32000)])
def test_filtered_walk_matches_the_oracle(top_k, top_p, T, V):
    w = W.CONFIGS[3].replace(B=48, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=30, depth=6, V=V, T=T,
                             seed=900 + V + top_k + int(100 * top_p))
    _check(W.generate(w, temperature=T), T, top_k, top_p)


def test_no_filter_options_are_the_plain_walk():
    w = W.CONFIGS[3].replace(B=32, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=30, depth=6, V=5000, T=1.0, seed=17)
    inp = W.generate(w)
    a = run_verify(inp)
    b = run_verify(inp, top_k=0, top_p=1.0)
    c = run_verify(inp, top_k=5000, top_p=1.0)  # top_k >= V keeps everything
    for key in ("accepted_nodes", "accept_len", "bonus_token", "out_tokens", "err"):
        assert np.array_equal(a[key], b[key]) and np.array_equal(a[key], c[key]), key


def test_top1_is_the_greedy_walk():
    w = W.CONFIGS[3].replace(B=48, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=25, depth=5, V=3000, T=1.0, seed=43)
    inp = W.generate(w)
    a = run_verify(inp, top_k=1)
    g = run_verify(inp, temperature=0.0)
    for key in ("accepted_nodes", "accept_len", "bonus_token", "out_tokens"):
        assert np.array_equal(a[key], g[key]), key


@pytest.mark.parametrize("top_k,top_p", [(7, 1.0), (0, 0.5), (12, 0.7)])
def test_boundary_inside_a_run_of_equal_logits(top_k, top_p):
    """Logits rounded to a coarse grid: many entries share the boundary value, so the cut
    falls inside a run of ties and is decided by index."""
    w = W.CONFIGS[3].replace(B=40, Hq=4, Hkv=1, D=64, prefix=(0, 0), N=20, depth=5, V=2000, T=1.0, seed=321 + top_k)
    inp = W.generate(w)
    inp["target_logits"] = (np.round(inp["target_logits"] * 2.0) / 2.0).astype(np.float32)
    _check(inp, 1.0, top_k, top_p)


def _filtered(p, top_k, top_p):
    order = np.lexsort((np.arange(len(p)), -p))
    keep = len(p) if top_k <= 0 else min(top_k, len(p))
    if top_p < 1.0:
        cum = np.cumsum(p[order[:keep]])
        keep = min(int(np.searchsorted(cum, top_p, side="left")) + 1, len(cum))
    out = np.zeros_like(p)
    out[order[:keep]] = p[order[:keep]] / p[order[:keep]].sum()
    return out


@pytest.mark.parametrize("top_k,top_p", [(0, 0.8), (6, 0.9), (3, 1.0)])
def test_filtered_output_follows_the_filtered_target_on_gpu(top_k, top_p):
    V, T, x0 = 16, 1.0, 3
    parent = [-1, 0, 0, 0, 1, 1, 2, 2, 3, 3]
    rng = np.random.default_rng(77)
    tgt = rng.normal(0.0, 1.0, (V, V)).astype(np.float32)
    z = (tgt + rng.normal(0.0, 0.8, (V, V))) / T
    q = np.exp(z - z.max(1, keepdims=True))
    q = q / q.sum(1, keepdims=True)
    drf = np.stack([_filtered(r, top_k, top_p) for r in q]).astype(np.float32)  # the drafter's own filter
    N = len(parent)
    kids = [[c for c in range(1, N) if parent[c] == i] for i in range(N)]
    counts = np.zeros(V, np.int64)
    for _ in range(3):
        n = 200_000
        tok = np.empty((n, N), np.int64)
        tok[:, 0] = x0
        for i in range(N):
            if kids[i]:
                with np.errstate(divide="ignore"):
                    key = np.log(drf[tok[:, i]].astype(np.float64)) + rng.gumbel(size=(n, V))
                tok[:, kids[i]] = np.argsort(-key, axis=1, kind="stable")[:, :len(kids[i])]
        inp = dict(B=n, N=N, V=V, T=T, target_logits=np.ascontiguousarray(tgt[tok], np.float32),
                   draft_probs=np.ascontiguousarray(drf[tok], np.float32), draft_tokens=tok.astype(np.int32),
                   parent=np.tile(np.array(parent, np.int32), (n, 1)),
                   u_accept=rng.random((n, N), dtype=np.float32), u_bonus=rng.random(n, dtype=np.float32))
        g = run_verify(inp, top_k=top_k, top_p=top_p)
        assert not g["err"].any()
        counts += np.bincount(g["out_tokens"][:, 0], minlength=V)
    zt = tgt[x0].astype(np.float64) / T
    p = np.exp(zt - zt.max())
    want = _filtered(p / p.sum(), top_k, top_p)
    assert np.all(counts[want == 0] == 0)
    m = want > 0
    assert m.sum() >= 2  # a support of one token would make the test trivial
    assert stats.chisquare(counts[m], want[m] * counts.sum()).pvalue > 1e-3


@pytest.mark.parametrize("opts", [dict(top_k=50, top_p=0.9), dict(top_k=0, top_p=0.8), dict(with_replacement=True)])
def test_serving_batch_layout(opts):
    """The serving mix's batch (64 sequences, 64-node trees, V = 128256) does not fit the
    512-thread layout at once, so the walk runs 384-thread CTAs with 16 vector steps a
    thread; the filtered and the with-replacement walks are pinned there too (the
    prefix plays no part in the walk and is left out)."""
    w = W.CONFIGS[4].replace(prefix=(0, 0), seed=4040 + len(opts))
    inp = W.generate(w)
    T = inp["T"]
    g = run_verify(inp, **opts)
    o = oracle.tree_reject_sample(inp, replacement=bool(opts.get("with_replacement", False)),
                                  top_k=opts.get("top_k", 0), top_p=opts.get("top_p", 1.0))
    exempt, fails = compare_decisions(inp, g, o, T)
    B = len(o["accept_len"])
    msg = f"{opts}: {exempt} of {B} exempt near ties; {len(fails)} mismatches: {fails[:5]}"
    assert not fails, msg
    assert exempt <= 0.05 * B + 1, msg
