"""Seeded synthetic inputs for the tree-verification step.

This module only *draws* inputs: trees, prefix lengths, paged-cache layouts,
query/key/value values, draft logits and their softmax (the draft model's
output, which the verification step consumes as given), target logits, draft
tokens and uniforms.  It holds none of the verification step's own arithmetic
(no attention, no rejection test, no residual, no compaction), so both the CPU
oracle and the CUDA library can be fed from it without sharing any of the
method's code.

Workload shapes follow the five synthetic configurations of the verification
study (tiny binary tree, chain, static top-k tree, Sequoia-scale random tree,
large ragged serving mix).  The pages measure on trained models and public
datasets (C4, MT-Bench); these seeded draws stand in for them.

Draw order for one workload (fixed so that every caller sees the same arrays):
tree(s) -> prefix lengths -> block-table permutation -> q/k/v -> draft logits
-> target noise (and the p == q subset) -> draft tokens -> uniforms.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Sequence

import numpy as np

BLOCK_SIZE = 16

# bf16 quiet NaN bit pattern, used to poison cache slots that no sequence owns
BF16_NAN = np.uint16(0x7FC0)


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and distribution recipe of one synthetic verification batch."""

    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    dtype: str  # "f32" | "bf16" (dtype of q, k, v and the attention output)
    prefix: tuple  # (lo, hi) inclusive range of cached prefix lengths; lo == hi for fixed
    tree: str  # "binary" | "chain" | "topk" | "random"
    N: int  # tree nodes including the root
    V: int
    T: float
    noise: float  # std of the target-minus-draft logit noise
    depth: int = 0  # depth cap for "random" trees
    branching: tuple = ()  # per-level children for "topk" trees
    pq_frac: float = 0.0  # fraction of sequences whose target logits equal the draft logits
    siblings: str = "without"  # "without": siblings drafted without replacement; "independent": i.i.d. from q
    seed: int = 1000
    block_size: int = BLOCK_SIZE

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five verification workloads (tiny oracle case, chain, static EAGLE-style
# tree, Sequoia-scale tree, large-model serving mix).
CONFIGS = [
    Workload("tiny_binary15_f32", B=1, Hq=8, Hkv=2, D=64, dtype="f32", prefix=(256, 256),
             tree="binary", N=15, V=1000, T=1.0, noise=0.5, seed=1000),
    Workload("chain5_b8_L2048_v128k", B=8, Hq=32, Hkv=8, D=128, dtype="bf16", prefix=(2048, 2048),
             tree="chain", N=6, V=128256, T=1.0, noise=0.5, seed=1001),
    Workload("eagle60_b32_L4096_v32k", B=32, Hq=32, Hkv=8, D=128, dtype="bf16", prefix=(4096, 4096),
             tree="topk", N=60, V=32000, T=1.0, noise=1.0, branching=(4, 3, 2, 2, 1, 1), seed=1002),
    Workload("sequoia128_b16_L8192_v32k", B=16, Hq=32, Hkv=8, D=128, dtype="bf16", prefix=(8192, 8192),
             tree="random", N=128, depth=10, V=32000, T=0.6, noise=0.5, seed=1003),
    Workload("serving64_b64_L512-32768_v128k", B=64, Hq=64, Hkv=8, D=128, dtype="bf16",
             prefix=(512, 32768), tree="random", N=64, depth=8, V=128256, T=1.0, noise=0.5,
             pq_frac=0.1, seed=1004),
]


# ----------------------------------------------------------------------------- trees

def binary_tree(N: int) -> np.ndarray:
    """Complete binary tree: parent[i] = (i-1)//2, root parent -1."""
    p = np.array([-1] + [(i - 1) // 2 for i in range(1, N)], dtype=np.int32)
    return p


def chain_tree(N: int) -> np.ndarray:
    """Chain (sequence-based speculation): node i's parent is i-1."""
    return np.arange(-1, N - 1, dtype=np.int32)


def _relabel_bfs(par_of: Sequence[int], order_children: Sequence[Sequence[int]]) -> np.ndarray:
    """Relabel a tree given as creation-order parent links into BFS order so that
    parent < child and each node's children are consecutive, in creation order."""
    new_id = {0: 0}
    queue = [0]
    out_par = [-1]
    head = 0
    while head < len(queue):
        u = queue[head]
        head += 1
        for c in order_children[u]:
            new_id[c] = len(queue)
            queue.append(c)
            out_par.append(new_id[u])
    assert len(out_par) == len(par_of)
    return np.array(out_par, dtype=np.int32)


def topk_tree(branching: Sequence[int], keep: int) -> np.ndarray:
    """Static top-k tree: expand the full tree (branching[d] children at depth d,
    sibling ranks 0..k-1), keep the `keep` nodes with the smallest key
    (sum of sibling ranks on the path, depth, BFS index).  The key never
    decreases from a parent to its child, so the kept set is ancestor-closed."""
    paths = [()]
    frontier = [()]
    for b in branching:
        nxt = [p + (r,) for p in frontier for r in range(b)]
        paths += nxt
        frontier = nxt
    order = sorted(range(len(paths)), key=lambda i: (sum(paths[i]), len(paths[i]), i))
    kept = sorted(order[:keep])  # BFS index order
    idx = {paths[i]: j for j, i in enumerate(kept)}
    par = [-1] * keep
    children = [[] for _ in range(keep)]
    for j, i in enumerate(kept):
        p = paths[i]
        if p:
            pj = idx[p[:-1]]
            par[j] = pj
            children[pj].append(j)
    return _relabel_bfs(par, children)


def random_tree(rng: np.random.Generator, N: int, max_depth: int) -> np.ndarray:
    """Sequoia-scale random tree: a first-child spine down to `max_depth`, then
    rounds over the nodes in creation order (depth < max_depth), each node
    receiving Poisson(3/(depth+1)) more children, until exactly N nodes."""
    par = [-1]
    depth = [0]
    children = [[]]
    while len(par) < N and depth[-1] < max_depth:  # spine
        u = len(par) - 1
        par.append(u)
        depth.append(depth[u] + 1)
        children.append([])
        children[u].append(len(par) - 1)
    while len(par) < N:
        for u in range(len(par)):
            if len(par) >= N:
                break
            if depth[u] >= max_depth:
                continue
            k = int(rng.poisson(3.0 / (depth[u] + 1)))
            for _ in range(k):
                if len(par) >= N:
                    break
                par.append(u)
                depth.append(depth[u] + 1)
                children.append([])
                children[u].append(len(par) - 1)
    return _relabel_bfs(par, children)


def tree_depth(parent: np.ndarray) -> int:
    d = np.zeros(len(parent), dtype=np.int64)
    for i in range(1, len(parent)):
        d[i] = d[parent[i]] + 1
    return int(d.max())


# ----------------------------------------------------------------------------- helpers

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest even), returned as uint16 bits.
    Input values here are finite normal draws."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + r) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _fill_normals(out: np.ndarray, seed: int, scale: float = 1.0, to_bf16: bool = False) -> None:
    """Fills `out` (any shape, C order) with N(0, scale^2) draws.  The array is cut
    into fixed slabs along axis 0; slab s draws from its own PCG64 stream seeded by
    (seed, s), so the values do not depend on how many threads fill them."""
    n0 = out.shape[0]
    per_row = int(np.prod(out.shape[1:], dtype=np.int64)) if out.ndim > 1 else 1
    rows = max(1, (1 << 22) // max(1, per_row))
    slabs = [(s, min(n0, s + rows)) for s in range(0, n0, rows)]

    def work(i):
        lo, hi = slabs[i]
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, i])))
        x = g.standard_normal((hi - lo,) + out.shape[1:], dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        out[lo:hi] = f32_to_bf16_bits(x) if to_bf16 else x

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        list(ex.map(work, range(len(slabs))))


def _softmax_rows_f32(x: np.ndarray, T: float, chunk: int = 64) -> np.ndarray:
    """Draft-model distribution q = softmax(draft_logits / T), computed in float64 and
    stored as float32 (the draft model's output, an input to verification)."""
    flat = x.reshape(-1, x.shape[-1])
    out = np.empty_like(flat, dtype=np.float32)

    def work(s):
        z = flat[s:s + chunk].astype(np.float64) / T
        z -= z.max(axis=1, keepdims=True)
        np.exp(z, out=z)
        z /= z.sum(axis=1, keepdims=True)
        out[s:s + chunk] = z

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        list(ex.map(work, range(0, flat.shape[0], chunk)))
    return out.reshape(x.shape)


# ----------------------------------------------------------------------------- generator

def generate(w: Workload, *, seed: Optional[int] = None, temperature: Optional[float] = None,
             pad_nan: bool = True) -> dict:
    """Draw one batch for workload `w`.  Returns numpy arrays:

    parent [B,N] i32, seq_lens [B] i32, block_table [B,max_blocks] i32,
    q [B,N,Hq,D], k_cache/v_cache [num_blocks,bs,Hkv,D] (float32, or uint16 bf16 bits),
    target_logits/draft_probs [B,N,V] f32, draft_tokens [B,N] i32,
    u_accept [B,N] f32, u_bonus [B] f32, plus scalar metadata.

    Cache slots that a sequence's blocks hold beyond its last tree slot are filled
    with NaN when `pad_nan` (they must never be read)."""
    T = float(w.T if temperature is None else temperature)
    rng = np.random.default_rng(w.seed if seed is None else seed)
    B, N, V, bs = w.B, w.N, w.V, w.block_size

    # 1. trees
    if w.tree == "binary":
        parent = np.tile(binary_tree(N), (B, 1))
    elif w.tree == "chain":
        parent = np.tile(chain_tree(N), (B, 1))
    elif w.tree == "topk":
        parent = np.tile(topk_tree(w.branching, N), (B, 1))
    elif w.tree == "random":
        parent = np.stack([random_tree(rng, N, w.depth) for _ in range(B)])
    else:
        raise ValueError(w.tree)
    parent = np.ascontiguousarray(parent, dtype=np.int32)

    # 2. prefix lengths
    lo, hi = w.prefix
    if lo == hi:
        seq_lens = np.full(B, lo, dtype=np.int32)
    else:
        seq_lens = rng.integers(lo, hi, endpoint=True, size=B).astype(np.int32)

    # 3. paged layout: every sequence owns ceil((L_b + N)/bs) blocks, assigned from a
    #    random permutation of all physical blocks
    nblk = (seq_lens.astype(np.int64) + N + bs - 1) // bs
    num_blocks = int(nblk.sum())
    max_blocks = int(nblk.max())
    perm = rng.permutation(num_blocks).astype(np.int32)
    block_table = np.full((B, max_blocks), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        block_table[b, :nblk[b]] = perm[off:off + nblk[b]]
        off += int(nblk[b])

    # 4. q / k / v ~ N(0, 1) (the caches are filled slab-parallel from one drawn seed)
    def normals(shape):
        return rng.standard_normal(shape, dtype=np.float32)

    q = normals((B, N, w.Hq, w.D))
    kv_seed = int(rng.integers(0, 2**63 - 1))
    cache_shape = (num_blocks, bs, w.Hkv, w.D)
    if w.dtype == "bf16":
        q = f32_to_bf16_bits(q)
        k_cache = np.empty(cache_shape, dtype=np.uint16)
        v_cache = np.empty(cache_shape, dtype=np.uint16)
        _fill_normals(k_cache, kv_seed * 2 % (2**63), to_bf16=True)
        _fill_normals(v_cache, (kv_seed * 2 + 1) % (2**63), to_bf16=True)
        nan_val = BF16_NAN
    elif w.dtype == "f32":
        k_cache = np.empty(cache_shape, dtype=np.float32)
        v_cache = np.empty(cache_shape, dtype=np.float32)
        _fill_normals(k_cache, kv_seed * 2 % (2**63))
        _fill_normals(v_cache, (kv_seed * 2 + 1) % (2**63))
        nan_val = np.float32(np.nan)
    else:
        raise ValueError(w.dtype)
    if pad_nan:
        for b in range(B):
            for t in range(int(seq_lens[b]) + N, int(nblk[b]) * bs):
                blk = block_table[b, t // bs]
                k_cache[blk, t % bs] = nan_val
                v_cache[blk, t % bs] = nan_val

    # 5. draft logits 2*N(0,1) and the draft distribution q = softmax(draft / T)
    draft_logits = np.empty((B, N, V), dtype=np.float32)
    _fill_normals(draft_logits, int(rng.integers(0, 2**63 - 1)), scale=2.0)
    draft_probs = _softmax_rows_f32(draft_logits, T if T > 0 else 1.0)

    # 6. target logits = draft + N(0, noise^2); a seeded subset gets target == draft
    target_logits = np.empty((B, N, V), dtype=np.float32)
    _fill_normals(target_logits, int(rng.integers(0, 2**63 - 1)), scale=w.noise)
    target_logits += draft_logits
    pq_seqs = np.zeros(0, dtype=np.int64)
    if w.pq_frac > 0:
        npq = int(round(w.pq_frac * B))
        pq_seqs = np.sort(rng.choice(B, size=npq, replace=False))
        target_logits[pq_seqs] = draft_logits[pq_seqs]

    # 7. draft tokens: the children of node i are drafted from node i's draft
    #    distribution without replacement (Gumbel-top-k), in child-index order, or
    #    independently (siblings="independent"); at T == 0 they are the top-k of the
    #    draft logits.  The root's own token is the
    #    last accepted token and is drawn uniformly.
    draft_tokens = np.zeros((B, N), dtype=np.int32)
    draft_tokens[:, 0] = rng.integers(0, V, size=B)
    for b in range(B):
        kids = [[] for _ in range(N)]
        for c in range(1, N):
            kids[parent[b, c]].append(c)
        for i in range(N):
            if not kids[i]:
                continue
            k = len(kids[i])
            if k > V:
                raise ValueError(f"node {i} has {k} children but the vocabulary has only {V} tokens")
            if T > 0 and w.siblings == "independent":
                # each child drawn independently from q (inverse CDF of one uniform each)
                cdf = np.cumsum(draft_probs[b, i].astype(np.float64))
                u = rng.random(k) * cdf[-1]
                draft_tokens[b, kids[i]] = np.minimum(np.searchsorted(cdf, u, side="right"), V - 1)
                continue
            if T > 0:
                key = np.log(draft_probs[b, i].astype(np.float64)) + rng.gumbel(size=V)
            else:
                key = draft_logits[b, i].astype(np.float64)
            cand = np.argpartition(-key, k - 1)[:k] if k < V else np.arange(V)
            top = cand[np.lexsort((cand, -key[cand]))]  # descending key, ties to the lower id
            draft_tokens[b, kids[i]] = top

    # 8. uniforms U[0, 1)
    u_accept = rng.random((B, N), dtype=np.float32)
    u_bonus = rng.random(B, dtype=np.float32)

    return dict(
        workload=w, T=T, scale=1.0 / math.sqrt(w.D), dtype=w.dtype,
        B=B, N=N, Hq=w.Hq, Hkv=w.Hkv, D=w.D, V=V, block_size=bs,
        num_blocks=num_blocks, max_blocks=max_blocks,
        parent=parent, seq_lens=seq_lens, block_table=block_table,
        q=q, k_cache=k_cache, v_cache=v_cache,
        target_logits=target_logits, draft_probs=draft_probs, draft_tokens=draft_tokens,
        u_accept=u_accept, u_bonus=u_bonus, pq_seqs=pq_seqs,
    )


def small_variant(w: Workload, **kw) -> Workload:
    """The same recipe at sizes the CPU oracle finishes in seconds."""
    return w.replace(**kw)
