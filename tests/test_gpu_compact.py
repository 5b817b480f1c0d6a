"""GPU parity of tsv_kv_compact_accepted against the oracle's array copy:
caches bit-identical, new lengths and error bits identical."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import run_compact

pytestmark = pytest.mark.gpu


def _paths(parent, rng):
    B, N = parent.shape
    nodes = np.full((B, N), -1, np.int32)
    lens = np.zeros(B, np.int32)
    for b in range(B):
        path = [0]
        while True:
            kids = np.nonzero(parent[b] == path[-1])[0]
            if len(kids) == 0 or rng.random() < 0.15:
                break
            path.append(int(rng.choice(kids)))
        nodes[b, :len(path)] = path
        lens[b] = len(path) - 1
    return nodes, lens


def _check(inp, nodes, lens):
    gk, gv, gl, ge = run_compact(inp, nodes, lens)
    ok_, ov, ol, oe = oracle.kv_compact_accepted(inp, nodes, lens)
    assert np.array_equal(ge, oe) and np.array_equal(gl, ol)
    assert np.array_equal(gk.view(np.uint8), ok_.view(np.uint8))
    assert np.array_equal(gv.view(np.uint8), ov.view(np.uint8))


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64), ("bf16", 64)])
def test_random_paths(dtype, D):
    w = W.CONFIGS[3].replace(B=24, Hq=8, Hkv=4, D=D, dtype=dtype, prefix=(0, 500), N=100, depth=10, V=128, seed=4)
    inp = W.generate(w)
    nodes, lens = _paths(inp["parent"], np.random.default_rng(1))
    lens[0] = -1
    nodes[0] = -1
    _check(inp, nodes, lens)


def test_overlapping_and_chain_paths_and_errors():
    inp = W.generate(W.CONFIGS[1].replace(B=5, Hq=8, Hkv=2, prefix=(33, 33), N=9, V=32, seed=2))
    nodes = np.full((5, 9), -1, np.int32)
    nodes[0, :3] = [0, 2, 5]          # sources overlap destinations (chain parents ignored here)
    nodes[1, :9] = np.arange(9)       # full accept: identity
    nodes[2, :3] = [0, 3, 2]          # not increasing -> error
    nodes[3, :2] = [0, 8]
    nodes[4, :4] = [0, 1, 4, 8]
    lens = np.array([2, 8, 2, 1, 3], np.int32)
    inp["block_table"] = inp["block_table"].copy()
    inp["block_table"][3, 1] = -3     # bad block id
    _check(inp, nodes, lens)


def test_full_size_sequoia():
    inp = W.generate(W.CONFIGS[3])
    nodes, lens = _paths(inp["parent"], np.random.default_rng(3))
    _check(inp, nodes, lens)
