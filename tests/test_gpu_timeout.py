"""Failure detection on the GPU without a fault: every mbarrier wait of the attention
kernel is bounded, and a wait that gives up reports TSV_DERR_TIMEOUT for its sequence
instead of hanging or trapping; the other roles see the abort, drain their copies
and MMAs, free TMEM and return, and the CUDA context stays usable.

The "hooks" test build (-DTSV_TEST_HOOKS) shortens the limit to 1 ms and, when
tsv_test_set_stall(1) is set, points warpgroup 0's first S wait of every CTA at a
barrier that nothing completes.  The product build has neither."""
import time

import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_03_gb300 as tsv
import workloads as W
from gpu_util import run_attn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hooks_lib():
    tsv.build(variant="hooks")
    lib = tsv.load("hooks")
    tsv.use_variant("hooks")
    yield lib
    lib.tsv_test_set_stall(0)
    tsv.use_variant(None)


def test_a_wait_that_runs_out_is_reported_and_the_context_survives(hooks_lib):
    w = W.CONFIGS[3].replace(B=4, Hq=16, Hkv=4, prefix=(200, 900), N=40, depth=6, V=64, seed=55)
    inp = W.generate(w)
    assert hooks_lib.tsv_test_set_stall(1) == 0
    t0 = time.perf_counter()
    _, err = run_attn(inp)  # returns: the stalled waits give up after 1 ms each
    elapsed = time.perf_counter() - t0
    assert (err & tsv.TSV_DERR_TIMEOUT).any(), err
    assert elapsed < 5.0, elapsed
    # the context still works: the same call without the stall gives the oracle's result
    assert hooks_lib.tsv_test_set_stall(0) == 0
    got, err = run_attn(inp)
    assert not err.any()
    want, _ = oracle.tree_verify_attn(inp)
    assert np.abs(got - want).max() <= 2e-2
    torch.cuda.synchronize()
