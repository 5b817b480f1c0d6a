"""tsv_tree_verify_attn_noalloc: the attention call for callers that cannot
allocate device memory (an engine plugin that only receives its inputs and
outputs, a loop that must not call cudaMalloc).  Its split-K scratch is the
library's own fixed device array, shared by every call and keeping whatever the
last call left there.

Every check call comes right after a call on other data -- the same shapes with
negated queries and shorter prefixes, so a different split of the keys, other
partial values and other per-unit records in the array -- and must give, bit for
bit, what the workspace-taking entry point gives on the same inputs: a read of a
scratch byte that the call itself did not write would show up as a difference.
A shape that needs more scratch than the array holds must be refused.

This file is collected last so that a failure here comes after every other test."""
import numpy as np
import pytest
import torch

import tree_speculative_decoding_03_gb300 as tsv
import workloads as W
from gpu_util import device_inputs

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).cpu().numpy()


def _with_workspace(inp, d):
    B, N, Hq, D = d["q"].shape
    out = torch.empty_like(d["q"])
    code = tsv.TSV_BF16 if inp["dtype"] == "bf16" else tsv.TSV_F32
    ws_bytes = tsv.attn_workspace_size(B, N, Hq, inp["Hkv"], D, inp["block_size"], inp["max_blocks"], code)
    assert ws_bytes > 0  # the shape really uses scratch
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    err = torch.empty(B, dtype=torch.int32, device="cuda")
    tsv.tree_verify_attn(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["parent"], out,
                         inp["scale"], workspace=ws, seq_err=err)
    torch.cuda.synchronize()
    return _bits(out), err.cpu().numpy()


def _no_alloc(inp, d, q=None, seq_lens=None):
    q = d["q"] if q is None else q
    out = torch.full_like(q, float("nan"))
    err = torch.full((inp["B"],), -1, dtype=torch.int32, device="cuda")
    tsv.tree_verify_attn_noalloc(q, d["k_cache"], d["v_cache"], d["block_table"],
                                 d["seq_lens"] if seq_lens is None else seq_lens, d["parent"], out, inp["scale"],
                                 seq_err=err)
    torch.cuda.synchronize()
    return _bits(out), err.cpu().numpy()


@pytest.mark.parametrize("cfg", [0, 1, 3])
def test_no_alloc_matches_workspace_call_twice(cfg):
    tsv.build()
    inp = W.generate(W.CONFIGS[cfg])
    d = device_inputs(inp, verify=False)
    want, want_err = _with_workspace(inp, d)
    assert not want_err.any()
    other_q = -d["q"]
    other_lens = torch.clamp(d["seq_lens"] - 37 - torch.arange(inp["B"], device="cuda", dtype=torch.int32), min=0)
    for _ in range(2):
        dirty, dirty_err = _no_alloc(inp, d, q=other_q, seq_lens=other_lens)  # other data in the scratch
        assert not dirty_err.any() and not np.array_equal(dirty, want)
        got, err = _no_alloc(inp, d)
        assert np.array_equal(err, want_err)
        assert np.array_equal(got, want), "no-alloc output differs from the workspace call's"


def test_no_alloc_refuses_shapes_beyond_its_scratch():
    inp = W.generate(W.CONFIGS[2].replace(B=2, V=64))
    d = device_inputs(inp, verify=False)
    B, N, Hq, D = d["q"].shape
    lib = tsv.load()
    cap = lib.tsv_noalloc_scratch_bytes()
    # fp32 key chunks: a block table wide enough that the planned scratch exceeds the array
    big_blocks = 1 << 20
    need = tsv.attn_workspace_size(B, N, Hq, inp["Hkv"], D, 16, big_blocks, tsv.TSV_F32)
    assert need > cap
    out = torch.empty_like(d["q"])
    err = torch.empty(B, dtype=torch.int32, device="cuda")
    st = lib.tsv_tree_verify_attn_noalloc(d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
                                          d["block_table"].data_ptr(), d["seq_lens"].data_ptr(),
                                          d["parent"].data_ptr(), out.data_ptr(), B, N, Hq, inp["Hkv"], D, 16,
                                          big_blocks, inp["num_blocks"], inp["scale"], tsv.TSV_F32,
                                          err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == tsv.TSV_ERR_UNSUPPORTED
    assert b"scratch" in lib.tsv_last_error()
