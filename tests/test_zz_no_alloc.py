"""tsv_tree_verify_attn_noalloc: the attention call for callers that cannot
allocate device memory (an engine plugin that only receives its inputs and
outputs, a loop that must not call cudaMalloc).  Its split-K scratch is the
library's own fixed device array.  Two calls in a row through the C ABI must give
what the workspace-taking entry point gives, within the attention tolerance, and
a shape that needs more scratch than the array holds must be refused.

This file is collected last so that a failure here comes after every other test."""
import numpy as np
import pytest
import torch

import tree_speculative_decoding_03_gb300 as tsv
import workloads as W
from gpu_util import device_inputs

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-4}


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
    return out.float().cpu().numpy(), err.cpu().numpy()


@pytest.mark.parametrize("cfg", [0, 1])
def test_no_alloc_matches_workspace_call_twice(cfg):
    tsv.build()
    inp = W.generate(W.CONFIGS[cfg])
    d = device_inputs(inp, verify=False)
    want, want_err = _with_workspace(inp, d)
    assert not want_err.any()
    for _ in range(2):
        out = torch.full_like(d["q"], float("nan"))
        err = torch.full((inp["B"],), -1, dtype=torch.int32, device="cuda")
        tsv.tree_verify_attn_noalloc(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                                     d["parent"], out, inp["scale"], seq_err=err)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.array_equal(err.cpu().numpy(), want_err)
        assert np.abs(got - want).max() <= TOL[inp["dtype"]]


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
