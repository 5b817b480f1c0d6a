"""The C ABI library builds for sm_103a, loads, and exports every entry point that
include/tsv.h declares; host-side argument checks answer without a GPU."""
import ctypes

import pytest

import tree_speculative_decoding_03_gb300 as tsv


@pytest.fixture(scope="module")
def lib():
    tsv.build()
    return tsv.load()


def test_exports_every_declared_symbol(lib):
    names = tsv.header_symbols()
    assert {"tsv_tree_verify_attn", "tsv_tree_reject_sample", "tsv_kv_compact_accepted",
            "tsv_attn_workspace_size", "tsv_last_error"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_host_argument_checks_need_no_gpu(lib):
    P = None
    # tree too large: rejected before any CUDA call
    st = lib.tsv_tree_reject_sample(P, P, P, P, P, P, 1.0, 4, 200, 100, P, P, P, P, P, P)
    assert st == tsv.TSV_ERR_UNSUPPORTED
    assert b"tree nodes" in lib.tsv_last_error()
    st = lib.tsv_tree_reject_sample(P, P, P, P, P, P, -1.0, 4, 8, 100, P, P, P, P, P, P)
    assert st == tsv.TSV_ERR_ARG
    st = lib.tsv_tree_reject_sample(P, P, P, P, P, P, 1.0, 4, 8, 100, P, P, P, P, P, P)
    assert st == tsv.TSV_ERR_ARG and b"null" in lib.tsv_last_error()
    # head dim 96 is not built
    st = lib.tsv_tree_verify_attn(P, P, P, P, P, P, P, 2, 8, 8, 2, 96, 16, 4, 8, 0.1, 0, P, 0, P, P)
    assert st == tsv.TSV_ERR_UNSUPPORTED
    st = lib.tsv_tree_verify_attn(P, P, P, P, P, P, P, 2, 8, 6, 4, 64, 16, 4, 8, 0.1, 0, P, 0, P, P)
    assert st == tsv.TSV_ERR_ARG  # Hq not a multiple of Hkv
    st = lib.tsv_kv_compact_accepted(P, P, P, P, P, P, P, 2, 8, 2, 64, 12, 4, 8, 0, P, P)
    assert st == tsv.TSV_ERR_UNSUPPORTED  # block size 12
    # empty batch is a no-op
    assert lib.tsv_kv_compact_accepted(P, P, P, P, P, P, P, 0, 8, 2, 64, 16, 4, 8, 0, P, P) == tsv.TSV_OK
    # the fused walk + rewrite checks both calls' arguments
    fused = lib.tsv_tree_reject_sample_compact
    walk = [P] * 6
    assert fused(*walk, 1.0, 4, 200, 100, *[P] * 5, *[P] * 5, 2, 64, 16, 4, 8, 0, P, P) == tsv.TSV_ERR_UNSUPPORTED
    assert fused(*walk, 1e-8, 4, 8, 100, *[P] * 5, *[P] * 5, 2, 64, 16, 4, 8, 0, P, P) == tsv.TSV_ERR_UNSUPPORTED
    fake = [16] * 5  # non-null, never dereferenced: the call is refused before any launch
    assert fused(*[16] * 6, 0.0, 4, 8, 100, *fake, *fake, 2, 64, 12, 4, 8, 0, 16, P) == tsv.TSV_ERR_UNSUPPORTED
    assert fused(*[16] * 6, 0.0, 4, 8, 100, *fake, *[P] * 5, 2, 64, 16, 4, 8, 0, P, P) == tsv.TSV_ERR_ARG
    assert fused(*walk, 1.0, 0, 8, 100, *[P] * 5, *[P] * 5, 2, 64, 16, 4, 8, 0, P, P) == tsv.TSV_OK
    # walk options: checked before anything else is looked at
    from tree_speculative_decoding_03_gb300 import WalkOptions
    ex = lib.tsv_tree_reject_sample_ex
    for opts, want in ((WalkOptions(2, 1, 0, 1.0), tsv.TSV_ERR_ARG), (WalkOptions(0, 7, 0, 1.0), tsv.TSV_ERR_ARG),
                       (WalkOptions(0, 1, -1, 1.0), tsv.TSV_ERR_ARG), (WalkOptions(0, 1, 0, 0.0), tsv.TSV_ERR_ARG),
                       (WalkOptions(0, 1, 0, 1.5), tsv.TSV_ERR_ARG), (WalkOptions(0, 1, 0, float("nan")), tsv.TSV_ERR_ARG)):
        assert ex(*[16] * 6, 1.0, ctypes.byref(opts), 4, 8, 100, *[16] * 5, P) == want
    assert ex(*walk, 1.0, None, 0, 8, 100, *[P] * 5, P) == tsv.TSV_OK  # NULL options, empty batch
    # single-chunk plans need no workspace
    assert lib.tsv_attn_workspace_size(1, 15, 8, 2, 64, 16, 16, tsv.TSV_F32) == 0
    assert lib.tsv_attn_workspace_size(1, 15, 8, 2, 64, 16, 17, tsv.TSV_F32) > 0  # prefix may need 2 chunks
    assert lib.tsv_attn_workspace_size(1, 15, 8, 2, 96, 16, 17, tsv.TSV_F32) == 0


def test_error_bits_match_the_header():
    import re
    text = open(tsv.HEADER if hasattr(tsv, "HEADER") else __import__("os").path.join(
        __import__("os").path.dirname(__file__), "..", "include", "tsv.h")).read()
    for name in ["TSV_DERR_PARENT", "TSV_DERR_BLOCK", "TSV_DERR_CAPACITY", "TSV_DERR_TOKEN", "TSV_DERR_NONFINITE",
                 "TSV_DERR_TIMEOUT"]:
        m = re.search(name + r"\s*=\s*(\d+)", text)
        assert m and int(m.group(1)) == getattr(tsv, name), name


def test_every_refusal_happens_before_any_launch(lib):
    """Each host-side check answers on a machine without a GPU: the fake (aligned,
    never dereferenced) pointers below would fault if anything reached the device."""
    P, A, M = None, 4096, 4104  # null, 16-byte aligned, misaligned
    attn = lib.tsv_tree_verify_attn

    def call(q=A, out=A, B=2, N=8, Hq=8, Hkv=2, D=64, bs=16, mb=4, nb=8, scale=0.125, dt=0, ws=P, wsb=0):
        return attn(q, A, A, A, A, A, out, B, N, Hq, Hkv, D, bs, mb, nb, scale, dt, ws, wsb, A, P)

    assert call(q=M) == tsv.TSV_ERR_ARG and b"aligned" in lib.tsv_last_error()
    assert call(out=M) == tsv.TSV_ERR_ARG
    for bad_scale in (0.0, -1.0, float("nan"), float("inf")):
        assert call(scale=bad_scale) == tsv.TSV_ERR_ARG, bad_scale
    assert call(N=128, Hq=64, Hkv=4) == tsv.TSV_ERR_UNSUPPORTED  # 2048 query rows per kv head
    assert call(dt=5) == tsv.TSV_ERR_ARG
    assert call(Hkv=0) == tsv.TSV_ERR_ARG
    assert call(N=0) == tsv.TSV_ERR_ARG
    assert call(bs=32 + 1) == tsv.TSV_ERR_UNSUPPORTED
    assert call(B=0, q=P, out=P) == tsv.TSV_OK  # empty batch: nothing to do, nothing read

    walk = lib.tsv_tree_reject_sample
    arrs = [A] * 6
    outs = [A] * 5
    assert walk(*arrs, 1.0, 2, 8, 0, *outs, P) == tsv.TSV_ERR_ARG  # V = 0
    assert walk(*arrs, 1.0, 2, 8, 16 * 512 * 32 + 1, *outs, P) == tsv.TSV_ERR_UNSUPPORTED
    for bad_t in (float("nan"), float("inf"), -0.5):
        assert walk(*arrs, bad_t, 2, 8, 100, *outs, P) == tsv.TSV_ERR_ARG, bad_t
    assert walk(*arrs, 1.0, 2, 0, 100, *outs, P) == tsv.TSV_ERR_ARG  # no root
    assert walk(*[P] * 6, 1.0, 0, 8, 100, *[P] * 5, P) == tsv.TSV_OK  # empty batch

    comp = lib.tsv_kv_compact_accepted
    assert comp(M, A, A, A, A, A, A, 2, 8, 2, 64, 16, 4, 8, 0, A, P) == tsv.TSV_ERR_ARG
    assert comp(A, A, A, A, A, A, A, 2, 8, 2, 96, 16, 4, 8, 0, A, P) == tsv.TSV_ERR_UNSUPPORTED
    assert comp(A, A, A, A, A, A, A, 2, 8, 2, 64, 16, 4, 8, 9, A, P) == tsv.TSV_ERR_ARG
    assert comp(A, A, A, A, P, A, A, 2, 8, 2, 64, 16, 4, 8, 0, A, P) == tsv.TSV_ERR_ARG

    assert lib.tsv_noalloc_scratch_bytes() == 64 << 20
