"""Helpers of the GPU parity tests: move a generated batch to the device, run the
three library calls, and compare decisions with the oracle's under the stated
near-tie exemption."""
from __future__ import annotations

import numpy as np
import torch

import tree_speculative_decoding_03_gb300 as tsv

EXEMPT_BAND = 1e-6  # |u - p/q| (or |u - CDF boundary|) below which a decision may differ


def dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def device_inputs(inp, attn=True, verify=True):
    d = dict(parent=dev(inp["parent"]))
    if attn:
        bf = inp["dtype"] == "bf16"
        el = torch.bfloat16 if bf else None

        def kv(x):
            return dev(x.view(np.int16) if bf else x, el)

        d.update(q=kv(inp["q"]), k_cache=kv(inp["k_cache"]), v_cache=kv(inp["v_cache"]),
                 block_table=dev(inp["block_table"]), seq_lens=dev(inp["seq_lens"]))
    if verify:
        tl = inp["target_logits"]
        d.update(target_logits=dev(tl.view(np.int16), torch.bfloat16) if tl.dtype == np.uint16 else dev(tl),
                 draft_probs=dev(inp["draft_probs"]),
                 draft_tokens=dev(inp["draft_tokens"]), u_accept=dev(inp["u_accept"]), u_bonus=dev(inp["u_bonus"]))
    return d


def run_attn(inp, d=None):
    d = d or device_inputs(inp, verify=False)
    B, N, Hq, D = d["q"].shape
    out = torch.empty_like(d["q"])
    ws_bytes = tsv.attn_workspace_size(B, N, Hq, inp["Hkv"], D, inp["block_size"], inp["max_blocks"],
                                       tsv.TSV_BF16 if inp["dtype"] == "bf16" else tsv.TSV_F32)
    ws = torch.empty(max(1, ws_bytes), dtype=torch.uint8, device="cuda") if ws_bytes else None
    err = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    tsv.tree_verify_attn(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], d["parent"], out,
                         inp["scale"], workspace=ws, seq_err=err)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().reshape(B * N * Hq, D).astype(np.float64), err.cpu().numpy()


def run_verify(inp, d=None, temperature=None, **opts):
    """The walk on the device (opts: with_replacement, top_k, top_p).  Target logits
    given as uint16 are bfloat16 bit patterns."""
    d = d or device_inputs(inp, attn=False)
    if d["target_logits"].dtype == torch.int16:
        d["target_logits"] = d["target_logits"].view(torch.bfloat16)
    B, N, V = d["target_logits"].shape
    T = inp["T"] if temperature is None else temperature
    an = torch.full((B, N), -9, dtype=torch.int32, device="cuda")
    al = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    bt = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    ot = torch.full((B, N), -9, dtype=torch.int32, device="cuda")
    err = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    tsv.tree_reject_sample(d["target_logits"], d["draft_probs"], d["draft_tokens"], d["parent"], d["u_accept"],
                           d["u_bonus"], T, an, al, bt, ot, err, **opts)
    torch.cuda.synchronize()
    return dict(accepted_nodes=an.cpu().numpy(), accept_len=al.cpu().numpy(), bonus_token=bt.cpu().numpy(),
                out_tokens=ot.cpu().numpy(), err=err.cpu().numpy())


def run_compact(inp, accepted_nodes, accept_len, d=None):
    d = d or device_inputs(inp, verify=False)
    B = len(accept_len)
    new_len = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    err = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    tsv.kv_compact_accepted(d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                            dev(accepted_nodes), dev(accept_len), new_len, err)
    torch.cuda.synchronize()
    bf = inp["dtype"] == "bf16"

    def host(t):
        a = t.cpu()
        return a.view(torch.int16).numpy().view(np.uint16) if bf else a.numpy()

    return host(d["k_cache"]), host(d["v_cache"]), new_len.cpu().numpy(), err.cpu().numpy()


def first_divergent_trial(inp, g, o, b):
    """For a sequence whose GPU and oracle walks differ, the child whose test
    decided differently first (both walks tried it), or -1 if the paths agree."""
    pg, po = g["accepted_nodes"][b], o["accepted_nodes"][b]
    parent = inp["parent"][b]
    for j in range(1, len(po)):
        if pg[j] != po[j]:
            p = po[j - 1]
            cands = [c for c in (pg[j], po[j]) if c >= 0]
            c_star = min(cands)
            assert parent[c_star] == p
            return int(c_star)
    return -1


def compare_decisions(inp, g, o, T):
    """Bit-exact comparison of the walk outputs, except sequences whose first
    differing decision is a near tie: |u - p/q| < 1e-6 for an accept test, or
    u_bonus within 1e-6 of a CDF boundary around the oracle's bonus token.
    Returns (n_exempt, list of failure strings)."""
    B = len(o["accept_len"])
    fails, exempt = [], 0
    assert np.array_equal(g["err"], o["err"]), (g["err"], o["err"])
    for b in range(B):
        same = (np.array_equal(g["accepted_nodes"][b], o["accepted_nodes"][b])
                and g["accept_len"][b] == o["accept_len"][b] and g["bonus_token"][b] == o["bonus_token"][b]
                and np.array_equal(g["out_tokens"][b], o["out_tokens"][b]))
        if same:
            continue
        if T == 0:
            fails.append(f"seq {b}: greedy walk differs")
            continue
        c = first_divergent_trial(inp, g, o, b)
        if c >= 0:
            r = o["ratio"][b, c]
            u = float(inp["u_accept"][b, c])
            if np.isfinite(r) and abs(u - r) < EXEMPT_BAND:
                exempt += 1
                continue
            fails.append(f"seq {b}: child {c} u={u!r} oracle ratio={r!r}")
        else:
            lo, hi = o["bonus_cdf"][b]
            u = float(inp["u_bonus"][b])
            if abs(u - lo) < EXEMPT_BAND or abs(u - hi) < EXEMPT_BAND:
                exempt += 1
                continue
            fails.append(f"seq {b}: bonus {g['bonus_token'][b]} vs {o['bonus_token'][b]} u={u!r} cdf=({lo!r},{hi!r})")
    return exempt, fails
