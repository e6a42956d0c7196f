"""Helpers for the GPU parity tests: move seeded inputs to the device, run
the CUDA path through the C ABI, compare with the CPU oracle.

Parity bar (per request whose oracle status is OK):
  - accept_len, out_len and out_tokens bit-exact, except for requests where
    some decision the oracle took lies within 1e-6 (relative) of its
    boundary ("near" draws; counted, must stay under 1e-4 of all draws);
  - p_i(x_i), q_i(x_i) within 1e-5 relative.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import speculative_decoding_verification_63_gb300 as sv

NEAR = 1e-6
RTOL = 1e-5


def dev(a):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_chain(inp, with_probs=True, ws=None, num_drafts=True, top_k=True):
    out = sv.verify_chain(dev(inp["target"]), dev(inp["draft"]), dev(inp["tokens"]),
                          dev(inp["temperature"]), dev(inp["uniforms"]),
                          num_drafts=dev(inp["num_drafts"]) if num_drafts else None,
                          top_k=dev(inp["top_k"]) if top_k and inp["top_k"].any() else None,
                          max_top_k=int(inp["top_k"].max()) if top_k and inp["top_k"].any()
                          else 0,
                          with_probs=with_probs, ws=ws)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def run_tree(inp, ws=None, mode=None):
    mode = mode or inp.get("mode", "mss")
    out = sv.verify_tree(dev(inp["target"]), None if mode == "naive" else dev(inp["draft"]),
                         dev(inp["node_tokens"]),
                         dev(inp["parent"]), dev(inp["q_row"]), dev(inp["temperature"]),
                         dev(inp["u_accept"]), dev(inp["u_sample"]),
                         max_depth=int(inp["max_depth"]), num_nodes=dev(inp["num_nodes"]),
                         ws=ws, mode=mode)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def compare(got, ref, draws_per_request, check_probs=True, prefix_tokens=None, V=None):
    """Assert parity.  Returns a dict of counts.

    Requests whose oracle decisions all lie farther than NEAR from their
    boundaries must match bit for bit.  A "near" request may differ from
    the oracle but must still be a valid result: the accepted prefix is the
    proposed tokens, the emitted token is in range.  Near accept tests must
    stay under 1e-4 of all accept tests; near inverse-CDF draws are counted
    (their share is a property of the input distribution: about
    sum_t min(p_t, 2 NEAR) per draw)."""
    ok = ref["status"] == 0
    near_acc = ok & (ref["margin_accept"] < NEAR)
    near_draw = ok & (ref["margin_draw"] < NEAR)
    near = near_acc | near_draw
    exact = ok & ~near
    for k in ("out_tokens", "out_len", "accept_len", "accepted_nodes"):
        if k in ref and k in got:
            bad = np.nonzero(np.any((got[k] != ref[k]).reshape(len(ok), -1), axis=1) & exact)[0]
            assert bad.size == 0, (k, bad[:10], got[k][bad[:3]], ref[k][bad[:3]],
                                   ref["margin"][bad[:3]])
    # failed requests report nothing
    assert np.all(got["out_len"][~ok] == 0)
    # near requests: a valid result
    mism = 0
    for b in np.nonzero(near)[0]:
        n = int(got["out_len"][b])
        assert 1 <= n <= got["out_tokens"].shape[1], (b, n)
        row = got["out_tokens"][b]
        if prefix_tokens is not None:
            assert np.array_equal(row[:n - 1], prefix_tokens[b][:n - 1]), b
        assert 0 <= row[n - 1] < (V if V is not None else 1 << 30)
        assert np.all(row[n:] == -1)
        mism += int(not np.array_equal(got["out_tokens"][b], ref["out_tokens"][b]))
    if check_probs and "p_at_draft" in got:
        for g, r in (("p_at_draft", "p_at"), ("q_at_draft", "q_at")):
            m = ok[:, None] & np.isfinite(ref[r])
            np.testing.assert_allclose(got[g][m], ref[r][m], rtol=RTOL, atol=1e-30)
            assert np.all(np.isnan(got[g][ok[:, None] & ~np.isfinite(ref[r])]))
    n_acc_tests = int((draws_per_request - 1) * ok.sum())
    assert near_acc.sum() <= max(1, 1e-4 * n_acc_tests), (int(near_acc.sum()), n_acc_tests)
    stats = dict(requests=int(ok.sum()), exact=int(exact.sum()), near_accept=int(near_acc.sum()),
                 near_draw=int(near_draw.sum()), near_mismatch=mism)
    print("parity", stats)
    return stats


def check_chain(inp, **kw):
    got = run_chain(inp, **kw)
    ref = oracle.verify_chain_inputs(inp)
    if kw.get("ws") is None:
        sv.check_device_errors(sv.workspace(1, "cuda", "chain"))
    return compare(got, ref, inp["K"] + 1, prefix_tokens=inp["tokens"], V=inp["V"]), got, ref


def tree_path_tokens(inp, got):
    """Tokens of the accepted nodes the GPU reports (for validity checks)."""
    B = inp["B"]
    out = np.full((B, inp["max_depth"] + 1), -1, np.int64)
    for b in range(B):
        L = max(int(got["accept_len"][b]), 0)
        for i in range(L):
            out[b, i] = inp["node_tokens"][b, got["accepted_nodes"][b, i]]
    return out


def check_tree(inp, **kw):
    got = run_tree(inp, **kw)
    ref = oracle.verify_tree_inputs(inp, mode=kw.get("mode"))
    return compare(got, ref, inp["N"], prefix_tokens=tree_path_tokens(inp, got),
                   V=inp["V"]), got, ref
