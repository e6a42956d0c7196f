"""Helpers for the GPU parity tests: move seeded inputs to the device, run
the CUDA path through the C ABI, compare with the CPU oracle.

Parity bar, per request whose oracle status is OK:
  - The path -- accept_len, the accepted tokens (tree: the accepted nodes)
    and out_len -- is bit-exact, unless a decision on it lies within NEAR =
    1e-6 (relative) of its boundary: an accept test with |u q - p| / q <
    NEAR, or, in naive tree sampling, a draw that chose a child.  Such
    "near-path" requests may differ and are only checked for validity; they
    must stay under 1e-4 of the accept tests.
  - The emitted token is bit-exact unless the final inverse-CDF draw is
    near (u S within NEAR S of a CDF step).  Then it must lie within the
    oracle's window: the ids whose CDF step meets [u S - NEAR S, u S +
    NEAR S] (oracle.icdf_window).  NEAR covers the kernel's arithmetic:
    fp32 weights from fp32 normalisers, about 3e-7 relative of the total
    mass in the worst case summed over a row, float-pair running sums.
  - p_i(x_i), q_i(x_i) within 1e-5 relative.
Each comparison's counts are recorded (PARITY_LOG) and summed up at the end
of the pytest session (tests/conftest.py).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import speculative_decoding_verification_63_gb300 as sv

NEAR = oracle.NEAR
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


PARITY_LOG: list[tuple[str, dict]] = []


def _current_test() -> str:
    import os
    return os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]


def compare(got, ref, draws_per_request, check_probs=True, prefix_tokens=None, V=None):
    """Assert parity (see the module docstring).  Returns a dict of counts:
    requests compared, exact (no near decision), near_accept (near path),
    near_draw (final draw near, path exact), draw_mismatch (near draws
    whose token differs from the oracle's, inside its window),
    path_mismatch (near-path requests whose result differs) and
    max_mismatch_margin (the largest oracle margin among the draw
    mismatches: how close to a CDF step the kernel's rounding reaches)."""
    B = len(ref["status"])
    ok = ref["status"] == 0
    walk = ref.get("margin_walk", np.full(B, np.inf))
    near_path = ok & ((ref["margin_accept"] < NEAR) | (walk < NEAR))
    near_draw = ok & ~near_path & (ref["margin_draw"] < NEAR)
    firm = ok & ~near_path
    exact = firm & ~near_draw
    # the path: bit-exact wherever no decision on it is near
    for k in ("out_len", "accept_len", "accepted_nodes"):
        if k in ref and k in got:
            bad = np.nonzero(np.any((got[k] != ref[k]).reshape(B, -1), axis=1) & firm)[0]
            assert bad.size == 0, (k, bad[:10], got[k][bad[:3]], ref[k][bad[:3]],
                                   ref["margin"][bad[:3]])
    gt, rt = got["out_tokens"], ref["out_tokens"]
    n_out = ref["out_len"]
    last = np.clip(n_out - 1, 0, gt.shape[1] - 1)
    rows = np.arange(B)
    # every token but the emitted one is bit-exact
    mask = np.ones_like(gt, dtype=bool)
    mask[rows, last] = False
    bad = np.nonzero(np.any((gt != rt) & mask, axis=1) & firm)[0]
    assert bad.size == 0, ("out_tokens", bad[:10], gt[bad[:3]], rt[bad[:3]])
    # the emitted token: the oracle's, or inside its near-draw window
    tok = gt[rows, last]
    lo, hi = ref["draw_lo"], ref["draw_hi"]
    bad = np.nonzero(firm & ~((tok >= lo) & (tok <= hi)))[0]
    assert bad.size == 0, ("emitted token", bad[:10], tok[bad[:3]], rt[bad[:3], last[bad[:3]]],
                           lo[bad[:3]], hi[bad[:3]], ref["margin_draw"][bad[:3]])
    bad = np.nonzero(exact & (tok != rt[rows, last]))[0]
    assert bad.size == 0, ("emitted token", bad[:10], ref["margin_draw"][bad[:3]])
    mism = near_draw & (tok != rt[rows, last])
    draw_mism = int(mism.sum())
    worst = float(ref["margin_draw"][mism].max()) if draw_mism else 0.0
    # failed requests report nothing
    assert np.all(got["out_len"][~ok] == 0)
    # near-path requests: a valid result
    path_mism = 0
    for b in np.nonzero(near_path)[0]:
        n = int(got["out_len"][b])
        assert 1 <= n <= got["out_tokens"].shape[1], (b, n)
        row = got["out_tokens"][b]
        if prefix_tokens is not None:
            assert np.array_equal(row[:n - 1], prefix_tokens[b][:n - 1]), b
        assert 0 <= row[n - 1] < (V if V is not None else 1 << 30)
        assert np.all(row[n:] == -1)
        path_mism += int(not np.array_equal(got["out_tokens"][b], ref["out_tokens"][b]))
    if check_probs and "p_at_draft" in got:
        for g, r in (("p_at_draft", "p_at"), ("q_at_draft", "q_at")):
            m = ok[:, None] & np.isfinite(ref[r])
            np.testing.assert_allclose(got[g][m], ref[r][m], rtol=RTOL, atol=1e-30)
            assert np.all(np.isnan(got[g][ok[:, None] & ~np.isfinite(ref[r])]))
    n_acc_tests = int((draws_per_request - 1) * ok.sum())
    assert near_path.sum() <= max(1, 1e-4 * n_acc_tests), (int(near_path.sum()), n_acc_tests)
    stats = dict(requests=int(ok.sum()), exact=int(exact.sum()),
                 near_accept=int(near_path.sum()), near_draw=int(near_draw.sum()),
                 draw_mismatch=draw_mism, path_mismatch=path_mism,
                 max_mismatch_margin=worst)
    PARITY_LOG.append((_current_test(), stats))
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
