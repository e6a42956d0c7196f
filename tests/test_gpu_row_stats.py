"""Per-position acceptance statistics on the GPU against the fp64 oracle.

Tolerance, from the arithmetic: alpha is a sum of V terms min(p, q), each
an fp32 2^x from the special-function unit (relative error about 2^-22),
accumulated per thread over at most 64 terms in fp32 (relative error at
most 64 * 2^-24 of that thread's part) and then in fp64; the row totals Z
come from fp32 (max, sum) pairs (a few 2^-24 relative).  That bounds the
error of alpha, which lies in [0, 1], well below 2e-5; the expected
tokens multiply up to K = 32 such rates: 1e-4 relative.  Greedy positions
(argmax agreement) must match exactly."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_63_gb300 as sv
from speculative_decoding_verification_63_gb300 import workloads as wl

from gpu_util import dev

pytestmark = pytest.mark.gpu

ATOL_ALPHA = 2e-5
RTOL_EXPECTED = 1e-4


def run_stats(inp, ws=None, target=None, draft=None, max_top_k=None):
    out = sv.row_stats(target if target is not None else dev(inp["target"]),
                       draft if draft is not None else dev(inp["draft"]),
                       dev(inp["temperature"]), num_drafts=dev(inp["num_drafts"]),
                       top_k=dev(inp["top_k"]) if inp["top_k"].any() else None, ws=ws,
                       max_top_k=max_top_k)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def check_stats(inp, **kw):
    got = run_stats(inp, **kw)
    ref = oracle.row_stats_inputs(inp)
    ok = ref["status"] == 0
    a, r = got["alpha"][ok], ref["alpha"][ok]
    assert np.array_equal(np.isnan(a), np.isnan(r))
    m = ~np.isnan(r)
    np.testing.assert_allclose(a[m], r[m], rtol=0, atol=ATOL_ALPHA)
    greedy = (inp["temperature"] == 0)[ok]
    if greedy.any():
        g = np.broadcast_to(greedy[:, None], r.shape) & m
        assert np.array_equal(a[g], r[g])
    np.testing.assert_allclose(got["expected"][ok], ref["expected"][ok], rtol=RTOL_EXPECTED)
    assert np.all(np.isnan(got["expected"][~ok]))
    return got, ref


def test_stats_headline_full_size():
    """B=64, K=6, V=128256 bf16, half greedy: every position checked."""
    got, ref = check_stats(wl.make_chain(3))
    sampled = wl.make_chain(3)["temperature"] > 0
    assert 0.0 < ref["alpha"][sampled].mean() < 1.0


def test_stats_small_chain_and_ragged():
    rng = np.random.default_rng(60)
    nd = rng.integers(0, 5, 40).astype(np.int32)
    inp = wl.make_chain(2, B=40, num_drafts=nd, seed=61)
    inp["temperature"] = rng.choice([0.0, 0.5, 0.8, 1.3], 40).astype(np.float32)
    check_stats(inp)


@pytest.mark.parametrize("V", [7, 1001, 70_000, 152_064])
def test_stats_row_lengths(V):
    """Unaligned rows (plain loads), fp32 rows past the register tile, and
    bf16 rows past it (workload 5's vocabulary)."""
    if V == 70_000:
        inp = wl.make_chain(1, B=6, V=V, seed=62)
    else:
        inp = wl.make_chain(5, B=6, K=4, V=V, seed=62 + V)
        inp["top_k"][:] = 0
    check_stats(inp)


def test_stats_no_drafts():
    inp = wl.make_chain(2, B=5, K=0, V=3000, seed=63)
    got = run_stats(inp, draft=torch.zeros((5, 0, 3000), dtype=torch.bfloat16, device="cuda"))
    assert np.all(got["expected"] == 1.0)


def test_stats_topk_workload_shape():
    """Workload 5's shape (K=8, V=152064 bf16, t=0.7, top-k 50 on p and
    q): alpha_i is the sum of min(p_i, q_i) over the tokens both kept sets
    hold, from the top-k pass's lists."""
    inp = wl.make_chain(5, B=24)
    got, ref = check_stats(inp)
    assert 0.0 < ref["alpha"].mean() < 1.0


def test_stats_topk_mixed_batch():
    """Filtered and unfiltered, greedy and sampled requests in one call,
    ragged drafts, ties at the k-th logit (rows of equal logits), and
    k = 1 and k = 64."""
    rng = np.random.default_rng(67)
    B = 16
    nd = rng.integers(0, 5, B).astype(np.int32)
    inp = wl.make_chain(5, B=B, K=4, V=9000, num_drafts=nd, seed=68)
    inp["top_k"] = rng.choice([0, 1, 7, 50, 64], B).astype(np.int32)
    inp["temperature"] = rng.choice([0.0, 0.7, 1.1], B).astype(np.float32)
    inp["target"][3, :, 100:200] = inp["target"][3, :, 150:151]   # a run of equal logits
    inp["draft"][3, :, 100:200] = inp["draft"][3, :, 150:151]
    check_stats(inp)
    ws = sv.workspace(sv.sv_chain_workspace_bytes(B, 4, 9000, sv.SV_BF16, 64), "cuda", "stk")
    for _ in range(2):  # the lists are left zero for the next call on the workspace
        check_stats(inp, ws=ws)
        from gpu_util import check_chain
        check_chain(inp, ws=ws)


def test_stats_data_errors():
    inp = wl.make_chain(2, B=6, V=2000, seed=64)
    inp["target"][1, 2, 77] = 0x7FC0      # NaN
    inp["draft"][2, 0, :] = 0xFF80        # a draft row with no mass
    inp["temperature"][3] = -1.0
    inp["top_k"][4] = 20                  # top-k filtering without lists (max_top_k 0)
    ws = sv.workspace(sv.sv_chain_workspace_bytes(6, 4, 2000, sv.SV_BF16), "cuda", "stats_err")
    got = run_stats(inp, ws=ws, max_top_k=0)
    st, flags = sv.sv_get_error(ws)
    assert st == sv.SV_EDATA
    assert flags & sv.SV_DERR_NONFINITE and flags & sv.SV_DERR_MASS and flags & sv.SV_DERR_ARG
    assert np.all(np.isnan(got["expected"][1:5]))
    inp["top_k"][4] = 0
    ref = oracle.row_stats_inputs(inp)
    for b in (0, 5):
        np.testing.assert_allclose(got["alpha"][b], ref["alpha"][b], atol=ATOL_ALPHA)
    sv.sv_workspace_init(ws)
    # the workspace serves a chain call afterwards
    from gpu_util import check_chain
    check_chain(wl.make_chain(2, B=6, V=2000, seed=65), ws=ws)


def test_stats_then_verify_share_a_workspace():
    """The statistics' per-request counters are left zero for the chain
    call that follows on the same workspace."""
    from gpu_util import check_chain
    inp = wl.make_chain(3, B=16, V=20_000, seed=66)
    ws = sv.workspace(sv.sv_chain_workspace_bytes(16, 6, 20_000, sv.SV_BF16), "cuda", "share")
    for _ in range(2):
        check_stats(inp, ws=ws)
        check_chain(inp, ws=ws)
    st, flags = sv.sv_get_error(ws)
    assert st == sv.SV_OK and flags == 0
