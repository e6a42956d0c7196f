"""Chain verification on the GPU against the fp64 oracle (bit-exact tokens
and lengths outside near-boundary draws; probabilities to 1e-5 relative)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_63_gb300 as sv
from speculative_decoding_verification_63_gb300 import workloads as wl

from gpu_util import check_chain, compare, dev, run_chain

pytestmark = pytest.mark.gpu


def test_toy_chain_10000_rounds():
    """Toy workload (B=4, K=4, V=5 fp32): 10,000 rounds of 4 requests, run
    as one batch of 40,000 independent requests."""
    total = dict(requests=0, exact=0, near_accept=0, near_draw=0)
    for r in range(40):
        inp = wl.make_chain(1, B=1000, seed=wl.SEED_BASE + 1 + 1000 * r)
        st, got, _ = check_chain(inp)
        for k in total:
            total[k] += st[k]
    assert total["requests"] == 40_000
    # with V = 5 every decision is a coarse one: near draws of either kind are rare
    assert total["near_accept"] + total["near_draw"] <= 1e-4 * 40_000 * 5


def test_small_chain_many_seeds():
    """Small-chain workload (K=4, V=32000 bf16, peaked target): 64 requests."""
    check_chain(wl.make_chain(2, B=64))


@pytest.mark.parametrize("B", [1, 3, 7])
def test_small_chain_odd_batches(B):
    """The small-chain workload as specified (B=1) and other odd batch sizes
    (per-request tables of odd length in shared memory)."""
    for seed in range(3):
        check_chain(wl.make_chain(2, B=B, seed=wl.SEED_BASE + 2 + 17 * seed + B))


def test_headline_full_size():
    """B=64, K=6, V=128256 bf16, half greedy: every request checked."""
    st, got, ref = check_chain(wl.make_chain(3))
    assert got["accept_len"].max() > 0 and st["exact"] >= 60


@pytest.mark.parametrize("mix", ["all", "none"])
def test_headline_greedy_and_sampled(mix):
    check_chain(wl.make_chain(3, B=12, greedy=mix, seed=7))


def test_ragged_num_drafts():
    rng = np.random.default_rng(3)
    nd = rng.integers(0, 7, 24).astype(np.int32)
    nd[:3] = [0, 6, 1]
    check_chain(wl.make_chain(3, B=24, num_drafts=nd, seed=8))


@pytest.mark.parametrize("V", [7, 1001, 40_003])
def test_unaligned_vocab_takes_direct_path(V):
    """bf16 rows of V not a multiple of 8 are not 16-byte aligned: the
    kernel reads them directly instead of through bulk copies."""
    check_chain(wl.make_chain(2, B=16, V=V, seed=V))


@pytest.mark.parametrize("V", [8, 16384, 16392, 65536 + 8])
def test_chunk_boundaries(V):
    """V around the 32 KB chunk size (16384 bf16): single, exact and ragged
    last chunks."""
    check_chain(wl.make_chain(3, B=8, V=V, seed=V + 1))


def test_rows_of_more_than_eight_chunks():
    """Rows longer than eight 32 KB chunks (bf16 V = 150000: ten chunks;
    fp32 V = 70000: nine), so a row's partials are merged in several batches."""
    inp = wl.make_chain(3, B=6, V=150_000, seed=150)
    inp["temperature"][:] = 1.0  # every request sampled: the (max, sum) merge
    check_chain(inp)
    check_chain(wl.make_chain(1, B=4, V=70_000, seed=70))


def test_fp32_aligned_rows():
    inp = wl.make_chain(1, B=16, V=12_000, seed=4)
    check_chain(inp)


def test_padded_row_stride():
    inp = wl.make_chain(3, B=6, V=5000, seed=9)
    pad = 5000 + 24
    t = np.zeros((6, 7, pad), np.uint16)
    d = np.zeros((6, 6, pad), np.uint16)
    t[..., :5000] = inp["target"]
    d[..., :5000] = inp["draft"]
    tt = dev(t)[..., :5000]
    dd = dev(d)[..., :5000]
    out = sv.verify_chain(tt, dd, dev(inp["tokens"]), dev(inp["temperature"]),
                          dev(inp["uniforms"]), num_drafts=dev(inp["num_drafts"]),
                          with_probs=True)
    torch.cuda.synchronize()
    got = {k: v.cpu().numpy() for k, v in out.items()}
    compare(got, oracle.verify_chain_inputs(inp), 7, prefix_tokens=inp["tokens"])


def test_mixed_temperatures():
    inp = wl.make_chain(2, B=40, V=3000, seed=11)
    rng = np.random.default_rng(0)
    inp["temperature"] = rng.choice([0.0, 0.3, 0.7, 1.0, 1.7], 40).astype(np.float32)
    check_chain(inp)


def test_no_drafts_is_plain_sampling():
    inp = wl.make_chain(2, B=10, K=0, V=3000, seed=12)
    st, got, ref = check_chain(inp)
    assert np.all(got["out_len"] == 1)


def test_many_requests():
    check_chain(wl.make_chain(2, B=1024, K=3, V=64, seed=13))


def test_workspace_reuse_gives_same_result():
    inp = wl.make_chain(3, B=16, V=20_000, seed=14)
    ws = sv.workspace(sv.sv_chain_workspace_bytes(16, 6, 20_000, sv.SV_BF16), "cuda", "reuse")
    a = run_chain(inp, ws=ws)
    b = run_chain(inp, ws=ws)
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True), k
    st, flags = sv.sv_get_error(ws)
    assert st == sv.SV_OK and flags == 0


def test_one_workspace_serves_calls_of_any_shape():
    """Chain calls of different shapes, a tree call and a top-k call in turn
    on one workspace: what one call writes anywhere in it must not be taken
    by the next for its own results (the sequence B = 64, 1, 1, 1, 3 once
    reused segment sums as chunk partials)."""
    from gpu_util import check_tree
    need = max(sv.sv_chain_workspace_bytes(64, 8, 32_000, sv.SV_BF16, 64),
               sv.sv_tree_workspace_bytes(16, 32, 32, 32_000, sv.SV_BF16))
    ws = sv.workspace(need, "cuda", "shapes")
    check_chain(wl.make_chain(2, B=64), ws=ws)
    for s_ in range(3):
        check_chain(wl.make_chain(2, B=1, seed=wl.SEED_BASE + 2 + 17 * s_ + 1), ws=ws)
    check_chain(wl.make_chain(2, B=3, seed=wl.SEED_BASE + 2 + 3), ws=ws)
    check_tree(wl.make_tree(B=6, seed=61), ws=ws)
    check_chain(wl.make_chain(3, B=5, V=20_000, seed=62), ws=ws)
    check_chain(wl.make_chain(5, B=8, V=20_000, seed=wl.SEED_BASE + 563), ws=ws)
    check_chain(wl.make_chain(2, B=3, seed=wl.SEED_BASE + 2 + 3), ws=ws)
    st, flags = sv.sv_get_error(ws)
    assert st == sv.SV_OK and flags == 0


def test_data_errors_are_reported_per_request():
    inp = wl.make_chain(2, B=6, V=2000, seed=15)
    t = wl.bf16_bits_to_f32(inp["target"]).copy()
    inp["target"][1, 2, 77] = 0x7FC0          # NaN in a target row of request 1
    inp["tokens"][2, 1] = 2000                # token out of range in request 2
    inp["temperature"][3] = -1.0              # invalid temperature in request 3
    inp["target"][4, 0, :] = 0xFF80           # an all -inf row: no mass
    ws = sv.workspace(sv.sv_chain_workspace_bytes(6, 4, 2000, sv.SV_BF16), "cuda", "errs")
    got = run_chain(inp, ws=ws)
    st, flags = sv.sv_get_error(ws)
    assert st == sv.SV_EDATA
    assert flags & sv.SV_DERR_NONFINITE and flags & sv.SV_DERR_TOKEN
    assert flags & sv.SV_DERR_ARG and flags & sv.SV_DERR_MASS
    assert list(got["out_len"][1:5]) == [0, 0, 0, 0]
    ref = oracle.verify_chain_inputs(inp)
    assert list(ref["status"][1:5]) == [oracle.ENONFINITE, oracle.ETOKEN, oracle.EARG,
                                        oracle.EMASS]
    ok = ref["status"] == 0
    assert np.array_equal(got["out_tokens"][ok], ref["out_tokens"][ok])
    # the workspace is usable again after re-initialisation
    sv.sv_workspace_init(ws)
    good = wl.make_chain(2, B=6, V=2000, seed=16)
    compare(run_chain(good, ws=ws), oracle.verify_chain_inputs(good), 5,
            prefix_tokens=good["tokens"])


def test_failed_requests_leave_the_workspace_clean():
    """Sampled requests that fail publish a failed draw, whose record the
    last of its draw-pass claims clears: the next call on the same
    workspace, with no re-initialisation, must see none of it."""
    bad = wl.make_chain(3, B=12, V=20_000, seed=18, greedy="none")
    for b in (1, 4, 7):
        bad["target"][b, 3, 500] = 0x7FC0     # NaN: request b fails
    bad["tokens"][10, 0] = 20_000             # out of range: request 10 fails
    ws = sv.workspace(sv.sv_chain_workspace_bytes(12, 6, 20_000, sv.SV_BF16), "cuda", "clean")
    got = run_chain(bad, ws=ws)
    assert list(got["out_len"][[1, 4, 7, 10]]) == [0, 0, 0, 0]
    st, flags = sv.sv_get_error(ws)
    assert st == sv.SV_EDATA
    for seed in (19, 20):
        good = wl.make_chain(3, B=12, V=20_000, seed=seed, greedy="none")
        compare(run_chain(good, ws=ws), oracle.verify_chain_inputs(good), 12,
                prefix_tokens=good["tokens"])
    st, flags = sv.sv_get_error(ws)
    assert st == sv.SV_OK and flags == 0


def test_greedy_with_nan_draft_rows_is_fine():
    """Greedy requests never read draft rows."""
    inp = wl.make_chain(3, B=4, V=4000, greedy="all", seed=17)
    inp["draft"][:] = 0x7FC0
    check_chain(inp)


def test_bounded_wait_reports_timeout():
    ws = sv.workspace(4096, "cuda", "timeout")
    assert sv.sv_selftest_wait_timeout(ws, 20_000_000) == sv.SV_ETIMEOUT
    sv.sv_workspace_init(ws)
    # the context stays usable
    check_chain(wl.make_chain(2, B=2, V=1000, seed=18))


def test_empty_batch():
    out = sv.verify_chain(torch.zeros((0, 5, 100), dtype=torch.bfloat16, device="cuda"),
                          torch.zeros((0, 4, 100), dtype=torch.bfloat16, device="cuda"),
                          torch.zeros((0, 4), dtype=torch.int32, device="cuda"),
                          torch.zeros(0, device="cuda"), torch.zeros((0, 5), device="cuda"))
    torch.cuda.synchronize()
    assert out["out_tokens"].shape == (0, 5)
