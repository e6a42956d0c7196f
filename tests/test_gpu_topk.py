"""Chain verification with top-k filtering on the GPU against the fp64
oracle: p and q each keep their k largest logits (ties to the lower token
id) before the accept tests and the residual ("LLM speculative decoding
study notes 02", sec. 5.4).  Tokens and lengths bit-exact outside
near-boundary decisions, probabilities to 1e-5 relative."""
import numpy as np
import pytest

from speculative_decoding_verification_63_gb300 import workloads as wl

from gpu_util import check_chain

pytestmark = pytest.mark.gpu


def _with_topk(inp, k):
    inp = dict(inp)
    inp["top_k"] = np.full(inp["B"], k, dtype=np.int32)
    return inp


def _rebuild(inp, target, draft, k, greedy=False):
    """Same shapes and uniforms, new logits (fp32 values, bf16-rounded when
    the workload is bf16) and drafts drawn from the new q."""
    rng = np.random.default_rng(99)
    dt = inp["dtype"]
    out = dict(inp)
    out["target"] = wl.to_bf16_bits(target) if dt == "bf16" else target.astype(np.float32)
    out["draft"] = wl.to_bf16_bits(draft) if dt == "bf16" else draft.astype(np.float32)
    dv = wl.bf16_bits_to_f32(out["draft"]) if dt == "bf16" else out["draft"]
    tok = np.zeros_like(inp["tokens"])
    for b in range(inp["B"]):
        for i in range(inp["K"]):
            tok[b, i] = wl.draw_draft(rng, dv[b, i], float(inp["temperature"][b]), k)
    out["tokens"] = tok
    out["top_k"] = np.full(inp["B"], k, dtype=np.int32)
    return out


def test_topk_workload_shape():
    """Top-k workload (K=8, V=152064 bf16, t=0.7, top-50) on 32 requests."""
    st, got, _ = check_chain(wl.make_chain(5, B=32))
    assert st["requests"] == 32 and got["accept_len"].max() > 0


@pytest.mark.parametrize("k", [1, 2, 50, 64])
def test_topk_sizes(k):
    inp = wl.make_chain(5, B=8, V=20000, seed=wl.SEED_BASE + 500 + k)
    rng = np.random.default_rng(k)
    t = rng.normal(0, 4, (8, 9, 20000)).astype(np.float32)
    d = t[:, :8] + rng.normal(0, 2, (8, 8, 20000)).astype(np.float32)
    check_chain(_rebuild(inp, t, d, k))


def test_topk_heavy_ties():
    """Integer logits: the k-th value is shared by many tokens, so the tie
    rule (lower token id first) decides which of them are kept."""
    inp = wl.make_chain(5, B=8, V=30000, seed=wl.SEED_BASE + 501)
    rng = np.random.default_rng(5)
    t = np.round(rng.normal(0, 2, (8, 9, 30000))).astype(np.float32)
    d = np.round(t[:, :8] + rng.normal(0, 1, (8, 8, 30000))).astype(np.float32)
    check_chain(_rebuild(inp, t, d, 50))


def test_topk_constant_and_masked_rows():
    """Rows that are constant (top-k = the k lowest ids) and rows masked to
    -inf outside a few hundred tokens."""
    inp = wl.make_chain(5, B=6, V=16384 * 3 + 512, seed=wl.SEED_BASE + 502)
    V = inp["V"]
    rng = np.random.default_rng(6)
    t = rng.normal(0, 3, (6, 9, V)).astype(np.float32)
    t[0] = 1.5                      # constant target rows
    t[1, :, 300:] = -np.inf         # masked rows: 300 live tokens
    t[2, :, :40] = 9.0              # fewer distinct maxima than k
    d = t[:, :8] + rng.normal(0, 1, (6, 8, V)).astype(np.float32)
    d[0] = 1.5
    check_chain(_rebuild(inp, t, d, 50))


def test_topk_no_filter_when_k_reaches_v():
    inp = wl.make_chain(5, B=6, V=60, seed=wl.SEED_BASE + 503)
    check_chain(_with_topk(inp, 60))


def test_topk_mixed_batch():
    """Top-k, plain sampled and greedy requests in one call."""
    inp = wl.make_chain(5, B=24, V=40000, seed=wl.SEED_BASE + 504)
    inp["top_k"] = inp["top_k"].copy()
    inp["temperature"] = inp["temperature"].copy()
    inp["top_k"][1::3] = 0
    inp["temperature"][2::3] = 0.0
    rng = np.random.default_rng(11)
    dv = wl.bf16_bits_to_f32(inp["draft"])
    for b in range(2, 24, 3):
        for i in range(inp["K"]):
            inp["tokens"][b, i] = int(np.argmax(dv[b, i].astype(np.float64)))
    check_chain(inp)


def test_topk_fp32_and_unaligned():
    """fp32 logits (rows read where they are) and a bf16 vocabulary that is
    not a multiple of eight (no bulk copies)."""
    rng = np.random.default_rng(12)
    for V, dt in ((20000, "fp32"), (20001, "bf16")):
        inp = wl.make_chain(5, B=6, V=V, seed=wl.SEED_BASE + 505)
        inp["dtype"] = dt
        t = rng.normal(0, 4, (6, 9, V)).astype(np.float32)
        d = t[:, :8] + rng.normal(0, 2, (6, 8, V)).astype(np.float32)
        check_chain(_rebuild(inp, t, d, 50))


def test_topk_above_host_bound_is_an_argument_error():
    """A request whose top_k exceeds the call's max_top_k fails alone."""
    import speculative_decoding_verification_63_gb300 as sv
    from gpu_util import dev
    import torch
    inp = wl.make_chain(5, B=4, V=5000, seed=wl.SEED_BASE + 506)
    tk = np.array([50, 60, 50, 60], dtype=np.int32)
    out = sv.verify_chain(dev(inp["target"]), dev(inp["draft"]), dev(inp["tokens"]),
                          dev(inp["temperature"]), dev(inp["uniforms"]),
                          num_drafts=dev(inp["num_drafts"]), top_k=dev(tk), max_top_k=55)
    torch.cuda.synchronize()
    st, flags = sv.sv_get_error(sv.workspace(1, "cuda", "chain"))
    assert flags & sv.SV_DERR_ARG
    n = out["out_len"].cpu().numpy()
    assert list(n[[1, 3]]) == [0, 0]
    assert np.all(n[[0, 2]] > 0)


def test_topk_negative_and_narrow_rows():
    """Rows whose logits are all negative (the row bound comes from the
    coarse bins below zero) and rows packed into a narrow band far from zero
    (many ties after bf16 rounding: the lists overflow and are cut exactly)."""
    inp = wl.make_chain(5, B=6, V=40000, seed=wl.SEED_BASE + 507)
    V = inp["V"]
    rng = np.random.default_rng(13)
    t = rng.normal(0, 3, (6, 9, V)).astype(np.float32)
    t[0] = -30.0 + rng.normal(0, 5, (9, V)).astype(np.float32)      # all negative
    t[1] = -1e4 + rng.normal(0, 50, (9, V)).astype(np.float32)       # far below zero
    t[2] = 100.0 + rng.normal(0, 0.05, (9, V)).astype(np.float32)    # narrow band
    t[3] = 0.0 + rng.normal(0, 1e-3, (9, V)).astype(np.float32)      # around zero
    d = t[:, :8] + rng.normal(0, 0.5, (6, 8, V)).astype(np.float32)
    check_chain(_rebuild(inp, t, d, 50))


@pytest.mark.parametrize("V,dt,K", [(262144, "bf16", 2), (600000, "bf16", 1), (131072, "fp32", 2)])
def test_topk_large_vocab_folded_groups(V, dt, K):
    """Vocabularies whose group maxima do not fit one map at 16 tokens per
    group (groups of 32 or 64 tokens, re-read in 16-token pieces), with a
    constant row (the k lowest ids) and rows of integer logits (ties at the
    k-th value spread over many groups)."""
    rng = np.random.default_rng(V)
    B = 3
    inp = wl.make_chain(5, B=B, K=K, V=V, seed=wl.SEED_BASE + 508)
    inp["dtype"] = dt
    t = rng.normal(0, 4, (B, K + 1, V)).astype(np.float32)
    t[1] = 2.0
    t[2] = np.round(rng.normal(0, 2, (K + 1, V))).astype(np.float32)
    d = t[:, :K] + rng.normal(0, 2, (B, K, V)).astype(np.float32)
    d[1] = 2.0
    d[2] = np.round(d[2])
    check_chain(_rebuild(inp, t, d, 50))
