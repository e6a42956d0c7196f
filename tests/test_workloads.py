"""The seeded input generators: shapes, determinism, value recipes, exact
uniforms, bf16 rounding and tree invariants (CPU)."""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_63_gb300 import workloads as wl


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).normal(0, 5, 100_000).astype(np.float32)
    ours = wl.to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = wl.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(ours.view(np.int16)).view(torch.bfloat16)
                          .float().numpy())


def test_uniforms_exact_and_in_range():
    u = wl.uniforms(np.random.default_rng(1), 100_000)
    assert u.dtype == np.float32 and u.min() >= 0.0 and u.max() < 1.0
    assert np.array_equal(u.astype(np.float64) * 2 ** 24,
                          np.round(u.astype(np.float64) * 2 ** 24))


def test_chain_shapes_and_determinism():
    a = wl.make_chain(2)
    b = wl.make_chain(2)
    for k in ("target", "draft", "tokens", "uniforms"):
        assert np.array_equal(a[k], b[k])
    assert a["target"].shape == (1, 5, 32000) and a["target"].dtype == np.uint16
    assert a["draft"].shape == (1, 4, 32000)
    assert a["tokens"].shape == (1, 4) and a["uniforms"].shape == (1, 5)
    c = wl.make_chain(2, seed=5)
    assert not np.array_equal(a["target"], c["target"])
    t1 = wl.make_chain(1)
    assert t1["target"].dtype == np.float32 and t1["target"].shape == (4, 5, 5)


def test_headline_recipe_and_bytes():
    inp = wl.make_chain(3, B=4, V=128256)
    assert list(inp["temperature"]) == [0.0, 1.0, 0.0, 1.0]
    # greedy drafts are argmax of the draft row
    d = wl.bf16_bits_to_f32(inp["draft"][0])
    assert np.array_equal(inp["tokens"][0], np.argmax(d, axis=1))
    # the Zipf term makes low ids likelier: mean logit falls with ln(id+1)
    t = wl.bf16_bits_to_f32(inp["target"]).astype(np.float64)
    assert t[..., :100].mean() > t[..., -1000:].mean() + 8
    full = dict(B=64, V=128256, dtype="bf16", num_drafts=np.full(64, 6),
                temperature=np.tile([0.0, 1.0], 32).astype(np.float32))
    assert wl.chain_algorithmic_bytes(full) == 640 * 128256 * 2 == 164_167_680


def test_topk_drafts_come_from_the_filtered_draft():
    inp = wl.make_chain(5, B=3, K=2, V=2000)
    for b in range(3):
        for i in range(2):
            row = wl.bf16_bits_to_f32(inp["draft"][b, i]).astype(np.float64)
            keep = sorted(range(2000), key=lambda j: (-row[j], j))[:50]
            assert inp["tokens"][b, i] in keep


@pytest.mark.parametrize("seed", range(5))
def test_tree_shape_invariants(seed):
    rng = np.random.default_rng(seed)
    par = wl.random_tree_shape(rng, 32, 5, 3)
    assert par.shape == (32,) and par[0] == -1
    depth = np.zeros(32, int)
    kids = np.zeros(32, int)
    for n in range(1, 32):
        assert 0 <= par[n] < n
        depth[n] = depth[par[n]] + 1
        kids[par[n]] += 1
    assert depth.max() <= 5 and kids.max() <= 3
    # depth-first order: every subtree is a contiguous index range
    for n in range(32):
        sub = [m for m in range(32) if _is_desc(par, m, n)]
        assert sub == list(range(n, n + len(sub)))


def _is_desc(par, m, n):
    while m > n:
        m = par[m]
    return m == n


def test_tree_workload():
    inp = wl.make_tree(B=3)
    assert inp["target"].shape == (3, 32, 32000)
    assert np.all(inp["num_nodes"] == 32)
    for b in range(3):
        assert np.array_equal(inp["q_row"][b, 1:], inp["parent"][b, 1:])
    assert wl.tree_algorithmic_bytes(inp) > 3 * 32 * 64000
