"""Tree verification with the other two stochastic rules on the GPU against
the fp64 oracle: multi-step speculative sampling for children drawn without
replacement, and naive sampling (CMU 15-779 Lecture 17 notes, sec. 4.5 and
sec. 10 exercises 6-7)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_63_gb300 as sv
from speculative_decoding_verification_63_gb300 import workloads as wl

from gpu_util import check_tree, dev
from oracle_pins import _tree_inputs, golden, logits_of

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["noreplace", "naive"])
def test_tree_mode_workload_full_size(mode):
    """B=16 trees of 32 nodes, depth <= 5, branching <= 3, V=32000 bf16;
    children drawn without replacement for the without-replacement rule."""
    inp = wl.make_tree(replace=mode != "noreplace")
    st, got, ref = check_tree(inp, mode=mode)
    assert got["out_len"].min() >= 1


@pytest.mark.parametrize("mode", ["noreplace", "naive"])
def test_tree_mode_small_vocab(mode):
    """V=6 fp32: most siblings get rejected, removals change q_j a lot and
    naive draws land off the tree often."""
    inp = wl.make_tree(B=256, N=12, V=6, max_depth=4, max_branch=3, seed=52, dtype="fp32",
                       replace=False)
    check_tree(inp, mode=mode)


def test_noreplace_rule_with_repeated_sibling_tokens():
    """Children drawn with replacement (repeats) under the without-
    replacement rule: a repeated token has q_j = 0 and the removal counts
    each token once."""
    inp = wl.make_tree(B=256, N=12, V=6, max_depth=4, max_branch=3, seed=53, dtype="fp32")
    check_tree(inp, mode="noreplace")


@pytest.mark.parametrize("mode", ["noreplace", "naive"])
def test_tree_mode_ragged_sizes(mode):
    inp = wl.make_tree(B=24, N=40, V=3000, nodes_min=1, seed=54, replace=mode != "noreplace")
    check_tree(inp, mode=mode)


def test_noreplace_thresholds_on_gpu():
    """The hand-derived case of the oracle pin: p = (.2, .5, .3),
    q = (.5, .25, .25), children propose tokens 0 then 2; after token 0 is
    rejected, token 2 passes for u < 1/3 without replacement (u < 2/3 with)."""
    p, q = [0.2, 0.5, 0.3], [0.5, 0.25, 0.25]
    cases = [((0.39, 0.9), 1, 1), ((0.41, 0.30), 2, 2), ((0.9, 0.34), 2, 0),
             ((0.9, 0.66), 2, 0), ((0.9, 0.68), 0, 0)]
    n = len(cases)
    t = np.zeros((n, 3, 3), np.float32)
    t[:, 0] = logits_of(p)
    d = np.broadcast_to(logits_of(q)[None, None], (n, 1, 3)).copy()
    tok = np.tile(np.array([0, 0, 2], np.int32), (n, 1))
    par = np.tile(np.array([-1, 0, 0], np.int32), (n, 1))
    qr = np.zeros((n, 3), np.int32)
    ua = np.array([[0.0, a, b] for (a, b), _, _ in cases], np.float32)
    us = np.full(n, 0.5, np.float32)
    for mode, col in (("mss", 1), ("noreplace", 2)):
        out = sv.verify_tree(dev(t), dev(d), dev(tok), dev(par), dev(qr),
                             dev(np.ones(n, np.float32)), dev(ua), dev(us), max_depth=1,
                             mode=mode)
        torch.cuda.synchronize()
        acc = out["accept_len"].cpu().numpy()
        nodes = np.where(acc == 1, out["accepted_nodes"].cpu().numpy()[:, 0], 0)
        assert nodes.tolist() == [c[col] for c in cases], (mode, nodes)
        ref = oracle.verify_tree(t, d, tok, par, qr, np.ones(n), ua, us, max_depth=1, mode=mode)
        assert np.array_equal(out["out_tokens"].cpu().numpy(), ref["out_tokens"])


def test_naive_examples_on_gpu():
    """Slides example and exercise 6: naive sampling accepts for exactly half
    of an even grid of root uniforms (p uniform on 4 tokens, two children)."""
    G = 64
    for key in ("slides_example", "exercise6"):
        g = golden("l17_exercises.json")[key]
        kids = [g["draft1"], g["draft2"]]
        t, d, tok, par, qr = _tree_inputs(g["p"], [g["q1"], g["q2"]], kids, 4)
        rep = lambda a: np.repeat(a, G, axis=0)
        ua = np.zeros((G, 3), np.float32)
        ua[:, 0] = (np.arange(G) + 0.5) / G
        ua[:, 1:] = 0.3
        out = sv.verify_tree(dev(rep(t)), None, dev(rep(tok)), dev(rep(par)), dev(rep(qr)),
                             dev(np.ones(G, np.float32)), dev(ua),
                             dev(np.full(G, 0.5, np.float32)), max_depth=1, mode="naive")
        torch.cuda.synchronize()
        x = np.arange(G) * 4 // G
        acc = out["accept_len"].cpu().numpy()
        assert np.array_equal(acc, np.isin(x, kids).astype(np.int32)), key
        assert np.array_equal(out["out_tokens"].cpu().numpy()[:, 0], x)
        assert acc.mean() == (g.get("naive_accept_this_draw") or g.get("naive_accept"))


def test_modes_agree_when_greedy_on_gpu():
    inp = wl.make_tree(B=16, temperature=0.0, greedy_hint=0.8, seed=55)
    outs = []
    for mode in ("mss", "noreplace", "naive"):
        st, got, ref = check_tree(inp, mode=mode)
        outs.append(got["out_tokens"])
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
