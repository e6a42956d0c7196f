"""Tree-attention mask and depth position ids on the GPU against the oracle
(CMU 15-779 Lecture 17 notes, sec. 4.3 and sec. 10 exercise 5): bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_63_gb300 as sv
from speculative_decoding_verification_63_gb300 import workloads as wl

from gpu_util import dev
from oracle_pins import golden

pytestmark = pytest.mark.gpu


def run_mask(parent, num_nodes=None, words=None, ws=None):
    out = sv.tree_mask(dev(parent), None if num_nodes is None else dev(num_nodes), words=words,
                       ws=ws)
    torch.cuda.synchronize()
    return out["mask"].cpu().numpy().view(np.uint32), out["depth"].cpu().numpy()


def random_trees(rng, B, N, reach=5):
    par = np.full((B, N), -1, np.int32)
    nn = rng.integers(1, N + 1, B).astype(np.int32)
    for b in range(B):
        for i in range(1, N):
            par[b, i] = rng.integers(max(0, i - reach), i)
    return par, nn


@pytest.mark.parametrize("N,words", [(64, 2), (33, 3), (7, 1), (1, 1)])
def test_mask_matches_oracle(N, words):
    rng = np.random.default_rng(N)
    par, nn = random_trees(rng, 300, N)
    mask, depth = run_mask(par, nn, words=words)
    ref = oracle.tree_mask(par, nn, words=words)
    assert np.all(ref["status"] == 0)
    assert np.array_equal(mask, ref["mask"])
    assert np.array_equal(depth, ref["depth"])


def test_mask_of_the_tree_workload():
    inp = wl.make_tree()
    mask, depth = run_mask(inp["parent"], inp["num_nodes"])
    ref = oracle.tree_mask(inp["parent"], inp["num_nodes"])
    assert np.array_equal(mask, ref["mask"]) and np.array_equal(depth, ref["depth"])
    assert depth.max() <= inp["max_depth"]


def test_mask_slides_example():
    g = golden("l17_tree_mask.json")
    names = g["nodes"]
    parent_name = {"machine": None, "learning": "machine", "algorithm": "learning",
                   "system": "learning", "design": "system", "translation": "machine",
                   "model": "translation"}
    par = np.array([[-1] + [0 if parent_name[x] is None else 1 + names.index(parent_name[x])
                            for x in names]], np.int32)
    mask, depth = run_mask(par)
    for i, row in enumerate(g["visible"]):
        want = {0} | {1 + names.index(x) for x in row}
        assert {j for j in range(8) if (mask[0, 1 + i, 0] >> j) & 1} == want, names[i]
    e5 = golden("l17_ex5_tree.json")
    mask, depth = run_mask(np.array([e5["parent"]], np.int32))
    assert depth[0].tolist() == e5["depth"]


def test_malformed_trees_are_reported():
    rng = np.random.default_rng(7)
    par, nn = random_trees(rng, 8, 16)
    nn[:] = 16
    par[1, 5] = 5      # parent not before the child
    par[2, 0] = 0      # the root has a parent
    nn[3] = 0          # no nodes
    nn[4] = 17         # more nodes than N
    ws = sv.workspace(sv.SV_MIN_WORKSPACE_BYTES, "cuda", "maskerr")
    mask, depth = run_mask(par, nn, ws=ws)
    st, flags = sv.sv_get_error(ws)
    assert st == sv.SV_EDATA and flags & sv.SV_DERR_TREE and flags & sv.SV_DERR_ARG
    ref = oracle.tree_mask(par, nn)
    assert list(ref["status"][1:5] != 0) == [True] * 4
    assert np.array_equal(mask, ref["mask"]) and np.array_equal(depth, ref["depth"])
    assert not mask[1:5].any() and np.all(depth[1:5] == -1)
    sv.sv_workspace_init(ws)
