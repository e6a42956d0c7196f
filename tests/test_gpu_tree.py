"""Token-tree verification on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_63_gb300 as sv
from speculative_decoding_verification_63_gb300 import workloads as wl

from gpu_util import check_tree, compare, dev, run_tree
from oracle_pins import golden, logits_of

pytestmark = pytest.mark.gpu


def test_tree_workload_full_size():
    """B=16 trees of 32 nodes, depth <= 5, branching <= 3, V=32000 bf16, MSS."""
    st, got, ref = check_tree(wl.make_tree())
    assert got["out_len"].min() >= 1


def test_tree_odd_batch():
    check_tree(wl.make_tree(B=5, seed=46))


def test_tree_greedy_deep_walks():
    inp = wl.make_tree(B=16, temperature=0.0, greedy_hint=0.8, seed=41)
    st, got, ref = check_tree(inp)
    assert ref["accept_len"].max() >= 2


def test_tree_small_vocab_many_rejections():
    """V=6: siblings often collide and residual updates chain up."""
    inp = wl.make_tree(B=256, N=12, V=6, max_depth=4, max_branch=3, seed=42, dtype="fp32")
    check_tree(inp)


def test_tree_ragged_sizes():
    inp = wl.make_tree(B=24, N=40, V=3000, nodes_min=1, seed=43)
    check_tree(inp)


def test_path_tree_equals_chain_on_gpu():
    inp = wl.make_chain(2, B=8, V=5000, seed=44)
    B, K, V = 8, inp["K"], 5000
    par = np.tile(np.arange(-1, K, dtype=np.int32), (B, 1))
    ntok = np.concatenate([np.zeros((B, 1), np.int32), inp["tokens"]], 1)
    ua = np.concatenate([np.zeros((B, 1), np.float32), inp["uniforms"][:, :K]], 1)
    draft = np.concatenate([inp["draft"], inp["draft"][:, :1]], 1)  # M = K + 1 rows
    out = sv.verify_tree(dev(inp["target"]), dev(draft), dev(ntok), dev(par),
                         dev(np.maximum(par, 0)), dev(inp["temperature"]), dev(ua),
                         dev(np.ascontiguousarray(inp["uniforms"][:, K])), max_depth=K)
    ch = sv.verify_chain(dev(inp["target"]), dev(inp["draft"]), dev(inp["tokens"]),
                         dev(inp["temperature"]), dev(inp["uniforms"]))
    torch.cuda.synchronize()
    assert np.array_equal(out["out_tokens"].cpu().numpy(), ch["out_tokens"].cpu().numpy())


def test_tree_ex5_bookkeeping_on_gpu():
    g = golden("l17_ex5_tree.json")
    par = np.array([g["parent"]], np.int32)
    N, V = par.shape[1], 8
    tok = np.arange(N, dtype=np.int32)[None]
    t = np.zeros((1, N, V), np.float32)
    for node, nxt in [(0, 1), (1, 2), (2, 4), (4, 5), (5, 0)]:
        t[0, node, nxt] = 3.0
    d = np.zeros((1, N, V), np.float32)
    out = sv.verify_tree(dev(t), dev(d), dev(tok), dev(par), dev(np.maximum(par, 0)),
                         dev(np.zeros(1, np.float32)), dev(np.zeros((1, N), np.float32)),
                         dev(np.array([0.5], np.float32)), max_depth=4)
    torch.cuda.synchronize()
    assert out["accepted_nodes"].cpu().numpy()[0].tolist() == [1, 2, 4, 5]
    assert out["out_tokens"].cpu().numpy()[0].tolist() == [1, 2, 4, 5, 0]


def test_tree_slides_example_on_gpu():
    s = golden("l17_exercises.json")["slides_example"]
    t = np.zeros((3, 3, 4), np.float32)
    t[:, 0] = logits_of(s["p"])
    d = np.stack([logits_of(s["q1"]), logits_of(s["q2"])])[None].repeat(3, 0)
    tok = np.array([[0, s["draft1"], s["draft2"]]] * 3, np.int32)
    par = np.array([[-1, 0, 0]] * 3, np.int32)
    qr = np.array([[0, 0, 1]] * 3, np.int32)
    ua = np.array([[0, 0.2499, 0.9], [0, 0.2501, 0.9], [0, 0.999, 0.999]], np.float32)
    out = sv.verify_tree(dev(t), dev(d), dev(tok), dev(par), dev(qr),
                         dev(np.ones(3, np.float32)), dev(ua),
                         dev(np.full(3, 0.5, np.float32)), max_depth=1)
    torch.cuda.synchronize()
    assert out["accepted_nodes"].cpu().numpy()[:, 0].tolist() == [1, 2, 2]


def test_tree_errors():
    inp = wl.make_tree(B=4, N=16, V=500, seed=45)
    inp["parent"][1, 5] = 7          # parent after the child: not depth-first
    inp["node_tokens"][2, 3] = 500   # token out of range
    ws = sv.workspace(sv.sv_tree_workspace_bytes(4, 16, 16, 500, sv.SV_BF16), "cuda", "terr")
    got = run_tree(inp, ws=ws)
    st, flags = sv.sv_get_error(ws)
    assert st == sv.SV_EDATA and flags & sv.SV_DERR_TREE and flags & sv.SV_DERR_TOKEN
    ref = oracle.verify_tree_inputs(inp)
    assert list(ref["status"][1:3]) == [oracle.ETREE, oracle.ETOKEN]
    assert list(got["out_len"][1:3]) == [0, 0]
    sv.sv_workspace_init(ws)
    compare(got, ref, 16, check_probs=False)
