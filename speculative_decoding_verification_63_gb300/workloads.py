"""Seeded synthetic inputs for the speculative-sampling verification step.

This module only *generates inputs*: target/draft logits, draft tokens,
trees and uniforms.  It holds none of the verification arithmetic (no
softmax, no acceptance test, no residual, no inverse CDF), so both the CUDA
path and the CPU oracle can be fed from it without sharing method code.

Draft tokens are drawn from the draft distribution q = softmax(d / T) with
the Gumbel-max construction (x = argmax_j d_j / T + G_j with G_j standard
Gumbel noise), which samples exactly from q without normalising it; with
top-k filtering the argmax runs over the k entries that come first in the
order (logit descending, id ascending).  Greedy requests propose argmax d.

Uniforms are 24 random bits scaled by 2^-24, so every value is exact in fp32
and fp64 and lies in [0, 1).

Workload shapes (logits generated in fp32, then rounded to bf16 where the
workload is bf16; seeds are 63000 + workload number unless given):
  1  toy chain        B=4,   K=4, V=5,      fp32, target ~ N(0, 2^2),
                      draft = target + N(0, 0.7^2), T = 1
  2  small chain      B=1,   K=4, V=32000,  bf16, target ~ N(0, 3^2) with
                      5 random ids per row raised by +8, draft = target +
                      N(0, 1), T = 0.8
  3  headline chain   B=64,  K=6, V=128256, bf16, target ~ N(0, 3^2) -
                      1.1 ln(id + 1) (ids read as Zipf ranks), draft =
                      target + N(0, 1.5^2); even requests greedy (T = 0,
                      drafts = argmax q), odd requests T = 1
  4  token tree       B=16,  N=32 nodes (root included), depth <= 5,
                      branching <= 3, V=32000 bf16; per-node target logits
                      as in 2, per-parent draft logits = target(parent) +
                      N(0, 1); children drawn i.i.d. from the parent's q;
                      T = 0.8
  5  top-k chain      B=256, K=8, V=152064, bf16, target ~ N(0, 4^2), draft
                      = target + N(0, 2^2), T = 0.7, top-k = 50 on p and q
"""
from __future__ import annotations

import numpy as np

SEED_BASE = 63000

CHAIN_SHAPES = {
    1: dict(B=4, K=4, V=5, dtype="fp32"),
    2: dict(B=1, K=4, V=32000, dtype="bf16"),
    3: dict(B=64, K=6, V=128256, dtype="bf16"),
    5: dict(B=256, K=8, V=152064, dtype="bf16"),
}
TREE_SHAPE = dict(B=16, N=32, V=32000, max_depth=5, max_branch=3, dtype="bf16")


# ----------------------------------------------------------------- helpers

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); returns
    the uint16 bit patterns.  Inputs are finite."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    return ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 values."""
    return (h.astype(np.uint32) << np.uint32(16)).view(np.float32)


def uniforms(rng: np.random.Generator, shape) -> np.ndarray:
    """U[0,1) values with 24 random bits each (exact in fp32 and fp64)."""
    bits = rng.integers(0, 1 << 24, size=shape, dtype=np.int64)
    return (bits.astype(np.float64) * 2.0 ** -24).astype(np.float32)


def _gumbel(rng: np.random.Generator, shape, dtype=np.float64) -> np.ndarray:
    u = rng.random(size=shape, dtype=dtype)
    tiny = np.finfo(dtype).tiny
    return -np.log(-np.log(np.clip(u, tiny, 1.0 - np.finfo(dtype).eps)))


def _values(logits: np.ndarray, dtype: str) -> np.ndarray:
    """The logits as the kernel will see them (after bf16 rounding)."""
    if dtype == "bf16":
        return bf16_bits_to_f32(to_bf16_bits(logits))
    return logits.astype(np.float32)


def _topk_ids(row: np.ndarray, k: int) -> np.ndarray:
    """Ids of the k entries first in the order (value descending, id
    ascending) -- the draft side's own filter."""
    order = np.argsort(-row.astype(np.float64), kind="stable")
    return order[:k]


def draw_draft(rng: np.random.Generator, d_row: np.ndarray, T: float,
               top_k: int = 0, gumbel_dtype=np.float64) -> int:
    """One draft token from the draft row (Gumbel-max; argmax for T = 0)."""
    d = d_row.astype(np.float64)
    if T == 0.0:
        return int(np.argmax(d))
    V = d.shape[0]
    if 0 < top_k < V:
        ids = _topk_ids(d, top_k)
        g = d[ids] / T + _gumbel(rng, ids.shape[0])
        return int(ids[int(np.argmax(g))])
    g = d / T + _gumbel(rng, V, gumbel_dtype).astype(np.float64)
    return int(np.argmax(g))


def _pack(logits: np.ndarray, dtype: str) -> np.ndarray:
    return to_bf16_bits(logits) if dtype == "bf16" else logits.astype(np.float32)


# ------------------------------------------------------------------- chain

def _chain_target_logits(rng, cfg: int, B: int, R: int, V: int) -> np.ndarray:
    if cfg == 1:
        return rng.normal(0.0, 2.0, size=(B, R, V)).astype(np.float32)
    if cfg == 2:
        t = rng.normal(0.0, 3.0, size=(B, R, V)).astype(np.float32)
        for b in range(B):
            for r in range(R):
                ids = rng.choice(V, size=min(5, V), replace=False)
                t[b, r, ids] += 8.0
        return t
    if cfg == 3:
        t = rng.normal(0.0, 3.0, size=(B, R, V)).astype(np.float32)
        t -= (1.1 * np.log(np.arange(V, dtype=np.float64) + 1.0)).astype(np.float32)
        return t
    if cfg == 5:
        return rng.normal(0.0, 4.0, size=(B, R, V)).astype(np.float32)
    raise ValueError(f"no chain workload {cfg}")


_DRAFT_SIGMA = {1: 0.7, 2: 1.0, 3: 1.5, 5: 2.0}


def make_chain(cfg: int, seed: int | None = None, B: int | None = None,
               K: int | None = None, V: int | None = None,
               num_drafts: np.ndarray | None = None,
               greedy: str | None = None) -> dict:
    """Seeded inputs for chain workload `cfg` (1, 2, 3 or 5).

    B, K, V override the workload's sizes (parity tests use reduced sizes
    with the same value distributions).  `greedy` overrides the temperature
    mix: "all", "none" or "half" (even requests greedy).  `num_drafts`
    gives ragged chains (drafts beyond num_drafts[b] are padding).

    Returns a dict of numpy arrays: target [B][K+1][V] and draft [B][K][V]
    (uint16 bf16 bit patterns, or float32), tokens [B][K] int32,
    num_drafts [B] int32, temperature [B] float32, top_k [B] int32,
    uniforms [B][K+1] float32, plus dtype / sizes.
    """
    shape = dict(CHAIN_SHAPES[cfg])
    B = shape["B"] if B is None else B
    K = shape["K"] if K is None else K
    V = shape["V"] if V is None else V
    dtype = shape["dtype"]
    rng = np.random.default_rng(SEED_BASE + cfg if seed is None else seed)

    t_logits = _chain_target_logits(rng, cfg, B, K + 1, V)
    d_logits = (t_logits[:, :K, :] +
                rng.normal(0.0, _DRAFT_SIGMA[cfg], size=(B, K, V)).astype(np.float32))

    temp = np.full(B, {1: 1.0, 2: 0.8, 3: 1.0, 5: 0.7}[cfg], dtype=np.float32)
    mix = greedy if greedy is not None else ("half" if cfg == 3 else "none")
    if mix == "half":
        temp[0::2] = 0.0
    elif mix == "all":
        temp[:] = 0.0
    top_k = np.full(B, 50 if cfg == 5 else 0, dtype=np.int32)
    nd = (np.full(B, K, dtype=np.int32) if num_drafts is None
          else np.asarray(num_drafts, dtype=np.int32))

    d_vals = _values(d_logits, dtype)
    gdt = np.float32 if V > 50000 else np.float64
    tokens = np.zeros((B, K), dtype=np.int32)
    for b in range(B):
        for i in range(K):
            tokens[b, i] = draw_draft(rng, d_vals[b, i], float(temp[b]),
                                      int(top_k[b]), gdt)
    u = uniforms(rng, (B, K + 1))
    return dict(target=_pack(t_logits, dtype), draft=_pack(d_logits, dtype),
                tokens=tokens, num_drafts=nd, temperature=temp, top_k=top_k,
                uniforms=u, dtype=dtype, B=B, K=K, V=V)


# -------------------------------------------------------------------- tree

def random_tree_shape(rng: np.random.Generator, n_nodes: int, max_depth: int,
                      max_branch: int) -> np.ndarray:
    """Parent array of a random rooted tree with n_nodes nodes (root
    included), depth <= max_depth below the root and at most max_branch
    children per node, relabelled in depth-first order (children in order of
    creation), so parent[n] < n and parent[0] = -1."""
    par = [-1]
    depth = [0]
    kids: list[list[int]] = [[]]
    while len(par) < n_nodes:
        open_nodes = [n for n in range(len(par))
                      if depth[n] < max_depth and len(kids[n]) < max_branch]
        if not open_nodes:
            break
        u = open_nodes[int(rng.integers(len(open_nodes)))]
        par.append(u)
        depth.append(depth[u] + 1)
        kids.append([])
        kids[u].append(len(par) - 1)
    order: list[int] = []
    stack = [0]
    while stack:
        n = stack.pop()
        order.append(n)
        stack.extend(reversed(kids[n]))
    new_id = {old: i for i, old in enumerate(order)}
    out = np.full(len(order), -1, dtype=np.int32)
    for old in order[1:]:
        out[new_id[old]] = new_id[par[old]]
    return out


def make_tree(seed: int | None = None, B: int | None = None,
              N: int | None = None, V: int | None = None,
              max_depth: int | None = None, max_branch: int | None = None,
              temperature: float = 0.8, greedy_hint: float = 0.0,
              dtype: str | None = None, nodes_min: int | None = None,
              replace: bool = True) -> dict:
    """Seeded inputs for the token-tree workload (4).

    Each request gets a random tree (see random_tree_shape) with between
    nodes_min and N nodes (default exactly N).  Target row n is the target
    distribution after the path root..n; draft row m is the draft
    distribution at node m, used by the children of m (q_row[n] =
    parent[n]).  Children tokens are drawn i.i.d. from the parent's draft
    distribution: i.i.d. (replace=True), or without replacement among the
    children of one node (replace=False: each child is drawn from the draft
    distribution with its earlier siblings' tokens excluded).  With
    greedy_hint > 0 (greedy trees), the first child of a node takes the
    argmax of the node's target row with that probability, so greedy walks
    go deep.
    """
    sh = TREE_SHAPE
    B = sh["B"] if B is None else B
    N = sh["N"] if N is None else N
    V = sh["V"] if V is None else V
    max_depth = sh["max_depth"] if max_depth is None else max_depth
    max_branch = sh["max_branch"] if max_branch is None else max_branch
    dtype = sh["dtype"] if dtype is None else dtype
    rng = np.random.default_rng(SEED_BASE + 4 if seed is None else seed)

    t_logits = rng.normal(0.0, 3.0, size=(B, N, V)).astype(np.float32)
    for b in range(B):
        for n in range(N):
            ids = rng.choice(V, size=min(5, V), replace=False)
            t_logits[b, n, ids] += 8.0
    d_logits = t_logits + rng.normal(0.0, 1.0, size=(B, N, V)).astype(np.float32)
    t_vals = _values(t_logits, dtype)
    d_vals = _values(d_logits, dtype)

    parent = np.full((B, N), -1, dtype=np.int32)
    q_row = np.zeros((B, N), dtype=np.int32)
    tokens = np.zeros((B, N), dtype=np.int32)
    num_nodes = np.zeros(B, dtype=np.int32)
    temp = np.full(B, temperature, dtype=np.float32)
    lo = N if nodes_min is None else nodes_min
    for b in range(B):
        n_b = int(rng.integers(lo, N + 1))
        par = random_tree_shape(rng, n_b, max_depth, max_branch)
        n_b = par.shape[0]
        num_nodes[b] = n_b
        parent[b, :n_b] = par
        q_row[b, 1:n_b] = par[1:]
        first_child_seen = set()
        used: dict[int, set] = {}
        for n in range(1, n_b):
            u = int(par[n])
            if (greedy_hint > 0.0 and u not in first_child_seen
                    and rng.random() < greedy_hint):
                tokens[b, n] = int(np.argmax(t_vals[b, u].astype(np.float64)))
            else:
                row = d_vals[b, u]
                if not replace and used.get(u):
                    row = row.astype(np.float64)
                    row[sorted(used[u])] = -np.inf
                tokens[b, n] = draw_draft(rng, row, float(temperature))
            first_child_seen.add(u)
            used.setdefault(u, set()).add(int(tokens[b, n]))
    u_acc = uniforms(rng, (B, N))
    u_smp = uniforms(rng, (B,))
    return dict(target=_pack(t_logits, dtype), draft=_pack(d_logits, dtype),
                node_tokens=tokens, parent=parent, q_row=q_row,
                num_nodes=num_nodes, temperature=temp,
                top_k=np.zeros(B, dtype=np.int32), u_accept=u_acc,
                u_sample=u_smp, dtype=dtype, B=B, N=N, M=N, V=V,
                max_depth=max_depth, mode="mss" if replace else "noreplace")


def chain_algorithmic_bytes(inp: dict) -> int:
    """Logit bytes the step must read once: target rows 0..nd_b of every
    request and, for sampled requests (T > 0), draft rows 0..nd_b-1."""
    es = 2 if inp["dtype"] == "bf16" else 4
    rows = 0
    for b in range(inp["B"]):
        nd = int(inp["num_drafts"][b])
        rows += nd + 1
        if inp["temperature"][b] > 0:
            rows += nd
    return rows * inp["V"] * es


def tree_algorithmic_bytes(inp: dict) -> int:
    """Every node's target row plus every draft row some node refers to."""
    es = 2 if inp["dtype"] == "bf16" else 4
    rows = 0
    for b in range(inp["B"]):
        n_b = int(inp["num_nodes"][b])
        rows += n_b + len(set(int(r) for r in inp["q_row"][b, 1:n_b]))
    return rows * inp["V"] * es
