"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each check_* function takes an oracle library handle (oracle.load() or a
deliberately broken build, see test_oracle_mutants.py) and raises
AssertionError when the oracle disagrees with the pin.  The fixtures in
tests/golden/ carry their citations.

Which pin covers which oracle function:
  svo_row_probs   check_row_probs_softmax (library softmax), check_topk_*,
                  check_greedy_* , the worked examples
  svo_residual    check_residual_lemma1, the worked examples
  svo_icdf        check_icdf_intervals, the worked examples, Monte Carlo
  svo_icdf_window check_icdf_window_examples (dyadic weights, exact sums),
                  check_icdf_window_bruteforce (the draws at a grid of
                  uniforms), check_chain_draw_window
  svo_verify_chain  worked examples, check_grid_one_position (exact output
                  law = p), check_mc_chain (accept-length law, per-position
                  law, E[N]), check_greedy_spec_on_off, check_ragged
  svo_verify_tree check_tree_* (slides example, exercise 6, exercise 5
                  bookkeeping, branching-1 = chain, Monte Carlo law = p)
"""
from __future__ import annotations

import json
import os

import numpy as np
from scipy.special import softmax
from scipy.stats import chi2

import oracle
from oracle import enumerate as en

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def logits_of(p) -> np.ndarray:
    """fp32 logits whose softmax at T = 1 is p (zeros become -inf)."""
    p = np.asarray(p, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.log(p).astype(np.float32)


def chi2_ok(counts, probs, alpha=1e-7) -> bool:
    """Pearson chi-square goodness of fit at significance alpha."""
    counts = np.asarray(counts, dtype=np.float64)
    probs = np.asarray(probs, dtype=np.float64)
    n = counts.sum()
    m = probs > 0
    if np.any(counts[~m] > 0):
        return False
    e = n * probs[m]
    stat = ((counts[m] - e) ** 2 / e).sum()
    return stat < chi2.ppf(1.0 - alpha, max(int(m.sum()) - 1, 1))


def _chain_rows(p_rows, q_rows):
    t = np.stack([logits_of(p) for p in p_rows])[None]
    d = np.stack([logits_of(q) for q in q_rows])[None]
    return t, d


# ------------------------------------------------------------ worked examples

def check_worked_round_n02_sec9(lib):
    g = golden("n02_sec9_worked_round.json")
    p, q, K = g["p"], g["q"], g["K"]
    t, d = _chain_rows([p] * (K + 1), [q] * K)
    r = list(g["accept_uniforms"])
    r[1] = 0.999  # not printed; position 2 accepts with probability 1
    for u_final, expect in [(0.10, 1), (0.50, 1), (0.7499, 1), (0.7501, 2), (0.90, 2)]:
        out = oracle.verify_chain(t, d, [g["drafts"]], [1.0], [r + [u_final]], lib=lib)
        assert out["status"][0] == 0
        assert out["accept_len"][0] == 2 and out["out_len"][0] == g["N"]
        assert list(out["out_tokens"][0][:3]) == [0, 1, expect], (u_final, out)
        acc = np.minimum(1.0, out["p_at"][0] / out["q_at"][0])
        assert np.allclose(acc, g["accept_probabilities"], atol=1e-6)
    # the accept threshold of position 1 is p(A)/q(A) = 0.6
    for u1, n_expect in [(0.5999, 2), (0.6001, 0)]:
        out = oracle.verify_chain(t, d, [g["drafts"]], [1.0], [[u1, 0.999, 0.8, 0.1]], lib=lib)
        assert out["accept_len"][0] == n_expect
    # alpha, beta, p_r of sec. 9.1
    st, pp = oracle.row_probs(t[0, 0], 1.0, lib=lib)
    st2, qq = oracle.row_probs(d[0, 0], 1.0, lib=lib)
    w, S = oracle.residual(pp, qq, lib=lib)
    assert abs(S - g["beta"]) < 1e-7 and abs((1 - S) - g["alpha"]) < 1e-7
    assert np.allclose(w / S, g["p_r"], atol=1e-6)
    assert abs(en.expected_tokens(1 - S, K) - g["E_N"]) < 1e-6


def check_exercise2_n02(lib):
    g = golden("n02_sec14_exercise2.json")
    t, d = _chain_rows([g["p"]] * (g["K"] + 1), [g["q"]] * g["K"])
    r = list(g["accept_uniforms"])
    r[1] = 0.5
    for u_final in (0.05, 0.5, 0.95):
        out = oracle.verify_chain(t, d, [g["drafts"]], [1.0], [r + [u_final]], lib=lib)
        assert list(out["out_tokens"][0][:3]) == g["emitted"], out
    st, pp = oracle.row_probs(t[0, 0], 1.0, lib=lib)
    st, qq = oracle.row_probs(d[0, 0], 1.0, lib=lib)
    w, S = oracle.residual(pp, qq, lib=lib)
    assert abs(S - g["beta"]) < 1e-7
    assert np.allclose(w / S, g["p_r"], atol=1e-6)


# ------------------------------------------- exact law over a uniform grid

def oracle_one_position_law(lib, p, q, G: int = 256, draft_fixed=None,
                            temperature=1.0, top_k=0, p_logits=None, q_logits=None):
    """Exact-up-to-grid law of the first emitted token of a K = 1 chain:
    drafts enumerated with weight q(x) (or fixed), (u0, u1) on the midpoint
    grid of G x G cells.  Returns the law over V."""
    tl = logits_of(p) if p_logits is None else np.asarray(p_logits, np.float32)
    dl = logits_of(q) if q_logits is None else np.asarray(q_logits, np.float32)
    V = tl.shape[0]
    grid = (np.arange(G) + 0.5) / G
    u0, u1 = np.meshgrid(grid, grid, indexing="ij")
    n = G * G
    law = np.zeros(V)
    drafts = [draft_fixed] if draft_fixed is not None else range(V)
    for x in drafts:
        wx = 1.0 if draft_fixed is not None else float(q[x])
        if wx == 0.0:
            continue
        t = np.broadcast_to(np.stack([tl, tl]), (n, 2, V))
        d = np.broadcast_to(dl[None], (n, 1, V))
        u = np.stack([u0.ravel(), u1.ravel()], 1).astype(np.float32)
        out = oracle.verify_chain(t, d, np.full((n, 1), x), np.full(n, temperature), u,
                                  top_k=np.full(n, top_k), lib=lib)
        assert np.all(out["status"] == 0)
        law += wx * np.bincount(out["out_tokens"][:, 0], minlength=V)[:V] / n
    return law


def check_grid_one_position(lib):
    """[L17] sec. 10 exercise 3: p = (0.6, 0.4), q = (0.5, 0.5) -> p; and two
    random V = 5 pairs; exact up to the grid resolution ([N02] Lemma 2)."""
    g = golden("l17_exercises.json")["exercise3"]
    law = oracle_one_position_law(lib, g["p"], g["q"], G=200)
    assert np.allclose(law, g["correct_output"], atol=2.0 / 200), law
    assert not np.allclose(law, g["greedy_rule_output"], atol=0.05)
    rng = np.random.default_rng(7)
    for _ in range(2):
        p = rng.dirichlet(np.ones(5))
        q = rng.dirichlet(np.ones(5))
        law = oracle_one_position_law(lib, p, q, G=160)
        assert np.abs(law - p).max() < 5 * 2.0 / 160, (law, p)


def check_deterministic_draft_bias(lib):
    """[L17] sec. 10 exercise 7: a fixed top-1 draft under the speculative
    rule emits (0.833, 0.167) for p = (0.5, 0.5), q = (0.6, 0.4)."""
    g = golden("l17_exercises.json")["exercise7"]
    law = oracle_one_position_law(lib, g["p"], g["q"], G=240, draft_fixed=0)
    assert np.allclose(law, g["biased_output"], atol=2.0 / 240), law


# ------------------------------------------------------------ closed forms

def check_residual_lemma1(lib):
    """[N02] sec. 5.1: sum max(0, p - q) = 1 - sum min(p, q) = TV(p, q)."""
    rng = np.random.default_rng(11)
    for V in (2, 5, 1000):
        p = rng.dirichlet(np.ones(V))
        q = rng.dirichlet(np.ones(V) * 0.5)
        w, S = oracle.residual(p, q, lib=lib)
        assert np.all(w >= 0) and np.all((w > 0) <= (p > q))
        assert abs(S - (1.0 - np.minimum(p, q).sum())) < 1e-14
        assert abs(S - 0.5 * np.abs(p - q).sum()) < 1e-14


def check_icdf_intervals(lib):
    w = np.array([0.0, 2.0, 0.0, 1.0, 1.0])
    for u, t in [(0.0, 1), (0.3, 1), (0.4999, 1), (0.5, 3), (0.7, 3), (0.75, 4), (0.999, 4)]:
        tok, m = oracle.icdf(w, u, lib=lib)
        assert tok == t, (u, tok)
    tok, m = oracle.icdf(w, 0.5 + 1e-9, lib=lib)
    assert m < 1e-8  # near the boundary between ids 1 and 3
    tok, m = oracle.icdf(np.zeros(4), 0.5, lib=lib)
    assert tok == -1


def check_icdf_window_examples(lib):
    """svo_icdf_window on dyadic weights, where every sum is exact: the
    tokens whose CDF step meets [u S - r S, u S + r S]."""
    w = np.array([0.0, 2.0, 0.0, 1.0, 1.0])  # S = 4, steps at 2 (id 1), 3 (id 3), 4 (id 4)
    cases = [
        (0.5, 0.0, (3, 3, 1)),     # u S = 2 sits on the 1|3 step: the draw is 3
        (0.5, 0.01, (1, 3, 2)),    # [1.96, 2.04] meets ids 1 and 3 (id 2 has no weight)
        (0.5, 0.3, (1, 4, 3)),     # [0.8, 3.2] meets 1, 3 and 4
        (0.999, 0.01, (4, 4, 1)),  # [3.956, 4.036]: the last step only
        (0.0, 0.1, (1, 1, 1)),     # [-0.4, 0.4]: id 0 has no weight
        (0.74, 0.02, (3, 4, 2)),   # [2.88, 3.04] meets 3 and 4
    ]
    for u, r, want in cases:
        got = oracle.icdf_window(w, u, r, lib=lib)
        assert got == want, (u, r, got, want)
        if r == 0.0:
            assert got[0] == oracle.icdf(w, u, lib=lib)[0]
    assert oracle.icdf_window(np.zeros(3), 0.5, 0.1, lib=lib) == (-1, -1, -1)


def check_icdf_window_bruteforce(lib):
    """The window against the draws themselves: on random small weight
    vectors (every positive weight at least 1e-3 of the total), the
    inverse-CDF token at both ends of [u - r, u + r] and on a grid 1e-4
    apart inside it hits every token whose step meets the window, and only
    those."""
    rng = np.random.default_rng(41)
    for case in range(120):
        V = int(rng.integers(2, 10))
        w = rng.dirichlet(np.ones(V)) + 2e-2
        w[rng.random(V) < 0.3] = 0.0
        if not w.any():
            w[rng.integers(V)] = 1.0
        u = float(rng.random())
        r = float(rng.choice([0.0, 1e-3, 0.02, 0.1]))
        us = np.concatenate([[u - r, u + r], np.arange(u - r, u + r, 1e-4)])
        hit = {oracle.icdf(w, float(x), lib=lib)[0] for x in us if 0.0 <= x < 1.0}
        if u - r < 0.0:
            hit.add(oracle.icdf(w, 0.0, lib=lib)[0])
        if u + r >= 1.0:
            hit.add(int(np.nonzero(w)[0][-1]))
        lo, hi, n = oracle.icdf_window(w, u, r, lib=lib)
        assert (lo, hi) == (min(hit), max(hit)), (case, w, u, r, lo, hi, sorted(hit))
        assert n == int((w[lo:hi + 1] > 0).sum()) == len(hit), (case, n, sorted(hit))


def check_chain_draw_window(lib):
    """The chain reports the window of a near draw: [N02] sec. 9's round
    (residual (0, .75, .25, 0, 0) after position 3 rejects).  A final
    uniform 1e-8 below the 0.75 step is near and may give id 1 or 2; one at
    0.5 is not near and gives id 1 alone."""
    g = golden("n02_sec9_worked_round.json")
    p, q, K = g["p"], g["q"], g["K"]
    t, d = _chain_rows([p] * (K + 1), [q] * K)
    r = list(g["accept_uniforms"])
    r[1] = 0.999
    near = oracle.verify_chain(t, d, [g["drafts"]], [1.0], [r + [0.75 - 1e-8]], lib=lib)
    assert near["out_tokens"][0][2] == 1 and near["margin_draw"][0] < 1e-6
    assert (near["draw_lo"][0], near["draw_hi"][0]) == (1, 2)
    far = oracle.verify_chain(t, d, [g["drafts"]], [1.0], [r + [0.5]], lib=lib)
    assert (far["draw_lo"][0], far["draw_hi"][0]) == (1, 1)


def check_row_probs_softmax(lib):
    """temperature softmax = scipy.special.softmax(l / T) (a library routine)."""
    rng = np.random.default_rng(5)
    for T in (0.5, 0.8, 1.0, 2.0):
        l = rng.normal(0, 3, 257).astype(np.float32)
        st, p = oracle.row_probs(l, T, lib=lib)
        assert st == 0
        ref = softmax(l.astype(np.float64) / T)
        assert np.abs(p - ref).max() < 1e-14
    # bf16 bit patterns decode exactly
    from speculative_decoding_verification_63_gb300.workloads import (
        to_bf16_bits, bf16_bits_to_f32)
    h = to_bf16_bits(rng.normal(0, 3, 300).astype(np.float32))
    st, p = oracle.row_probs(h, 0.7, lib=lib)
    ref = softmax(bf16_bits_to_f32(h).astype(np.float64) / 0.7)
    assert np.abs(p - ref).max() < 1e-14


def check_topk_bruteforce(lib):
    """top-k keeps exactly k entries, ties at the k-th value to the lower id
    ([N02] sec. 5.4 top-k applied to both p and q)."""
    rng = np.random.default_rng(3)
    for V, k in [(12, 1), (12, 3), (12, 5), (12, 11), (12, 12), (12, 0), (40, 7)]:
        l = rng.integers(-3, 3, V).astype(np.float32)  # many ties
        st, p = oracle.row_probs(l, 0.9, k, lib=lib)
        assert st == 0
        order = sorted(range(V), key=lambda j: (-float(l[j]), j))
        keep = set(order[:k]) if 0 < k < V else set(range(V))
        ref = np.zeros(V)
        ids = sorted(keep)
        ref[ids] = softmax(l[ids].astype(np.float64) / 0.9)
        assert np.abs(p - ref).max() < 1e-14, (V, k, p, ref)


def check_greedy_chain(lib):
    """[L17] sec. 2.2, [N02] sec. 10: accept iff x_i = argmax p_i; at the
    first mismatch emit argmax p_i; all accepted -> argmax p_{K+1}; argmax
    ties go to the lowest id; uniforms and draft rows are unused."""
    V, K = 8, 4
    t = np.zeros((1, K + 1, V), np.float32)
    am = [3, 5, 0, 7, 2]
    for i, a in enumerate(am):
        t[0, i, a] = 5.0
    t[0, 2, 6] = 5.0  # tie at row 2 between ids 0 and 6 -> 0
    d = np.full((1, K, V), np.nan, np.float32)  # never read for T = 0
    for toks, n, last in [([3, 5, 0, 7], 4, 2), ([3, 5, 6, 7], 2, 0),
                          ([1, 5, 0, 7], 0, 3), ([3, 5, 0, 1], 3, 7)]:
        for u in (0.0, 0.999):
            out = oracle.verify_chain(t, d, [toks], [0.0], [[u] * (K + 1)], lib=lib)
            assert out["status"][0] == 0
            assert out["accept_len"][0] == n
            assert list(out["out_tokens"][0][:n + 1]) == toks[:n] + [last]


def check_greedy_spec_on_off(lib):
    """[S14] 'temperature=0 ... spec on and off give identical tokens';
    [L17] sec. 2.2: speculative greedy equals plain greedy token for token."""
    m = en.ToyModel(V=5, ctx=2, seed=4)
    L = 12
    ref = [0, 1]
    while len(ref) < 2 + L:
        ref.append(int(np.argmax(m.target(ref))))
    for K in (1, 2, 3, 4):
        h = [0, 1]
        while len(h) < 2 + L:
            drafts, hh = [], list(h)
            for _ in range(K):
                x = int(np.argmax(m.draft(hh)))
                drafts.append(x)
                hh.append(x)
            t = np.stack([m.p_logits[m.key(h + drafts[:i])] for i in range(K + 1)])[None]
            d = np.stack([m.q_logits[m.key(h + drafts[:i])] for i in range(K)])[None]
            out = oracle.verify_chain(t.astype(np.float32), d.astype(np.float32),
                                      [drafts], [0.0], [[0.5] * (K + 1)], lib=lib)
            h += list(out["out_tokens"][0][:out["out_len"][0]])
        assert h[:2 + L] == ref, (K, h, ref)


def check_topk1_is_greedy(lib):
    """top-k = 1 at T > 0 makes p and q one-hot: the sampled rule then
    reduces to greedy argmax equality ([N02] sec. 10)."""
    rng = np.random.default_rng(9)
    B, K, V = 64, 4, 30
    t = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    d = (t[:, :K] + rng.normal(0, 2, (B, K, V))).astype(np.float32)
    toks = np.argmax(d, axis=2).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    a = oracle.verify_chain(t, d, toks, np.full(B, 0.9), u, top_k=np.ones(B), lib=lib)
    b = oracle.verify_chain(t, d, toks, np.zeros(B), u, lib=lib)
    assert np.array_equal(a["out_tokens"], b["out_tokens"])
    assert np.array_equal(a["accept_len"], b["accept_len"])


def check_ragged(lib):
    """num_drafts[b] < K ([N02] sec. 11.3 padding): rows beyond num_drafts
    are unused; num_drafts = 0 is a plain draw from p_1."""
    rng = np.random.default_rng(12)
    B, K, V = 6, 5, 9
    t = rng.normal(0, 1, (B, K + 1, V)).astype(np.float32)
    d = (t[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    toks = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    nd = np.array([0, 1, 2, 3, 4, 5], np.int32)
    full = oracle.verify_chain(t, d, toks, np.ones(B), u, num_drafts=nd, lib=lib)
    for b in range(B):
        n = int(nd[b])
        tt = np.concatenate([t[b:b + 1, :n + 1], np.zeros((1, K - n, V), np.float32)], 1)
        tt[0, n + 1:] = np.nan  # unused rows
        dd = np.concatenate([d[b:b + 1, :n], np.full((1, K - n, V), np.nan, np.float32)], 1)
        one = oracle.verify_chain(tt, dd, toks[b:b + 1], [1.0], u[b:b + 1],
                                  num_drafts=[n], lib=lib)
        assert one["status"][0] == 0
        assert np.array_equal(one["out_tokens"], full["out_tokens"][b:b + 1])
    # nd = 0: the emitted token is the inverse-CDF draw from p_1 with u[K]
    st, p1 = oracle.row_probs(t[0, 0], 1.0, lib=lib)
    tok, _ = oracle.icdf(p1, float(u[0, K]), lib=lib)
    assert full["out_tokens"][0, 0] == tok and full["out_len"][0] == 1


def check_data_errors(lib):
    t = np.zeros((1, 3, 4), np.float32)
    d = np.zeros((1, 2, 4), np.float32)
    u = [[0.5, 0.5, 0.5]]
    assert oracle.verify_chain(t, d, [[0, 9]], [1.0], u, lib=lib)["status"][0] == oracle.ETOKEN
    t2 = t.copy()
    t2[0, 1, 2] = np.nan
    assert oracle.verify_chain(t2, d, [[0, 1]], [1.0], u, lib=lib)["status"][0] == oracle.ENONFINITE
    assert oracle.verify_chain(t2, d, [[0, 1]], [0.0], u, lib=lib)["status"][0] == oracle.ENONFINITE
    t3 = t.copy()
    t3[0, 0, :] = -np.inf
    assert oracle.verify_chain(t3, d, [[0, 1]], [1.0], u, lib=lib)["status"][0] == oracle.EMASS
    assert oracle.verify_chain(t, d, [[0, 1]], [-1.0], u, lib=lib)["status"][0] == oracle.EARG


# --------------------------------------------------------------- Monte Carlo

def check_mc_chain(lib, n=150_000, seed=21):
    """Position-specific p_i, q_i (V = 5, K = 3), drafts x_i ~ q_i: the
    accept-length law is prod(alpha)(1 - alpha) ([L17] sec. 2.5), and the
    token emitted at position i, given the round reached i, has law p_i
    ([N02] Lemma 2); positions beyond the first rejection are never used."""
    rng = np.random.default_rng(seed)
    V, K = 5, 3
    P = rng.dirichlet(np.ones(V), K + 1)
    Q = rng.dirichlet(np.ones(V), K)
    t = np.broadcast_to(np.stack([logits_of(p) for p in P])[None], (n, K + 1, V))
    d = np.broadcast_to(np.stack([logits_of(q) for q in Q])[None], (n, K, V))
    toks = np.stack([rng.choice(V, n, p=Q[i]) for i in range(K)], 1).astype(np.int32)
    u = rng.random((n, K + 1)).astype(np.float32)
    out = oracle.verify_chain(t, d, toks, np.ones(n), u, lib=lib)
    assert np.all(out["status"] == 0)
    alphas = [en.overlap(P[i], Q[i]) for i in range(K)]
    law = en.accept_length_law(alphas)
    assert chi2_ok(np.bincount(out["accept_len"], minlength=K + 1), law)
    for i in range(K + 1):
        reached = out["accept_len"] >= i
        emitted = out["out_tokens"][reached, i]
        assert chi2_ok(np.bincount(emitted, minlength=V), P[i]), i
    exact = en.chain_exact(P, Q)
    assert np.allclose(exact["accept_len_law"], law, atol=1e-12)


def check_mc_expected_tokens(lib, n=120_000, seed=22):
    """Identical rows with alpha = 0.8 ([N02] sec. 9 p, q), K = 4:
    mean tokens per round -> (1 - 0.8^5) / 0.2 = 3.36 ([L17] sec. 2.5)."""
    g = golden("n02_sec9_worked_round.json")
    rng = np.random.default_rng(seed)
    K, V = 4, 5
    t = np.broadcast_to(logits_of(g["p"])[None, None], (n, K + 1, V))
    d = np.broadcast_to(logits_of(g["q"])[None, None], (n, K, V))
    toks = rng.choice(V, (n, K), p=g["q"]).astype(np.int32)
    u = rng.random((n, K + 1)).astype(np.float32)
    out = oracle.verify_chain(t, d, toks, np.ones(n), u, lib=lib)
    E = en.expected_tokens(0.8, K)
    N = out["out_len"].astype(np.float64)
    assert abs(N.mean() - E) < 5 * N.std() / np.sqrt(n), (N.mean(), E)


def check_mc_temperature_topk(lib, n=120_000, seed=23):
    """Any decoding strategy applied to both p and q (temperature, top-k)
    keeps the output law equal to the filtered target ([N02] sec. 5.4)."""
    rng = np.random.default_rng(seed)
    V, K, T, k = 7, 2, 0.6, 4
    tl = rng.normal(0, 1.5, (K + 1, V)).astype(np.float32)
    dl = (tl[:K] + rng.normal(0, 1.0, (K, V))).astype(np.float32)

    def filt(l):
        order = sorted(range(V), key=lambda j: (-float(l[j]), j))[:k]
        p = np.zeros(V)
        p[order] = softmax(l[order].astype(np.float64) / T)
        return p

    P = [filt(tl[i]) for i in range(K + 1)]
    Q = [filt(dl[i]) for i in range(K)]
    toks = np.stack([rng.choice(V, n, p=Q[i]) for i in range(K)], 1).astype(np.int32)
    u = rng.random((n, K + 1)).astype(np.float32)
    out = oracle.verify_chain(np.broadcast_to(tl[None], (n, K + 1, V)),
                              np.broadcast_to(dl[None], (n, K, V)), toks,
                              np.full(n, T), u, top_k=np.full(n, k), lib=lib)
    assert np.all(out["status"] == 0)
    for i in range(K + 1):
        reached = out["accept_len"] >= i
        assert chi2_ok(np.bincount(out["out_tokens"][reached, i], minlength=V), P[i]), i


def check_mc_toy_sequences(lib, n=60_000, K=3, L=3, seed=24):
    """[L17] sec. 2.3 exact check, by Monte Carlo through the oracle: the
    first L tokens of repeated speculative rounds on a context-dependent toy
    model follow the autoregressive law of p ([N02] sec. 5.3)."""
    m = en.ToyModel(V=4, ctx=2, seed=6)
    rng = np.random.default_rng(seed)
    prefix = [0, 1]
    P0 = len(prefix)
    hist = np.zeros((n, P0 + L + K + 1), np.int64)
    hist[:, :P0] = prefix
    length = np.full(n, P0)

    def key(h, ln):
        r = np.arange(h.shape[0])
        return h[r, ln - 2] * m.V + h[r, ln - 1]

    while True:
        todo = np.nonzero(length < P0 + L)[0]
        if todo.size == 0:
            break
        B = todo.size
        h = hist[todo].copy()
        ln = length[todo].copy()
        t = np.zeros((B, K + 1, m.V), np.float32)
        d = np.zeros((B, K, m.V), np.float32)
        toks = np.zeros((B, K), np.int32)
        r = np.arange(B)
        for i in range(K):
            kk = key(h, ln)
            q = m.q[kk]
            x = (rng.random(B)[:, None] >= np.cumsum(q, 1)).sum(1)
            x = np.minimum(x, m.V - 1)
            t[:, i] = m.p_logits[kk]
            d[:, i] = m.q_logits[kk]
            toks[:, i] = x
            h[r, ln] = x
            ln = ln + 1
        t[:, K] = m.p_logits[key(h, ln)]
        u = rng.random((B, K + 1)).astype(np.float32)
        out = oracle.verify_chain(t, d, toks, np.ones(B), u, lib=lib)
        for j in range(K + 1):
            sel = out["out_len"] > j
            rows = todo[sel]
            hist[rows, length[rows]] = out["out_tokens"][sel, j]
            length[rows] += 1
    exact = en.autoregressive_law(m, prefix, L)
    keys = sorted(exact)
    code = np.zeros(n, np.int64)
    for j in range(L):
        code = code * m.V + hist[:, P0 + j]
    counts = np.bincount(code, minlength=m.V ** L)
    probs = np.zeros(m.V ** L)
    for k in keys:
        c = 0
        for tkn in k:
            c = c * m.V + tkn
        probs[c] = exact[k]
    assert chi2_ok(counts, probs)


# -------------------------------------------------------------------- tree

def _tree_inputs(p_root, q_rows, child_tokens, V):
    """Root with len(child_tokens) children; child j proposed by q_rows[j];
    children are leaves whose target rows are uniform."""
    n = 1 + len(child_tokens)
    t = np.zeros((1, n, V), np.float32)
    t[0, 0] = logits_of(p_root)
    d = np.stack([logits_of(q) for q in q_rows])[None]
    tok = np.array([[0] + list(child_tokens)], np.int32)
    par = np.array([[-1] + [0] * len(child_tokens)], np.int32)
    qr = np.array([[0] + list(range(len(child_tokens)))], np.int32)
    return t, d, tok, par, qr


def check_tree_slides_example(lib):
    """[L17] sec. 4.5 slides example: p uniform on 4 tokens, SSM 1 always
    proposes t1, SSM 2 (uniform) proposed t2: t1 accepted w.p. 0.25; after
    its rejection r = (0, 1/3, 1/3, 1/3) and t2 is accepted w.p. 1."""
    g = golden("l17_exercises.json")["slides_example"]
    t, d, tok, par, qr = _tree_inputs(g["p"], [g["q1"], g["q2"]],
                                      [g["draft1"], g["draft2"]], 4)
    for u1, node in [(0.2499, 1), (0.2501, 2), (0.999, 2)]:
        out = oracle.verify_tree(t, d, tok, par, qr, [1.0], [[0.0, u1, 0.999]], [0.5],
                                 max_depth=1, lib=lib)
        assert out["status"][0] == 0
        assert out["accepted_nodes"][0][0] == node, (u1, out)
        assert out["out_tokens"][0][0] == tok[0][node]


def check_tree_exercise6(lib):
    """[L17] sec. 10 exercise 6: q1 = (.5, .5, 0, 0) proposed t2: accepted
    w.p. 0.5; residual (0, 0, .5, .5); t3 from a uniform SSM then accepted
    w.p. 1 (min(1, 0.5 / 0.25))."""
    g = golden("l17_exercises.json")["exercise6"]
    t, d, tok, par, qr = _tree_inputs(g["p"], [g["q1"], g["q2"]],
                                      [g["draft1"], g["draft2"]], 4)
    for u1, node in [(0.4999, 1), (0.5001, 2), (0.999, 2)]:
        out = oracle.verify_tree(t, d, tok, par, qr, [1.0], [[0.0, u1, 0.9999]], [0.5],
                                 max_depth=1, lib=lib)
        assert out["accepted_nodes"][0][0] == node, (u1, out)
    # a third child proposing t1 after both rejections can never pass
    # (residual is zero on t1); with a third uniform child proposing t1 and
    # the first two rejected by construction, the final draw is from r
    p = np.full(4, 0.25)
    w, S = oracle.residual(p, np.array(g["q1"]), lib=lib)
    assert np.allclose(w / S, g["residual_after_first"])


def check_tree_ex5_bookkeeping(lib):
    """[L17] sec. 10 exercise 5: the merged tree r a b c d e f g in DFS
    order; a greedy walk to e returns accepted nodes a, b, d, e (the
    ancestors of e plus e: the KV entries to keep)."""
    g = golden("l17_ex5_tree.json")
    par = np.array([g["parent"]], np.int32)
    N = par.shape[1]
    V = 8
    tok = np.array([[0, 1, 2, 3, 4, 5, 6, 7]], np.int32)  # token id = node id
    t = np.zeros((1, N, V), np.float32)
    # greedy target: r -> a, a -> b, b -> d, d -> e, e -> (id 0, not a child)
    for node, nxt in [(0, 1), (1, 2), (2, 4), (4, 5), (5, 0)]:
        t[0, node, nxt] = 3.0
    d = np.zeros((1, N, V), np.float32)
    out = oracle.verify_tree(t, d, tok, par, np.maximum(par, 0), [0.0],
                             np.zeros((1, N)), [0.5], max_depth=4, lib=lib)
    assert out["status"][0] == 0
    names = g["dfs_order"]
    path = [names[i] for i in out["accepted_nodes"][0][:out["accept_len"][0]]]
    assert path == g["ancestors_of_e"][1:] + ["e"], path
    assert out["out_tokens"][0][4] == 0 and out["out_len"][0] == 5


def check_tree_branching1_is_chain(lib):
    """A path-shaped tree is a chain ([L17] sec. 7.3: MSS on a single
    child is speculative sampling)."""
    rng = np.random.default_rng(31)
    B, K, V = 40, 4, 11
    t = rng.normal(0, 1.5, (B, K + 1, V)).astype(np.float32)
    d = (t[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    toks = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    for T in (1.0, 0.0):
        ch = oracle.verify_chain(t, d, toks, np.full(B, T), u, lib=lib)
        par = np.tile(np.arange(-1, K, dtype=np.int32), (B, 1))
        ntok = np.concatenate([np.zeros((B, 1), np.int32), toks], 1)
        ua = np.concatenate([np.zeros((B, 1), np.float32), u[:, :K]], 1)
        tr = oracle.verify_tree(t, d, ntok, par, np.maximum(par, 0), np.full(B, T), ua,
                                u[:, K], max_depth=K, lib=lib)
        assert np.array_equal(ch["out_tokens"], tr["out_tokens"]), T
        assert np.array_equal(ch["accept_len"], tr["accept_len"])


def check_tree_mc_lossless(lib, n=100_000, seed=32):
    """Theorem 4.2 ([L17] sec. 4.5): with children drawn i.i.d. from their
    proposers' q, the first token MSS emits has law p_root; its accept rate
    matches the exact enumeration and is >= naive sampling (Theorem 4.3)."""
    rng = np.random.default_rng(seed)
    V = 5
    p = rng.dirichlet(np.ones(V))
    qs = [rng.dirichlet(np.ones(V)) for _ in range(3)]
    ex = en.mss_exact(p, qs)
    assert np.abs(ex["emitted"] - p).max() < 1e-12
    assert ex["accept"] >= ex["naive_accept"] - 1e-12
    N = 4
    t = np.zeros((n, N, V), np.float32)
    t[:, 0] = logits_of(p)
    d = np.broadcast_to(np.stack([logits_of(q) for q in qs])[None], (n, 3, V))
    tok = np.zeros((n, N), np.int32)
    for j in range(3):
        tok[:, j + 1] = rng.choice(V, n, p=qs[j])
    par = np.tile(np.array([-1, 0, 0, 0], np.int32), (n, 1))
    qr = np.tile(np.array([0, 0, 1, 2], np.int32), (n, 1))
    ua = rng.random((n, N)).astype(np.float32)
    us = rng.random(n).astype(np.float32)
    out = oracle.verify_tree(t, d, tok, par, qr, np.ones(n), ua, us, max_depth=1, lib=lib)
    assert np.all(out["status"] == 0)
    assert chi2_ok(np.bincount(out["out_tokens"][:, 0], minlength=V), p)
    acc = (out["accept_len"] == 1).mean()
    assert abs(acc - ex["accept"]) < 5 * np.sqrt(ex["accept"] * (1 - ex["accept"]) / n)


def check_tree_deeper_mc(lib, n=60_000, seed=33):
    """Two levels: the emitted path law factorises as p_root then p_child
    (MSS is lossless level by level)."""
    rng = np.random.default_rng(seed)
    V = 4
    # tree: 0 -> {1, 2}; 1 -> {3}; all tokens drawn from their parent's q
    P = [rng.dirichlet(np.ones(V)) for _ in range(4)]
    Q = [rng.dirichlet(np.ones(V)) for _ in range(4)]
    par = np.array([-1, 0, 0, 1], np.int32)
    t = np.broadcast_to(np.stack([logits_of(x) for x in P])[None], (n, 4, V))
    d = np.broadcast_to(np.stack([logits_of(x) for x in Q])[None], (n, 4, V))
    tok = np.zeros((n, 4), np.int32)
    for c in (1, 2, 3):
        tok[:, c] = rng.choice(V, n, p=Q[par[c]])
    out = oracle.verify_tree(t, d, tok, np.tile(par, (n, 1)),
                             np.tile(np.maximum(par, 0), (n, 1)), np.ones(n),
                             rng.random((n, 4)).astype(np.float32),
                             rng.random(n).astype(np.float32), max_depth=2, lib=lib)
    assert chi2_ok(np.bincount(out["out_tokens"][:, 0], minlength=V), P[0])
    # given that node 1 was accepted, the next token follows p_1
    sel = (out["accept_len"] >= 1) & (out["accepted_nodes"][:, 0] == 1)
    assert chi2_ok(np.bincount(out["out_tokens"][sel, 1], minlength=V), P[1])


ALL_FAST = [check_worked_round_n02_sec9, check_exercise2_n02, check_residual_lemma1,
            check_icdf_intervals, check_row_probs_softmax, check_topk_bruteforce,
            check_greedy_chain, check_greedy_spec_on_off, check_topk1_is_greedy,
            check_ragged, check_data_errors, check_tree_slides_example,
            check_tree_exercise6, check_tree_ex5_bookkeeping,
            check_tree_branching1_is_chain, check_grid_one_position,
            check_deterministic_draft_bias]
ALL_MC = [check_mc_chain, check_mc_expected_tokens, check_mc_temperature_topk,
          check_mc_toy_sequences, check_tree_mc_lossless, check_tree_deeper_mc]


# ---------------------------------------- tree: MSS without replacement, naive

def _one_level_tree(p, q, child_tokens, ua_children, us=0.5, mode="mss", lib=None):
    """Root with children proposing child_tokens, all from the one draft row q."""
    V = len(p)
    n = 1 + len(child_tokens)
    t = np.zeros((1, n, V), np.float32)
    t[0, 0] = logits_of(p)
    d = logits_of(q)[None, None]
    tok = np.array([[0] + list(child_tokens)], np.int32)
    par = np.array([[-1] + [0] * len(child_tokens)], np.int32)
    qr = np.zeros((1, n), np.int32)
    ua = np.array([[0.0] + list(ua_children)], np.float32)
    return oracle.verify_tree(t, d, tok, par, qr, [1.0], ua, [us], max_depth=1,
                              mode=mode, lib=lib)


def check_tree_noreplace_thresholds(lib):
    """[L17] sec. 4.5 (the MSS proof needs the j-th draft to be drawn from
    q_j) and sec. 10 exercise 7 (the fix: children drawn without replacement,
    the j-th tested against q with the earlier tokens removed, renormalised).

    p = (.2, .5, .3), q = (.5, .25, .25); children propose token 0 then
    token 2.  Token 0 is rejected for u >= p(0)/q(0) = 0.4; the residual is
    max(0, p - q) / 0.3 = (0, 5/6, 1/6).  Token 2 is then tested against
    q_1 = (0, .5, .5) without replacement (threshold (1/6)/0.5 = 1/3), and
    against q = (.5, .25, .25) with replacement (threshold (1/6)/0.25 = 2/3).
    After a rejection of token 2, max(0, r - q_1) = (0, 1/3, 0): the draw is
    token 1 whatever u_sample is."""
    p, q = [0.2, 0.5, 0.3], [0.5, 0.25, 0.25]
    cases = [  # (u for child 0, u for child 1) -> accepted node per mode
        ((0.39, 0.9), 1, 1),
        ((0.41, 0.30), 2, 2),
        ((0.9, 0.34), 2, 0),   # accepted with replacement only
        ((0.9, 0.66), 2, 0),
        ((0.9, 0.68), 0, 0),
    ]
    for ua, mss_node, nor_node in cases:
        for mode, want in (("mss", mss_node), ("noreplace", nor_node)):
            for us in (0.01, 0.5, 0.999):
                out = _one_level_tree(p, q, [0, 2], ua, us=us, mode=mode, lib=lib)
                assert out["status"][0] == 0
                got = int(out["accepted_nodes"][0][0]) if out["accept_len"][0] else 0
                assert got == want, (mode, ua, got)
                if want == 0 and mode == "noreplace":
                    assert out["out_tokens"][0][0] == 1, out  # residual (0, 1, 0)
    # the removed token can no longer be accepted: a third child repeating
    # token 0 has q_2(0) = 0 and r(0) = 0
    out = _one_level_tree(p, q, [0, 2, 0], (0.9, 0.9, 0.0), mode="noreplace", lib=lib)
    assert out["accept_len"][0] == 0 and out["out_tokens"][0][0] == 1


def check_tree_noreplace_mc_lossless(lib, n=120_000, seed=34):
    """Children drawn without replacement from one q, tested with the
    renormalised q_j: the emitted first token still follows p_root (the
    unbiased fix of [L17] sec. 10 exercise 7), at the accept rate the exact
    enumeration gives."""
    rng = np.random.default_rng(seed)
    V = 5
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V) * 0.7)
    ex = en.mss_exact(p, [q] * 3, mode="without_replacement")
    assert np.abs(ex["emitted"] - p).max() < 1e-12
    N = 4
    t = np.zeros((n, N, V), np.float32)
    t[:, 0] = logits_of(p)
    d = np.broadcast_to(logits_of(q)[None, None], (n, 1, V))
    # sequential sampling without replacement: Gumbel top-3 of log q
    g = np.log(q)[None] + rng.gumbel(size=(n, V))
    order = np.argsort(-g, axis=1)[:, :3].astype(np.int32)
    tok = np.concatenate([np.zeros((n, 1), np.int32), order], 1)
    par = np.tile(np.array([-1, 0, 0, 0], np.int32), (n, 1))
    qr = np.zeros((n, N), np.int32)
    ua = rng.random((n, N)).astype(np.float32)
    us = rng.random(n).astype(np.float32)
    out = oracle.verify_tree(t, d, tok, par, qr, np.ones(n), ua, us, max_depth=1,
                             mode="noreplace", lib=lib)
    assert np.all(out["status"] == 0)
    assert chi2_ok(np.bincount(out["out_tokens"][:, 0], minlength=V), p)
    acc = (out["accept_len"] == 1).mean()
    assert abs(acc - ex["accept"]) < 5 * np.sqrt(ex["accept"] * (1 - ex["accept"]) / n)


def check_tree_naive_examples(lib):
    """[L17] sec. 4.5 slides example and sec. 10 exercise 6: naive sampling
    draws from p (uniform on 4 tokens) and accepts when the draw is a child's
    token: 50 % in both.  The draw is the inverse CDF of p at the root's
    uniform, so over an even grid of u exactly half the points accept."""
    for key in ("slides_example", "exercise6"):
        g = golden("l17_exercises.json")[key]
        want = g.get("naive_accept_this_draw", g.get("naive_accept"))
        kids = [g["draft1"], g["draft2"]]
        hits = 0
        G = 64
        for k in range(G):
            u = (k + 0.5) / G
            t, d, tok, par, qr = _tree_inputs(g["p"], [g["q1"], g["q2"]], kids, 4)
            out = oracle.verify_tree(t, d, tok, par, qr, [1.0], [[u, 0.3, 0.3]], [0.5],
                                     max_depth=1, mode="naive", lib=lib)
            assert out["status"][0] == 0
            x = int(k * 4 // G)  # inverse CDF of the uniform p
            if x in kids:
                hits += 1
                assert out["accept_len"][0] == 1
                assert out["accepted_nodes"][0][0] == 1 + kids.index(x)
                assert out["out_tokens"][0][0] == x
            else:
                assert out["accept_len"][0] == 0 and out["out_tokens"][0][0] == x
        assert hits / G == want, (key, hits)


def check_tree_naive_mc(lib, n=100_000, seed=35):
    """Naive sampling is lossless (it only ever emits draws from p) and, on
    the same inputs, accepts no more often than MSS (Theorem 4.3); its rate
    matches the exact enumeration's naive rate."""
    rng = np.random.default_rng(seed)
    V = 5
    p = rng.dirichlet(np.ones(V))
    qs = [rng.dirichlet(np.ones(V)) for _ in range(3)]
    ex = en.mss_exact(p, qs)
    N = 4
    t = np.zeros((n, N, V), np.float32)
    t[:, 0] = logits_of(p)
    d = np.broadcast_to(np.stack([logits_of(q) for q in qs])[None], (n, 3, V))
    tok = np.zeros((n, N), np.int32)
    for j in range(3):
        tok[:, j + 1] = rng.choice(V, n, p=qs[j])
    par = np.tile(np.array([-1, 0, 0, 0], np.int32), (n, 1))
    qr = np.tile(np.array([0, 0, 1, 2], np.int32), (n, 1))
    ua = rng.random((n, N)).astype(np.float32)
    us = rng.random(n).astype(np.float32)
    nv = oracle.verify_tree(t, d, tok, par, qr, np.ones(n), ua, us, max_depth=1,
                            mode="naive", lib=lib)
    ms = oracle.verify_tree(t, d, tok, par, qr, np.ones(n), ua, us, max_depth=1, lib=lib)
    assert np.all(nv["status"] == 0)
    assert chi2_ok(np.bincount(nv["out_tokens"][:, 0], minlength=V), p)
    a_nv = (nv["accept_len"] == 1).mean()
    a_ms = (ms["accept_len"] == 1).mean()
    sd = np.sqrt(0.25 / n)
    assert abs(a_nv - ex["naive_accept"]) < 5 * sd
    assert a_ms >= a_nv - 5 * sd and abs(a_ms - ex["accept"]) < 5 * sd


def check_tree_modes_agree_when_greedy(lib):
    """VerifyGreedy ([L17] sec. 4.4) does not depend on the stochastic rule."""
    rng = np.random.default_rng(36)
    B, N, V = 30, 9, 7
    t = rng.normal(0, 2, (B, N, V)).astype(np.float32)
    d = rng.normal(0, 2, (B, N, V)).astype(np.float32)
    par = np.tile(np.array([-1, 0, 1, 1, 0, 4, 4, 6, 0], np.int32), (B, 1))
    tok = rng.integers(0, V, (B, N)).astype(np.int32)
    ua = rng.random((B, N)).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    outs = [oracle.verify_tree(t, d, tok, par, np.maximum(par, 0), np.zeros(B), ua, us,
                               max_depth=3, mode=m, lib=lib)
            for m in ("mss", "noreplace", "naive")]
    for o in outs[1:]:
        assert np.array_equal(o["out_tokens"], outs[0]["out_tokens"])


# ------------------------------------------------------- tree attention mask

def check_tree_mask_slides(lib):
    """[L17] sec. 4.3: the slides' mask (machine / learning / algorithm /
    system / design / translation / model) and sec. 10 exercise 5 (what e
    sees; depths as position offsets)."""
    g = golden("l17_tree_mask.json")
    names = g["nodes"]
    parent_name = {"machine": None, "learning": "machine", "algorithm": "learning",
                   "system": "learning", "design": "system", "translation": "machine",
                   "model": "translation"}
    # node 0 is the verified root; the speculated tokens follow in the
    # order the slides list them (a depth-first order)
    par = [-1] + [0 if parent_name[x] is None else 1 + names.index(parent_name[x])
                  for x in names]
    out = oracle.tree_mask(np.array([par], np.int32), lib=lib)
    assert out["status"][0] == 0
    m = out["mask"][0][:, 0]
    for i, row in enumerate(g["visible"]):
        want = {0} | {1 + names.index(x) for x in row}
        got = {j for j in range(len(par)) if (m[1 + i] >> j) & 1}
        assert got == want, (names[i], got, want)
    e5 = golden("l17_ex5_tree.json")
    out = oracle.tree_mask(np.array([e5["parent"]], np.int32), lib=lib)
    assert list(out["depth"][0]) == e5["depth"]
    sees = {e5["dfs_order"][j] for j in range(8) if (out["mask"][0][5][0] >> j) & 1}
    assert sees == set(e5["ancestors_of_e"]) | {"e"}


def check_tree_mask_closure(lib):
    """Random DFS trees (up to 64 nodes, two mask words): the mask is the
    reflexive-transitive closure of the parent relation (boolean matrix
    powers) and the depth is the number of proper ancestors; malformed
    trees and padding rows come back empty."""
    rng = np.random.default_rng(37)
    B, N = 40, 64
    par = np.full((B, N), -1, np.int32)
    nn = rng.integers(1, N + 1, B).astype(np.int32)
    for b in range(B):
        for i in range(1, nn[b]):
            par[b, i] = rng.integers(max(0, i - 5), i)  # a parent shortly before
    bad = 3
    par[bad, 7] = 7 if nn[bad] > 7 else par[bad, 7]
    nn[bad] = max(nn[bad], 8)
    out = oracle.tree_mask(par, nn, lib=lib)
    for b in range(B):
        if b == bad:
            assert out["status"][b] != 0 and not out["mask"][b].any()
            assert np.all(out["depth"][b] == -1)
            continue
        n = nn[b]
        A = np.zeros((n, n), bool)
        for i in range(1, n):
            A[i, par[b, i]] = True
        R = np.eye(n, dtype=bool)
        step = np.eye(n, dtype=bool)
        for _ in range(n):
            step = (step.astype(int) @ A.astype(int)) > 0
            R |= step
        bits = np.zeros((N, 64), bool)
        words = out["mask"][b]
        for w in range(2):
            for k in range(32):
                bits[:, 32 * w + k] = (words[:, w] >> np.uint32(k)) & 1
        assert np.array_equal(bits[:n, :n], R), b
        assert not bits[:n, n:].any() and not bits[n:].any()
        assert np.array_equal(out["depth"][b][:n], R.sum(1) - 1)
        assert np.all(out["depth"][b][n:] == -1)


# -------------------------------------------------- per-position statistics

def check_row_stats_worked(lib):
    """[N02] sec. 9: q = (.5, .2, .15, .1, .05), p = (.3, .35, .2, .1, .05)
    gives alpha = 0.8, and with three such positions E[N] = 2.952; the
    printed E[tokens] examples for identical positions; p == q accepts
    everything (E[N] = K + 1)."""
    g = golden("n02_sec9_worked_round.json")
    p, q = np.array(g["p"]), np.array(g["q"])
    K = 3
    t = np.tile(logits_of(p), (1, K + 1, 1)).astype(np.float32)
    d = np.tile(logits_of(q), (1, K, 1)).astype(np.float32)
    out = oracle.row_stats(t, d, [1.0], lib=lib)
    assert np.allclose(out["alpha"][0], 0.8, atol=1e-6)
    assert abs(out["expected"][0] - 2.952) < 1e-5
    for ex in golden("l17_exercises.json")["E_examples"]:
        a = ex["alpha"]
        pp = np.array([a, 1 - a])
        qq = np.array([1.0, 0.0])  # sum min = a
        t = np.tile(logits_of(pp), (1, ex["K"] + 1, 1)).astype(np.float32)
        with np.errstate(divide="ignore"):
            d = np.tile(np.log(qq), (1, ex["K"], 1)).astype(np.float32)
        out = oracle.row_stats(t, d, [1.0], lib=lib)
        assert round(out["expected"][0], ex["digits"]) == ex["E"], ex
    r = np.random.default_rng(38).normal(0, 2, (2, 5, 9)).astype(np.float32)
    out = oracle.row_stats(r, r[:, :4].copy(), [0.7, 0.0], lib=lib)
    assert np.allclose(out["alpha"], 1.0) and np.allclose(out["expected"], 5.0)


def check_row_stats_tv(lib):
    """alpha = 1 - TV(p, q) (Thm 3.5) on random rows with temperature, top-k
    and ragged drafts: TV from a library softmax; greedy positions give the
    argmax-agreement indicator; positions past num_drafts are NaN."""
    rng = np.random.default_rng(39)
    B, K, V = 12, 4, 33
    t = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    d = (t[:, :K] + rng.normal(0, 1.5, (B, K, V))).astype(np.float32)
    temp = rng.choice([0.0, 0.5, 1.0, 1.6], B).astype(np.float32)
    nd = rng.integers(0, K + 1, B).astype(np.int32)
    tk = rng.choice([0, 5], B).astype(np.int32)
    out = oracle.row_stats(t, d, temp, num_drafts=nd, top_k=tk, lib=lib)
    for b in range(B):
        e, reach = 0.0, 1.0
        for i in range(K):
            a = out["alpha"][b, i]
            if i >= nd[b]:
                assert np.isnan(a)
                continue
            if temp[b] == 0:
                want = float(np.argmax(t[b, i]) == np.argmax(d[b, i]))
            else:
                def dist(l):
                    y = l.astype(np.float64) / temp[b]
                    if tk[b]:
                        keep = np.lexsort((np.arange(V), -y))[:tk[b]]
                        z = np.full(V, -np.inf)
                        z[keep] = y[keep]
                        y = z
                    return softmax(y)
                want = 1.0 - 0.5 * np.abs(dist(t[b, i]) - dist(d[b, i])).sum()
            assert abs(a - want) < 1e-12, (b, i, a, want)
        for j in range(nd[b] + 1):
            e += reach
            if j < nd[b]:
                reach *= out["alpha"][b, j]
        assert abs(out["expected"][b] - e) < 1e-12


ALL_FAST += [check_icdf_window_examples, check_icdf_window_bruteforce, check_chain_draw_window]
ALL_FAST += [check_tree_noreplace_thresholds, check_tree_naive_examples,
             check_tree_modes_agree_when_greedy, check_tree_mask_slides,
             check_tree_mask_closure, check_row_stats_worked, check_row_stats_tv]
ALL_MC += [check_tree_noreplace_mc_lossless, check_tree_naive_mc]
