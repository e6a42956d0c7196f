"""Exact (fp64, numpy) distributions of the verification step.

TEST INFRASTRUCTURE ONLY.  These functions integrate the method over its
randomness analytically -- every draft sequence weighted by its draft
probability, every accept test by its probability min(1, p/q) -- and so give
the exact distribution of what the step emits.  They pin the C oracle
(sv_oracle.c) through Monte Carlo and grid tests, and reproduce the numbers
the pages print for correct and for deliberately wrong verification rules.

Sources (cited by page title and section):
  [L17] CMU 15-779 Lecture 17 notes, "Speculative Decoding": sec. 2.3
        (speculative sampling, its proof, exact enumeration over 625
        sequences, the three wrong implementations), 2.5 (E = (1 -
        a^(g+1)) / (1 - a)), 4.5 (naive sampling vs multi-step speculative
        sampling, Theorems 4.2 / 4.3, the requirement that tree children are
        sampled), sec. 10 exercises 2, 3, 6, 7.
  [N02] "LLM speculative decoding study notes 02", sec. 5.1-5.3 (Lemma 1,
        Lemma 2, sequence-level theorem by induction), 9 (worked example),
        10 (greedy), 14 (exercises 1, 2, 6).
  [S14] "Speculative decoding" tutorial: E[tokens] examples.
"""
from __future__ import annotations

import itertools

import numpy as np


# ------------------------------------------------------------ closed forms

def expected_tokens(alpha: float, K: int) -> float:
    """E[N] = (1 - alpha^(K+1)) / (1 - alpha), and K + 1 when alpha = 1
    ([L17] sec. 2.5 formula 1; [N02] sec. 6)."""
    if alpha == 1.0:
        return float(K + 1)
    return (1.0 - alpha ** (K + 1)) / (1.0 - alpha)


def accept_length_law(alphas) -> np.ndarray:
    """P(accept_len = j), j = 0..K, when position i is accepted with
    probability alphas[i] independently: (prod_{i<j} a_i)(1 - a_j) for j < K
    and prod a_i for j = K."""
    K = len(alphas)
    out = np.zeros(K + 1)
    run = 1.0
    for j in range(K):
        out[j] = run * (1.0 - alphas[j])
        run *= alphas[j]
    out[K] = run
    return out


def overlap(p, q) -> float:
    """alpha = sum min(p, q) = 1 - TV(p, q) ([L17] sec. 2.3, Thm 3.5)."""
    return float(np.minimum(p, q).sum())


# ------------------------------------------------------- one position, exact

def emitted_one_position(p, q, rule: str = "speculative") -> np.ndarray:
    """Exact distribution of the token emitted at one position when the
    draft x ~ q is verified against p.

    rule = "speculative": accept w.p. min(1, p(x)/q(x)), else draw from
           norm(max(0, p - q))  -> equals p ([N02] Lemma 2).
    rule = "greedy_rule": the greedy rule misused under sampling -- accept
           iff x = argmax p, else draw from p ([L17] sec. 10 exercise 3
           gives (0.8, 0.2) for p = (0.6, 0.4), q = (0.5, 0.5)).
    rule = "no_resample": accept w.p. min(1, p/q); a rejection emits nothing
           (returned unnormalised; its mass is the accept rate).
    """
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    V = p.shape[0]
    out = np.zeros(V)
    w = np.maximum(0.0, p - q)
    S = w.sum()
    a = int(np.argmax(p))
    for x in range(V):
        if q[x] == 0.0:
            continue
        if rule == "greedy_rule":
            acc = 1.0 if x == a else 0.0
            out[x] += q[x] * acc
            out += q[x] * (1.0 - acc) * p
            continue
        acc = min(1.0, p[x] / q[x])
        out[x] += q[x] * acc
        if rule == "speculative" and S > 0.0:
            out += q[x] * (1.0 - acc) * (w / S)
    return out


def emitted_deterministic_draft(p, q, draft: int) -> np.ndarray:
    """Exact output when the draft is fixed (e.g. always argmax q) but the
    speculative accept / residual rule is applied as if x ~ q.  Biased:
    [L17] sec. 10 exercise 7 gives (0.833, 0.167) for p = (0.5, 0.5),
    q = (0.6, 0.4)."""
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    out = np.zeros_like(p)
    acc = min(1.0, p[draft] / q[draft])
    out[draft] += acc
    w = np.maximum(0.0, p - q)
    if w.sum() > 0:
        out += (1.0 - acc) * w / w.sum()
    return out


# ------------------------------------------ chain, context-free positions

def chain_exact(p_rows, q_rows) -> dict:
    """Exact law of one chain round with position-specific, context-free
    distributions p_1..p_{K+1}, q_1..q_K (draft x_i ~ q_i independently).

    Sums over all V^K draft sequences weighted by prod q_i(x_i); each accept
    test contributes min(1, p_i/q_i) analytically ([L17] sec. 2.4).
    Returns accept_len law [K+1] and, for each position i = 0..K, the
    distribution of the token emitted there given the round reached it.
    """
    p_rows = np.asarray(p_rows, dtype=np.float64)
    q_rows = np.asarray(q_rows, dtype=np.float64)
    K, V = q_rows.shape
    law = np.zeros(K + 1)
    emit = np.zeros((K + 1, V))
    reach = np.zeros(K + 1)
    for xs in itertools.product(range(V), repeat=K):
        wq = 1.0
        for i, x in enumerate(xs):
            wq *= q_rows[i, x]
        if wq == 0.0:
            continue
        run = wq  # probability of reaching position i with these drafts
        for i, x in enumerate(xs):
            reach[i] += run
            acc = min(1.0, p_rows[i, x] / q_rows[i, x])
            emit[i, x] += run * acc
            w = np.maximum(0.0, p_rows[i] - q_rows[i])
            S = w.sum()
            rej = run * (1.0 - acc)
            law[i] += rej
            if S > 0.0:
                emit[i] += rej * w / S
            else:
                emit[i] += rej * p_rows[i]
            run *= acc
        reach[K] += run
        law[K] += run
        emit[K] += run * p_rows[K]
    cond = emit / np.where(reach > 0, reach, 1.0)[:, None]
    return dict(accept_len_law=law, emitted_given_reached=cond, reach=reach)


# ------------------------------- chain over a context-dependent toy model

class ToyModel:
    """A toy language model in the spirit of [L17] sec. 0.4: V tokens, the
    next-token distribution depends on the last `ctx` tokens through a fixed
    random table; the draft is softmax(log p + noise)."""

    def __init__(self, V: int = 5, ctx: int = 2, noise: float = 0.8, seed: int = 0):
        rng = np.random.default_rng(seed)
        self.V, self.ctx = V, ctx
        n_ctx = V ** ctx
        lp = rng.normal(0.0, 1.5, size=(n_ctx, V))
        self.p = np.exp(lp - lp.max(1, keepdims=True))
        self.p /= self.p.sum(1, keepdims=True)
        lq = np.log(self.p) + rng.normal(0.0, noise, size=(n_ctx, V))
        self.q = np.exp(lq - lq.max(1, keepdims=True))
        self.q /= self.q.sum(1, keepdims=True)
        self.p_logits = np.log(self.p)
        self.q_logits = np.log(self.q)

    def key(self, hist) -> int:
        k = 0
        for t in hist[-self.ctx:]:
            k = k * self.V + int(t)
        return k

    def target(self, hist) -> np.ndarray:
        return self.p[self.key(hist)]

    def draft(self, hist) -> np.ndarray:
        return self.q[self.key(hist)]


def autoregressive_law(model: ToyModel, prefix, L: int) -> dict:
    """Exact distribution of the next L tokens sampled from p alone."""
    out = {}
    for seq in itertools.product(range(model.V), repeat=L):
        h = list(prefix)
        pr = 1.0
        for t in seq:
            pr *= model.target(h)[t]
            h.append(t)
        out[seq] = pr
    return out


def speculative_law(model: ToyModel, prefix, L: int, K: int) -> dict:
    """Exact distribution of the first L tokens produced by repeated rounds
    of speculative sampling with K drafts ([L17] sec. 2.3 "exact check":
    every branch enumerated; [N02] sec. 5.3 theorem: equals the
    autoregressive law)."""
    out: dict = {}

    def rounds(hist, weight):
        if len(hist) - len(prefix) >= L:
            seq = tuple(hist[len(prefix):len(prefix) + L])
            out[seq] = out.get(seq, 0.0) + weight
            return
        # one round: enumerate drafts position by position
        def step(h, i, w):
            if w == 0.0:
                return
            p = model.target(h)
            if i == K:  # all accepted: bonus from p_{K+1}
                for t in range(model.V):
                    rounds(h + [t], w * p[t])
                return
            q = model.draft(h)
            r = np.maximum(0.0, p - q)
            S = r.sum()
            for x in range(model.V):
                if q[x] == 0.0:
                    continue
                acc = min(1.0, p[x] / q[x])
                step(h + [x], i + 1, w * q[x] * acc)
                rej = w * q[x] * (1.0 - acc)
                if rej > 0.0:
                    dist = r / S if S > 0 else p
                    for t in range(model.V):
                        rounds(h + [t], rej * dist[t])
        step(list(hist), 0, weight)

    rounds(list(prefix), 1.0)
    return out


def tv(a: dict, b: dict) -> float:
    keys = set(a) | set(b)
    return 0.5 * sum(abs(a.get(k, 0.0) - b.get(k, 0.0)) for k in keys)


# --------------------------------------------------------- tree, one level

def mss_exact(p, q_list, children_from=None, mode: str = "with_replacement") -> dict:
    """Exact law of one multi-step speculative sampling step at a node with
    len(q_list) children ([L17] sec. 4.5).

    Child j's token is drawn from q_list[j]: independently ("with_replacement",
    the SpecInfer setting), or without replacement from one shared q
    ("without_replacement": q_j = q with earlier siblings' tokens removed and
    renormalised, also used as the accept distribution), or deterministically
    as the j-th most likely token of q ("deterministic_topk", biased).
    Children are tried in order: accept child j iff u*q_j(x_j) < r(x_j); on
    rejection r <- norm(max(0, r - q_j)); if all are rejected, draw from r.

    Returns dict(emitted = exact output distribution, accept = probability
    that some child is accepted, naive_accept = probability that a draw from
    p lands on a child token (naive sampling)).
    """
    p = np.asarray(p, dtype=np.float64)
    V = p.shape[0]
    n = len(q_list)
    qs = [np.asarray(q, dtype=np.float64) for q in q_list]
    emitted = np.zeros(V)
    accept = 0.0
    naive = 0.0

    def walk(tokens, wt):
        nonlocal accept, naive
        r = p.copy()
        run = wt
        naive += wt * p[list(set(tokens))].sum()
        for j, x in enumerate(tokens):
            qj = qs[j] if mode != "without_replacement" else _without(qs[0], tokens[:j])
            if qj[x] == 0.0:
                acc = 1.0 if r[x] > 0 else 0.0
            else:
                acc = min(1.0, r[x] / qj[x])
            emitted[x] += run * acc
            accept += run * acc
            run *= (1.0 - acc)
            w = np.maximum(0.0, r - qj)
            if w.sum() > 0.0:
                r = w / w.sum()
        emitted[:] += run * r

    if mode == "deterministic_topk":
        order = np.argsort(-qs[0], kind="stable")
        walk([int(order[j]) for j in range(n)], 1.0)
    else:
        for toks in itertools.product(range(V), repeat=n):
            if mode == "without_replacement" and len(set(toks)) < n:
                continue
            wt = 1.0
            for j, x in enumerate(toks):
                qj = qs[j] if mode != "without_replacement" else _without(qs[0], toks[:j])
                wt *= qj[x]
            if wt > 0.0:
                walk(list(toks), wt)
    return dict(emitted=emitted, accept=accept, naive_accept=naive)


def _without(q, removed) -> np.ndarray:
    q = np.array(q, dtype=np.float64)
    for t in removed:
        q[t] = 0.0
    s = q.sum()
    return q / s if s > 0 else q
