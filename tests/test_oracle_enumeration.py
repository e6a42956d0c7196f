"""Pins of the exact enumerator (oracle/enumerate.py) against the numbers
the pages print and against the losslessness theorem."""
import numpy as np
import pytest

from oracle import enumerate as en
from oracle_pins import golden


def test_expected_tokens_printed_values():
    """[L17] sec. 2.5 / exercise 1, [N02] sec. 9.3, [S14] E[tokens]."""
    for ex in golden("l17_exercises.json")["E_examples"]:
        assert round(en.expected_tokens(ex["alpha"], ex["K"]), ex["digits"]) == ex["E"]
    assert en.expected_tokens(1.0, 5) == 6.0  # [N02] sec. 11.3: alpha = 1 -> K+1
    # E is capped by 1 / (1 - alpha)  ([L17] sec. 2.5)
    assert en.expected_tokens(0.8, 200) <= 5.0 + 1e-12


def test_one_position_rules_printed_values():
    g = golden("l17_exercises.json")
    e3 = g["exercise3"]
    assert np.allclose(en.emitted_one_position(e3["p"], e3["q"]), e3["correct_output"])
    assert np.allclose(en.emitted_one_position(e3["p"], e3["q"], "greedy_rule"),
                       e3["greedy_rule_output"])
    assert abs(en.overlap(e3["p"], e3["q"]) - e3["alpha"]) < 1e-15
    e7 = g["exercise7"]
    assert np.allclose(en.emitted_deterministic_draft(e7["p"], e7["q"], 0),
                       e7["biased_output"])
    # dropping the resample loses exactly the rejection mass 1 - alpha
    out = en.emitted_one_position(e3["p"], e3["q"], "no_resample")
    assert abs(out.sum() - e3["alpha"]) < 1e-15


def test_mss_printed_values():
    """[L17] sec. 4.5 slides example: MSS 81.25 %, naive 43.75 % averaged
    over SSM 2's draw; MSS is lossless (Thm 4.2) and beats naive (Thm 4.3)."""
    s = golden("l17_exercises.json")["slides_example"]
    r = en.mss_exact(s["p"], [s["q1"], s["q2"]])
    assert abs(r["accept"] - s["mss_accept_averaged"]) < 1e-15
    assert abs(r["naive_accept"] - s["naive_accept_averaged"]) < 1e-15
    assert np.allclose(r["emitted"], s["p"], atol=1e-15)


@pytest.mark.parametrize("seed", range(4))
def test_mss_lossless_and_beats_naive(seed):
    rng = np.random.default_rng(seed)
    V = 5
    p = rng.dirichlet(np.ones(V))
    qs = [rng.dirichlet(np.ones(V)) for _ in range(2 + seed % 2)]
    r = en.mss_exact(p, qs)
    assert np.abs(r["emitted"] - p).max() < 1e-12
    assert r["accept"] >= r["naive_accept"] - 1e-12
    shared = en.mss_exact(p, [qs[0]] * 3)
    assert np.abs(shared["emitted"] - p).max() < 1e-12
    # without replacement, with the renormalised q_j, stays lossless
    wor = en.mss_exact(p, [qs[0]] * 3, mode="without_replacement")
    assert np.abs(wor["emitted"] - p).max() < 1e-12
    # deterministic top-k children under the same rule are biased
    det = en.mss_exact(p, [qs[0]] * 2, mode="deterministic_topk")
    assert np.abs(det["emitted"] - p).max() > 1e-3


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_toy_model_625_sequences(K):
    """[L17] sec. 2.3: exact enumeration of every branch on a 5-token toy
    model; the first 4 tokens (625 sequences) match the target to ~1e-16."""
    m = en.ToyModel(V=5, ctx=2, seed=1)
    a = en.autoregressive_law(m, [0, 1], 4)
    b = en.speculative_law(m, [0, 1], 4, K)
    assert len(a) == 625
    assert en.tv(a, b) < 1e-12


def test_chain_exact_position_laws():
    """[N02] Lemma 2 per position, and the accept-length law."""
    rng = np.random.default_rng(2)
    K, V = 3, 4
    P = rng.dirichlet(np.ones(V), K + 1)
    Q = rng.dirichlet(np.ones(V), K)
    r = en.chain_exact(P, Q)
    assert np.abs(r["emitted_given_reached"] - P).max() < 1e-12
    law = en.accept_length_law([en.overlap(P[i], Q[i]) for i in range(K)])
    assert np.abs(r["accept_len_law"] - law).max() < 1e-12
    # identical rows: E[N] = (1 - a^(K+1)) / (1 - a)
    Pi = np.tile(P[0], (K + 1, 1))
    Qi = np.tile(Q[0], (K, 1))
    r = en.chain_exact(Pi, Qi)
    EN = (r["accept_len_law"] * np.arange(1, K + 2)).sum()
    assert abs(EN - en.expected_tokens(en.overlap(P[0], Q[0]), K)) < 1e-12
