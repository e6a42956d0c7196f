"""Planted mistakes in the CPU oracle must be caught by its pins.

Each case copies sv_oracle.c, applies one textual mutation (a dropped term,
a wrong sign or index, swapped operands, a wrong tie rule), builds the copy
with gcc into a temporary directory and runs the pin suite of
tests/oracle_pins.py against it; at least one pin must fail.  Nothing here
touches the real oracle build."""
import os
import subprocess

import pytest

import oracle
import oracle_pins as pins

MUTANTS = {
    "residual_drops_max": ("w[t] = d > 0.0 ? d : 0.0;", "w[t] = d;"),
    "accept_test_swapped": ("if ((double)u[n] * qi < pi) ++n;",
                            "if ((double)u[n] * pi < qi) ++n;"),
    "accept_test_ignores_q": ("if ((double)u[n] * qi < pi) ++n;",
                              "if ((double)u[n] < pi) ++n;"),
    "residual_from_next_row": (
        "st = svo_row_probs(trow0 + (size_t)n * V * es, dtype, V, T, tk, p);",
        "st = svo_row_probs(trow0 + (size_t)(n < nd ? n + 1 : n) * V * es, dtype, V, T, tk, p);"),
    "icdf_reversed": ("double target = u * S;", "double target = (1.0 - u) * S;"),
    "temperature_multiplies": ("y[j] = logit_at(row, dtype, j) / T;",
                               "y[j] = logit_at(row, dtype, j) * T;"),
    "argmax_ties_to_highest": ("if (l > best) { best = l; a = j; }",
                               "if (l >= best) { best = l; a = j; }"),
    "topk_keeps_all_ties": ("else if (y[j] == thr && ties_left > 0)",
                            "else if (y[j] == thr)"),
    "mss_no_residual_update": ("for (int t = 0; t < V; ++t) r[t] = w[t] / S;",
                               "for (int t = 0; t < V; ++t) r[t] = r[t];"),
    "mss_accept_against_p": ("if ((double)ua[c] * q[xc] < r[xc]) { next = c; break; }",
                             "if ((double)ua[c] * q[xc] < p[xc]) { next = c; break; }"),
    "bonus_from_draft_row": (
        "          /* all drafts accepted: bonus token from p_{nd+1} */\n"
        "          token = svo_icdf(p, V, (double)u[K], &mg);",
        "          /* all drafts accepted: bonus token from p_{nd+1} */\n"
        "          svo_row_probs(drow0 + (size_t)(nd - 1) * V * es, dtype, V, T, tk, q);\n"
        "          token = svo_icdf(nd > 0 ? q : p, V, (double)u[K], &mg);"),
    "greedy_emits_draft": ("      token = a[n];", "      token = n < nd ? x[n] : a[n];"),
    "noreplace_keeps_tried": ("for (int j = 0; j < n_tried; ++j) q[tried[j]] = 0.0;",
                              "for (int j = 0; j < n_tried; ++j) q[tried[j]] = q[tried[j]];"),
    "noreplace_not_renormalised": ("for (int t = 0; t < V; ++t) q[t] /= sq;",
                                   "for (int t = 0; t < V; ++t) q[t] = q[t];"),
    "naive_takes_any_child": ("if (par[c] == node && tok[c] == x) { next = c; break; }",
                              "if (par[c] == node) { next = c; break; }"),
    "naive_draws_with_u_sample": ("int x = svo_icdf(p, V, (double)ua[node], &mgn);",
                                  "int x = svo_icdf(p, V, (double)u_sample[b], &mgn);"),
    "mask_drops_self": ("mrow[(size_t)i * W + j / 32] |= 1u << (j % 32);",
                        "if (j != i) mrow[(size_t)i * W + j / 32] |= 1u << (j % 32);"),
    "mask_depth_off_by_one": ("      int d = -1;", "      int d = 0;"),
    "stats_sum_of_max": ("a += p[t] < q[t] ? p[t] : q[t];", "a += p[t] > q[t] ? p[t] : q[t];"),
    "window_ignores_radius": ("const double a = (u - radius) * S, b = (u + radius) * S;",
                              "const double a = u * S, b = u * S;"),
    "window_keeps_zero_weights": ("    if (!(w[t] > 0.0)) continue;\n    if (c > a && c_prev <= b) {",
                                  "    if (c > a && c_prev <= b) {"),
    "stats_expected_stops_early": ("for (int j = 0; j <= nd; ++j) {",
                                   "for (int j = 0; j < nd; ++j) {"),
}


def _build_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = os.path.join(tmp_path, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(tmp_path, f"lib{name}.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", lib, path, "-lm"],
                   check=True)
    return oracle.load(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    lib = _build_mutant(str(tmp_path), name)
    failed = []
    for check in pins.ALL_FAST + pins.ALL_MC:
        try:
            if check in pins.ALL_MC:
                check(lib, n=20_000)
            else:
                check(lib)
        except AssertionError:
            failed.append(check.__name__)
            break
        except Exception as e:  # a crash or bad status also counts as caught
            failed.append(f"{check.__name__}: {type(e).__name__}")
            break
    assert failed, f"mutant {name} passed every pin"
