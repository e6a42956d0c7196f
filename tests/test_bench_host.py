"""Host-side pieces of bench.py: the key that ties a stored ncu figure to the
chain kernel's code, and the committed ncu summary it is read from."""
import os
import re
import shutil

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _hash_of(tmp_path, edit):
    """source_hash() of a copy of the kernel sources with `edit` applied to sv_chain.cuh."""
    pkg = tmp_path / "speculative_decoding_verification_63_gb300" / "csrc"
    shutil.copytree(os.path.join(ROOT, "speculative_decoding_verification_63_gb300", "csrc"), pkg)
    p = pkg / "sv_chain.cuh"
    p.write_text(edit(p.read_text()))
    old = bench.ROOT
    bench.ROOT = str(tmp_path)
    try:
        return bench.source_hash()
    finally:
        bench.ROOT = old


def test_hash_ignores_comments_and_blank_lines(tmp_path):
    base = bench.source_hash()
    assert _hash_of(tmp_path / "a", lambda s: s.replace("#pragma once", "// a note\n\n#pragma once")) == base


def test_hash_changes_with_the_code(tmp_path):
    base = bench.source_hash()
    assert _hash_of(tmp_path / "b", lambda s: s.replace("#pragma once", "#pragma once\nint x_;")) != base


def test_committed_ncu_summary_has_the_figures():
    text = open(os.path.join(ROOT, "profiles", "verify_chain_b64_k6_v128256.md")).read()
    assert re.search(r"^- source_hash: `[0-9a-f]{16}`$", text, re.M)
    m = re.search(r"^- dram_bytes_per_launch: `(\d+)`$", text, re.M)
    assert m and int(m.group(1)) > 0
    assert "--clock-control none" in text


def test_hash_ignores_block_comments(tmp_path):
    base = bench.source_hash()
    edit = lambda s: s.replace("#pragma once", "/* a block\n   comment */\n#pragma once")
    assert _hash_of(tmp_path / "c", edit) == base


def test_hash_of_the_tree_kernel_is_its_own():
    assert bench.source_hash("tree") != bench.source_hash("chain")


def _ref(B, tokens, lo, hi, margin_accept, margin_draw, out_len):
    import numpy as np
    return {"status": np.zeros(B, np.int32), "out_tokens": np.array(tokens, np.int32),
            "out_len": np.array(out_len, np.int32), "accept_len": np.array(out_len, np.int32) - 1,
            "draw_lo": np.array(lo, np.int32), "draw_hi": np.array(hi, np.int32),
            "margin_accept": np.array(margin_accept), "margin_draw": np.array(margin_draw)}


def test_parity_counts_follow_the_test_rule():
    """bench.parity_counts: a near final draw may move within the oracle's
    window; anything else that differs is a firm mismatch."""
    import numpy as np
    inf = np.inf
    ref = _ref(4, [[5, 7, -1], [5, 9, -1], [3, -1, -1], [4, 4, 8]], lo=[7, 8, 3, 8],
               hi=[7, 10, 3, 8], margin_accept=[inf, inf, inf, 1e-8],
               margin_draw=[0.1, 1e-7, inf, 0.2], out_len=[2, 2, 1, 3])
    got = {k: ref[k].copy() for k in ("out_tokens", "out_len", "accept_len")}
    got["out_tokens"][1, 1] = 10      # near draw, inside its window
    got["out_tokens"][3] = [4, 6, -1]  # near accept test: only counted
    got["out_len"][3] = 2
    got["accept_len"][3] = 1
    c = bench.parity_counts(got, ref)
    assert c["near_draw"] == 1 and c["near_draw_mismatch"] == 1
    assert c["near_accept"] == 1 and c["near_accept_mismatch"] == 1
    assert c["firm_mismatch"] == 0
    got["out_tokens"][0, 1] = 8       # a firm draw that moved
    assert bench.parity_counts(got, ref)["firm_mismatch"] == 1
    got["out_tokens"][0, 1] = 7
    got["out_tokens"][1, 1] = 11      # outside the near draw's window
    assert bench.parity_counts(got, ref)["firm_mismatch"] == 1


def test_cpu_oracle_one_thread_and_all_cores():
    """The CPU baseline leg on a small pool: one thread, then every core in
    spawned workers; the one-thread pass's outputs come back for the parity
    counts."""
    import numpy as np
    from speculative_decoding_verification_63_gb300 import workloads as wl
    wk = bench.Workload(2)
    wk.pool = wl.make_chain(2, B=6, V=3000, seed=5)
    wk.Btot, wk.B, wk.windows, wk.V = 6, 1, 6, 3000
    base, ref = bench.cpu_oracle(wk, 0.2, 0.5, np.arange(6))
    assert base["cores"] == 1 and base["cores_all"] == os.cpu_count()
    assert base["value"] > 0 and base["value_all_cores"] > 0
    import oracle
    want = oracle.verify_chain_inputs(wk.pool)
    assert np.array_equal(ref["out_tokens"], want["out_tokens"])


def test_committed_dram_figures_match_the_current_sources():
    """Each workload's committed ncu summary was taken on the kernel sources
    as they are: bench.py finds its DRAM bytes (a stale summary gives null)."""
    for key in (2, 3, 4, 5):
        wk = bench.Workload(key)
        assert bench.stored_traffic(wk.profile, wk.kernel), (wk.profile, wk.kernel)
