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
