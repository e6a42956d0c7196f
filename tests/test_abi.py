"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function include/specverify.h declares, its structs match the ctypes
binding field for field, and host-side argument checks answer before any
device work."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="session")
def svlib():
    from speculative_decoding_verification_63_gb300 import _binding, _build
    _build.build_library()
    return _binding.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sv_[a-z_]+)\s*\(", src)))


def test_header_declares_binding_exports():
    from speculative_decoding_verification_63_gb300 import _binding
    assert declared_functions() == sorted(_binding.EXPORTS)


def test_every_declared_symbol_is_exported(svlib):
    for name in declared_functions():
        assert hasattr(svlib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", svlib._name], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (sv_\w+)", out))
    assert set(declared_functions()) <= exported


def test_struct_layout_matches_binding(tmp_path):
    from speculative_decoding_verification_63_gb300 import _binding
    lines = ['#include "specverify.h"', "#include <stdio.h>", "#include <stddef.h>",
             "int main(void) {"]
    expect = []
    for cname, cls in [("sv_chain_args", _binding.SvChainArgs),
                       ("sv_tree_args", _binding.SvTreeArgs),
                       ("sv_tree_mask_args", _binding.SvTreeMaskArgs)]:
        lines.append(f'printf("%zu\\n", sizeof({cname}));')
        expect.append(ctypes.sizeof(cls))
        for f, _ in cls._fields_:
            lines.append(f'printf("%zu\\n", offsetof({cname}, {f}));')
            expect.append(getattr(cls, f).offset)
    lines.append("return 0; }")
    c = tmp_path / "layout.c"
    c.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", f"-I{os.path.dirname(HEADER)}", "-o", str(exe), str(c)],
                   check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert got == expect


def test_workspace_sizes(svlib):
    from speculative_decoding_verification_63_gb300 import _binding as b
    assert b.sv_chain_workspace_bytes(64, 6, 128256, b.SV_BF16) > 0
    assert b.sv_chain_workspace_bytes(0, 6, 128256, b.SV_BF16) > 0
    assert b.sv_tree_workspace_bytes(16, 32, 32, 32000, b.SV_BF16) > 0
    bad = [(b.SV_MAX_B + 1, 6, 100, 0, 0), (4, b.SV_MAX_K + 1, 100, 0, 0), (4, 6, 0, 0, 0),
           (4, 6, b.SV_MAX_V + 1, 0, 0), (4, 6, 100, 7, 0), (4, 6, 100, 0, b.SV_MAX_TOPK + 1),
           (-1, 6, 100, 0, 0)]
    for args in bad:
        assert b.sv_chain_workspace_bytes(*args) == 0, args
    assert b.sv_tree_workspace_bytes(4, b.SV_MAX_TREE_NODES + 1, 4, 100, 0) == 0
    assert b.sv_tree_workspace_bytes(b.SV_MAX_TREE_B + 1, 4, 4, 100, 0) == 0
    # grows with the batch
    assert (b.sv_chain_workspace_bytes(128, 6, 128256, 0)
            > b.sv_chain_workspace_bytes(64, 6, 128256, 0))


def _chain_args(b, **kw):
    a = b.SvChainArgs()
    a.B, a.K, a.V, a.dtype = 4, 4, 1000, b.SV_BF16
    fake = 0x100000
    for f in ("target_logits", "draft_logits", "draft_tokens", "temperature", "uniforms",
              "out_tokens", "out_len", "accept_len"):
        setattr(a, f, fake)
    a.target_row_stride = a.draft_row_stride = 1000
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_host_side_checks(svlib):
    """Every case below is rejected (or accepted as empty) before any CUDA
    call, so it runs without a GPU."""
    from speculative_decoding_verification_63_gb300 import _binding as b
    ws_ok = ctypes.c_void_p(0x200000)
    big = 1 << 30
    call = lambda a, ws=ws_ok, n=big: svlib.sv_verify_chain(ctypes.byref(a), ws, n, None)
    assert svlib.sv_verify_chain(None, ws_ok, big, None) == b.SV_EINVAL
    assert call(_chain_args(b, B=0)) == b.SV_OK
    assert call(_chain_args(b, K=b.SV_MAX_K + 1)) == b.SV_EINVAL
    assert call(_chain_args(b, V=0)) == b.SV_EINVAL
    assert call(_chain_args(b, dtype=3)) == b.SV_EINVAL
    assert call(_chain_args(b, target_logits=None)) == b.SV_EINVAL
    assert call(_chain_args(b, uniforms=None)) == b.SV_EINVAL
    assert call(_chain_args(b, target_row_stride=999)) == b.SV_EINVAL
    assert call(_chain_args(b, max_top_k=b.SV_MAX_TOPK + 1)) == b.SV_EINVAL
    assert call(_chain_args(b), ws=ctypes.c_void_p(0)) == b.SV_EWORKSPACE
    assert call(_chain_args(b), ws=ctypes.c_void_p(0x200010)) == b.SV_EWORKSPACE
    assert call(_chain_args(b), n=16) == b.SV_EWORKSPACE
    assert svlib.sv_verify_tree(None, ws_ok, big, None) == b.SV_EINVAL
    t = b.SvTreeArgs()
    t.B, t.N, t.M, t.V, t.max_depth = 2, 8, 8, 100, 8  # max_depth must be < N
    assert svlib.sv_verify_tree(ctypes.byref(t), ws_ok, big, None) == b.SV_EINVAL
    t.max_depth = 3
    t.mode = 3  # no such tree mode
    assert svlib.sv_verify_tree(ctypes.byref(t), ws_ok, big, None) == b.SV_EINVAL
    # tree mask
    m = b.SvTreeMaskArgs()
    m.B, m.N, m.words = 4, 40, 2
    m.parent = m.mask = m.depth = 0x100000
    mcall = lambda a, ws=ws_ok, n=big: svlib.sv_tree_mask(ctypes.byref(a), ws, n, None)
    assert svlib.sv_tree_mask(None, ws_ok, big, None) == b.SV_EINVAL
    m0 = b.SvTreeMaskArgs()
    m0.B, m0.N, m0.words = 0, 8, 1
    assert mcall(m0) == b.SV_OK
    m.words = 1  # 40 nodes need two words
    assert mcall(m) == b.SV_EINVAL
    m.words, m.N = 2, b.SV_MAX_TREE_NODES + 1
    assert mcall(m) == b.SV_EINVAL
    m.N, m.parent = 40, None
    assert mcall(m) == b.SV_EINVAL
    m.parent = 0x100000
    assert mcall(m, n=b.SV_MIN_WORKSPACE_BYTES - 1) == b.SV_EWORKSPACE
    assert mcall(m, ws=ctypes.c_void_p(0x200010)) == b.SV_EWORKSPACE
    # row statistics
    al, ex = ctypes.c_void_p(0x300000), ctypes.c_void_p(0x400000)
    scall = lambda a, al=al, ex=ex, ws=ws_ok, n=big: svlib.sv_row_stats(ctypes.byref(a), al, ex,
                                                                        ws, n, None)
    assert svlib.sv_row_stats(None, al, ex, ws_ok, big, None) == b.SV_EINVAL
    assert scall(_chain_args(b, B=0)) == b.SV_OK
    assert scall(_chain_args(b, K=b.SV_MAX_K + 1)) == b.SV_EINVAL
    assert scall(_chain_args(b), ex=None) == b.SV_EINVAL
    assert scall(_chain_args(b), al=None) == b.SV_EINVAL
    assert scall(_chain_args(b, draft_logits=None)) == b.SV_EINVAL
    assert scall(_chain_args(b, temperature=None)) == b.SV_EINVAL
    assert scall(_chain_args(b), n=1024) == b.SV_EWORKSPACE
    assert svlib.sv_get_error(None, None, None) == b.SV_EWORKSPACE
    assert svlib.sv_selftest_wait_timeout(None, 0, 1000, None) == b.SV_EWORKSPACE
    assert svlib.sv_workspace_init(None, 0, None) == b.SV_EWORKSPACE


def test_status_strings(svlib):
    from speculative_decoding_verification_63_gb300 import _binding as b
    names = [b.sv_status_string(s) for s in range(8)]
    assert names[0] == "SV_OK" and all(n.startswith("SV_E") for n in names[1:])
    assert len(set(names)) == 8
    assert names[b.SV_ECORESIDENT].startswith("SV_ECORESIDENT")
    assert b.sv_version() >= 100


def test_status_codes_match_the_header():
    """Every status the header defines (among them SV_ECORESIDENT, the
    answer to a grid that cannot be resident at once) has the same value in
    the binding."""
    import re
    from speculative_decoding_verification_63_gb300 import _binding as b
    text = open(os.path.join(ROOT, "include", "specverify.h")).read()
    enum = dict(re.findall(r"\b(SV_OK|SV_E[A-Z]+)\s*=\s*(\d+)", text))
    assert "SV_ECORESIDENT" in enum and len(enum) == 8
    for name, value in enum.items():
        assert getattr(b, name) == int(value), name


def test_product_has_no_cpu_fallback():
    """The package never imports the oracle, and fails loudly without the
    built library."""
    import speculative_decoding_verification_63_gb300 as pkg
    from speculative_decoding_verification_63_gb300 import _binding
    pkg_dir = os.path.dirname(pkg.__file__)
    for root, _, files in os.walk(pkg_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh")):
                txt = open(os.path.join(root, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", txt, re.M), f
    with pytest.raises(RuntimeError):
        _binding.lib(os.path.join(pkg_dir, "does_not_exist.so"))


def test_nvtx_build_opens_a_range_per_entry_point():
    """The traced build (-DSV_NVTX) wraps every entry point that enqueues
    device work in an NVTX range named after it (preprocessed only: the
    ranges need no GPU)."""
    import re
    import subprocess
    from speculative_decoding_verification_63_gb300 import _build
    src = os.path.join(_build.CSRC, "specverify.cu")
    flags = [f for f in _build.compile_flags(nvtx=True) if f.startswith(("-I", "-D", "-std"))]
    out = subprocess.run([_build.nvcc(), "-E", "-x", "cu", *flags, src], capture_output=True,
                         text=True, check=True).stdout
    for name in ("sv_verify_chain", "sv_verify_tree", "sv_row_stats", "sv_tree_mask",
                 "sv_verify_chain_noalloc", "sv_workspace_init"):
        body = re.search(r"sv_status\s+" + name + r"\s*\([^{]*\{\s*const\s+SvRange\s+sv_range_\s*\(\s*\"" +
                         name + r"\"\s*\)", out)
        assert body, name
    assert "nvtxRangePushA" in out
    plain = subprocess.run([_build.nvcc(), "-E", "-x", "cu",
                            *[f for f in _build.compile_flags() if f.startswith(("-I", "-D", "-std"))],
                            src], capture_output=True, text=True, check=True).stdout
    assert "SvRange" not in plain


def test_checks_build_guards_the_bulk_copies():
    """The debug build (-DSV_CHECKS) guards the bulk copies of the persistent
    kernel, the top-k pass and the tree walk, and the top-k map and piece
    indices, with checks that set SV_DERR_CHECK (preprocessed only: the
    checks need no GPU); the release build has none of them."""
    from speculative_decoding_verification_63_gb300 import _binding, _build
    src = os.path.join(_build.CSRC, "specverify.cu")

    def pre(checks):
        flags = [f for f in _build.compile_flags(checks=checks) if f.startswith(("-I", "-D", "-std"))]
        return subprocess.run([_build.nvcc(), "-E", "-x", "cu", *flags, src], capture_output=True,
                              text=True, check=True).stdout
    debug, release = pre(True), pre(False)
    n_checks = debug.count("::sv::sv_check(")
    assert n_checks >= 6, n_checks
    assert "::sv::sv_check(" not in release
    assert _binding.SV_DERR_CHECK == 0x40
