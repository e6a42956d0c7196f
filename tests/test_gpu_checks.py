"""The debug build (-DSV_CHECKS: device-side bounds and alignment checks on
the kernels' own indexing, a failed check setting SV_DERR_CHECK) on the
GPU: the chain path with and without top-k filtering (map groups of 16
and of 32 tokens), unaligned rows and the tree walk, compared with the
fp64 oracle like the release build, and no check may fire."""
import numpy as np
import pytest

import speculative_decoding_verification_63_gb300 as sv
from speculative_decoding_verification_63_gb300 import _binding, _build
from speculative_decoding_verification_63_gb300 import workloads as wl

from gpu_util import check_chain, check_tree

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checks_lib():
    h = _binding.lib(_build.build_library(checks=True))
    old = _binding._lib_handle
    _binding._lib_handle = h
    try:
        yield h
    finally:
        _binding._lib_handle = old


def _flags(kind):
    st, flags = sv.sv_get_error(sv.workspace(1, "cuda", kind))
    return st, flags


@pytest.mark.parametrize("cfg,kw", [
    (3, dict(B=8, V=40000)),
    (5, dict(B=6, K=4, V=40000)),
    (5, dict(B=2, K=2, V=262144)),
    (2, dict(B=3, V=5001)),
])
def test_checks_build_chain(checks_lib, cfg, kw):
    inp = wl.make_chain(cfg, seed=wl.SEED_BASE + 900 + cfg, **kw)
    check_chain(inp)  # raises on any device flag, SV_DERR_CHECK included
    assert _flags("chain") == (sv.SV_OK, 0)


def test_checks_build_tree(checks_lib):
    inp = wl.make_tree(B=4, seed=wl.SEED_BASE + 904)
    check_tree(inp)
    assert _flags("tree") == (sv.SV_OK, 0)
