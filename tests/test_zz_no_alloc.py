"""The allocation-free chain entry point, sv_verify_chain_noalloc, against
the fp64 oracle and against the workspace entry point sv_verify_chain on the
same inputs.

Its scratch is the library's per-device static array; the test checks that
two calls in a row both meet the oracle's parity bar (tests/gpu_util.py)
and give the workspace call's results (tokens and lengths bit for bit,
probabilities within 1e-5 relative), and that a call too large for the
scratch is refused before any device work.  This file is collected last so
that it also runs after every other GPU test.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_63_gb300 as sv
from speculative_decoding_verification_63_gb300 import workloads as wl

from gpu_util import compare

pytestmark = pytest.mark.gpu

RTOL = 1e-5


def _dev(a):
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _outputs(B, K):
    return dict(out_tokens=torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda"),
                out_len=torch.full((B,), -7, dtype=torch.int32, device="cuda"),
                accept_len=torch.full((B,), -7, dtype=torch.int32, device="cuda"),
                p_at=torch.zeros((B, K), dtype=torch.float32, device="cuda"),
                q_at=torch.zeros((B, K), dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("cfg,B", [(3, 16), (2, 8)])
def test_noalloc_matches_workspace_entry(cfg, B):
    inp = wl.make_chain(cfg, B=B, seed=wl.SEED_BASE + 900 + cfg)
    K = inp["K"]
    d = {k: _dev(inp[k]) for k in ("target", "draft", "tokens", "temperature", "uniforms",
                                   "num_drafts")}
    ref = sv.verify_chain(d["target"], d["draft"], d["tokens"], d["temperature"],
                          d["uniforms"], num_drafts=d["num_drafts"], with_probs=True)
    torch.cuda.synchronize()
    sv.check_device_errors(sv.workspace(1, "cuda", "chain"))
    want = oracle.verify_chain_inputs(inp)
    for call in range(2):
        o = _outputs(B, K)
        sv.sv_verify_chain_noalloc(d["target"], d["draft"], d["tokens"], d["temperature"],
                                   d["uniforms"], o["out_tokens"], o["out_len"],
                                   o["accept_len"], num_drafts=d["num_drafts"],
                                   p_at_draft=o["p_at"], q_at_draft=o["q_at"])
        st, flags = sv.sv_noalloc_get_error()
        assert st == sv.SV_OK, (call, st, flags)
        got = {k: v.cpu().numpy() for k, v in o.items()}
        got["p_at_draft"], got["q_at_draft"] = got.pop("p_at"), got.pop("q_at")
        compare(got, want, K + 1, prefix_tokens=inp["tokens"], V=inp["V"])
        for k in ("out_tokens", "out_len", "accept_len"):
            assert torch.equal(o[k], ref[k]), (call, k)
        for k, rk in (("p_at", "p_at_draft"), ("q_at", "q_at_draft")):
            a, b = o[k].cpu().numpy(), ref[rk].cpu().numpy()
            fin = np.isfinite(b)
            np.testing.assert_allclose(a[fin], b[fin], rtol=RTOL, atol=1e-30)
            assert np.array_equal(np.isnan(a), np.isnan(b))


def test_noalloc_refuses_calls_beyond_its_scratch():
    B, K, V = sv.SV_MAX_B, 16, 1 << 18
    need = sv.sv_chain_workspace_bytes(B, K, V, sv.SV_BF16, 0)
    assert need > sv.SV_NOALLOC_SCRATCH_BYTES
    # shapes only (the call is refused before the data is looked at): one row, expanded
    row = torch.zeros((1, 1, V), dtype=torch.bfloat16, device="cuda")
    t = row.expand(B, K + 1, V)
    dft = row.expand(B, K, V)
    o = _outputs(B, K)
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.sv_verify_chain_noalloc(t, dft, torch.zeros((B, K), dtype=torch.int32, device="cuda"),
                                   torch.ones(B, dtype=torch.float32, device="cuda"),
                                   torch.zeros((B, K + 1), dtype=torch.float32, device="cuda"),
                                   o["out_tokens"], o["out_len"], o["accept_len"])
    assert e.value.status == sv.SV_EWORKSPACE
    assert "SV_NOALLOC_SCRATCH_BYTES" in str(e.value)
