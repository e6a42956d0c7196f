"""GB300 (sm_103a) speculative-sampling verification step.

The computation runs in libspecverify.so (hand-written CUDA for sm_103a,
C ABI in include/specverify.h).  This package holds the ctypes binding
(_binding), the build (_build), the seeded synthetic workloads (workloads)
and a thin convenience layer that allocates outputs and workspaces with
torch and calls the C ABI.  There is no CPU fallback: without the built
library every call raises.
"""
from __future__ import annotations

import threading

import torch

from ._binding import (  # noqa: F401
    EXPORTS, SV_BF16, SV_DERR_ARG, SV_DERR_CHECK, SV_DERR_MASS, SV_DERR_NONFINITE, SV_DERR_TIMEOUT,
    SV_DERR_TOKEN, SV_DERR_TREE, SV_ECORESIDENT, SV_EDATA, SV_EINVAL, SV_ETIMEOUT, SV_EUNSUPPORTED,
    SV_EWORKSPACE, SV_FP32, SV_MAX_B, SV_MAX_K, SV_MAX_TOPK, SV_MAX_TREE_B,
    SV_MAX_TREE_NODES, SV_MAX_V, SV_OK, SpecVerifyError, lib, sv_chain_workspace_bytes,
    sv_get_error, sv_selftest_wait_timeout, sv_status_string, sv_tree_workspace_bytes,
    sv_verify_chain, sv_verify_tree, sv_version, sv_workspace_init,
    SV_NOALLOC_SCRATCH_BYTES, sv_noalloc_get_error, sv_verify_chain_noalloc,
    SV_TREE_MSS, SV_TREE_MSS_NOREPLACE, SV_TREE_NAIVE, TREE_MODES, SV_MIN_WORKSPACE_BYTES,
    sv_tree_mask, sv_row_stats)
from ._build import build_library  # noqa: F401

_ws_lock = threading.Lock()
_ws_cache: dict = {}


def workspace(nbytes: int, device=None, key=None) -> torch.Tensor:
    """A zeroed, 256-byte aligned device workspace of at least nbytes,
    cached per (device, key).  Calls sharing one workspace must not overlap
    on the GPU."""
    device = torch.device(device if device is not None else "cuda")
    if device.index is None:
        device = torch.device("cuda", torch.cuda.current_device())
    k = (device, key)
    with _ws_lock:
        buf = _ws_cache.get(k)
        if buf is None or buf.numel() < nbytes:
            buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
            if buf.data_ptr() % 256:
                raise RuntimeError("torch returned a workspace that is not 256-byte aligned")
            sv_workspace_init(buf)
            _ws_cache[k] = buf
        return buf


def dtype_code(t: torch.Tensor) -> int:
    return SV_BF16 if t.dtype == torch.bfloat16 else SV_FP32


def verify_chain(target_logits, draft_logits, draft_tokens, temperature, uniforms,
                 num_drafts=None, top_k=None, max_top_k: int | None = None,
                 with_probs: bool = False, ws: torch.Tensor | None = None) -> dict:
    """Chain verification of a batch on the current stream (asynchronous).

    target_logits [B][K+1][V] and draft_logits [B][K][V] (bf16 or fp32),
    draft_tokens [B][K] int32, temperature [B] fp32 (0 = greedy), uniforms
    [B][K+1] fp32; optional num_drafts [B] int32 and top_k [B] int32.
    Returns device tensors out_tokens [B][K+1], out_len [B], accept_len [B]
    (and p_at_draft, q_at_draft [B][K] when with_probs)."""
    B, K1, V = target_logits.shape
    K = K1 - 1
    dev = target_logits.device
    if max_top_k is None:
        max_top_k = 0 if top_k is None else SV_MAX_TOPK
    out = dict(out_tokens=torch.empty((B, K1), dtype=torch.int32, device=dev),
               out_len=torch.empty(B, dtype=torch.int32, device=dev),
               accept_len=torch.empty(B, dtype=torch.int32, device=dev))
    if with_probs:
        out["p_at_draft"] = torch.empty((B, K), dtype=torch.float32, device=dev)
        out["q_at_draft"] = torch.empty((B, K), dtype=torch.float32, device=dev)
    need = sv_chain_workspace_bytes(B, K, V, dtype_code(target_logits), max_top_k)
    if need == 0:
        raise SpecVerifyError(SV_EINVAL, "verify_chain (sizes)")
    if ws is None:
        ws = workspace(need, dev, "chain")
    sv_verify_chain(target_logits, draft_logits, draft_tokens, temperature, uniforms,
                    out["out_tokens"], out["out_len"], out["accept_len"], ws,
                    num_drafts=num_drafts, top_k=top_k, max_top_k=max_top_k,
                    p_at_draft=out.get("p_at_draft"), q_at_draft=out.get("q_at_draft"))
    return out


def verify_tree(target_logits, draft_logits, node_tokens, parent, q_row, temperature,
                u_accept, u_sample, max_depth: int, num_nodes=None,
                ws: torch.Tensor | None = None, mode: str = "mss") -> dict:
    """Token-tree verification on the current stream: VerifyGreedy for
    temperature 0, otherwise the stochastic rule `mode` ("mss", "noreplace"
    for children drawn without replacement, or "naive" sampling).
    Returns out_tokens [B][max_depth+1], out_len, accept_len and
    accepted_nodes [B][max_depth] (device tensors)."""
    B, N, V = target_logits.shape
    M = draft_logits.shape[1] if draft_logits is not None else 1
    dev = target_logits.device
    out = dict(out_tokens=torch.empty((B, max_depth + 1), dtype=torch.int32, device=dev),
               out_len=torch.empty(B, dtype=torch.int32, device=dev),
               accept_len=torch.empty(B, dtype=torch.int32, device=dev),
               accepted_nodes=torch.empty((B, max(max_depth, 1)), dtype=torch.int32,
                                          device=dev))
    need = sv_tree_workspace_bytes(B, N, M, V, dtype_code(target_logits), 0)
    if need == 0:
        raise SpecVerifyError(SV_EINVAL, "verify_tree (sizes)")
    if ws is None:
        ws = workspace(need, dev, "tree")
    sv_verify_tree(target_logits, draft_logits, node_tokens, parent, q_row, temperature,
                   u_accept, u_sample, out["out_tokens"], out["out_len"], out["accept_len"],
                   out["accepted_nodes"], ws, max_depth=max_depth, num_nodes=num_nodes,
                   mode=TREE_MODES[mode])
    if max_depth == 0:
        out["accepted_nodes"] = out["accepted_nodes"][:, :0]
    return out


def tree_mask(parent, num_nodes=None, words: int | None = None,
              ws: torch.Tensor | None = None) -> dict:
    """Tree-attention mask and depth position ids of DFS-linearised trees
    (parent [B][N] int32 on the device).  Returns mask [B][N][words] (the
    uint32 words in int32 storage: bit j of row i set iff j is i or an
    ancestor of i) and depth [B][N] (device tensors)."""
    B, N = parent.shape
    W = (N + 31) // 32 if words is None else words
    dev = parent.device
    out = dict(mask=torch.empty((B, N, W), dtype=torch.int32, device=dev),
               depth=torch.empty((B, N), dtype=torch.int32, device=dev))
    if ws is None:
        ws = workspace(SV_MIN_WORKSPACE_BYTES, dev, "mask")
    sv_tree_mask(parent, out["mask"], out["depth"], ws, num_nodes=num_nodes)
    return out


def row_stats(target_logits, draft_logits, temperature, num_drafts=None, top_k=None,
              ws: torch.Tensor | None = None, max_top_k: int | None = None) -> dict:
    """Per-position acceptance rates alpha [B][K] (sum min(p_i, q_i), over
    the top-k sets of filtered requests) and the expected tokens per round
    [B] of a chain batch (device tensors)."""
    B, K1, V = target_logits.shape
    K = K1 - 1
    dev = target_logits.device
    if max_top_k is None:
        max_top_k = 0 if top_k is None else SV_MAX_TOPK
    out = dict(alpha=torch.empty((B, K), dtype=torch.float32, device=dev),
               expected=torch.empty(B, dtype=torch.float32, device=dev))
    if ws is None:
        ws = workspace(sv_chain_workspace_bytes(max(B, 1), K, V, dtype_code(target_logits),
                                                max_top_k), dev, "chain")
    sv_row_stats(target_logits, draft_logits, temperature, out["alpha"], out["expected"], ws,
                 num_drafts=num_drafts, top_k=top_k, max_top_k=max_top_k)
    return out


def check_device_errors(ws: torch.Tensor) -> None:
    """Synchronise and raise if the last calls on `ws` recorded a device
    error (the workspace is re-initialised in that case)."""
    st, flags = sv_get_error(ws)
    if st != SV_OK:
        sv_workspace_init(ws)
        raise SpecVerifyError(st, "device", flags)
