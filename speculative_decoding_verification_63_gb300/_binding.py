"""ctypes binding of libspecverify (include/specverify.h).

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the cudaStream_t.  Every step of the verification runs in the
library's CUDA kernels; there is no CPU fallback, and every call raises when
the library is missing or returns an error status.
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIBRARY

SV_OK, SV_EINVAL, SV_ECUDA, SV_ETIMEOUT, SV_EDATA, SV_EWORKSPACE, SV_EUNSUPPORTED, SV_ECORESIDENT = range(8)
SV_BF16, SV_FP32 = 0, 1
SV_TREE_MSS, SV_TREE_MSS_NOREPLACE, SV_TREE_NAIVE = 0, 1, 2
TREE_MODES = {"mss": SV_TREE_MSS, "noreplace": SV_TREE_MSS_NOREPLACE, "naive": SV_TREE_NAIVE}
SV_DERR_TOKEN, SV_DERR_NONFINITE, SV_DERR_MASS = 0x01, 0x02, 0x04
SV_DERR_TREE, SV_DERR_TIMEOUT, SV_DERR_ARG = 0x08, 0x10, 0x20
SV_DERR_CHECK = 0x40
SV_MAX_K, SV_MAX_B, SV_MAX_V, SV_MAX_TOPK = 32, 1024, 1 << 20, 64
SV_MAX_TREE_NODES, SV_MAX_TREE_B = 64, 1024

# every symbol include/specverify.h declares
EXPORTS = ("sv_chain_workspace_bytes", "sv_tree_workspace_bytes", "sv_workspace_init",
           "sv_verify_chain", "sv_verify_tree", "sv_get_error", "sv_selftest_wait_timeout",
           "sv_verify_chain_noalloc", "sv_noalloc_get_error", "sv_tree_mask", "sv_row_stats",
           "sv_status_string", "sv_version")
SV_MIN_WORKSPACE_BYTES = 8192
SV_NOALLOC_SCRATCH_BYTES = 8 << 20

_P = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64


class SvChainArgs(ctypes.Structure):
    _fields_ = [("B", _i32), ("K", _i32), ("V", _i32), ("dtype", _i32),
                ("target_logits", _P), ("target_row_stride", _i64),
                ("draft_logits", _P), ("draft_row_stride", _i64),
                ("draft_tokens", _P), ("num_drafts", _P), ("temperature", _P),
                ("top_k", _P), ("max_top_k", _i32), ("uniforms", _P),
                ("out_tokens", _P), ("out_len", _P), ("accept_len", _P),
                ("p_at_draft", _P), ("q_at_draft", _P)]


class SvTreeArgs(ctypes.Structure):
    _fields_ = [("B", _i32), ("N", _i32), ("M", _i32), ("V", _i32), ("max_depth", _i32),
                ("dtype", _i32), ("mode", _i32),
                ("target_logits", _P), ("target_row_stride", _i64),
                ("draft_logits", _P), ("draft_row_stride", _i64),
                ("node_tokens", _P), ("parent", _P), ("q_row", _P), ("num_nodes", _P),
                ("temperature", _P), ("top_k", _P), ("max_top_k", _i32),
                ("u_accept", _P), ("u_sample", _P), ("out_tokens", _P), ("out_len", _P),
                ("accept_len", _P), ("accepted_nodes", _P)]


class SvTreeMaskArgs(ctypes.Structure):
    _fields_ = [("B", _i32), ("N", _i32), ("words", _i32), ("parent", _P), ("num_nodes", _P),
                ("mask", _P), ("depth", _P)]


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, what: str = "", flags: int = 0):
        self.status = status
        self.flags = flags
        msg = sv_status_string(status) if _lib_or_none() else f"status {status}"
        super().__init__(f"{what}: {msg}" + (f" (device flags 0x{flags:x})" if flags else ""))


_lib_handle = None


def _lib_or_none():
    return _lib_handle


def lib(path: str | None = None):
    """Load libspecverify.so.  Raises if it has not been built."""
    global _lib_handle
    if _lib_handle is not None and path is None:
        return _lib_handle
    p = path or LIBRARY
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with __graft_entry__.build() "
                           "(nvcc, sm_103a); there is no CPU fallback")
    h = ctypes.CDLL(p)
    h.sv_chain_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32, _i32]
    h.sv_chain_workspace_bytes.restype = ctypes.c_size_t
    h.sv_tree_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32]
    h.sv_tree_workspace_bytes.restype = ctypes.c_size_t
    h.sv_workspace_init.argtypes = [_P, ctypes.c_size_t, _P]
    h.sv_workspace_init.restype = ctypes.c_int
    h.sv_verify_chain.argtypes = [ctypes.POINTER(SvChainArgs), _P, ctypes.c_size_t, _P]
    h.sv_verify_chain.restype = ctypes.c_int
    h.sv_verify_tree.argtypes = [ctypes.POINTER(SvTreeArgs), _P, ctypes.c_size_t, _P]
    h.sv_verify_tree.restype = ctypes.c_int
    h.sv_get_error.argtypes = [_P, _P, ctypes.POINTER(_i32)]
    h.sv_get_error.restype = ctypes.c_int
    h.sv_selftest_wait_timeout.argtypes = [_P, ctypes.c_size_t, _i64, _P]
    h.sv_selftest_wait_timeout.restype = ctypes.c_int
    h.sv_verify_chain_noalloc.argtypes = [ctypes.POINTER(SvChainArgs), _P]
    h.sv_verify_chain_noalloc.restype = ctypes.c_int
    h.sv_noalloc_get_error.argtypes = [_P, ctypes.POINTER(_i32)]
    h.sv_noalloc_get_error.restype = ctypes.c_int
    h.sv_tree_mask.argtypes = [ctypes.POINTER(SvTreeMaskArgs), _P, ctypes.c_size_t, _P]
    h.sv_tree_mask.restype = ctypes.c_int
    h.sv_row_stats.argtypes = [ctypes.POINTER(SvChainArgs), _P, _P, _P, ctypes.c_size_t, _P]
    h.sv_row_stats.restype = ctypes.c_int
    h.sv_status_string.argtypes = [ctypes.c_int]
    h.sv_status_string.restype = ctypes.c_char_p
    h.sv_version.argtypes = []
    h.sv_version.restype = _i32
    if path is None:
        _lib_handle = h
    return h


# ---------------------------------------------------------------- marshalling

def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libspecverify takes device tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t) -> int:
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_FP32
    raise ValueError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _row_stride(t, rows_per_req: int) -> int:
    """Element stride between consecutive rows of a [B][R][V] tensor whose
    rows are evenly spaced."""
    if t.stride(-1) != 1:
        raise ValueError("logit rows must be contiguous")
    if t.shape[0] > 1 and rows_per_req > 0 and t.stride(0) != rows_per_req * t.stride(1):
        raise ValueError("logit rows must be evenly spaced across requests")
    return t.stride(1)


def _check(t, dtype, shape, what):
    if t is None:
        return
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{what}: expected contiguous {dtype} {tuple(shape)}, "
                         f"got {t.dtype} {tuple(t.shape)}")


def sv_status_string(status: int) -> str:
    return lib().sv_status_string(int(status)).decode()


def sv_version() -> int:
    return lib().sv_version()


def sv_chain_workspace_bytes(B: int, K: int, V: int, dtype: int, max_top_k: int = 0) -> int:
    return lib().sv_chain_workspace_bytes(B, K, V, dtype, max_top_k)


def sv_tree_workspace_bytes(B: int, N: int, M: int, V: int, dtype: int,
                            max_top_k: int = 0) -> int:
    return lib().sv_tree_workspace_bytes(B, N, M, V, dtype, max_top_k)


def sv_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    st = lib().sv_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "sv_workspace_init")


def sv_verify_chain(target_logits, draft_logits, draft_tokens, temperature, uniforms,
                    out_tokens, out_len, accept_len, workspace, num_drafts=None, top_k=None,
                    max_top_k: int = 0, p_at_draft=None, q_at_draft=None, stream=None) -> None:
    """Enqueue sv_verify_chain on the current (or given) stream."""
    B, K1, V = target_logits.shape
    K = K1 - 1
    a = SvChainArgs()
    a.B, a.K, a.V = B, K, V
    a.dtype = _dtype_code(target_logits)
    a.target_logits = _ptr(target_logits)
    a.target_row_stride = _row_stride(target_logits, K1)
    if draft_logits is not None:
        if draft_logits.dtype != target_logits.dtype or tuple(draft_logits.shape) != (B, K, V):
            raise ValueError("draft_logits must be [B][K][V] of the target's dtype")
        if draft_logits.numel() > 0:
            a.draft_logits = _ptr(draft_logits)
            a.draft_row_stride = _row_stride(draft_logits, K)
    _check(draft_tokens, torch.int32, (B, K), "draft_tokens")
    if draft_tokens is not None and draft_tokens.numel() == 0:
        draft_tokens = None
    _check(temperature, torch.float32, (B,), "temperature")
    _check(uniforms, torch.float32, (B, K + 1), "uniforms")
    _check(num_drafts, torch.int32, (B,), "num_drafts")
    _check(top_k, torch.int32, (B,), "top_k")
    _check(out_tokens, torch.int32, (B, K + 1), "out_tokens")
    _check(out_len, torch.int32, (B,), "out_len")
    _check(accept_len, torch.int32, (B,), "accept_len")
    _check(p_at_draft, torch.float32, (B, K), "p_at_draft")
    _check(q_at_draft, torch.float32, (B, K), "q_at_draft")
    a.draft_tokens = _ptr(draft_tokens)
    a.num_drafts = _ptr(num_drafts)
    a.temperature = _ptr(temperature)
    a.top_k = _ptr(top_k)
    a.max_top_k = max_top_k
    a.uniforms = _ptr(uniforms)
    a.out_tokens = _ptr(out_tokens)
    a.out_len = _ptr(out_len)
    a.accept_len = _ptr(accept_len)
    a.p_at_draft = _ptr(p_at_draft)
    a.q_at_draft = _ptr(q_at_draft)
    st = lib().sv_verify_chain(ctypes.byref(a), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "sv_verify_chain")


def sv_verify_tree(target_logits, draft_logits, node_tokens, parent, q_row, temperature,
                   u_accept, u_sample, out_tokens, out_len, accept_len, accepted_nodes,
                   workspace, max_depth: int, num_nodes=None, top_k=None, max_top_k: int = 0,
                   mode: int = SV_TREE_MSS, stream=None) -> None:
    """Enqueue sv_verify_tree on the current (or given) stream."""
    B, N, V = target_logits.shape
    a = SvTreeArgs()
    a.B, a.N, a.V, a.max_depth = B, N, V, max_depth
    a.M = draft_logits.shape[1] if draft_logits is not None else 1
    a.dtype = _dtype_code(target_logits)
    a.mode = mode
    a.target_logits = _ptr(target_logits)
    a.target_row_stride = _row_stride(target_logits, N)
    if draft_logits is not None:
        if draft_logits.dtype != target_logits.dtype or draft_logits.shape[0] != B \
                or draft_logits.shape[2] != V:
            raise ValueError("draft_logits must be [B][M][V] of the target's dtype")
        a.draft_logits = _ptr(draft_logits)
        a.draft_row_stride = _row_stride(draft_logits, a.M)
    for t, dt, shp, nm in [(node_tokens, torch.int32, (B, N), "node_tokens"),
                           (parent, torch.int32, (B, N), "parent"),
                           (q_row, torch.int32, (B, N), "q_row"),
                           (temperature, torch.float32, (B,), "temperature"),
                           (u_accept, torch.float32, (B, N), "u_accept"),
                           (u_sample, torch.float32, (B,), "u_sample"),
                           (num_nodes, torch.int32, (B,), "num_nodes"),
                           (top_k, torch.int32, (B,), "top_k"),
                           (out_tokens, torch.int32, (B, max_depth + 1), "out_tokens"),
                           (out_len, torch.int32, (B,), "out_len"),
                           (accept_len, torch.int32, (B,), "accept_len")]:
        _check(t, dt, shp, nm)
    if accepted_nodes.dtype != torch.int32 or accepted_nodes.shape[0] != B \
            or accepted_nodes.numel() < B * max_depth:
        raise ValueError("accepted_nodes: expected int32 [B][max_depth]")
    a.node_tokens, a.parent, a.q_row = _ptr(node_tokens), _ptr(parent), _ptr(q_row)
    a.num_nodes, a.temperature, a.top_k = _ptr(num_nodes), _ptr(temperature), _ptr(top_k)
    a.max_top_k = max_top_k
    a.u_accept, a.u_sample = _ptr(u_accept), _ptr(u_sample)
    a.out_tokens, a.out_len, a.accept_len = _ptr(out_tokens), _ptr(out_len), _ptr(accept_len)
    a.accepted_nodes = _ptr(accepted_nodes)
    st = lib().sv_verify_tree(ctypes.byref(a), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "sv_verify_tree")


def sv_get_error(workspace, stream=None) -> tuple[int, int]:
    """(status, device flags); synchronises the stream and clears the word."""
    flags = _i32(0)
    st = lib().sv_get_error(_ptr(workspace), _stream(stream), ctypes.byref(flags))
    return st, flags.value


def sv_selftest_wait_timeout(workspace, limit_ns: int, stream=None) -> int:
    return lib().sv_selftest_wait_timeout(_ptr(workspace),
                                          workspace.numel() * workspace.element_size(),
                                          int(limit_ns), _stream(stream))


# ------------------------------------------------ allocation-free chain call

def sv_verify_chain_noalloc(target_logits, draft_logits, draft_tokens, temperature, uniforms,
                            out_tokens, out_len, accept_len, num_drafts=None, top_k=None,
                            max_top_k: int = 0, p_at_draft=None, q_at_draft=None,
                            stream=None) -> None:
    """Enqueue sv_verify_chain_noalloc: the chain verification with the
    library's own per-device scratch (no workspace argument)."""
    B, K1, V = target_logits.shape
    K = K1 - 1
    a = SvChainArgs()
    a.B, a.K, a.V = B, K, V
    a.dtype = _dtype_code(target_logits)
    a.target_logits = _ptr(target_logits)
    a.target_row_stride = _row_stride(target_logits, K1)
    if draft_logits is not None:
        if draft_logits.dtype != target_logits.dtype or tuple(draft_logits.shape) != (B, K, V):
            raise ValueError("draft_logits must be [B][K][V] of the target's dtype")
        if draft_logits.numel() > 0:
            a.draft_logits = _ptr(draft_logits)
            a.draft_row_stride = _row_stride(draft_logits, K)
    if draft_tokens is not None and draft_tokens.numel() == 0:
        draft_tokens = None
    for t, dt, shp, nm in [(draft_tokens, torch.int32, (B, K), "draft_tokens"),
                           (temperature, torch.float32, (B,), "temperature"),
                           (uniforms, torch.float32, (B, K + 1), "uniforms"),
                           (num_drafts, torch.int32, (B,), "num_drafts"),
                           (top_k, torch.int32, (B,), "top_k"),
                           (out_tokens, torch.int32, (B, K + 1), "out_tokens"),
                           (out_len, torch.int32, (B,), "out_len"),
                           (accept_len, torch.int32, (B,), "accept_len"),
                           (p_at_draft, torch.float32, (B, K), "p_at_draft"),
                           (q_at_draft, torch.float32, (B, K), "q_at_draft")]:
        _check(t, dt, shp, nm)
    a.draft_tokens, a.num_drafts = _ptr(draft_tokens), _ptr(num_drafts)
    a.temperature, a.top_k, a.max_top_k = _ptr(temperature), _ptr(top_k), max_top_k
    a.uniforms = _ptr(uniforms)
    a.out_tokens, a.out_len, a.accept_len = _ptr(out_tokens), _ptr(out_len), _ptr(accept_len)
    a.p_at_draft, a.q_at_draft = _ptr(p_at_draft), _ptr(q_at_draft)
    st = lib().sv_verify_chain_noalloc(ctypes.byref(a), _stream(stream))
    if st == SV_EWORKSPACE:
        need = sv_chain_workspace_bytes(B, K, V, a.dtype, max_top_k)
        raise SpecVerifyError(st, f"sv_verify_chain_noalloc: the call needs {need} bytes of "
                                  f"scratch, more than SV_NOALLOC_SCRATCH_BYTES "
                                  f"({SV_NOALLOC_SCRATCH_BYTES}); use sv_verify_chain with a "
                                  "workspace")
    if st != SV_OK:
        raise SpecVerifyError(st, "sv_verify_chain_noalloc")


def sv_noalloc_get_error(stream=None) -> tuple[int, int]:
    """(status, device flags) of the allocation-free scratch of the current
    device; synchronises the stream; re-zeroes the scratch after an error."""
    flags = _i32(0)
    st = lib().sv_noalloc_get_error(_stream(stream), ctypes.byref(flags))
    return st, flags.value


# ------------------------------------------------- tree mask, row statistics

def sv_tree_mask(parent, mask, depth, workspace, num_nodes=None, stream=None) -> None:
    """Enqueue sv_tree_mask: ancestor bitmask rows mask [B][N][words] (int32
    storage of the uint32 words) and depths [B][N] of DFS-linearised trees."""
    B, N = parent.shape
    if mask.dim() != 3 or tuple(mask.shape[:2]) != (B, N):
        raise ValueError("mask: expected [B][N][words]")
    _check(parent, torch.int32, (B, N), "parent")
    _check(num_nodes, torch.int32, (B,), "num_nodes")
    _check(mask, torch.int32, (B, N, mask.shape[2]), "mask")
    _check(depth, torch.int32, (B, N), "depth")
    a = SvTreeMaskArgs()
    a.B, a.N, a.words = B, N, mask.shape[2]
    a.parent, a.num_nodes = _ptr(parent), _ptr(num_nodes)
    a.mask, a.depth = _ptr(mask), _ptr(depth)
    st = lib().sv_tree_mask(ctypes.byref(a), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "sv_tree_mask")


def sv_row_stats(target_logits, draft_logits, temperature, alpha, expected, workspace,
                 num_drafts=None, top_k=None, max_top_k: int = 0, stream=None) -> None:
    """Enqueue sv_row_stats: alpha [B][K] = sum min(p_i, q_i) per position
    and expected [B] tokens per round."""
    B, K1, V = target_logits.shape
    K = K1 - 1
    a = SvChainArgs()
    a.B, a.K, a.V = B, K, V
    a.dtype = _dtype_code(target_logits)
    a.target_logits = _ptr(target_logits)
    a.target_row_stride = _row_stride(target_logits, K1)
    if K > 0:
        if draft_logits is None or draft_logits.dtype != target_logits.dtype \
                or tuple(draft_logits.shape) != (B, K, V):
            raise ValueError("draft_logits must be [B][K][V] of the target's dtype")
        a.draft_logits = _ptr(draft_logits)
        a.draft_row_stride = _row_stride(draft_logits, K)
    _check(temperature, torch.float32, (B,), "temperature")
    _check(num_drafts, torch.int32, (B,), "num_drafts")
    _check(top_k, torch.int32, (B,), "top_k")
    _check(alpha, torch.float32, (B, K), "alpha")
    _check(expected, torch.float32, (B,), "expected")
    a.temperature, a.num_drafts, a.top_k = _ptr(temperature), _ptr(num_drafts), _ptr(top_k)
    a.max_top_k = max_top_k
    st = lib().sv_row_stats(ctypes.byref(a), _ptr(alpha), _ptr(expected), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "sv_row_stats")
