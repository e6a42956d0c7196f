"""fp64 CPU oracle for the speculative-sampling verification step.

TEST INFRASTRUCTURE ONLY.  The oracle is the plain definition of what the
verification step computes, written out in C (sv_oracle.c) with fp64 loops,
and loaded here through ctypes.  Only the tests, the package smoke check and
the benchmark's CPU-baseline leg may import this package; the product path
never does.  It shares no code with the CUDA library.

Every oracle function is pinned by tests/test_oracle_*.py against values the
pages print, closed forms, exact enumeration and brute force (see the
docstrings there for which pin covers which function).

Sources are cited in sv_oracle.c; the short names used here are
[L17] (CMU 15-779 Lecture 17 notes, Speculative Decoding), [S14]
(llminference "Speculative decoding" tutorial), [N02] ("LLM speculative
decoding study notes 02") and [DVP] ("Speculative decoding: draft, verify
and payoff").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "sv_oracle.c")
LIBRARY = os.path.join(_HERE, "libsv_oracle.so")

# oracle status codes (mirror the #defines in sv_oracle.c)
OK, ENONFINITE, ETOKEN, EMASS, ETREE, EARG = 0, 1, 2, 3, 4, 5

# Relative distance from a decision boundary below which a decision is
# "near": an accept test with |u q - p| / q < NEAR, or an inverse-CDF draw
# whose u S lies within NEAR S of a CDF step.  For such draws the batch
# functions also report the range of tokens a target perturbed by up to
# NEAR S can give (draw_lo .. draw_hi).
NEAR = 1e-6

_lock = threading.Lock()
_lib = None


def build(force: bool = False, source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile the oracle with gcc (-O2, plain C11, no vector intrinsics)."""
    if force or not os.path.exists(output) or (
            os.path.getmtime(output) < os.path.getmtime(source)):
        tmp = output + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp,
                        source, "-lm"], check=True)
        os.replace(tmp, output)
    return output


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


_P = ctypes.c_void_p


def _declare(lib):
    lib.svo_row_probs.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                  ctypes.c_int, _P]
    lib.svo_row_probs.restype = ctypes.c_int
    lib.svo_row_argmax.argtypes = [_P, ctypes.c_int, ctypes.c_int]
    lib.svo_row_argmax.restype = ctypes.c_int
    lib.svo_residual.argtypes = [_P, _P, ctypes.c_int, _P]
    lib.svo_residual.restype = ctypes.c_double
    lib.svo_icdf.argtypes = [_P, ctypes.c_int, ctypes.c_double, _P]
    lib.svo_icdf.restype = ctypes.c_int
    lib.svo_icdf_window.argtypes = [_P, ctypes.c_int, ctypes.c_double, ctypes.c_double, _P, _P]
    lib.svo_icdf_window.restype = ctypes.c_int
    lib.svo_verify_chain.argtypes = ([ctypes.c_int] * 4 + [_P] * 7 + [_P] * 8 +
                                     [ctypes.c_double, _P, _P])
    lib.svo_verify_chain.restype = ctypes.c_int
    lib.svo_verify_tree.argtypes = ([ctypes.c_int] * 7 + [_P] * 10 + [_P] * 7 +
                                    [ctypes.c_double, _P, _P, _P])
    lib.svo_verify_tree.restype = ctypes.c_int
    lib.svo_tree_mask.argtypes = [ctypes.c_int] * 3 + [_P] * 5
    lib.svo_tree_mask.restype = ctypes.c_int
    lib.svo_row_stats.argtypes = [ctypes.c_int] * 4 + [_P] * 8
    lib.svo_row_stats.restype = ctypes.c_int
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a):
    """(dtype code, contiguous array): uint16 arrays are bf16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return 0, a
    if a.dtype == np.float32:
        return 1, a
    return 1, np.ascontiguousarray(a, dtype=np.float32)


# ------------------------------------------------------------ single pieces

def row_probs(row, temperature: float, top_k: int = 0, lib=None):
    """p = decoding distribution of one logit row (fp64).  Returns (status, p)."""
    lib = lib or load()
    dt, row = _logits(row)
    V = row.shape[-1]
    p = np.zeros(V, dtype=np.float64)
    st = lib.svo_row_probs(_ptr(row), dt, V, float(temperature), int(top_k), _ptr(p))
    return st, p


def row_argmax(row, lib=None) -> int:
    lib = lib or load()
    dt, row = _logits(row)
    return lib.svo_row_argmax(_ptr(row), dt, row.shape[-1])


def residual(p, q, lib=None):
    """(w, S): w = max(0, p - q), S = sum w."""
    lib = lib or load()
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    w = np.zeros_like(p)
    S = lib.svo_residual(_ptr(p), _ptr(q), p.shape[0], _ptr(w))
    return w, S


def icdf(w, u: float, lib=None):
    """(token, margin) of the inverse-CDF draw from weights w with uniform u."""
    lib = lib or load()
    w = np.ascontiguousarray(w, dtype=np.float64)
    m = np.zeros(1, dtype=np.float64)
    t = lib.svo_icdf(_ptr(w), w.shape[0], float(u), _ptr(m))
    return t, float(m[0])


def icdf_window(w, u: float, radius: float, lib=None):
    """(lo, hi, count): the ids of the first and last positive-weight token
    whose CDF step meets [u S - radius S, u S + radius S], and how many
    positive-weight tokens lie between them (see svo_icdf_window)."""
    lib = lib or load()
    w = np.ascontiguousarray(w, dtype=np.float64)
    lo = np.zeros(1, dtype=np.int32)
    hi = np.zeros(1, dtype=np.int32)
    n = lib.svo_icdf_window(_ptr(w), w.shape[0], float(u), float(radius), _ptr(lo), _ptr(hi))
    return int(lo[0]), int(hi[0]), int(n)


# ------------------------------------------------------------------- chain

def verify_chain(target, draft, tokens, temperature, uniforms,
                 num_drafts=None, top_k=None, lib=None, near: float = NEAR) -> dict:
    """Chain verification of a batch (see svo_verify_chain in sv_oracle.c).

    target [B][K+1][V], draft [B][K][V] (uint16 bf16 bits or float32),
    tokens [B][K], temperature [B], uniforms [B][K+1]; optional
    num_drafts [B] and top_k [B].
    """
    lib = lib or load()
    dt, target = _logits(target)
    dt2, draft = _logits(draft)
    assert dt == dt2
    B, K1, V = target.shape
    K = K1 - 1
    assert draft.shape == (B, K, V)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, K)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, K + 1)
    nd = None if num_drafts is None else np.ascontiguousarray(num_drafts, dtype=np.int32)
    tk = None if top_k is None else np.ascontiguousarray(top_k, dtype=np.int32)
    out = dict(out_tokens=np.zeros((B, K + 1), np.int32), out_len=np.zeros(B, np.int32),
               accept_len=np.zeros(B, np.int32), p_at=np.zeros((B, K)),
               q_at=np.zeros((B, K)), margin_accept=np.zeros(B), margin_draw=np.zeros(B),
               status=np.zeros(B, np.int32), draw_lo=np.zeros(B, np.int32),
               draw_hi=np.zeros(B, np.int32))
    lib.svo_verify_chain(B, K, V, dt, _ptr(target), _ptr(draft), _ptr(tokens), _ptr(nd),
                         _ptr(temperature), _ptr(tk), _ptr(uniforms),
                         _ptr(out["out_tokens"]), _ptr(out["out_len"]),
                         _ptr(out["accept_len"]), _ptr(out["p_at"]), _ptr(out["q_at"]),
                         _ptr(out["margin_accept"]), _ptr(out["margin_draw"]),
                         _ptr(out["status"]), float(near), _ptr(out["draw_lo"]),
                         _ptr(out["draw_hi"]))
    out["margin"] = np.minimum(out["margin_accept"], out["margin_draw"])
    out["margin_walk"] = np.full(B, np.inf)
    return out


def verify_chain_inputs(inp: dict, requests=None, lib=None) -> dict:
    """verify_chain on a workloads.make_chain() dict, optionally on a subset
    of requests (rows are sliced, the computation per request is unchanged)."""
    sel = slice(None) if requests is None else np.asarray(requests)
    return verify_chain(inp["target"][sel], inp["draft"][sel], inp["tokens"][sel],
                        inp["temperature"][sel], inp["uniforms"][sel],
                        num_drafts=inp["num_drafts"][sel], top_k=inp["top_k"][sel],
                        lib=lib)


# -------------------------------------------------------------------- tree

TREE_MODES = {"mss": 0, "noreplace": 1, "naive": 2}


def verify_tree(target, draft, node_tokens, parent, q_row, temperature,
                u_accept, u_sample, num_nodes=None, top_k=None, max_depth=None,
                mode: str = "mss", lib=None, near: float = NEAR) -> dict:
    """Token-tree verification (VerifyGreedy, and MSS, MSS without
    replacement or naive sampling by `mode`), see svo_verify_tree."""
    lib = lib or load()
    dt, target = _logits(target)
    dt2, draft = _logits(draft)
    assert dt == dt2
    B, N, V = target.shape
    M = draft.shape[1]
    i32 = lambda a: np.ascontiguousarray(a, dtype=np.int32)
    node_tokens, parent, q_row = i32(node_tokens), i32(parent), i32(q_row)
    nn = None if num_nodes is None else i32(num_nodes)
    tk = None if top_k is None else i32(top_k)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    u_accept = np.ascontiguousarray(u_accept, dtype=np.float32)
    u_sample = np.ascontiguousarray(u_sample, dtype=np.float32)
    if max_depth is None:
        max_depth = N - 1
    out = dict(out_tokens=np.zeros((B, max_depth + 1), np.int32),
               out_len=np.zeros(B, np.int32), accept_len=np.zeros(B, np.int32),
               accepted_nodes=np.zeros((B, max(max_depth, 1)), np.int32),
               margin_accept=np.zeros(B), margin_draw=np.zeros(B),
               status=np.zeros(B, np.int32), margin_walk=np.zeros(B),
               draw_lo=np.zeros(B, np.int32), draw_hi=np.zeros(B, np.int32))
    lib.svo_verify_tree(B, N, M, V, dt, max_depth, TREE_MODES[mode], _ptr(target),
                        _ptr(draft),
                        _ptr(node_tokens), _ptr(parent), _ptr(q_row), _ptr(nn),
                        _ptr(temperature), _ptr(tk), _ptr(u_accept), _ptr(u_sample),
                        _ptr(out["out_tokens"]), _ptr(out["out_len"]),
                        _ptr(out["accept_len"]), _ptr(out["accepted_nodes"]),
                        _ptr(out["margin_accept"]), _ptr(out["margin_draw"]),
                        _ptr(out["status"]), float(near), _ptr(out["margin_walk"]),
                        _ptr(out["draw_lo"]), _ptr(out["draw_hi"]))
    out["margin"] = np.minimum(out["margin_accept"], out["margin_draw"])
    if max_depth == 0:
        out["accepted_nodes"] = out["accepted_nodes"][:, :0]
    return out


def verify_tree_inputs(inp: dict, requests=None, mode: str | None = None, lib=None) -> dict:
    sel = slice(None) if requests is None else np.asarray(requests)
    return verify_tree(inp["target"][sel], inp["draft"][sel], inp["node_tokens"][sel],
                       inp["parent"][sel], inp["q_row"][sel], inp["temperature"][sel],
                       inp["u_accept"][sel], inp["u_sample"][sel],
                       num_nodes=inp["num_nodes"][sel], top_k=inp["top_k"][sel],
                       max_depth=inp["max_depth"],
                       mode=mode if mode is not None else inp.get("mode", "mss"), lib=lib)


# ------------------------------------------------------- tree attention mask

def tree_mask(parent, num_nodes=None, words: int | None = None, lib=None) -> dict:
    """Ancestor bitmask rows and depths of DFS-linearised trees, see
    svo_tree_mask.  Returns mask [B][N][words] uint32, depth [B][N], status."""
    lib = lib or load()
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    B, N = parent.shape
    W = (N + 31) // 32 if words is None else words
    nn = None if num_nodes is None else np.ascontiguousarray(num_nodes, dtype=np.int32)
    out = dict(mask=np.zeros((B, N, W), np.uint32), depth=np.zeros((B, N), np.int32),
               status=np.zeros(B, np.int32))
    lib.svo_tree_mask(B, N, W, _ptr(parent), _ptr(nn), _ptr(out["mask"]),
                      _ptr(out["depth"]), _ptr(out["status"]))
    return out


# --------------------------------------------------- per-position statistics

def row_stats(target, draft, temperature, num_drafts=None, top_k=None, lib=None) -> dict:
    """alpha_i = sum min(p_i, q_i) per position and the expected tokens
    per round, see svo_row_stats."""
    lib = lib or load()
    dt, target = _logits(target)
    dt2, draft = _logits(draft)
    assert dt == dt2
    B, R, V = target.shape
    K = R - 1
    assert draft.shape[:2] == (B, K)
    nd = None if num_drafts is None else np.ascontiguousarray(num_drafts, dtype=np.int32)
    tk = None if top_k is None else np.ascontiguousarray(top_k, dtype=np.int32)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    out = dict(alpha=np.zeros((B, K)), expected=np.zeros(B), status=np.zeros(B, np.int32))
    lib.svo_row_stats(B, K, V, dt, _ptr(target), _ptr(draft), _ptr(nd), _ptr(temperature),
                      _ptr(tk), _ptr(out["alpha"]), _ptr(out["expected"]),
                      _ptr(out["status"]))
    return out


def row_stats_inputs(inp: dict, lib=None) -> dict:
    return row_stats(inp["target"], inp["draft"], inp["temperature"],
                     num_drafts=inp["num_drafts"], top_k=inp["top_k"], lib=lib)
