"""fp64 CPU oracle for MInference-style dynamic sparse prefill attention.

TEST INFRASTRUCTURE ONLY.  This package is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``; the
library's compute path never imports, links or runs it.  It shares no code with
the CUDA library: the arithmetic lives in ``msa_oracle.c`` (plain C, double
precision), and this module only marshals numpy arrays into it.

Every function cites the passage of the source pages it follows (see the
header of ``msa_oracle.c`` for the page list and the readings taken where the
pages are silent).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_LIB = os.path.join(_HERE, "_msa_oracle.so")
_lock = threading.Lock()
_lib = None

ASHAPE, VS, BLOCK, DENSE = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile msa_oracle.c into oracle/_msa_oracle.so with gcc."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Head(ctypes.Structure):
    _fields_ = [("pattern", ctypes.c_int32), ("sink", ctypes.c_int32), ("window", ctypes.c_int32),
                ("block", ctypes.c_int32), ("topk", ctypes.c_int32)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, f64, P = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.ora_num_threads.restype = ctypes.c_int
            lib.ora_set_threads.argtypes = [ctypes.c_int]
            lib.ora_ashape_set.restype = i64
            lib.ora_ashape_set.argtypes = [i64, i64, i64, P]
            lib.ora_vs_logical_set.restype = i64
            lib.ora_vs_logical_set.argtypes = [i64, P, i64, P, i64, P]
            lib.ora_vs_block_index.restype = i64
            lib.ora_vs_block_index.argtypes = [i64, i64, i64, P, i64, P, i64, P, P, P, P]
            lib.ora_vs_physical_set.restype = i64
            lib.ora_vs_physical_set.argtypes = [i64, i64, i64, P, i64, P, i64, P]
            lib.ora_bs_set.restype = i64
            lib.ora_bs_set.argtypes = [i64, i64, i64, P, P, i64, P]
            lib.ora_vs_proxy_probs.argtypes = [i64, i64, i64, f64, P, P, P]
            lib.ora_proxy_aggregate.argtypes = [P, i64, i64, P, P, P, ctypes.c_int32]
            lib.ora_vs_proxy.argtypes = [i64, i64, i64, f64, P, P, P, P, ctypes.c_int32]
            lib.ora_topk.restype = i64
            lib.ora_topk.argtypes = [P, i64, i64, P]
            lib.ora_bs_pool.argtypes = [P, i64, i64, i64, P]
            lib.ora_bs_index.argtypes = [P, P, i64, i64, i64, i64, P, P]
            lib.ora_attend.argtypes = [P, P, P, i64, f64, i64, P, i64, P, P]
            lib.ora_head_rows.argtypes = [P, i64, i64, f64, P, P, P, P, i64, P, i64, P, P, P, i64, P, P, P]
            lib.ora_head_edges.restype = i64
            lib.ora_head_edges.argtypes = [P, i64, P, i64, P, i64, P, P]
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _i32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32).reshape(-1))


def num_threads() -> int:
    """Threads the oracle's parallel loops use."""
    return int(_load().ora_num_threads())


def set_threads(t: int) -> None:
    _load().ora_set_threads(int(t))


# ----------------------------------------------------------------- sets
def ashape_set(i: int, sink: int, window: int) -> np.ndarray:
    """MInference page, eq.(3): N_A(i) = {0..min(g-1,i)} ∪ {max(0,i-w+1)..i}."""
    out = np.empty(int(i) + 1, dtype=np.int64)
    m = _load().ora_ashape_set(int(i), int(sink), int(window), _p(out))
    return out[:m].copy()


def vs_logical_set(i: int, C, D) -> np.ndarray:
    """MInference page, eq.(5): {j in C, j <= i} ∪ {i - δ : δ in D, i - δ >= 0}."""
    C, D = _i32(C), _i32(D)
    out = np.empty(len(C) + len(D) + 1, dtype=np.int64)
    m = _load().ora_vs_logical_set(int(i), _p(C), len(C), _p(D), len(D), _p(out))
    return out[:m].copy()


def vs_block_index(u: int, n: int, block: int, C, D):
    """Per-query-block Vertical-Slash index (MInference page §2.1/§4.1 and the
    MInference blog §2.3.3): merged key ranges [[lo, hi], ...] (inclusive) and
    the vertical columns they leave uncovered."""
    C, D = _i32(C), _i32(D)
    ranges = np.empty(2 * max(len(D), 1), dtype=np.int64)
    cols = np.empty(max(len(C), 1), dtype=np.int64)
    nr = np.zeros(1, dtype=np.int64)
    nc = np.zeros(1, dtype=np.int64)
    _load().ora_vs_block_index(int(u), int(n), int(block), _p(C), len(C), _p(D), len(D), _p(ranges), _p(nr),
                               _p(cols), _p(nc))
    return ranges[:2 * nr[0]].reshape(-1, 2).copy(), cols[:nc[0]].copy()


def vs_physical_set(i: int, n: int, block: int, C, D) -> np.ndarray:
    """Keys row i attends under Vertical-Slash with query blocks of `block` rows."""
    C, D = _i32(C), _i32(D)
    out = np.empty(int(n) + len(C) + 1, dtype=np.int64)
    m = _load().ora_vs_physical_set(int(i), int(n), int(block), _p(C), len(C), _p(D), len(D), _p(out))
    return out[:m].copy()


def bs_set(i: int, n: int, block: int, J, cnt) -> np.ndarray:
    """MInference page eq.(6): keys of the selected blocks J_u with j <= i."""
    J = _i32(J)
    cnt = _i32(cnt)
    kb = J.size // cnt.size
    out = np.empty(int(n) + 1, dtype=np.int64)
    m = _load().ora_bs_set(int(i), int(n), int(block), _p(J), _p(cnt), kb, _p(out))
    return out[:m].copy()


# ----------------------------------------------------------------- proxy / top-k
def vs_proxy_probs(q, k, last_q: int, scale: float) -> np.ndarray:
    """MInference page §6.2: Ã rows for the last `last_q` queries, [L][n] (0 for j > i)."""
    q, k = _f32(q), _f32(k)
    n, d = k.shape
    L = min(int(last_q), n)
    A = np.empty((L, n), dtype=np.float64)
    _load().ora_vs_proxy_probs(n, d, L, float(scale), _p(q), _p(k), _p(A))
    return A


# proxy conventions (bits): column maximum instead of the sum, slash mean instead of the sum
PROXY_SUM, PROXY_COL_MAX, PROXY_SLASH_MEAN = 0, 1, 2


def proxy_aggregate(A, pos, mode: int = PROXY_SUM):
    """MInference page §3.1/§6.2: column sums c_j = Σ_t A[t, j] and slash sums
    r_d = Σ_t A[t, pos[t] - d] of a proxy matrix whose row t is query pos[t]
    (mode: PROXY_COL_MAX takes the column maximum, PROXY_SLASH_MEAN divides each
    slash sum by its number of legal pairs)."""
    A = np.ascontiguousarray(np.asarray(A, dtype=np.float64))
    rows, n = A.shape
    pos = np.ascontiguousarray(np.asarray(pos, dtype=np.int64))
    c = np.empty(n, dtype=np.float64)
    r = np.empty(n, dtype=np.float64)
    _load().ora_proxy_aggregate(_p(A), rows, n, _p(pos), _p(c), _p(r), int(mode))
    return c, r


def vs_proxy(q, k, last_q: int, scale: float, mode: int = PROXY_SUM):
    """Column scores c [n] and slash scores r [n] of one head (fp64)."""
    q, k = _f32(q), _f32(k)
    n, d = k.shape
    c = np.empty(n, dtype=np.float64)
    r = np.empty(n, dtype=np.float64)
    _load().ora_vs_proxy(n, d, min(int(last_q), n), float(scale), _p(q), _p(k), _p(c), _p(r), int(mode))
    return c, r


def topk(score, k: int) -> np.ndarray:
    """Indices of the k largest scores, ties to the lower index, best first."""
    s = np.ascontiguousarray(np.asarray(score, dtype=np.float64))
    out = np.empty(max(min(int(k), s.size), 1), dtype=np.int32)
    m = _load().ora_topk(_p(s), s.size, int(k), _p(out))
    return out[:m].copy()


def vs_index(q, k, last_q: int, n_vertical: int, n_slash: int, scale: float, mode: int = PROXY_SUM):
    """Vertical-Slash index of one head: (C ascending, D descending, c, r)."""
    c, r = vs_proxy(q, k, last_q, scale, mode)
    C = np.sort(topk(c, n_vertical))
    D = np.sort(topk(r, n_slash))[::-1].copy()
    return C, D, c, r


def bs_pool(x, block: int) -> np.ndarray:
    x = _f32(x)
    n, d = x.shape
    nb = (n + block - 1) // block
    out = np.empty((nb, d), dtype=np.float64)
    _load().ora_bs_pool(_p(x), n, d, int(block), _p(out))
    return out


def bs_index(q, k, block: int, topk_blocks: int):
    """Block-sparse index of one head: J [N_b, k_b] ascending (-1 padded), cnt [N_b]."""
    q, k = _f32(q), _f32(k)
    n, d = k.shape
    nb = (n + block - 1) // block
    J = np.empty((nb, int(topk_blocks)), dtype=np.int32)
    cnt = np.empty(nb, dtype=np.int32)
    _load().ora_bs_index(_p(q), _p(k), n, d, int(block), int(topk_blocks), _p(J), _p(cnt))
    return J, cnt


# ----------------------------------------------------------------- attention
def attend(q, k, v, i: int, keyset, scale: float):
    """MInference page eq.(2) over the given key set: (o [d], lse)."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    d = q.shape[1]
    s = np.ascontiguousarray(np.asarray(keyset, dtype=np.int64))
    o = np.empty(d, dtype=np.float64)
    lse = np.empty(1, dtype=np.float64)
    _load().ora_attend(_p(q), _p(k), _p(v), d, float(scale), int(i), _p(s), s.size, _p(o), _p(lse))
    return o, float(lse[0])


def merge(o_a, lse_a, o_b, lse_b):
    """Attention over two disjoint key sets combined into the attention over
    their union (MInference page §3.2, eq.(7)-(8): each part's softmax state is
    its LSE; the union's LSE is log(e^lse_a + e^lse_b) and each part's output is
    weighted by e^(lse_part - lse)).  o_*: [rows, d]; lse_*: [rows]; fp64.
    Empty parts have lse = -inf."""
    o_a, o_b = np.asarray(o_a, np.float64), np.asarray(o_b, np.float64)
    lse_a, lse_b = np.asarray(lse_a, np.float64), np.asarray(lse_b, np.float64)
    m = np.maximum(lse_a, lse_b)
    both_empty = np.isneginf(m)
    ms = np.where(both_empty, 0.0, m)
    wa = np.where(np.isneginf(lse_a), 0.0, np.exp(lse_a - ms))
    wb = np.where(np.isneginf(lse_b), 0.0, np.exp(lse_b - ms))
    s = wa + wb
    lse = np.where(both_empty, -np.inf, ms + np.log(np.where(both_empty, 1.0, s)))
    s = np.where(both_empty, 1.0, s)
    o = (wa / s)[:, None] * o_a + (wb / s)[:, None] * o_b
    return o, lse


def captured_mass(q, k, rows, keysets, scale: float):
    """Mean over the given rows of the dense causal softmax mass that falls in
    each row's key set (MInference page §5.1): Σ_{j in set} p_ij with
    p_ij = e^{s_ij} / Σ_{j' <= i} e^{s_ij'} (fp64, plain loops over rows)."""
    q, k = np.asarray(q, np.float64), np.asarray(k, np.float64)
    total = 0.0
    for i, ks in zip(rows, keysets):
        s = (k[:i + 1] @ q[i]) * scale
        p = np.exp(s - s.max())
        p /= p.sum()
        total += p[np.asarray(ks, np.int64)].sum() if len(ks) else 0.0
    return total / len(rows)


def _head(cfg: dict) -> _Head:
    return _Head(int(cfg["pattern"]), int(cfg.get("sink", 0)), int(cfg.get("window", 0)),
                 int(cfg.get("block", 64)), int(cfg.get("topk", 0)))


def head_rows(cfg: dict, q, k, v, rows, scale: float, C=None, D=None, J=None, cnt=None, want_output=True):
    """Attention output of the given rows of one head under its pattern.

    q, k, v: [n, d] of that head (k, v of its KV head).  Returns (o [rows, d],
    lse [rows], set_size [rows]); o and lse are None when want_output is False.
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    n, d = k.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    C = _i32(C if C is not None else [])
    D = _i32(D if D is not None else [])
    J = _i32(J if J is not None else [])
    cnt = _i32(cnt if cnt is not None else [])
    h = _head(cfg)
    o = np.empty((rows.size, d), dtype=np.float64) if want_output else None
    lse = np.empty(rows.size, dtype=np.float64) if want_output else None
    size = np.empty(rows.size, dtype=np.int64)
    _load().ora_head_rows(ctypes.byref(h), n, d, float(scale), _p(q), _p(k), _p(v), _p(C), C.size, _p(D), D.size,
                          _p(J), _p(cnt), _p(rows), rows.size, _p(o), _p(lse), _p(size))
    return o, lse, size


def head_edges(cfg: dict, n: int, C=None, D=None, J=None, cnt=None) -> int:
    """E_h = Σ_i |N_h(i)| (MInference page eq.(4), any pattern)."""
    C = _i32(C if C is not None else [])
    D = _i32(D if D is not None else [])
    J = _i32(J if J is not None else [])
    cnt = _i32(cnt if cnt is not None else [])
    h = _head(cfg)
    return int(_load().ora_head_edges(ctypes.byref(h), int(n), _p(C), C.size, _p(D), D.size, _p(J), _p(cnt)))
