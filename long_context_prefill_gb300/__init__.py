"""Python binding of libmsa (MInference-style dynamic sparse prefill attention
on sm_103a).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  There is no fallback:
if ``libmsa.so`` is missing or cannot be loaded, every call raises.

Function names mirror the C ABI in ``include/msa.h`` without the ``msa_``
prefix.  Tensors: Q/O [B,Hq,n,d] bf16, K/V [B,Hkv,n,d] bf16 (contiguous, on
the current CUDA device); ``heads`` is a list of query-head indices.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmsa.so")

MSA_OK, MSA_ERR_INVALID_ARG, MSA_ERR_UNSUPPORTED, MSA_ERR_WORKSPACE_TOO_SMALL = 0, 1, 2, 3
MSA_ERR_CUDA, MSA_ERR_DEVICE_TIMEOUT, MSA_ERR_INDEX = 4, 5, 6
ASHAPE, VS, BLOCK = 0, 1, 2
PATTERNS = {"ashape": ASHAPE, "vs": VS, "block": BLOCK}

EXPORTS = ("msa_status_string", "msa_vs_index_workspace", "msa_block_index_workspace", "msa_layer_workspace",
           "msa_build_vs_index", "msa_build_block_index", "msa_attn_ashape", "msa_attn_vs", "msa_attn_block",
           "msa_prefill_layer", "msa_layer_index", "msa_layer_attend", "msa_kernel_launches", "msa_layer_indices",
           "msa_vs_expand", "msa_poll_device_status", "msa_build_block_index_static",
           "msa_check_wait_timeout", "msa_attn_dense", "msa_layer_varlen_workspace", "msa_prefill_layer_varlen",
           "msa_layer_attend_rows", "msa_merge_attention", "msa_captured_mass", "msa_layer_varlen_indices",
           "msa_layer_attend_stats")


class MsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("n", ctypes.c_int32),
                ("d_h", ctypes.c_int32), ("scale", ctypes.c_float)]


class HeadCfg(ctypes.Structure):
    _fields_ = [("pattern", ctypes.c_int32), ("sink", ctypes.c_int32), ("window", ctypes.c_int32),
                ("last_q", ctypes.c_int32), ("n_vertical", ctypes.c_int32), ("n_slash", ctypes.c_int32),
                ("block", ctypes.c_int32), ("topk", ctypes.c_int32), ("proxy", ctypes.c_int32)]


class VSIndexC(ctypes.Structure):
    _fields_ = [("vertical", ctypes.c_void_p), ("vertical_cnt", ctypes.c_void_p), ("slash", ctypes.c_void_p),
                ("slash_cnt", ctypes.c_void_p), ("vertical_bits", ctypes.c_void_p), ("slash_bits", ctypes.c_void_p),
                ("slash_cover", ctypes.c_void_p), ("v_cap", ctypes.c_int32), ("s_cap", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH):
    """Load libmsa.so (raises if it is missing: there is no CPU fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"libmsa.so not built ({path}); run __graft_entry__.build()")
            lib = ctypes.CDLL(path)
            P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            st = ctypes.c_int
            lib.msa_status_string.restype = ctypes.c_char_p
            lib.msa_status_string.argtypes = [st]
            lib.msa_vs_index_workspace.restype = sz
            lib.msa_vs_index_workspace.argtypes = [P, P, i32]
            lib.msa_block_index_workspace.restype = sz
            lib.msa_block_index_workspace.argtypes = [P, i32, i32]
            lib.msa_layer_workspace.restype = sz
            lib.msa_layer_workspace.argtypes = [P, P]
            lib.msa_build_vs_index.restype = st
            lib.msa_build_vs_index.argtypes = [P, P, P, P, i32, P, P, P, sz, P]
            lib.msa_build_block_index.restype = st
            lib.msa_build_block_index.argtypes = [P, P, P, P, i32, i32, i32, P, P, P, sz, P]
            lib.msa_attn_ashape.restype = st
            lib.msa_attn_ashape.argtypes = [P, P, P, P, P, i32, i32, i32, P, P, P, P]
            lib.msa_attn_vs.restype = st
            lib.msa_attn_vs.argtypes = [P, P, P, P, P, i32, i32, P, P, P, P, P]
            lib.msa_attn_block.restype = st
            lib.msa_attn_block.argtypes = [P, P, P, P, P, i32, i32, i32, P, P, P, P, P, P]
            lib.msa_prefill_layer.restype = st
            lib.msa_prefill_layer.argtypes = [P, P, P, P, P, P, P, P, P, sz, P]
            lib.msa_layer_index.restype = st
            lib.msa_layer_index.argtypes = [P, P, P, P, P, sz, P]
            lib.msa_layer_attend.restype = st
            lib.msa_layer_attend.argtypes = [P, P, P, P, P, P, P, P, P, sz, P]
            lib.msa_kernel_launches.restype = ctypes.c_uint64
            lib.msa_kernel_launches.argtypes = []
            lib.msa_layer_indices.restype = st
            lib.msa_layer_indices.argtypes = [P, P, P, P, P, P]
            lib.msa_vs_expand.restype = st
            lib.msa_vs_expand.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P]
            lib.msa_poll_device_status.restype = st
            lib.msa_poll_device_status.argtypes = [P]
            lib.msa_attn_dense.restype = st
            lib.msa_attn_dense.argtypes = [P, P, P, P, P, i32, P, P, P, P]
            lib.msa_check_wait_timeout.restype = st
            lib.msa_check_wait_timeout.argtypes = [i32, P]
            lib.msa_layer_varlen_workspace.restype = sz
            lib.msa_layer_varlen_workspace.argtypes = [P, P, P, i32]
            lib.msa_prefill_layer_varlen.restype = st
            lib.msa_prefill_layer_varlen.argtypes = [P, P, i32, P, P, P, P, P, P, P, P, sz, P]
            lib.msa_layer_attend_stats.restype = st
            lib.msa_layer_attend_stats.argtypes = [P, P, P, P, P, P, P, P, P, P, sz, P]
            lib.msa_layer_varlen_indices.restype = st
            lib.msa_layer_varlen_indices.argtypes = [P, P, P, i32, P, i32, P, P, P]
            lib.msa_layer_attend_rows.restype = st
            lib.msa_layer_attend_rows.argtypes = [P, P, P, P, P, P, P, P, P, sz, i32, i32, P]
            lib.msa_merge_attention.restype = st
            lib.msa_merge_attention.argtypes = [ctypes.c_int64, i32, P, P, P, P, P, P, P]
            lib.msa_captured_mass.restype = st
            lib.msa_captured_mass.argtypes = [ctypes.c_int64, ctypes.c_int64, P, P, P, P]
            lib.msa_build_block_index_static.restype = st
            lib.msa_build_block_index_static.argtypes = [P, P, P, P, i32, i32, i32, P, P, P]
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().msa_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != MSA_OK:
        raise MsaError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _heads(heads):
    arr = (ctypes.c_int32 * len(heads))(*[int(h) for h in heads])
    return arr, len(heads)


def make_shape(q: torch.Tensor, k: torch.Tensor, scale: float | None = None) -> Shape:
    B, Hq, n, d = q.shape
    return Shape(B, Hq, k.shape[1], n, d, float(scale) if scale else 0.0)


def head_cfg(entry: dict) -> HeadCfg:
    """A config-table entry from a dict: pattern 'ashape' | 'vs' | 'block' plus its budgets."""
    pat = entry["pattern"]
    pat = PATTERNS[pat] if isinstance(pat, str) else int(pat)
    return HeadCfg(pat, int(entry.get("sink", 0)), int(entry.get("window", 1)), int(entry.get("last_q", 64)),
                   int(entry.get("n_vertical", 0)), int(entry.get("n_slash", 0)), int(entry.get("block", 64)),
                   int(entry.get("topk", 1)), int(entry.get("proxy", 0)))


def table_array(table):
    arr = (HeadCfg * len(table))()
    for h, e in enumerate(table):
        arr[h] = head_cfg(e)
    return arr


def _out_like(q, o):
    return torch.empty_like(q) if o is None else o


def _want(t, what, dtype, shape=None, min_numel=None, device=None):
    """Raise ValueError unless t (None passes) is a contiguous tensor of this
    dtype and shape (on `device` if given): the library sees only a pointer,
    so a smaller or strided buffer would be read or written out of bounds."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{what}: a torch.Tensor is required")
    if t.dtype != dtype:
        raise ValueError(f"{what}: dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{what}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError(f"{what}: {t.numel()} elements, at least {min_numel} needed")
    if not t.is_contiguous():
        raise ValueError(f"{what}: must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{what}: on {t.device}, expected {device}")


def _cuda(**tensors):
    """Raise ValueError for the first given tensor (None passes) not on a CUDA device."""
    for what, t in tensors.items():
        if t is not None and not t.is_cuda:
            raise ValueError(f"{what}: must be on a CUDA device")


def _check_attn(q, k, v=None, o=None, lse=None, edges=None, dims=None):
    """Q/O [B,Hq,n,d], K/V [B,Hkv,n,d] bf16, LSE [B,Hq,n] fp32, edges >= B*Hq int64.
    dims: (B, Hq, Hkv, n, d) the tensors must have (a layer's shape), else taken from q and k."""
    for t, what in ((q, "q"), (k, "k")):
        if not isinstance(t, torch.Tensor) or t.dim() != 4:
            raise ValueError(f"{what}: a 4-d tensor [B, H, n, d] is required")
    if dims:
        B, Hq, Hkv, n, d = dims
    else:
        B, Hq, n, d = q.shape
        Hkv = k.shape[1]
    dev = q.device
    _want(q, "q", torch.bfloat16, (B, Hq, n, d), device=dev)
    _want(k, "k", torch.bfloat16, (B, Hkv, n, d), device=dev)
    _want(v, "v", torch.bfloat16, (B, Hkv, n, d), device=dev)
    _want(o, "o", torch.bfloat16, (B, Hq, n, d), device=dev)
    _want(lse, "lse", torch.float32, (B, Hq, n), device=dev)
    _want(edges, "edges", torch.int64, min_numel=B * Hq, device=dev)
    _cuda(q=q, k=k, v=v, o=o, lse=lse, edges=edges)


# ----------------------------------------------------------------- attention
def attn_ashape(q, k, v, heads, sink, window, o=None, lse=None, edges=None, scale=None, stream=None):
    """A-shape heads (sink g, window w); returns o."""
    _check_attn(q, k, v, o, lse, edges)
    lib = load()
    o = _out_like(q, o)
    sh = make_shape(q, k, scale)
    hp, nh = _heads(heads)
    _check(lib.msa_attn_ashape(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), hp, nh, int(sink), int(window), _ptr(o),
                               _ptr(lse), _ptr(edges), _stream(stream)), "msa_attn_ashape")
    return o


def attn_dense(q, k, v, heads, o=None, lse=None, edges=None, scale=None, stream=None):
    """Dense causal attention of the listed heads on the same engine; returns o."""
    _check_attn(q, k, v, o, lse, edges)
    lib = load()
    o = _out_like(q, o)
    sh = make_shape(q, k, scale)
    hp, nh = _heads(heads)
    _check(lib.msa_attn_dense(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), hp, nh, _ptr(o), _ptr(lse), _ptr(edges),
                              _stream(stream)), "msa_attn_dense")
    return o


class VSIndex:
    """Device buffers of a Vertical-Slash index (see msa_vs_index in msa.h)."""

    def __init__(self, slots: int, n: int, n_vertical: int, n_slash: int, device):
        self.slots, self.n = int(slots), int(n)
        self.v_cap = max(min(int(n_vertical), n), 0)
        self.s_cap = max(min(int(n_slash), n), 0)
        words = (n + 31) // 32
        self.vertical = torch.empty(slots, max(self.v_cap, 1), dtype=torch.int32, device=device)
        self.vertical_cnt = torch.empty(slots, dtype=torch.int32, device=device)
        self.slash = torch.empty(slots, max(self.s_cap, 1), dtype=torch.int32, device=device)
        self.slash_cnt = torch.empty(slots, dtype=torch.int32, device=device)
        self.vertical_bits = torch.zeros(slots, words, dtype=torch.int32, device=device)
        self.slash_bits = torch.zeros(slots, words, dtype=torch.int32, device=device)
        self.slash_cover = torch.zeros(slots, (n + 63 + 31) // 32, dtype=torch.int32, device=device)

    def check(self, slots: int, n: int, device=None):
        """Raise ValueError unless the buffers hold `slots` slots of an n-token index (on `device`)."""
        if self.n != n or self.slots < slots:
            raise ValueError(f"VSIndex: {self.slots} slots for n = {self.n}, need {slots} for n = {n}")
        if device is not None and self.vertical_bits.device != device:
            raise ValueError(f"VSIndex: on {self.vertical_bits.device}, expected {device}")

    def c(self) -> VSIndexC:
        return VSIndexC(self.vertical.data_ptr(), self.vertical_cnt.data_ptr(), self.slash.data_ptr(),
                        self.slash_cnt.data_ptr(), self.vertical_bits.data_ptr(), self.slash_bits.data_ptr(),
                        self.slash_cover.data_ptr(), self.v_cap, self.s_cap)

    @staticmethod
    def from_c(c: VSIndexC, slots: int, n: int, ws: torch.Tensor):
        """View of an index that lives in the layer workspace `ws` (the views keep it alive)."""
        ix = VSIndex.__new__(VSIndex)
        ix.slots, ix.n = int(slots), int(n)
        ix.v_cap, ix.s_cap = c.v_cap, c.s_cap
        words = (n + 31) // 32
        ix.vertical = _view_i32(ws, c.vertical, slots * max(c.v_cap, 1)).view(slots, max(c.v_cap, 1))
        ix.vertical_cnt = _view_i32(ws, c.vertical_cnt, slots)
        ix.slash = _view_i32(ws, c.slash, slots * max(c.s_cap, 1)).view(slots, max(c.s_cap, 1))
        ix.slash_cnt = _view_i32(ws, c.slash_cnt, slots)
        ix.vertical_bits = _view_i32(ws, c.vertical_bits, slots * words).view(slots, words)
        ix.slash_bits = _view_i32(ws, c.slash_bits, slots * words).view(slots, words)
        cw = (n + 63 + 31) // 32
        ix.slash_cover = _view_i32(ws, c.slash_cover, slots * cw).view(slots, cw)
        return ix


def _view_i32(base: torch.Tensor, ptr: int, count: int) -> torch.Tensor:
    """A torch int32 view of `count` elements at device address `ptr` inside the uint8 workspace `base`."""
    off = ptr - base.data_ptr()
    assert off % 4 == 0 and 0 <= off and off + 4 * count <= base.numel()
    return base[off:off + 4 * count].view(torch.int32)


def attn_vs(q, k, v, heads, index: VSIndex, o=None, lse=None, edges=None, scale=None, stream=None):
    _check_attn(q, k, v, o, lse, edges)
    index.check(q.shape[0] * len(heads), q.shape[2], q.device)
    lib = load()
    o = _out_like(q, o)
    sh = make_shape(q, k, scale)
    hp, nh = _heads(heads)
    ic = index.c()
    _check(lib.msa_attn_vs(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), hp, nh, 64, ctypes.byref(ic), _ptr(o),
                           _ptr(lse), _ptr(edges), _stream(stream)), "msa_attn_vs")
    return o


def attn_block(q, k, v, heads, topk, block_idx, block_cnt, o=None, lse=None, edges=None, scale=None, stream=None):
    _check_attn(q, k, v, o, lse, edges)
    B, nb = q.shape[0], (q.shape[2] + 63) // 64
    _want(block_idx, "block_idx", torch.int32, (B, len(heads), nb, int(topk)), device=q.device)
    _want(block_cnt, "block_cnt", torch.int32, (B, len(heads), nb), device=q.device)
    lib = load()
    o = _out_like(q, o)
    sh = make_shape(q, k, scale)
    hp, nh = _heads(heads)
    _check(lib.msa_attn_block(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), hp, nh, 64, int(topk), _ptr(block_idx),
                              _ptr(block_cnt), _ptr(o), _ptr(lse), _ptr(edges), _stream(stream)), "msa_attn_block")
    return o


# ----------------------------------------------------------------- indices
def build_vs_index(q, k, heads, last_q, n_vertical, n_slash, index: VSIndex | None = None, scale=None, stream=None,
                   proxy: int = 0):
    _check_attn(q, k)
    lib = load()
    sh = make_shape(q, k, scale)
    hp, nh = _heads(heads)
    cfg = HeadCfg(VS, 0, 1, int(last_q), int(n_vertical), int(n_slash), 64, 1, int(proxy))
    if index is None:
        index = VSIndex(q.shape[0] * nh, q.shape[2], n_vertical, n_slash, q.device)
    index.check(q.shape[0] * nh, q.shape[2], q.device)
    if index.v_cap < min(int(n_vertical), q.shape[2]) or index.s_cap < min(int(n_slash), q.shape[2]):
        raise ValueError("VSIndex: list capacity below the requested budgets")
    ws_bytes = lib.msa_vs_index_workspace(ctypes.byref(sh), ctypes.byref(cfg), nh)
    ws = torch.empty(max(int(ws_bytes), 1), dtype=torch.uint8, device=q.device)
    ic = index.c()
    _check(lib.msa_build_vs_index(ctypes.byref(sh), _ptr(q), _ptr(k), hp, nh, ctypes.byref(cfg), ctypes.byref(ic),
                                  _ptr(ws), int(ws_bytes), _stream(stream)), "msa_build_vs_index")
    index._ws = ws  # keep the scratch alive until the stream has used it
    return index


def build_block_index(q, k, heads, topk, block_idx=None, block_cnt=None, scale=None, stream=None):
    _check_attn(q, k)
    lib = load()
    sh = make_shape(q, k, scale)
    hp, nh = _heads(heads)
    B, n = q.shape[0], q.shape[2]
    nb = (n + 63) // 64
    if block_idx is None:
        block_idx = torch.empty(B, nh, nb, int(topk), dtype=torch.int32, device=q.device)
    if block_cnt is None:
        block_cnt = torch.empty(B, nh, nb, dtype=torch.int32, device=q.device)
    _want(block_idx, "block_idx", torch.int32, (B, nh, nb, int(topk)), device=q.device)
    _want(block_cnt, "block_cnt", torch.int32, (B, nh, nb), device=q.device)
    ws_bytes = lib.msa_block_index_workspace(ctypes.byref(sh), 64, nh)
    ws = torch.empty(max(int(ws_bytes), 1), dtype=torch.uint8, device=q.device)
    _check(lib.msa_build_block_index(ctypes.byref(sh), _ptr(q), _ptr(k), hp, nh, 64, int(topk), _ptr(block_idx),
                                     _ptr(block_cnt), _ptr(ws), int(ws_bytes), _stream(stream)),
           "msa_build_block_index")
    block_idx._ws = ws
    return block_idx, block_cnt


def build_block_index_static(q, k, heads, topk, block_idx=None, block_cnt=None, scale=None, stream=None):
    """msa_build_block_index_static: the Block-Sparse index built in the
    library's own scratch (no workspace); outputs as build_block_index."""
    _check_attn(q, k)
    lib = load()
    sh = make_shape(q, k, scale)
    hp, nh = _heads(heads)
    B, n = q.shape[0], q.shape[2]
    nb = (n + 63) // 64
    if block_idx is None:
        block_idx = torch.empty(B, nh, nb, int(topk), dtype=torch.int32, device=q.device)
    if block_cnt is None:
        block_cnt = torch.empty(B, nh, nb, dtype=torch.int32, device=q.device)
    _want(block_idx, "block_idx", torch.int32, (B, nh, nb, int(topk)), device=q.device)
    _want(block_cnt, "block_cnt", torch.int32, (B, nh, nb), device=q.device)
    _check(lib.msa_build_block_index_static(ctypes.byref(sh), _ptr(q), _ptr(k), hp, nh, 64, int(topk),
                                            _ptr(block_idx), _ptr(block_cnt), _stream(stream)),
           "msa_build_block_index_static")
    return block_idx, block_cnt


def vs_expand(q_shape, index: VSIndex, slot, u_begin, u_count, range_cap, col_cap, stream=None):
    """Explicit per-block ranges and columns of one slot (device tensors)."""
    lib = load()
    B, Hq, n, d = q_shape
    sh = Shape(B, Hq, 1, n, d, 0.0)
    dev = index.vertical.device
    rc = torch.empty(u_count, dtype=torch.int32, device=dev)
    rg = torch.empty(u_count, max(range_cap, 1), 2, dtype=torch.int32, device=dev)
    cc = torch.empty(u_count, dtype=torch.int32, device=dev)
    cl = torch.empty(u_count, max(col_cap, 1), dtype=torch.int32, device=dev)
    ic = index.c()
    _check(lib.msa_vs_expand(ctypes.byref(sh), ctypes.byref(ic), int(slot), int(u_begin), int(u_count), int(range_cap),
                             int(col_cap), _ptr(rc), _ptr(rg), _ptr(cc), _ptr(cl), _stream(stream)), "msa_vs_expand")
    return rc, rg, cc, cl


# ----------------------------------------------------------------- layer
class Layer:
    """One layer's config table plus its workspace; call() runs msa_prefill_layer."""

    def __init__(self, table, B, Hq, Hkv, n, d, device, scale=None):
        self.table = list(table)
        assert len(self.table) == Hq
        self.tarr = table_array(self.table)
        self.shape = Shape(B, Hq, Hkv, n, d, float(scale) if scale else 0.0)
        lib = load()
        self.ws_bytes = int(lib.msa_layer_workspace(ctypes.byref(self.shape), self.tarr))
        if self.ws_bytes == 0:
            raise MsaError(MSA_ERR_INVALID_ARG, "msa_layer_workspace")
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)

    def _dims(self):
        s = self.shape
        return (s.B, s.Hq, s.Hkv, s.n, s.d_h)

    def __call__(self, q, k, v, o=None, lse=None, edges=None, stream=None):
        _check_attn(q, k, v, o, lse, edges, self._dims())
        lib = load()
        o = _out_like(q, o)
        _check(lib.msa_prefill_layer(ctypes.byref(self.shape), _ptr(q), _ptr(k), _ptr(v), self.tarr, _ptr(o), _ptr(lse),
                                     _ptr(edges), _ptr(self.ws), self.ws_bytes, _stream(stream)), "msa_prefill_layer")
        return o

    def index(self, q, k, stream=None):
        """First half of the layer (T_index): build every online index into the workspace."""
        _check_attn(q, k, dims=self._dims())
        _check(load().msa_layer_index(ctypes.byref(self.shape), _ptr(q), _ptr(k), self.tarr, _ptr(self.ws),
                                      self.ws_bytes, _stream(stream)), "msa_layer_index")

    def attend(self, q, k, v, o, lse=None, edges=None, stream=None):
        """Second half (T_sparse): the single attention launch over the indices in the workspace."""
        _check_attn(q, k, v, o, lse, edges, self._dims())
        _check(load().msa_layer_attend(ctypes.byref(self.shape), _ptr(q), _ptr(k), _ptr(v), self.tarr, _ptr(o),
                                       _ptr(lse), _ptr(edges), _ptr(self.ws), self.ws_bytes, _stream(stream)),
               "msa_layer_attend")
        return o

    def attend_stats(self, q, k, v, o, lse=None, edges=None, tiles=None, stream=None):
        """attend() with work counters: edges (E_h) and tiles (64-row x 128-key tiles per query head),
        both [B*Hq] int64 device tensors that are ADDED to."""
        _check_attn(q, k, v, o, lse, edges, self._dims())
        if tiles is not None:
            _want(tiles, "tiles", torch.int64, (self.shape.B * self.shape.Hq,), device=q.device)
        _check(load().msa_layer_attend_stats(ctypes.byref(self.shape), _ptr(q), _ptr(k), _ptr(v), self.tarr, _ptr(o),
                                             _ptr(lse), _ptr(edges), _ptr(tiles), _ptr(self.ws), self.ws_bytes,
                                             _stream(stream)), "msa_layer_attend_stats")
        return o

    def attend_rows(self, q, k, v, o, row_begin, row_end, lse=None, edges=None, stream=None):
        """Chunked T_sparse: the attention of query rows [row_begin, row_end) only (indices from index())."""
        _check_attn(q, k, v, o, lse, edges, self._dims())
        _check(load().msa_layer_attend_rows(ctypes.byref(self.shape), _ptr(q), _ptr(k), _ptr(v), self.tarr, _ptr(o),
                                            _ptr(lse), _ptr(edges), _ptr(self.ws), self.ws_bytes, int(row_begin),
                                            int(row_end), _stream(stream)), "msa_layer_attend_rows")
        return o

    def indices(self):
        """(VSIndex view, block_idx, block_cnt) left in the workspace by the last call."""
        lib = load()
        vc = VSIndexC()
        bi = ctypes.c_void_p()
        bc = ctypes.c_void_p()
        _check(lib.msa_layer_indices(ctypes.byref(self.shape), self.tarr, _ptr(self.ws), ctypes.byref(vc),
                                     ctypes.byref(bi), ctypes.byref(bc)), "msa_layer_indices")
        B, n = self.shape.B, self.shape.n
        nvs = sum(1 for e in self.table if head_cfg(e).pattern == VS)
        nbs = [e for e in self.table if head_cfg(e).pattern == BLOCK]
        vs = VSIndex.from_c(vc, B * nvs, n, self.ws) if nvs else None
        blk = cnt = None
        if nbs:
            nb = (n + 63) // 64
            topk = head_cfg(nbs[0]).topk
            blk = _view_i32(self.ws, bi.value, B * len(nbs) * nb * topk).view(B, len(nbs), nb, topk)
            cnt = _view_i32(self.ws, bc.value, B * len(nbs) * nb).view(B, len(nbs), nb)
        return vs, blk, cnt


# ----------------------------------------------------------------- varlen
def pack_varlen(seqs) -> torch.Tensor:
    """Pack per-sequence [H, n_s, d] tensors back to back (the varlen layout)."""
    return torch.cat([x.contiguous().reshape(-1) for x in seqs])


def unpack_varlen(flat: torch.Tensor, H: int, cu_seqlens, d: int):
    """Split a packed varlen buffer into per-sequence [H, n_s, d] views."""
    out = []
    for s in range(len(cu_seqlens) - 1):
        a, b = int(cu_seqlens[s]), int(cu_seqlens[s + 1])
        out.append(flat[H * a * d:H * b * d].view(H, b - a, d))
    return out


class VarlenLayer:
    """A varlen batch (cumulative lengths cu_seqlens) of one layer's table plus
    its workspace; call() runs msa_prefill_layer_varlen on packed buffers (see
    pack_varlen) and indices(seq) views what it left for one sequence."""

    def __init__(self, table, cu_seqlens, Hq, Hkv, d, device, scale=None):
        self.table = list(table)
        if len(self.table) != int(Hq):
            raise ValueError(f"table: {len(self.table)} entries, expected Hq = {int(Hq)}")
        self.cu_list = [int(x) for x in cu_seqlens]
        self.n_seqs = len(self.cu_list) - 1
        self.cu = (ctypes.c_int32 * len(self.cu_list))(*self.cu_list)
        lens = [self.cu_list[s + 1] - self.cu_list[s] for s in range(self.n_seqs)]
        self.Hq, self.Hkv, self.d = int(Hq), int(Hkv), int(d)
        self.shape = Shape(1, self.Hq, self.Hkv, max([1] + lens), self.d, float(scale) if scale else 0.0)
        self.tarr = table_array(self.table)
        lib = load()
        self.ws_bytes = int(lib.msa_layer_varlen_workspace(ctypes.byref(self.shape), self.tarr, self.cu, self.n_seqs))
        if self.ws_bytes == 0:
            raise MsaError(MSA_ERR_INVALID_ARG, "msa_layer_varlen_workspace")
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)

    def __call__(self, q, k, v, o=None, lse=None, edges=None, stream=None):
        _check_varlen(q, k, v, o, lse, edges, self.cu_list, self.Hq, self.Hkv, self.d)
        o = torch.empty_like(q) if o is None else o
        _check(load().msa_prefill_layer_varlen(ctypes.byref(self.shape), self.cu, self.n_seqs, _ptr(q), _ptr(k),
                                               _ptr(v), self.tarr, _ptr(o), _ptr(lse), _ptr(edges), _ptr(self.ws),
                                               self.ws_bytes, _stream(stream)), "msa_prefill_layer_varlen")
        return o

    def indices(self, seq: int):
        """(VSIndex view, block_idx [n_bs, N_b, topk], block_cnt [n_bs, N_b]) of sequence seq."""
        lib = load()
        vc = VSIndexC()
        bi = ctypes.c_void_p()
        bc = ctypes.c_void_p()
        _check(lib.msa_layer_varlen_indices(ctypes.byref(self.shape), self.tarr, self.cu, self.n_seqs,
                                            _ptr(self.ws), int(seq), ctypes.byref(vc), ctypes.byref(bi),
                                            ctypes.byref(bc)), "msa_layer_varlen_indices")
        n = self.cu_list[seq + 1] - self.cu_list[seq]
        nvs = sum(1 for e in self.table if head_cfg(e).pattern == VS)
        nbs = [e for e in self.table if head_cfg(e).pattern == BLOCK]
        vs = VSIndex.from_c(vc, nvs, n, self.ws) if nvs else None
        blk = cnt = None
        if nbs:
            nb = (n + 63) // 64
            topk = head_cfg(nbs[0]).topk
            blk = _view_i32(self.ws, bi.value, len(nbs) * nb * topk).view(len(nbs), nb, topk)
            cnt = _view_i32(self.ws, bc.value, len(nbs) * nb).view(len(nbs), nb)
        return vs, blk, cnt


def _check_varlen(q, k, v, o, lse, edges, cu_seqlens, Hq, Hkv, d):
    total = int(cu_seqlens[-1]) if len(cu_seqlens) else 0
    _want(q, "q", torch.bfloat16, min_numel=Hq * total * d)
    _want(k, "k", torch.bfloat16, min_numel=Hkv * total * d, device=q.device)
    _want(v, "v", torch.bfloat16, min_numel=Hkv * total * d, device=q.device)
    _want(o, "o", torch.bfloat16, tuple(q.shape), device=q.device)
    _want(lse, "lse", torch.float32, min_numel=Hq * total, device=q.device)
    _want(edges, "edges", torch.int64, min_numel=(len(cu_seqlens) - 1) * Hq, device=q.device)
    _cuda(q=q)


def prefill_layer_varlen(q, k, v, table, cu_seqlens, Hq, Hkv, d, o=None, lse=None, edges=None, scale=None,
                         stream=None):
    """msa_prefill_layer_varlen on packed buffers (see pack_varlen); returns o."""
    _check_varlen(q, k, v, o, lse, edges, cu_seqlens, Hq, Hkv, d)
    layer = VarlenLayer(table, cu_seqlens, Hq, Hkv, d, q.device, scale=scale)
    return layer(q, k, v, o=o, lse=lse, edges=edges, stream=stream)


def merge_attention(o_a, lse_a, o_b, lse_b, o=None, lse=None, stream=None):
    """Combine two attention results over disjoint key sets (msa_merge_attention); returns (o, lse)."""
    if not isinstance(o_a, torch.Tensor) or o_a.dim() < 1:
        raise ValueError("o_a: a tensor [..., d] is required")
    d = o_a.shape[-1]
    rows = o_a.numel() // d
    for t, what in ((o_a, "o_a"), (o_b, "o_b"), (o, "o")):
        _want(t, what, torch.bfloat16, tuple(o_a.shape), device=o_a.device)
    for t, what in ((lse_a, "lse_a"), (lse_b, "lse_b"), (lse, "lse")):
        _want(t, what, torch.float32, tuple(o_a.shape[:-1]), device=o_a.device)
    _cuda(o_a=o_a)
    o = torch.empty_like(o_a) if o is None else o
    lse = torch.empty_like(lse_a) if lse is None else lse
    _check(load().msa_merge_attention(rows, d, _ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(o), _ptr(lse),
                                      _stream(stream)), "msa_merge_attention")
    return o, lse


def captured_mass(lse_sparse, lse_dense, stream=None):
    """Per-head share of the dense softmax mass kept by the sparse sets (msa_captured_mass).
    lse_*: [..., n] with the leading dims flattened into heads; returns [heads] fp32."""
    if not isinstance(lse_sparse, torch.Tensor) or lse_sparse.dim() < 1:
        raise ValueError("lse_sparse: a tensor [..., n] is required")
    _want(lse_sparse, "lse_sparse", torch.float32, device=lse_sparse.device)
    _want(lse_dense, "lse_dense", torch.float32, tuple(lse_sparse.shape), device=lse_sparse.device)
    _cuda(lse_sparse=lse_sparse)
    n = lse_sparse.shape[-1]
    heads = lse_sparse.numel() // n
    mass = torch.empty(heads, dtype=torch.float32, device=lse_sparse.device)
    _check(load().msa_captured_mass(heads, n, _ptr(lse_sparse), _ptr(lse_dense), _ptr(mass), _stream(stream)),
           "msa_captured_mass")
    return mass


def kernel_launches() -> int:
    """Kernels launched through the library by this process so far."""
    return int(load().msa_kernel_launches())


def check_wait_timeout(limit_ms: int, stream=None):
    """Launch the failure-detection check (a bounded wait that runs out)."""
    _check(load().msa_check_wait_timeout(int(limit_ms), _stream(stream)), "msa_check_wait_timeout")


def poll_device_status(stream=None) -> int:
    """Synchronise the stream and read/clear the device error word (status code)."""
    return int(load().msa_poll_device_status(_stream(stream)))
