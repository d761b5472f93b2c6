"""CPU checks of the C ABI: the library loads, exports every symbol msa.h
declares, and rejects bad arguments on the host before any launch (these
calls return before touching the GPU, so they run without one)."""
import ctypes
import os
import re

import pytest

import long_context_prefill_gb300 as msa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from long_context_prefill_gb300 import build
    build.build()
    return msa.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "msa.h")).read()
    return sorted(set(re.findall(r"MSA_API\s+[\w\s\*]+?\b(msa_\w+)\s*\(", src)))


def test_header_declares_every_binding_export():
    assert declared_functions() == sorted(msa.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(7):
        assert msa.status_string(code)
    assert msa.status_string(0) == "ok"


def _shape(**kw):
    base = dict(B=1, Hq=4, Hkv=2, n=256, d_h=128, scale=0.0)
    base.update(kw)
    return msa.Shape(**base)


FAKE = ctypes.c_void_p(0x10000)  # 16-byte aligned, never dereferenced: validation fails first or no launch


def _heads(hs):
    return (ctypes.c_int32 * len(hs))(*hs), len(hs)


@pytest.mark.parametrize("shape_kw,code", [
    (dict(Hq=3, Hkv=2), msa.MSA_ERR_INVALID_ARG),   # Hq % Hkv != 0
    (dict(n=0), msa.MSA_ERR_INVALID_ARG),
    (dict(d_h=96), msa.MSA_ERR_UNSUPPORTED),
    (dict(B=0), msa.MSA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), msa.MSA_ERR_INVALID_ARG),
])
def test_bad_shapes_rejected(lib, shape_kw, code):
    sh = _shape(**shape_kw)
    hp, nh = _heads([0])
    st = lib.msa_attn_ashape(ctypes.byref(sh), FAKE, FAKE, FAKE, hp, nh, 4, 16, FAKE, None, None, None)
    assert st == code


def test_bad_heads_and_budgets_rejected(lib):
    sh = _shape()
    for hs in ([4], [-1], [0, 0], []):
        hp, nh = _heads(hs) if hs else (None, 0)
        assert lib.msa_attn_ashape(ctypes.byref(sh), FAKE, FAKE, FAKE, hp, nh, 4, 16, FAKE, None, None,
                                   None) == msa.MSA_ERR_INVALID_ARG
    hp, nh = _heads([1])
    assert lib.msa_attn_ashape(ctypes.byref(sh), FAKE, FAKE, FAKE, hp, nh, -1, 16, FAKE, None, None,
                               None) == msa.MSA_ERR_INVALID_ARG
    assert lib.msa_attn_ashape(ctypes.byref(sh), FAKE, FAKE, FAKE, hp, nh, 4, 0, FAKE, None, None,
                               None) == msa.MSA_ERR_INVALID_ARG
    # misaligned tensor
    assert lib.msa_attn_ashape(ctypes.byref(sh), ctypes.c_void_p(0x10008), FAKE, FAKE, hp, nh, 4, 16, FAKE, None,
                               None, None) == msa.MSA_ERR_INVALID_ARG
    assert lib.msa_attn_block(ctypes.byref(sh), FAKE, FAKE, FAKE, hp, nh, 64, 0, FAKE, FAKE, FAKE, None, None,
                              None) == msa.MSA_ERR_INVALID_ARG
    assert lib.msa_attn_block(ctypes.byref(sh), FAKE, FAKE, FAKE, hp, nh, 32, 4, FAKE, FAKE, FAKE, None, None,
                              None) == msa.MSA_ERR_UNSUPPORTED
    cfg = msa.HeadCfg(msa.VS, 0, 1, 0, 10, 10, 64, 1)  # last_q = 0
    ix = msa.VSIndexC()
    assert lib.msa_build_vs_index(ctypes.byref(sh), FAKE, FAKE, hp, nh, ctypes.byref(cfg), ctypes.byref(ix), FAKE,
                                  1 << 20, None) == msa.MSA_ERR_INVALID_ARG


def test_layer_workspace_and_table_validation(lib):
    sh = _shape()
    table = msa.table_array([dict(pattern="ashape", sink=4, window=64), dict(pattern="vs", last_q=64, n_vertical=10,
                                                                              n_slash=20),
                             dict(pattern="block", topk=3), dict(pattern="vs", last_q=64, n_vertical=10, n_slash=20)])
    ws = lib.msa_layer_workspace(ctypes.byref(sh), table)
    assert ws > 0
    bad = msa.table_array([dict(pattern="ashape", sink=4, window=0)] * 4)
    assert lib.msa_layer_workspace(ctypes.byref(sh), bad) == 0
    mixed_vs = msa.table_array([dict(pattern="vs", last_q=64, n_vertical=10, n_slash=20),
                                dict(pattern="vs", last_q=64, n_vertical=11, n_slash=20)] * 2)
    assert lib.msa_layer_workspace(ctypes.byref(sh), mixed_vs) == 0
    # workspace too small is reported before anything runs
    st = lib.msa_prefill_layer(ctypes.byref(sh), FAKE, FAKE, FAKE, table, FAKE, None, None, FAKE, 16, None)
    assert st == msa.MSA_ERR_WORKSPACE_TOO_SMALL


def test_missing_library_fails_loudly(tmp_path):
    import importlib
    mod = importlib.import_module("long_context_prefill_gb300")
    saved = mod._lib
    try:
        mod._lib = None
        with pytest.raises(RuntimeError):
            mod.load(str(tmp_path / "nope.so"))
    finally:
        mod._lib = saved


def test_binding_validates_tensors():
    """The binding refuses tensors whose dtype, shape, layout or device would
    make the library read or write outside them (the C ABI sees pointers only);
    the checks run before the library is called, so CPU tensors exercise them."""
    import torch
    bf = torch.bfloat16
    q = torch.zeros(1, 2, 64, 128, dtype=bf)
    k = torch.zeros(1, 1, 64, 128, dtype=bf)
    cases = [
        (lambda: msa.attn_ashape(q, k, torch.zeros(1, 1, 32, 128, dtype=bf), [0], 4, 16), "v: shape"),
        (lambda: msa.attn_ashape(q, k, k, [0], 4, 16, o=torch.zeros(1, 2, 64, 128)), "o: dtype"),
        (lambda: msa.attn_ashape(q, k, k, [0], 4, 16, o=torch.zeros(1, 2, 128, 64, dtype=bf).transpose(2, 3)),
         "o: must be contiguous"),
        (lambda: msa.attn_ashape(q, k, k, [0], 4, 16, lse=torch.zeros(1, 2, 63)), "lse: shape"),
        (lambda: msa.attn_ashape(q, k, k, [0], 4, 16, edges=torch.zeros(1, dtype=torch.int64)), "edges: 1 elements"),
        (lambda: msa.attn_ashape(q.float(), k, k, [0], 4, 16), "q: dtype"),
        (lambda: msa.attn_ashape(q, k, k, [0], 4, 16), "q: must be on a CUDA device"),
        (lambda: msa.attn_block(q, k, k, [0], 4, torch.zeros(1, 1, 1, 4, dtype=torch.int32),
                                torch.zeros(1, 1, 1, dtype=torch.int32)), "q: must be on a CUDA device"),
        (lambda: msa.merge_attention(torch.zeros(8, 128, dtype=bf), torch.zeros(8), torch.zeros(8, 64, dtype=bf),
                                     torch.zeros(8)), "o_b: shape"),
        (lambda: msa.captured_mass(torch.zeros(2, 64), torch.zeros(2, 65)), "lse_dense: shape"),
        (lambda: msa.prefill_layer_varlen(torch.zeros(100, dtype=bf), k, k, [dict(pattern="ashape", sink=4, window=8)],
                                          [0, 64], 2, 1, 128), "q: 100 elements"),
    ]
    for call, msg in cases:
        with pytest.raises(ValueError, match=msg):
            call()
    ix = msa.VSIndex.__new__(msa.VSIndex)
    ix.slots, ix.n = 1, 64
    with pytest.raises(ValueError, match="VSIndex"):
        ix.check(2, 64)


def test_empty_inputs_are_no_ops(lib):
    """Valid calls with nothing to do return MSA_OK before touching the
    device (so they run here without one): a merge of zero rows, the captured
    mass of zero heads, and a varlen batch whose sequences are all empty."""
    P = ctypes.c_void_p
    a, b, la, lb = P(0x10000), P(0x20000), P(0x30000), P(0x40000)
    assert lib.msa_merge_attention(0, 128, a, la, b, lb, a, None, None) == msa.MSA_OK
    assert lib.msa_captured_mass(0, 16, la, lb, P(0x50000), None) == msa.MSA_OK
    table = msa.table_array([dict(pattern="ashape", sink=4, window=64),
                             dict(pattern="vs", last_q=64, n_vertical=10, n_slash=20)])
    cu = (ctypes.c_int32 * 3)(0, 0, 0)
    sh = msa.Shape(1, 2, 1, 1, 128, 0.0)
    need = lib.msa_layer_varlen_workspace(ctypes.byref(sh), table, cu, 2)
    assert need > 0
    assert lib.msa_prefill_layer_varlen(ctypes.byref(sh), cu, 2, a, a, a, table, a, None, None, a, need,
                                        None) == msa.MSA_OK
