"""Varlen prefill (msa_prefill_layer_varlen): sequences of different lengths
packed without padding, each with its own online indices and attention.

CPU: the host checks of cu_seqlens and the workspace rule (no launch).  GPU:
every sequence's output, LSE and edge counts equal those of msa_prefill_layer
run on that sequence alone (the same kernels, so bit for bit), and A-shape
heads match the fp64 oracle directly."""
import ctypes

import numpy as np
import pytest
import torch

import long_context_prefill_gb300 as msa
import oracle
import synth
from helpers import compare_rows, f32, oracle_cfg

TABLE = [synth.ashape(16, 100), synth.vslash(64, 20, 50), synth.blocksparse(4), synth.vslash(64, 20, 50)]
HQ, HKV, D = 4, 2, 128
LENS = [1000, 0, 64, 2500, 777]


def _cu(lens):
    return [0] + list(np.cumsum(lens).astype(int))


@pytest.fixture(scope="module")
def lib():
    from long_context_prefill_gb300 import build
    build.build()
    return msa.load()


def _shape():
    return msa.Shape(1, HQ, HKV, 1, D, 0.0)


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first


@pytest.mark.parametrize("cu", [[1, 5], [0, 5, 3], [0]])
def test_varlen_rejects_bad_cu_seqlens(lib, cu):
    arr = (ctypes.c_int32 * len(cu))(*cu)
    n_seqs = len(cu) - 1
    tarr = msa.table_array(TABLE)
    assert lib.msa_layer_varlen_workspace(ctypes.byref(_shape()), tarr, arr, n_seqs) == 0
    st = lib.msa_prefill_layer_varlen(ctypes.byref(_shape()), arr, n_seqs, FAKE, FAKE, FAKE, tarr, FAKE, None, None,
                                      FAKE, 1 << 30, None)
    assert st == msa.MSA_ERR_INVALID_ARG


def test_varlen_workspace_is_the_largest_sequence(lib):
    cu = _cu(LENS)
    arr = (ctypes.c_int32 * len(cu))(*cu)
    tarr = msa.table_array(TABLE)
    want = max(lib.msa_layer_workspace(ctypes.byref(msa.Shape(1, HQ, HKV, n, D, 0.0)), tarr) for n in LENS if n)
    assert lib.msa_layer_varlen_workspace(ctypes.byref(_shape()), tarr, arr, len(LENS)) == want


def _sequences(device):
    return [synth.random_qkv(1, HQ, HKV, n, D, seed=500 + s, device=device) if n else None
            for s, n in enumerate(LENS)]


@pytest.mark.gpu
def test_varlen_equals_each_sequence_alone(cuda_lib):
    seqs = _sequences("cuda")
    cu = _cu(LENS)
    empty = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    q = cuda_lib.pack_varlen([x[0][0] if x else empty for x in seqs])
    k = cuda_lib.pack_varlen([x[1][0] if x else empty for x in seqs])
    v = cuda_lib.pack_varlen([x[2][0] if x else empty for x in seqs])
    lse = torch.empty(HQ * cu[-1], device="cuda")
    edges = torch.zeros(len(LENS) * HQ, dtype=torch.int64, device="cuda")
    o = cuda_lib.prefill_layer_varlen(q, k, v, TABLE, cu, HQ, HKV, D, lse=lse, edges=edges)
    assert cuda_lib.poll_device_status() == 0
    outs = cuda_lib.unpack_varlen(o, HQ, cu, D)
    lses = [lse[HQ * cu[s]:HQ * cu[s + 1]].view(HQ, -1) for s in range(len(LENS))]
    for s, n in enumerate(LENS):
        if not n:
            continue
        qs, ks, vs = seqs[s]
        layer = cuda_lib.Layer(TABLE, 1, HQ, HKV, n, D, "cuda")
        o1 = torch.empty_like(qs)
        l1 = torch.empty(1, HQ, n, device="cuda")
        e1 = torch.zeros(HQ, dtype=torch.int64, device="cuda")
        layer(qs, ks, vs, o=o1, lse=l1, edges=e1)
        assert cuda_lib.poll_device_status() == 0
        assert torch.equal(outs[s], o1[0]), f"sequence {s}: output"
        assert torch.equal(lses[s], l1[0]), f"sequence {s}: lse"
        assert torch.equal(edges[s * HQ:(s + 1) * HQ], e1), f"sequence {s}: edges"


@pytest.mark.gpu
def test_varlen_ashape_heads_against_oracle(cuda_lib):
    seqs = _sequences("cuda")
    cu = _cu(LENS)
    empty = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    q = cuda_lib.pack_varlen([x[0][0] if x else empty for x in seqs])
    k = cuda_lib.pack_varlen([x[1][0] if x else empty for x in seqs])
    v = cuda_lib.pack_varlen([x[2][0] if x else empty for x in seqs])
    lse = torch.empty(HQ * cu[-1], device="cuda")
    o = cuda_lib.prefill_layer_varlen(q, k, v, TABLE, cu, HQ, HKV, D, lse=lse)
    assert cuda_lib.poll_device_status() == 0
    outs = cuda_lib.unpack_varlen(o, HQ, cu, D)
    cfg = oracle_cfg(TABLE[0])
    for s, n in enumerate(LENS):
        if not n:
            continue
        qs, ks, vs = seqs[s]
        rows = synth.sample_rows(n, 150, seed=n)
        ro, rl, _ = oracle.head_rows(cfg, f32(qs[0, 0]), f32(ks[0, 0]), f32(vs[0, 0]), rows, D ** -0.5)
        lh = lse[HQ * cu[s]:HQ * cu[s + 1]].view(HQ, n)
        compare_rows(f32(outs[s][0])[rows], f32(lh[0])[rows], ro, rl, f"sequence {s} A-shape head")


# ----------------------------------------------------------------- chunked rows
@pytest.mark.parametrize("lo,hi", [(100, 512), (0, 0), (256, 300), (512, 256)])
def test_attend_rows_rejects_bad_ranges(lib, lo, hi):
    shape = msa.Shape(1, HQ, HKV, 1000, D, 0.0)
    st = lib.msa_layer_attend_rows(ctypes.byref(shape), FAKE, FAKE, FAKE, msa.table_array(TABLE), FAKE, None, None,
                                   FAKE, 1 << 30, lo, hi, None)
    assert st == msa.MSA_ERR_INVALID_ARG


@pytest.mark.gpu
def test_chunked_rows_reproduce_the_whole_layer(cuda_lib):
    """Indices built once; the attention run in three row chunks (out of
    order) equals the whole-layer attention bit for bit, rows outside a chunk
    are left untouched, and the chunks' edge counts add up."""
    n, B = 1300, 2
    q, k, v = synth.random_qkv(B, HQ, HKV, n, D, seed=901, device="cuda")
    layer = cuda_lib.Layer(TABLE, B, HQ, HKV, n, D, "cuda")
    o_all = torch.empty_like(q)
    l_all = torch.empty(B, HQ, n, device="cuda")
    e_all = torch.zeros(B * HQ, dtype=torch.int64, device="cuda")
    layer.index(q, k)
    layer.attend(q, k, v, o_all, lse=l_all, edges=e_all)
    sentinel = torch.full_like(q, 7.0)
    o = sentinel.clone()
    lse = torch.full((B, HQ, n), 7.0, device="cuda")
    edges = torch.zeros(B * HQ, dtype=torch.int64, device="cuda")
    layer.attend_rows(q, k, v, o, 512, 1024, lse=lse, edges=edges)
    assert cuda_lib.poll_device_status() == 0
    assert torch.equal(o[:, :, 512:1024], o_all[:, :, 512:1024])
    assert torch.equal(o[:, :, :512], sentinel[:, :, :512]) and torch.equal(o[:, :, 1024:], sentinel[:, :, 1024:])
    for lo, hi in [(1024, n), (0, 512)]:
        layer.attend_rows(q, k, v, o, lo, hi, lse=lse, edges=edges)
    assert cuda_lib.poll_device_status() == 0
    assert torch.equal(o, o_all) and torch.equal(lse, l_all) and torch.equal(edges, e_all)
