"""Varlen prefill (msa_prefill_layer_varlen): sequences of different lengths
packed without padding, each with its own online indices and attention
(cost-model page §2.2: no window, index or tile reaches a neighbour's tokens).

CPU: the host checks of cu_seqlens and the workspace rule (no launch).  GPU:
every sequence's output, LSE and edge counts equal those of msa_prefill_layer
run on that sequence alone (bit for bit), the launches of a batch do not grow
with its number of sequences, and every head of every packed
sequence matches the fp64 oracle: its online index against the oracle's index
of that sequence alone, its rows on the packed layout against eq.(2) over the
device's sets, and its edge count exactly.  Chunked prefill (MInference page
§5.2): each row chunk's attention against the oracle on the index built once."""
import ctypes

import numpy as np
import pytest
import torch

import long_context_prefill_gb300 as msa
import oracle
import synth
from helpers import check_block_index, check_topk_set, compare_rows, f32, oracle_cfg

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


def test_varlen_workspace_of_equal_lengths_is_the_uniform_batch(lib):
    """One plan covers every sequence (sequence-major regions): a varlen batch
    of equal lengths needs exactly the workspace of the uniform batch, and a
    longer batch needs more."""
    tarr = msa.table_array(TABLE)
    cu = _cu([512, 512, 512])
    arr = (ctypes.c_int32 * len(cu))(*cu)
    uni = lib.msa_layer_workspace(ctypes.byref(msa.Shape(3, HQ, HKV, 512, D, 0.0)), tarr)
    assert uni > 0 and lib.msa_layer_varlen_workspace(ctypes.byref(_shape()), tarr, arr, 3) == uni
    cu2 = _cu(LENS)
    arr2 = (ctypes.c_int32 * len(cu2))(*cu2)
    more = lib.msa_layer_varlen_workspace(ctypes.byref(_shape()), tarr, arr2, len(LENS))
    assert more > lib.msa_layer_workspace(ctypes.byref(msa.Shape(1, HQ, HKV, max(LENS), D, 0.0)), tarr)


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


def check_sequence_against_oracle(layer, s, n, q, k, v, outs, lses, edges, table, rows=None, what=""):
    """Every head of packed sequence s against the oracle run on that sequence
    alone (q, k, v: its [1, H, n, d] tensors)."""
    vs, bidx, bcnt = layer.indices(s)
    vs_heads = [h for h, e in enumerate(table) if e["pattern"] == "vs"]
    bs_heads = [h for h, e in enumerate(table) if e["pattern"] == "block"]
    g = HQ // HKV
    rows = np.arange(n) if rows is None else rows
    scale = D ** -0.5
    for h, entry in enumerate(table):
        qn, kn, vn = f32(q[0, h]), f32(k[0, h // g]), f32(v[0, h // g])
        cfg = oracle_cfg(entry)
        idx = {}
        if entry["pattern"] == "vs":
            x = vs_heads.index(h)
            C = vs.vertical[x, :int(vs.vertical_cnt[x])].cpu().numpy()
            Dl = vs.slash[x, :int(vs.slash_cnt[x])].cpu().numpy()
            Co, Do, c, r = oracle.vs_index(qn, kn, entry["last_q"], entry["n_vertical"], entry["n_slash"], scale)
            check_topk_set(C, Co, c, min(entry["n_vertical"], n), f"{what} seq {s} vertical h{h}")
            check_topk_set(Dl, Do, r, min(entry["n_slash"], n), f"{what} seq {s} slash h{h}")
            idx = dict(C=C, D=Dl)
        elif entry["pattern"] == "block":
            x = bs_heads.index(h)
            J, cnt = bidx[x].cpu().numpy(), bcnt[x].cpu().numpy()
            Jo, co = oracle.bs_index(qn, kn, 64, entry["topk"])
            check_block_index(J, cnt, Jo, co, oracle.bs_pool(qn, 64), oracle.bs_pool(kn, 64), entry["topk"],
                              f"{what} seq {s} blocks h{h}")
            idx = dict(J=J, cnt=cnt)
        ro, rl, _ = oracle.head_rows(cfg, qn, kn, vn, rows, scale, **idx)
        compare_rows(f32(outs[s][h])[rows], f32(lses[s][h])[rows], ro, rl, f"{what} seq {s} h{h} {entry['pattern']}")
        assert int(edges[s * HQ + h]) == oracle.head_edges(cfg, n, **idx), f"{what} seq {s} edges h{h}"


def _run_varlen(cuda_lib, seqs, lens, table):
    cu = _cu(lens)
    empty = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    q = cuda_lib.pack_varlen([x[0][0] if x else empty for x in seqs])
    k = cuda_lib.pack_varlen([x[1][0] if x else empty for x in seqs])
    v = cuda_lib.pack_varlen([x[2][0] if x else empty for x in seqs])
    lse = torch.empty(HQ * cu[-1], device="cuda")
    edges = torch.zeros(len(lens) * HQ, dtype=torch.int64, device="cuda")
    layer = cuda_lib.VarlenLayer(table, cu, HQ, HKV, D, "cuda")
    o = layer(q, k, v, lse=lse, edges=edges)
    assert cuda_lib.poll_device_status() == 0
    outs = cuda_lib.unpack_varlen(o, HQ, cu, D)
    lses = [lse[HQ * cu[s]:HQ * cu[s + 1]].view(HQ, -1) for s in range(len(lens))]
    return layer, outs, lses, edges


@pytest.mark.gpu
def test_varlen_every_head_against_oracle(cuda_lib):
    """All rows of every head of every sequence of the packed batch."""
    seqs = _sequences("cuda")
    layer, outs, lses, edges = _run_varlen(cuda_lib, seqs, LENS, TABLE)
    for s, n in enumerate(LENS):
        if n:
            check_sequence_against_oracle(layer, s, n, *seqs[s], outs, lses, edges, TABLE)


@pytest.mark.gpu
@pytest.mark.timeout(900)
def test_varlen_many_sequences_against_oracle(cuda_lib):
    """72 sequences of mixed lengths (empty, a single row, ragged tails, up to
    5000 tokens) in one index pass and one attention pass: every head's
    index against the oracle and 96 seeded rows per head and sequence (rows 0,
    63, 64 and n-1 included)."""
    rng = np.random.default_rng(4242)
    lens = [int(x) for x in rng.integers(1, 5000, size=68)] + [0, 1, 64, 129]
    rng.shuffle(lens)
    seqs = [synth.random_qkv(1, HQ, HKV, n, D, seed=7000 + s, device="cuda") if n else None
            for s, n in enumerate(lens)]
    l0 = cuda_lib.kernel_launches()
    layer, outs, lses, edges = _run_varlen(cuda_lib, seqs, lens, TABLE)
    launches = cuda_lib.kernel_launches() - l0
    for s, n in enumerate(lens):
        if n:
            check_sequence_against_oracle(layer, s, n, *seqs[s], outs, lses, edges, TABLE,
                                          rows=synth.sample_rows(n, 96, seed=s), what="batch of 72")
    # one index pass (6 Vertical-Slash + 4 Block-Sparse launches) and one attention launch per
    # pattern of the table, the same as for a batch of two sequences
    two = [s for s, n in enumerate(lens) if n][:2]
    l0 = cuda_lib.kernel_launches()
    _run_varlen(cuda_lib, [seqs[s] for s in two], [lens[s] for s in two], TABLE)
    n_patterns = len({e["pattern"] for e in TABLE})
    assert cuda_lib.kernel_launches() - l0 == launches == 10 + n_patterns


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


@pytest.mark.gpu
def test_chunked_rows_against_oracle(cuda_lib):
    """Chunked prefill: indices built once over the whole sequence, then the
    attention run chunk by chunk (out of order); every row of every head of
    each chunk equals eq.(2) over the once-built sets (fp64 oracle)."""
    n, B = 1300, 2
    q, k, v = synth.random_qkv(B, HQ, HKV, n, D, seed=903, device="cuda")
    layer = cuda_lib.Layer(TABLE, B, HQ, HKV, n, D, "cuda")
    layer.index(q, k)
    o = torch.zeros_like(q)
    lse = torch.empty(B, HQ, n, device="cuda")
    edges = torch.zeros(B * HQ, dtype=torch.int64, device="cuda")
    vs, bidx, bcnt = layer.indices()
    vs_heads = [h for h, e in enumerate(TABLE) if e["pattern"] == "vs"]
    bs_heads = [h for h, e in enumerate(TABLE) if e["pattern"] == "block"]
    g = HQ // HKV
    for lo, hi in [(768, n), (0, 256), (256, 768)]:
        layer.attend_rows(q, k, v, o, lo, hi, lse=lse, edges=edges)
        assert cuda_lib.poll_device_status() == 0
        rows = np.arange(lo, hi)
        for b in range(B):
            for h, entry in enumerate(TABLE):
                qn, kn, vn = f32(q[b, h]), f32(k[b, h // g]), f32(v[b, h // g])
                idx = {}
                if entry["pattern"] == "vs":
                    x = b * len(vs_heads) + vs_heads.index(h)
                    idx = dict(C=vs.vertical[x, :int(vs.vertical_cnt[x])].cpu().numpy(),
                               D=vs.slash[x, :int(vs.slash_cnt[x])].cpu().numpy())
                elif entry["pattern"] == "block":
                    x = bs_heads.index(h)
                    idx = dict(J=bidx[b, x].cpu().numpy(), cnt=bcnt[b, x].cpu().numpy())
                ro, rl, _ = oracle.head_rows(oracle_cfg(entry), qn, kn, vn, rows, D ** -0.5, **idx)
                compare_rows(f32(o[b, h])[rows], f32(lse[b, h])[rows], ro, rl, f"rows [{lo}, {hi}) b{b} h{h}")
    for b in range(B):
        for h, entry in enumerate(TABLE):
            idx = {}
            if entry["pattern"] == "vs":
                x = b * len(vs_heads) + vs_heads.index(h)
                idx = dict(C=vs.vertical[x, :int(vs.vertical_cnt[x])].cpu().numpy(),
                           D=vs.slash[x, :int(vs.slash_cnt[x])].cpu().numpy())
            elif entry["pattern"] == "block":
                x = bs_heads.index(h)
                idx = dict(J=bidx[b, x].cpu().numpy(), cnt=bcnt[b, x].cpu().numpy())
            assert int(edges[b * HQ + h]) == oracle.head_edges(oracle_cfg(entry), n, **idx), f"edges b{b} h{h}"
