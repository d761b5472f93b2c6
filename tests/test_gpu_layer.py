"""GPU parity of msa_prefill_layer (table dispatch, online indices and the
single attention launch) against the fp64 oracle.

Attention is checked on the GPU's own index sets (so the comparison isolates
the kernels); the index sets themselves are checked against the oracle's."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import compare_rows, f32, head_qkv, oracle_cfg
from test_gpu_index import check_bs_against_oracle, check_vs_against_oracle

pytestmark = pytest.mark.gpu


def run_layer(msa, w, rows_per_head=None, check_index=True, exact_index=False):
    q, k, v, table, sh = w["q"], w["k"], w["v"], w["table"], w["shape"]
    B, Hq, Hkv, n, d = sh["B"], sh["Hq"], sh["Hkv"], sh["n"], sh["d"]
    layer = msa.Layer(table, B, Hq, Hkv, n, d, q.device)
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, n, device=q.device)
    edges = torch.zeros(B * Hq, dtype=torch.int64, device=q.device)
    layer(q, k, v, o=o, lse=lse, edges=edges)
    assert msa.poll_device_status() == 0
    vs, bidx, bcnt = layer.indices()
    vs_heads = [h for h, e in enumerate(table) if e["pattern"] == "vs"]
    bs_heads = [h for h, e in enumerate(table) if e["pattern"] == "block"]
    if check_index and vs_heads:
        e = table[vs_heads[0]]
        check_vs_against_oracle(vs, q, k, vs_heads, e["last_q"], e["n_vertical"], e["n_slash"], exact=exact_index)
    if check_index and bs_heads:
        check_bs_against_oracle(bidx, bcnt, q, k, bs_heads, table[bs_heads[0]]["topk"])
    rows = np.arange(n) if rows_per_head is None else synth.sample_rows(n, rows_per_head, seed=n)
    for b in range(B):
        for h, entry in enumerate(table):
            qn, kn, vn = head_qkv(q, k, v, b, h, Hq, Hkv)
            cfg = oracle_cfg(entry)
            idx = {}
            if entry["pattern"] == "vs":
                slot = b * len(vs_heads) + vs_heads.index(h)
                idx = dict(C=vs.vertical[slot, :int(vs.vertical_cnt[slot])].cpu().numpy(),
                           D=vs.slash[slot, :int(vs.slash_cnt[slot])].cpu().numpy())
            elif entry["pattern"] == "block":
                x = bs_heads.index(h)
                idx = dict(J=bidx[b, x].cpu().numpy(), cnt=bcnt[b, x].cpu().numpy())
            ro, rl, _ = oracle.head_rows(cfg, qn, kn, vn, rows, sh["scale"], **idx)
            compare_rows(f32(o[b, h])[rows], f32(lse[b, h])[rows], ro, rl, f"layer b{b} h{h} {entry['pattern']}")
            assert int(edges[b * Hq + h]) == oracle.head_edges(cfg, n, **idx), f"edges h{h}"
    return layer


def test_layer_tiny_all_rows(cuda_lib):
    """The tiny workload end to end: every row of both heads, exact indices."""
    run_layer(cuda_lib, synth.make_workload("tiny", device="cuda"), exact_index=True)


def test_layer_mixed_reduced(cuda_lib):
    """Mixed-pattern table (A-shape / Vertical-Slash / Block-Sparse, 1:6:1) at
    n = 4096 with 8 query heads over 2 KV heads, sampled rows."""
    w = synth.make_workload("mixed", device="cuda", n=4096, Hq=8, Hkv=2)
    run_layer(cuda_lib, w, rows_per_head=300)


def test_layer_ragged_batch(cuda_lib):
    """B = 2, ragged n, a table with every pattern and paired Block-Sparse heads."""
    q, k, v = synth.random_qkv(2, 8, 2, 1111, 128, seed=77, device="cuda")
    table = [synth.ashape(16, 100), synth.vslash(64, 20, 50), synth.blocksparse(6), synth.blocksparse(6),
             synth.vslash(64, 20, 50), synth.ashape(0, 64), synth.blocksparse(6), synth.vslash(64, 20, 50)]
    w = dict(q=q, k=k, v=v, table=table, shape=dict(B=2, Hq=8, Hkv=2, n=1111, d=128, scale=128 ** -0.5))
    run_layer(cuda_lib, w, rows_per_head=200)


def test_layer_one_group_pairings(cuda_lib):
    """One KV group: an A-shape pair with different sink/window, four
    Block-Sparse heads in one item, a Vertical-Slash pair (d = 64)."""
    q, k, v = synth.random_qkv(1, 8, 1, 1000, 64, seed=78, device="cuda")
    table = [synth.ashape(16, 100), synth.blocksparse(5), synth.vslash(32, 30, 40), synth.blocksparse(5),
             synth.ashape(0, 300), synth.blocksparse(5), synth.vslash(32, 30, 40), synth.blocksparse(5)]
    w = dict(q=q, k=k, v=v, table=table, shape=dict(B=1, Hq=8, Hkv=1, n=1000, d=64, scale=64 ** -0.5))
    run_layer(cuda_lib, w)


def test_attend_stats_counts(cuda_lib):
    """msa_layer_attend_stats: the same output and edge counts as
    msa_layer_attend, and per head a tile count whose (row, key) area covers
    the head's attended edges."""
    w = synth.make_workload("mixed", device="cuda", n=3000, Hq=8, Hkv=2)
    q, k, v, table, sh = w["q"], w["k"], w["v"], w["table"], w["shape"]
    layer = cuda_lib.Layer(table, 1, sh["Hq"], sh["Hkv"], sh["n"], sh["d"], "cuda")
    layer.index(q, k)
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    e1 = torch.zeros(sh["Hq"], dtype=torch.int64, device="cuda")
    e2 = torch.zeros_like(e1)
    tiles = torch.zeros_like(e1)
    layer.attend(q, k, v, o1, edges=e1)
    layer.attend_stats(q, k, v, o2, edges=e2, tiles=tiles)
    assert cuda_lib.poll_device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(e1, e2)
    t, e = tiles.cpu().numpy(), e1.cpu().numpy()
    assert np.all(t * 64 * 128 >= e) and np.all(t > 0)
    # every query block of a head is processed in at least one tile
    assert np.all(t >= (sh["n"] + 63) // 64)


def test_pattern_kernels_agree_with_the_mixed_kernel(cuda_lib):
    """A launch of one pattern runs a kernel compiled for that pattern alone;
    a mixed table runs the kernel that holds all three.  On the same heads and
    the same index the two must produce the same bits (same items, same tiles,
    same arithmetic; the calls group the heads as the layer does).  A-shape
    heads are left out: the layer pairs them across heads, a lone call pairs a
    head's even and odd tiles."""
    w = synth.make_workload("mixed", device="cuda", n=3000, Hq=8, Hkv=2)
    q, k, v, table, sh = w["q"], w["k"], w["v"], w["table"], w["shape"]
    layer = cuda_lib.Layer(table, 1, sh["Hq"], sh["Hkv"], sh["n"], sh["d"], "cuda")
    o_mix = torch.empty_like(q)
    layer(q, k, v, o=o_mix)
    assert cuda_lib.poll_device_status() == 0
    vs, bidx, bcnt = layer.indices()
    vs_heads = [h for h, e in enumerate(table) if e["pattern"] == "vs"]
    bs_heads = [h for h, e in enumerate(table) if e["pattern"] == "block"]
    assert vs_heads and bs_heads
    o_one = torch.zeros_like(q)
    cuda_lib.attn_vs(q, k, v, vs_heads, vs, o=o_one)
    cuda_lib.attn_block(q, k, v, bs_heads, table[bs_heads[0]]["topk"], bidx, bcnt, o=o_one)
    assert cuda_lib.poll_device_status() == 0
    for h in vs_heads + bs_heads:
        assert torch.equal(o_one[0, h], o_mix[0, h]), f"head {h} ({table[h]['pattern']})"
