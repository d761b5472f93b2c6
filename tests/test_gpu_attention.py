"""GPU parity of the three sparse attention kernels with a fixed index (the
MInference page's first test layer, §5.2: fixed index, kernel vs plain masked
attention).  The oracle evaluates eq.(2) over each row's set in fp64; the
kernels run through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import compare_rows, cover_bits, f32, head_qkv, pack_bits, scale_of

pytestmark = pytest.mark.gpu


def _ashape_case(msa, B, Hq, Hkv, n, d, heads, sink, window, seed, rows=None):
    q, k, v = synth.random_qkv(B, Hq, Hkv, n, d, seed, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.full((B, Hq, n), 7.0, device="cuda")
    edges = torch.zeros(B * Hq, dtype=torch.int64, device="cuda")
    msa.attn_ashape(q, k, v, heads, sink, window, o=o, lse=lse, edges=edges)
    assert msa.poll_device_status() == 0
    rows = np.arange(n) if rows is None else rows
    cfg = dict(pattern=oracle.ASHAPE, sink=sink, window=window)
    for b in range(B):
        for h in heads:
            qn, kn, vn = head_qkv(q, k, v, b, h, Hq, Hkv)
            ro, rl, _ = oracle.head_rows(cfg, qn, kn, vn, rows, scale_of(d))
            compare_rows(f32(o[b, h])[rows], f32(lse[b, h])[rows], ro, rl, f"ashape b{b} h{h}")
            assert int(edges[b * Hq + h]) == oracle.head_edges(cfg, n)
    untouched = [h for h in range(Hq) if h not in heads]
    for h in untouched:
        assert torch.all(o[:, h] == 0) and torch.all(lse[:, h] == 7.0)


def test_ashape_tiny_head(cuda_lib):
    """The tiny workload's A-shape head (sink 64, window 512, d=64), all rows."""
    w = synth.make_workload("tiny", device="cuda")
    q, k, v = w["q"], w["k"], w["v"]
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 2048, device="cuda")
    cuda_lib.attn_ashape(q, k, v, [0], 64, 512, o=o, lse=lse)
    assert cuda_lib.poll_device_status() == 0
    qn, kn, vn = head_qkv(q, k, v, 0, 0, 2, 1)
    ro, rl, _ = oracle.head_rows(dict(pattern=oracle.ASHAPE, sink=64, window=512), qn, kn, vn, np.arange(2048), 0.125)
    compare_rows(f32(o[0, 0]), f32(lse[0, 0]), ro, rl, "tiny ashape")


@pytest.mark.parametrize("n,d,sink,window", [
    (1000, 128, 128, 300),   # ragged tail, window not a tile multiple
    (777, 64, 0, 1),         # no sink, diagonal only
    (300, 128, 5, 1000),     # budgets cover every key: dense causal
    (1024, 128, 200, 129),   # sink wider than a tile
    (65, 128, 3, 17),        # a single partial tile
])
def test_ashape_shapes(cuda_lib, n, d, sink, window):
    _ashape_case(cuda_lib, 1, 4, 2, n, d, [0, 3], sink, window, seed=n + d)


@pytest.mark.parametrize("heads", [[1, 2], [0, 1, 3]])
def test_ashape_batch_gqa(cuda_lib, heads):
    """Heads of one KV group share an item (a pair; a pair plus a single)."""
    _ashape_case(cuda_lib, 2, 4, 1, 513, 128, heads, 64, 256, seed=7)


def _bs_index_host(q, k, b, heads, Hq, Hkv, topk):
    J, C = [], []
    for h in heads:
        qn, kn, _ = head_qkv(q, k, k, b, h, Hq, Hkv)
        Jh, ch = oracle.bs_index(qn, kn, 64, topk)
        J.append(Jh)
        C.append(ch)
    return np.stack(J), np.stack(C)


@pytest.mark.parametrize("heads,Hq,Hkv", [
    ([0, 1], 4, 1),              # a pair
    ([2], 4, 2),                 # a single head
    ([0, 1, 3], 4, 2),           # a pair and a single in two groups
    ([0, 1, 2, 3], 4, 1),        # four heads of one group
    ([0, 1, 2, 3, 4, 6], 8, 1),  # four heads, then a pair
    ([7, 1, 2, 0, 5], 8, 1),     # four heads, then a single
])
def test_block_with_oracle_index(cuda_lib, heads, Hq, Hkv):
    """Block-Sparse attention on the oracle's J for every way heads are grouped into items."""
    B, n, d, topk = 1, 1000, 128, 4
    q, k, v = synth.random_qkv(B, Hq, Hkv, n, d, seed=11 + len(heads), device="cuda")
    J, C = _bs_index_host(q, k, 0, heads, Hq, Hkv, topk)
    bidx = torch.from_numpy(J[None]).cuda()
    bcnt = torch.from_numpy(C[None]).cuda()
    o = torch.zeros_like(q)
    lse = torch.empty(B, Hq, n, device="cuda")
    edges = torch.zeros(B * Hq, dtype=torch.int64, device="cuda")
    cuda_lib.attn_block(q, k, v, heads, topk, bidx, bcnt, o=o, lse=lse, edges=edges)
    assert cuda_lib.poll_device_status() == 0
    for x, h in enumerate(heads):
        qn, kn, vn = head_qkv(q, k, v, 0, h, Hq, Hkv)
        cfg = dict(pattern=oracle.BLOCK, block=64, topk=topk)
        ro, rl, _ = oracle.head_rows(cfg, qn, kn, vn, np.arange(n), scale_of(d), J=J[x], cnt=C[x])
        compare_rows(f32(o[0, h]), f32(lse[0, h]), ro, rl, f"block h{h}")
        assert int(edges[h]) == oracle.head_edges(cfg, n, J=J[x], cnt=C[x])


def _vs_case(msa, n, d, C, D, seed, Hq=2, Hkv=1):
    q, k, v = synth.random_qkv(1, Hq, Hkv, n, d, seed, device="cuda")
    index = msa.VSIndex(Hq, n, max(len(C), 1), max(len(D), 1), "cuda")
    for h in range(Hq):
        index.vertical_bits[h] = torch.from_numpy(pack_bits(C[h], n)).cuda()
        index.slash_bits[h] = torch.from_numpy(pack_bits(D[h], n)).cuda()
        index.slash_cover[h] = torch.from_numpy(cover_bits(D[h], n)).cuda()
    o = torch.zeros_like(q)
    lse = torch.empty(1, Hq, n, device="cuda")
    edges = torch.zeros(Hq, dtype=torch.int64, device="cuda")
    msa.attn_vs(q, k, v, list(range(Hq)), index, o=o, lse=lse, edges=edges)
    assert msa.poll_device_status() == 0
    for h in range(Hq):
        qn, kn, vn = head_qkv(q, k, v, 0, h, Hq, Hkv)
        cfg = dict(pattern=oracle.VS, block=64)
        ro, rl, _ = oracle.head_rows(cfg, qn, kn, vn, np.arange(n), scale_of(d), C=C[h], D=D[h])
        compare_rows(f32(o[0, h]), f32(lse[0, h]), ro, rl, f"vs h{h}")
        assert int(edges[h]) == oracle.head_edges(cfg, n, C=C[h], D=D[h])


def test_vs_with_given_index(cuda_lib):
    rng = np.random.default_rng(3)
    n = 1500
    C = [np.sort(rng.choice(n, 40, replace=False)), np.array([0, 5, 700, 1499])]
    D = [np.sort(rng.choice(n, 30, replace=False))[::-1], np.array([0, 37, 300])]
    _vs_case(cuda_lib, n, 128, C, D, seed=5)


def test_vs_sparse_slashes_gather_columns(cuda_lib):
    """Few far slashes leave most 128-key windows without slash coverage, so
    the verticals there go through the column-gather tiles."""
    rng = np.random.default_rng(9)
    n = 4000
    C = [np.sort(rng.choice(n, 300, replace=False)), np.sort(rng.choice(n, 7, replace=False))]
    D = [np.array([3000, 1000, 0]), np.array([2500])]
    _vs_case(cuda_lib, n, 64, C, D, seed=6)


def test_vs_single_heads_odd_tiles(cuda_lib):
    """One head per KV group (each head's even and odd tiles share an item) with
    an odd number of query tiles, so the last item has one tile."""
    rng = np.random.default_rng(12)
    n = 1100
    C = [np.sort(rng.choice(n, 25, replace=False)), np.sort(rng.choice(n, 60, replace=False))]
    D = [np.array([900, 400, 130, 64, 1, 0]), np.sort(rng.choice(n, 40, replace=False))[::-1]]
    _vs_case(cuda_lib, n, 128, C, D, seed=13, Hq=2, Hkv=2)


def test_vs_empty_sets(cuda_lib):
    """No verticals and no slashes: every row's set is empty (o = 0, lse = -inf)."""
    _vs_case(cuda_lib, 300, 128, [np.array([], np.int64)] * 2, [np.array([], np.int64)] * 2, seed=8)


def test_vs_dense_when_all_offsets(cuda_lib):
    n = 700
    _vs_case(cuda_lib, n, 128, [np.array([], np.int64)] * 2, [np.arange(n)[::-1]] * 2, seed=10)


@pytest.mark.parametrize("n,d", [(1000, 128), (333, 64)])
def test_dense_causal_matches_sdpa(cuda_lib, n, d):
    """msa_attn_dense against the oracle's dense pattern and against torch's
    fp64 causal SDPA (eq.(1)-(2) with N(i) = {0..i}); E = n(n+1)/2 per head."""
    q, k, v = synth.random_qkv(1, 4, 2, n, d, seed=n, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(1, 4, n, device="cuda")
    edges = torch.zeros(4, dtype=torch.int64, device="cuda")
    cuda_lib.attn_dense(q, k, v, [0, 1, 2, 3], o=o, lse=lse, edges=edges)
    assert cuda_lib.poll_device_status() == 0
    for h in range(4):
        qn, kn, vn = head_qkv(q, k, v, 0, h, 4, 2)
        ro, rl, _ = oracle.head_rows(dict(pattern=oracle.DENSE), qn, kn, vn, np.arange(n), scale_of(d))
        compare_rows(f32(o[0, h]), f32(lse[0, h]), ro, rl, f"dense h{h}")
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qn).double()[None], torch.from_numpy(kn).double()[None],
            torch.from_numpy(vn).double()[None], is_causal=True, scale=scale_of(d))[0].numpy()
        assert np.abs(f32(o[0, h]) - ref).max() <= 1.5e-2
        assert int(edges[h]) == n * (n + 1) // 2


@pytest.mark.parametrize("pattern", ["dense", "ashape"])
def test_extreme_logits(cuda_lib, pattern):
    """Logits of order ±100 whose scale grows along the key axis, so later
    key tiles raise each row's running maximum by tens of units and the
    online rescale of eq.(7)-(8) (MInference page §3.2) drops earlier
    partial sums to underflow; the result must still be eq.(2) over the set."""
    n, d, Hq, Hkv = 1000, 128, 2, 1
    q, k, v = synth.random_qkv(1, Hq, Hkv, n, d, seed=91, device="cuda", scale_q=8.0)
    ramp = torch.linspace(1.0, 4.0, n, device="cuda")[None, None, :, None]
    k = (k.float() * ramp).to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(1, Hq, n, device="cuda")
    if pattern == "dense":
        cuda_lib.attn_dense(q, k, v, [0, 1], o=o, lse=lse)
        cfg = dict(pattern=oracle.DENSE)
    else:
        cuda_lib.attn_ashape(q, k, v, [0, 1], 16, 300, o=o, lse=lse)
        cfg = dict(pattern=oracle.ASHAPE, sink=16, window=300)
    assert cuda_lib.poll_device_status() == 0
    for h in range(Hq):
        qn, kn, vn = head_qkv(q, k, v, 0, h, Hq, Hkv)
        ro, rl, _ = oracle.head_rows(cfg, qn, kn, vn, np.arange(n), scale_of(d))
        assert rl.max() > 60.0  # the case really reaches large logits
        compare_rows(f32(o[0, h]), f32(lse[0, h]), ro, rl, f"{pattern} extreme h{h}")


def test_extreme_logits_vs(cuda_lib):
    """The same ramped large logits on Vertical-Slash heads. Keys that a whole
    64-row half leaves out reach the softmax as the most negative finite bf16
    added to their score (the tensor-core masking step), so attended scores of
    any sign and size must still give eq.(2) over the physical set."""
    n, d, Hq, Hkv = 1000, 128, 2, 1
    q, k, v = synth.random_qkv(1, Hq, Hkv, n, d, seed=92, device="cuda", scale_q=8.0)
    ramp = torch.linspace(1.0, 4.0, n, device="cuda")[None, None, :, None]
    k = (k.float() * ramp).to(torch.bfloat16)
    rng = np.random.default_rng(93)
    C = [np.sort(rng.choice(n, 30, replace=False)), np.array([0, 999])]
    D = [np.sort(rng.choice(n, 20, replace=False))[::-1], np.array([400, 3, 0])]
    index = cuda_lib.VSIndex(Hq, n, 30, 20, "cuda")
    for h in range(Hq):
        index.vertical_bits[h] = torch.from_numpy(pack_bits(C[h], n)).cuda()
        index.slash_bits[h] = torch.from_numpy(pack_bits(D[h], n)).cuda()
        index.slash_cover[h] = torch.from_numpy(cover_bits(D[h], n)).cuda()
    o = torch.empty_like(q)
    lse = torch.empty(1, Hq, n, device="cuda")
    cuda_lib.attn_vs(q, k, v, [0, 1], index, o=o, lse=lse)
    assert cuda_lib.poll_device_status() == 0
    for h in range(Hq):
        qn, kn, vn = head_qkv(q, k, v, 0, h, Hq, Hkv)
        cfg = dict(pattern=oracle.VS, block=64)
        ro, rl, _ = oracle.head_rows(cfg, qn, kn, vn, np.arange(n), scale_of(d), C=C[h], D=D[h])
        assert np.nanmax(rl[np.isfinite(rl)]) > 60.0
        compare_rows(f32(o[0, h]), f32(lse[0, h]), ro, rl, f"vs extreme h{h}")


@pytest.mark.parametrize("n,topk", [
    (700, 20),            # k_b above N_b = 11
    (64 * 520 + 17, 521),  # k_b = N_b = 521: the last rows' lists exceed the 512 entries staged in shared memory
])
def test_block_budget_covering_every_key_is_dense(cuda_lib, n, topk):
    """Block-Sparse with k_b >= N_b (index built on the device, attention on
    its lists) reduces to dense causal attention, eq.(1)-(2): J_u = {0..u},
    E = n(n+1)/2.  The long case takes the path that reads lists longer than
    the shared-memory stage straight from global memory."""
    d, Hq, Hkv = 128, 2, 1
    q, k, v = synth.random_qkv(1, Hq, Hkv, n, d, seed=n, device="cuda")
    bidx, bcnt = cuda_lib.build_block_index(q, k, [1], topk)
    assert cuda_lib.poll_device_status() == 0
    nb = (n + 63) // 64
    cnt = bcnt[0, 0].cpu().numpy()
    assert (cnt == np.minimum(np.arange(nb) + 1, topk)).all()
    idx = bidx[0, 0].cpu().numpy()
    for u in range(nb):
        assert (idx[u, :u + 1] == np.arange(u + 1)).all(), f"block {u}"
    o = torch.zeros_like(q)
    lse = torch.empty(1, Hq, n, device="cuda")
    edges = torch.zeros(Hq, dtype=torch.int64, device="cuda")
    cuda_lib.attn_block(q, k, v, [1], topk, bidx, bcnt, o=o, lse=lse, edges=edges)
    assert cuda_lib.poll_device_status() == 0
    rows = np.arange(n) if n <= 1000 else synth.sample_rows(n, 96, seed=3)
    if n > 1000:
        rows = np.unique(np.concatenate([rows, np.arange(n - 130, n)]))  # the blocks with > 512 entries
    qn, kn, vn = head_qkv(q, k, v, 0, 1, Hq, Hkv)
    ro, rl, _ = oracle.head_rows(dict(pattern=oracle.DENSE), qn, kn, vn, rows, scale_of(d))
    compare_rows(f32(o[0, 1])[rows], f32(lse[0, 1])[rows], ro, rl, f"block dense n{n}")
    assert int(edges[1]) == n * (n + 1) // 2
    assert torch.all(o[0, 0] == 0)


@pytest.mark.parametrize("heads,Hq,Hkv", [
    ([0, 1], 4, 1),                 # a pair of heads
    ([2], 4, 2),                    # a single head: its even and odd tiles
    ([0, 1, 2, 3], 4, 1),           # two pairs of one group
    ([0, 1, 2, 3, 4, 6], 8, 1),     # three pairs
    ([7, 1, 2, 0, 5], 8, 1),        # two pairs, then a single
    ([0, 1, 3, 4, 5, 6, 7], 8, 2),  # a pair and a single in one group, two pairs in the other
])
def test_vs_head_groupings(cuda_lib, heads, Hq, Hkv):
    """Vertical-Slash attention on head subsets that pair into items in every
    way (each sub-item reads its own head's index); per-head random verticals
    and slashes, partly shared, so that an item's key stream mixes common and
    private keys."""
    n, d = 1000, 128
    rng = np.random.default_rng(31 + len(heads))
    q, k, v = synth.random_qkv(1, Hq, Hkv, n, d, seed=17 + len(heads), device="cuda")
    C0, D0 = rng.choice(n, 30, replace=False), rng.choice(n, 20, replace=False)
    C, D = [], []
    index = cuda_lib.VSIndex(len(heads), n, 60, 40, "cuda")
    for x in range(len(heads)):
        Cx = np.unique(np.concatenate([C0[:20], rng.choice(n, 25, replace=False)]))
        Dx = np.unique(np.concatenate([D0[:12], rng.choice(n, 15, replace=False), [0]]))[::-1]
        C.append(Cx)
        D.append(Dx)
        index.vertical_bits[x] = torch.from_numpy(pack_bits(Cx, n)).cuda()
        index.slash_bits[x] = torch.from_numpy(pack_bits(Dx, n)).cuda()
        index.slash_cover[x] = torch.from_numpy(cover_bits(Dx, n)).cuda()
    o = torch.zeros_like(q)
    lse = torch.empty(1, Hq, n, device="cuda")
    edges = torch.zeros(Hq, dtype=torch.int64, device="cuda")
    cuda_lib.attn_vs(q, k, v, heads, index, o=o, lse=lse, edges=edges)
    assert cuda_lib.poll_device_status() == 0
    cfg = dict(pattern=oracle.VS, block=64)
    for x, h in enumerate(heads):
        qn, kn, vn = head_qkv(q, k, v, 0, h, Hq, Hkv)
        ro, rl, _ = oracle.head_rows(cfg, qn, kn, vn, np.arange(n), scale_of(d), C=C[x], D=D[x])
        compare_rows(f32(o[0, h]), f32(lse[0, h]), ro, rl, f"vs h{h}")
        assert int(edges[h]) == oracle.head_edges(cfg, n, C=C[x], D=D[x])
    for h in range(Hq):
        if h not in heads:
            assert torch.all(o[0, h] == 0)
