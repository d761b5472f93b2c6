"""Pins of the fp64 oracle to what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a value the
pages print (fixtures under tests/golden/, each with its citation), a closed
form, an invariant, a library routine the case reduces to, or brute force on a
tiny input.  The tests are chosen so that a dropped term, a wrong sign or index
or a transposed operand in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------- worked example
def _worked_inputs(g):
    n = g["n"]
    q = np.tile(np.asarray(g["filler_k"], np.float32), (n, 1))
    k = np.tile(np.asarray(g["filler_k"], np.float32), (n, 1))
    v = np.tile(np.asarray(g["filler_v"], np.float32), (n, 1))
    q[g["row"]] = g["q6"]
    for j, x in g["k"].items():
        k[int(j)] = x
    for j, x in g["v"].items():
        v[int(j)] = x
    return q, k, v


def test_worked_example_set_and_output():
    g = gold("vs_worked_example.json")
    q, k, v = _worked_inputs(g)
    i = g["row"]
    s = oracle.vs_logical_set(i, g["C"], g["D"])
    assert s.tolist() == g["expected_set"]
    # the physical set with one-row query blocks is the logical set
    assert oracle.vs_physical_set(i, g["n"], 1, g["C"], g["D"]).tolist() == g["expected_set"]
    o, lse = oracle.attend(q, k, v, i, s, g["scale"])
    np.testing.assert_allclose(o, g["printed_o6"], atol=g["printed_tolerance"])
    e = math.e
    np.testing.assert_allclose(o, [3 * e / (2 * e + 1), (e + 2) / (2 * e + 1)], rtol=0, atol=1e-13)
    assert abs(lse - math.log(2 * e * e + e)) < 1e-13  # eq.(10): Z = 2e^2 + e
    # through the per-head driver, Vertical-Slash pattern with 1-row blocks
    o2, lse2, size = oracle.head_rows(dict(pattern=oracle.VS, block=1), q, k, v, [i], g["scale"], C=g["C"], D=g["D"])
    assert size.tolist() == [3]
    np.testing.assert_allclose(o2[0], o, atol=1e-15)


def test_worked_example_dedup_and_negative_offset():
    g = gold("vs_worked_example.json")
    q, k, v = _worked_inputs(g)
    # vertical and slash both hit 6: it enters the softmax once -> output v6 exactly
    s = oracle.vs_logical_set(6, [6], [0])
    assert s.tolist() == [6]
    o, _ = oracle.attend(q, k, v, 6, s, 1.0)
    np.testing.assert_array_equal(o, v[6])
    # offset 2 at row 1 is negative and is clipped: nothing left
    assert oracle.vs_logical_set(1, [], [2]).size == 0
    o, lse = oracle.attend(q, k, v, 1, np.zeros(0, np.int64), 1.0)
    assert np.all(o == 0) and lse == -math.inf
    assert oracle.vs_logical_set(1, [], [0, 2]).tolist() == [1]


# ----------------------------------------------------------------- proxy aggregation
def test_proxy_topk_example_eq12():
    g = gold("proxy_topk_example.json")
    P = np.asarray(g["P"])
    c, _ = oracle.proxy_aggregate(P, [6, 7])
    np.testing.assert_allclose(c, g["column_sum"], atol=1e-15)
    assert oracle.topk(c, 1).tolist() == [g["selected_top1"]]
    assert oracle.topk(P.max(axis=0), 1).tolist() == [g["selected_top1"]]
    np.testing.assert_allclose(P.max(axis=0), g["printed_column_max"])
    # the column-maximum convention reproduces the printed maxima and the same choice
    cm, _ = oracle.proxy_aggregate(P, [6, 7], oracle.PROXY_COL_MAX)
    np.testing.assert_allclose(cm, g["printed_column_max"], atol=1e-15)
    assert oracle.topk(cm, 1).tolist() == [g["selected_top1"]]


def test_proxy_slash_mean_counts_legal_pairs():
    """Slash mean (MInference page §6.2: offset d has fewer legal pairs than a
    short one): with every proxy probability 1 on the causal part, each legal
    pair adds 1, so the sum of r_d is the number of legal pairs (rows with
    pos >= d) and the mean is exactly 1 for every offset that has one, 0 else."""
    n, pos = 10, [6, 7, 8, 9]
    A = np.zeros((4, n))
    for t, i in enumerate(pos):
        A[t, :i + 1] = 1.0
    _, rs = oracle.proxy_aggregate(A, pos)
    assert rs.tolist() == [sum(1 for i in pos if i >= d) for d in range(n)]
    _, rm = oracle.proxy_aggregate(A, pos, oracle.PROXY_SLASH_MEAN)
    assert rm.tolist() == [1.0] * n
    A2 = A.copy()
    A2[:, 0] = 0.0  # key 0 dropped: offsets d = pos reach only key 0
    _, rm2 = oracle.proxy_aggregate(A2, pos, oracle.PROXY_SLASH_MEAN)
    for d in range(n):
        legal = [i for i in pos if i >= d]
        want = sum(1.0 for i in legal if i - d != 0) / len(legal)
        assert rm2[d] == want
    # column max and sum agree when a single row is sampled
    c1, _ = oracle.proxy_aggregate(A[:1], pos[:1])
    cm1, _ = oracle.proxy_aggregate(A[:1], pos[:1], oracle.PROXY_COL_MAX)
    assert c1.tolist() == cm1.tolist()


def test_proxy_slash_indexing_one_hot():
    """A proxy matrix with a single 1 per row on the diagonal offset 3 puts all
    of its mass on r_3 and spreads c over the columns i-3 (a transposed or
    sign-flipped slash index fails this)."""
    n, pos = 12, [8, 9, 10, 11]
    A = np.zeros((4, n))
    for t, i in enumerate(pos):
        A[t, i - 3] = 1.0
    c, r = oracle.proxy_aggregate(A, pos)
    assert r[3] == 4 and r.sum() == 4
    assert c.tolist() == [0, 0, 0, 0, 0, 1, 1, 1, 1, 0, 0, 0]


def _onehot_qk(n, d, targets, big):
    """k_j = e_j; q_i = big * e_{targets[i]} so s_ij = big iff j == targets[i]."""
    k = np.eye(n, d, dtype=np.float32)
    q = np.zeros((n, d), np.float32)
    for i, j in targets.items():
        q[i, j] = big
    return q, k


def test_proxy_vertical_concentration():
    """Every sampled row puts (numerically) all of its probability on column 5:
    c = L e_5 and r_d = 1 at d = i - 5 for each sampled row i."""
    n, L = 40, 6
    q, k = _onehot_qk(n, n, {i: 5 for i in range(n - L, n)}, 1000.0)
    c, r = oracle.vs_proxy(q, k, L, 1.0)
    exp_c = np.zeros(n)
    exp_c[5] = L
    np.testing.assert_array_equal(c, exp_c)
    exp_r = np.zeros(n)
    exp_r[[i - 5 for i in range(n - L, n)]] = 1.0
    np.testing.assert_array_equal(r, exp_r)


def test_proxy_slash_concentration():
    """Every sampled row i puts its probability on key i-7: r = L e_7."""
    n, L = 40, 5
    q, k = _onehot_qk(n, n, {i: i - 7 for i in range(n - L, n)}, 1000.0)
    c, r = oracle.vs_proxy(q, k, L, 1.0)
    exp_r = np.zeros(n)
    exp_r[7] = L
    np.testing.assert_array_equal(r, exp_r)
    exp_c = np.zeros(n)
    exp_c[[i - 7 for i in range(n - L, n)]] = 1.0
    np.testing.assert_array_equal(c, exp_c)


def test_proxy_uniform_closed_form():
    """Identical keys give Ã_ij = 1/(i+1) on the causal prefix, so
    c_j = Σ_{i in R, i >= j} 1/(i+1) and the same sum for r_d."""
    n, L, d = 50, 7, 4
    k = np.tile(np.array([0.5, -1.0, 2.0, 0.25], np.float32), (n, 1))
    q = np.random.default_rng(0).standard_normal((n, d)).astype(np.float32)
    c, r = oracle.vs_proxy(q, k, L, 0.5)
    rows = np.arange(n - L, n)
    want = np.array([sum(1.0 / (i + 1) for i in rows if i >= j) for j in range(n)])
    np.testing.assert_allclose(c, want, rtol=1e-13, atol=0)
    np.testing.assert_allclose(r, want, rtol=1e-13, atol=0)


def test_proxy_probs_match_library_softmax_and_mass():
    """Ã is a causal softmax of the scaled scores (torch.softmax in fp64); each
    sampled row carries mass 1, so Σ c = Σ r = L."""
    rng = np.random.default_rng(3)
    n, d, L, scale = 97, 16, 9, 0.37
    q = rng.standard_normal((n, d)).astype(np.float32)
    k = rng.standard_normal((n, d)).astype(np.float32)
    A = oracle.vs_proxy_probs(q, k, L, scale)
    qs = torch.from_numpy(q).double()[n - L:]
    s = scale * qs @ torch.from_numpy(k).double().T
    rows = torch.arange(n - L, n)[:, None]
    s = s.masked_fill(torch.arange(n)[None, :] > rows, float("-inf"))
    np.testing.assert_allclose(A, torch.softmax(s, dim=1).numpy(), rtol=1e-12, atol=1e-15)
    c, r = oracle.vs_proxy(q, k, L, scale)
    assert abs(c.sum() - L) < 1e-10 and abs(r.sum() - L) < 1e-10
    # last_q larger than n uses every row
    c2, r2 = oracle.vs_proxy(q[:5], k[:5], 64, scale)
    assert abs(c2.sum() - 5) < 1e-12 and abs(r2.sum() - 5) < 1e-12


# ----------------------------------------------------------------- top-k
@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 40))
    s = rng.integers(0, 6, size=n).astype(np.float64)  # many ties
    for kk in range(0, n + 3):
        got = oracle.topk(s, kk)
        beats = [sum(1 for l in range(n) if s[l] > s[j] or (s[l] == s[j] and l < j)) for j in range(n)]
        want = [j for j in range(n) if beats[j] < kk]
        assert sorted(got.tolist()) == want
        assert len(got) == min(kk, n)
        # best first
        assert all(s[got[t]] >= s[got[t + 1]] for t in range(len(got) - 1))


# ----------------------------------------------------------------- edge counts
def test_ashape_edge_counts_from_pages():
    g = gold("edge_counts.json")
    for case in g["cases"]:
        E = oracle.head_edges(dict(pattern=oracle.ASHAPE, sink=case["sink"], window=case["window"]), case["n"])
        assert E == case["E"], case["what"]


def test_ashape_count_closed_form():
    """|N_A(i)| = min(i+1, g+w); with g = 0 the total is n w - w(w-1)/2."""
    for (n, g, w) in [(300, 0, 17), (300, 5, 17), (64, 64, 1), (130, 3, 200), (257, 31, 64)]:
        sizes = [oracle.ashape_set(i, g, w).size for i in range(n)]
        assert sizes == [min(i + 1, g + w) for i in range(n)]
        assert oracle.head_edges(dict(pattern=oracle.ASHAPE, sink=g, window=w), n) == sum(sizes)
        if g == 0 and w <= n:
            assert sum(sizes) == n * w - w * (w - 1) // 2


def test_ashape_set_brute_force():
    n, g, w = 40, 3, 6
    for i in range(n):
        want = [j for j in range(i + 1) if j < g or j > i - w]
        assert oracle.ashape_set(i, g, w).tolist() == want


def test_vertical_edge_count():
    g = gold("edge_counts.json")["vertical"]
    cfg = dict(pattern=oracle.VS, block=64)
    assert oracle.head_edges(cfg, g["n"], C=g["C"], D=[]) == g["E"]
    assert sum(oracle.vs_logical_set(i, g["C"], []).size for i in range(g["n"])) == g["E"]


# ----------------------------------------------------------------- VS index
def test_vs_block_index_hand_example():
    g = gold("vs_block_example.json")
    for blk in g["blocks"]:
        ranges, cols = oracle.vs_block_index(blk["u"], g["n"], g["block"], g["C"], g["D"])
        assert ranges.tolist() == blk["ranges"], blk["why"]
        assert cols.tolist() == blk["cols"], blk["why"]


@pytest.mark.parametrize("seed", range(4))
def test_vs_physical_set_vs_logical(seed):
    """Block size 1 reduces the physical set to eq.(5); at block 64 the
    physical set contains the logical one, and the edge counter agrees with
    the per-row sets."""
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(70, 260))
    C = rng.choice(n, size=int(rng.integers(0, 12)), replace=False)
    D = rng.choice(n, size=int(rng.integers(0, 9)), replace=False)
    tot = 0
    for i in range(n):
        lg = oracle.vs_logical_set(i, C, D)
        assert oracle.vs_physical_set(i, n, 1, C, D).tolist() == lg.tolist()
        ph = oracle.vs_physical_set(i, n, 64, C, D)
        assert set(lg.tolist()) <= set(ph.tolist())
        assert ph.size == 0 or ph.max() <= i
        # definition of the 64-row tile: j covered iff some δ has a-δ <= j <= e-δ, or j in C
        a = (i // 64) * 64
        e = min(a + 64, n) - 1
        want = [j for j in range(i + 1) if j in set(C.tolist()) or any(a - dl <= j <= e - dl for dl in D)]
        assert ph.tolist() == want
        tot += ph.size
    assert oracle.head_edges(dict(pattern=oracle.VS, block=64), n, C=C, D=D) == tot
    assert oracle.head_edges(dict(pattern=oracle.VS, block=1), n, C=C, D=D) == sum(
        oracle.vs_logical_set(i, C, D).size for i in range(n))


# ----------------------------------------------------------------- block-sparse index
def test_bs_pool_partial_block():
    n, d, b = 150, 3, 64
    x = np.repeat(np.arange(n, dtype=np.float32)[:, None], d, axis=1)
    xb = oracle.bs_pool(x, b)
    np.testing.assert_allclose(xb[:, 0], [31.5, 95.5, (128 + 149) / 2.0])


def test_bs_index_planted_scores():
    """Block v of K is w_v e_v and every query is all-ones, so r_uv = w_v; J_u
    is {u} plus the k_b-1 best earlier blocks by w (ties to lower v)."""
    b, nb, kb = 4, 12, 4
    n = b * nb
    w = np.array([3, 7, 1, 7, 5, 2, 9, 4, 4, 6, 8, 0], np.float32)
    k = np.zeros((n, nb), np.float32)
    for vb in range(nb):
        k[vb * b:(vb + 1) * b, vb] = w[vb]
    q = np.ones((n, nb), np.float32)
    J, cnt = oracle.bs_index(q, k, b, kb)
    for u in range(nb):
        prev = sorted(range(u), key=lambda vb: (-w[vb], vb))[:kb - 1]
        want = sorted([u] + prev)
        assert J[u, :cnt[u]].tolist() == want
        assert cnt[u] == min(kb, u + 1)
        assert all(x == -1 for x in J[u, cnt[u]:])


def test_bs_edge_closed_form():
    rng = np.random.default_rng(5)
    b, nb, kb = 64, 9, 3
    n = b * nb
    q = rng.standard_normal((n, 8)).astype(np.float32)
    k = rng.standard_normal((n, 8)).astype(np.float32)
    J, cnt = oracle.bs_index(q, k, b, kb)
    E = oracle.head_edges(dict(pattern=oracle.BLOCK, block=b, topk=kb), n, J=J, cnt=cnt)
    assert E == sum((min(kb, u + 1) - 1) * b * b + b * (b + 1) // 2 for u in range(nb))
    # per-row sets agree with the counter
    assert E == sum(oracle.bs_set(i, n, b, J, cnt).size for i in range(n))


# ----------------------------------------------------------------- dense reduction
def _dense_ref(q, k, v, scale):
    qt, kt, vt = (torch.from_numpy(x).double()[None, None] for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale)
    return out[0, 0].numpy()


@pytest.mark.parametrize("n", [1, 5, 64, 150, 200])
def test_budgets_covering_every_key_equal_dense(n):
    """When the budgets cover every causal key, each pattern is dense causal
    attention (torch SDPA in fp64) and E = n(n+1)/2."""
    rng = np.random.default_rng(n)
    d = 16
    q = rng.standard_normal((n, d)).astype(np.float32)
    k = rng.standard_normal((n, d)).astype(np.float32)
    v = rng.standard_normal((n, d)).astype(np.float32)
    scale = 1 / math.sqrt(d)
    ref = _dense_ref(q, k, v, scale)
    rows = np.arange(n)
    nb = (n + 63) // 64
    J, cnt = oracle.bs_index(q, k, 64, nb)
    cases = [
        (dict(pattern=oracle.ASHAPE, sink=0, window=n), {}),
        (dict(pattern=oracle.ASHAPE, sink=n // 3, window=n - n // 3), {}),
        (dict(pattern=oracle.VS, block=64), dict(C=[], D=np.arange(n))),
        (dict(pattern=oracle.VS, block=64), dict(C=np.arange(n), D=[])),
        (dict(pattern=oracle.BLOCK, block=64, topk=nb), dict(J=J, cnt=cnt)),
        (dict(pattern=oracle.DENSE), {}),
    ]
    for cfg, idx in cases:
        o, lse, size = oracle.head_rows(cfg, q, k, v, rows, scale, **idx)
        np.testing.assert_allclose(o, ref, rtol=1e-10, atol=1e-12)
        assert size.tolist() == [i + 1 for i in range(n)]
        assert oracle.head_edges(cfg, n, **idx) == n * (n + 1) // 2
    # lse against the library's logsumexp
    s = scale * torch.from_numpy(q).double() @ torch.from_numpy(k).double().T
    s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=1).numpy(), rtol=1e-12)


def test_attend_extreme_logits():
    """A logit far above the others takes all the weight; huge negative
    logits do not produce NaN (the max is subtracted first)."""
    d = 4
    q = np.array([[100.0, 0, 0, 0]], np.float32)
    k = np.array([[0, 0, 0, 0], [50, 0, 0, 0], [-50, 0, 0, 0]], np.float32)
    v = np.array([[1, 0, 0, 0], [0, 1, 0, 0], [0, 0, 1, 0]], np.float32)
    q3 = np.zeros((3, d), np.float32)
    q3[2] = q[0]
    o, lse = oracle.attend(q3, k, v, 2, [0, 1, 2], 1.0)
    np.testing.assert_allclose(o, [0, 1, 0, 0], atol=1e-300)
    assert abs(lse - 5000.0) < 1e-9
