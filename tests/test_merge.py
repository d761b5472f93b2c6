"""Merging attention results over disjoint key sets (msa_merge_attention,
MInference page §3.2, eq.(7)-(8)).

CPU: the oracle's merge is pinned to the oracle's attention itself (the merge
of two disjoint parts equals the attention over their union, for any split),
including empty parts; the library rejects bad arguments on the host.  GPU: the
kernel against the oracle's merge, and a Vertical-Slash head computed as two
disjoint vertical sets merged, against the oracle's attention over the union."""
import ctypes

import numpy as np
import pytest
import torch

import long_context_prefill_gb300 as msa
import oracle
import synth
from helpers import compare_rows, cover_bits, f32, head_qkv, pack_bits, scale_of


def _parts(rng, n, d, i, frac):
    q = rng.standard_normal((n, d))
    k = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    keys = np.arange(i + 1)
    pick = rng.random(i + 1) < frac
    return q, k, v, keys[pick], keys[~pick]


@pytest.mark.parametrize("seed,frac", [(1, 0.5), (2, 0.1), (3, 0.9)])
def test_oracle_merge_equals_attention_over_union(seed, frac):
    rng = np.random.default_rng(seed)
    n, d, scale = 200, 16, 0.25
    for i in (0, 37, 199):
        q, k, v, A, B = _parts(rng, n, d, i, frac)
        ou, lu = oracle.attend(q, k, v, i, np.arange(i + 1), scale)
        oa, la = oracle.attend(q, k, v, i, A, scale) if len(A) else (np.zeros(d), -np.inf)
        ob, lb = oracle.attend(q, k, v, i, B, scale) if len(B) else (np.zeros(d), -np.inf)
        om, lm = oracle.merge(oa[None], np.array([la]), ob[None], np.array([lb]))
        np.testing.assert_allclose(om[0], ou, rtol=1e-12, atol=1e-12)
        assert abs(lm[0] - lu) < 1e-12


def test_oracle_merge_empty_parts():
    o = np.arange(6.0).reshape(2, 3)
    z = np.zeros((2, 3))
    ninf = np.full(2, -np.inf)
    om, lm = oracle.merge(o, np.array([0.5, -2.0]), z, ninf)
    np.testing.assert_array_equal(om, o)
    np.testing.assert_array_equal(lm, [0.5, -2.0])
    om, lm = oracle.merge(z, ninf, z, ninf)
    assert np.all(om == 0) and np.all(np.isneginf(lm))


@pytest.fixture(scope="module")
def lib():
    from long_context_prefill_gb300 import build
    build.build()
    return msa.load()


def test_merge_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    a, b = P(0x10000), P(0x20000)
    la, lb = P(0x30000), P(0x40000)
    assert lib.msa_merge_attention(-1, 128, a, la, b, lb, a, None, None) == msa.MSA_ERR_INVALID_ARG
    assert lib.msa_merge_attention(4, 96, a, la, b, lb, a, None, None) == msa.MSA_ERR_UNSUPPORTED
    assert lib.msa_merge_attention(4, 128, P(0x10008), la, b, lb, a, None, None) == msa.MSA_ERR_INVALID_ARG
    assert lib.msa_merge_attention(4, 128, a, la, b, lb, a, la, None) == msa.MSA_ERR_INVALID_ARG  # lse aliases lse_a
    assert lib.msa_merge_attention(4, 128, None, la, b, lb, a, None, None) == msa.MSA_ERR_INVALID_ARG


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
def test_merge_kernel_against_oracle(cuda_lib, d):
    g = torch.Generator(device="cuda").manual_seed(40 + d)
    rows = 3000
    oa = torch.randn(rows, d, generator=g, device="cuda").to(torch.bfloat16)
    ob = torch.randn(rows, d, generator=g, device="cuda").to(torch.bfloat16)
    la = 3 * torch.randn(rows, generator=g, device="cuda")
    lb = 3 * torch.randn(rows, generator=g, device="cuda")
    la[::7] = -float("inf")   # empty first part
    lb[::11] = -float("inf")  # empty second part (and both on rows divisible by 77)
    o, lse = cuda_lib.merge_attention(oa, la, ob, lb)
    assert cuda_lib.poll_device_status() == 0
    ro, rl = oracle.merge(f32(oa), f32(la), f32(ob), f32(lb))
    compare_rows(f32(o), f32(lse), ro, rl, f"merge d={d}")


@pytest.mark.gpu
def test_vertical_sets_computed_apart_and_merged(cuda_lib):
    """A Vertical-Slash head whose verticals are split into two disjoint sets,
    each attended by its own msa_attn_vs call, then merged: equals the oracle's
    attention over the union (the split-kernel form of the pattern)."""
    n, d, Hq, Hkv = 1500, 128, 2, 1
    rng = np.random.default_rng(21)
    q, k, v = synth.random_qkv(1, Hq, Hkv, n, d, 31, device="cuda")
    C = [np.sort(rng.choice(n, 120, replace=False)) for _ in range(Hq)]
    split = [rng.random(len(c)) < 0.5 for c in C]
    parts = []
    for take in (True, False):
        Cs = [C[h][split[h] == take] for h in range(Hq)]
        index = cuda_lib.VSIndex(Hq, n, max(max(len(c) for c in Cs), 1), 1, "cuda")
        for h in range(Hq):
            index.vertical_bits[h] = torch.from_numpy(pack_bits(Cs[h], n)).cuda()
            index.slash_bits[h] = torch.from_numpy(pack_bits(np.array([], np.int64), n)).cuda()
            index.slash_cover[h] = torch.from_numpy(cover_bits(np.array([], np.int64), n)).cuda()
        o = torch.zeros_like(q)
        lse = torch.empty(1, Hq, n, device="cuda")
        cuda_lib.attn_vs(q, k, v, list(range(Hq)), index, o=o, lse=lse)
        parts.append((o, lse))
    o, lse = cuda_lib.merge_attention(parts[0][0], parts[0][1], parts[1][0], parts[1][1])
    assert cuda_lib.poll_device_status() == 0
    for h in range(Hq):
        qn, kn, vn = head_qkv(q, k, v, 0, h, Hq, Hkv)
        ro, rl, _ = oracle.head_rows(dict(pattern=oracle.VS, block=64), qn, kn, vn, np.arange(n), scale_of(d), C=C[h],
                                     D=np.array([], np.int64))
        compare_rows(f32(o[0, h]), f32(lse[0, h]), ro, rl, f"merged verticals h{h}")


# ----------------------------------------------------------------- captured mass
def test_oracle_captured_mass_pins():
    rng = np.random.default_rng(5)
    n, d = 120, 8
    # fp32-representable inputs: oracle.attend takes fp32 tensors, so both paths see the same values
    q, k = (rng.standard_normal((n, d)).astype(np.float32).astype(np.float64) for _ in range(2))
    rows = np.arange(n)
    full = [np.arange(i + 1) for i in rows]
    assert abs(oracle.captured_mass(q, k, rows, full, 0.3) - 1.0) < 1e-12
    assert oracle.captured_mass(q, k, rows, [np.array([], np.int64)] * n, 0.3) == 0.0
    # a set and its complement share the mass; the share is e^(lse_set - lse_dense)
    sets = [np.flatnonzero(rng.random(i + 1) < 0.4) for i in rows]
    comp = [np.setdiff1d(np.arange(i + 1), s) for i, s in zip(rows, sets)]
    a = oracle.captured_mass(q, k, rows, sets, 0.3)
    b = oracle.captured_mass(q, k, rows, comp, 0.3)
    assert abs(a + b - 1.0) < 1e-12
    v = rng.standard_normal((n, d)).astype(np.float32)
    shares = []
    for i, s in zip(rows, sets):
        if len(s) == 0:
            shares.append(0.0)
            continue
        _, ls = oracle.attend(q, k, v, i, s, 0.3)
        _, ld = oracle.attend(q, k, v, i, np.arange(i + 1), 0.3)
        shares.append(np.exp(ls - ld))
    assert abs(np.mean(shares) - a) < 1e-12


@pytest.mark.gpu
def test_captured_mass_of_ashape_heads(cuda_lib):
    n, d, Hq, Hkv = 2048, 128, 4, 2
    q, k, v = synth.random_qkv(1, Hq, Hkv, n, d, 61, device="cuda", scale_q=2.0)
    cfgs = [(4, 64), (0, 256), (64, 512), (0, n)]
    lse_s = torch.empty(1, Hq, n, device="cuda")
    for h, (g, w) in enumerate(cfgs):
        cuda_lib.attn_ashape(q, k, v, [h], g, w, lse=lse_s)
    lse_d = torch.empty(1, Hq, n, device="cuda")
    cuda_lib.attn_dense(q, k, v, list(range(Hq)), lse=lse_d)
    mass = cuda_lib.captured_mass(lse_s, lse_d)
    assert cuda_lib.poll_device_status() == 0
    rows = np.arange(n)
    for h, (g, w) in enumerate(cfgs):
        qn, kn, _ = head_qkv(q, k, v, 0, h, Hq, Hkv)
        sets = [oracle.ashape_set(i, g, w) for i in rows]
        ref = oracle.captured_mass(qn, kn, rows, sets, scale_of(d))
        assert abs(float(mass[h]) - ref) < 2e-3, (h, float(mass[h]), ref)
    assert abs(float(mass[3]) - 1.0) < 1e-4
