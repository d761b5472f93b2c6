"""Shared test helpers: tolerances, oracle marshalling, bitmap packing, and
the index-set comparison rule.

Index sets (a top-k of fp64 oracle scores against the device's fp32 scores):
- where the oracle's k-th and (k+1)-th scores are separated by more than
  MARGIN (relative), the structure is well separated and the sets must be
  equal;
- otherwise a member may differ only if its oracle score lies within REL
  (relative) of the oracle's k-th score, for both the missing and the extra
  member (fp32 device scores against fp64)."""
import math

import numpy as np
import torch

import oracle  # noqa: F401  (test-side helpers only)

# Output tolerance against the fp64 oracle: bf16 inputs and fp32 accumulation
# within O_MAX_ABS (max-abs) and O_MEAN_ABS (mean-abs over the compared rows).
# The output tensor itself is bf16: rounding a value to bf16 (round to nearest
# even, 8 significant bits) moves it by up to BF16_U of its magnitude, which on
# its own exceeds 1.5e-2 once |o| >= 3.84 (half a bf16 step in [4, 8) is
# 2^-6).  So each element may differ by O_MAX_ABS plus that storage rounding,
# BF16_U * |o_ref|; the mean-abs bound is unchanged.
O_MAX_ABS = 1.5e-2
O_MEAN_ABS = 2e-3
BF16_U = 2.0 ** -8
# LSE is fp32 on the device; scores come from exact bf16 products summed in fp32.
LSE_ABS = 2e-3


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def head_qkv(q, k, v, b, h, Hq, Hkv):
    """fp32 numpy [n, d] matrices of query head h (and its KV head) of batch b."""
    g = Hq // Hkv
    return f32(q[b, h]), f32(k[b, h // g]), f32(v[b, h // g])


def compare_rows(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """o_gpu (bf16 values)/o_ref: [rows, d]; lse_*: [rows].  Asserts the
    output tolerance above: per element |o_gpu - o_ref| <= O_MAX_ABS +
    BF16_U * |o_ref|, and the mean-abs error <= O_MEAN_ABS."""
    o_gpu = np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    err = np.abs(o_gpu - o_ref)
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite output"
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    if err.size:
        excess = err - BF16_U * np.abs(o_ref)
        w = np.unravel_index(int(np.argmax(excess)), err.shape)
        assert excess[w] <= O_MAX_ABS, (f"{what}: abs err {err[w]:.3e} at |o_ref| = {abs(o_ref[w]):.3f} exceeds "
                                        f"{O_MAX_ABS} + {BF16_U:.4g} * |o_ref| (max abs err {mx:.3e})")
    assert mean <= O_MEAN_ABS, f"{what}: mean abs err {mean:.3e} > {O_MEAN_ABS}"
    if lse_gpu is not None:
        lse_gpu = np.asarray(lse_gpu, np.float64)
        inf_ref = np.isneginf(lse_ref)
        assert (np.isneginf(lse_gpu) == inf_ref).all(), f"{what}: empty-set rows differ"
        fin = ~inf_ref
        if fin.any():
            le = float(np.abs(lse_gpu[fin] - lse_ref[fin]).max())
            assert le <= LSE_ABS, f"{what}: lse err {le:.3e}"
    return mx, mean


def pack_bits(idx, n) -> np.ndarray:
    """int32 words with bit j set for j in idx (the library's bitmap layout)."""
    words = np.zeros((n + 31) // 32, dtype=np.uint32)
    for j in np.asarray(idx, dtype=np.int64).reshape(-1):
        words[j >> 5] |= np.uint32(1) << np.uint32(j & 31)
    return words.view(np.int32)


def cover_bits(D, n) -> np.ndarray:
    """The index's dilated slash-coverage map (msa_vs_index.slash_cover): bit z
    set iff D holds an offset in [n-1-z, n+62-z], z < n+63."""
    Dset = np.zeros(n, dtype=bool)
    Dset[np.asarray(D, dtype=np.int64)] = True
    pre = np.concatenate([[0], np.cumsum(Dset)])
    z = np.arange(n + 63)
    lo = np.clip(n - 1 - z, 0, n - 1)
    hi = np.clip(n + 62 - z, -1, n - 1)
    has = (hi >= lo) & ((pre[hi + 1] - pre[lo]) > 0)
    return pack_bits(np.nonzero(has)[0], n + 63)


def unpack_bits(words, n) -> np.ndarray:
    w = np.asarray(words).view(np.uint32)
    bits = ((w[:, None] >> np.arange(32, dtype=np.uint32)[None, :]) & 1).astype(bool).reshape(-1)[:n]
    return np.nonzero(bits)[0]


def oracle_cfg(entry: dict) -> dict:
    pat = {"ashape": oracle.ASHAPE, "vs": oracle.VS, "block": oracle.BLOCK}[entry["pattern"]]
    return dict(pattern=pat, sink=entry.get("sink", 0), window=entry.get("window", 1), block=entry.get("block", 64),
                topk=entry.get("topk", 1))


def scale_of(d):
    return 1.0 / math.sqrt(d)


REL = 1e-4      # a differing member's oracle score must lie this close to the k-th score
MARGIN = 1e-3   # k-th vs (k+1)-th gap above which the sets must be equal


def topk_margin(scores, k: int) -> float:
    """Relative gap between the k-th and (k+1)-th largest oracle scores
    (inf when k takes every candidate or none)."""
    s = np.asarray(scores, dtype=np.float64).reshape(-1)
    if k <= 0 or k >= s.size:
        return float("inf")
    part = -np.partition(-s, (k - 1, k))
    kth, nxt = part[k - 1], part[k]
    if kth == nxt:
        return 0.0
    return float((kth - nxt) / abs(kth)) if kth != 0 else float("inf")


def check_topk_set(got, want, scores, k: int, what: str) -> int:
    """The index-set rule above; returns the number of differing members."""
    got, want = set(int(x) for x in got), set(int(x) for x in want)
    assert len(got) == len(want), f"{what}: {len(got)} vs {len(want)} members"
    if got == want:
        return 0
    margin = topk_margin(scores, k)
    assert margin <= MARGIN, f"{what}: sets differ although the oracle's top-{k} is separated by {margin:.2e}"
    sc = np.asarray(scores, dtype=np.float64)
    kth = min(sc[x] for x in want)
    for x in got ^ want:
        assert abs(sc[x] - kth) <= REL * abs(kth), f"{what}: member {x} score {sc[x]!r} vs k-th {kth!r}"
    return len(got ^ want)


def check_block_index(Jg, Cg, Jo, Co, qb, kb, topk: int, what: str) -> int:
    """Every row of a Block-Sparse index against the oracle's: counts equal,
    each row strictly ascending, ending with its own (diagonal) block, -1
    padded; rows that differ follow the index-set rule on the block scores
    Q̄_u . K̄_v (v < u; the diagonal is forced).  Returns the differing rows."""
    Jg, Cg, Jo, Co = (np.asarray(x) for x in (Jg, Cg, Jo, Co))
    nb = Jo.shape[0]
    assert np.array_equal(Cg, Co), f"{what}: block counts"
    cols = np.arange(Jg.shape[1])[None, :]
    inside = cols < Cg[:, None]
    assert np.all(Jg[~inside] == -1), f"{what}: padding"
    steps = np.diff(Jg, axis=1) > 0
    assert np.all(steps | ~inside[:, 1:]), f"{what}: rows not strictly ascending"
    assert np.array_equal(Jg[np.arange(nb), Cg - 1], np.arange(nb)), f"{what}: diagonal block"
    bad = np.nonzero(~np.all(Jg == Jo, axis=1))[0]
    for u in bad:
        sc = qb[u] @ kb[:u].T
        check_topk_set([v for v in Jg[u, :Cg[u]] if v != u], [v for v in Jo[u, :Co[u]] if v != u], sc,
                       min(topk - 1, int(u)), f"{what} u{u}")
    return int(bad.size)
