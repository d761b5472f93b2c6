"""Shared test helpers: tolerances, oracle marshalling, bitmap packing."""
import math

import numpy as np
import torch

import oracle  # noqa: F401  (test-side helpers only)

# Output tolerance: bf16 inputs, fp32 accumulation, bf16 output, against the
# fp64 oracle (max-abs and mean-abs over the compared rows).
O_MAX_ABS = 1.5e-2
O_MEAN_ABS = 2e-3
# LSE is fp32 on the device; scores come from exact bf16 products summed in fp32.
LSE_ABS = 2e-3


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def head_qkv(q, k, v, b, h, Hq, Hkv):
    """fp32 numpy [n, d] matrices of query head h (and its KV head) of batch b."""
    g = Hq // Hkv
    return f32(q[b, h]), f32(k[b, h // g]), f32(v[b, h // g])


def compare_rows(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """o_gpu/o_ref: [rows, d]; lse_*: [rows].  Asserts the benchmark spec's tolerance."""
    o_gpu = np.asarray(o_gpu, np.float64)
    err = np.abs(o_gpu - o_ref)
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite output"
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= O_MAX_ABS, f"{what}: max abs err {mx:.3e} > {O_MAX_ABS}"
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
