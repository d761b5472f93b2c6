"""Seeded synthetic inputs shaped like long-context prefill (one attention layer).

This module only draws random tensors and plants structure in them; it holds
none of the method's arithmetic.  The CUDA path and the oracle both take what
it produces (the oracle gets the exact bf16 values copied to the host).

Workloads (B = 1 throughout; Q [B,Hq,n,d], K/V [B,Hkv,n,d], bf16):

* ``tiny``    Hq=2, Hkv=1, n=2048, d=64.  Q, K, V ~ N(0,1); 16 random key
  columns get K += 3u and every query Q += u (verticals); q_i += 2 rot(u_s, i)
  and k_j += 2 Σ_{δ in {0,37,300}} rot(u_s, j+δ) (slashes).  Head 0 is A-shape
  (sink 64, window 512), head 1 Vertical-Slash (last_q 64, v 64, s 128).
* ``mixed``   Hq=32, Hkv=8, n=32768, d=128.  Per KV head: U{8..64} vertical
  columns with strength U[2,4]; U{2..8} slash offsets, log-uniform in [1,n),
  plus offset 0, strength U[1.5,3].  A seeded permutation assigns 4 heads
  A-shape (128, 1024), 24 Vertical-Slash (64, 1000, 6096), 4 Block-Sparse
  (block 64, top-k 64).
* ``vs128k``  Hq=32, Hkv=8, n=131072, d=128; 50 verticals per KV head
  (strength 3), 16 slashes per KV head with δ = floor(exp(U[0, ln n))) - 1
  (strength 2); every head Vertical-Slash (64, 1000, 6096).
* ``bs128k``  Hq=32, Hkv=8, n=131072, d=128; each (KV head, 64-token block)
  gets a mean μ ~ N(0, 1.5² I) added to its K rows and to the Q rows of every
  query head of the group, plus N(0,1) noise; V ~ N(0,1); every head
  Block-Sparse (block 64, top-k 100).
* ``million`` the ``mixed`` generator and table at n = 1,048,576.
* ``ashape128k`` the ``vs128k`` generator at n = 131072 with every head
  A-shape (sink 128, window 1024): the A-shape pattern measured on its own.

rot(u, p) rotates dimension pairs (2k, 2k+1) of u by the angle
p * 10000^(-2k/d) (a RoPE-style rotation), so rot(u,p).rot(u,p') depends only
on p - p' and peaks at p = p'.
"""
from __future__ import annotations

import math

import numpy as np
import torch

WORKLOADS = {
    "tiny": dict(B=1, Hq=2, Hkv=1, n=2048, d=64),
    "mixed": dict(B=1, Hq=32, Hkv=8, n=32768, d=128),
    "vs128k": dict(B=1, Hq=32, Hkv=8, n=131072, d=128),
    "bs128k": dict(B=1, Hq=32, Hkv=8, n=131072, d=128),
    "million": dict(B=1, Hq=32, Hkv=8, n=1048576, d=128),
    "ashape128k": dict(B=1, Hq=32, Hkv=8, n=131072, d=128),
}
SEEDS = {"tiny": 1001, "mixed": 1002, "vs128k": 1003, "bs128k": 1004, "million": 1005, "ashape128k": 1006}


def ashape(sink, window):
    return dict(pattern="ashape", sink=int(sink), window=int(window))


def vslash(last_q, v, s, block=64, proxy=0):
    return dict(pattern="vs", last_q=int(last_q), n_vertical=int(v), n_slash=int(s), block=int(block),
                proxy=int(proxy))


def blocksparse(topk, block=64):
    return dict(pattern="block", block=int(block), topk=int(topk))


def table_for(name: str, Hq: int, seed: int):
    """Per-query-head pattern table of a workload."""
    if name == "tiny":
        return [ashape(64, 512), vslash(64, 64, 128)]
    if name in ("mixed", "million"):
        g = np.random.default_rng(seed + 7)
        kinds = ["ashape"] * (Hq // 8) + ["vs"] * (Hq - 2 * (Hq // 8)) + ["block"] * (Hq // 8)
        kinds = [kinds[i] for i in g.permutation(Hq)]
        out = []
        for k in kinds:
            out.append(ashape(128, 1024) if k == "ashape" else vslash(64, 1000, 6096) if k == "vs" else blocksparse(64))
        return out
    if name == "vs128k":
        return [vslash(64, 1000, 6096) for _ in range(Hq)]
    if name == "bs128k":
        return [blocksparse(100) for _ in range(Hq)]
    if name == "ashape128k":
        return [ashape(128, 1024) for _ in range(Hq)]
    raise KeyError(name)


def _rot(u: torch.Tensor, pos: torch.Tensor) -> torch.Tensor:
    """rot(u, p) for a batch of positions: u [d], pos [m] -> [m, d] (fp32)."""
    d = u.numel()
    k = torch.arange(d // 2, device=u.device, dtype=torch.float64)
    theta = torch.pow(torch.tensor(10000.0, device=u.device, dtype=torch.float64), -2.0 * k / d)
    ang = (pos.to(torch.float64)[:, None] * theta[None, :])
    c, s = torch.cos(ang).float(), torch.sin(ang).float()
    ue, uo = u[0::2].float(), u[1::2].float()
    out = torch.empty(pos.numel(), d, device=u.device, dtype=torch.float32)
    out[:, 0::2] = ue * c - uo * s
    out[:, 1::2] = ue * s + uo * c
    return out


def _plant_vs(q, k, kvh, g, gen, n, d, cols, vstrength, offsets, sstrength, chunk=1 << 16):
    """Plant verticals and slashes for one KV head (in place, fp32 work buffers).

    q: [g, n, d] fp32 query heads of the group; k: [n, d] fp32.
    """
    dev = k.device
    u_v = torch.randn(d, generator=gen, device=dev)
    u_s = torch.randn(d, generator=gen, device=dev)
    if len(cols):
        k[torch.as_tensor(cols, device=dev)] += vstrength * u_v
        q += u_v
    for s0 in range(0, n, chunk):
        pos = torch.arange(s0, min(n, s0 + chunk), device=dev)
        q[:, s0:s0 + pos.numel()] += sstrength * _rot(u_s, pos)
        acc = torch.zeros(pos.numel(), d, device=dev)
        for dl in offsets:
            acc += _rot(u_s, pos + int(dl))
        k[s0:s0 + pos.numel()] += sstrength * acc


def make_workload(name: str, device="cpu", n: int | None = None, seed: int | None = None, Hq: int | None = None,
                  Hkv: int | None = None, d: int | None = None):
    """Seeded inputs of a workload; n / Hq / Hkv / d override its sizes (for
    scaled-down parity cases).  Returns dict(q, k, v, table, shape, name)."""
    base = dict(WORKLOADS[name])
    if n is not None:
        base["n"] = int(n)
    if Hq is not None:
        base["Hq"] = int(Hq)
    if Hkv is not None:
        base["Hkv"] = int(Hkv)
    if d is not None:
        base["d"] = int(d)
    B, Hq_, Hkv_, n_, d_ = base["B"], base["Hq"], base["Hkv"], base["n"], base["d"]
    seed = SEEDS[name] if seed is None else int(seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    rng = np.random.default_rng(seed)
    g = Hq_ // Hkv_
    q = torch.empty(B, Hq_, n_, d_, dtype=torch.bfloat16, device=device)
    k = torch.empty(B, Hkv_, n_, d_, dtype=torch.bfloat16, device=device)
    v = torch.empty(B, Hkv_, n_, d_, dtype=torch.bfloat16, device=device)
    for b in range(B):
        for kvh in range(Hkv_):
            qf = torch.randn(g, n_, d_, generator=gen, device=device)
            kf = torch.randn(n_, d_, generator=gen, device=device)
            vf = torch.randn(n_, d_, generator=gen, device=device)
            if name == "tiny":
                cols = rng.choice(n_, size=min(16, n_), replace=False)
                _plant_vs(qf, kf, kvh, g, gen, n_, d_, cols, 3.0, [0, 37, 300], 2.0)
            elif name in ("mixed", "million"):
                nv = int(rng.integers(8, 65))
                cols = rng.choice(n_, size=min(nv, n_), replace=False)
                vs_ = float(rng.uniform(2.0, 4.0))
                ns = int(rng.integers(2, 9))
                offs = [0] + [int(math.exp(rng.uniform(0.0, math.log(n_)))) for _ in range(ns)]
                offs = [min(o, n_ - 1) for o in offs]
                ss = float(rng.uniform(1.5, 3.0))
                _plant_vs(qf, kf, kvh, g, gen, n_, d_, cols, vs_, offs, ss)
            elif name in ("vs128k", "ashape128k"):
                cols = rng.choice(n_, size=min(50, n_), replace=False)
                offs = [int(math.exp(rng.uniform(0.0, math.log(n_)))) - 1 for _ in range(16)]
                _plant_vs(qf, kf, kvh, g, gen, n_, d_, cols, 3.0, offs, 2.0)
            elif name == "bs128k":
                nb = (n_ + 63) // 64
                mu = 1.5 * torch.randn(nb, d_, generator=gen, device=device)
                mu_rows = mu.repeat_interleave(64, dim=0)[:n_]
                kf += mu_rows
                qf += mu_rows[None]
            q[b, kvh * g:(kvh + 1) * g] = qf.to(torch.bfloat16)
            k[b, kvh] = kf.to(torch.bfloat16)
            v[b, kvh] = vf.to(torch.bfloat16)
            del qf, kf, vf
    table = table_for(name, Hq_, seed)
    shape = dict(B=B, Hq=Hq_, Hkv=Hkv_, n=n_, d=d_, scale=1.0 / math.sqrt(d_))
    return dict(q=q, k=k, v=v, table=table, shape=shape, name=name)


def random_qkv(B, Hq, Hkv, n, d, seed, device="cpu", scale_q=1.0):
    """Plain N(0,1) bf16 tensors (Q optionally scaled) for edge-case tests."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    q = (scale_q * torch.randn(B, Hq, n, d, generator=gen, device=device)).to(torch.bfloat16)
    k = torch.randn(B, Hkv, n, d, generator=gen, device=device).to(torch.bfloat16)
    v = torch.randn(B, Hkv, n, d, generator=gen, device=device).to(torch.bfloat16)
    return q, k, v


def sample_rows(n: int, count: int, seed: int, block: int = 64) -> np.ndarray:
    """Seeded sample of query rows, always including 0, block-1, block, n-1."""
    rng = np.random.default_rng(seed)
    must = [r for r in (0, block - 1, block, n - 1) if 0 <= r < n]
    rest = rng.choice(n, size=min(n, count), replace=False)
    return np.unique(np.concatenate([np.asarray(must, dtype=np.int64), rest.astype(np.int64)]))
