"""Parity at the benchmark's full sizes, through the same layer call bench.py
times (msa_layer_index + msa_layer_attend on one workspace).

At these sizes the oracle cannot evaluate every row, so for a few heads of
each pattern it rebuilds the online index at full length (compared by the
same rule as the small cases) and evaluates eq.(2) on seeded sampled query
rows (always including rows 0, 63, 64 and n-1) over the GPU's own index sets;
the per-head edge count E_h is compared exactly on the GPU's sets."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import compare_rows, f32, head_qkv, oracle_cfg
from test_gpu_index import check_set

pytestmark = pytest.mark.gpu


def _check_layer(msa, name, n=None, heads_per_pattern=2, rows=40, check_edges=True):
    w = synth.make_workload(name, device="cuda", n=n)
    q, k, v, table, sh = w["q"], w["k"], w["v"], w["table"], w["shape"]
    B, Hq, Hkv, n, d = sh["B"], sh["Hq"], sh["Hkv"], sh["n"], sh["d"]
    layer = msa.Layer(table, B, Hq, Hkv, n, d, q.device)
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, n, device=q.device)
    edges = torch.zeros(B * Hq, dtype=torch.int64, device=q.device)
    layer.index(q, k)
    layer.attend(q, k, v, o, lse=lse, edges=edges)
    assert msa.poll_device_status() == 0
    vs, bidx, bcnt = layer.indices()
    vs_heads = [h for h, e in enumerate(table) if e["pattern"] == "vs"]
    bs_heads = [h for h, e in enumerate(table) if e["pattern"] == "block"]
    picked = []
    for pat in ("ashape", "vs", "block"):
        hs = [h for h, e in enumerate(table) if e["pattern"] == pat]
        picked += sorted({hs[0], hs[-1]})[:heads_per_pattern] if hs else []
    sample = synth.sample_rows(n, rows, seed=n + 17)
    for h in picked:
        entry = table[h]
        qn, kn, vn = head_qkv(q, k, v, 0, h, Hq, Hkv)
        cfg = oracle_cfg(entry)
        idx = {}
        if entry["pattern"] == "vs":
            slot = vs_heads.index(h)
            C = vs.vertical[slot, :int(vs.vertical_cnt[slot])].cpu().numpy()
            D = vs.slash[slot, :int(vs.slash_cnt[slot])].cpu().numpy()
            Co, Do, c, r = oracle.vs_index(qn, kn, entry["last_q"], entry["n_vertical"], entry["n_slash"], sh["scale"])
            check_set(C, Co, c, f"{name} vertical h{h}")
            check_set(D, Do, r, f"{name} slash h{h}")
            idx = dict(C=C, D=D)
        elif entry["pattern"] == "block":
            x = bs_heads.index(h)
            J, cnt = bidx[0, x].cpu().numpy(), bcnt[0, x].cpu().numpy()
            Jo, co = oracle.bs_index(qn, kn, 64, entry["topk"])
            assert np.array_equal(cnt, co), f"{name} block counts h{h}"
            qb, kb = oracle.bs_pool(qn, 64), oracle.bs_pool(kn, 64)
            for u in np.random.default_rng(h).choice(len(cnt), size=min(64, len(cnt)), replace=False):
                g = J[u, :cnt[u]]
                assert np.all(np.diff(g) > 0) and g[-1] == u
                sc = qb[u] @ kb[:u].T if u else np.zeros(0)
                check_set([t for t in g if t != u], [t for t in Jo[u, :co[u]] if t != u], sc, f"{name} blocks h{h} u{u}")
            idx = dict(J=J, cnt=cnt)
        ro, rl, _ = oracle.head_rows(cfg, qn, kn, vn, sample, sh["scale"], **idx)
        compare_rows(f32(o[0, h])[sample], f32(lse[0, h])[sample], ro, rl, f"{name} h{h} {entry['pattern']}")
        if check_edges:
            assert int(edges[h]) == oracle.head_edges(cfg, n, **idx), f"{name} edges h{h}"


@pytest.mark.timeout(900)
@pytest.mark.parametrize("name", ["mixed", "vs128k", "bs128k"])
def test_bench_layers_full_size(cuda_lib, name):
    _check_layer(cuda_lib, name)


@pytest.mark.timeout(1500)
def test_million_token_layer(cuda_lib):
    """The mixed table at n = 1,048,576: one head per pattern, sampled rows."""
    _check_layer(cuda_lib, "million", heads_per_pattern=1, rows=12)
