#!/usr/bin/env python
"""Sparse-prefill benchmark (one GPU per rank; replicas when run under torchrun).

One step = one msa_prefill_layer call on each layer of the workload: the
mixed-pattern layer at n = 32768 and the two n = 131072 layers
(Vertical-Slash only, Block-Sparse only), seeded synthetic inputs resident in
HBM.  Each layer call is split into its two halves (index build, attention) so
the CUDA events give T_index and T_sparse separately.

Metric: effective TFLOP/s = Σ_h 4 E_h d_h / t over the whole step (E_h =
attended causal edges, counted by the kernel in an untimed pass), plus
ms/layer and index-build GB/s.  The JSON line also carries the attention
kernel's roofline, an end-to-end figure through host buffers, the clocks seen
during the timed region and the fp64 oracle timed on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

WORKLOADS = ("mixed", "vs128k", "bs128k")
METRIC = "sparse-prefill effective TFLOP/s (4·E·d_h) & ms/layer at 128K; index-build GB/s"
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except OSError:
        return FALLBACK_PEAKS, "fallback"


# ----------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "200"], stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


def gpu_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v for v in vis.split(",") if v.strip() != ""]
    if ids and local_rank < len(ids) and ids[local_rank].strip().isdigit():
        return int(ids[local_rank])
    return local_rank


# ----------------------------------------------------------------- workload
def algorithmic_index_bytes(w) -> int:
    """Bytes the online indices must move at least (read Q/K once, write and
    read the score vectors and pooled means once, write the indices)."""
    sh, table = w["shape"], w["table"]
    B, Hq, Hkv, n, d = sh["B"], sh["Hq"], sh["Hkv"], sh["n"], sh["d"]
    g = Hq // Hkv
    vs = [h for h, e in enumerate(table) if e["pattern"] == "vs"]
    bs = [h for h, e in enumerate(table) if e["pattern"] == "block"]
    total = 0
    if vs:
        e = table[vs[0]]
        kv = {h // g for h in vs}
        total += B * len(kv) * n * d * 2                    # K of the groups, once
        total += B * len(vs) * min(e["last_q"], n) * d * 2  # proxy query rows
        total += 4 * B * len(vs) * n * 4                    # c and r written and read
        total += B * len(vs) * (4 * (e["n_vertical"] + e["n_slash"]) + 2 * 4 * ((n + 31) // 32))
    if bs:
        nb = (n + 63) // 64
        kv = {h // g for h in bs}
        topk = table[bs[0]]["topk"]
        total += B * (len(bs) + len(kv)) * n * d * 2        # Q of the heads, K of the groups
        total += 2 * B * (len(bs) + len(kv)) * nb * d * 4   # pooled means written and read
        total += B * len(bs) * nb * (topk + 1) * 4          # J and counts
    return total


def logical_edges(n: int, C, D) -> int:
    """Edge count of eq.(5)'s logical Vertical-Slash sets over all rows,
    Σ_i |{j in C : j <= i} ∪ {i - δ : δ in D, δ <= i}|: each column c is
    attended by the n - c rows i >= c, each offset δ by the n - δ rows i >= δ,
    and a pair (c, δ) with c + δ <= n - 1 names the same (row, key) twice."""
    C = np.unique(np.asarray(C, dtype=np.int64))
    D = np.unique(np.asarray(D, dtype=np.int64))
    C, D = C[(C >= 0) & (C < n)], D[(D >= 0) & (D < n)]
    both = int(np.searchsorted(D, n - 1 - C, side="right").sum())
    return int((n - C).sum() + (n - D).sum() - both)


class LayerRun:
    def __init__(self, name, device, msa, synth, n=None):
        self.name = name
        self.w = synth.make_workload(name, device=device, n=n)
        sh = self.w["shape"]
        self.sh = sh
        self.layer = msa.Layer(self.w["table"], sh["B"], sh["Hq"], sh["Hkv"], sh["n"], sh["d"], device)
        self.o = torch.empty_like(self.w["q"])
        self.lse = torch.empty(sh["B"], sh["Hq"], sh["n"], device=device)
        # untimed counting pass: attended edges E_h and 64-row x 128-key tiles per head
        edges = torch.zeros(sh["B"] * sh["Hq"], dtype=torch.int64, device=device)
        tiles = torch.zeros(sh["B"] * sh["Hq"], dtype=torch.int64, device=device)
        self.layer.index(self.w["q"], self.w["k"])
        self.layer.attend_stats(self.w["q"], self.w["k"], self.w["v"], self.o, lse=self.lse, edges=edges, tiles=tiles)
        torch.cuda.synchronize()
        self.edges = edges.cpu().numpy()
        self.tiles = tiles.cpu().numpy()
        self.flops = float(4.0 * self.edges.sum() * sh["d"])
        # Vertical-Slash heads: physical edges (the tile-expanded sets attended) against eq.(5)'s logical sets
        table = self.w["table"]
        vs_heads = [h for h, e in enumerate(table) if e["pattern"] == "vs"]
        self.vs_edges = None
        if vs_heads:
            vs, _, _ = self.layer.indices()
            logical = 0
            for b in range(sh["B"]):
                for x, h in enumerate(vs_heads):
                    slot = b * len(vs_heads) + x
                    C = vs.vertical[slot, :int(vs.vertical_cnt[slot])].cpu().numpy()
                    D = vs.slash[slot, :int(vs.slash_cnt[slot])].cpu().numpy()
                    logical += logical_edges(sh["n"], C, D)
            phys = int(sum(self.edges[b * sh["Hq"] + h] for b in range(sh["B"]) for h in vs_heads))
            self.vs_edges = {"heads": len(vs_heads) * sh["B"], "physical": phys, "logical": logical,
                             "physical_over_logical": round(phys / max(logical, 1), 4)}
        self.index_bytes = algorithmic_index_bytes(self.w)
        self.bytes_in = sum(t.numel() * t.element_size() for t in (self.w["q"], self.w["k"], self.w["v"]))
        self.bytes_out = self.o.numel() * self.o.element_size()

    def index(self):
        self.layer.index(self.w["q"], self.w["k"])

    def attend(self):
        self.layer.attend(self.w["q"], self.w["k"], self.w["v"], self.o, lse=self.lse)


# ----------------------------------------------------------------- oracle (CPU) sample
def oracle_sample(runs, target_s=20.0, seed=5):
    """Time the fp64 oracle on a bounded sample of the workload.

    For every layer, the first head of each pattern it uses: its online index
    at full length (timed once), then seeded sampled query rows, sized from a
    32-row pilot so that all rows together take about target_s seconds (the
    pilot overestimates the per-row cost, so the rows take somewhat less).  The
    index time is charged to the sample in proportion to the rows sampled
    (R / n of it), so the value is the same effective metric a full layer
    would give.  Returns (TFLOP/s, seconds spent, sampled FLOPs, description).
    """
    import oracle
    import synth
    heads = []
    for r in runs:
        w, sh = r.w, r.sh
        g = sh["Hq"] // sh["Hkv"]
        seen = set()
        for h, e in enumerate(w["table"]):
            if e["pattern"] in seen:
                continue
            seen.add(e["pattern"])
            qn = w["q"][0, h].float().cpu().numpy()
            kn = w["k"][0, h // g].float().cpu().numpy()
            vn = w["v"][0, h // g].float().cpu().numpy()
            t0 = time.perf_counter()
            idx = {}
            if e["pattern"] == "vs":
                C, D, _, _ = oracle.vs_index(qn, kn, e["last_q"], e["n_vertical"], e["n_slash"], sh["scale"])
                idx = dict(C=C, D=D)
                cfg = dict(pattern=oracle.VS, block=64)
            elif e["pattern"] == "block":
                J, cnt = oracle.bs_index(qn, kn, 64, e["topk"])
                idx = dict(J=J, cnt=cnt)
                cfg = dict(pattern=oracle.BLOCK, block=64, topk=e["topk"])
            else:
                cfg = dict(pattern=oracle.ASHAPE, sink=e["sink"], window=e["window"])
            heads.append(dict(cfg=cfg, q=qn, k=kn, v=vn, idx=idx, n=sh["n"], d=sh["d"], scale=sh["scale"],
                              t_index=time.perf_counter() - t0, seed=seed + h))

    def rows_pass(count):
        flops, secs, t_idx, R = 0.0, 0.0, 0.0, 0
        for x in heads:
            rows = synth.sample_rows(x["n"], count, x["seed"] + count)
            t0 = time.perf_counter()
            _, _, size = oracle.head_rows(x["cfg"], x["q"], x["k"], x["v"], rows, x["scale"], **x["idx"])
            secs += time.perf_counter() - t0
            flops += 4.0 * float(size.sum()) * x["d"]
            t_idx += x["t_index"] * len(rows) / x["n"]
            R += len(rows)
        return flops, secs, t_idx, R

    pilot = rows_pass(32)
    count = int(max(32, min(min(x["n"] for x in heads), 32 * target_s / max(pilot[1], 1e-3))))
    flops, secs, t_idx, R = rows_pass(count)
    spent = sum(x["t_index"] for x in heads) + pilot[1] + secs
    desc = (f"per layer ({', '.join(r.name for r in runs)}): the first head of each pattern, its online index "
            f"at full length (time charged by rows sampled / n) and {count} seeded sampled query rows "
            f"({R} rows in all, {secs:.1f} s of rows; fp64, {oracle.num_threads()} threads)")
    return flops / (secs + t_idx) / 1e12, spent, flops, desc


def attention_traffic(names, n_override):
    """DRAM bytes of each layer's attention launches from the committed ncu
    capture (profiles/sparse_attn_kernel_traffic.json), if the kernel sources
    still hash to the captured ones and the workloads are the captured full
    sizes."""
    import hashlib
    here = os.path.dirname(os.path.abspath(__file__))
    try:
        rec = json.load(open(os.path.join(here, "profiles", "sparse_attn_kernel_traffic.json")))
        h = hashlib.sha256()
        for f in rec["sources"]:
            h.update(open(os.path.join(here, f), "rb").read())
    except (OSError, KeyError, ValueError):
        return None, None
    if h.hexdigest() != rec["source_sha256"] or n_override or any(nm not in rec["bytes_per_layer"] for nm in names):
        return None, None
    per = {nm: rec["bytes_per_layer"][nm] for nm in names}
    return int(sum(per.values())), per


# ----------------------------------------------------------------- curves
def _timed(fn, reps, flush):
    """Median CUDA-event time (ms) of fn over reps calls, L2 flushed before each."""
    stream = torch.cuda.current_stream()
    ts = []
    for _ in range(reps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def curves(kind, local, reps=5):
    """The curves the MInference page asks for beside the headline (§5.2: the
    time decomposition eq.(13) and the length where sparse overtakes dense;
    §6.2: sampled rows vs captured mass vs index time), on the seeded layers:

    crossover: for each layer type and n, T_index + T_sparse of the sparse
      layer against dense causal attention (msa_attn_dense) of every head on
      the same inputs; speedup = dense / (index + sparse).
    lastq: the Vertical-Slash and mixed layers at n = 131072 with last_q =
      16 .. 128 sampled proxy rows: index time and attention time.
    proxy: the same layers with each proxy aggregation convention (§3.1,
      §6.2: column sum or maximum, slash sum or mean over legal pairs).
    Every point also gives the captured dense mass per head (the mean over
    rows of e^{lse_sparse - lse_dense}), as its mean and minimum over the heads
    of each pattern."""
    import long_context_prefill_gb300 as msa
    import synth
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    msa.load()
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=device)
    if kind == "crossover":
        points = [(wl, n) for wl in ("vs128k", "bs128k", "mixed")
                  for n in (4096, 8192, 16384, 32768, 65536, 131072)]
    else:
        points = [("vs128k", 131072), ("mixed", 131072)]
    for wl, n in points:
        w = synth.make_workload(wl, device=device, n=n)
        sh = w["shape"]
        q, k, v = w["q"], w["k"], w["v"]
        o = torch.empty_like(q)
        lse_d = torch.empty(sh["B"], sh["Hq"], n, device=device)
        heads = list(range(sh["Hq"]))
        dense = lambda: msa.attn_dense(q, k, v, heads, o=o, lse=lse_d)
        dense()
        t_dense = _timed(dense, reps, flush)
        variants = {"crossover": [{}], "lastq": [{"last_q": x} for x in (16, 32, 64, 128)],
                    "proxy": [{"proxy": x} for x in (0, 1, 2, 3)]}[kind]
        for var in variants:
            table = [dict(e) for e in w["table"]]
            for e in table:
                if e["pattern"] == "vs":
                    e.update(var)
            layer = msa.Layer(table, sh["B"], sh["Hq"], sh["Hkv"], n, sh["d"], device)
            lse_s = torch.empty_like(lse_d)
            edges = torch.zeros(sh["B"] * sh["Hq"], dtype=torch.int64, device=device)
            layer(q, k, v, o=o, lse=lse_s, edges=edges)
            t_idx = _timed(lambda: layer.index(q, k), reps, flush)
            t_att = _timed(lambda: layer.attend(q, k, v, o, lse=lse_s), reps, flush)
            assert msa.poll_device_status() == 0
            E = float(edges.sum().item())
            rec = {"curve": kind, "workload": wl, "n": n, "heads": sh["Hq"], "kv_heads": sh["Hkv"], "d_h": sh["d"],
                   "t_index_ms": round(t_idx, 4), "t_sparse_ms": round(t_att, 4), "dense_ms": round(t_dense, 4),
                   "speedup_vs_dense": round(t_dense / (t_idx + t_att), 3),
                   "density": round(E / (sh["B"] * sh["Hq"] * n * (n + 1) / 2), 4),
                   "effective_tflops": round(4.0 * E * sh["d"] / ((t_idx + t_att) * 1e-3) / 1e12, 1),
                   "l2": "flushed (256 MiB write) before every timed call"}
            rec.update(var)
            mass = msa.captured_mass(lse_s, lse_d).cpu().numpy().reshape(sh["B"], sh["Hq"])
            for pat in ("ashape", "vs", "block"):
                hs = [h for h, e in enumerate(table) if e["pattern"] == pat]
                if hs:
                    rec[f"captured_mass_{pat}"] = {"mean": round(float(mass[:, hs].mean()), 5),
                                                   "min": round(float(mass[:, hs].min()), 5)}
            print(json.dumps(rec), flush=True)
            del layer
        del w, q, k, v, o
        torch.cuda.empty_cache()


# ----------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workloads", default=",".join(WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-dense", action="store_true", help="skip the dense-baseline and cold-L2 measurements")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the per-config lines outside the step (A-shape-only 128K layer, 1M-token layer)")
    ap.add_argument("--n", type=int, default=None,
                    help="override the sequence length (scaled-down runs for profiling; not a headline number)")
    ap.add_argument("--curve", choices=["crossover", "lastq", "proxy"], default=None,
                    help="instead of the step: the sparse-vs-dense crossover over sequence lengths, the sampled "
                         "proxy rows sweep, or the proxy aggregation conventions, each with index time and "
                         "captured mass (one JSON line per point)")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    names = [x for x in args.workloads.split(",") if x]

    if args.impl == "reference":
        return reference_arm(args, world, rank, local, names)
    if args.curve:
        if rank == 0:
            curves(args.curve, local)
        return

    import long_context_prefill_gb300 as msa
    import synth
    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    msa.load()
    runs = [LayerRun(nm, device, msa, synth, n=args.n) for nm in names]
    assert msa.poll_device_status() == 0
    step_flops = sum(r.flops for r in runs)
    stream = torch.cuda.current_stream()

    def step(evs=None):
        for x, r in enumerate(runs):
            if evs is not None:
                evs[x][0].record(stream)
            r.index()
            if evs is not None:
                evs[x][1].record(stream)
            r.attend()
            if evs is not None:
                evs[x][2].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert msa.poll_device_status() == 0

    K = args.steps
    events = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in runs] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0 = msa.kernel_launches()
    with ClockSampler(gpu_index(local)) as clk:
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for s in range(K):
            step(events[s])
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    launches = msa.kernel_launches() - l0
    assert msa.poll_device_status() == 0
    ms_total = max_over_ranks(start.elapsed_time(end), world, device)
    ms_step = ms_total / K
    value = world * step_flops * K / (ms_total * 1e-3) / 1e12

    per_layer = {}
    attn_ms_sum, attn_flops_sum = 0.0, 0.0
    for x, r in enumerate(runs):
        idx_ms = statistics.mean(events[s][x][0].elapsed_time(events[s][x][1]) for s in range(K))
        att_ms = statistics.mean(events[s][x][1].elapsed_time(events[s][x][2]) for s in range(K))
        attn_ms_sum += att_ms
        attn_flops_sum += r.flops
        per_layer[r.name] = {
            "n": r.sh["n"], "heads": r.sh["Hq"], "kv_heads": r.sh["Hkv"], "d_h": r.sh["d"],
            "ms_per_layer": round(idx_ms + att_ms, 4), "t_index_ms": round(idx_ms, 4), "t_sparse_ms": round(att_ms, 4),
            "edges": int(r.edges.sum()), "effective_tflops": round(r.flops / ((idx_ms + att_ms) * 1e-3) / 1e12, 2),
            "attention_tflops": round(r.flops / (att_ms * 1e-3) / 1e12, 2),
            "index_gbs": round(r.index_bytes / (idx_ms * 1e-3) / 1e9, 1) if idx_ms > 0 else None,
            "index_bytes": r.index_bytes,
            "density": round(float(r.edges.sum()) / (r.sh["Hq"] * r.sh["n"] * (r.sh["n"] + 1) / 2), 4),
            "tiles_64x128": int(r.tiles.sum()),
            "tile_fill": round(float(r.edges.sum()) / max(float(r.tiles.sum()) * 64 * 128, 1.0), 4),
        }
        if r.vs_edges:
            per_layer[r.name]["vs_edges"] = r.vs_edges
    if not args.no_dense:
        dense_and_cold(runs, msa, per_layer, stream)
    pk, pk_src = peaks()
    achieved = attn_flops_sum / (attn_ms_sum * 1e-3) / 1e12
    burst = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    clocks = clk.summary()
    # the burst peak unless the clock record shows the power cap throttling the timed region
    capped = bool(clocks) and "sw_power_cap" in clocks.get("reasons", [])
    peak = sustained if capped else burst
    traffic, traffic_per = attention_traffic([r.name for r in runs], args.n)
    roofline = {"bound": "tensor", "kernel": "sparse_attn_kernel", "achieved": round(achieved, 2), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                "traffic_note": "DRAM bytes (read + write) of the attention launches of one step (one per pattern of each layer), from "
                                "the committed ncu capture; null once the kernel source differs from the captured one",
                "traffic_per_layer": traffic_per,
                "peak_source": (f"{pk_src} bf16 " + ("sustained (the clock record shows sw_power_cap)" if capped else
                                                     "burst (no power cap in the clock record of the timed region)")),
                "frac_of_burst": round(achieved / burst, 4), "frac_of_sustained": round(achieved / sustained, 4),
                "flops_per_launch": {r.name: r.flops for r in runs},
                "launch_ms": {r.name: per_layer[r.name]["t_sparse_ms"] for r in runs}}
    idx_bytes = sum(r.index_bytes for r in runs)
    idx_ms = sum(per_layer[r.name]["t_index_ms"] for r in runs)

    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(runs, msa, K, world, device, stream)

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded generators, planted structure)",
        "config": {"workload": "+".join(names) + " prefill layers (B=1, Hq=32, Hkv=8, d_h=128)"
                   + (f", n overridden to {args.n}" if args.n else ""),
                   "layers": per_layer, "l2": "inputs larger than L2 (129 MB) between timed iterations",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "index_gbs_total": round(idx_bytes / (idx_ms * 1e-3) / 1e9, 1),
                   "index_frac_of_hbm": round(idx_bytes / (idx_ms * 1e-3) / 1e9 / float(pk.get("hbm_gbs", 6800.0)), 4)},
        "roofline": roofline, "e2e": e2e, "gpu_launches": int(launches), "clocks": clocks,
    }
    if not args.no_extra and args.n is None:
        line["extra_layers"] = extra_layers(msa, synth, device, stream)
    if rank == 0 and world == 1 and not args.no_cpu:
        v, secs, fl, desc = oracle_sample(runs)
        import oracle
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": desc, "seconds": round(secs, 2)}
    if rank == 0:
        print(json.dumps(line), flush=True)


def extra_layers(msa, synth, device, stream, names=("ashape128k", "million"), reps=3):
    """Per-config figures outside the headline step (their own runs, after it):
    the A-shape pattern alone at n = 131072 and the mixed table at n =
    1,048,576 (the MInference page §5.2 million-token bucket).  Each layer is
    timed over `reps` calls after one warm-up; inputs exceed L2."""
    out = {}
    for nm in names:
        r = LayerRun(nm, device, msa, synth)
        r.index()
        r.attend()
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        idx, att = [], []
        for _ in range(reps):
            a.record(stream)
            r.index()
            b.record(stream)
            r.attend()
            c.record(stream)
            torch.cuda.synchronize()
            idx.append(a.elapsed_time(b))
            att.append(b.elapsed_time(c))
        assert msa.poll_device_status() == 0
        ti, ta = statistics.median(idx), statistics.median(att)
        sh = r.sh
        rec = {"n": sh["n"], "heads": sh["Hq"], "kv_heads": sh["Hkv"], "d_h": sh["d"],
               "patterns": {p: sum(1 for e in r.w["table"] if e["pattern"] == p) for p in ("ashape", "vs", "block")},
               "ms_per_layer": round(ti + ta, 4), "t_index_ms": round(ti, 4), "t_sparse_ms": round(ta, 4),
               "edges": int(r.edges.sum()), "effective_tflops": round(r.flops / ((ti + ta) * 1e-3) / 1e12, 2),
               "attention_tflops": round(r.flops / (ta * 1e-3) / 1e12, 2),
               "index_gbs": round(r.index_bytes / (ti * 1e-3) / 1e9, 1) if ti > 0 and r.index_bytes else None,
               "density": round(float(r.edges.sum()) / (sh["Hq"] * sh["n"] * (sh["n"] + 1) / 2), 5),
               "tiles_64x128": int(r.tiles.sum()),
               "tile_fill": round(float(r.edges.sum()) / max(float(r.tiles.sum()) * 64 * 128, 1.0), 4)}
        if r.vs_edges:
            rec["vs_edges"] = r.vs_edges
        out[nm] = rec
        del r
        torch.cuda.empty_cache()
    out["varlen_mixed64"] = varlen_batch(msa, synth, device, stream, reps=reps)
    return out


def varlen_batch(msa, synth, device, stream, n_seqs=64, lo=1024, hi=16384, seed=77, reps=3):
    """A varlen batch (cost-model page §2.2): n_seqs sequences with seeded
    log-uniform lengths in [lo, hi], each the mixed-pattern generator and
    table, packed back to back; one msa_prefill_layer_varlen call (one index
    pass and one attention launch per pattern over all sequences), timed after a warm-up."""
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in np.exp(rng.uniform(np.log(lo), np.log(hi), size=n_seqs))]
    ws = [synth.make_workload("mixed", device=device, n=n, seed=3000 + i) for i, n in enumerate(lens)]
    sh = ws[0]["shape"]
    table = ws[0]["table"]
    q = msa.pack_varlen([w["q"][0] for w in ws])
    k = msa.pack_varlen([w["k"][0] for w in ws])
    v = msa.pack_varlen([w["v"][0] for w in ws])
    del ws
    cu = [0] + [int(x) for x in np.cumsum(lens)]
    layer = msa.VarlenLayer(table, cu, sh["Hq"], sh["Hkv"], sh["d"], device)
    edges = torch.zeros(n_seqs * sh["Hq"], dtype=torch.int64, device=device)
    o = layer(q, k, v, edges=edges)
    torch.cuda.synchronize()
    flops = 4.0 * float(edges.sum().item()) * sh["d"]
    l0 = msa.kernel_launches()
    layer(q, k, v, o=o)
    launches = msa.kernel_launches() - l0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts = []
    for _ in range(reps):
        a.record(stream)
        layer(q, k, v, o=o)
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    assert msa.poll_device_status() == 0
    ms = statistics.median(ts)
    dense = sum(n * (n + 1) / 2 for n in lens) * sh["Hq"]
    rec = {"sequences": n_seqs, "tokens": cu[-1], "lengths": f"log-uniform in [{lo}, {hi}] (seed {seed})",
           "heads": sh["Hq"], "kv_heads": sh["Hkv"], "d_h": sh["d"], "table": "mixed (A-shape : VS : BS = 1 : 6 : 1)",
           "ms_per_batch": round(ms, 4), "effective_tflops": round(flops / (ms * 1e-3) / 1e12, 2),
           "density": round(float(edges.sum().item()) / dense, 4), "launches_per_batch": int(launches)}
    del q, k, v, o, layer
    torch.cuda.empty_cache()
    return rec


def dense_and_cold(runs, msa, per_layer, stream, reps=2):
    """Outside the timed region: (1) dense causal attention of every head on
    the same engine and inputs, the baseline the sparse layer is measured
    against (speedup_vs_dense = dense attention time / sparse layer time);
    (2) the sparse layer once right after a 512 MiB write has flushed L2."""
    scrub = torch.empty(512 << 20, dtype=torch.uint8, device=runs[0].o.device)
    for r in runs:
        sh = r.sh
        heads = list(range(sh["Hq"]))
        q, k, v = r.w["q"], r.w["k"], r.w["v"]
        msa.attn_dense(q, k, v, heads, o=r.o, stream=stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            msa.attn_dense(q, k, v, heads, o=r.o, stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        dense_ms = a.elapsed_time(b) / reps
        dense_flops = 4.0 * sh["d"] * sh["B"] * sh["Hq"] * sh["n"] * (sh["n"] + 1) / 2
        cold = []
        for _ in range(reps):
            scrub.fill_(1)
            a.record(stream)
            r.index()
            r.attend()
            b.record(stream)
            torch.cuda.synchronize()
            cold.append(a.elapsed_time(b))
        lay = per_layer[r.name]
        lay["dense_ms"] = round(dense_ms, 4)
        lay["dense_tflops"] = round(dense_flops / (dense_ms * 1e-3) / 1e12, 2)
        lay["speedup_vs_dense"] = round(dense_ms / lay["ms_per_layer"], 3)
        lay["ms_per_layer_cold_l2"] = round(statistics.median(cold), 4)
    assert msa.poll_device_status() == 0
    del scrub


def end_to_end(runs, msa, K, world, device, stream):
    """The same metric through host buffers: every step copies each layer's
    Q/K/V from pinned host memory, runs msa_prefill_layer, and reads its O
    back.  Each layer has two device buffer sets used by alternate steps, so
    the uploads of the next step and the downloads of this one run on two copy
    streams while the current step computes (a set is rewritten only after the
    step two back has finished computing from it and its output has reached
    the host)."""
    host, dev = [], []
    for r in runs:
        hq = r.w["q"].cpu().pin_memory()
        hk = r.w["k"].cpu().pin_memory()
        hv = r.w["v"].cpu().pin_memory()
        ho = torch.empty(r.o.shape, dtype=r.o.dtype).pin_memory()
        host.append((hq, hk, hv, ho))
        dev.append([(r.w["q"], r.w["k"], r.w["v"], r.o),
                    (torch.empty_like(r.w["q"]), torch.empty_like(r.w["k"]), torch.empty_like(r.w["v"]),
                     torch.empty_like(r.o))])
    up_stream, down_stream = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    uploaded = [[ev(), ev()] for _ in runs]  # [layer][set]: inputs are on the device
    computed = [[ev(), ev()] for _ in runs]  # the layer's compute from this set has finished
    fetched = [[ev(), ev()] for _ in runs]   # the layer's output in this set has reached the host
    count = [0]

    def upload(x):
        for L, (hq, hk, hv, _) in enumerate(host):
            q, k, v, _ = dev[L][x % 2]
            with torch.cuda.stream(up_stream):
                if x >= 2:
                    up_stream.wait_event(computed[L][x % 2])
                q.copy_(hq, non_blocking=True)
                k.copy_(hk, non_blocking=True)
                v.copy_(hv, non_blocking=True)
                uploaded[L][x % 2].record(up_stream)

    def compute(x):
        for L, r in enumerate(runs):
            q, k, v, o = dev[L][x % 2]
            stream.wait_event(uploaded[L][x % 2])
            if x >= 2:
                stream.wait_event(fetched[L][x % 2])
            r.layer(q, k, v, o=o, stream=stream)
            computed[L][x % 2].record(stream)
            with torch.cuda.stream(down_stream):
                down_stream.wait_event(computed[L][x % 2])
                host[L][3].copy_(o, non_blocking=True)
                fetched[L][x % 2].record(down_stream)

    def step():
        x = count[0]
        if x == 0:
            upload(0)
        upload(x + 1)  # the next step's inputs go up while this one computes
        compute(x)
        count[0] += 1

    step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    a.record(stream)
    for _ in range(K):
        step()
    last = (count[0] - 1) % 2
    for L in range(len(runs)):  # K uploads (steps 2 .. K+1), K computes and K downloads in the timed region
        stream.wait_event(fetched[L][last])
        stream.wait_event(uploaded[L][count[0] % 2])
    b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(a.elapsed_time(b), world, device)
    flops = sum(r.flops for r in runs)
    del dev
    return {"value": round(world * flops * K / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(sum(r.bytes_in for r in runs)),
            "d2h_bytes_per_step": int(sum(r.bytes_out for r in runs)), "ms_per_step": round(ms / K, 4),
            "overlap": "two device buffer sets per layer: the next step's uploads and this step's downloads "
                       "run on two copy streams during this step's compute"}


def reference_arm(args, world, rank, local, names):
    """The oracle (fp64, host cores) on a bounded sample of the same workload."""
    if rank != 0:
        return
    import oracle
    import synth

    class HostRun:
        def __init__(self, name):
            self.name = name
            self.w = synth.make_workload(name, device="cuda" if torch.cuda.is_available() else "cpu")
            self.sh = self.w["shape"]

    runs = [HostRun(nm) for nm in names]
    per_step = 4.0  # seconds of sampled rows per step: warm-up and timed steps end within a few minutes
    for _ in range(max(args.warmup, 3)):
        oracle_sample(runs, target_s=per_step)
    vals, secs_all = [], 0.0
    desc = ""
    for _ in range(args.steps):
        v, secs, fl, desc = oracle_sample(runs, target_s=per_step)
        vals.append(v)
        secs_all += secs
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(1e3 * secs_all / args.steps, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generators, planted structure)",
            "config": {"workload": "+".join(names) + " prefill layers (B=1, Hq=32, Hkv=8, d_h=128)",
                       "sample": desc},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
