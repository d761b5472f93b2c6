"""The seeded input generators: the same seed gives the same tensors, and the
structure they plant is what the oracle's proxy finds (the planted slash
offsets of the tiny workload rank among its top slashes)."""
import numpy as np
import torch

import oracle
import synth


def test_generators_are_deterministic():
    a = synth.make_workload("tiny", device="cpu")
    b = synth.make_workload("tiny", device="cpu")
    c = synth.make_workload("tiny", device="cpu", seed=synth.SEEDS["tiny"] + 1)
    for name in ("q", "k", "v"):
        assert torch.equal(a[name], b[name])
        assert not torch.equal(a[name], c[name])
    assert a["table"] == b["table"]
    q1, k1, v1 = synth.random_qkv(1, 2, 1, 100, 64, seed=3)
    q2, k2, v2 = synth.random_qkv(1, 2, 1, 100, 64, seed=3)
    assert torch.equal(q1, q2) and torch.equal(k1, k2) and torch.equal(v1, v2)


def test_planted_slashes_are_found_by_the_proxy():
    w = synth.make_workload("tiny", device="cpu")
    h = [x for x, e in enumerate(w["table"]) if e["pattern"] == "vs"][0]
    e = w["table"][h]
    _, D, _, _ = oracle.vs_index(w["q"][0, h].float().numpy(), w["k"][0, 0].float().numpy(), e["last_q"],
                                 e["n_vertical"], e["n_slash"], w["shape"]["scale"])
    assert {0, 37, 300} <= set(np.asarray(D).tolist())
