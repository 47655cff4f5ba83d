"""The seeded input recipe: shapes, determinism and the advantage construction."""
import math

import torch

from long_context_grpo_gb300 import workloads as wl


def test_tiny_shapes_and_determinism():
    w = wl.WORKLOADS["tiny"]
    assert wl.response_lengths(w) == [32, 48, 64, 17]
    k1, v1 = wl.prefix_kv(w, seed=0)
    k2, v2 = wl.prefix_kv(w, seed=0)
    assert k1.shape == (256, 2, 64) and k1.dtype == torch.bfloat16
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert not torch.equal(k1, v1)
    q, k, v, do = wl.response_attention(w, 2, 64)
    assert q.shape == (64, 2, 64) and k.shape == (64, 2, 64) and do.shape == (64, 2, 64)
    logits, ids, noise = wl.response_loss_inputs(w, 2, 64)
    assert logits.shape == (64, 1024) and ids.dtype == torch.int32
    assert int(ids.min()) >= 0 and int(ids.max()) < 1024
    # distributions: N(0,1)/sqrt(D) for q/k/v, std 2 logits
    assert abs(float(k1.float().std()) - 1 / 8) < 0.01
    assert abs(float(logits.float().std()) - 2.0) < 0.05


def test_response_lengths_in_range():
    for name in ("p32k", "p262k", "p1m", "p2m"):
        w = wl.WORKLOADS[name]
        R = wl.response_lengths(w, seed=0)
        assert len(R) == w.G
        assert all(w.R_range[0] <= r <= w.R_range[1] for r in R)


def test_group_advantage_recipe():
    A = wl.group_advantages([1.0, 0.0, 1.0, 0.0])
    assert all(abs(abs(a) - 1.0) < 1e-5 for a in A)
    assert abs(sum(A)) < 1e-12
    assert wl.group_advantages([1.0, 1.0, 1.0]) == [0.0, 0.0, 0.0]
    r = [1.0, 0.0, 0.0, 0.0, 1.0]
    m = sum(r) / 5
    sd = math.sqrt(sum((x - m) ** 2 for x in r) / 5)
    assert wl.group_advantages(r)[0] == (1.0 - m) / (sd + 1e-6)
