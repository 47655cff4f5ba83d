"""Pins for the float64 GRPO-loss oracle against values fixed outside the oracle."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import grpo

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "clip_cases.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_clip_cases_hand_worked():
    g = _golden()
    eps = g["eps"]
    for c in g["cases"]:
        surr, clipped, d = grpo.surrogate(np.array([c["rho"]]), c["A"], eps)
        assert surr[0] == pytest.approx(c["surr"], abs=1e-15), c
        assert bool(clipped[0]) == c["clipped"], c
        assert d[0] == pytest.approx(c["dsurr_drho"], abs=1e-15), c


def test_worked_loss_example():
    w = _golden()["worked_loss"]
    logits = np.array(w["logits"])
    ids = np.array(w["ids"])
    logp = math.log(0.5)
    old = np.array([logp - math.log(w["rho"][0]), logp - math.log(w["rho"][1])])
    out = grpo.grpo_loss(logits, ids, old, w["A"], w["eps"], w["G"])
    assert out["loss"] == pytest.approx(w["loss"], rel=1e-14)
    np.testing.assert_allclose(out["rho"], w["rho"], rtol=1e-14)
    assert list(out["clipped"]) == w["clipped"]
    np.testing.assert_allclose(out["dlogits"], np.array(w["dlogits"]), atol=1e-15)


def _rand_case(R=37, V=301, seed=1, std=2.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(R, V, generator=g) * std).to(torch.bfloat16)
    ids = torch.randint(0, V, (R,), generator=g)
    return x, ids


def test_logp_matches_torch_log_softmax_fp64():
    x, ids = _rand_case()
    ref = torch.log_softmax(x.double(), dim=1)[torch.arange(x.shape[0]), ids].numpy()
    np.testing.assert_allclose(grpo.token_logp(x, ids), ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("A", [1.3, -0.7])
def test_rho_one_is_scaled_cross_entropy_gradient(A):
    # With logp_old == logp, rho == 1 in every token: the surrogate is A, nothing is
    # clipped and the logit gradient is -(A/(G R)) * (onehot - softmax), i.e. A/(G R)
    # times the gradient of the summed cross-entropy.
    x, ids = _rand_case(R=23, V=157, seed=3)
    G = 5
    logp = grpo.token_logp(x, ids)
    out = grpo.grpo_loss(x, ids, logp, A, 0.2, G)
    R = x.shape[0]
    xx = x.double().clone().requires_grad_(True)
    torch.nn.functional.cross_entropy(xx, ids.long(), reduction="sum").backward()
    np.testing.assert_allclose(out["dlogits"], (A / (G * R)) * xx.grad.numpy(),
                               rtol=1e-12, atol=1e-15)
    assert out["loss"] == pytest.approx(-A / G, rel=1e-13)
    assert not out["clipped"].any()


def test_dlogits_rows_sum_to_zero():
    x, ids = _rand_case(seed=5)
    noise = torch.randn(x.shape[0], generator=torch.Generator().manual_seed(9)).numpy() * 0.3
    old = grpo.token_logp(x, ids) + noise
    out = grpo.grpo_loss(x, ids, old, 0.9, 0.2, 4)
    np.testing.assert_allclose(out["dlogits"].sum(axis=1), 0.0, atol=1e-15)
    assert out["clipped"].any() and (~out["clipped"]).any()


def test_mask_rule_matches_sign_cases():
    # clipped iff (A>0 and rho>1+eps) or (A<0 and rho<1-eps)
    rho = np.linspace(0.5, 1.5, 101)
    for A in (1.0, -1.0, 0.0):
        _, clipped, _ = grpo.surrogate(rho, A, 0.2)
        want = ((A > 0) & (rho > 1.2)) | ((A < 0) & (rho < 0.8))
        # exact ties at the band edges are excluded from the comparison
        edge = (np.abs(rho - 1.2) < 1e-9) | (np.abs(rho - 0.8) < 1e-9)
        assert (clipped[~edge] == want[~edge]).all()


@pytest.mark.parametrize("A", [0.8, -1.1])
def test_finite_differences_of_loss_wrt_logits(A):
    rng = np.random.default_rng(11)
    R, V, G, eps = 6, 13, 3, 0.2
    x = rng.normal(0, 2, (R, V))
    ids = rng.integers(0, V, R)
    logp = grpo.token_logp(x, ids)
    # old log-probs chosen so every rho sits well away from the band edges 1 +- eps
    offs = np.array([0.5, -0.5, 0.05, -0.05, 0.3, -0.35])
    old = logp + offs
    rho = np.exp(logp - old)
    assert np.all(np.abs(rho - 1.2) > 1e-2) and np.all(np.abs(rho - 0.8) > 1e-2)
    out = grpo.grpo_loss(x, ids, old, A, eps, G)
    h = 1e-6
    num = np.zeros_like(x)
    for r in range(R):
        for v in range(V):
            xp = x.copy(); xp[r, v] += h
            xm = x.copy(); xm[r, v] -= h
            num[r, v] = (grpo.grpo_loss(xp, ids, old, A, eps, G)["loss"]
                         - grpo.grpo_loss(xm, ids, old, A, eps, G)["loss"]) / (2 * h)
    np.testing.assert_allclose(out["dlogits"], num, rtol=1e-6, atol=1e-10)


def test_row_selection_matches_full():
    x, ids = _rand_case(seed=7)
    old = grpo.token_logp(x, ids) + 0.1
    full = grpo.grpo_loss(x, ids, old, 0.5, 0.2, 2)
    rows = [3, 0, 20]
    part = grpo.grpo_loss(x, ids, old, 0.5, 0.2, 2, rows=rows)
    np.testing.assert_array_equal(part["dlogits"], full["dlogits"][rows])
    assert part["loss"] == full["loss"]


def test_finalize_is_scaled_accumulator():
    acc = np.arange(12, dtype=np.float32).reshape(3, 4)
    np.testing.assert_array_equal(grpo.finalize(acc, 0.5), acc.astype(np.float64) * 0.5)
