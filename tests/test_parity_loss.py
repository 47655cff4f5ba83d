"""GPU fused GRPO loss against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from long_context_grpo_gb300 import workloads as wl
from replay_harness import MASK_BAND, TOL_BF16, TOL_LOSS, f64, rel_l2

pytestmark = pytest.mark.gpu


def _run(R, V, A, eps=0.2, G=4, seed=0, noise=0.1, logit_std=2.0, rows=None):
    import long_context_grpo_gb300 as ls
    w = wl.Workload("loss", P=1, G=G, Hq=1, Hkv=1, D=64, V=V, R_fixed=(R,), logit_std=logit_std,
                    old_logp_noise=noise, eps=eps)
    logits, ids, nz = wl.response_loss_inputs(w, 0, R, seed, "cuda")
    logp_ref = oracle.token_logp(logits, ids)
    old = torch.tensor(logp_ref, dtype=torch.float64) + nz.cpu().double()
    old = old.float().cuda()
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    dlog, mask, logp = ls.grpo_loss(logits, ids, old, A, eps, G, loss)
    torch.cuda.synchronize()
    ref = oracle.grpo_loss(logits, ids, old, A, eps, G, rows=rows)
    return dict(loss=float(loss.item()), dlogits=dlog, mask=mask, logp=logp, ref=ref,
                status=ls.device_status())


def _check(out, rows=None):
    ref = out["ref"]
    assert out["status"] == (0, 0)
    assert abs(out["loss"] - ref["loss"]) <= TOL_LOSS * abs(ref["loss"]), (out["loss"], ref["loss"])
    np.testing.assert_allclose(f64(out["logp"]), ref["logp"], atol=2e-5, rtol=0)
    mask = out["mask"].cpu().numpy().astype(bool)
    rho = ref["rho"]
    band = (np.abs(rho - 1.2) < MASK_BAND) | (np.abs(rho - 0.8) < MASK_BAND)
    assert np.array_equal(mask[~band], ref["clipped"][~band])
    d = out["dlogits"] if rows is None else out["dlogits"][torch.tensor(rows, device="cuda")]
    assert rel_l2(d, ref["dlogits"]) < TOL_BF16


@pytest.mark.parametrize("A", [1.0, -0.7])
def test_loss_small_vocab(A):
    out = _run(64, 1024, A, noise=0.3)
    _check(out)
    assert out["ref"]["clipped"].any()


def test_loss_32k_vocab_many_rows():
    out = _run(2048, 32000, 0.9, G=8, seed=1)
    _check(out)


def test_loss_qwen_vocab_sampled_rows():
    rows = [0, 1, 77, 511, 1023]
    out = _run(1024, 151936, -1.1, G=8, seed=2, rows=rows)
    _check(out, rows=rows)


def test_loss_unaligned_vocab_scalar_path():
    out = _run(33, 1001, 0.5, seed=4)
    _check(out)


def test_zero_advantage_gives_zero_gradient():
    out = _run(16, 512, 0.0)
    assert out["loss"] == 0.0
    assert int(out["mask"].sum()) == 0
    assert torch.count_nonzero(out["dlogits"]) == 0


def test_loss_single_row():
    """One token row (the cluster kernel with a single row to walk)."""
    _check(_run(1, 151936, 0.9))


def test_loss_extreme_logits():
    """Logits with standard deviation 20 (row maxima far above the bulk): the running
    maximum and the compensated exp sum stay exact to the oracle's tolerances."""
    _check(_run(256, 32000, -0.6, logit_std=20.0))


@pytest.mark.parametrize("V", [151936, 1003], ids=["cluster_kernel", "row_kernel"])
def test_out_of_range_token_id_sets_status_and_zeroes_its_row(V):
    """An id outside [0, V) sets the index bit of the device status; that row's loss term,
    dlogits, clip mask and log-prob are zero, and every other row is the oracle's (the loss
    still normalised by all R rows)."""
    import long_context_grpo_gb300 as ls
    R, A, eps, G = 64, 1.0, 0.2, 4
    w = wl.Workload("loss", P=1, G=G, Hq=1, Hkv=1, D=64, V=V, R_fixed=(R,), logit_std=2.0,
                    old_logp_noise=0.1, eps=eps)
    logits, ids, nz = wl.response_loss_inputs(w, 0, R, 3, "cuda")
    old = (torch.tensor(oracle.token_logp(logits, ids), dtype=torch.float64) + nz.cpu().double()).float().cuda()
    ref = oracle.grpo_loss(logits, ids, old, A, eps, G)
    bad = [5, 40]
    ids_bad = ids.clone()
    ids_bad[bad[0]] = -1
    ids_bad[bad[1]] = V
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    dlog, mask, logp = ls.grpo_loss(logits, ids_bad, old, A, eps, G, loss)
    torch.cuda.synchronize()
    st, bits = ls.device_status()
    assert bits & 2, (st, bits)
    good = np.setdiff1d(np.arange(R), bad)
    surr, _, _ = oracle.surrogate(ref["rho"], A, eps)
    expect = -(surr[good].sum()) / (G * R)
    assert abs(float(loss.item()) - expect) <= TOL_LOSS * abs(expect)
    d = f64(dlog)
    assert np.all(d[bad] == 0.0)
    assert rel_l2(dlog[torch.tensor(good, device="cuda")], ref["dlogits"][good]) < TOL_BF16
    lp = f64(logp)
    assert np.all(lp[bad] == 0.0)
    np.testing.assert_allclose(lp[good], ref["logp"][good], atol=2e-5, rtol=0)
    m = mask.cpu().numpy().astype(bool)
    assert not m[bad].any()
    assert ls.device_status() == (0, 0)
