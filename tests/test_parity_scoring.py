"""Old/reference-policy scoring without gradients: the forward replay plus token
log-probabilities (ls_token_logp), against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from long_context_grpo_gb300 import workloads as wl
from replay_harness import TOL_BF16, TOL_LSE, f64, gpu_replay, make_group, rel_l2

pytestmark = pytest.mark.gpu


def _logits(R, V, seed):
    w = wl.Workload("score", P=1, G=1, Hq=1, Hkv=1, D=64, V=V, R_fixed=(R,))
    return wl.response_loss_inputs(w, 0, R, seed, "cuda")[:2]


@pytest.mark.parametrize("R,V", [(64, 1024), (700, 32000), (257, 151936), (33, 1001)])
def test_token_logp_matches_oracle(R, V):
    import long_context_grpo_gb300 as ls
    logits, ids = _logits(R, V, seed=R + V)
    lp = ls.token_logp(logits, ids)
    torch.cuda.synchronize()
    np.testing.assert_allclose(f64(lp), oracle.token_logp(logits, ids), atol=3e-5, rtol=0)
    assert ls.device_status() == (0, 0)


def test_token_logp_equals_the_loss_pass_logp():
    import long_context_grpo_gb300 as ls
    logits, ids = _logits(300, 4096, seed=5)
    lp = ls.token_logp(logits, ids)
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    _, _, lp2 = ls.grpo_loss(logits, ids, torch.zeros(300, device="cuda"), 0.5, 0.2, 2, loss)
    torch.cuda.synchronize()
    assert torch.equal(lp, lp2)


def test_bad_token_id_sets_device_status():
    import long_context_grpo_gb300 as ls
    logits, ids = _logits(8, 512, seed=1)
    ids = ids.clone()
    ids[3] = 512                     # out of range: recorded, row output 0, no fault
    lp = ls.token_logp(logits, ids)
    torch.cuda.synchronize()
    st, bits = ls.device_status()
    assert bits == 2 and st == 7
    assert float(lp[3]) == 0.0
    assert ls.device_status() == (0, 0)   # reading cleared it


def test_scoring_pass_forward_matches_oracle():
    """The attention half of scoring is the forward replay alone (no backward)."""
    import long_context_grpo_gb300 as ls
    w = wl.small("score_fwd", 500, (200, 77), 8, 2, 128)
    R, kp, vp, resp = make_group(w, seed=9)
    dk = torch.empty(kp.shape, dtype=torch.float32, device="cuda")
    dv = torch.empty_like(dk)
    pre = ls.Prefix(kp, vp, dk, dv, Hq=w.Hq)
    for (q, ks, vs, do) in resp:
        o, lse = pre.fwd(q, ks, vs)
        torch.cuda.synchronize()
        ref = oracle.replay_response(kp, vp, q, ks, vs, do, want_grads=False)
        assert rel_l2(o, ref["o"]) < TOL_BF16
        assert np.max(np.abs(f64(lse) - ref["lse"])) < TOL_LSE
    pre.close()
