"""GPU replay attention (forward + backward + prompt-gradient accumulation) against the
float64 oracle, element by element, at sizes that span several tiles and ragged tails."""
import numpy as np
import pytest
import torch

import oracle
from long_context_grpo_gb300 import workloads as wl
from replay_harness import (TOL_BF16, TOL_LSE, TOL_PREFIX, f64, gpu_replay, make_group,
                            rel_l2)

pytestmark = pytest.mark.gpu

SMALL = {
    # name: (P, R tuple, Hq, Hkv, D)
    "tiny": None,
    "g4_ragged": (300, (1, 130, 257), 8, 2, 128),
    "g5_pad": (200, (70, 33), 10, 2, 128),
    "g6_d64": (129, (50, 200), 12, 2, 64),
    "g8_two_tiles": (1000, (300, 129), 16, 2, 128),
    "g16_short": (64, (20, 3), 16, 1, 128),
    "g1_d128_long": (700, (400,), 2, 2, 128),
    "p1_one_prompt_token": (1, (5, 130), 4, 1, 64),
    "exact_tiles": (256, (128, 16), 4, 4, 128),
}


def _workload(name):
    if name == "tiny":
        return wl.WORKLOADS["tiny"]
    P, R, Hq, Hkv, D = SMALL[name]
    return wl.small(name, P, R, Hq, Hkv, D)


def _check_group(w, kp, vp, resp, outs, dk, dv, st):
    assert st == (0, 0), "device status %s" % (st,)
    res, dk_ref, dv_ref = oracle.replay_group(kp, vp, [tuple(x) for x in resp])
    for i, (r, g) in enumerate(zip(res, outs)):
        assert rel_l2(g["o"], r["o"]) < TOL_BF16, ("o", i, rel_l2(g["o"], r["o"]))
        assert np.max(np.abs(f64(g["lse"]) - r["lse"])) < TOL_LSE, ("lse", i)
        assert rel_l2(g["dq"], r["dq"]) < TOL_BF16, ("dq", i, rel_l2(g["dq"], r["dq"]))
        assert rel_l2(g["dk_suffix"], r["dk_suffix"]) < TOL_BF16, ("dk_suffix", i, rel_l2(g["dk_suffix"], r["dk_suffix"]))
        assert rel_l2(g["dv_suffix"], r["dv_suffix"]) < TOL_BF16, ("dv_suffix", i, rel_l2(g["dv_suffix"], r["dv_suffix"]))
    assert rel_l2(dk, dk_ref) < TOL_PREFIX, ("dk_prefix", rel_l2(dk, dk_ref))
    assert rel_l2(dv, dv_ref) < TOL_PREFIX, ("dv_prefix", rel_l2(dv, dv_ref))


@pytest.mark.parametrize("name", list(SMALL))
def test_group_replay_matches_oracle(name):
    w = _workload(name)
    R, kp, vp, resp = make_group(w, seed=0)
    outs, dk, dv, st = gpu_replay(w, kp, vp, resp)
    _check_group(w, kp, vp, resp, outs, dk, dv, st)


def test_peaked_attention_exercises_online_rescale():
    """Keys of the last prompt tile are scaled up so the running max jumps late in the
    sweep and the output rows held in tensor memory must be rescaled."""
    w = wl.small("peaked", 1000, (100, 37), 8, 2, 128)
    R, kp, vp, resp = make_group(w, seed=3, q_scale=8.0)
    kp = kp.clone()
    kp[896:] = (kp[896:].float() * 30.0).to(torch.bfloat16)
    outs, dk, dv, st = gpu_replay(w, kp, vp, resp)
    _check_group(w, kp, vp, resp, outs, dk, dv, st)


def test_prompt_state_is_not_mutated_and_replay_is_deterministic():
    w = _workload("g8_two_tiles")
    R, kp, vp, resp = make_group(w, seed=1)
    k0, v0 = kp.clone(), vp.clone()
    a = gpu_replay(w, kp, vp, resp)
    b = gpu_replay(w, kp, vp, resp)
    assert torch.equal(kp, k0) and torch.equal(vp, v0)
    for x, y in zip(a[0], b[0]):
        for key in x:
            assert torch.equal(x[key], y[key]), key
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
