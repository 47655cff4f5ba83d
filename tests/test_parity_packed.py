"""Packed (tree) replay of a whole group in one launch per kernel against the float64
oracle and against the serial per-response calls.

Every response sees the prompt and, causally, only itself, so the packed results are the
serial ones: the forward outputs, dq and the suffix key gradients come from the same tiles
and are bitwise equal; the fp32 prompt accumulators differ only by summation order (the
packed backward adds all responses of a prompt tile on chip, then once into HBM).
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_grpo_gb300 import workloads as wl
from replay_harness import TOL_BF16, TOL_LSE, TOL_PREFIX, f64, gpu_replay, make_group, rel_l2

pytestmark = pytest.mark.gpu

CASES = {
    # name: (P, R tuple, Hq, Hkv, D)
    "g4_ragged": (300, (1, 130, 257), 8, 2, 128),
    "g8_eight_responses": (1000, (300, 129, 17, 128, 255, 64, 1, 400), 16, 2, 128),
    "g6_d64": (129, (50, 200), 12, 2, 64),
    "g1_long": (700, (400, 333), 2, 2, 128),
}


def packed_replay(w, kp, vp, resp):
    import long_context_grpo_gb300 as ls
    dev = kp.device
    Rs = [x[0].shape[0] for x in resp]
    cu = [0]
    for r in Rs:
        cu.append(cu[-1] + r)
    q, ks, vs, do = (torch.cat([x[i] for x in resp]).contiguous() for i in range(4))
    dk_acc = torch.empty(kp.shape, dtype=torch.float32, device=dev)
    dv_acc = torch.empty_like(dk_acc)
    pre = ls.Prefix(kp, vp, dk_acc, dv_acc, Hq=w.Hq)
    o, lse = pre.fwd_packed(cu, q, ks, vs)
    dq, dks, dvs = pre.bwd_packed(cu, q, ks, vs, o, lse, do)
    dk = torch.empty_like(dk_acc)
    dv = torch.empty_like(dk_acc)
    pre.finalize(1.0, dk, dv, out_fp32=True)
    torch.cuda.synchronize()
    st = ls.device_status()
    pre.close()
    outs = [dict(o=o[a:b], lse=lse[a:b], dq=dq[a:b], dk_suffix=dks[a:b], dv_suffix=dvs[a:b])
            for a, b in zip(cu[:-1], cu[1:])]
    return outs, dk, dv, st


@pytest.mark.parametrize("name", list(CASES))
def test_packed_replay_matches_oracle_and_serial_calls(name):
    P, Rs, Hq, Hkv, D = CASES[name]
    w = wl.small(name, P, Rs, Hq, Hkv, D)
    R, kp, vp, resp = make_group(w, seed=4)
    outs, dk, dv, st = packed_replay(w, kp, vp, resp)
    assert st == (0, 0), "device status %s" % (st,)
    res, dk_ref, dv_ref = oracle.replay_group(kp, vp, [tuple(x) for x in resp])
    for i, (r, g) in enumerate(zip(res, outs)):
        assert rel_l2(g["o"], r["o"]) < TOL_BF16, ("o", i)
        assert np.max(np.abs(f64(g["lse"]) - r["lse"])) < TOL_LSE, ("lse", i)
        assert rel_l2(g["dq"], r["dq"]) < TOL_BF16, ("dq", i)
        assert rel_l2(g["dk_suffix"], r["dk_suffix"]) < TOL_BF16, ("dk_suffix", i)
        assert rel_l2(g["dv_suffix"], r["dv_suffix"]) < TOL_BF16, ("dv_suffix", i)
    assert rel_l2(dk, dk_ref) < TOL_PREFIX and rel_l2(dv, dv_ref) < TOL_PREFIX
    a, dka, dva, sta = gpu_replay(w, kp, vp, resp)
    assert sta == (0, 0)
    for x, y in zip(a, outs):
        for key in x:
            assert torch.equal(x[key], y[key]), key
    # same fp32 terms summed in another order (per tile on chip, then once into HBM, instead
    # of once per response); the prompt gradient nearly cancels across the group, so the
    # relative reordering error is a few fp32 ulps times that cancellation factor
    assert rel_l2(dk, dka) < 1e-4 and rel_l2(dv, dva) < 1e-4


def test_packed_arguments_are_checked_before_launch():
    import long_context_grpo_gb300 as ls
    w = wl.small("args", 128, (64,), 2, 2, 64)
    R, kp, vp, resp = make_group(w, seed=0)
    dk_acc = torch.empty(kp.shape, dtype=torch.float32, device=kp.device)
    dv_acc = torch.empty_like(dk_acc)
    pre = ls.Prefix(kp, vp, dk_acc, dv_acc, Hq=w.Hq)
    q, ks, vs, do = resp[0]
    for cu in ([1, 64], [0, 30, 30, 64], [0] + list(range(1, 66))):
        T = cu[-1]
        with pytest.raises(ls.LongStrawError):
            pre.fwd_packed(cu, q[:T] if T <= 64 else torch.zeros((T, 2, 64), dtype=torch.bfloat16, device=kp.device),
                           ks[:T] if T <= 64 else torch.zeros((T, 2, 64), dtype=torch.bfloat16, device=kp.device),
                           vs[:T] if T <= 64 else torch.zeros((T, 2, 64), dtype=torch.bfloat16, device=kp.device))
    assert pre.bwd_packed_workspace_bytes([0, 30, 30, 64]) == 0
    pre.close()
