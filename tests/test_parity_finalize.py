"""Parity of the prompt-gradient finalization (LongStraw review, section 2-1 step 5, "one
gradient finalization"; section 3-2 (7)) in every form the C ABI offers, against the
float64 oracle: bf16 and fp32 outputs, scales other than 1, in-place scaling, reset of the
accumulators, and the row-range variant.

Each case replays a small group through the library (so the accumulators hold a real
group-summed prompt gradient), keeps a copy of the fp32 accumulators, then finalizes:
  - against the oracle's group sum: relative L2 within the prompt-gradient tolerance;
  - against the oracle's finalize of the library's own accumulators: exact where the
    arithmetic is exact (a power-of-two scale, then one rounding to bf16 by round to
    nearest even, oracle.numerics.to_bf16), within one fp32 rounding otherwise.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.numerics import to_bf16
from long_context_grpo_gb300 import workloads as wl
from replay_harness import TOL_PREFIX, f64, make_group, rel_l2

pytestmark = pytest.mark.gpu

SHAPES = [("d128_g4", 1000, (77, 130, 5), 8, 2, 128), ("d64_g1", 333, (40, 1), 2, 2, 64)]


def _group(name, P, R, Hq, Hkv, D):
    import long_context_grpo_gb300 as ls
    w = wl.small(name, P=P, R=R, Hq=Hq, Hkv=Hkv, D=D)
    _, kp, vp, resp = make_group(w, seed=4)
    dk_acc = torch.empty(kp.shape, dtype=torch.float32, device="cuda")
    dv_acc = torch.empty_like(dk_acc)
    pre = ls.Prefix(kp, vp, dk_acc, dv_acc, Hq=Hq)
    for (q, ks, vs, do) in resp:
        o, lse = pre.fwd(q, ks, vs)
        pre.bwd(q, ks, vs, o, lse, do)
    torch.cuda.synchronize()
    _, dk_ref, dv_ref = oracle.replay_group(kp, vp, resp)
    return pre, dk_acc, dv_acc, dk_ref, dv_ref


@pytest.mark.parametrize("name,P,R,Hq,Hkv,D", SHAPES, ids=[s[0] for s in SHAPES])
def test_finalize_bf16_with_group_scale(name, P, R, Hq, Hkv, D):
    import long_context_grpo_gb300 as ls
    pre, dk_acc, dv_acc, dk_ref, dv_ref = _group(name, P, R, Hq, Hkv, D)
    scale = 1.0 / 8.0                           # 1/G for a group of 8: exact in fp32
    acc_k, acc_v = f64(dk_acc), f64(dv_acc)
    dk = torch.empty(dk_acc.shape, dtype=torch.bfloat16, device="cuda")
    dv = torch.empty_like(dk)
    pre.finalize(scale, dk, dv)
    torch.cuda.synchronize()
    assert ls.device_status() == (0, 0)
    assert rel_l2(dk, oracle.finalize(dk_ref, scale)) < TOL_PREFIX
    assert rel_l2(dv, oracle.finalize(dv_ref, scale)) < TOL_PREFIX
    assert np.array_equal(f64(dk), to_bf16(oracle.finalize(acc_k, scale)))
    assert np.array_equal(f64(dv), to_bf16(oracle.finalize(acc_v, scale)))
    # without reset the accumulators are untouched
    assert np.array_equal(f64(dk_acc), acc_k) and np.array_equal(f64(dv_acc), acc_v)
    pre.close()


@pytest.mark.parametrize("name,P,R,Hq,Hkv,D", SHAPES, ids=[s[0] for s in SHAPES])
def test_finalize_fp32_with_inexact_scale(name, P, R, Hq, Hkv, D):
    pre, dk_acc, dv_acc, dk_ref, dv_ref = _group(name, P, R, Hq, Hkv, D)
    scale = 0.3
    acc_k, acc_v = f64(dk_acc), f64(dv_acc)
    dk = torch.empty_like(dk_acc)
    dv = torch.empty_like(dv_acc)
    pre.finalize(scale, dk, dv, out_fp32=True)
    torch.cuda.synchronize()
    assert rel_l2(dk, oracle.finalize(dk_ref, scale)) < TOL_PREFIX
    assert rel_l2(dv, oracle.finalize(dv_ref, scale)) < TOL_PREFIX
    # fp32(0.3) and one fp32 product: at most two roundings of 2^-24 each
    np.testing.assert_allclose(f64(dk), oracle.finalize(acc_k, scale), rtol=2.0 ** -22, atol=0)
    np.testing.assert_allclose(f64(dv), oracle.finalize(acc_v, scale), rtol=2.0 ** -22, atol=0)
    pre.close()


def test_finalize_in_place_scaling():
    name, P, R, Hq, Hkv, D = SHAPES[0]
    pre, dk_acc, dv_acc, dk_ref, dv_ref = _group(name, P, R, Hq, Hkv, D)
    acc_k, acc_v = f64(dk_acc), f64(dv_acc)
    pre.finalize(0.25)                          # both outputs NULL: acc *= scale
    torch.cuda.synchronize()
    assert np.array_equal(f64(dk_acc), oracle.finalize(acc_k, 0.25))
    assert np.array_equal(f64(dv_acc), oracle.finalize(acc_v, 0.25))
    assert rel_l2(dk_acc, oracle.finalize(dk_ref, 0.25)) < TOL_PREFIX
    pre.close()


def test_finalize_with_reset_zeroes_the_accumulators():
    import long_context_grpo_gb300 as ls
    name, P, R, Hq, Hkv, D = SHAPES[0]
    pre, dk_acc, dv_acc, dk_ref, dv_ref = _group(name, P, R, Hq, Hkv, D)
    acc_k, acc_v = f64(dk_acc), f64(dv_acc)
    dk = torch.empty(dk_acc.shape, dtype=torch.bfloat16, device="cuda")
    dv = torch.empty_like(dk)
    pre.finalize(1.0, dk, dv, reset=True)
    torch.cuda.synchronize()
    assert np.array_equal(f64(dk), to_bf16(acc_k))
    assert np.array_equal(f64(dv), to_bf16(acc_v))
    assert rel_l2(dk, dk_ref) < TOL_PREFIX
    assert int(torch.count_nonzero(dk_acc)) == 0 and int(torch.count_nonzero(dv_acc)) == 0
    assert ls.device_status() == (0, 0)
    pre.close()


def test_finalize_rows_bf16_with_reset():
    name, P, R, Hq, Hkv, D = SHAPES[0]
    pre, dk_acc, dv_acc, dk_ref, dv_ref = _group(name, P, R, Hq, Hkv, D)
    acc_k, acc_v = f64(dk_acc), f64(dv_acc)
    row0, nrows, scale = 129, 517, 0.125
    dk = torch.empty((nrows, Hkv, D), dtype=torch.bfloat16, device="cuda")
    dv = torch.empty_like(dk)
    pre.finalize_rows(row0, nrows, scale, dk, dv, reset=True)
    torch.cuda.synchronize()
    rows = slice(row0, row0 + nrows)
    assert np.array_equal(f64(dk), to_bf16(oracle.finalize(acc_k[rows], scale)))
    assert np.array_equal(f64(dv), to_bf16(oracle.finalize(acc_v[rows], scale)))
    assert rel_l2(dk, oracle.finalize(dk_ref[rows], scale)) < TOL_PREFIX
    after_k, after_v = f64(dk_acc), f64(dv_acc)
    assert not after_k[rows].any() and not after_v[rows].any()       # the range is reset
    keep = np.ones(P, dtype=bool)
    keep[rows] = False
    assert np.array_equal(after_k[keep], acc_k[keep]) and np.array_equal(after_v[keep], acc_v[keep])
    pre.close()
