"""Blockwise suffix replay (LongStraw review, section 3-2 (4)) against the float64 oracle.

Causal attention over [prompt; response] does not depend on how the response rows are
grouped, so a response replayed block by block -- each block seeing the prompt, the earlier
blocks and (causally) itself, its key/value gradients added into the accumulator rows of
every row it sees -- must give the whole-response oracle's outputs and gradients.  The
oracle is the plain whole-response replay; no block arithmetic is restated here.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_grpo_gb300 import workloads as wl
from replay_harness import TOL_BF16, TOL_LSE, TOL_PREFIX, f64, gpu_replay, make_group, rel_l2

pytestmark = pytest.mark.gpu

CASES = {
    # name: (P, R tuple, Hq, Hkv, D, block length)
    "g4_blocks64": (300, (1, 130, 257), 8, 2, 128, 64),
    "g4_blocks100_ragged": (300, (1, 130, 257), 8, 2, 128, 100),
    "g8_blocks128": (1000, (300, 129), 16, 2, 128, 128),
    "g6_d64_blocks37": (129, (50, 200), 12, 2, 64, 37),
    "g1_one_block": (700, (400,), 2, 2, 128, 4096),
}


def spans(R, block):
    return [(t0, min(R, t0 + block)) for t0 in range(0, R, block)]


def block_replay(w, kp, vp, resp, block, bwd_reverse=True):
    """Run a group through the blockwise entry points; the K/V buffers hold
    [prompt; current response] and the response rows of the accumulators are read out
    (and cleared) after each response."""
    import long_context_grpo_gb300 as ls
    dev = kp.device
    P0, Hkv, D = kp.shape
    Rmax = max(x[0].shape[0] for x in resp)
    kbuf = torch.zeros((P0 + Rmax, Hkv, D), dtype=torch.bfloat16, device=dev)
    vbuf = torch.zeros_like(kbuf)
    kbuf[:P0] = kp
    vbuf[:P0] = vp
    dk_acc = torch.empty(kbuf.shape, dtype=torch.float32, device=dev)
    dv_acc = torch.empty(kbuf.shape, dtype=torch.float32, device=dev)
    pre = ls.Prefix(kbuf, vbuf, dk_acc, dv_acc, Hq=w.Hq)
    outs = []
    for (q, ks, vs, do) in resp:
        R = q.shape[0]
        kbuf[P0:P0 + R] = ks
        vbuf[P0:P0 + R] = vs
        o = torch.empty_like(q)
        lse = torch.empty((R, w.Hq), dtype=torch.float32, device=dev)
        dq = torch.empty_like(q)
        sp = spans(R, block)
        for t0, t1 in sp:
            pre.block_fwd(P0 + t0, q[t0:t1], o[t0:t1], lse[t0:t1])
        for t0, t1 in (reversed(sp) if bwd_reverse else sp):
            pre.block_bwd(P0 + t0, q[t0:t1], o[t0:t1], lse[t0:t1], do[t0:t1], dq[t0:t1])
        dks = torch.empty((R, Hkv, D), dtype=torch.float32, device=dev)
        dvs = torch.empty_like(dks)
        pre.finalize_rows(P0, R, 1.0, dks, dvs, out_fp32=True, reset=True)
        outs.append(dict(o=o, lse=lse, dq=dq, dk_suffix=dks, dv_suffix=dvs))
    dk = torch.empty(kp.shape, dtype=torch.float32, device=dev)
    dv = torch.empty(kp.shape, dtype=torch.float32, device=dev)
    pre.finalize_rows(0, P0, 1.0, dk, dv, out_fp32=True)
    torch.cuda.synchronize()
    st = ls.device_status()
    pre.close()
    return outs, dk, dv, st


@pytest.mark.parametrize("name", list(CASES))
def test_block_replay_matches_whole_response_oracle(name):
    P, Rs, Hq, Hkv, D, block = CASES[name]
    w = wl.small(name, P, Rs, Hq, Hkv, D)
    R, kp, vp, resp = make_group(w, seed=5)
    outs, dk, dv, st = block_replay(w, kp, vp, resp, block)
    assert st == (0, 0), "device status %s" % (st,)
    res, dk_ref, dv_ref = oracle.replay_group(kp, vp, [tuple(x) for x in resp])
    for i, (r, g) in enumerate(zip(res, outs)):
        assert rel_l2(g["o"], r["o"]) < TOL_BF16, ("o", i, rel_l2(g["o"], r["o"]))
        assert np.max(np.abs(f64(g["lse"]) - r["lse"])) < TOL_LSE, ("lse", i)
        assert rel_l2(g["dq"], r["dq"]) < TOL_BF16, ("dq", i, rel_l2(g["dq"], r["dq"]))
        assert rel_l2(g["dk_suffix"], r["dk_suffix"]) < TOL_BF16, ("dk_suffix", i)
        assert rel_l2(g["dv_suffix"], r["dv_suffix"]) < TOL_BF16, ("dv_suffix", i)
    assert rel_l2(dk, dk_ref) < TOL_PREFIX, ("dk_prefix", rel_l2(dk, dk_ref))
    assert rel_l2(dv, dv_ref) < TOL_PREFIX, ("dv_prefix", rel_l2(dv, dv_ref))


def test_one_block_is_bitwise_the_whole_response_replay():
    """With a single block the tiling is that of ls_replay_fwd/bwd; only the suffix key
    gradients take the accumulator route (fp32, then one rounding to bf16)."""
    w = wl.small("one_block", 1000, (300, 129), 16, 2, 128)
    R, kp, vp, resp = make_group(w, seed=2)
    a, dka, dva, sta = gpu_replay(w, kp, vp, resp)
    b, dkb, dvb, stb = block_replay(w, kp, vp, resp, block=1 << 20)
    assert sta == (0, 0) and stb == (0, 0)
    for x, y in zip(a, b):
        for key in ("o", "lse", "dq"):
            assert torch.equal(x[key], y[key]), key
        for key in ("dk_suffix", "dv_suffix"):
            assert torch.equal(x[key], y[key].to(torch.bfloat16)), key
    assert torch.equal(dka, dkb) and torch.equal(dva, dvb)


def test_block_replay_is_deterministic_and_backward_order_only_reorders_sums():
    w = wl.small("det", 300, (257,), 8, 2, 128)
    R, kp, vp, resp = make_group(w, seed=7)
    a = block_replay(w, kp, vp, resp, 64)
    b = block_replay(w, kp, vp, resp, 64)
    c = block_replay(w, kp, vp, resp, 64, bwd_reverse=False)
    for x, y in zip(a[0], b[0]):
        for key in x:
            assert torch.equal(x[key], y[key]), key
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    # forward outputs and dq do not depend on the backward order; accumulated key
    # gradients differ at most by the fp32 rounding of the summation order
    for x, y in zip(a[0], c[0]):
        for key in ("o", "lse", "dq"):
            assert torch.equal(x[key], y[key]), key
        for key in ("dk_suffix", "dv_suffix"):
            assert rel_l2(x[key], y[key]) < 1e-5, key
    assert rel_l2(a[1], c[1]) < 1e-5 and rel_l2(a[2], c[2]) < 1e-5


def test_block_arguments_are_checked_before_launch():
    import long_context_grpo_gb300 as ls
    w = wl.small("args", 128, (64,), 2, 2, 64)
    R, kp, vp, resp = make_group(w, seed=0)
    dk_acc = torch.empty(kp.shape, dtype=torch.float32, device=kp.device)
    dv_acc = torch.empty_like(dk_acc)
    pre = ls.Prefix(kp, vp, dk_acc, dv_acc, Hq=w.Hq)
    q = resp[0][0][:32].contiguous()
    with pytest.raises(ls.LongStrawError):
        pre.block_fwd(0, q)                    # prefix_len must be >= 1
    with pytest.raises(ls.LongStrawError):
        pre.block_fwd(100, q)                  # 100 + 32 rows > P = 128
    with pytest.raises(ls.LongStrawError):
        pre.finalize_rows(120, 16, 1.0, torch.empty((16, 2, 64), dtype=torch.float32, device=kp.device),
                          torch.empty((16, 2, 64), dtype=torch.float32, device=kp.device), out_fp32=True)
    pre.close()


# ------------------------------------------------------------------ full-size workloads
def _slice(w, kv, kp, vp, q, ks, vs, do):
    g = w.group
    hs = slice(kv * g, (kv + 1) * g)
    return (kp[:, kv:kv + 1].cpu(), vp[:, kv:kv + 1].cpu(), q[:, hs].cpu(),
            ks[:, kv:kv + 1].cpu(), vs[:, kv:kv + 1].cpu(), do[:, hs].cpu())


@pytest.mark.slow
@pytest.mark.parametrize("name,block", [("p262k", 1000), ("p2m", 4096)])
def test_block_replay_full_size_sampled(name, block):
    """First response of the workload replayed in blocks against the full prompt: O, LSE
    and dQ of sampled rows (each row exact on its own), dK/dV of the last 16 response keys
    (exact from the rows at or after them), and over every key the sum rules
    sum dV = sum dO and sum dK = 0."""
    torch.cuda.empty_cache()
    w = wl.WORKLOADS[name]
    R = wl.response_lengths(w, 0)[0]
    kp, vp = wl.prefix_kv(w, 0, "cuda")
    q, ks, vs, do = wl.response_attention(w, 0, R, 0, "cuda")
    outs, dk, dv, st = block_replay(w, kp, vp, [(q, ks, vs, do)], block)
    assert st == (0, 0)
    out = outs[0]
    kv, g = 1, w.group
    sl = _slice(w, kv, kp, vp, q, ks, vs, do)
    rng = np.random.default_rng(11)
    ts = sorted(set([0, R - 1, block - 1, block, R // 2] + [int(x) for x in rng.integers(0, R, 7)]))
    rows = [(t, int(rng.integers(0, g))) for t in ts if t < R]
    o_ref, lse_ref, dq_ref = oracle.response_rows(*sl, rows)
    o = torch.stack([out["o"][t, kv * g + h] for t, h in rows])
    lse = torch.stack([out["lse"][t, kv * g + h] for t, h in rows])
    dq = torch.stack([out["dq"][t, kv * g + h] for t, h in rows])
    assert rel_l2(o, o_ref) < TOL_BF16
    assert np.max(np.abs(f64(lse) - lse_ref)) < TOL_LSE
    assert rel_l2(dq, dq_ref) < TOL_BF16
    ref = oracle.replay_response(*sl, row_range=(R - 16, R))
    assert rel_l2(out["dk_suffix"][R - 16:, kv:kv + 1], ref["dk_suffix"][R - 16:]) < TOL_BF16
    assert rel_l2(out["dv_suffix"][R - 16:, kv:kv + 1], ref["dv_suffix"][R - 16:]) < TOL_BF16
    dv_sum = dv.double().sum(dim=0) + out["dv_suffix"].double().sum(dim=0)
    want = do.double().view(R, w.Hkv, g, w.D).sum(dim=(0, 2))
    assert rel_l2(dv_sum, want) < TOL_PREFIX
    dk_sum = dk.double().sum(dim=0) + out["dk_suffix"].double().sum(dim=0)
    dk_norm = ((dk.double() ** 2).sum(dim=0) + (out["dk_suffix"].double() ** 2).sum(dim=0)).sum().sqrt()
    assert (dk_sum.norm() / dk_norm).item() < TOL_PREFIX
