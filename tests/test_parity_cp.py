"""Context-parallel prompt sharding (LongStraw review, section 3-2 (2)) emulated on one GPU:
each prompt shard is its own handle (a rank's pages), the last shard also owns the
response's causal suffix.  Forward partials are merged by the cross-shard log-sum-exp; the
backward of every shard uses the merged O and LSE, so each shard's key gradients are exact
and the dQ parts add up.  Compared with the float64 oracle's replay over the whole prompt.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_grpo_gb300 import workloads as wl
from replay_harness import TOL_BF16, TOL_LSE, TOL_PREFIX, f64, gpu_replay, make_group, rel_l2

pytestmark = pytest.mark.gpu

CASES = {
    # name: (P, R tuple, Hq, Hkv, D, shard boundaries of the prompt)
    "three_ragged_shards": (1000, (300, 129, 1), 16, 2, 128, (0, 300, 777, 1000)),
    "two_shards_d64": (257, (50, 200), 12, 2, 64, (0, 128, 257)),
    "eight_shards": (1024, (130,), 8, 2, 128, tuple(range(0, 1025, 128))),
    "tiny_first_shard": (400, (64, 17), 4, 4, 128, (0, 1, 400)),
}


def cp_replay(w, kp, vp, resp, bounds):
    import long_context_grpo_gb300 as ls
    dev = kp.device
    shards = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        dk = torch.empty((b - a,) + tuple(kp.shape[1:]), dtype=torch.float32, device=dev)
        dv = torch.empty_like(dk)
        shards.append(ls.Prefix(kp[a:b], vp[a:b], dk, dv, Hq=w.Hq))
    owner = shards[-1]
    outs = []
    for (q, ks, vs, do) in resp:
        parts = [s.fwd_prompt_only(q) for s in shards[:-1]] + [owner.fwd(q, ks, vs)]
        o, lse = ls.attn_merge([p[0] for p in parts], [p[1] for p in parts])
        dq_parts = [s.bwd_prompt_only(q, o, lse, do) for s in shards[:-1]]
        dq_o, dks, dvs = owner.bwd(q, ks, vs, o, lse, do)
        dq = ls.sum_bf16(dq_parts + [dq_o])
        outs.append(dict(o=o, lse=lse, dq=dq, dk_suffix=dks, dv_suffix=dvs))
    dk_parts, dv_parts = [], []
    for s, (a, b) in zip(shards, zip(bounds[:-1], bounds[1:])):
        dk = torch.empty((b - a,) + tuple(kp.shape[1:]), dtype=torch.float32, device=dev)
        dv = torch.empty_like(dk)
        s.finalize(1.0, dk, dv, out_fp32=True)
        dk_parts.append(dk)
        dv_parts.append(dv)
    torch.cuda.synchronize()
    st = ls.device_status()
    for s in shards:
        s.close()
    return outs, torch.cat(dk_parts), torch.cat(dv_parts), st


@pytest.mark.parametrize("name", list(CASES))
def test_context_parallel_replay_matches_whole_prompt_oracle(name):
    P, Rs, Hq, Hkv, D, bounds = CASES[name]
    w = wl.small(name, P, Rs, Hq, Hkv, D)
    R, kp, vp, resp = make_group(w, seed=6)
    outs, dk, dv, st = cp_replay(w, kp, vp, resp, bounds)
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


def test_one_shard_is_bitwise_the_ordinary_replay():
    """A single shard owning everything: the merge of one part and the sum of one part are
    exact, so the results are the ordinary replay's bit for bit."""
    w = wl.small("one_shard", 500, (200, 33), 8, 2, 128)
    R, kp, vp, resp = make_group(w, seed=3)
    a, dka, dva, sta = gpu_replay(w, kp, vp, resp)
    b, dkb, dvb, stb = cp_replay(w, kp, vp, resp, (0, 500))
    assert sta == (0, 0) and stb == (0, 0)
    for x, y in zip(a, b):
        for key in x:
            assert torch.equal(x[key], y[key]), key
    assert torch.equal(dka, dkb) and torch.equal(dva, dvb)


def test_merge_kernel_matches_oracle_merge():
    import long_context_grpo_gb300 as ls
    g = torch.Generator(device="cuda").manual_seed(5)
    R, Hq, D, n = 77, 6, 128, 5
    o_parts = [torch.randn(R, Hq, D, device="cuda", generator=g).to(torch.bfloat16) for _ in range(n)]
    lse_parts = [torch.randn(R, Hq, device="cuda", generator=g) * 4.0 for _ in range(n)]
    o, lse = ls.attn_merge(o_parts, lse_parts)
    o_ref, lse_ref = oracle.merge_partials([x.cpu() for x in o_parts], [x.cpu() for x in lse_parts])
    assert rel_l2(o, o_ref) < TOL_BF16
    assert np.max(np.abs(f64(lse) - lse_ref)) < 1e-5
    s = ls.sum_bf16(o_parts)
    s_ref = sum(f64(x) for x in o_parts)
    assert rel_l2(s, s_ref) < TOL_BF16


def test_merge_arguments_are_checked_before_launch():
    import long_context_grpo_gb300 as ls
    parts = [torch.zeros(4, 2, 64, dtype=torch.bfloat16, device="cuda") for _ in range(17)]
    lses = [torch.zeros(4, 2, device="cuda") for _ in range(17)]
    with pytest.raises(ls.LongStrawError):
        ls.attn_merge(parts, lses)               # more than 16 parts
    with pytest.raises(ls.LongStrawError):
        ls.sum_bf16([torch.zeros(12, dtype=torch.bfloat16, device="cuda")] * 2)   # count % 8


def test_rank_driver_with_a_one_rank_group():
    """long_context_grpo_gb300.cp.replay_response through a real (one-rank, NCCL) process
    group on this GPU: the exchange is the identity, the results are the oracle's."""
    import os
    import socket
    import torch.distributed as dist
    from long_context_grpo_gb300 import cp
    import long_context_grpo_gb300 as ls
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        w = wl.small("rank_driver", 300, (130,), 8, 2, 128)
        R, kp, vp, resp = make_group(w, seed=8)
        dk = torch.empty(kp.shape, dtype=torch.float32, device="cuda")
        dv = torch.empty_like(dk)
        pre = ls.Prefix(kp, vp, dk, dv, Hq=w.Hq)
        q, ks, vs, do = resp[0]
        o, lse, dq, dks, dvs = cp.replay_response(pre, 0, 1, q, ks, vs, do)
        dkf = torch.empty_like(dk)
        dvf = torch.empty_like(dk)
        pre.finalize(1.0, dkf, dvf, out_fp32=True)
        torch.cuda.synchronize()
        pre.close()
    finally:
        dist.destroy_process_group()
    ref = oracle.replay_response(kp, vp, q, ks, vs, do)
    assert rel_l2(o, ref["o"]) < TOL_BF16 and rel_l2(dq, ref["dq"]) < TOL_BF16
    assert np.max(np.abs(f64(lse) - ref["lse"])) < TOL_LSE
    assert rel_l2(dks, ref["dk_suffix"]) < TOL_BF16 and rel_l2(dvs, ref["dv_suffix"]) < TOL_BF16
    assert rel_l2(dkf, ref["dk_prefix"]) < TOL_PREFIX and rel_l2(dvf, ref["dv_prefix"]) < TOL_PREFIX


def test_dq_exchange_conversions_against_the_oracle_rounding():
    """ls_bf16_to_f32 widens exactly; ls_f32_to_bf16 rounds to nearest, ties to even, bit
    for bit as oracle.numerics.to_bf16 (values across the exponent range, ties included)."""
    import long_context_grpo_gb300 as ls
    from oracle.numerics import to_bf16
    g = torch.Generator(device="cpu").manual_seed(21)
    bits = torch.randint(0, 2 ** 31 - 1, (4096,), generator=g, dtype=torch.int64)
    bits[::2] |= 0x8000                                 # half of the low halves at a tie
    x = (bits.to(torch.int32)).view(torch.float32)
    x = torch.where(torch.isfinite(x), x, torch.zeros_like(x))
    x = torch.cat([x, -x])
    got = ls.f32_to_bf16(x.cuda())
    want = to_bf16(x.double().numpy())
    assert np.array_equal(f64(got), want)
    back = ls.bf16_to_f32(got)
    torch.cuda.synchronize()
    assert np.array_equal(f64(back), want)
    with pytest.raises(ls.LongStrawError):
        ls.f32_to_bf16(torch.zeros(12, device="cuda"))   # count % 8
