"""Prefix reuse across steps (LongStraw review, section 4-2 "Qwen prefix-reuse extension";
section 4-3 (4), the prompt reuse policy): the prompt state is captured once and kept resident
while several groups are replayed against it, each group's gradient read out by a
finalization that clears the accumulators.  The library part of that mode is the handle:
kept across groups, it must give each group exactly what a freshly prepared one gives
(whether reusing a stale prompt state is acceptable is the caller's policy)."""
import pytest
import torch

from long_context_grpo_gb300 import workloads as wl
from replay_harness import gpu_replay, make_group

pytestmark = pytest.mark.gpu


def test_handle_reused_across_groups_equals_fresh_handles():
    import long_context_grpo_gb300 as ls
    w = wl.small("reuse", 1000, (300, 129, 40), 16, 2, 128)
    R, kp, vp, groups = make_group(w, seed=1)
    groups_b = make_group(w, seed=2)[3]
    dk_acc = torch.empty(kp.shape, dtype=torch.float32, device=kp.device)
    dv_acc = torch.empty_like(dk_acc)
    pre = ls.Prefix(kp, vp, dk_acc, dv_acc, Hq=w.Hq)
    got = []
    for resp in (groups, groups_b, groups):
        outs = []
        for (q, ks, vs, do) in resp:
            o, lse = pre.fwd(q, ks, vs)
            dq, dks, dvs = pre.bwd(q, ks, vs, o, lse, do)
            outs.append((o, lse, dq, dks, dvs))
        dk = torch.empty_like(dk_acc)
        dv = torch.empty_like(dk_acc)
        pre.finalize(1.0, dk, dv, out_fp32=True, reset=True)
        got.append((outs, dk, dv))
    torch.cuda.synchronize()
    assert ls.device_status() == (0, 0)
    pre.close()
    for resp, (outs, dk, dv) in zip((groups, groups_b, groups), got):
        ref, dk_ref, dv_ref, st = gpu_replay(w, kp, vp, resp)
        assert st == (0, 0)
        for x, y in zip(ref, outs):
            for key, t in zip(("o", "lse", "dq", "dk_suffix", "dv_suffix"), y):
                assert torch.equal(x[key], t), key
        assert torch.equal(dk, dk_ref) and torch.equal(dv, dv_ref)
