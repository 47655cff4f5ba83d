"""Failure detection without a GPU fault: a kernel wait that can never complete gives up
after a short limit, records the timeout in the device status word and exits; the host
reads LS_ERR_TIMEOUT and the context keeps working.  Host-side errors are checked too."""
import ctypes

import pytest
import torch

from long_context_grpo_gb300 import build as lsbuild


def _L():
    lsbuild.build()
    from long_context_grpo_gb300 import _lib as b
    return b._lib()


@pytest.mark.gpu
def test_bounded_wait_expires_and_context_stays_usable():
    import long_context_grpo_gb300 as ls
    L = _L()
    assert ls.device_status() == (0, 0)
    s = torch.cuda.current_stream().cuda_stream
    assert L.ls_debug_wait_timeout(50_000_000, s) == 0          # 50 ms
    torch.cuda.synchronize()
    st, bits = ls.device_status()
    assert (st, bits) == (6, 1)                                   # LS_ERR_TIMEOUT, wait bit
    assert ls.device_status() == (0, 0)                           # cleared by the read
    # the context still runs real work correctly
    x = torch.randn(16, 256, device="cuda").to(torch.bfloat16)
    ids = torch.randint(0, 256, (16,), device="cuda", dtype=torch.int32)
    lp = ls.token_logp(x, ids)
    ref = torch.log_softmax(x.double(), dim=1)[torch.arange(16), ids.long()]
    assert torch.allclose(lp.double(), ref, atol=3e-5)


def test_wait_limit_is_validated_on_the_host():
    L = _L()
    assert L.ls_debug_wait_timeout(0, None) == 1
    assert L.ls_debug_wait_timeout(20_000_000_000, None) == 1


def test_launch_failure_injection_arms_and_disarms_on_the_host():
    L = _L()
    assert L.ls_debug_fail_launch(-1) == 0
    assert L.ls_debug_fail_launch_pending() == -1
    assert L.ls_debug_fail_launch(2) == 0
    assert L.ls_debug_fail_launch_pending() == 2
    # a call rejected by its argument checks makes no launch attempt
    assert L.ls_grpo_loss(0, 64, 1, 0x1000, 0x2000, 0x3000, 1.0, 0.2, 0x4000, 0x5000, 0x6000,
                          0x7000, 0x8000, 1 << 20, None) == 1
    assert L.ls_sum_bf16(2, 12, None, 0x5000, None) == 1
    assert L.ls_debug_fail_launch_pending() == 2
    assert L.ls_debug_fail_launch(-5) == 0
    assert L.ls_debug_fail_launch_pending() == -1


def _case():
    from long_context_grpo_gb300 import workloads as wl
    from replay_harness import make_group
    w = wl.small("inject", 300, (70,), 8, 2, 128, V=1024)
    R, kp, vp, resp = make_group(w, seed=12)
    return w, kp, vp, resp[0]


@pytest.mark.gpu
def test_every_entry_point_reports_an_injected_launch_failure_and_recovers():
    """Each compute entry point, with a launch failure injected at each of its launch
    attempts: LS_ERR_CUDA with the injected message, the countdown disarmed, no device
    status set; the same call then succeeds.  A failure placed between the backward's
    launches leaves the prompt accumulators as far as the launches before it took them."""
    import long_context_grpo_gb300 as ls
    L = _L()
    w, kp, vp, (q, ks, vs, do) = _case()
    R = q.shape[0]
    dk = torch.empty(kp.shape, dtype=torch.float32, device="cuda")
    dv = torch.empty_like(dk)
    pre = ls.Prefix(kp, vp, dk, dv, Hq=w.Hq)
    logits = torch.randn((R, w.V), device="cuda").to(torch.bfloat16)
    ids = torch.randint(0, w.V, (R,), device="cuda", dtype=torch.int32)
    old = torch.zeros((R,), device="cuda")
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    parts = [torch.randn(R, w.Hq, w.D, device="cuda").to(torch.bfloat16) for _ in range(2)]
    lses = [torch.randn(R, w.Hq, device="cuda") for _ in range(2)]
    o, lse = pre.fwd(q, ks, vs)
    torch.cuda.synchronize()

    calls = {
        "prepare": (2, lambda: ls.Prefix(kp, vp, torch.empty_like(dk), torch.empty_like(dv), Hq=w.Hq).close()),
        "fwd": (1, lambda: pre.fwd(q, ks, vs, o=o, lse=lse)),
        "fwd_packed": (1, lambda: pre.fwd_packed([0, 30, R], q, ks, vs)),
        "fwd_prompt_only": (1, lambda: pre.fwd_prompt_only(q)),
        "block_fwd": (1, lambda: pre.block_fwd(100, q[:50])),
        "bwd": (3, lambda: pre.bwd(q, ks, vs, o, lse, do)),
        "bwd_packed": (3, lambda: pre.bwd_packed([0, 30, R], q, ks, vs, o, lse, do)),
        "bwd_prompt_only": (3, lambda: pre.bwd_prompt_only(q, o, lse, do)),
        "block_bwd": (3, lambda: pre.block_bwd(100, q[:50], o[:50], lse[:50], do[:50])),
        "grpo_loss": (1, lambda: ls.grpo_loss(logits, ids, old, 0.5, 0.2, 4, loss)),
        "token_logp": (1, lambda: ls.token_logp(logits, ids)),
        "merge": (1, lambda: ls.attn_merge(parts, lses)),
        "sum": (1, lambda: ls.sum_bf16(parts)),
        "bf16_to_f32": (1, lambda: ls.bf16_to_f32(parts[0])),
        "f32_to_bf16": (1, lambda: ls.f32_to_bf16(lses[0])),
        "finalize": (2, lambda: pre.finalize(1.0, torch.empty_like(dk), torch.empty_like(dv), out_fp32=True)),
        "finalize_rows": (2, lambda: pre.finalize_rows(5, 40, 0.5, torch.empty(40, w.Hkv, w.D, device="cuda"),
                                                       torch.empty(40, w.Hkv, w.D, device="cuda"), out_fp32=True)),
    }
    for name, (attempts, fn) in calls.items():
        for k in range(attempts):
            assert L.ls_debug_fail_launch(k) == 0
            with pytest.raises(ls.LongStrawError) as ex:
                fn()
            assert ex.value.status == 5, name
            assert "injected" in str(ex.value), (name, str(ex.value))
            assert L.ls_debug_fail_launch_pending() == -1, name
            torch.cuda.synchronize()
            assert ls.device_status() == (0, 0), name
            fn()                                   # the same call now succeeds
            torch.cuda.synchronize()
    # the no-allocation loss reports through the same path
    s = torch.cuda.current_stream().cuda_stream
    dl = torch.empty_like(logits)
    mask = torch.empty((R,), dtype=torch.uint8, device="cuda")
    assert L.ls_debug_fail_launch(0) == 0
    st = L.ls_grpo_loss_noalloc(R, w.V, 4, logits.data_ptr(), ids.data_ptr(), old.data_ptr(), 0.5,
                                0.2, loss.data_ptr(), dl.data_ptr(), mask.data_ptr(), None, s)
    assert st == 5 and b"injected" in L.ls_last_error()
    # the backward failing at its dK/dV launch leaves the prompt accumulators untouched
    torch.cuda.synchronize()
    before = dk.clone()
    assert L.ls_debug_fail_launch(1) == 0
    with pytest.raises(ls.LongStrawError):
        pre.bwd(q, ks, vs, o, lse, do)
    torch.cuda.synchronize()
    assert torch.equal(dk, before)
    pre.close()
    assert ls.device_status() == (0, 0)
