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
