"""The allocation-free GRPO loss entry point, called through the C ABI.

ls_grpo_loss_noalloc serves callers that cannot allocate device memory where they run (a
fixed memory plan, an allocator that must not be re-entered, a host runtime that may only
hand over buffers it already owns), so it keeps its per-row scratch in a fixed array inside
the library instead of a caller workspace.  Every call reuses that array, so its results
must match ls_grpo_loss and the float64 oracle call after call: here on three calls in a
row, across both loss kernels (the 4-CTA cluster kernel for V a multiple of 8, the
one-CTA-per-row kernel otherwise) and with a later call larger than an earlier one.  This
file is collected last on purpose: if it fails, every other test has already run.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_grpo_gb300 import build as lsbuild
from long_context_grpo_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2
TOL_LOSS = 1e-4
MASK_BAND = 1e-6


def _lib():
    lsbuild.build()
    from long_context_grpo_gb300 import _lib as b
    return b._lib()


def _inputs(R, V, seed):
    w = wl.Workload("noalloc", P=1, G=4, Hq=1, Hkv=1, D=64, V=V, R_fixed=(R,), old_logp_noise=0.3)
    logits, ids, noise = wl.response_loss_inputs(w, 0, R, seed, "cuda")
    # old-policy log-probs near the current ones, so both clip branches occur
    old = (torch.tensor(oracle.token_logp(logits, ids)) + noise.cpu().double()).float().cuda()
    return logits, ids, old


def _run(L, fn, R, V, logits, ids, old, A, eps, G, with_ws):
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    dl = torch.empty((R, V), dtype=torch.bfloat16, device="cuda")
    mask = torch.empty((R,), dtype=torch.uint8, device="cuda")
    logp = torch.empty((R,), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    args = [R, V, G, logits.data_ptr(), ids.data_ptr(), old.data_ptr(), A, eps,
            loss.data_ptr(), dl.data_ptr(), mask.data_ptr(), logp.data_ptr()]
    if with_ws:
        nbytes = L.ls_grpo_loss_workspace_bytes(R)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        st = fn(*args, ws.data_ptr(), nbytes, s)
    else:
        st = fn(*args, s)
    assert st == 0, L.ls_last_error()
    torch.cuda.synchronize()
    return loss.item(), dl, mask, logp


def _rel_l2(a, b):
    a = a.double().cpu().numpy() if isinstance(a, torch.Tensor) else a
    b = b.double().cpu().numpy() if isinstance(b, torch.Tensor) else b
    return np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-30)


def test_noalloc_matches_workspace_entry_point_and_oracle_on_consecutive_calls():
    L = _lib()
    assert L.ls_grpo_loss_noalloc_max_rows() == 65536
    G, eps = 4, 0.2
    # (R, V, A, seed): cluster kernel; one-CTA-per-row kernel (V % 8 != 0) with a larger R;
    # cluster kernel again with a larger R still
    cases = [(777, 4096, 0.8, 11), (1500, 1001, -1.3, 12), (2048, 4096, 1.1, 13)]
    rng = np.random.default_rng(5)
    for call, (R, V, A, seed) in enumerate(cases):
        logits, ids, old = _inputs(R, V, seed)
        ref = _run(L, L.ls_grpo_loss, R, V, logits, ids, old, A, eps, G, with_ws=True)
        got = _run(L, L.ls_grpo_loss_noalloc, R, V, logits, ids, old, A, eps, G, with_ws=False)
        # against the workspace entry point: the same kernels, so the same values
        assert abs(got[0] - ref[0]) <= TOL_LOSS * abs(ref[0]), (call, got[0], ref[0])
        assert _rel_l2(got[1], ref[1]) < TOL_BF16, call
        assert torch.equal(got[2], ref[2]), call
        assert torch.allclose(got[3], ref[3], rtol=0, atol=1e-6), call
        # against the float64 oracle
        rows = sorted(set([0, R - 1] + [int(x) for x in rng.integers(0, R, 14)]))
        o = oracle.grpo_loss(logits, ids, old, A, eps, G, rows=rows)
        assert abs(got[0] - o["loss"]) <= TOL_LOSS * abs(o["loss"]), (call, got[0], o["loss"])
        band = (np.abs(o["rho"] - (1 + eps)) < MASK_BAND) | (np.abs(o["rho"] - (1 - eps)) < MASK_BAND)
        m = got[2].cpu().numpy().astype(bool)
        assert m.any() and (~m).any(), call          # both branches exercised
        assert np.array_equal(m[~band], o["clipped"][~band]), call
        np.testing.assert_allclose(got[3].double().cpu().numpy(), o["logp"], atol=3e-5, rtol=0)
        assert _rel_l2(got[1][torch.tensor(rows, device="cuda")], o["dlogits"]) < TOL_BF16, call


def test_noalloc_rejects_rows_beyond_capacity():
    L = _lib()
    R = L.ls_grpo_loss_noalloc_max_rows() + 1
    st = L.ls_grpo_loss_noalloc(R, 64, 1, 0x1000, 0x2000, 0x3000, 1.0, 0.2, 0x4000, 0x5000,
                                0x6000, 0x7000, None)
    assert st == 2
    assert b"65536" in L.ls_last_error()
