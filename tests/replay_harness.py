"""Shared helpers for the GPU parity tests: run a group through the C ABI (via the thin
binding) and compare against the float64 oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

from long_context_grpo_gb300 import workloads as wl

# Tolerances (relative L2 unless stated): bf16 outputs and dQ 1e-2; the fp32 group-summed
# prompt gradients 2e-2; the loss scalar 1e-4 relative; LSE 2e-3 absolute (natural log).
TOL_BF16 = 1e-2
TOL_PREFIX = 2e-2
TOL_LOSS = 1e-4
TOL_LSE = 2e-3
MASK_BAND = 1e-6


def f64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def rel_l2(got, ref):
    got, ref = f64(got), f64(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in GPU output"
    den = np.linalg.norm(ref.ravel())
    return float(np.linalg.norm((got - ref).ravel()) / max(den, 1e-30))


def make_group(w, seed=0, device="cuda", q_scale=1.0):
    R = wl.response_lengths(w, seed)
    kp, vp = wl.prefix_kv(w, seed, device)
    resp = [wl.response_attention(w, i, R[i], seed, device, q_scale) for i in range(w.G)]
    return R, kp, vp, resp


def gpu_replay(w, kp, vp, resp, dtype_out_fp32=True):
    import long_context_grpo_gb300 as ls
    dev = kp.device
    dk_acc = torch.empty(kp.shape, dtype=torch.float32, device=dev)
    dv_acc = torch.empty(kp.shape, dtype=torch.float32, device=dev)
    pre = ls.Prefix(kp, vp, dk_acc, dv_acc, Hq=w.Hq)
    outs = []
    for (q, ks, vs, do) in resp:
        o, lse = pre.fwd(q, ks, vs)
        dq, dks, dvs = pre.bwd(q, ks, vs, o, lse, do)
        outs.append(dict(o=o, lse=lse, dq=dq, dk_suffix=dks, dv_suffix=dvs))
    dk = torch.empty(kp.shape, dtype=torch.float32, device=dev)
    dv = torch.empty(kp.shape, dtype=torch.float32, device=dev)
    pre.finalize(1.0, dk, dv, out_fp32=True)
    torch.cuda.synchronize()
    st = ls.device_status()
    pre.close()
    return outs, dk, dv, st
