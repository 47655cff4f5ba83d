"""Seeded synthetic workloads for branch replay (shapes and value distributions only).

This module draws random numbers and nothing else: it holds none of the replay or loss
arithmetic, so both the CUDA path and the float64 oracle can be fed from it without
sharing any computation.  Every tensor gets its own generator stream, derived from
(seed, tensor name, response index), so a tensor can be regenerated on its own.

The workload table mirrors the configurations the LongStraw review measures at
(dimensionstp.github.io "LongStraw" review, section 4-2, the Qwen exact-2M receipt:
2,088,960 prompt + 8,192 response positions), scaled to one GPU and one attention
layer.  The old-policy log-probabilities are "current log-prob + noise": the noise
is drawn here, the log-prob itself is computed by whoever consumes the workload.
"""
from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    P: int                      # shared prompt (prefix) length
    G: int                      # group size (responses per prompt)
    Hq: int
    Hkv: int
    D: int
    V: int                      # loss vocabulary
    R_fixed: tuple = ()         # explicit response lengths, else drawn from R_range
    R_range: tuple = (1, 1)     # inclusive bounds for uniform integer draws
    qkv_std: float = 1.0        # multiplied by 1/sqrt(D)
    logit_std: float = 2.0
    old_logp_noise: float = 0.1
    reward_p: float = 0.5
    eps: float = 0.2
    notes: str = ""

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv


WORKLOADS = {
    "tiny": Workload("tiny", P=256, G=4, Hq=2, Hkv=2, D=64, V=1024,
                     R_fixed=(32, 48, 64, 17)),
    "p32k": Workload("p32k", P=32768, G=8, Hq=32, Hkv=8, D=128, V=32000,
                     R_range=(512, 2048)),
    "p262k": Workload("p262k", P=262144, G=16, Hq=40, Hkv=8, D=128, V=151936,
                      R_range=(1024, 4096), reward_p=0.3, old_logp_noise=0.2),
    "p1m": Workload("p1m", P=1048576, G=8, Hq=48, Hkv=8, D=128, V=151936,
                    R_range=(4096, 8192),
                    notes="logit std and old-logp noise not stated: 2.0 and 0.1 assumed"),
    "p2m": Workload("p2m", P=2097152, G=8, Hq=64, Hkv=8, D=128, V=151936,
                    R_range=(8192, 16384),
                    notes="logit std not stated: 2.0 assumed"),
}


def _stream_seed(seed: int, *parts) -> int:
    h = hashlib.sha256(("%d|" % seed + "|".join(str(p) for p in parts)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, seed, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_stream_seed(seed, *parts))
    return g


def response_lengths(w: Workload, seed: int = 0) -> list:
    if w.R_fixed:
        return list(w.R_fixed)
    g = _gen("cpu", seed, "R")
    lo, hi = w.R_range
    return [int(x) for x in torch.randint(lo, hi + 1, (w.G,), generator=g)]


def rewards(w: Workload, seed: int = 0) -> list:
    g = _gen("cpu", seed, "reward")
    return [float(x) for x in (torch.rand((w.G,), generator=g, dtype=torch.float64) < w.reward_p)]


def group_advantages(r) -> list:
    """Group-normalised advantage A_i = (r_i - mean) / (std + 1e-6), population std.

    This is the input recipe the workload table specifies for A_i; the library takes
    A_i as a given scalar per response and never computes it.
    """
    n = len(r)
    mean = sum(r) / n
    std = math.sqrt(sum((x - mean) ** 2 for x in r) / n)
    return [(x - mean) / (std + 1e-6) for x in r]


def _normal(shape, std, device, gen, dtype=torch.bfloat16):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def prefix_kv(w: Workload, seed: int = 0, device="cpu", P: int = None):
    """Resident prompt K/V, bf16 [P, Hkv, D]."""
    P = w.P if P is None else P
    std = w.qkv_std / math.sqrt(w.D)
    k = _normal((P, w.Hkv, w.D), std, device, _gen(device, seed, "k_prefix"))
    v = _normal((P, w.Hkv, w.D), std, device, _gen(device, seed, "v_prefix"))
    return k, v


def response_attention(w: Workload, i: int, R: int, seed: int = 0, device="cpu",
                       q_scale: float = 1.0):
    """Suffix Q [R,Hq,D], K/V [R,Hkv,D] and upstream gradient dO [R,Hq,D], bf16."""
    std = w.qkv_std / math.sqrt(w.D)
    q = _normal((R, w.Hq, w.D), std * q_scale, device, _gen(device, seed, "q", i))
    k = _normal((R, w.Hkv, w.D), std, device, _gen(device, seed, "k_suffix", i))
    v = _normal((R, w.Hkv, w.D), std, device, _gen(device, seed, "v_suffix", i))
    do = _normal((R, w.Hq, w.D), 1.0, device, _gen(device, seed, "d_out", i))
    return q, k, v, do


def response_loss_inputs(w: Workload, i: int, R: int, seed: int = 0, device="cpu"):
    """Logits bf16 [R,V], sampled token ids int32 [R], old-logp noise fp32 [R]."""
    logits = _normal((R, w.V), w.logit_std, device, _gen(device, seed, "logits", i))
    ids = torch.randint(0, w.V, (R,), generator=_gen(device, seed, "ids", i),
                        device=device, dtype=torch.int32)
    noise = torch.randn((R,), generator=_gen(device, seed, "old_logp_noise", i),
                        device=device, dtype=torch.float32) * w.old_logp_noise
    return logits, ids, noise


def small(name: str, P: int, R: tuple, Hq: int, Hkv: int, D: int, V: int = 4096,
          eps: float = 0.2) -> Workload:
    """A reduced workload with the same distributions, for full element-wise parity."""
    return Workload(name, P=P, G=len(R), Hq=Hq, Hkv=Hkv, D=D, V=V, R_fixed=tuple(R), eps=eps)
