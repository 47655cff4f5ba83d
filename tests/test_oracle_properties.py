"""Property-based pins of the float64 oracle on random shapes (hypothesis; CPU only).

Each property compares the oracle with something computed another way:
  - the replay of one response (outputs and every gradient) against torch fp64 autograd
    through softmax attention over the concatenated [prompt; response] sequence with an
    explicit causal mask;
  - the hand-derived logit gradient of the GRPO loss against torch autograd through the
    L_policy expression (away from the clip kinks, where the derivative is one-sided);
  - the shard merge against torch attention over all keys, for random shard boundaries.
"""
import numpy as np
import pytest
import torch

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from oracle import attention as att  # noqa: E402
from oracle import grpo  # noqa: E402


def _torch_replay(kp, vp, q, ks, vs, do, scale):
    """Autograd through attention over [prompt; response]: response row t sees prompt keys
    and response keys 0..t; kv head of query head h is h // (Hq // Hkv)."""
    P, Hkv, D = kp.shape
    R, Hq, _ = q.shape
    g = Hq // Hkv
    t = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)
    kp_, vp_, q_, ks_, vs_ = t(kp), t(vp), t(q), t(ks), t(vs)
    k = torch.cat([kp_, ks_]).repeat_interleave(g, dim=1)        # [P+R, Hq, D]
    v = torch.cat([vp_, vs_]).repeat_interleave(g, dim=1)
    s = torch.einsum("thd,jhd->htj", q_, k) * scale               # [Hq, R, P+R]
    key = torch.arange(P + R)[None, :]
    row = torch.arange(R)[:, None]
    s = s.masked_fill(key > P + row, float("-inf"))
    lse = torch.logsumexp(s, dim=2)                               # [Hq, R]
    o = torch.einsum("htj,jhd->thd", torch.softmax(s, dim=2), v)
    (o * torch.tensor(do)).sum().backward()
    return (o.detach().numpy(), lse.T.detach().numpy(), q_.grad.numpy(), kp_.grad.numpy(),
            vp_.grad.numpy(), ks_.grad.numpy(), vs_.grad.numpy())


@settings(max_examples=30, deadline=None)
@given(P=st.integers(1, 12), R=st.integers(1, 8), Hkv=st.integers(1, 3), g=st.integers(1, 3),
       D=st.integers(1, 8), seed=st.integers(0, 2**31 - 1), std=st.floats(0.1, 2.5))
def test_replay_matches_autograd_on_random_shapes(P, R, Hkv, g, D, seed, std):
    rng = np.random.default_rng(seed)
    Hq = Hkv * g
    kp, vp = rng.normal(0, std, (P, Hkv, D)), rng.normal(0, std, (P, Hkv, D))
    q = rng.normal(0, std, (R, Hq, D))
    ks, vs = rng.normal(0, std, (R, Hkv, D)), rng.normal(0, std, (R, Hkv, D))
    do = rng.normal(0, 1, (R, Hq, D))
    scale = 1.0 / np.sqrt(D)
    got = att.replay_response(kp, vp, q, ks, vs, do, scale=scale)
    o, lse, dq, dkp, dvp, dks, dvs = _torch_replay(kp, vp, q, ks, vs, do, scale)
    for name, ref in (("o", o), ("lse", lse), ("dq", dq), ("dk_prefix", dkp),
                      ("dv_prefix", dvp), ("dk_suffix", dks), ("dv_suffix", dvs)):
        np.testing.assert_allclose(got[name], ref, rtol=1e-10, atol=1e-12, err_msg=name)


@settings(max_examples=30, deadline=None)
@given(R=st.integers(1, 9), V=st.integers(2, 40), G=st.integers(1, 16),
       A=st.floats(-3.0, 3.0), eps=st.floats(0.01, 0.5), seed=st.integers(0, 2**31 - 1),
       spread=st.floats(0.0, 0.8))
def test_loss_gradient_matches_autograd_on_random_cases(R, V, G, A, eps, seed, spread):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 2, (R, V))
    ids = rng.integers(0, V, R)
    logp = grpo.token_logp(x, ids)
    old = logp + rng.uniform(-spread, spread, R)
    rho = np.exp(logp - old)
    hyp.assume(np.all(np.abs(rho - (1 + eps)) > 1e-6) and np.all(np.abs(rho - (1 - eps)) > 1e-6))
    out = grpo.grpo_loss(x, ids, old, A, eps, G)
    xx = torch.tensor(x, requires_grad=True)
    lp = torch.log_softmax(xx, dim=1)[torch.arange(R), torch.tensor(ids)]
    r = torch.exp(lp - torch.tensor(old))
    surr = torch.minimum(r * A, torch.clamp(r, 1 - eps, 1 + eps) * A)
    loss = -surr.sum() / (G * R)
    loss.backward()
    np.testing.assert_allclose(out["loss"], loss.item(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(out["dlogits"], xx.grad.numpy(), rtol=1e-10, atol=1e-14)


@settings(max_examples=30, deadline=None)
@given(N=st.integers(1, 40), T=st.integers(1, 6), D=st.integers(1, 8),
       cuts=st.lists(st.floats(0.0, 1.0), min_size=0, max_size=6),
       seed=st.integers(0, 2**31 - 1))
def test_merge_matches_full_attention_for_random_shards(N, T, D, cuts, seed):
    rng = np.random.default_rng(seed)
    q, k, v = rng.normal(size=(T, D)), rng.normal(size=(N, D)) * 2, rng.normal(size=(N, D))
    bounds = sorted(set([0, N] + [int(c * N) for c in cuts]))
    s = torch.tensor(q @ k.T / np.sqrt(D))
    vt = torch.tensor(v)
    o_parts, l_parts = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b > a:
            o_parts.append((torch.softmax(s[:, a:b], dim=1) @ vt[a:b]).numpy())
            l_parts.append(torch.logsumexp(s[:, a:b], dim=1).numpy())
    o, lse = att.merge_partials(o_parts, l_parts)
    np.testing.assert_allclose(o, (torch.softmax(s, dim=1) @ vt).numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=1).numpy(), rtol=1e-12, atol=1e-12)
