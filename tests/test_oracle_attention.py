"""Pins for the float64 branch-replay attention oracle against facts fixed outside it:
finite differences, torch fp64 autograd on one packed shared-prefix sequence, torch's
scaled_dot_product_attention, closed forms and sum rules."""
import numpy as np
import pytest
import torch

from oracle import attention as att


def _rand(shape, rng, std=1.0):
    return rng.normal(0.0, std, shape)


def _case(P=5, R=3, Hq=4, Hkv=2, D=3, seed=0, std=0.7):
    rng = np.random.default_rng(seed)
    return dict(k_prefix=_rand((P, Hkv, D), rng, std), v_prefix=_rand((P, Hkv, D), rng, std),
                q=_rand((R, Hq, D), rng, std), k_suffix=_rand((R, Hkv, D), rng, std),
                v_suffix=_rand((R, Hkv, D), rng, std), d_out=_rand((R, Hq, D), rng, 1.0))


def _objective(c):
    o = att.replay_response(c["k_prefix"], c["v_prefix"], c["q"], c["k_suffix"],
                            c["v_suffix"], c["d_out"], want_grads=False)["o"]
    return float((o * c["d_out"]).sum())


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (3, 3), (6, 1)])
def test_finite_differences_every_input(Hq, Hkv):
    c = _case(Hq=Hq, Hkv=Hkv, seed=Hq * 10 + Hkv)
    r = att.replay_response(**c)
    grads = {"q": r["dq"], "k_prefix": r["dk_prefix"], "v_prefix": r["dv_prefix"],
             "k_suffix": r["dk_suffix"], "v_suffix": r["dv_suffix"]}
    h = 1e-6
    for name, g in grads.items():
        num = np.zeros_like(c[name])
        for idx in np.ndindex(c[name].shape):
            cp = {k: v.copy() for k, v in c.items()}
            cm = {k: v.copy() for k, v in c.items()}
            cp[name][idx] += h
            cm[name][idx] -= h
            num[idx] = (_objective(cp) - _objective(cm)) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-9, err_msg=name)


def test_packed_shared_prefix_tree_equals_sum_of_replays():
    """One sequence [prompt; y_1; ...; y_G] with a block mask (y_i sees the prompt and its
    own causal past), differentiated by torch autograd in fp64, must give per-response
    outputs equal to the serial replays and prompt gradients equal to their sum."""
    rng = np.random.default_rng(3)
    P, Hq, Hkv, D = 7, 4, 2, 5
    Rs = [3, 1, 4]
    g = Hq // Hkv
    kp, vp = _rand((P, Hkv, D), rng, 0.8), _rand((P, Hkv, D), rng, 0.8)
    resp = [(_rand((R, Hq, D), rng, 0.8), _rand((R, Hkv, D), rng, 0.8),
             _rand((R, Hkv, D), rng, 0.8), _rand((R, Hq, D), rng)) for R in Rs]
    results, dk_sum, dv_sum = att.replay_group(kp, vp, resp)

    N = P + sum(Rs)
    K = torch.tensor(np.concatenate([kp] + [r[1] for r in resp]), requires_grad=True)
    V = torch.tensor(np.concatenate([vp] + [r[2] for r in resp]), requires_grad=True)
    Q = torch.tensor(np.concatenate([r[0] for r in resp]), requires_grad=True)
    dO = torch.tensor(np.concatenate([r[3] for r in resp]))
    allowed = torch.zeros(sum(Rs), N, dtype=torch.bool)
    row, col = 0, P
    for R in Rs:
        for t in range(R):
            allowed[row + t, :P] = True
            allowed[row + t, col:col + t + 1] = True
        row += R
        col += R
    Kx = K.repeat_interleave(g, dim=1)            # [N, Hq, D], head h -> kv h // g
    Vx = V.repeat_interleave(g, dim=1)
    S = torch.einsum("thd,jhd->htj", Q, Kx) / np.sqrt(D)
    S = S.masked_fill(~allowed[None], float("-inf"))
    O = torch.einsum("htj,jhd->thd", torch.softmax(S, dim=-1), Vx)
    (O * dO).sum().backward()

    row = 0
    for R, r in zip(Rs, results):
        np.testing.assert_allclose(r["o"], O.detach().numpy()[row:row + R], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(r["dq"], Q.grad.numpy()[row:row + R], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(r["dk_suffix"], K.grad.numpy()[P + row:P + row + R], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(r["dv_suffix"], V.grad.numpy()[P + row:P + row + R], rtol=1e-10, atol=1e-12)
        row += R
    np.testing.assert_allclose(dk_sum, K.grad.numpy()[:P], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv_sum, V.grad.numpy()[:P], rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (6, 2), (2, 2)])
def test_forward_matches_torch_sdpa_causal_fp64(Hq, Hkv):
    rng = np.random.default_rng(Hq + Hkv)
    P, R, D = 19, 11, 8
    c = _case(P=P, R=R, Hq=Hq, Hkv=Hkv, D=D, seed=5)
    r = att.replay_response(**c, want_grads=False)
    # queries at prompt positions are zero-filled; is_causal on the full square sequence
    Qf = np.concatenate([np.zeros((P, Hq, D)), c["q"]])
    Kf = np.concatenate([c["k_prefix"], c["k_suffix"]])
    Vf = np.concatenate([c["v_prefix"], c["v_suffix"]])
    t = lambda a: torch.tensor(a).permute(1, 0, 2)[None]   # [1, H, N, D]
    O = torch.nn.functional.scaled_dot_product_attention(t(Qf), t(Kf), t(Vf), is_causal=True,
                                                         enable_gqa=True)
    np.testing.assert_allclose(r["o"], O[0].permute(1, 0, 2).numpy()[P:], rtol=1e-12, atol=1e-13)


def test_equal_keys_give_mean_of_visible_values():
    rng = np.random.default_rng(8)
    P, R, Hq, Hkv, D = 6, 5, 2, 1, 4
    k = rng.normal(size=D)
    c = dict(k_prefix=np.tile(k, (P, Hkv, 1)), v_prefix=rng.normal(size=(P, Hkv, D)),
             q=rng.normal(size=(R, Hq, D)), k_suffix=np.tile(k, (R, Hkv, 1)),
             v_suffix=rng.normal(size=(R, Hkv, D)), d_out=rng.normal(size=(R, Hq, D)))
    r = att.replay_response(**c)
    allv = np.concatenate([c["v_prefix"][:, 0], c["v_suffix"][:, 0]])
    for t in range(R):
        want = allv[:P + t + 1].mean(axis=0)        # prompt + suffix keys 0..t
        for h in range(Hq):
            np.testing.assert_allclose(r["o"][t, h], want, rtol=1e-13, atol=1e-14)
            # uniform attention over n keys: LSE = s q.k + log n
            lse = (c["q"][t, h] @ k) / np.sqrt(D) + np.log(P + t + 1)
            assert r["lse"][t, h] == pytest.approx(lse, rel=1e-13)


def test_constant_values_give_that_value_and_no_key_gradient():
    rng = np.random.default_rng(9)
    P, R, Hq, Hkv, D = 5, 4, 4, 2, 3
    c = _case(P=P, R=R, Hq=Hq, Hkv=Hkv, D=D, seed=9)
    cv = rng.normal(size=(Hkv, D))
    c["v_prefix"] = np.broadcast_to(cv, (P, Hkv, D)).copy()
    c["v_suffix"] = np.broadcast_to(cv, (R, Hkv, D)).copy()
    r = att.replay_response(**c)
    for h in range(Hq):
        np.testing.assert_allclose(r["o"][:, h], np.broadcast_to(cv[h // 2], (R, D)), rtol=1e-13)
    np.testing.assert_allclose(r["dq"], 0.0, atol=1e-13)
    np.testing.assert_allclose(r["dk_prefix"], 0.0, atol=1e-13)
    np.testing.assert_allclose(r["dk_suffix"], 0.0, atol=1e-13)


def test_key_shift_invariance():
    c = _case(P=6, R=4, Hq=4, Hkv=2, D=5, seed=12)
    r0 = att.replay_response(**c)
    shift = np.random.default_rng(1).normal(size=(1, 2, 5))
    c2 = dict(c)
    c2["k_prefix"] = c["k_prefix"] + shift
    c2["k_suffix"] = c["k_suffix"] + shift
    r1 = att.replay_response(**c2)
    np.testing.assert_allclose(r1["o"], r0["o"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r1["dq"], r0["dq"], rtol=1e-10, atol=1e-12)


def test_sum_rules_over_keys():
    """sum_j dK_j = 0 and sum_j dV_j = sum over the group's rows of dO, per kv head."""
    c = _case(P=9, R=6, Hq=6, Hkv=2, D=4, seed=21)
    r = att.replay_response(**c)
    dk = np.concatenate([r["dk_prefix"], r["dk_suffix"]]).sum(axis=0)
    dv = np.concatenate([r["dv_prefix"], r["dv_suffix"]]).sum(axis=0)
    np.testing.assert_allclose(dk, 0.0, atol=1e-12)
    want = c["d_out"].reshape(6, 2, 3, 4).sum(axis=(0, 2))
    np.testing.assert_allclose(dv, want, rtol=1e-12, atol=1e-12)


def test_response_rows_match_full_replay():
    c = _case(P=33, R=9, Hq=4, Hkv=1, D=6, seed=4)
    full = att.replay_response(**c)
    rows = [(0, 0), (8, 3), (4, 2), (8, 0)]
    o, lse, dq = att.response_rows(c["k_prefix"], c["v_prefix"], c["q"], c["k_suffix"],
                                   c["v_suffix"], c["d_out"], rows)
    for i, (t, h) in enumerate(rows):
        np.testing.assert_allclose(o[i], full["o"][t, h], rtol=1e-12)
        assert lse[i] == pytest.approx(full["lse"][t, h], rel=1e-13)
        np.testing.assert_allclose(dq[i], full["dq"][t, h], rtol=1e-10, atol=1e-13)


def test_prompt_gradient_is_linear_in_the_group():
    """The group's prompt gradient is the sum of the responses' (replays are independent)."""
    rng = np.random.default_rng(2)
    P, Hq, Hkv, D = 8, 2, 1, 4
    kp, vp = rng.normal(size=(P, Hkv, D)), rng.normal(size=(P, Hkv, D))
    resp = [(rng.normal(size=(R, Hq, D)), rng.normal(size=(R, Hkv, D)),
             rng.normal(size=(R, Hkv, D)), rng.normal(size=(R, Hq, D))) for R in (2, 5)]
    _, dk, dv = att.replay_group(kp, vp, resp)
    a = att.replay_response(kp, vp, *resp[0])
    b = att.replay_response(kp, vp, *resp[1])
    np.testing.assert_allclose(dk, a["dk_prefix"] + b["dk_prefix"], rtol=1e-14)
    np.testing.assert_allclose(dv, a["dv_prefix"] + b["dv_prefix"], rtol=1e-14)


def test_row_range_gives_exact_tail_key_gradients():
    """Suffix keys j >= t0 are seen only by rows t >= t0, so replaying just those rows
    reproduces their key gradients (and those rows' outputs) exactly."""
    c = _case(P=13, R=9, Hq=4, Hkv=2, D=5, seed=31)
    full = att.replay_response(**c)
    part = att.replay_response(**c, row_range=(6, 9))
    np.testing.assert_allclose(part["o"][6:], full["o"][6:], rtol=1e-13)
    np.testing.assert_allclose(part["dq"][6:], full["dq"][6:], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(part["dk_suffix"][6:], full["dk_suffix"][6:], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(part["dv_suffix"][6:], full["dv_suffix"][6:], rtol=1e-12, atol=1e-14)
    assert np.all(part["o"][:6] == 0.0)


def test_merge_of_key_shards_equals_attention_over_all_keys():
    """Attention over a key set split into disjoint shards, each computed on its own by
    torch (fp64 softmax and logsumexp), then merged by the oracle, equals torch's attention
    over all keys; one part merges to itself; equal lse gives the plain average."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(21)
    T, D, N = 7, 16, 53
    q = torch.tensor(rng.normal(size=(T, D)))
    k = torch.tensor(rng.normal(size=(N, D)) * 1.5)
    v = torch.tensor(rng.normal(size=(N, D)))
    s = q @ k.T / np.sqrt(D)
    o_full = torch.softmax(s, dim=1) @ v
    lse_full = torch.logsumexp(s, dim=1)
    bounds = [0, 5, 6, 30, 53]
    o_parts, lse_parts = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        sp = s[:, a:b]
        o_parts.append((torch.softmax(sp, dim=1) @ v[a:b]).numpy())
        lse_parts.append(torch.logsumexp(sp, dim=1).numpy())
    o, lse = att.merge_partials(o_parts, lse_parts)
    assert np.allclose(o, o_full.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(lse, lse_full.numpy(), rtol=0, atol=1e-12)
    o1, l1 = att.merge_partials(o_parts[:1], lse_parts[:1])
    assert np.array_equal(o1, o_parts[0]) and np.allclose(l1, lse_parts[0], atol=0)
    o2, l2 = att.merge_partials([o_parts[0], o_parts[1]], [lse_parts[0], lse_parts[0]])
    assert np.allclose(o2, 0.5 * (o_parts[0] + o_parts[1]), atol=1e-15)
    assert np.allclose(l2, lse_parts[0] + np.log(2.0), atol=1e-15)


@pytest.mark.parametrize("Hq,Hkv,D", [(4, 2, 5), (3, 3, 4), (6, 1, 8)])
def test_prompt_key_grads_match_autograd_at_selected_keys(Hq, Hkv, D):
    """prompt_key_grads against torch fp64 autograd of plain causal attention over each
    concatenated [prompt; response_i] (explicit mask, explicit softmax), the prompt
    gradients summed over the group, at an unsorted subset of prompt rows with a repeat."""
    rng = np.random.default_rng(Hq * 100 + Hkv * 10 + D)
    P, Rs = 11, [4, 1, 6]
    g = Hq // Hkv
    s = 1.0 / np.sqrt(D)
    kp, vp = _rand((P, Hkv, D), rng, 0.9), _rand((P, Hkv, D), rng, 0.9)
    resp = [(_rand((R, Hq, D), rng, 0.9), _rand((R, Hkv, D), rng, 0.9),
             _rand((R, Hkv, D), rng, 0.9), _rand((R, Hq, D), rng)) for R in Rs]
    Kp = torch.tensor(kp, requires_grad=True)
    Vp = torch.tensor(vp, requires_grad=True)
    total = 0.0
    for q, ks, vs, do in resp:
        R = q.shape[0]
        K = torch.cat([Kp, torch.tensor(ks)])                     # [P+R, Hkv, D]
        V = torch.cat([Vp, torch.tensor(vs)])
        Q = torch.tensor(q)
        mask = torch.arange(P + R)[None, :] <= (P + torch.arange(R))[:, None]
        for h in range(Hq):
            S = s * Q[:, h, :] @ K[:, h // g, :].T
            A = torch.softmax(S.masked_fill(~mask, float("-inf")), dim=1)
            total = total + (A @ V[:, h // g, :] * torch.tensor(do[:, h, :])).sum()
    total.backward()
    keys = [7, 0, P - 1, 3, 7]
    dk, dv = att.prompt_key_grads(kp, vp, resp, keys)
    np.testing.assert_allclose(dk, Kp.grad.numpy()[keys], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, Vp.grad.numpy()[keys], rtol=1e-10, atol=1e-12)
    # small row chunks split the forward statistics across chunks: same result
    dk2, dv2 = att.prompt_key_grads(kp, vp, resp, keys, row_chunk=2)
    np.testing.assert_allclose(dk2, dk, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dv2, dv, rtol=1e-12, atol=1e-14)
