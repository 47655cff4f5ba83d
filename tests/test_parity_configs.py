"""Parity on the five workload configurations at full size, in the launch configuration the
benchmark times (one prepare, G serial fwd/loss/bwd calls on one stream, one finalize).

What the float64 oracle can afford to compute at each size:
  tiny, p32k  every output of one kv-head group (tiny: all heads), prompt gradients
              included, element by element.
  p262k, p1m, p2m
              - O, LSE and dQ of sampled query rows of the first and last responses (each
                row is exact on its own);
              - dK/dV of the last 16 suffix keys of the first response (only the rows at
                or after a suffix key see it, so replaying those rows is exact);
              - the loss scalar and the clip mask over every token, and dlogits on sampled
                rows, for the first response;
              - for the fp32 prompt accumulators, properties that hold at any size: the
                sum over all keys of dV equals the sum of dO over the group's rows, the sum
                over all keys of dK vanishes, and the prompt K/V are bit-identical after the
                replay;
              - the fp32 prompt accumulators element by element at 512+ seeded prompt
                positions (the first and last prompt tiles among them) of one kv head, on a
                fresh handle over the full prompt with two short ragged responses, against
                the oracle's per-key gradient (oracle.prompt_key_grads), through the whole
                call sequence (prepare, fwd, bwd, bf16 finalize with scale 1/G); also on a
                prompt 1,000 rows past 2M (a ragged last tile, element offsets past 2^31).
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_grpo_gb300 import workloads as wl
from replay_harness import (MASK_BAND, TOL_BF16, TOL_LOSS, TOL_LSE, TOL_PREFIX, f64,
                            make_group, rel_l2)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

LARGE = ["p262k", "p1m", "p2m"]
SAMPLED_KV = 1          # not kv head 0, so head-offset mistakes cannot hide


def _replay(w, kp, vp, resp):
    import long_context_grpo_gb300 as ls
    dk_acc = torch.empty(kp.shape, dtype=torch.float32, device="cuda")
    dv_acc = torch.empty_like(dk_acc)
    pre = ls.Prefix(kp, vp, dk_acc, dv_acc, Hq=w.Hq)
    outs = []
    for (q, ks, vs, do) in resp:
        o, lse = pre.fwd(q, ks, vs)
        dq, dks, dvs = pre.bwd(q, ks, vs, o, lse, do)
        outs.append(dict(o=o, lse=lse, dq=dq, dk_suffix=dks, dv_suffix=dvs))
    dk = torch.empty_like(dk_acc)
    dv = torch.empty_like(dk_acc)
    pre.finalize(1.0, dk, dv, out_fp32=True)
    torch.cuda.synchronize()
    st = ls.device_status()
    pre.close()
    del dk_acc, dv_acc
    return outs, dk, dv, st


_CACHE = {}


def _group(name):
    if name not in _CACHE:
        _CACHE.clear()
        torch.cuda.empty_cache()
        w = wl.WORKLOADS[name]
        R, kp, vp, resp = make_group(w, seed=0)
        k0 = kp[:, SAMPLED_KV].clone()
        v0 = vp[:, SAMPLED_KV].clone()
        outs, dk, dv, st = _replay(w, kp, vp, resp)
        _CACHE[name] = dict(w=w, R=R, kp=kp, vp=vp, resp=resp, outs=outs, dk=dk, dv=dv,
                            st=st, k0=k0, v0=v0)
    return _CACHE[name]


def _kv_slice(w, kv, kp, vp, q, ks, vs, do):
    g = w.group
    hs = slice(kv * g, (kv + 1) * g)
    return (kp[:, kv:kv + 1].cpu(), vp[:, kv:kv + 1].cpu(), q[:, hs].cpu(),
            ks[:, kv:kv + 1].cpu(), vs[:, kv:kv + 1].cpu(), do[:, hs].cpu())


# --------------------------------------------------------------------------- checks
def _check_full_kv_group(G):
    w, kv, g = G["w"], SAMPLED_KV, G["w"].group
    sl = [_kv_slice(w, kv, G["kp"], G["vp"], *r) for r in G["resp"]]
    res, dk_ref, dv_ref = oracle.replay_group(sl[0][0], sl[0][1], [s[2:] for s in sl])
    hs = slice(kv * g, (kv + 1) * g)
    for i, (r, o) in enumerate(zip(res, G["outs"])):
        assert rel_l2(o["o"][:, hs], r["o"]) < TOL_BF16, ("o", i)
        assert np.max(np.abs(f64(o["lse"][:, hs]) - r["lse"])) < TOL_LSE, ("lse", i)
        assert rel_l2(o["dq"][:, hs], r["dq"]) < TOL_BF16, ("dq", i)
        assert rel_l2(o["dk_suffix"][:, kv:kv + 1], r["dk_suffix"]) < TOL_BF16, ("dk_suffix", i)
        assert rel_l2(o["dv_suffix"][:, kv:kv + 1], r["dv_suffix"]) < TOL_BF16, ("dv_suffix", i)
    assert rel_l2(G["dk"][:, kv:kv + 1], dk_ref) < TOL_PREFIX
    assert rel_l2(G["dv"][:, kv:kv + 1], dv_ref) < TOL_PREFIX


def _rows(R, g, rng, n=12):
    ts = sorted(set([0, R - 1, R // 2] + [int(x) for x in rng.integers(0, R, n - 3)]))
    return [(t, int(rng.integers(0, g))) for t in ts]


def _check_sampled_rows(G):
    w, kv, g = G["w"], SAMPLED_KV, G["w"].group
    rng = np.random.default_rng(7)
    for i in (0, w.G - 1):
        q, ks, vs, do = G["resp"][i]
        sl = _kv_slice(w, kv, G["kp"], G["vp"], q, ks, vs, do)
        rows = _rows(G["R"][i], g, rng)
        o_ref, lse_ref, dq_ref = oracle.response_rows(*sl, rows)
        out = G["outs"][i]
        o = torch.stack([out["o"][t, kv * g + h] for t, h in rows])
        lse = torch.stack([out["lse"][t, kv * g + h] for t, h in rows])
        dq = torch.stack([out["dq"][t, kv * g + h] for t, h in rows])
        assert rel_l2(o, o_ref) < TOL_BF16, (w.name, i, "o")
        assert np.max(np.abs(f64(lse) - lse_ref)) < TOL_LSE, (w.name, i, "lse")
        assert rel_l2(dq, dq_ref) < TOL_BF16, (w.name, i, "dq")


def _check_last_suffix_keys(G):
    w, kv = G["w"], SAMPLED_KV
    R = G["R"][0]
    q, ks, vs, do = G["resp"][0]
    sl = _kv_slice(w, kv, G["kp"], G["vp"], q, ks, vs, do)
    t0 = R - 16
    ref = oracle.replay_response(*sl, row_range=(t0, R))
    out = G["outs"][0]
    assert rel_l2(out["dk_suffix"][t0:, kv:kv + 1], ref["dk_suffix"][t0:]) < TOL_BF16
    assert rel_l2(out["dv_suffix"][t0:, kv:kv + 1], ref["dv_suffix"][t0:]) < TOL_BF16


def _check_sum_rules_and_prompt_unchanged(G):
    w = G["w"]
    g = w.group
    # sum over every key (prompt + all suffixes) of dV == sum over the group's rows of dO
    dv_sum = G["dv"].double().sum(dim=0)                   # [Hkv, D]
    dk_sum = G["dk"].double().sum(dim=0)
    dk_norm2 = (G["dk"].double() ** 2).sum(dim=0)
    want = torch.zeros_like(dv_sum)
    for o, (q, ks, vs, do) in zip(G["outs"], G["resp"]):
        dv_sum += o["dv_suffix"].double().sum(dim=0)
        dk_sum += o["dk_suffix"].double().sum(dim=0)
        dk_norm2 += (o["dk_suffix"].double() ** 2).sum(dim=0)
        want += do.double().view(do.shape[0], w.Hkv, g, w.D).sum(dim=(0, 2))
    assert rel_l2(dv_sum, want) < TOL_PREFIX, w.name
    # sum over keys of dK vanishes up to rounding: compare with the keys' total magnitude
    ratio = (dk_sum.norm() / dk_norm2.sum().sqrt()).item()
    assert ratio < TOL_PREFIX, (w.name, ratio)
    # the replays never wrote the resident prompt state
    assert torch.equal(G["kp"][:, SAMPLED_KV], G["k0"])
    assert torch.equal(G["vp"][:, SAMPLED_KV], G["v0"])


def test_p32k_full_size():
    G = _group("p32k")
    assert G["st"] == (0, 0)
    _check_full_kv_group(G)
    _check_sum_rules_and_prompt_unchanged(G)
    # bitwise determinism of the whole group (no atomics anywhere)
    outs, dk, dv, st = _replay(G["w"], G["kp"], G["vp"], G["resp"])
    assert st == (0, 0)
    assert torch.equal(dk, G["dk"]) and torch.equal(dv, G["dv"])
    for a, b in zip(outs, G["outs"]):
        for k in a:
            assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("name", LARGE)
def test_large_config_full_size(name):
    G = _group(name)
    assert G["st"] == (0, 0)
    _check_sampled_rows(G)
    _check_last_suffix_keys(G)
    _check_sum_rules_and_prompt_unchanged(G)


# --------------------------------------------------------------------------- loss
@pytest.mark.parametrize("name", ["tiny", "p32k"] + LARGE)
def test_grpo_loss_full_response_against_oracle(name):
    import long_context_grpo_gb300 as ls
    _CACHE.clear()
    torch.cuda.empty_cache()
    w = wl.WORKLOADS[name]
    R_all = wl.response_lengths(w, 0)
    A_all = wl.group_advantages(wl.rewards(w, 0))
    if all(a == 0.0 for a in A_all):
        A_all = wl.group_advantages([float(i % 2) for i in range(w.G)])
    idx = [i for i in range(w.G) if A_all[i] != 0.0][:1] or [0]
    if name in ("tiny", "p32k"):
        idx = list(range(w.G))
    total_gpu = torch.zeros(1, dtype=torch.float64, device="cuda")
    total_ref = 0.0
    rng = np.random.default_rng(3)
    for i in idx:
        R = R_all[i]
        logits, ids, noise = wl.response_loss_inputs(w, i, R, 0, "cuda")
        old = (torch.tensor(oracle.token_logp(logits, ids)) + noise.cpu().double()).float().cuda()
        dl, mask, logp = ls.grpo_loss(logits, ids, old, A_all[i], w.eps, w.G, total_gpu)
        torch.cuda.synchronize()
        rows = sorted(set([0, R - 1] + [int(x) for x in rng.integers(0, R, 6)]))
        ref = oracle.grpo_loss(logits, ids, old, A_all[i], w.eps, w.G, rows=rows)
        total_ref += ref["loss"]
        band = (np.abs(ref["rho"] - (1 + w.eps)) < MASK_BAND) | (np.abs(ref["rho"] - (1 - w.eps)) < MASK_BAND)
        m = mask.cpu().numpy().astype(bool)
        assert np.array_equal(m[~band], ref["clipped"][~band]), (name, i)
        np.testing.assert_allclose(f64(logp), ref["logp"], atol=3e-5, rtol=0)
        assert rel_l2(dl[torch.tensor(rows, device="cuda")], ref["dlogits"]) < TOL_BF16, (name, i)
        del logits, dl
    assert abs(total_gpu.item() - total_ref) <= TOL_LOSS * abs(total_ref), (name, total_gpu.item(), total_ref)
    assert ls.device_status() == (0, 0)


# --------------------------------------------------------------------------- schedule
def test_peak_memory_is_flat_in_group_size():
    """Serial replay keeps one response's buffers live at a time: the peak device memory
    of the replay loop does not grow with G beyond one response's outputs."""
    import long_context_grpo_gb300 as ls
    w = wl.WORKLOADS["p32k"]
    R, kp, vp, resp = make_group(w, seed=5)
    Rmax = max(R)
    per_resp = Rmax * (2 * w.Hq * w.D * 2 + 2 * w.Hkv * w.D * 2 + w.Hq * 4) + (1 << 22)

    def peak(nresp):
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats()
        base = torch.cuda.memory_allocated()
        dk_acc = torch.empty(kp.shape, dtype=torch.float32, device="cuda")
        dv_acc = torch.empty_like(dk_acc)
        pre = ls.Prefix(kp, vp, dk_acc, dv_acc, Hq=w.Hq)
        for (q, ks, vs, do) in resp[:nresp]:
            o, lse = pre.fwd(q, ks, vs)
            out = pre.bwd(q, ks, vs, o, lse, do)
            del o, lse, out
        pre.close()
        torch.cuda.synchronize()
        p = torch.cuda.max_memory_allocated() - base
        del dk_acc, dv_acc
        return p

    p2, p8 = peak(2), peak(8)
    assert p8 - p2 <= per_resp, (p2, p8, per_resp)


# --------------------------------------------------------------------------- prompt gradients
PROMPT_GRAD_R = (300, 77)
# (workload, prompt rows, kv head checked): never kv head 0, so a head offset cannot hide; on
# the prompt past 2M the last kv head puts elements (row * Hkv + kv) * D beyond 2^31.
PROMPT_GRAD_CASES = [("p262k", 262144, 5), ("p1m", 1048576, 3), ("p2m", 2097152, 6),
                     ("p2m", 2097152 + 1000, 7)]


def _sampled_positions(P, rng, n_random=256):
    """The first and the last prompt tiles (the last one ragged when P % 128 != 0) and
    n_random seeded positions in between."""
    first = np.arange(0, 128)
    last = np.arange((P - 1) // 128 * 128, P)
    mid = np.sort(rng.choice(np.arange(128, (P - 1) // 128 * 128), n_random, replace=False))
    return first, mid, last


@pytest.mark.parametrize("name,P,kv", PROMPT_GRAD_CASES,
                         ids=["p262k", "p1m", "p2m", "p2m_plus_1000"])
def test_large_config_prompt_gradients_at_sampled_positions(name, P, kv):
    import long_context_grpo_gb300 as ls
    _CACHE.clear()
    torch.cuda.empty_cache()
    w = wl.WORKLOADS[name]
    g = w.group
    kp, vp = wl.prefix_kv(w, 0, "cuda", P=P)
    resp = [wl.response_attention(w, i, R, 0, "cuda") for i, R in enumerate(PROMPT_GRAD_R)]
    dk_acc = torch.empty((P, w.Hkv, w.D), dtype=torch.float32, device="cuda")
    dv_acc = torch.empty_like(dk_acc)
    pre = ls.Prefix(kp, vp, dk_acc, dv_acc, Hq=w.Hq)
    outs = []
    for (q, ks, vs, do) in resp:
        o, lse = pre.fwd(q, ks, vs)
        outs.append(pre.bwd(q, ks, vs, o, lse, do))
    scale = 1.0 / len(resp)
    dk_out = torch.empty(dk_acc.shape, dtype=torch.bfloat16, device="cuda")
    dv_out = torch.empty_like(dk_out)
    pre.finalize(scale, dk_out, dv_out)
    torch.cuda.synchronize()
    assert ls.device_status() == (0, 0)
    pre.close()

    first, mid, last = _sampled_positions(P, np.random.default_rng(P + kv))
    keys = np.concatenate([first, mid, last])
    hs = slice(kv * g, (kv + 1) * g)
    sl = [(q[:, hs].cpu(), ks[:, kv:kv + 1].cpu(), vs[:, kv:kv + 1].cpu(), do[:, hs].cpu())
          for (q, ks, vs, do) in resp]
    dk_ref, dv_ref = oracle.prompt_key_grads(kp[:, kv:kv + 1].cpu(), vp[:, kv:kv + 1].cpu(),
                                             sl, keys)
    idx = torch.tensor(keys, device="cuda")
    got_k = dk_acc.index_select(0, idx)[:, kv:kv + 1]
    got_v = dv_acc.index_select(0, idx)[:, kv:kv + 1]
    n1, n2 = len(first), len(first) + len(mid)
    for part, sel in (("first tile", slice(0, n1)), ("random", slice(n1, n2)),
                      ("last tile", slice(n2, None)), ("all", slice(None))):
        assert rel_l2(got_k[sel], dk_ref[sel]) < TOL_PREFIX, (name, P, "dk", part)
        assert rel_l2(got_v[sel], dv_ref[sel]) < TOL_PREFIX, (name, P, "dv", part)
    # the finalized bf16 gradient the benchmark produces: scale * the group sum
    fin_k = dk_out.index_select(0, idx)[:, kv:kv + 1]
    fin_v = dv_out.index_select(0, idx)[:, kv:kv + 1]
    assert rel_l2(fin_k, scale * dk_ref) < TOL_PREFIX, (name, P, "finalized dk")
    assert rel_l2(fin_v, scale * dv_ref) < TOL_PREFIX, (name, P, "finalized dv")
    # any size: the sum rules over every key of the group (prompt + both suffixes)
    dv_sum = dv_acc.double().sum(dim=0)
    want = torch.zeros_like(dv_sum)
    for (dq, dks, dvs), (q, ks, vs, do) in zip(outs, resp):
        dv_sum += dvs.double().sum(dim=0)
        want += do.double().view(do.shape[0], w.Hkv, g, w.D).sum(dim=(0, 2))
    assert rel_l2(dv_sum, want) < TOL_PREFIX, (name, P)
    del kp, vp, dk_acc, dv_acc, dk_out, dv_out
