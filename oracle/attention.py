"""Float64 CPU oracle for branch-replay attention.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this
module.  It shares no code with the CUDA path.

What it computes (LongStraw review, dimensionstp.github.io "LongStraw", sections 2-1 and
3-2 (4): the prompt is captured once without autograd and each response is replayed on
its own against it, forward and backward, and the gradients are summed over the group):

  for one response i, build the concatenated sequence X_i = [prompt; response_i] of
  length N = P + R_i and run ordinary causal softmax attention for the response rows.
  Suffix row t (0-based) sees every prompt key and the response keys 0..t, i.e. the
  keys j <= P + t of X_i.

  S = s * Q K^T (s = 1/sqrt(D) unless given), P = softmax_row(S), O = P V,
  LSE = log sum_j exp(S_j)  (natural log).

  The backward is written out by the explicit formulas of softmax attention, with the
  upstream gradient dO given on the response rows and zero on the prompt rows (the
  prompt rows carry no loss: the prompt is captured without a graph):
    dV = P^T dO,  dP = dO V^T,  dS = P * (dP - rowsum(P * dP)),
    dQ = s dS K,  dK = s dS^T Q.
  Grouped-query attention: query head h reads kv head floor(h / g), g = Hq / Hkv, and the
  kv-head gradients sum over the g query heads of the group.

  The gradient w.r.t. the prompt keys/values, summed over the G responses of a group, is
  the quantity the prompt-side term of the gradient decomposition (review section 2-2,
  the equation splitting the total gradient at the prompt boundary state z_P) needs for
  this layer.

Pins (tests/test_oracle_attention.py): central finite differences of <O, dO>, torch fp64
autograd on one packed prompt+all-responses sequence with a block mask (the shared
prefix tree), scaled_dot_product_attention in fp64, closed forms (equal keys -> mean of
the visible values, constant values -> that value), shift invariance of the keys and the
sum rules over keys; prompt_key_grads against torch fp64 autograd of causal attention over
each [prompt; response_i] at selected prompt rows.
"""
from __future__ import annotations

import numpy as np

__all__ = ["replay_response", "replay_group", "response_rows", "merge_partials",
           "prompt_key_grads"]

_ROW_CHUNK = 256


def _f64(x):
    """Exact upcast of a bf16/fp32 torch tensor or array to a float64 numpy array."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _kv_of(h: int, Hq: int, Hkv: int) -> int:
    return h // (Hq // Hkv)


def replay_response(k_prefix, v_prefix, q, k_suffix, v_suffix, d_out, scale=None,
                    heads=None, want_grads=True, row_range=None):
    """Forward and backward of one response replayed against the prompt.

    Shapes: k_prefix, v_prefix [P, Hkv, D]; q, d_out [R, Hq, D]; k_suffix, v_suffix
    [R, Hkv, D].  `heads` restricts the work to a subset of query heads (the kv-head
    gradients then contain only those heads' contributions).

    Returns a dict of float64 arrays: o [R,Hq,D], lse [R,Hq], and with want_grads
    dq [R,Hq,D], dk_prefix/dv_prefix [P,Hkv,D], dk_suffix/dv_suffix [R,Hkv,D].
    Entries for query heads outside `heads` stay zero.
    """
    Kp, Vp, Q, Ks, Vs = (_f64(a) for a in (k_prefix, v_prefix, q, k_suffix, v_suffix))
    dO = _f64(d_out) if want_grads else None
    P, Hkv, D = Kp.shape
    R, Hq, _ = Q.shape
    s = (1.0 / np.sqrt(D)) if scale is None else float(scale)
    heads = range(Hq) if heads is None else heads
    N = P + R

    o = np.zeros((R, Hq, D))
    lse = np.zeros((R, Hq))
    if want_grads:
        dq = np.zeros((R, Hq, D))
        dk = np.zeros((N, Hkv, D))
        dv = np.zeros((N, Hkv, D))

    for h in heads:
        kv = _kv_of(h, Hq, Hkv)
        K = np.concatenate([Kp[:, kv, :], Ks[:, kv, :]], axis=0)   # keys of X_i
        Vv = np.concatenate([Vp[:, kv, :], Vs[:, kv, :]], axis=0)
        r0, r1 = (0, R) if row_range is None else row_range
        for t0 in range(r0, r1, _ROW_CHUNK):
            t1 = min(r1, t0 + _ROW_CHUNK)
            t = np.arange(t0, t1)
            S = s * (Q[t0:t1, h, :] @ K.T)                           # [c, N]
            visible = np.arange(N)[None, :] <= (P + t)[:, None]
            S = np.where(visible, S, -np.inf)
            m = S.max(axis=1, keepdims=True)
            E = np.exp(S - m)
            l = E.sum(axis=1, keepdims=True)
            Pm = E / l
            lse[t0:t1, h] = (m + np.log(l))[:, 0]
            o[t0:t1, h, :] = Pm @ Vv
            if want_grads:
                g = dO[t0:t1, h, :]
                dP = g @ Vv.T
                dS = Pm * (dP - (Pm * dP).sum(axis=1, keepdims=True))
                dq[t0:t1, h, :] = s * (dS @ K)
                dk[:, kv, :] += s * (dS.T @ Q[t0:t1, h, :])
                dv[:, kv, :] += Pm.T @ g

    out = {"o": o, "lse": lse}
    if want_grads:
        out.update(dq=dq, dk_prefix=dk[:P], dv_prefix=dv[:P],
                   dk_suffix=dk[P:], dv_suffix=dv[P:])
    return out


def replay_group(k_prefix, v_prefix, responses, scale=None, heads=None):
    """Serial replay of every response of a group; prompt gradients summed over the group.

    `responses` is a sequence of (q, k_suffix, v_suffix, d_out) tuples.  Returns
    (per_response_results, dk_prefix_sum, dv_prefix_sum).
    """
    Kp, Vp = _f64(k_prefix), _f64(v_prefix)
    dk_sum = np.zeros(Kp.shape)
    dv_sum = np.zeros(Vp.shape)
    results = []
    for (q, ks, vs, do) in responses:
        r = replay_response(Kp, Vp, q, ks, vs, do, scale=scale, heads=heads)
        dk_sum += r["dk_prefix"]
        dv_sum += r["dv_prefix"]
        results.append(r)
    return results, dk_sum, dv_sum


def response_rows(k_prefix, v_prefix, q, k_suffix, v_suffix, d_out, rows, scale=None):
    """O, LSE and dQ of selected (t, h) query rows of one response, each row exact.

    The outputs of one row depend only on that row's query, its upstream gradient and
    the keys/values it sees, so a row can be checked on its own at any prompt length.
    Returns (o [n,D], lse [n], dq [n,D]) in the order of `rows`.
    """
    Q = _f64(q)
    dO = _f64(d_out)
    P, Hkv, D = k_prefix.shape
    R, Hq, _ = Q.shape
    s = (1.0 / np.sqrt(D)) if scale is None else float(scale)
    n = len(rows)
    o = np.zeros((n, D))
    lse = np.zeros(n)
    dq = np.zeros((n, D))
    by_kv = {}
    for idx, (t, h) in enumerate(rows):
        by_kv.setdefault(_kv_of(h, Hq, Hkv), []).append(idx)
    for kv, idxs in by_kv.items():
        K = np.concatenate([_f64(k_prefix[:, kv, :]), _f64(k_suffix[:, kv, :])], axis=0)
        Vv = np.concatenate([_f64(v_prefix[:, kv, :]), _f64(v_suffix[:, kv, :])], axis=0)
        for idx in idxs:
            t, h = rows[idx]
            Kt = K[:P + t + 1]                        # keys visible from suffix row t
            Vt = Vv[:P + t + 1]
            S = s * (Kt @ Q[t, h, :])
            m = S.max()
            E = np.exp(S - m)
            l = E.sum()
            Pm = E / l
            lse[idx] = m + np.log(l)
            o[idx] = Pm @ Vt
            dP = Vt @ dO[t, h, :]
            dS = Pm * (dP - (Pm * dP).sum())
            dq[idx] = s * (dS @ Kt)
    return o, lse, dq


def merge_partials(o_parts, lse_parts):
    """Combine attention results computed over disjoint key sets (one per prompt shard of a
    context-parallel prompt; LongStraw review, section 3-2 (2): the cross-rank log-sum-exp
    and output merge).  With lse_r = log sum_{j in K_r} exp(S_j) and o_r the softmax average
    of the values over K_r, the attention over the union of the key sets is
        lse = log sum_r exp(lse_r),   o = sum_r exp(lse_r - lse) o_r.
    o_parts: list of [..., D]; lse_parts: list of [...] (natural log).  float64."""
    lse_parts = [_f64(x) for x in lse_parts]
    o_parts = [_f64(x) for x in o_parts]
    m = np.max(np.stack(lse_parts), axis=0)
    w = [np.exp(l - m) for l in lse_parts]
    total = np.sum(np.stack(w), axis=0)
    lse = m + np.log(total)
    o = sum(wr[..., None] / total[..., None] * orr for wr, orr in zip(w, o_parts))
    return o, lse


def prompt_key_grads(k_prefix, v_prefix, responses, keys, scale=None, row_chunk=64):
    """Group-summed gradient w.r.t. selected prompt keys and values, float64.

    The same quantity as replay_group's dk_prefix / dv_prefix, restricted to the prompt
    rows `keys`, for prompts too long to differentiate whole on the CPU.  The gradient of a
    single key is written out from the same explicit formulas: for response i, query head h
    (kv head floor(h / g)) and suffix row t,
      forward over every key the row sees (all P prompt keys, suffix keys 0..t):
        lse_t = log sum_j exp(s q_t . k_j),  o_t = sum_j exp(s q_t . k_j - lse_t) v_j,
        Delta_t = sum_d dO_t,d o_t,d;
      then for a selected prompt key j (every suffix row sees every prompt key):
        P_tj = exp(s q_t . k_j - lse_t),  dP_tj = dO_t . v_j,  dS_tj = P_tj (dP_tj - Delta_t),
        dk_j += s sum_t dS_tj q_t,         dv_j += sum_t P_tj dO_t,
    summed over the query heads of the kv head and over the G responses.  Only the
    forward touches every key, so the cost is about a third of the whole-prompt backward.

    k_prefix, v_prefix [P, Hkv, D]; `responses` a sequence of (q [R,Hq,D], k_suffix,
    v_suffix [R,Hkv,D], d_out [R,Hq,D]); keys: prompt row indices.  Returns
    (dk [n, Hkv, D], dv [n, Hkv, D]) in the order of `keys`.  Plain torch CPU ops in
    float64 (multithreaded elementwise work); rows are processed `row_chunk` at a time.
    """
    import torch
    f64 = torch.float64

    def t64(x):
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", f64)
        return torch.as_tensor(np.asarray(x, dtype=np.float64))

    Kp, Vp = t64(k_prefix), t64(v_prefix)
    P, Hkv, D = Kp.shape
    s = (1.0 / np.sqrt(D)) if scale is None else float(scale)
    J = torch.as_tensor(np.asarray(keys, dtype=np.int64))
    dk = torch.zeros((len(J), Hkv, D), dtype=f64)
    dv = torch.zeros((len(J), Hkv, D), dtype=f64)
    for (q, ks, vs, do) in responses:
        Q, Ks, Vs, dO = t64(q), t64(ks), t64(vs), t64(do)
        R, Hq, _ = Q.shape
        for h in range(Hq):
            kv = _kv_of(h, Hq, Hkv)
            Kh, Vh = Kp[:, kv, :], Vp[:, kv, :]
            Ksh, Vsh = Ks[:, kv, :], Vs[:, kv, :]
            lse = torch.empty(R, dtype=f64)
            delta = torch.empty(R, dtype=f64)
            for t0 in range(0, R, row_chunk):
                t1 = min(R, t0 + row_chunk)
                Qc = Q[t0:t1, h, :]
                S_p = s * (Qc @ Kh.T)                                   # [c, P], all visible
                S_s = s * (Qc @ Ksh.T)                                  # [c, R], causal
                t = torch.arange(t0, t1)
                S_s = torch.where(torch.arange(R)[None, :] <= t[:, None], S_s,
                                  torch.full_like(S_s, -np.inf))
                m = torch.maximum(S_p.amax(dim=1), S_s.amax(dim=1))[:, None]
                E_p = torch.exp(S_p - m)
                E_s = torch.exp(S_s - m)
                l = E_p.sum(dim=1) + E_s.sum(dim=1)
                o = (E_p @ Vh + E_s @ Vsh) / l[:, None]
                lse[t0:t1] = m[:, 0] + torch.log(l)
                delta[t0:t1] = (dO[t0:t1, h, :] * o).sum(dim=1)
            KJ, VJ = Kh[J], Vh[J]
            Pm = torch.exp(s * (Q[:, h, :] @ KJ.T) - lse[:, None])        # [R, n]
            dP = dO[:, h, :] @ VJ.T
            dS = Pm * (dP - delta[:, None])
            dk[:, kv, :] += s * (dS.T @ Q[:, h, :])
            dv[:, kv, :] += Pm.T @ dO[:, h, :]
    return dk.numpy(), dv.numpy()
