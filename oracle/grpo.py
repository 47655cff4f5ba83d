"""Float64 CPU oracle for the fused GRPO clipped-surrogate loss.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this
module.  It shares no code with the CUDA path.

The objective is the policy loss of the LongStraw review (dimensionstp.github.io
"LongStraw", section 1-1, equation L_policy):

  L = -(1/G) sum_i (1/R_i) sum_t min(rho_{i,t} A_i, clip(rho_{i,t}, 1-eps, 1+eps) A_i)

with rho_{i,t} the ratio of the current to the old policy probability of the sampled
token.  Per token of response i (the library is called once per response):

  lse    = log sum_v exp(x_v)                  (natural log over the vocabulary)
  logp   = x_y - lse                           (y = sampled token id)
  rho    = exp(logp - logp_old)
  surr   = min(rho A, clip(rho, 1-eps, 1+eps) A)
  loss  += -surr / (G R)
  clipped: the min picks the constant clipped branch, i.e. (A > 0 and rho > 1+eps) or
           (A < 0 and rho < 1-eps); on a tie both branches have the same value and the
           unclipped derivative is taken
  g      = d loss / d logp = -A rho [not clipped] / (G R)
  dlogits_v = g (1[v = y] - softmax_v)

Readings where the page is silent: no KL or entropy term (the equation has none); the
log is natural; the advantage is a given per-response scalar.

Pins (tests/test_oracle_grpo.py): hand-worked clip cases (tests/golden/clip_cases.json),
the rho == 1 special case against torch's cross-entropy gradient in fp64, the sum of
each dlogits row being zero, log-softmax against torch in fp64, and central finite
differences of the loss w.r.t. the logits away from the clip kinks.
"""
from __future__ import annotations

import numpy as np

__all__ = ["token_logp", "grpo_loss", "surrogate", "finalize"]

_ROW_CHUNK = 512


def _f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _ids(ids):
    try:
        import torch
        if isinstance(ids, torch.Tensor):
            return ids.detach().to("cpu", torch.int64).numpy().reshape(-1)
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(ids).astype(np.int64).reshape(-1)


def _row_index(t, rows):
    import torch
    return torch.as_tensor(rows, dtype=torch.long, device=t.device)


def _lse_rows(X):
    m = X.max(axis=1, keepdims=True)
    return (m + np.log(np.exp(X - m).sum(axis=1, keepdims=True)))[:, 0]


def token_logp(logits, ids):
    """log softmax(x)_y per row, float64.  logits [R, V], ids [R].  Rows are upcast to
    float64 a chunk at a time, so a full response's logits need not fit in fp64 at once."""
    y = _ids(ids)
    R = logits.shape[0]
    out = np.empty(R)
    for r0 in range(0, R, _ROW_CHUNK):
        r1 = min(R, r0 + _ROW_CHUNK)
        X = _f64(logits[r0:r1])
        out[r0:r1] = X[np.arange(r1 - r0), y[r0:r1]] - _lse_rows(X)
    return out


def surrogate(rho, A, eps):
    """min(rho A, clip(rho, 1-eps, 1+eps) A), the clipped decision and d surr / d rho."""
    rho = np.asarray(rho, dtype=np.float64)
    unclipped = rho * A
    clipped_val = np.clip(rho, 1.0 - eps, 1.0 + eps) * A
    surr = np.minimum(unclipped, clipped_val)
    clipped = clipped_val < unclipped           # strictly: the constant branch wins
    dsurr_drho = np.where(clipped, 0.0, A)
    return surr, clipped, dsurr_drho


def grpo_loss(logits, ids, logp_old, A, eps, G, rows=None):
    """Loss contribution of one response and its gradients, float64.

    logits [R, V] (the exact bf16 values), ids [R], logp_old [R], A scalar, G group size.
    Returns dict(loss=scalar, logp [R], rho [R], clipped bool [R], dlogits [R, V] or the
    selected rows' [n, V] when `rows` is given).  The loss always covers every token.
    """
    y = _ids(ids)
    old = _f64(logp_old).reshape(-1)
    R, V = logits.shape
    A = float(A)
    coef = 1.0 / (G * R)

    logp = np.empty(R)
    lse = np.empty(R)
    for r0 in range(0, R, _ROW_CHUNK):       # rows upcast a chunk at a time
        r1 = min(R, r0 + _ROW_CHUNK)
        X = _f64(logits[r0:r1])
        lse[r0:r1] = _lse_rows(X)
        logp[r0:r1] = X[np.arange(r1 - r0), y[r0:r1]] - lse[r0:r1]
    rho = np.exp(logp - old)
    surr, clipped, dsurr = surrogate(rho, A, eps)
    loss = -coef * surr.sum()
    g = -coef * dsurr * rho                     # d loss / d logp (chain through rho)

    sel = np.arange(R) if rows is None else np.asarray(rows, dtype=np.int64)
    dlogits = np.empty((len(sel), V))
    for k0 in range(0, len(sel), _ROW_CHUNK):
        k1 = min(len(sel), k0 + _ROW_CHUNK)
        rr = sel[k0:k1]
        Xr = _f64(logits[rr] if not hasattr(logits, "index_select") else
                  logits.index_select(0, _row_index(logits, rr)))
        soft = np.exp(Xr - lse[rr, None])
        onehot = np.zeros_like(soft)
        onehot[np.arange(len(rr)), y[rr]] = 1.0
        dlogits[k0:k1] = g[rr, None] * (onehot - soft)
    return {"loss": loss, "logp": logp, "rho": rho, "clipped": clipped, "g": g,
            "dlogits": dlogits}


def finalize(acc, scale=1.0):
    """Group finalization of a prompt-gradient accumulator: scale * sum over the group.

    One finalization per group (review section 2-1, step 5); on one GPU there is no
    collective, so this is the scaled accumulator itself.
    """
    return float(scale) * _f64(acc)
