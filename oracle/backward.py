"""fp64 CPU oracle for the gradients of the CCQ-GLA forward -- TEST
INFRASTRUCTURE (used by ``tests/`` and ``bench.py``'s CPU-baseline leg only).

The gradient is the plain definition: the derivative of the forward.  The
forward is written out token by token in float64 PyTorch CPU ops, one (b, h)
at a time, and PyTorch's reverse-mode autodiff (a library primitive) gives the
gradients.  The recurrence is the one the C oracle follows (10100.com
article, "method", item 1; gist.science summary of 2606.01294, section 2,
"mechanism" and "integration"):

    S_t = Diag(alpha_t) S_{t-1} + k_t v_t^T,  C_t = C_{t-1} + k_t k_t^T,
    m_t = m_{t-1} + k_t,  n_t = t0 + t + 1,  mu_t = m_t / n_t,
    Sigma_t q_t = C_t q_t / n_t - mu_t (mu_t . q_t),
    lambda_t = sigmoid(w_lambda[h] . q_t + b_lambda[h])  (or lambda_in),
    o_t = S_t^T (q_t - lambda_t Sigma_t q_t).

Pins (tests/test_oracle_pins.py): its forward equals the C oracle's; its
gradients equal central finite differences; with lambda = 0 they reduce to the
closed forms of the plain GLA read.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np
import torch


def _t(x) -> Optional[torch.Tensor]:
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64).clone()
    return torch.as_tensor(np.asarray(x, dtype=np.float64))


def forward_torch(q, k, v, log_alpha, w, b, lambda_in, S0, C0, m0, t0: int):
    """One (b, h): q, k [T, dk]; v [T, dv]; log_alpha [T, dk]; w [dk]; b
    scalar tensor (or lambda_in [T]); S0 [dk, dv], C0 [dk, dk], m0 [dk].
    Returns o [T, dv] and the final S, C, m (autograd-tracked)."""
    T = q.shape[0]
    S, C, m = S0, C0, m0
    outs = []
    for t in range(T):
        qt, kt, vt = q[t], k[t], v[t]
        S = torch.exp(log_alpha[t])[:, None] * S + torch.outer(kt, vt)
        C = C + torch.outer(kt, kt)
        m = m + kt
        n = float(t0 + t + 1)
        mu = m / n
        sq = C @ qt / n - mu * (mu @ qt)
        lam = lambda_in[t] if lambda_in is not None else torch.sigmoid(w @ qt + b)
        outs.append(S.T @ (qt - lam * sq))
    return torch.stack(outs) if outs else torch.zeros((0, v.shape[-1]), dtype=torch.float64), S, C, m


def gla_backward(q, k, v, log_alpha, w_lambda, b_lambda, do, lambda_in=None, S0=None, C0=None,
                 m0=None, t0: int = 0, dS=None, dC=None, dm=None) -> Dict[str, np.ndarray]:
    """Gradients of  L = sum(o * do) + sum(S_T * dS) + sum(C_T * dC) + sum(m_T * dm)
    for every (b, h).  Shapes as the forward ([B,H,T,...]); dS, dC, dm are the
    optional upstream gradients of the final state.  Returns dq, dk, dv,
    dlog_alpha [B,H,T,...], dw_lambda and db_lambda per (b, h) ([B,H,dk],
    [B,H]; zero when lambda_in is given), dS0, dC0, dm0."""
    q, k, v, log_alpha, do = (_t(x) for x in (q, k, v, log_alpha, do))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    W = _t(w_lambda) if w_lambda is not None else torch.zeros((H, dk), dtype=torch.float64)
    Bl = _t(b_lambda) if b_lambda is not None else torch.zeros(H, dtype=torch.float64)
    lin = _t(lambda_in)
    S0, C0, m0, dS, dC, dm = (_t(x) for x in (S0, C0, m0, dS, dC, dm))
    out = {name: np.zeros(shape) for name, shape in (
        ("dq", (B, H, T, dk)), ("dk", (B, H, T, dk)), ("dv", (B, H, T, dv)),
        ("dlog_alpha", (B, H, T, dk)), ("dw_lambda", (B, H, dk)), ("db_lambda", (B, H)),
        ("dS0", (B, H, dk, dv)), ("dC0", (B, H, dk, dk)), ("dm0", (B, H, dk)))}
    for bi in range(B):
        for h in range(H):
            leaves = [q[bi, h].clone().requires_grad_(), k[bi, h].clone().requires_grad_(),
                      v[bi, h].clone().requires_grad_(), log_alpha[bi, h].clone().requires_grad_(),
                      W[h].clone().requires_grad_(), Bl[h].clone().requires_grad_(),
                      (S0[bi, h] if S0 is not None else torch.zeros((dk, dv), dtype=torch.float64)).clone().requires_grad_(),
                      (C0[bi, h] if C0 is not None else torch.zeros((dk, dk), dtype=torch.float64)).clone().requires_grad_(),
                      (m0[bi, h] if m0 is not None else torch.zeros(dk, dtype=torch.float64)).clone().requires_grad_()]
            o, S, C, m = forward_torch(*leaves[:6], lin[bi, h] if lin is not None else None,
                                       *leaves[6:], t0)
            loss = (o * do[bi, h]).sum()
            if dS is not None:
                loss = loss + (S * dS[bi, h]).sum()
            if dC is not None:
                loss = loss + (C * dC[bi, h]).sum()
            if dm is not None:
                loss = loss + (m * dm[bi, h]).sum()
            grads = torch.autograd.grad(loss, leaves, allow_unused=True)
            names = ("dq", "dk", "dv", "dlog_alpha", "dw_lambda", "db_lambda", "dS0", "dC0", "dm0")
            for name, g in zip(names, grads):
                if g is not None:
                    out[name][bi, h] = g.numpy()
    return out
