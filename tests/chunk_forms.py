"""Chunked (parallel-in-chunk) forms of the CCQ forward, fp64 numpy.

A second, independent algorithm that must reach the oracle's token-by-token
result up to rounding order.  It is used two ways: as a pin on the oracle
(a dropped term, wrong sign or transposed operand in either one makes them
disagree) and as the written-out statement of the chunk algebra that the
CUDA kernels implement.  Test helper only.

Derivation (per chunk of L tokens, 0-based i, j; state S0, C0, m0, n0 at the
chunk start; t_i = n0 + i + 1 tokens seen after token i):

  CCQ read (Sigma_t q as defined on the CCQ pages, expanded over the chunk):
    A_ij  = q_i . k_j                      (j <= i)
    s_i   = m_t . q_i = m0 . q_i + sum_{j<=i} A_ij
    P_i   = C0 q_i + sum_{j<=i} (A_ij - s_i/t_i) k_j - (s_i/t_i) m0
          = t_i * Sigma_{t_i} q_i
    qc_i  = q_i - (lambda_i / t_i) P_i

  GLA (per-channel decay; Bc_i = sum_{j<=i} log alpha_j, R = Bc_{L-1}):
    Qt = qc * exp(Bc - R),  Kh = K * exp(R - Bc),  Sb = exp(R) * S0 (rows)
    O  = tril(Qt Kh^T) V + Qt Sb,     S <- Sb + Kh^T V

  Gated DeltaNet (scalar decay; g_i = sum_{j<=i} log alpha_j):
    Gam_ij = exp(g_i - g_j);  A_ij = beta_i Gam_ij k_i . k_j  (i > j)
    U  = (I + A)^-1 (beta V - (beta exp(g)) * (K S0))
    O  = exp(g) * (Qc S0) + tril(Gam * (Qc K^T)) U
    S <- exp(g_L) S0 + (K * exp(g_L - g))^T U
"""
from __future__ import annotations

import numpy as np


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def ccq_chunked(backbone, q, k, v, log_alpha, w_lambda, b_lambda, beta=None, lambda_in=None,
                S0=None, C0=None, m0=None, t0=0, chunk=64):
    """Same arguments/shapes as oracle.run (fp64 arrays). Returns o, lambda, S, C, m."""
    q, k, v, log_alpha = (np.asarray(a, np.float64) for a in (q, k, v, log_alpha))
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, T, dv))
    lam_all = np.zeros((B, H, T))
    S_out = np.zeros((B, H, dk, dv))
    C_out = np.zeros((B, H, dk, dk))
    m_out = np.zeros((B, H, dk))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[b, h], np.float64)
            C = np.zeros((dk, dk)) if C0 is None else np.array(C0[b, h], np.float64)
            m = np.zeros(dk) if m0 is None else np.array(m0[b, h], np.float64)
            n = float(t0)
            for c0 in range(0, T, chunk):
                sl = slice(c0, min(T, c0 + chunk))
                Q, K, V = q[b, h, sl], k[b, h, sl], v[b, h, sl]
                L = Q.shape[0]
                t = n + np.arange(1, L + 1)
                A = np.tril(Q @ K.T)
                s = Q @ m + A.sum(axis=1)
                if lambda_in is None:
                    lam = _sigmoid(Q @ w_lambda[h] + b_lambda[h])
                else:
                    lam = np.asarray(lambda_in[b, h, sl], np.float64)
                Ahat = np.tril(A - (s / t)[:, None])
                P = Q @ C + Ahat @ K - np.outer(s / t, m)
                Qc = Q - (lam / t)[:, None] * P
                if backbone == "gla":
                    Bc = np.cumsum(log_alpha[b, h, sl], axis=0)
                    R = Bc[-1]
                    Qt = Qc * np.exp(Bc - R)
                    Kh = K * np.exp(R - Bc)
                    Sb = np.exp(R)[:, None] * S
                    O = np.tril(Qt @ Kh.T) @ V + Qt @ Sb
                    S = Sb + Kh.T @ V
                else:
                    g = np.cumsum(log_alpha[b, h, sl])
                    bt = np.asarray(beta[b, h, sl], np.float64)
                    Gam = np.exp(g[:, None] - g[None, :])
                    Aw = np.tril(bt[:, None] * Gam * (K @ K.T), -1)
                    X = bt[:, None] * V - (bt * np.exp(g))[:, None] * (K @ S)
                    U = np.linalg.solve(np.eye(L) + Aw, X)
                    O = np.exp(g)[:, None] * (Qc @ S) + np.tril(Gam * (Qc @ K.T)) @ U
                    S = np.exp(g[-1]) * S + (K * np.exp(g[-1] - g)[:, None]).T @ U
                C = C + K.T @ K
                m = m + K.sum(axis=0)
                n += L
                o[b, h, sl] = O
                lam_all[b, h, sl] = lam
            S_out[b, h], C_out[b, h], m_out[b, h] = S, C, m
    return {"o": o, "lambda": lam_all, "S": S_out, "C": C_out, "m": m_out}
