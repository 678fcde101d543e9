"""The chunked two-sweep gradient algorithm, written out in numpy, against the
fp64 autograd oracle (oracle/backward.py).

This is the algebra the CUDA gradient kernels implement, checked on the CPU
and independent of their code: a forward sweep that forms everything that
needs the forward state (dq, qc, gy and the scalars that rebuild dL/dmu), with
C_u gy_u obtained from the chunk's last C minus the later keys' share; a
reverse sweep over the adjoints of S, C and m, with the S adjoint moved a
chunk at a time (GS_u = P_u X + sum_{u' >= u} (P_u / P_u') qc_u' g_u'^T) and
the decay gradient from the identity

    dL/dlog A_t = qc_t * gqc_t - k_t * (GS_t v_t)   (+ rowsum(dS * S_T) at T),

summed over t' >= t.  Agreement to 1e-10 pins every one of these steps."""
import numpy as np
import pytest

from oracle.backward import gla_backward


def two_sweeps(q, k, v, la, w, b, go, t0=0, S0=None, C0=None, m0=None, dS=None, dC=None,
               dm=None, lam_in=None, L=8):
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else S0.copy()
    C = np.zeros((dk, dk)) if C0 is None else C0.copy()
    m = np.zeros(dk) if m0 is None else m0.copy()
    dS = np.zeros((dk, dv)) if dS is None else dS
    dC = np.zeros((dk, dk)) if dC is None else dC
    dm = np.zeros(dk) if dm is None else dm
    nch = (T + L - 1) // L
    dq = np.zeros((T, dk))
    QC, GY, T1, SC = np.zeros((T, dk)), np.zeros((T, dk)), np.zeros((T, dk)), np.zeros((T, 2))
    dw, db = np.zeros(dk), 0.0
    # ---- forward sweep
    for c in range(nch):
        tc, n = c * L, min(L, T - c * L)
        cq, gqc, mb = np.zeros((n, dk)), np.zeros((n, dk)), np.zeros((n, dk))
        for u in range(n):  # the writes, token by token, and the products with them
            t = tc + u
            C = C + np.outer(k[t], k[t])
            S = np.exp(la[t])[:, None] * S + np.outer(k[t], v[t])
            m = m + k[t]
            cq[u], gqc[u], mb[u] = C @ q[t], S @ go[t], m
        gy, keep = np.zeros((n, dk)), []
        for u in range(n):  # one token at a time: the read and its local gradients
            t = tc + u
            rn = 1.0 / (t0 + t + 1)
            mu = mb[u] * rn
            mqn = mu @ q[t]
            lam = lam_in[t] if lam_in is not None else 1 / (1 + np.exp(-(w @ q[t] + b)))
            y = cq[u] * rn - mu * mqn
            gy[u] = -lam * gqc[u]
            keep.append((rn, mqn, lam, mu, q[t] - lam * y, -(y @ gqc[u]), mu @ gy[u]))
        cgy_end = gy @ C.T  # C at the chunk's last token
        for u in range(n):
            t = tc + u
            rn, mqn, lam, mu, qc, gl, mg = keep[u]
            cgy = cgy_end[u] - sum(k[tc + up] * (k[tc + up] @ gy[u]) for up in range(u + 1, n))
            gz = 0.0 if lam_in is not None else gl * lam * (1 - lam)
            dq[t] = gqc[u] + cgy * rn - mu * mg + gz * w
            QC[t], GY[t], T1[t], SC[t] = qc, gy[u], qc * gqc[u], (mqn * rn, mg * rn)
            dw, db = dw + gz * q[t], db + gz
    acc = (dS * S).sum(1)
    # ---- reverse sweep
    GS, G, Gm, la_next = dS.copy(), dC + dC.T, dm.copy(), np.zeros(dk)
    dK, dV, dLA = np.zeros((T, dk)), np.zeros((T, dv)), np.zeros((T, dk))
    for c in reversed(range(nch)):
        tc, n = c * L, min(L, T - c * L)
        Lc, s = np.zeros((n, dk)), la_next.copy()
        for u in reversed(range(n)):  # log P_u: the decay from token u to the chunk's end
            Lc[u] = s
            s = s + la[tc + u]
        gk = np.zeros((n, dk))
        for u in reversed(range(n)):  # symmetric C adjoint, token by token
            t = tc + u
            G = G + (np.outer(GY[t], q[t]) + np.outer(q[t], GY[t])) / (t0 + t + 1)
            gk[u] = G @ k[t]
        gsv = np.zeros((n, dk))
        for u in range(n):
            t = tc + u
            r = lambda up: np.exp(Lc[u] - Lc[up]) * QC[tc + up]  # noqa: E731  (P_u/P_u') qc_u'
            gsv[u] = np.exp(Lc[u]) * (GS @ v[t]) + sum(r(up) * (go[tc + up] @ v[t])
                                                       for up in range(u, n))
            dV[t] = GS.T @ (np.exp(Lc[u]) * k[t]) + sum(go[tc + up] * (r(up) @ k[t])
                                                       for up in range(u, n))
            gm = Gm + sum(-GY[tc + up] * SC[tc + up, 0] - q[tc + up] * SC[tc + up, 1]
                          for up in range(u, n))
            dK[t] = gk[u] + gm + gsv[u]
        GS = np.exp(Lc[0])[:, None] * GS + sum(
            np.outer(np.exp(Lc[0] - Lc[up]) * QC[tc + up], go[tc + up]) for up in range(n))
        Gm = Gm + sum(-GY[tc + up] * SC[tc + up, 0] - q[tc + up] * SC[tc + up, 1] for up in range(n))
        for u in reversed(range(n)):
            acc = acc + T1[tc + u] - k[tc + u] * gsv[u]
            dLA[tc + u] = acc
        la_next = la[tc]
    return dict(dq=dq, dk=dK, dv=dV, dlog_alpha=dLA, dw_lambda=dw, db_lambda=db,
                dS0=np.exp(la_next)[:, None] * GS, dC0=0.5 * G, dm0=Gm)


def _case(seed, T, dk, dv, state, lam):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, dk))
    k = rng.standard_normal((T, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, dv))
    la = -np.abs(rng.standard_normal((T, dk))) / 3
    w, b = rng.standard_normal(dk) / 3, 0.2
    go = rng.standard_normal((T, dv))
    kw = dict(lam_in=rng.uniform(0, 1, T) if lam else None)
    if state:
        K0 = rng.standard_normal((9, dk))
        kw.update(t0=9, S0=rng.standard_normal((dk, dv)), C0=K0.T @ K0, m0=K0.sum(0),
                  dS=rng.standard_normal((dk, dv)), dC=rng.standard_normal((dk, dk)),
                  dm=rng.standard_normal(dk))
    return q, k, v, la, w, b, go, kw


@pytest.mark.parametrize("T,dk,dv,state,lam", [(1, 4, 3, False, False), (8, 5, 4, False, False),
                                               (29, 6, 5, True, False), (17, 4, 6, True, True)])
def test_two_sweep_algebra_matches_autograd(T, dk, dv, state, lam):
    q, k, v, la, w, b, go, kw = _case(T + dk, T, dk, dv, state, lam)
    got = two_sweeps(q, k, v, la, w, b, go, **kw)
    A = lambda x: None if x is None else np.asarray(x)[None, None]  # noqa: E731
    ref = gla_backward(A(q), A(k), A(v), A(la), w[None], np.array([b]), A(go),
                       lambda_in=A(kw.get("lam_in")), S0=A(kw.get("S0")), C0=A(kw.get("C0")),
                       m0=A(kw.get("m0")), t0=kw.get("t0", 0), dS=A(kw.get("dS")),
                       dC=A(kw.get("dC")), dm=A(kw.get("dm")))
    for name in ("dq", "dk", "dv", "dlog_alpha", "dw_lambda", "db_lambda", "dS0", "dm0"):
        np.testing.assert_allclose(got[name], ref[name][0, 0], rtol=1e-10, atol=1e-10,
                                   err_msg=name)
    r = ref["dC0"][0, 0]
    np.testing.assert_allclose(got["dC0"], 0.5 * (r + r.T), rtol=1e-10, atol=1e-10)
