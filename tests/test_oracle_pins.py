"""Pins for the fp64 oracle: checks against what the CCQ pages and the
mathematics fix, never against the oracle itself.

Sources of each pin:
  * hand-worked example (tests/golden/hand_worked_3tok.json);
  * brute-force explicit covariance (numpy.cov, bias=True) on tiny T;
  * the Hessian of log-sum-exp at q = 0 (closed form and central differences)
    -- gist.science summary of 2606.01294, section 2 "theory";
  * the score-correction identity k_j^T Sigma q = Cov_i(k_j.k_i, k_i.q)
    -- 10100.com article, "method";
  * lambda = 0 reduces to plain GLA / the gated delta rule; alpha = 1 and
    lambda = 0 reduce to the causal masked product tril(QK^T)V;
  * unit keys give eig(I - lambda Sigma) in [1-lambda, 1]; identical keys give
    Sigma = 0 -- 10100.com article, "method", item 2;
  * Gated DeltaNet special cases (beta = 0 is pure decay; alpha = beta = 1 with
    unit keys stores v exactly; the residual contracts by 1 - beta);
  * an independent chunked algorithm (tests/chunk_forms.py);
  * state-split and thread-count invariance.
"""
import json
import os

import numpy as np
import pytest
from scipy.special import expit, logsumexp

import oracle
from chunk_forms import ccq_chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng0 = np.random.default_rng(1234)


def _rand(B, H, T, dk, dv, unit=True, seed=0, backbone="gla"):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, H, T, dk))
    k = r.standard_normal((B, H, T, dk))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((B, H, T, dv))
    if backbone == "gla":
        la = -np.logaddexp(0, -r.standard_normal((B, H, T, dk))) / 4
    else:
        la = -np.logaddexp(0, r.standard_normal((B, H, T))) / 4
    w = r.standard_normal((H, dk)) / np.sqrt(dk)
    b = r.standard_normal(H) * 0.5
    beta = expit(r.standard_normal((B, H, T)))
    return dict(q=q, k=k, v=v, log_alpha=la, w_lambda=w, b_lambda=b, beta=beta)


# --------------------------------------------------------------------------- golden
def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_3tok.json")))
    q = np.array(g["q"], float)[None, None]
    k = np.array(g["k"], float)[None, None]
    v = np.array(g["v"], float)[None, None]
    w = np.array(g["w_lambda"], float)[None]
    b = np.array([g["b_lambda"]], float)
    for name, case in g["cases"].items():
        alpha = np.array(case["alpha"], float)
        la = np.log(alpha)[None, None]
        beta = None
        if case["backbone"] == "gdn":
            beta = np.array(case["beta"], float)[None, None]
        out = oracle.run(case["backbone"], q, k, v, la, w, b, beta=beta, want_sigq=True)
        np.testing.assert_allclose(out["o"][0, 0], np.array(case["o"]), rtol=0, atol=1e-15,
                                   err_msg=name)
        np.testing.assert_allclose(out["S"][0, 0], np.array(case["final_S"]), atol=1e-15)
        np.testing.assert_allclose(out["lambda"][0, 0], g["lambda"], atol=1e-15)
        np.testing.assert_allclose(out["sigq"][0, 0], np.array(g["sigma_q"]), atol=1e-15)
        np.testing.assert_allclose(out["C"][0, 0], np.array(g["final_C"]), atol=0)
        np.testing.assert_allclose(out["m"][0, 0], np.array(g["final_m"]), atol=0)


# --------------------------------------------------------------------------- Sigma
@pytest.mark.parametrize("unit", [True, False])
def test_sigma_matches_bruteforce_covariance(unit):
    d = _rand(1, 2, 13, 5, 3, unit=unit, seed=1)
    out = oracle.run("gla", **d, want_sigq=True)
    for h in range(2):
        K, Q = d["k"][0, h], d["q"][0, h]
        for t in range(13):
            Sig = np.cov(K[: t + 1].T, bias=True) if t > 0 else np.zeros((5, 5))
            np.testing.assert_allclose(out["sigq"][0, h, t], Sig @ Q[t], rtol=1e-12, atol=1e-13)


def test_sigma_with_carried_prefix_matches_full_history():
    d = _rand(1, 1, 20, 6, 4, seed=2)
    pre = {k: (v[:, :, :8] if v.ndim >= 3 and k not in ("w_lambda",) else v) for k, v in d.items()}
    pre["w_lambda"], pre["b_lambda"] = d["w_lambda"], d["b_lambda"]
    s = oracle.run("gla", **pre)
    rest = {k: (v[:, :, 8:] if k in ("q", "k", "v", "log_alpha", "beta") else v)
            for k, v in d.items()}
    out = oracle.run("gla", **rest, S0=s["S"], C0=s["C"], m0=s["m"], t0=8, want_sigq=True)
    K, Q = d["k"][0, 0], d["q"][0, 0]
    for t in range(8, 20):
        Sig = np.cov(K[: t + 1].T, bias=True)
        np.testing.assert_allclose(out["sigq"][0, 0, t - 8], Sig @ Q[t], rtol=1e-12, atol=1e-13)


def test_final_sigma_is_hessian_of_logsumexp_at_zero():
    """Sigma_T = C/n - mu mu^T must equal the Hessian of
    A(q) = log sum_j exp(k_j^T q) at q = 0, by central differences."""
    d = _rand(1, 1, 9, 4, 2, unit=False, seed=3)
    out = oracle.run("gla", **d)
    n = 9
    mu = out["m"][0, 0] / n
    Sig = out["C"][0, 0] / n - np.outer(mu, mu)
    K = d["k"][0, 0]
    f = lambda x: logsumexp(K @ x)  # noqa: E731
    h = 1e-3
    I = np.eye(4)
    Hfd = np.zeros((4, 4))
    for a in range(4):
        for b in range(4):
            Hfd[a, b] = (f(h * I[a] + h * I[b]) - f(h * I[a] - h * I[b])
                         - f(-h * I[a] + h * I[b]) + f(-h * I[a] - h * I[b])) / (4 * h * h)
    np.testing.assert_allclose(Sig, Hfd, atol=5e-6)
    # closed form: softmax weights are uniform at q = 0; gradient there is mu
    np.testing.assert_allclose(Sig, np.cov(K.T, bias=True), atol=1e-13)
    g = np.array([(f(h * I[a]) - f(-h * I[a])) / (2 * h) for a in range(4)])
    np.testing.assert_allclose(mu, g, atol=5e-6)


def test_score_correction_identity():
    """k_j^T Sigma_t q = mean_i[(k_j.k_i)(k_i.q)] - mean_i[k_j.k_i] mean_i[k_i.q]."""
    d = _rand(1, 1, 11, 6, 2, seed=4)
    out = oracle.run("gla", **d, want_sigq=True)
    K, Q = d["k"][0, 0], d["q"][0, 0]
    for t in range(11):
        Kt = K[: t + 1]
        kk = K @ Kt.T                # [all j, i<=t]
        kq = Kt @ Q[t]               # [i<=t]
        rhs = (kk * kq).mean(axis=1) - kk.mean(axis=1) * kq.mean()
        np.testing.assert_allclose(K @ out["sigq"][0, 0, t], rhs, atol=1e-13)


# --------------------------------------------------------------------------- gate
def test_gate_is_sigmoid_of_query_projection():
    d = _rand(2, 3, 7, 5, 4, seed=5)
    out = oracle.run("gla", **d)
    z = np.einsum("bhtd,hd->bht", d["q"], d["w_lambda"]) + d["b_lambda"][None, :, None]
    np.testing.assert_allclose(out["lambda"], expit(z), rtol=1e-14)


def test_lambda_in_overrides_gate():
    d = _rand(1, 2, 6, 4, 3, seed=6)
    lam = np.full((1, 2, 6), 0.1)
    out = oracle.run("gla", **d, lambda_in=lam)
    np.testing.assert_array_equal(out["lambda"], lam)


# --------------------------------------------------------------------------- reductions
def _plain_gla_bruteforce(q, k, v, la):
    """o_t = sum_{j<=t} (sum_c q_tc k_jc prod_{j<i<=t} alpha_ic) v_j (no recurrence)."""
    T = q.shape[0]
    o = np.zeros((T, v.shape[1]))
    for t in range(T):
        for j in range(t + 1):
            decay = np.exp(la[j + 1: t + 1].sum(axis=0))
            o[t] += np.sum(q[t] * k[j] * decay) * v[j]
    return o


def test_lambda_zero_is_plain_gla():
    d = _rand(1, 2, 10, 4, 3, seed=7)
    out = oracle.run("gla", **d, lambda_in=np.zeros((1, 2, 10)))
    for h in range(2):
        ref = _plain_gla_bruteforce(d["q"][0, h], d["k"][0, h], d["v"][0, h], d["log_alpha"][0, h])
        np.testing.assert_allclose(out["o"][0, h], ref, rtol=1e-12, atol=1e-13)


def test_alpha_one_lambda_zero_is_causal_masked_product():
    d = _rand(1, 1, 12, 5, 4, unit=False, seed=8)
    d["log_alpha"] = np.zeros_like(d["log_alpha"])
    out = oracle.run("gla", **d, lambda_in=np.zeros((1, 1, 12)))
    Q, K, V = d["q"][0, 0], d["k"][0, 0], d["v"][0, 0]
    np.testing.assert_allclose(out["o"][0, 0], np.tril(Q @ K.T) @ V, rtol=1e-12, atol=1e-12)


def _plain_gdn_bruteforce(q, k, v, la, beta):
    """Gated delta rule with explicit (I - beta k k^T) matrices, read with q."""
    dk, dv = k.shape[1], v.shape[1]
    S = np.zeros((dk, dv))
    o = []
    for t in range(q.shape[0]):
        S = np.exp(la[t]) * (np.eye(dk) - beta[t] * np.outer(k[t], k[t])) @ S \
            + beta[t] * np.outer(k[t], v[t])
        o.append(S.T @ q[t])
    return np.array(o)


def test_lambda_zero_is_plain_gated_deltanet():
    d = _rand(1, 2, 9, 4, 3, seed=9, backbone="gdn")
    out = oracle.run("gdn", **d, lambda_in=np.zeros((1, 2, 9)))
    for h in range(2):
        ref = _plain_gdn_bruteforce(d["q"][0, h], d["k"][0, h], d["v"][0, h],
                                    d["log_alpha"][0, h], d["beta"][0, h])
        np.testing.assert_allclose(out["o"][0, h], ref, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------- stability
@pytest.mark.parametrize("lam", [0.1, 0.5, 1.0])
def test_unit_keys_eigenvalue_bound(lam):
    d = _rand(1, 1, 40, 8, 2, seed=10)
    for T in (1, 2, 3, 5, 17, 40):
        sub = {k: (v[:, :, :T] if k in ("q", "k", "v", "log_alpha") else v) for k, v in d.items()}
        out = oracle.run("gla", **sub)
        mu = out["m"][0, 0] / T
        Sig = out["C"][0, 0] / T - np.outer(mu, mu)
        ev = np.linalg.eigvalsh(np.eye(8) - lam * Sig)
        assert ev.min() >= 1 - lam - 1e-12 and ev.max() <= 1 + 1e-12
        # trace(Sigma) = 1 - |mu|^2 <= 1 for unit keys
        assert abs(np.trace(Sig) - (1 - mu @ mu)) < 1e-12


def test_identical_keys_leave_query_unchanged():
    d = _rand(1, 1, 15, 6, 3, seed=11)
    d["k"][:] = d["k"][:, :, :1]
    out = oracle.run("gla", **d, want_sigq=True)
    assert np.abs(out["sigq"]).max() < 1e-14
    ref = oracle.run("gla", **d, lambda_in=np.zeros((1, 1, 15)))
    np.testing.assert_allclose(out["o"], ref["o"], atol=1e-13)


# --------------------------------------------------------------------------- GDN cases
def test_gdn_beta_zero_is_pure_decay():
    d = _rand(1, 1, 8, 4, 3, seed=12, backbone="gdn")
    d["beta"] = np.zeros_like(d["beta"])
    S0 = np.random.default_rng(0).standard_normal((1, 1, 4, 3))
    C0 = np.zeros((1, 1, 4, 4))
    m0 = np.zeros((1, 1, 4))
    out = oracle.run("gdn", **d, S0=S0, C0=C0, m0=m0, t0=0, lambda_in=np.zeros((1, 1, 8)))
    g = np.cumsum(d["log_alpha"][0, 0])
    np.testing.assert_allclose(out["S"][0, 0], np.exp(g[-1]) * S0[0, 0], rtol=1e-13)
    np.testing.assert_allclose(out["o"][0, 0], np.exp(g)[:, None] * (d["q"][0, 0] @ S0[0, 0]),
                               rtol=1e-12, atol=1e-14)


def test_gdn_unit_keys_alpha_beta_one_stores_value():
    d = _rand(1, 1, 10, 6, 4, seed=13, backbone="gdn")
    d["log_alpha"] = np.zeros_like(d["log_alpha"])
    d["beta"] = np.ones_like(d["beta"])
    d["q"] = d["k"].copy()
    out = oracle.run("gdn", **d, lambda_in=np.zeros((1, 1, 10)))
    np.testing.assert_allclose(out["o"][0, 0], d["v"][0, 0], atol=1e-12)


def test_gdn_residual_contracts_by_one_minus_beta():
    d = _rand(1, 1, 6, 5, 3, seed=14, backbone="gdn")
    d["log_alpha"] = np.zeros_like(d["log_alpha"])
    prev = np.zeros((5, 3))
    for T in range(1, 7):
        sub = {k: (v[:, :, :T] if k in ("q", "k", "v", "log_alpha", "beta") else v)
               for k, v in d.items()}
        S = oracle.run("gdn", **sub)["S"][0, 0]
        k, v, b = d["k"][0, 0, T - 1], d["v"][0, 0, T - 1], d["beta"][0, 0, T - 1]
        r_new = np.linalg.norm(S.T @ k - v)
        r_old = np.linalg.norm(prev.T @ k - v)
        assert abs(r_new - (1 - b) * r_old) < 1e-12
        prev = S


# --------------------------------------------------------------------------- algorithms
@pytest.mark.parametrize("backbone", ["gla", "gdn"])
@pytest.mark.parametrize("chunk", [4, 16])
def test_independent_chunk_algorithm_agrees(backbone, chunk):
    d = _rand(2, 2, 37, 8, 6, seed=15, backbone=backbone)   # ragged tail
    S0 = np.random.default_rng(1).standard_normal((2, 2, 8, 6)) * 0.1
    K0 = np.random.default_rng(2).standard_normal((2, 2, 30, 8))
    K0 /= np.linalg.norm(K0, axis=-1, keepdims=True)
    C0 = np.einsum("bhti,bhtj->bhij", K0, K0)
    m0 = K0.sum(axis=2)
    ref = oracle.run(backbone, **d, S0=S0, C0=C0, m0=m0, t0=30)
    got = ccq_chunked(backbone, d["q"], d["k"], d["v"], d["log_alpha"], d["w_lambda"],
                      d["b_lambda"], beta=d["beta"], S0=S0, C0=C0, m0=m0, t0=30, chunk=chunk)
    for key in ("o", "lambda", "S", "C", "m"):
        np.testing.assert_allclose(got[key], ref[key], rtol=1e-10, atol=1e-11, err_msg=key)


@pytest.mark.parametrize("backbone", ["gla", "gdn"])
def test_state_split_invariance(backbone):
    d = _rand(1, 2, 30, 6, 5, seed=16, backbone=backbone)
    full = oracle.run(backbone, **d)
    tok = ("q", "k", "v", "log_alpha", "beta")
    a = oracle.run(backbone, **{k: (v[:, :, :11] if k in tok else v) for k, v in d.items()})
    b = oracle.run(backbone, **{k: (v[:, :, 11:] if k in tok else v) for k, v in d.items()},
                   S0=a["S"], C0=a["C"], m0=a["m"], t0=11)
    np.testing.assert_allclose(np.concatenate([a["o"], b["o"]], axis=2), full["o"], atol=1e-13)
    for key in ("S", "C", "m"):
        np.testing.assert_allclose(b[key], full[key], atol=1e-12)


def test_thread_count_does_not_change_bits():
    d = _rand(2, 3, 20, 6, 5, seed=17)
    a = oracle.run("gla", **d, nthreads=1)
    b = oracle.run("gla", **d, nthreads=5)
    for key in ("o", "lambda", "S", "C", "m"):
        np.testing.assert_array_equal(a[key], b[key])


def test_l2norm_switch_normalises_q_and_k():
    d = _rand(1, 2, 9, 5, 3, unit=False, seed=18)
    got = oracle.run("gla", **d, l2norm=True)
    dd = dict(d)
    for key in ("q", "k"):
        dd[key] = d[key] / np.sqrt((d[key] ** 2).sum(-1, keepdims=True) + 1e-6)
    ref = oracle.run("gla", **dd)
    np.testing.assert_allclose(got["o"], ref["o"], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(got["C"], ref["C"], rtol=1e-13, atol=1e-14)


def test_rejects_bad_arguments():
    d = _rand(1, 1, 3, 2, 2, seed=19)
    with pytest.raises(ValueError):
        oracle.run("gla", **d, t0=5)          # t0 without a carried state
    with pytest.raises(ValueError):
        oracle.run("gdn", **{**d, "beta": None})


# ----------------------------------------------------------------- backward oracle
def _bwd_case(seed, B=1, H=2, T=9, dk=5, dv=4, state=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, T, dk))
    k = rng.standard_normal((B, H, T, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, T, dv))
    la = -np.abs(rng.standard_normal((B, H, T, dk))) / 8
    w = rng.standard_normal((H, dk)) / np.sqrt(dk)
    b = rng.standard_normal(H) * 0.1
    S0 = rng.standard_normal((B, H, dk, dv)) * 0.3 if state else None
    K0 = rng.standard_normal((B, H, 7, dk))
    C0 = np.einsum("bhti,bhtj->bhij", K0, K0) if state else None
    m0 = K0.sum(2) if state else None
    return q, k, v, la, w, b, S0, C0, m0, (7 if state else 0)


def test_backward_oracle_forward_equals_the_c_oracle():
    """The autograd forward is an independent implementation of the same
    recurrence: it must reproduce the C oracle's outputs and final state."""
    import torch
    from oracle.backward import forward_torch
    q, k, v, la, w, b, S0, C0, m0, t0 = _bwd_case(1)
    ref = oracle.run("gla", q, k, v, la, w, b, S0=S0, C0=C0, m0=m0, t0=t0)
    for h in range(2):
        T = lambda x: torch.as_tensor(x)  # noqa: E731
        o, S, C, m = forward_torch(T(q[0, h]), T(k[0, h]), T(v[0, h]), T(la[0, h]), T(w[h]),
                                   T(b[h]), None, T(S0[0, h]), T(C0[0, h]), T(m0[0, h]), t0)
        np.testing.assert_allclose(o.numpy(), ref["o"][0, h], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(S.numpy(), ref["S"][0, h], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(C.numpy(), ref["C"][0, h], rtol=1e-12, atol=1e-12)


def test_backward_oracle_matches_finite_differences():
    import torch
    from oracle.backward import forward_torch
    q, k, v, la, w, b, S0, C0, m0, t0 = _bwd_case(2, T=3, dk=3, dv=2)
    T = lambda x: torch.as_tensor(x[0, 0]).clone().requires_grad_()  # noqa: E731
    args = [T(q), T(k), T(v), T(la), torch.as_tensor(w[0]).clone().requires_grad_(),
            torch.as_tensor(b[0]).clone().requires_grad_()]
    st = [T(S0), T(C0), T(m0)]

    def f(*xs):
        o, S, C, m = forward_torch(*xs[:6], None, *xs[6:], t0)
        return o.sum() + (S * 0.3).sum() + (C * 0.1).sum() + m.sum()

    assert torch.autograd.gradcheck(f, tuple(args + st), eps=1e-6, atol=1e-7, rtol=1e-5)


def test_backward_oracle_plain_read_closed_forms():
    """lambda = 0: o_t = S_t^T q_t, so dq_t = S_t do_t; one token from a zero
    state: o = v (k . q), so dv = do (k . q) and dk = q (v . do)."""
    from oracle.backward import gla_backward
    q, k, v, la, w, b, S0, C0, m0, t0 = _bwd_case(3, state=False)
    do = np.random.default_rng(4).standard_normal(v.shape)
    lin = np.zeros(q.shape[:3])
    g = gla_backward(q, k, v, la, w, b, do, lambda_in=lin)
    fwd = oracle.run("gla", q, k, v, la, lambda_in=lin)
    # S_t from the forward of each prefix
    for t in range(q.shape[2]):
        st = oracle.run("gla", q[:, :, :t + 1], k[:, :, :t + 1], v[:, :, :t + 1],
                        la[:, :, :t + 1], lambda_in=lin[:, :, :t + 1])["S"]
        np.testing.assert_allclose(g["dq"][:, :, t], np.einsum("bhij,bhj->bhi", st, do[:, :, t]),
                                   rtol=1e-10, atol=1e-12)
    assert fwd["o"].shape == do.shape
    g1 = gla_backward(q[:, :, :1], k[:, :, :1], v[:, :, :1], la[:, :, :1], w, b, do[:, :, :1],
                      lambda_in=lin[:, :, :1])
    kq = (k[:, :, 0] * q[:, :, 0]).sum(-1)
    np.testing.assert_allclose(g1["dv"][:, :, 0], do[:, :, 0] * kq[..., None], rtol=1e-12)
    vd = (v[:, :, 0] * do[:, :, 0]).sum(-1)
    np.testing.assert_allclose(g1["dk"][:, :, 0], q[:, :, 0] * vd[..., None], rtol=1e-12)
    assert np.all(g1["dw_lambda"] == 0) and np.all(g1["db_lambda"] == 0)
