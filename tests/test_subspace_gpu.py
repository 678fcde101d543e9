"""GPU checks of the key-covariance diagnostics (top-k eigenspace of Sigma_T
from a final state, captured energy of keys) against numpy.linalg.eigh in
fp64 on the same C, m, n."""
import numpy as np
import pytest
import torch

import ccq_read_side_gb300 as ccq
from ccq_read_side_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def _state_with_gap(rng, BH, dk, n, r=16, boost=10.0):
    """C, m of n unit keys concentrated in a random rank-r subspace."""
    C = np.empty((BH, dk, dk))
    m = np.empty((BH, dk))
    for b in range(BH):
        Ub, _ = np.linalg.qr(rng.standard_normal((dk, r)))
        K = np.sqrt(boost) * rng.standard_normal((n, r)) @ Ub.T + rng.standard_normal((n, dk))
        K /= np.linalg.norm(K, axis=1, keepdims=True)
        C[b] = K.T @ K
        m[b] = K.sum(0)
    return C.astype(np.float32), m.astype(np.float32)


def _reference(C, m, n, k):
    """Top-k eigenpairs of Sigma = C/n - mu mu^T (fp64, from the fp32 inputs)."""
    C = C.astype(np.float64)
    mu = m.astype(np.float64) / n
    Sig = C / n - mu[:, :, None] * mu[:, None, :]
    w, V = np.linalg.eigh(Sig)
    return w[:, ::-1][:, :k], V[:, :, ::-1][:, :, :k]


@pytest.mark.parametrize("dk,k", [(128, 16), (64, 8), (128, 1)])
def test_top_subspace_matches_eigh(dk, k):
    rng = np.random.default_rng(dk + k)
    BH, n = 6, 3000
    C, m = _state_with_gap(rng, BH, dk, n, r=k)  # the gap sits after the k-th eigenvalue
    U, ritz = ccq.sigma_subspace(torch.from_numpy(C).cuda(), torch.from_numpy(m).cuda(), n, k=k,
                                 iters=100)
    torch.cuda.synchronize()
    U, ritz = U.double().cpu().numpy(), ritz.double().cpu().numpy()
    w_ref, V_ref = _reference(C, m, n, k)
    # orthonormal basis of the same subspace, Ritz values = top eigenvalues
    eye = np.eye(k)
    assert np.abs(np.einsum("bia,bic->bac", U, U) - eye).max() < 1e-4
    P = np.einsum("bia,bja->bij", U, U)
    P_ref = np.einsum("bia,bja->bij", V_ref, V_ref)
    assert np.linalg.norm(P - P_ref, axis=(1, 2)).max() < 1e-3
    np.testing.assert_allclose(ritz, w_ref, rtol=1e-4, atol=1e-7)
    assert (np.diff(ritz, axis=1) <= 1e-7).all()  # descending


def test_alignment_matches_projection():
    rng = np.random.default_rng(7)
    BH, dk, k, n, nx = 4, 128, 16, 2000, 37
    C, m = _state_with_gap(rng, BH, dk, n)
    Ug, _ = ccq.sigma_subspace(torch.from_numpy(C).cuda(), torch.from_numpy(m).cuda(), n, k=k)
    X = rng.standard_normal((BH, nx, dk)).astype(np.float32)
    X[0, 3] = 0.0  # a zero key captures nothing
    got = ccq.subspace_alignment(Ug, torch.from_numpy(X).cuda())
    torch.cuda.synchronize()
    _, V_ref = _reference(C, m, n, k)
    proj = np.einsum("bia,bji->bja", V_ref, X.astype(np.float64))
    xx = (X.astype(np.float64) ** 2).sum(-1)
    ref = np.where(xx > 0, (proj ** 2).sum(-1) / np.where(xx > 0, xx, 1), 0.0)
    np.testing.assert_allclose(got.double().cpu().numpy(), ref, atol=2e-4)
    assert got[0, 3].item() == 0.0


def test_needle_lies_off_the_dominant_subspace():
    """The article's premise on the benchmark workload's key geometry: after
    the forward, the needle key captures far less energy in the top-16
    eigenspace of Sigma_T than an ordinary key does."""
    w = WORKLOADS[2]
    inp = make_inputs(w, T=1024, B=1, H=4)
    d = {k_: (v.cuda() if isinstance(v, torch.Tensor) else v) for k_, v in inp.items()}
    _, st = ccq.gla_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["w_lambda"], d["b_lambda"])
    U, _ = ccq.sigma_subspace(st["C"], st["m"], 1024, k=16, iters=100)
    align = ccq.subspace_alignment(U, d["k"].contiguous())  # every key of every head
    torch.cuda.synchronize()
    a = align.double().cpu().numpy()
    pos = np.asarray(inp["needle_pos"]).reshape(1, -1)
    for h in range(4):
        p = int(pos[0, h]) if pos.shape[1] > h else int(pos[0, 0])
        others = np.delete(a[0, h], p)
        assert a[0, h, p] < 0.2 * np.median(others), (h, a[0, h, p], np.median(others))
    # and the same numbers as numpy on the GPU's own final state
    _, V_ref = _reference(st["C"].cpu().numpy().reshape(4, 128, 128),
                          st["m"].cpu().numpy().reshape(4, 128), 1024, 16)
    K = inp["k"].double().numpy()[0]
    proj = np.einsum("hia,hti->hta", V_ref, K)
    ref = (proj ** 2).sum(-1) / (K ** 2).sum(-1)
    np.testing.assert_allclose(a[0], ref, atol=2e-3)


def test_bad_sizes_are_rejected():
    C = torch.zeros((1, 128, 128), device="cuda")
    m = torch.zeros((1, 128), device="cuda")
    with pytest.raises(ccq.CcqError) as e:
        ccq.sigma_subspace(C, m, 10, k=33)
    assert e.value.code == 2
    with pytest.raises(ccq.CcqError) as e:
        ccq.sigma_subspace(C, m, 0, k=4)
    assert e.value.code == 1
