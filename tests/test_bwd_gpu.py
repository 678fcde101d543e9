"""GPU parity of the CCQ-GLA gradients (ccq_gla_bwd through the C ABI)
against the fp64 autograd oracle (oracle/backward.py) on the same seeded
inputs.

Tolerance: the kernels accumulate in fp32 (C, S and their adjoints over every
token, the decay gradient as a reverse running sum), so each gradient is
compared by its largest error relative to its largest magnitude: 2e-4 for
the short cases, 1e-3 at T = 4096 (a few thousand fp32 additions in a row)."""
import numpy as np
import pytest
import torch

import ccq_read_side_gb300 as ccq
from ccq_read_side_gb300.workloads import WORKLOADS, Workload, make_inputs
from oracle.backward import gla_backward

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "log_alpha", "w_lambda", "b_lambda")


def _rel(got, ref):
    """Largest error over the largest reference magnitude, floored at 1e-3: a
    gradient that is exactly zero (the decay gradient of a first token read
    from a zero state) is compared with an absolute bound instead; the
    kernel's value there is the fp32 rounding of two equal terms' difference."""
    got = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else got
    scale = max(np.abs(ref).max(), 1e-3)
    return np.abs(got - ref).max() / scale


def _case(dk, dv, T, B=1, H=2, seed=11, state=False, lam=False, up=False, keys="iso"):
    w = Workload("bwd", "gla", "f32", B, H, T, dk, dv, 64, seed, keys)
    inp = make_inputs(w)
    rng = np.random.default_rng(seed + 100)
    f32 = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float32))  # noqa: E731
    extra = {"grad_o": f32(rng.standard_normal((B, H, T, dv)))}
    if lam:
        extra["lambda_in"] = f32(rng.uniform(0.0, 1.0, (B, H, T)))
    if state:
        K0 = rng.standard_normal((B, H, 50, dk)) / np.sqrt(dk)
        extra["S0"] = f32(rng.standard_normal((B, H, dk, dv)) * 0.2)
        extra["C0"] = f32(np.einsum("bhti,bhtj->bhij", K0, K0))
        extra["m0"] = f32(K0.sum(2))
        extra["t0"] = 50
    if up:
        extra["grad_S"] = f32(rng.standard_normal((B, H, dk, dv)) * 0.1)
        extra["grad_C"] = f32(rng.standard_normal((B, H, dk, dk)) * 0.01)
        extra["grad_m"] = f32(rng.standard_normal((B, H, dk)) * 0.1)
    return inp, extra


def _run(inp, extra, want_state_grads=False):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in {**inp, **extra}.items()}
    g = ccq.gla_bwd(d["q"], d["k"], d["v"], d["log_alpha"], d["w_lambda"], d["b_lambda"],
                    d["grad_o"], lambda_in=d.get("lambda_in"), S0=d.get("S0"), C0=d.get("C0"),
                    m0=d.get("m0"), t0=d.get("t0", 0), grad_S=d.get("grad_S"),
                    grad_C=d.get("grad_C"), grad_m=d.get("grad_m"),
                    want_state_grads=want_state_grads)
    torch.cuda.synchronize()
    return g


def _oracle(inp, extra):
    n = lambda key: None if extra.get(key) is None else extra[key].double().numpy()  # noqa: E731
    return gla_backward(inp["q"].double().numpy(), inp["k"].double().numpy(),
                        inp["v"].double().numpy(), inp["log_alpha"].double().numpy(),
                        inp["w_lambda"].double().numpy(), inp["b_lambda"].double().numpy(),
                        extra["grad_o"].double().numpy(), lambda_in=n("lambda_in"), S0=n("S0"),
                        C0=n("C0"), m0=n("m0"), t0=extra.get("t0", 0), dS=n("grad_S"),
                        dC=n("grad_C"), dm=n("grad_m"))


def _compare(g, ref, tol, state=False):
    for name in NAMES:
        err = _rel(g[name], ref["d" + name])
        assert err <= tol, (name, err)
    if state:
        assert _rel(g["S0"], ref["dS0"]) <= tol
        sym = 0.5 * (ref["dC0"] + np.swapaxes(ref["dC0"], -1, -2))
        assert _rel(g["C0"], sym) <= tol
        assert _rel(g["m0"], ref["dm0"]) <= tol


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("T", [1, 45])
def test_gradients_match_oracle(dk, dv, T):
    inp, extra = _case(dk, dv, T)
    _compare(_run(inp, extra), _oracle(inp, extra), 2e-4)


@pytest.mark.parametrize("dk,dv", [(64, 128), (128, 128)])
def test_gradients_with_carried_state_and_state_gradients(dk, dv):
    inp, extra = _case(dk, dv, 37, state=True, up=True, seed=5)
    _compare(_run(inp, extra, True), _oracle(inp, extra), 2e-4, state=True)


def test_given_lambda_has_no_gate_gradient():
    inp, extra = _case(128, 64, 30, lam=True, seed=6)
    g = _run(inp, extra)
    _compare(g, _oracle(inp, extra), 2e-4)
    assert torch.count_nonzero(g["w_lambda"]).item() == 0
    assert torch.count_nonzero(g["b_lambda"]).item() == 0


def test_no_tokens_passes_the_state_gradients_through():
    inp, extra = _case(64, 64, 0, state=True, up=True, seed=7)
    g = _run(inp, extra, True)
    np.testing.assert_array_equal(g["S0"].cpu().numpy(), extra["grad_S"].numpy())
    gc = extra["grad_C"].double().numpy()
    np.testing.assert_allclose(g["C0"].double().cpu().numpy(),
                               0.5 * (gc + np.swapaxes(gc, -1, -2)), rtol=1e-6, atol=1e-9)
    np.testing.assert_array_equal(g["m0"].cpu().numpy(), extra["grad_m"].numpy())


def test_needle_keys_many_chunks():
    inp, extra = _case(128, 128, 301, B=2, H=1, seed=8, keys="aniso_needle")
    _compare(_run(inp, extra), _oracle(inp, extra), 2e-4)


def test_full_size_sampled_heads():
    """B4 H16 T4096 dk = dv = 128 (the benchmark's shape) in one call, two
    (b, h) heads checked against the oracle run on those heads alone."""
    w = WORKLOADS[2]
    inp = make_inputs(Workload("bwd_full", "gla", "f32", w.B, w.H, w.T, 128, 128, 64, w.seed,
                               w.keys))
    rng = np.random.default_rng(99)
    go = torch.from_numpy(rng.standard_normal((w.B, w.H, w.T, 128)).astype(np.float32))
    g = _run(inp, {"grad_o": go})
    for b, h in ((0, 0), (3, 11)):
        one = {key: inp[key][b:b + 1, h:h + 1] for key in ("q", "k", "v", "log_alpha")}
        one["w_lambda"] = inp["w_lambda"][h:h + 1]
        one["b_lambda"] = inp["b_lambda"][h:h + 1]
        ref = _oracle(one, {"grad_o": go[b:b + 1, h:h + 1]})
        for name in NAMES:
            assert _rel(g[name][b:b + 1, h:h + 1], ref["d" + name]) <= 1e-3, (b, h, name)


def test_workspace_too_small_is_rejected():
    inp, extra = _case(64, 64, 16)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in {**inp, **extra}.items()}
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(ccq.CcqError) as e:
        ccq.gla_bwd(d["q"], d["k"], d["v"], d["log_alpha"], d["w_lambda"], d["b_lambda"],
                    d["grad_o"], workspace=small)
    assert e.value.code == 1


@pytest.mark.parametrize("T", [8, 9, 16])
def test_chunk_boundaries(T):
    """T at a chunk multiple and one past it (chunks of 8 tokens)."""
    inp, extra = _case(128, 64, T, seed=40 + T, state=True, up=True)
    _compare(_run(inp, extra, True), _oracle(inp, extra), 2e-4, state=True)


def test_many_heads_given_lambda_with_state():
    """B3 H5: fifteen CTA pairs; a given lambda, carried state and state
    gradients together, d_k = 64, d_v = 128."""
    inp, extra = _case(64, 128, 23, B=3, H=5, seed=50, state=True, lam=True, up=True)
    _compare(_run(inp, extra, True), _oracle(inp, extra), 2e-4, state=True)


def test_strong_decay():
    """log alpha about -5 per token and channel: the decay products across a
    chunk underflow; the sweeps only ever form exp of non-positive
    differences, so nothing divides by a vanishing product."""
    inp, extra = _case(128, 128, 40, seed=60)
    inp["log_alpha"] = (inp["log_alpha"] * 80.0).clamp(min=-12.0)
    assert inp["log_alpha"].min().item() < -8.0
    _compare(_run(inp, extra), _oracle(inp, extra), 2e-4)
