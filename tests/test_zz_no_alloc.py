"""The no-allocation gradient entry point (ccq_gla_bwd_noalloc, workspace in
a fixed array inside the library) against the workspace entry point
(ccq_gla_bwd), both called through the C ABI.  Collected last on purpose: it
must also pass after every other test has used the library in this process."""
import ctypes

import numpy as np
import pytest
import torch

import ccq_read_side_gb300 as ccq
from ccq_read_side_gb300 import build as ccq_build
from ccq_read_side_gb300.workloads import Workload, make_inputs

SCRATCH_BYTES = 16 << 20  # CCQ_GLA_BWD_NOALLOC_SCRATCH_BYTES
TOL = 2e-4                # the gradient parity tolerance of the short backward cases
FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: the call is rejected first


@pytest.fixture(scope="module")
def lib():
    ccq_build.build()
    return ccq.library()


def _call(lib, a):
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.ccq_gla_bwd_noalloc(
        P(a["q"]), P(a["k"]), P(a["v"]), P(a["log_alpha"]), P(a["w_lambda"]), P(a["b_lambda"]),
        P(a.get("lambda_in")), P(a.get("S0")), P(a.get("C0")), P(a.get("m0")), a.get("t0", 0),
        P(a["grad_o"]), P(a.get("grad_S")), P(a.get("grad_C")), P(a.get("grad_m")),
        P(a["out_q"]), P(a["out_k"]), P(a["out_v"]), P(a["out_log_alpha"]), P(a["out_w_lambda"]),
        P(a["out_b_lambda"]), P(a.get("out_S0")), P(a.get("out_C0")), P(a.get("out_m0")),
        a["B"], a["H"], a["T"], a["dk"], a["dv"], 0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_sizes_beyond_the_scratch_are_rejected(lib):
    # B1 H16 T4096 at dk = 128 needs about 25 MB: rejected before any CUDA call
    assert lib.ccq_gla_bwd_workspace_bytes(1, 16, 4096, 128, 128) > SCRATCH_BYTES
    args = [FAKE] * 10 + [0] + [FAKE] * 13 + [1, 16, 4096, 128, 128, 0, None]
    assert lib.ccq_gla_bwd_noalloc(*args) == 6
    assert "TOO_LARGE" in ccq.status_string(6)
    # an empty batch needs no pointers and makes no CUDA call
    empty = [None] * 10 + [0] + [None] * 13 + [0, 16, 4096, 128, 128, 0, None]
    assert lib.ccq_gla_bwd_noalloc(*empty) == 0


def _inputs(dk, dv, T, B, H, seed, state):
    inp = make_inputs(Workload("noalloc", "gla", "f32", B, H, T, dk, dv, 64, seed, "iso"))
    rng = np.random.default_rng(seed + 7)
    f32 = lambda x: torch.from_numpy(np.asarray(x, dtype=np.float32)).cuda()  # noqa: E731
    a = {key: inp[key].cuda() for key in ("q", "k", "v", "log_alpha", "w_lambda", "b_lambda")}
    a["grad_o"] = f32(rng.standard_normal((B, H, T, dv)))
    if state:
        K0 = rng.standard_normal((B, H, 40, dk)) / np.sqrt(dk)
        a["S0"] = f32(rng.standard_normal((B, H, dk, dv)) * 0.2)
        a["C0"] = f32(np.einsum("bhti,bhtj->bhij", K0, K0))
        a["m0"] = f32(K0.sum(2))
        a["t0"] = 40
        a["grad_S"] = f32(rng.standard_normal((B, H, dk, dv)) * 0.1)
        a["grad_C"] = f32(rng.standard_normal((B, H, dk, dk)) * 0.01)
        a["grad_m"] = f32(rng.standard_normal((B, H, dk)) * 0.1)
    a.update(B=B, H=H, T=T, dk=dk, dv=dv)
    return a


def _rel(got, ref):
    return ((got.double() - ref.double()).abs().max() / ref.double().abs().max().clamp_min(1e-3)).item()


@pytest.mark.gpu
def test_matches_the_workspace_entry_point_on_two_calls_in_a_row(lib):
    cases = [(128, 128, 4096, 1, 2, 31, False),   # 12.7 MB of the 16 MiB array
             (64, 128, 777, 2, 3, 32, True)]      # carried state and state gradients
    for dk, dv, T, B, H, seed, state in cases:
        assert lib.ccq_gla_bwd_workspace_bytes(B, H, T, dk, dv) <= SCRATCH_BYTES
        a = _inputs(dk, dv, T, B, H, seed, state)
        ref = ccq.gla_bwd(a["q"], a["k"], a["v"], a["log_alpha"], a["w_lambda"], a["b_lambda"],
                          a["grad_o"], S0=a.get("S0"), C0=a.get("C0"), m0=a.get("m0"),
                          t0=a.get("t0", 0), grad_S=a.get("grad_S"), grad_C=a.get("grad_C"),
                          grad_m=a.get("grad_m"), want_state_grads=state)
        for name, t in ref.items():
            a["out_" + name] = torch.full_like(t, float("nan"))
        assert _call(lib, a) == 0
        torch.cuda.synchronize()
        for name, t in ref.items():
            got = a["out_" + name]
            assert torch.isfinite(got).all(), name
            assert _rel(got, t) <= TOL, (dk, dv, T, name, _rel(got, t))
