"""GPU parity: the CUDA path against the fp64 oracle on identical seeded inputs.

Small cases span several chunks and a ragged tail; the five workloads run at
their full sizes in the same launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import ccq_read_side_gb300 as ccq
import oracle
from ccq_read_side_gb300.workloads import WORKLOADS, Workload, make_inputs
from parity import check, check_all, np64, run_both, to_dev

pytestmark = pytest.mark.gpu


def _small(backbone, dtype, dk, dv, T, B=2, H=3, seed=0, keys="iso"):
    w = Workload("small", backbone, dtype, B, H, T, dk, dv, 64, seed, keys)
    return make_inputs(w)


# ----------------------------------------------------------------- full workloads
def test_workload0_gla_f32():
    w = WORKLOADS[0]
    inp = make_inputs(w)
    gpu, ref = run_both("gla", inp, w.dtype)
    check_all(gpu, ref, w.dtype, w.name)


@pytest.mark.parametrize("idx", [1, 2])
def test_workload_gla_bf16_full(idx):
    w = WORKLOADS[idx]
    inp = make_inputs(w)
    gpu, ref = run_both("gla", inp, w.dtype)
    check_all(gpu, ref, w.dtype, w.name)


def test_workload3_length_extrapolation_from_carried_state():
    """4096-token prefix -> fp32 state (from the oracle) -> 20480-token
    continuation on the GPU, compared with the oracle's continuation from the
    same fp32 state.  A second run chains the GPU's own prefix state."""
    w = WORKLOADS[3]
    inp = make_inputs(w)
    P = w.prefix
    pre = {k: (v[:, :, :P] if isinstance(v, torch.Tensor) and v.dim() >= 3 else v)
           for k, v in inp.items()}
    cont = {k: (v[:, :, P:].contiguous() if isinstance(v, torch.Tensor) and v.dim() >= 3 else v)
            for k, v in inp.items()}
    st = oracle.run("gla", pre["q"], pre["k"], pre["v"], pre["log_alpha"], pre["w_lambda"],
                    pre["b_lambda"])
    S0, C0, m0 = (st[k].astype(np.float32) for k in ("S", "C", "m"))
    gpu, ref = run_both("gla", cont, w.dtype, S0=S0, C0=C0, m0=m0, t0=P)
    check_all(gpu, ref, w.dtype, w.name)

    # chained: the GPU's own prefix state feeds the continuation
    d = to_dev(pre)
    _, gst = ccq.gla_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["w_lambda"], d["b_lambda"])
    dc = to_dev(cont)
    o2, _ = ccq.gla_fwd(dc["q"], dc["k"], dc["v"], dc["log_alpha"], dc["w_lambda"],
                        dc["b_lambda"], S0=gst["S"], C0=gst["C"], m0=gst["m"], t0=P)
    torch.cuda.synchronize()
    check(np64(o2), ref["o"], w.dtype, w.name + " chained")


def test_workload4_gdn_bf16_full():
    w = WORKLOADS[4]
    inp = make_inputs(w)
    gpu, ref = run_both("gdn", inp, w.dtype)
    check_all(gpu, ref, w.dtype, w.name)


# ----------------------------------------------------------------- shapes and tails
@pytest.mark.parametrize("backbone", ["gla", "gdn"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("T", [1, 17, 64, 130])
def test_small_shapes(backbone, dtype, dk, dv, T):
    inp = _small(backbone, dtype, dk, dv, T, seed=T + dk + dv)
    gpu, ref = run_both(backbone, inp, dtype)
    check_all(gpu, ref, dtype, f"{backbone}/{dtype}/{dk}x{dv}/T{T}")


@pytest.mark.parametrize("backbone", ["gla", "gdn"])
@pytest.mark.parametrize("T", [63, 65, 127, 129, 191, 200])
def test_ragged_tails_bf16_d128(backbone, T):
    inp = _small(backbone, "bf16", 128, 128, T, B=1, H=2, seed=100 + T)
    gpu, ref = run_both(backbone, inp, "bf16")
    check_all(gpu, ref, "bf16", f"{backbone}/T{T}")


@pytest.mark.parametrize("backbone", ["gla", "gdn"])
def test_zero_length_passes_state_through(backbone):
    inp = _small(backbone, "bf16", 128, 128, 0, B=1, H=2)
    rng = np.random.default_rng(0)
    S0 = rng.standard_normal((1, 2, 128, 128)).astype(np.float32)
    C0 = rng.standard_normal((1, 2, 128, 128)).astype(np.float32)
    m0 = rng.standard_normal((1, 2, 128)).astype(np.float32)
    gpu, _ = run_both(backbone, inp, "bf16", S0=S0, C0=C0, m0=m0, t0=5)
    np.testing.assert_array_equal(gpu["S"], S0)
    np.testing.assert_array_equal(gpu["C"], C0)
    np.testing.assert_array_equal(gpu["m"], m0)


# ----------------------------------------------------------------- lambda modes
@pytest.mark.parametrize("backbone", ["gla", "gdn"])
@pytest.mark.parametrize("lam", [0.0, 0.1])
def test_given_lambda(backbone, lam):
    inp = _small(backbone, "bf16", 128, 128, 150, B=1, H=2, seed=7)
    lin = np.full((1, 2, 150), lam, np.float32)
    gpu, ref = run_both(backbone, inp, "bf16", lambda_in=lin)
    check_all(gpu, ref, "bf16", f"lambda={lam}")
    np.testing.assert_array_equal(gpu["lambda"], lin)


def test_l2norm_flag_on_raw_inputs():
    inp = _small("gla", "bf16", 128, 128, 100, B=1, H=2, seed=8)
    g = torch.Generator().manual_seed(0)
    inp["q"] = (torch.randn(inp["q"].shape, generator=g) * 3).to(torch.bfloat16)
    inp["k"] = (torch.randn(inp["k"].shape, generator=g) * 3).to(torch.bfloat16)
    gpu, ref = run_both("gla", inp, "bf16", l2norm=True)
    check_all(gpu, ref, "bf16", "l2norm")


# ----------------------------------------------------------------- state
@pytest.mark.parametrize("backbone", ["gla", "gdn"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_state_chaining_matches_one_pass(backbone, dtype):
    inp = _small(backbone, dtype, 128, 128, 300, B=1, H=2, seed=9)
    d = to_dev(inp)
    fn = ccq.gla_fwd if backbone == "gla" else ccq.gdn_fwd

    def call(sl, **kw):
        args = [d["q"][:, :, sl].contiguous(), d["k"][:, :, sl].contiguous(),
                d["v"][:, :, sl].contiguous(), d["log_alpha"][:, :, sl].contiguous()]
        if backbone == "gdn":
            args.append(d["beta"][:, :, sl].contiguous())
        return fn(*args, d["w_lambda"], d["b_lambda"], **kw)

    o1, s1 = call(slice(0, 137))
    o2, s2 = call(slice(137, 300), S0=s1["S"], C0=s1["C"], m0=s1["m"], t0=137)
    torch.cuda.synchronize()
    ref = oracle.run(backbone, inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["w_lambda"],
                     inp["b_lambda"], beta=inp.get("beta"))
    check(np.concatenate([np64(o1), np64(o2)], axis=2), ref["o"], dtype, "chained o")
    for key in ("S", "C", "m"):
        check(np64(s2[key]), ref[key], dtype, "chained " + key, per_head=False)


def test_state_out_may_alias_state_in():
    inp = _small("gla", "bf16", 128, 128, 70, B=1, H=2, seed=10)
    d = to_dev(inp)
    rng = np.random.default_rng(1)
    K0 = rng.standard_normal((1, 2, 40, 128))
    K0 /= np.linalg.norm(K0, axis=-1, keepdims=True)
    C0 = np.einsum("bhti,bhtj->bhij", K0, K0).astype(np.float32)
    m0 = K0.sum(2).astype(np.float32)
    S0 = (rng.standard_normal((1, 2, 128, 128)) * 0.1).astype(np.float32)
    S = torch.from_numpy(S0).cuda()
    C = torch.from_numpy(C0).cuda()
    m = torch.from_numpy(m0).cuda()
    lib = ccq.library()
    o = torch.empty_like(d["v"])
    p = lambda t: None if t is None else __import__("ctypes").c_void_p(t.data_ptr())  # noqa
    rc = lib.ccq_gla_fwd(p(d["q"]), p(d["k"]), p(d["v"]), p(d["log_alpha"]), p(d["w_lambda"]),
                         p(d["b_lambda"]), None, None, p(o), p(S), p(C), p(m), 40, p(S), p(C),
                         p(m), 1, 2, 70, 128, 128, 0, 1, 0,
                         __import__("ctypes").c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    ref = oracle.run("gla", inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["w_lambda"],
                     inp["b_lambda"], S0=S0, C0=C0, m0=m0, t0=40)
    check(np64(o), ref["o"], "bf16", "aliased o")
    check(np64(S), ref["S"], "bf16", "aliased S", per_head=False)
    check(np64(C), ref["C"], "bf16", "aliased C", per_head=False)


# ----------------------------------------------------------------- invariances
def test_fp32_path_chunk_hint_invariance():
    inp = _small("gla", "f32", 64, 64, 90, B=1, H=2, seed=11)
    ref = None
    for chunk in (1, 5, 16):
        gpu, r = run_both("gla", inp, "f32", chunk=chunk)
        ref = r
        check_all(gpu, ref, "f32", f"chunk={chunk}")


def test_heads_are_independent():
    inp = _small("gla", "bf16", 128, 128, 96, B=2, H=4, seed=12)
    d = to_dev(inp)
    o, _ = ccq.gla_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["w_lambda"], d["b_lambda"])
    perm = torch.tensor([2, 0, 3, 1])
    dp = {k: (v[:, perm].contiguous() if isinstance(v, torch.Tensor) and v.dim() >= 3 else v)
          for k, v in d.items()}
    dp["w_lambda"] = d["w_lambda"][perm].contiguous()
    dp["b_lambda"] = d["b_lambda"][perm].contiguous()
    op, _ = ccq.gla_fwd(dp["q"], dp["k"], dp["v"], dp["log_alpha"], dp["w_lambda"],
                        dp["b_lambda"])
    torch.cuda.synchronize()
    assert torch.equal(op, o[:, perm])


def test_fp32_path_flag_on_bf16_matches_oracle():
    inp = _small("gla", "bf16", 128, 128, 200, B=1, H=2, seed=13)
    gpu, ref = run_both("gla", inp, "bf16", flags=ccq.FLAG_FP32_PATH)
    check_all(gpu, ref, "bf16", "fp32 path")


# ----------------------------------------------------------------- plain GLA baseline
@pytest.mark.parametrize("T", [64, 200, 4096])
def test_plain_gla_baseline_is_the_lambda_zero_read(T):
    """CCQ_FLAG_PLAIN_GLA computes the backbone's own read o_t = S_t^T q_t:
    the oracle with lambda = 0 gives it exactly (q_clean = q)."""
    inp = _small("gla", "bf16", 128, 128, T, B=1, H=4, seed=30 + T, keys="aniso")
    d = to_dev(inp)
    rng = np.random.default_rng(T)
    S0 = (rng.standard_normal((1, 4, 128, 128)) * 0.1).astype(np.float32)
    o, st = ccq.gla_fwd(d["q"], d["k"], d["v"], d["log_alpha"], flags=ccq.FLAG_PLAIN_GLA,
                        S0=torch.from_numpy(S0).cuda())
    torch.cuda.synchronize()
    assert ccq.last_device_status() == 0
    assert st["C"] is None and st["m"] is None
    lin = np.zeros((1, 4, T), np.float32)
    C0 = np.zeros((1, 4, 128, 128), np.float32)
    m0 = np.zeros((1, 4, 128), np.float32)
    ref = oracle.run("gla", inp["q"], inp["k"], inp["v"], inp["log_alpha"], lambda_in=lin,
                     S0=S0, C0=C0, m0=m0)
    check(np64(o), ref["o"], "bf16", f"plain T={T} o")
    check(np64(st["S"]), ref["S"], "bf16", f"plain T={T} S", per_head=False)


def test_plain_gla_flag_refuses_statistics_and_other_paths():
    inp = _small("gla", "bf16", 128, 128, 64, B=1, H=2, seed=3)
    d = to_dev(inp)
    with pytest.raises(ccq.CcqError) as e:  # lambda_out is a statistic of the CCQ read
        ccq.gla_fwd(d["q"], d["k"], d["v"], d["log_alpha"], flags=ccq.FLAG_PLAIN_GLA,
                    lambda_out=torch.empty((1, 2, 64), device="cuda"))
    assert e.value.code == 1
    inp32 = _small("gla", "f32", 64, 64, 64, B=1, H=2, seed=3)
    d32 = to_dev(inp32)
    with pytest.raises(ccq.CcqError) as e:  # tensor-core shapes only
        ccq.gla_fwd(d32["q"], d32["k"], d32["v"], d32["log_alpha"], flags=ccq.FLAG_PLAIN_GLA)
    assert e.value.code == 2
