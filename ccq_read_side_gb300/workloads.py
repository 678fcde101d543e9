"""Seeded synthetic inputs for the CCQ forward.

This module only draws random numbers and shapes them into the five
workloads the library is measured and checked on.  It holds none of the
method's arithmetic: it never forms a covariance, a gate, a decay product or
an output.  Both the fp64 oracle (via the tests) and the CUDA path read the
arrays it returns, so the two sides see bit-identical inputs.

Distributions follow the CCQ pages' setting (linear-attention heads with
L2-normalised keys, a learned per-head gate vector, GLA per-channel decay and
Gated DeltaNet scalar decay); the anisotropic key geometry with one needle
per sequence mirrors the "memory check-up" section of the 10100.com article
(needle keys lie off the top-16 covariance subspace of the keys).

Every array is generated in float64 with ``numpy.random.default_rng(seed)``
in the fixed order q, k, v, log_alpha, w_lambda, [beta], needle, then rounded
once (round-to-nearest-even, via float32) to the storage dtype.  The oracle
upcasts the stored values exactly, so rounding is not a source of mismatch.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np
import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "l2_normalise_rows"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    backbone: str          # "gla" or "gdn"
    dtype: str             # "f32" or "bf16"
    B: int
    H: int
    T: int                 # tokens computed and compared
    dk: int
    dv: int
    chunk: int
    seed: int
    keys: str              # "iso" or "aniso_needle"
    prefix: int = 0        # tokens of carried prefix state (length extrapolation)

    @property
    def head_tokens(self) -> int:
        return self.B * self.H * self.T


# The five measured/checked workloads.  Index i is the i-th configuration.
WORKLOADS = [
    Workload("gla_f32_b1h2t256d64", "gla", "f32", 1, 2, 256, 64, 64, 64, 0, "iso"),
    Workload("gla_bf16_b8h8t2048d128", "gla", "bf16", 8, 8, 2048, 128, 128, 64, 1, "iso"),
    Workload("gla_bf16_b4h16t4096d128_needle", "gla", "bf16", 4, 16, 4096, 128, 128, 64, 2,
             "aniso_needle"),
    Workload("gla_bf16_b1h16t20480d128_from4096", "gla", "bf16", 1, 16, 20480, 128, 128, 64, 3,
             "aniso_needle", prefix=4096),
    Workload("gdn_bf16_b2h16t8192d128", "gdn", "bf16", 2, 16, 8192, 128, 128, 64, 4, "iso"),
]


def l2_normalise_rows(x: np.ndarray) -> np.ndarray:
    """x / ||x|| along the last axis (input preparation, float64)."""
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True))


def _to_storage(x: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == "bf16":
        return t.to(torch.bfloat16)
    if dtype == "f32":
        return t
    raise ValueError(dtype)


def _iso_keys(rng, B, H, T, dk):
    return l2_normalise_rows(rng.standard_normal((B, H, T, dk)))


def _aniso_keys(rng, B, H, T, dk, rank=16, var_hi=10.0):
    """Per head: a random rank-16 orthonormal basis U (QR of a Gaussian);
    k = sqrt(var_hi) U z1 + (I - U U^T) z2, then L2-normalised.  One needle
    per sequence at a uniform position in [T/4, 3T/4) (same for all heads):
    its key is drawn from the complement (I - U U^T) z, normalised."""
    U = np.empty((H, dk, rank))
    for h in range(H):
        U[h], _ = np.linalg.qr(rng.standard_normal((dk, rank)))
    z1 = rng.standard_normal((B, H, T, rank))
    z2 = rng.standard_normal((B, H, T, dk))
    k = np.empty((B, H, T, dk))
    for h in range(H):
        Uh = U[h]
        lo = z2[:, h] - (z2[:, h] @ Uh) @ Uh.T
        k[:, h] = np.sqrt(var_hi) * (z1[:, h] @ Uh.T) + lo
    return k, U


def make_inputs(w: Workload, T: Optional[int] = None, B: Optional[int] = None,
                H: Optional[int] = None, seed: Optional[int] = None) -> Dict[str, object]:
    """Draw one workload's inputs.

    ``T``, ``B``, ``H`` and ``seed`` override the workload's own values (used
    for reduced-size parity cases with the same distributions).  For a
    workload with a carried prefix, the returned sequence holds
    ``prefix + T`` tokens; ``out["prefix"]`` says where the compared part
    starts.

    Returns a dict of CPU torch tensors in the storage dtype (q, k, v,
    log_alpha, [beta]) plus float32 ``w_lambda [H, dk]``, ``b_lambda [H]`` and
    the needle positions (or None).
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    T_cmp = w.T if T is None else T
    Ttot = T_cmp + w.prefix
    rng = np.random.default_rng(w.seed if seed is None else seed)
    dk, dv = w.dk, w.dv

    q = l2_normalise_rows(rng.standard_normal((B, H, Ttot, dk)))
    needle_pos = None
    if w.keys == "iso":
        k = _iso_keys(rng, B, H, Ttot, dk)
        U = None
    else:
        k, U = _aniso_keys(rng, B, H, Ttot, dk)
    v = rng.standard_normal((B, H, Ttot, dv))
    if w.backbone == "gla":
        # log(sigmoid(x)) / 16 per channel, x ~ N(0,1)
        x = rng.standard_normal((B, H, Ttot, dk))
        log_alpha = -np.logaddexp(0.0, -x) / 16.0
    else:
        # -softplus(x) / 8 per token and head, x ~ N(0,1)
        x = rng.standard_normal((B, H, Ttot))
        log_alpha = -np.logaddexp(0.0, x) / 8.0
    w_lambda = rng.standard_normal((H, dk)) * np.sqrt(1.0 / dk)
    b_lambda = np.zeros(H)
    beta = None
    if w.backbone == "gdn":
        beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, H, Ttot))))
    if U is not None:
        lo = w.prefix + T_cmp // 4
        hi = w.prefix + (3 * T_cmp) // 4
        needle_pos = rng.integers(lo, max(hi, lo + 1), size=B)
        for b in range(B):
            for h in range(H):
                z = rng.standard_normal(dk)
                z = z - U[h] @ (U[h].T @ z)
                k[b, h, needle_pos[b]] = z / np.linalg.norm(z)
        k = l2_normalise_rows(k)

    out = {
        "q": _to_storage(q, w.dtype),
        "k": _to_storage(k, w.dtype),
        "v": _to_storage(v, w.dtype),
        "log_alpha": _to_storage(log_alpha, w.dtype),
        "w_lambda": torch.from_numpy(w_lambda.astype(np.float32)),
        "b_lambda": torch.from_numpy(b_lambda.astype(np.float32)),
        "beta": None if beta is None else _to_storage(beta, w.dtype),
        "needle_pos": needle_pos,
        "prefix": w.prefix,
    }
    return out
