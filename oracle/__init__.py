"""fp64 CPU oracle for the CCQ forward -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it.

``run(...)`` calls the token-by-token recurrence in ``ccq_oracle.c`` (built
by ``oracle.build``).  Every function cites the CCQ page passage it follows;
the recurrence itself is documented in the C file.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.library_path()
        if not os.path.exists(path):
            _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        lib.ccq_oracle_fwd.restype = ctypes.c_int
        lib.ccq_oracle_fwd.argtypes = [
            ctypes.c_int, P, P, P, P, P, P, P, P, ctypes.c_int, P, P, P, ctypes.c_int64,
            P, P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int]
        _LIB = lib
    return _LIB


def _f64(x) -> Optional[np.ndarray]:
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (any dtype): exact upcast
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def run(backbone: str, q, k, v, log_alpha, w_lambda=None, b_lambda=None, beta=None,
        lambda_in=None, l2norm: bool = False, S0=None, C0=None, m0=None, t0: int = 0,
        want_sigq: bool = False, nthreads: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Token-by-token fp64 CCQ forward for every (b, h).

    q, k: [B,H,T,dk]; v: [B,H,T,dv]; log_alpha: [B,H,T,dk] (GLA) or [B,H,T]
    (GDN); beta: [B,H,T] (GDN); w_lambda [H,dk]; b_lambda [H]; lambda_in
    [B,H,T] replaces the learned gate when given.  S0 [B,H,dk,dv], C0
    [B,H,dk,dk], m0 [B,H,dk] with count t0 carry a prefix.

    Returns o, lambda, S, C, m (and sigq = Sigma_t q_t when asked).
    """
    bb = {"gla": 0, "gdn": 1}[backbone]
    q, k, v, log_alpha = _f64(q), _f64(k), _f64(v), _f64(log_alpha)
    beta, lambda_in = _f64(beta), _f64(lambda_in)
    w_lambda, b_lambda = _f64(w_lambda), _f64(b_lambda)
    S0, C0, m0 = _f64(S0), _f64(C0), _f64(m0)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, T, dv))
    lam = np.zeros((B, H, T))
    sigq = np.zeros((B, H, T, dk)) if want_sigq else None
    S = np.zeros((B, H, dk, dv))
    C = np.zeros((B, H, dk, dk))
    m = np.zeros((B, H, dk))
    rc = _lib().ccq_oracle_fwd(
        bb, _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(w_lambda),
        _ptr(b_lambda), _ptr(lambda_in), int(bool(l2norm)), _ptr(S0), _ptr(C0), _ptr(m0),
        int(t0), _ptr(o), _ptr(lam), _ptr(sigq), _ptr(S), _ptr(C), _ptr(m), B, H, T, dk, dv,
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"ccq_oracle_fwd failed with status {rc}")
    out = {"o": o, "lambda": lam, "S": S, "C": C, "m": m, "n": int(t0) + T}
    if want_sigq:
        out["sigq"] = sigq
    return out


def run_inputs(backbone: str, inputs: dict, start: int = 0, stop: Optional[int] = None,
               bh: Optional[list] = None, **kw) -> Dict[str, np.ndarray]:
    """Convenience: run on a dict from the workload generator, optionally on a
    token window [start, stop) and a subset of (b, h) pairs (list of (b, h))."""
    sl = slice(start, stop)

    def pick(x, tok_axis=True):
        if x is None:
            return None
        a = _f64(x)
        if bh is not None:
            a = np.stack([a[b, h] for (b, h) in bh])[None]
        return a[:, :, sl] if tok_axis else a

    wl = _f64(inputs["w_lambda"])
    bl = _f64(inputs["b_lambda"])
    if bh is not None:
        wl = np.stack([wl[h] for (_, h) in bh])
        bl = np.stack([bl[h] for (_, h) in bh])
    return run(backbone, pick(inputs["q"]), pick(inputs["k"]), pick(inputs["v"]),
               pick(inputs["log_alpha"]), wl, bl, beta=pick(inputs.get("beta")), **kw)
