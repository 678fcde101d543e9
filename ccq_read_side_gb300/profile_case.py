"""Runs the CCQ forward a few times on one seeded workload, for profilers.

    python -m ccq_read_side_gb300.profile_case [--backbone gla|gdn|gla_bwd] [--T 2048]
                                               [--launches 3]

No checking, no timing: it exists so that a profiler command line (for
example an Nsight Compute capture of one launch of the tensor-core kernel) can
name a small, reproducible case.  The workload is the B4 H16 d128 bf16
benchmark workload with T tokens (same distributions, seed 2), or the Gated
DeltaNet workload (B2 H16, seed 4) with --backbone gdn, or the gradients of
the CCQ-GLA forward on the benchmark workload in fp32 with --backbone gla_bwd.
"""
from __future__ import annotations

import argparse

import torch

import ccq_read_side_gb300 as ccq
from ccq_read_side_gb300.workloads import WORKLOADS, Workload, make_inputs


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--backbone", choices=["gla", "gdn", "gla_bwd"], default="gla")
    ap.add_argument("--T", type=int, default=2048)
    ap.add_argument("--launches", type=int, default=3)
    args = ap.parse_args()
    w = WORKLOADS[4] if args.backbone == "gdn" else WORKLOADS[2]
    if args.backbone == "gla_bwd":
        w = Workload(w.name + "_f32", "gla", "f32", w.B, w.H, w.T, w.dk, w.dv, w.chunk, w.seed,
                     w.keys)
    inp = make_inputs(w, T=args.T)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    for _ in range(args.launches):
        if args.backbone == "gla_bwd":
            ccq.gla_bwd(d["q"], d["k"], d["v"], d["log_alpha"], d["w_lambda"], d["b_lambda"],
                        d["v"])
        elif args.backbone == "gla":
            ccq.gla_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["w_lambda"], d["b_lambda"],
                        want_state=False)
        else:
            ccq.gdn_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["w_lambda"],
                        d["b_lambda"], want_state=False)
    torch.cuda.synchronize()
    status = ccq.last_device_status()
    if status != 0:
        raise SystemExit("device status: " + ccq.status_string(status))
    print(f"ran {args.launches} x {args.backbone}, T={args.T}")


if __name__ == "__main__":
    main()
