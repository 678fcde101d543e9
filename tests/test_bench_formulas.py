"""The benchmark's algorithmic work counts (the numerators of its roofline
fractions), checked against the per-head-token figures written out for the
measured workloads: CCQ-GLA 8 L d + 8 d^2 = 196,608 FLOPs and 5 d s = 1,280
bytes at L = 64, d = 128, bf16; CCQ-GDN 14 L d + 10 d^2 + (2/3) L^2 FLOPs;
the whole B4 H16 T4096 forward moving 335.5 MB and doing 51.54 GFLOP; a
decode step moving S and C of every head once in and once out."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

bench = pytest.importorskip("bench")


def test_gla_forward_counts():
    assert bench.flops_per_head_token(128) == 196_608
    assert bench.bytes_per_head_token(128) == 1_280
    head_tokens = 4 * 16 * 4096
    assert abs(bench.flops_per_head_token(128) * head_tokens / 1e9 - 51.54) < 0.01
    assert abs(bench.bytes_per_head_token(128) * head_tokens / 1e6 - 335.5) < 0.1


def test_gdn_forward_count():
    assert abs(bench.gdn_flops_per_head_token(128) - (14 * 64 * 128 + 10 * 128 ** 2 + 64 ** 2 * 2 / 3)) < 1e-9
    assert abs(bench.gdn_flops_per_head_token(128) - 281_259) < 1


def test_gradient_count():
    # forward sweep 6 dk^2 + 5 dk dv, reverse sweep 6 dk^2 + 7 dk dv (FMA = 2)
    assert bench.bwd_flops_per_head_token(128, 128) == 393_216
    assert bench.bwd_flops_per_head_token(64, 128) == 12 * 64 * 64 + 12 * 64 * 128


def test_decode_step_bytes():
    # S and C in fp32, read and written; m read and written; q, k, v, o bf16;
    # log alpha per channel (GLA) or log alpha and beta scalars (GDN)
    d = 128
    assert bench.step_bytes_per_head(d, False) == 2 * 4 * 2 * d * d + 2 * 4 * d + 4 * d * 2 + 2 * d
    assert bench.step_bytes_per_head(d, True) == 2 * 4 * 2 * d * d + 2 * 4 * d + 4 * d * 2 + 4
    # the GLA step over B64 H16 moves about 270.8 MB
    assert abs(bench.step_bytes_per_head(d, False) * 64 * 16 / 1e6 - 270.8) < 0.1
