"""The tcgen05 kernels' failure path, made to run out without any GPU fault.

Every wait of the batched-decode (16 < M <= 128) and prefill (M > 128)
kernels on a barrier that another role completes is bounded. These tests
shorten the bound through the library's test hook and, in one case, make each
CTA skip its first operand copy (a barrier that nothing completes), then check
that the kernel leaves cleanly: fp8act_check_status() reports
FP8ACT_ERR_TIMEOUT, the context stays usable, and the next call on the same
stream is exact against the oracle with a clean status.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

TIMEOUT = 5  # FP8ACT_ERR_TIMEOUT

# (M, N, K): the weight-streaming tcgen05 kernel with K split over a cluster
# (8 tiles x 8 CTAs) and with several tiles per CTA (160 tiles); the
# token-tiled kernel with split K (40 tiles x 3) and with two token tiles.
CASES = [(32, 1024, 2048), (48, 20480, 512), (64, 5120, 3072), (200, 256, 512)]


@pytest.fixture(scope="module")
def fp8act():
    from block_scaled_fp8_act_gb300 import fp8act as mod
    mod.load(build=True)
    yield mod
    mod.set_wait_limit(-1, False)


def _clean_call_matches_oracle(fp8act, p, q, sa, q_ref, sa_ref):
    from parity_util import compare_gemm, oracle_gemm
    out = fp8act.fp8_block_gemm(q, sa, p.w, p.sw)
    out32 = fp8act.fp8_block_gemm_f32(q, sa, p.w, p.sw)
    assert fp8act.check_status() == 0
    y, aabs, ref = oracle_gemm(q_ref, sa_ref, p.w_ref, p.sw_ref)
    compare_gemm(out, out32, y, aabs, ref, p.K)
    return out32


@pytest.mark.parametrize("M,N,K", CASES)
def test_withheld_copy_times_out_and_recovers(fp8act, M, N, K):
    """Each CTA skips its first operand copy: the MMA thread's first wait runs
    out after 1 ms, every role stops, the issued copies and MMAs drain, and
    the status says so. The next call is exact and clean."""
    from parity_util import Problem
    p = Problem(N, K, seed=N + K + 3)
    q, sa, q_ref, sa_ref = p.activations(M, seed=M + 1)
    ref32 = _clean_call_matches_oracle(fp8act, p, q, sa, q_ref, sa_ref)
    fp8act.set_wait_limit(1_000_000, True)
    try:
        fp8act.fp8_block_gemm_f32(q, sa, p.w, p.sw)
        status = fp8act.check_status()
    finally:
        fp8act.set_wait_limit(-1, False)
    assert status == TIMEOUT
    assert fp8act.check_status() == 0  # read once, then cleared
    again = _clean_call_matches_oracle(fp8act, p, q, sa, q_ref, sa_ref)
    assert torch.equal(again, ref32)


@pytest.mark.parametrize("M,N,K", CASES)
def test_zero_wait_limit_stops_anywhere_and_recovers(fp8act, M, N, K):
    """A zero bound: any wait that is not complete within a few polls gives
    up, wherever it is in the pipeline (mid-ring, at the accumulator
    hand-off, in the epilogue). Whatever happened, the kernels leave, the
    status is OK or TIMEOUT, and the next call is exact and clean."""
    from parity_util import Problem
    p = Problem(N, K, seed=N + K + 4)
    q, sa, q_ref, sa_ref = p.activations(M, seed=M + 2)
    ref32 = _clean_call_matches_oracle(fp8act, p, q, sa, q_ref, sa_ref)
    fp8act.set_wait_limit(0, False)
    try:
        for _ in range(4):
            fp8act.fp8_block_gemm_f32(q, sa, p.w, p.sw)
        status = fp8act.check_status()
    finally:
        fp8act.set_wait_limit(-1, False)
    assert status in (0, TIMEOUT)
    again = _clean_call_matches_oracle(fp8act, p, q, sa, q_ref, sa_ref)
    assert torch.equal(again, ref32)


# Grouped batched decode: three problems whose 190 weight tiles fill the SMs,
# so one launch of the grouped tile kernel takes them all.
GROUPED = [(9000, 1024, 100), (10000, 640, 17), (5000, 512, 77)]


def _grouped_args(fp8act):
    from parity_util import Problem
    probs = [Problem(N, K, seed=N + K + 5) for N, K, _ in GROUPED]
    acts = [p.activations(M, seed=M + 3) for p, (_, _, M) in zip(probs, GROUPED)]
    return [(q, sa, p.w, p.sw) for (q, sa, _, _), p in zip(acts, probs)]


@pytest.mark.parametrize("withhold,limit", [(True, 1_000_000), (False, 0)])
def test_grouped_tile_launch_times_out_and_recovers(fp8act, withhold, limit):
    """The grouped tile kernel's waits are bounded like the single-problem
    kernel's: with each CTA's first copy withheld (or a zero bound) the launch
    leaves, the status reports the timeout (withheld) or OK / TIMEOUT (zero
    bound), and the next grouped call gives the same bits as before with a
    clean status."""
    assert sum((N + 127) // 128 for N, _, _ in GROUPED) >= 152
    args = _grouped_args(fp8act)
    ref = fp8act.fp8_block_gemm_grouped_f32(args)
    assert fp8act.check_status() == 0
    fp8act.set_wait_limit(limit, withhold)
    try:
        for _ in range(1 if withhold else 4):
            fp8act.fp8_block_gemm_grouped_f32(args)
        status = fp8act.check_status()
    finally:
        fp8act.set_wait_limit(-1, False)
    assert status == TIMEOUT if withhold else status in (0, TIMEOUT)
    assert fp8act.check_status() == 0
    again = fp8act.fp8_block_gemm_grouped_f32(args)
    assert fp8act.check_status() == 0
    for a, b in zip(ref, again):
        assert torch.equal(a, b)
