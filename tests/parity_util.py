"""Shared pieces of the GPU parity tests: seeded problems and the comparison rules.

Tolerances (fixed by the layer's definition, not tuned):
* quantisation: bit-exact codes and scales;
* GEMM, fp32 output: relative L2 error <= 1e-4 against the oracle's fp64 y;
* GEMM, bf16 output: every element within 1 bf16 ulp of the oracle's
  correctly rounded bf16(y) (adjacent in the bf16 ordering), or, where y is so
  close to zero that no fp32 accumulation order can promise that, with the
  fp32 output inside the fp32 accumulation bound KB * 2^-23 * A, where
  A = sum_kb |sa sw P_kb| is the size of the terms summed;
* the bf16 output equals the round-to-nearest-even cast of the fp32 output of
  the same kernels (both entry points share them).
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from block_scaled_fp8_act_gb300 import inputs

G = 128
REL_L2_TOL = 1e-4

# Every compare_gemm result of the session (test id, shape, statistics); the
# conftest prints them at the end of the run.
STATS: list = []


def bf16_ordinal(bits: np.ndarray) -> np.ndarray:
    """Position in the bf16 total order (+0 and -0 both 0)."""
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def gpu_bits(t: torch.Tensor) -> np.ndarray:
    assert t.dtype == torch.bfloat16
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def compare_gemm(out_bf16: torch.Tensor, out_f32: torch.Tensor, y: np.ndarray, aabs: np.ndarray,
                 ref_bits: np.ndarray, K: int) -> dict:
    """Check one GEMM result against the oracle; returns error statistics."""
    gb = gpu_bits(out_bf16)
    gf = out_f32.cpu().numpy().astype(np.float64)
    assert gb.shape == ref_bits.shape == gf.shape == y.shape
    assert np.all(np.isfinite(gf)), "non-finite GPU output"
    # bf16 entry point == RNE(fp32 entry point)
    rne = out_f32.to(torch.bfloat16)
    assert np.array_equal(gpu_bits(rne), gb), "bf16 output is not the rounded fp32 output"
    ny = np.linalg.norm(y)
    rel = np.linalg.norm(gf - y) / ny if ny > 0 else np.linalg.norm(gf)
    assert rel <= REL_L2_TOL, f"fp32 rel-L2 {rel:.3e} > {REL_L2_TOL}"
    dist = np.abs(bf16_ordinal(gb) - bf16_ordinal(ref_bits))
    KB = K // G
    floor_ok = np.abs(gf - y) <= KB * 2.0 ** -23 * aabs
    bad = (dist > 1) & ~floor_ok
    assert not bad.any(), (f"{int(bad.sum())} elements beyond 1 bf16 ulp and the fp32 bound; first at "
                           f"{np.argwhere(bad)[0]}: gpu {gf[bad][0]!r} ref {y[bad][0]!r}")
    stats = {"rel_l2": float(rel), "max_ulp": int(dist.max()) if dist.size else 0,
             "floor_used": int(((dist > 1) & floor_ok).sum()), "elements": int(dist.size),
             "exact_bf16": float((dist == 0).mean()) if dist.size else 1.0}
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    STATS.append({"test": test, "rows": int(y.shape[0]), "N": int(y.shape[1]), "K": int(K), **stats})
    return stats


class Problem:
    """Seeded weights of one (N, K), quantised by both sides."""

    def __init__(self, N: int, K: int, seed: int, device="cuda"):
        from block_scaled_fp8_act_gb300 import fp8act
        self.N, self.K = N, K
        W = inputs.weights_bf16(N, K, seed)
        self.w_ref, self.sw_ref = oracle.weight_quant(inputs.bf16_bits(W))
        self.w, self.sw = fp8act.fp8_weight_quant(W.to(device))
        torch.cuda.synchronize()

    def activations(self, M: int, seed: int, edge: bool = False):
        from block_scaled_fp8_act_gb300 import fp8act
        x = (inputs.edge_activations_bf16(M, self.K, seed) if edge
             else inputs.activations_bf16(M, self.K, seed))
        q_ref, sa_ref = oracle.act_quant(inputs.bf16_bits(x))
        q, sa = fp8act.fp8_act_quant(x.cuda())
        return q, sa, q_ref, sa_ref

    def run_and_compare(self, M: int, seed: int, rows=None, edge: bool = False) -> dict:
        from block_scaled_fp8_act_gb300 import fp8act
        q, sa, q_ref, sa_ref = self.activations(M, seed, edge)
        assert np.array_equal(q.cpu().numpy(), q_ref) and np.array_equal(sa.cpu().numpy(), sa_ref)
        out = fp8act.fp8_block_gemm(q, sa, self.w, self.sw)
        out32 = fp8act.fp8_block_gemm_f32(q, sa, self.w, self.sw)
        torch.cuda.synchronize()
        y, aabs, ref = oracle_gemm(q_ref, sa_ref, self.w_ref, self.sw_ref, rows=rows)
        if rows is not None:
            idx = torch.as_tensor(np.asarray(rows), device=out.device)
            out, out32 = out.index_select(0, idx), out32.index_select(0, idx)
        return compare_gemm(out, out32, y, aabs, ref, self.K)


def oracle_gemm(q, sa, w, sw, rows=None, chunk: int = 256):
    """oracle.block_gemm over whole 128-row weight blocks at a time,
    concatenated along N: the same definition, on sub-problems whose weights
    stay in a host core's cache while every sampled row passes over them."""
    N = w.shape[0]
    if N <= chunk:
        return oracle.block_gemm(q, sa, w, sw, rows=rows)
    parts = [oracle.block_gemm(q, sa, w[n0:n0 + chunk], sw[n0 // G:(n0 + chunk + G - 1) // G], rows=rows)
             for n0 in range(0, N, chunk)]
    return tuple(np.concatenate([p[i] for p in parts], axis=1) for i in range(3))


def tile_rows(M: int, n_random: int, seed: int, edge: int = 128) -> np.ndarray:
    """Rows of an M-token GEMM to compare against the oracle: the first and
    last `edge` rows, a seeded random row of every 32-row lane quadrant of
    every 128-row token tile (m = 128 t + 32 q + r: every tile and every
    tensor-memory lane group of the token-tiled kernel), and `n_random`
    seeded random rows."""
    rng = np.random.default_rng(seed)
    rows = set(range(min(edge, M))) | set(range(max(0, M - edge), M))
    for t in range((M + 127) // 128):
        for qd in range(4):
            lo = 128 * t + 32 * qd
            if lo < M:
                rows.add(int(lo + rng.integers(0, min(32, M - lo))))
    rows |= set(rng.choice(M, size=min(n_random, M), replace=False).tolist())
    return np.array(sorted(rows), np.int64)


def sample_rows(M: int, n_random: int, seed: int) -> np.ndarray:
    """First and last 8 rows plus a seeded random subset, sorted and unique."""
    rng = np.random.default_rng(seed)
    rows = set(range(min(8, M))) | set(range(max(0, M - 8), M))
    rows |= set(rng.choice(M, size=min(n_random, M), replace=False).tolist())
    return np.array(sorted(rows), np.int64)
