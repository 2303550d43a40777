"""Seeded synthetic inputs for the block-FP8 linear layer.

This module only draws numbers: it holds none of the quantisation or GEMM
arithmetic. Both the CUDA path and the CPU oracle consume what it returns,
so a parity test feeds the two sides bit-identical bf16 inputs.

Workload recipe (the served model's linear-layer inputs, synthetic
stand-ins for the ShareGPT / GSM8K traffic the pages measured on):

* weights  W[N, K]: bf16 of N(0, 0.02), one independent stream per shape;
* activations x[M, K]: bf16 of N(0, 1), and each entry independently, with
  probability 0.001, multiplied by 20 before the bf16 rounding (outliers);
* fp32 draws from numpy's PCG64 ``default_rng(seed)``, rounded to bf16 by
  torch (round to nearest even);
* seeds: weights ``1000 + shape_index``, activations
  ``2000 + 16 * shape_index + m_index``.

The five (N, K) projection shapes are the ones the dual-L20 Qwen3.8-27B-FP8
tuning report lists as missing tuned W8A8 block-FP8 configs (section 8, "L20
FP8 Kernel tuning experiment"). The M values are decode (1), the k+1 tokens of
an MTP / draft verify step with k = 1..7 (2..8), batched decode with k = 2
(64 and 34 sequences x 3 = 102) and a 4096-token prefill chunk.
"""
from __future__ import annotations

import numpy as np
import torch

#: (N, K) of the five block-FP8 projections (dual-L20 report, section 8).
SHAPES: tuple[tuple[int, int], ...] = (
    (17408, 5120),
    (5120, 3072),
    (5120, 8704),
    (7168, 5120),
    (8192, 5120),
)

#: (N, K) of a vocabulary-sized head (the draft / LM head that reads the whole
#: vocabulary every decode step, single-RTX-PRO-6000 Qwen3.8-27B post, section
#: "单并发优化"). The pages give no vocabulary size; 151936 (1187 blocks of 128)
#: is the vocabulary of the model family, K = 5120 its hidden size.
VOCAB_SHAPE: tuple[int, int] = (151936, 5120)
#: Seed index of the vocabulary head's weights (after the five projections).
VOCAB_SEED_INDEX = len(SHAPES)

#: Token counts per call: decode, speculative verify, batched decode, prefill.
M_DECODE = (1,)
M_VERIFY = (2, 3, 4, 5, 6, 7, 8)
M_BATCHED = (64, 102)
M_PREFILL = (4096,)
M_ALL = M_DECODE + M_VERIFY + M_BATCHED + M_PREFILL

WEIGHT_SIGMA = 0.02
OUTLIER_P = 0.001
OUTLIER_MULT = 20.0


def weight_seed(shape_index: int) -> int:
    return 1000 + shape_index


def activation_seed(shape_index: int, m_index: int) -> int:
    return 2000 + 16 * shape_index + m_index


def _to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def weights_bf16(N: int, K: int, seed: int, sigma: float = WEIGHT_SIGMA) -> torch.Tensor:
    """bf16 [N, K] drawn from N(0, sigma^2), CPU tensor."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((N, K), dtype=np.float32)
    w *= np.float32(sigma)
    return _to_bf16(w)


def activations_bf16(M: int, K: int, seed: int, outlier_p: float = OUTLIER_P,
                     outlier_mult: float = OUTLIER_MULT) -> torch.Tensor:
    """bf16 [M, K] drawn from N(0, 1) with sparse x20 outliers, CPU tensor."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K), dtype=np.float32)
    if M * K:
        mask = rng.random((M, K)) < outlier_p
        x[mask] *= np.float32(outlier_mult)
    return _to_bf16(x)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw uint16 encoding of a bf16 CPU tensor, as a numpy array."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def edge_activations_bf16(M: int, K: int, seed: int) -> torch.Tensor:
    """Activations that hit the quantiser's corner cases, group by group.

    Each 1x128 group gets one of: ordinary normals; all zeros; all -0.0;
    a single non-zero entry; the smallest normal bf16 magnitude; bf16
    subnormals only; one huge outlier among small values; a group whose
    values sit exactly on E4M3 rounding midpoints after scaling by a power
    of two; and a constant group.
    """
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K), dtype=np.float32)
    G = 128
    tiny_normal = np.float32(2.0 ** -126)
    for m in range(M):
        for kb in range(K // G):
            kind = (m * (K // G) + kb) % 9
            g = slice(kb * G, (kb + 1) * G)
            if kind == 1:
                x[m, g] = 0.0
            elif kind == 2:
                x[m, g] = -0.0
            elif kind == 3:
                x[m, g] = 0.0
                x[m, kb * G + int(rng.integers(G))] = np.float32(rng.standard_normal())
            elif kind == 4:
                x[m, g] = tiny_normal * np.sign(rng.standard_normal(G)).astype(np.float32)
            elif kind == 5:
                # bf16 subnormals: multiples of 2^-133 below 2^-126
                x[m, g] = (rng.integers(-127, 128, G).astype(np.float32) * np.float32(2.0 ** -133))
            elif kind == 6:
                x[m, g] = rng.standard_normal(G).astype(np.float32) * np.float32(1e-3)
                x[m, kb * G + int(rng.integers(G))] = np.float32(3.0e4)
            elif kind == 7:
                # amax = 448 * 2^-4 makes the scale an exact power of two, so
                # x / s lands exactly on E4M3 midpoints (e.g. 1.0625, 17.0).
                vals = np.array([1.0625, 1.1875, 17.0, 19.0, 0.5 + 1 / 32, 2.0 ** -10,
                                 3 * 2.0 ** -10, 7.5 * 2.0 ** -9, 232.0, 448.0],
                                dtype=np.float64)
                pick = vals[rng.integers(len(vals), size=G)]
                sgn = np.where(rng.random(G) < 0.5, -1.0, 1.0)
                x[m, g] = (pick * sgn * 2.0 ** -4).astype(np.float32)
                x[m, kb * G] = np.float32(448.0 * 2.0 ** -4)
            elif kind == 8:
                x[m, g] = np.float32(-2.5)
    return _to_bf16(x)
