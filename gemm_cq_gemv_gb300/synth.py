"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no arithmetic of the quantization method: it only draws random
numbers (NumPy ``default_rng``) and names the matrix shapes of the workloads.  Both the
CUDA path and the CPU oracle receive these arrays as plain inputs.

Recipe (no public dataset is involved; every input is synthetic):
  * weights ``W = N(0, 1) * 0.02`` as float32, ``[out, in]``; with ``outliers=True``,
    1 % of the entries (``rng.random() < 0.01``) are multiplied by 10;
  * activations ``X = N(0, 1)`` as float32, ``[tokens, in]``;
  * Lloyd-Max samples: 400,000 float64 N(0, 1) draws;
  * seeds: workload ``c``, matrix ``m``, batch ``B`` -> weight seed ``1000*c + m``,
    activation seed ``1000*c + 500 + B``.
"""

from dataclasses import dataclass

import numpy as np

LLOYD_MAX_SAMPLES = 400_000


def weights(N: int, K: int, seed: int, outliers: bool = False) -> np.ndarray:
    rng = np.random.default_rng(seed)
    W = rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)
    if outliers:
        mask = rng.random((N, K)) < 0.01
        W[mask] *= np.float32(10.0)
    return W


def activations(B: int, K: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.standard_normal((B, K), dtype=np.float32)


def gaussian_samples(n: int = LLOYD_MAX_SAMPLES, seed: int = 0) -> np.ndarray:
    return np.random.default_rng(seed).standard_normal(n)


def weight_seed(workload: int, matrix: int) -> int:
    return 1000 * workload + matrix


def activation_seed(workload: int, batch: int) -> int:
    return 1000 * workload + 500 + batch


@dataclass(frozen=True)
class Mat:
    name: str
    N: int  # out
    K: int  # in


# Workload 0: one CQ-W4A8 matrix [512, 512], batch 1.
CQ_SMALL = (Mat("w", 512, 512),)

# Workload 1: one Mistral-style decoder layer of Minueza-32M (dim 312, 12 heads,
# 4 kv heads, head_dim 26, ffn 1092) plus the tied lm_head, in Q4_0.
MINUEZA_LAYER = (
    Mat("q", 312, 312), Mat("k", 104, 312), Mat("v", 104, 312), Mat("o", 312, 312),
    Mat("gate", 1092, 312), Mat("up", 1092, 312), Mat("down", 312, 1092),
    Mat("lm_head", 32002, 312),
)

# Workload 2: CQ mixed widths, b = 1..4, batch 1 / 4 / 16, 1 % x10 outliers.
CQ_MIXED = (Mat("sq", 4096, 4096), Mat("up", 11008, 4096))
CQ_MIXED_BITS = (1, 2, 3, 4)
CQ_MIXED_BATCHES = (1, 4, 16)

# Workload 3: the 20 layers of a synthetic 45M-parameter model (d_model 512, ffn 1536,
# kv width 128), layer-major, prefill M = 512 and 2048 tokens.
PREFILL_LAYER = (
    Mat("q", 512, 512), Mat("k", 128, 512), Mat("v", 128, 512), Mat("o", 512, 512),
    Mat("up", 1536, 512), Mat("down", 512, 1536),
)
PREFILL_LAYERS = 20
PREFILL_TOKENS = (512, 2048)

# Workload 4: large-shape bandwidth sweep, CQ-W4A8 and Q4_0, batch 1 / 2 / 8 / 32.
LARGE = (Mat("sq8k", 8192, 8192), Mat("up28k", 28672, 8192), Mat("down28k", 8192, 28672),
         Mat("lm_head", 128256, 4096))
LARGE_BATCHES = (1, 2, 8, 32)


def prefill_matrices():
    """The 120 matrices of the prefill model in layer-major order: (layer, Mat)."""
    return [(layer, m) for layer in range(PREFILL_LAYERS) for m in PREFILL_LAYER]
