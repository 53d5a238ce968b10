"""Lloyd-Max fit of the Gaussian codebooks ([CACT] §一).

The page states the codebooks ``cb2[4] | cb3[8] | cb4[16]`` are fitted offline by the
Lloyd-Max algorithm on 400,000 Gaussian samples for 200 iterations, and [MMAP] gives
the 1-bit codebook in closed form, ``{-sqrt(2/pi), +sqrt(2/pi)}``, and the ternary one
(bits = 5) as ``{-c, 0, +c}``, both hard-coded in the engine with no table.

Readings taken where the pages are silent:

* the samples are drawn by the caller (they are an input here; the seeded generator
  lives in ``gemm_cq_gemv_gb300.synth``);
* the initial levels are the N(0, 1) quantiles at probabilities (t + 0.5) / L;
* one iteration = thresholds at the midpoints of adjacent levels, then every level
  moves to the mean of the samples in its cell; a sample equal to a threshold belongs
  to the lower cell; an empty cell keeps its level;
* all arithmetic in float64, the result cast to float32 (the table the kernels read).
"""

import math
from statistics import NormalDist

import numpy as np

# [MMAP]: the 1-bit codebook is +-sqrt(2/pi), the mean of |N(0,1)|.
ONE_BIT_LEVEL = math.sqrt(2.0 / math.pi)


def ternary_gaussian_level(iters: int = 200) -> float:
    """``c`` of the ternary codebook ``{-c, 0, +c}`` ([MMAP], bits = 5).

    The page does not give ``c``.  Reading: the three-level Lloyd-Max quantizer of
    N(0, 1), the same optimality rule as the fitted codebooks, solved on the exact
    density instead of samples (like the 1-bit value).  Its middle level is 0 by
    symmetry, its thresholds are the midpoints +-c/2, and the outer level is the mean of
    N(0, 1) above its threshold:  ``c = phi(c/2) / (1 - Phi(c/2))``.  The iteration from
    c = 1 contracts (float64) to 1.2240063619...
    """
    c = 1.0
    for _ in range(iters):
        t = c / 2.0
        tail = 0.5 * math.erfc(t / math.sqrt(2.0))              # 1 - Phi(t)
        c = math.exp(-0.5 * t * t) / math.sqrt(2.0 * math.pi) / tail
    return c


TERNARY_LEVEL = ternary_gaussian_level()


def gaussian_quantile_init(L: int) -> np.ndarray:
    """Initial levels: N(0,1) quantiles at (t + 0.5) / L, t = 0..L-1 (float64)."""
    nd = NormalDist(0.0, 1.0)
    return np.array([nd.inv_cdf((t + 0.5) / L) for t in range(L)], dtype=np.float64)


def lloyd_max_gaussian_fit(samples: np.ndarray, L: int, iters: int = 200) -> np.ndarray:
    """Lloyd-Max quantizer levels (ascending, float32) for the given samples.

    Steps per iteration (the algorithm as the page names it):
      1. thresholds[t] = (levels[t] + levels[t+1]) / 2 for t = 0..L-2;
      2. cell(s) = number of thresholds strictly below s;
      3. levels[c] = mean of the samples with cell c (unchanged if the cell is empty).
    """
    s = np.asarray(samples, dtype=np.float64).ravel()
    levels = gaussian_quantile_init(L)
    for _ in range(iters):
        thr = (levels[:-1] + levels[1:]) / 2.0
        cell = np.searchsorted(thr, s, side="left")
        sums = np.bincount(cell, weights=s, minlength=L)
        counts = np.bincount(cell, minlength=L)
        nz = counts > 0
        levels = levels.copy()
        levels[nz] = sums[nz] / counts[nz]
    return levels.astype(np.float32)
