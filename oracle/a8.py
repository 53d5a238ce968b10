"""Per-token symmetric int8 activation quantization ("A8", [CACT] §一: ``ACT_BITS 8``).

The pages only say activations are 8-bit.  Reading taken (per-token symmetric, as the
CQ-W4A8 decode workload states it): for each token t,
  ``s_t = float32(amax_t) / 127`` (one IEEE float32 division),
  ``q = clip(rint(x / s_t), -127, 127)`` (float32 division, round half to even),
and an all-zero token gets ``s_t = 1`` and ``q = 0``.
"""

import numpy as np


def a8_quantize(X: np.ndarray):
    """``X`` float32 ``[B, K]`` -> (``q`` int8 ``[B, K]``, ``s`` float32 ``[B]``)."""
    X = np.asarray(X, dtype=np.float32)
    if X.ndim != 2:
        raise ValueError("X must be [B, K]")
    amax = np.max(np.abs(X), axis=1) if X.shape[1] > 0 else np.zeros(X.shape[0], np.float32)
    s = np.where(amax > 0, amax / np.float32(127.0), np.float32(1.0)).astype(np.float32)
    ratio = (X / s[:, None]).astype(np.float32)
    q = np.clip(np.rint(ratio), -127, 127).astype(np.int8)
    return q, s


def a8_dequantize(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """``x_hat = s_t * q`` in float64."""
    return np.asarray(q, np.float64) * np.asarray(s, np.float64)[:, None]
