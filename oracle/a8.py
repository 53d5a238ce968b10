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


# ---------------------------------------------------------------------------------------
# Grouped A8 for the attention side ([CACT] §四, KV cache budget: the key / value cache is
# int8 (``kv_bits = 8``), the query gets per-head symmetric A8 quantization, keys and
# values a per-head A8 fake-quant, and the per-layer budget stores one 4-byte scale per
# ``KV_GROUP = 32`` cached values).  Reading: the same per-token symmetric rule as
# ``a8_quantize``, applied to every group of G consecutive features of a row (a head, or
# a KV_GROUP of 32 values); the fake-quant returns ``q * s`` (float32 product).
# ---------------------------------------------------------------------------------------
def a8_quantize_groups(X: np.ndarray, G: int):
    """``X`` float32 ``[T, D]``, ``G | D`` -> (``q`` int8 ``[T, D]``, ``s`` float32 ``[T, D/G]``)."""
    X = np.asarray(X, dtype=np.float32)
    T, D = X.shape
    if G < 1 or D % G:
        raise ValueError("G must divide D")
    q, s = a8_quantize(X.reshape(T * (D // G), G))
    return q.reshape(T, D), s.reshape(T, D // G)


def a8_fake_quant_groups(X: np.ndarray, G: int) -> np.ndarray:
    """Quantize then dequantize every G-group: ``float32(q * s)``, float32 ``[T, D]``."""
    X = np.asarray(X, dtype=np.float32)
    T, D = X.shape
    q, s = a8_quantize_groups(X, G)
    s_full = np.repeat(s, G, axis=1)
    return (q.astype(np.float32) * s_full).astype(np.float32)
