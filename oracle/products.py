"""Dense float64 products that define what the GEMV / GEMM kernels compute.

The CQ kernels never materialise ``W_hat``; they use the rotation identity
``dot(w_g, x_g) = (norm / g) * dot(cb[idx], Hu @ x_g)``.  The oracle does not: it
reconstructs ``W_hat`` by the page's formula ([CACT] §一, ``cq_reconstruct``),
dequantises the activations (``x_hat = s * q``) and multiplies in float64.  For Q4_0 it
dequantises the blocks ([KMCU] §2) and multiplies by the float32 activations.

Large matrices are processed in row chunks (a float64 ``W_hat`` of 128256 x 4096 would
take 4.2 GB); ``rows`` restricts the product to selected output rows so that sampled
outputs of the full-size workloads can be checked one by one.
"""

import numpy as np

from .a8 import a8_dequantize
from .cq import cq_reconstruct
from .q4_0 import q4_0_dequantize

_CHUNK = 4096


def cq_gemv_ref(packed, norms16, b, cb28, Xq, scale, rows=None):
    """``Y[t, o] = sum_k W_hat[o, k] * s_t * q[t, k]`` in float64, ``[B, N]`` (or ``[B, len(rows)]``)."""
    packed = np.asarray(packed, dtype=np.uint8)
    norms16 = np.asarray(norms16, dtype=np.uint16)
    xhat = a8_dequantize(Xq, scale)                       # [B, K]
    sel = np.arange(packed.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.empty((xhat.shape[0], sel.shape[0]), dtype=np.float64)
    for c0 in range(0, sel.shape[0], _CHUNK):
        r = sel[c0:c0 + _CHUNK]
        w_hat = cq_reconstruct(packed[r], norms16[r], b, cb28)
        out[:, c0:c0 + r.shape[0]] = xhat @ w_hat.T
    return out


def cq_gemm_ref(packed, norms16, b, cb28, Xq, scale, rows=None):
    """Prefill product: the same definition as :func:`cq_gemv_ref` for M tokens."""
    return cq_gemv_ref(packed, norms16, b, cb28, Xq, scale, rows=rows)


def q4_0_gemv_ref(blocks, n_cols, X, rows=None):
    """``Y[t, o] = sum_k W_hat[o, k] * X[t, k]`` in float64 for Q4_0 weights."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    X = np.asarray(X, dtype=np.float32).astype(np.float64)
    sel = np.arange(blocks.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.empty((X.shape[0], sel.shape[0]), dtype=np.float64)
    for c0 in range(0, sel.shape[0], _CHUNK):
        r = sel[c0:c0 + _CHUNK]
        w_hat = q4_0_dequantize(blocks[r], n_cols)
        out[:, c0:c0 + r.shape[0]] = X @ w_hat.T
    return out
