"""Pins for the product definitions: the float64 dense product of the reconstructed
weights (Needle .cact page §一 reconstruction; §三 GEMV over [out, in] rows) and of the
dequantised Q4_0 blocks (Minueza -> KMCU v1 page §2)."""

import numpy as np

from gemm_cq_gemv_gb300.synth import activations, weights
from oracle import (TERNARY, a8_quantize, codebook_levels, cq_encode, cq_gemv_ref, cq_reconstruct,
                    field_bits, q4_0_dequantize, q4_0_gemv_ref, q4_0_quantize, sylvester_hadamard,
                    unpack_indices)
from util import fitted_cb28


def test_unit_vector_picks_a_column():
    cb = fitted_cb28()
    W = weights(24, 256, seed=8)
    packed, norms = cq_encode(W, 4, cb)
    W_hat = cq_reconstruct(packed, norms, 4, cb)
    for k in (0, 1, 130, 255):
        q = np.zeros((1, 256), np.int8)
        q[0, k] = 1
        y = cq_gemv_ref(packed, norms, 4, cb, q, np.array([1.0], np.float32))
        assert np.array_equal(y[0], W_hat[:, k])


def test_rotation_identity_route():
    """y = s * sum_j (norm/g) * sum_i cb[idx_i] * (Hu q_g)_i, evaluated with plain loops
    and the dense Hu, equals the oracle's dense product of W_hat and s*q."""
    cb = fitted_cb28()
    W = weights(6, 384, seed=12, outliers=True)
    X = activations(3, 384, seed=13)
    q, s = a8_quantize(X)
    Hu = sylvester_hadamard(128)
    for b in (1, 2, 3, 4, TERNARY):
        packed, norms = cq_encode(W, b, cb)
        idx = unpack_indices(packed, field_bits(b))
        lv = codebook_levels(cb, b).astype(np.float64)
        nrm = norms.view(np.float16).astype(np.float64)
        y = np.zeros((3, 6))
        for t in range(3):
            for o in range(6):
                acc = 0.0
                for j in range(3):
                    xr = Hu @ q[t, j * 128:(j + 1) * 128].astype(np.float64)
                    acc += nrm[o, j] / 128.0 * float(np.dot(lv[idx[o, j]], xr))
                y[t, o] = float(s[t]) * acc
        ref = cq_gemv_ref(packed, norms, b, cb, q, s)
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_row_selection_matches_full():
    cb = fitted_cb28()
    W = weights(40, 256, seed=2)
    X = activations(2, 256, seed=3)
    q, s = a8_quantize(X)
    packed, norms = cq_encode(W, 3, cb)
    full = cq_gemv_ref(packed, norms, 3, cb, q, s)
    rows = np.array([0, 7, 39, 12])
    assert np.array_equal(cq_gemv_ref(packed, norms, 3, cb, q, s, rows=rows), full[:, rows])


def test_q4_0_product_by_blocks():
    W = weights(10, 100, seed=6)
    X = activations(2, 100, seed=7)
    blocks = q4_0_quantize(W)
    y = q4_0_gemv_ref(blocks, 100, X)
    # explicit per-block loop: sum_b d_b * sum_k (nib - 8) * x_k, padding skipped
    raw = blocks.reshape(10, 4, 18)
    for t in range(2):
        for o in range(10):
            acc = 0.0
            for b in range(4):
                d = float(raw[o, b, :2].view(np.float16)[0])
                for k in range(32):
                    col = 32 * b + k
                    if col >= 100:
                        continue
                    byte = int(raw[o, b, 2 + k // 2])
                    nib = (byte >> 4) if (k & 1) else (byte & 0x0F)
                    acc += d * (nib - 8) * float(X[t, col])
            assert abs(acc - y[t, o]) <= 1e-12 * max(1.0, abs(acc))
    assert np.array_equal(q4_0_dequantize(blocks, 100).shape, (10, 100))
