"""Pins for int8 activations ("ACT_BITS 8", Needle .cact page §一; grouped for the query and
the KV cache, §四) and Q4_0
(Minueza -> KMCU v1 page §2 "Q4_0 量化", §3 "行对齐到 32")."""

import json
import os

import numpy as np
import pytest

from gemm_cq_gemv_gb300.synth import MINUEZA_LAYER, activations, weights
import oracle
from oracle import (Q4_0_BLOCK, Q4_0_BLOCK_BYTES, a8_quantize, q4_0_dequantize,
                    q4_0_quantize, q4_0_row_bytes)


def test_a8_hand_example():
    x = np.array([[0.9, -2.0, 0.3, 2.0, 0.0]], dtype=np.float32)
    q, s = a8_quantize(x)
    assert s[0] == np.float32(2.0) / np.float32(127.0)
    assert q.tolist() == [[57, -127, 19, 127, 0]]


def test_a8_properties():
    X = activations(16, 1024, seed=4)
    X[3] = 0.0
    q, s = a8_quantize(X)
    assert q.dtype == np.int8 and s.dtype == np.float32
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    assert s[3] == 1.0 and not q[3].any()
    for t in (0, 1, 2, 5):
        k = np.argmax(np.abs(X[t]))
        assert abs(int(q[t, k])) == 127 and np.sign(q[t, k]) == np.sign(X[t, k])
    # reconstruction within half a step
    err = np.abs(q.astype(np.float64) * s[:, None] - X)
    assert np.all(err <= 0.5 * s[:, None] * (1 + 1e-6))


def test_q4_0_hand_blocks(golden_dir):
    with open(os.path.join(golden_dir, "q4_0_block_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        W = np.array([c["row"]], dtype=np.float32)
        out = q4_0_quantize(W)
        assert bytes(out[0]).hex() == c["bytes_hex"], c["name"]
        if "dequant_first4" in c:
            assert np.array_equal(q4_0_dequantize(out, c["n_cols"])[0, :4], c["dequant_first4"])


def test_q4_0_density_and_minueza_sizes(golden_dir):
    assert Q4_0_BLOCK == 32 and Q4_0_BLOCK_BYTES == 18
    assert Q4_0_BLOCK_BYTES * 8 / Q4_0_BLOCK == 4.5
    with open(os.path.join(golden_dir, "minueza_q4_0_sizes.json")) as f:
        sizes = json.load(f)
    total = 0
    for m in MINUEZA_LAYER:
        rows, cols, nbytes = sizes["matrices"][m.name]
        assert (m.N, m.K) == (rows, cols)
        assert rows * q4_0_row_bytes(cols) == nbytes
        total += nbytes
    assert total == sizes["total_bytes"] == 6_499_800


def test_q4_0_exact_round_trip_of_scaled_integers():
    rng = np.random.default_rng(2)
    d = np.float32(0.125)             # fp16-exact scale
    q = rng.integers(-7, 8, size=(5, 96)).astype(np.float32)
    q[:, ::32] = 8                    # amax = 8 d in every block -> d recovered exactly
    W = q * d
    out = q4_0_quantize(W)
    back = q4_0_dequantize(out, 96)
    expect = np.clip(q, -8, 7) * np.float64(d)   # +8d clips to +7d
    assert np.array_equal(back, expect)


def test_q4_0_padding_and_shapes():
    W = weights(3, 312, seed=1)
    out = q4_0_quantize(W)
    assert out.shape == (3, 10 * 18)
    nib_last = out.reshape(3, 10, 18)[:, 9, 2:]
    # columns 312..319 are padding -> nibble 8 in the last block's last 8 positions
    assert np.all((nib_last[:, 12:] & 0x0F) == 8) and np.all((nib_last[:, 12:] >> 4) == 8)
    back = q4_0_dequantize(out, 312)
    assert back.shape == (3, 312)
    # per-block error at most d / 2, except the clipped maximum (at most d), plus the
    # fp16 rounding of d applied to |nibble - 8| <= 8
    blocks = np.zeros((3, 320), np.float32)
    blocks[:, :312] = W
    amax = np.abs(blocks.reshape(3, 10, 32)).max(axis=2)
    d = (amax / 8).repeat(32, axis=1)[:, :312]
    assert np.all(np.abs(back - W) <= d * (1 + 8 * 2.0 ** -11) + 1e-9)


# ---- grouped A8 (attention side: per-head query quantization, KV fake-quant) -----------

def test_a8_groups_worked_example():
    """One group whose max is 127 (scale exactly 1): the codes are the rounded values,
    half to even (-63.5 -> -64, 0.25 -> 0), and the fake-quant returns them; a zero group
    gets scale 1 and zeros."""
    X = np.array([[127.0, -63.5, 0.25, 1.0, 0.0, 0.0, 0.0, 0.0]], np.float32)
    q, s = oracle.a8_quantize_groups(X, 4)
    assert q.tolist() == [[127, -64, 0, 1, 0, 0, 0, 0]]
    assert s.tolist() == [[1.0, 1.0]]
    assert oracle.a8_fake_quant_groups(X, 4).tolist() == [[127.0, -64.0, 0.0, 1.0, 0.0, 0.0, 0.0, 0.0]]


def test_a8_groups_reduce_to_per_token_when_one_group():
    rng = np.random.default_rng(3)
    X = rng.standard_normal((5, 96)).astype(np.float32)
    q, s = oracle.a8_quantize_groups(X, 96)
    q1, s1 = oracle.a8_quantize(X)
    assert np.array_equal(q, q1) and np.array_equal(s[:, 0], s1)


def test_a8_groups_are_independent_and_scale_exactly():
    """Scaling one group by a power of two scales its scale by it and leaves every code
    (and every other group) unchanged: a misplaced group index would break this."""
    rng = np.random.default_rng(4)
    X = rng.standard_normal((3, 128)).astype(np.float32)
    q, s = oracle.a8_quantize_groups(X, 32)
    Y = X.copy()
    Y[1, 64:96] *= np.float32(8.0)
    q2, s2 = oracle.a8_quantize_groups(Y, 32)
    assert np.array_equal(q, q2)
    expect = s.copy()
    expect[1, 2] *= np.float32(8.0)
    assert np.array_equal(s2, expect)


def test_a8_fake_quant_error_bound_and_extremes():
    """|fq(x) - x| <= s/2 (plus float32 rounding of the product), and each group's largest
    magnitude maps to +-127."""
    rng = np.random.default_rng(5)
    X = (rng.standard_normal((16, 256)) * rng.uniform(0.01, 100.0, (16, 1))).astype(np.float32)
    q, s = oracle.a8_quantize_groups(X, 32)
    fq = oracle.a8_fake_quant_groups(X, 32)
    s_full = np.repeat(s, 32, axis=1).astype(np.float64)
    err = np.abs(fq.astype(np.float64) - X.astype(np.float64))
    assert np.all(err <= 0.5 * s_full * (1 + 1e-6) + np.abs(X) * 2.0**-23)
    qg = np.abs(q.astype(np.int32)).reshape(16, 8, 32)
    assert np.all(qg.max(axis=2) == 127)
