"""GPU parity of the quantizers against the oracle: CQ encode and pack (Needle .cact
page §一), per-token int8 (§一, ACT_BITS 8), Q4_0 (Minueza -> KMCU page §2, §3) and the
Lloyd-Max fit (§一).  Bit-exact except the fit (float64 sums in another order)."""

import numpy as np
import pytest
import torch

import gemm_cq_gemv_gb300 as cq
from gemm_cq_gemv_gb300 import synth
from gpu_util import require_gpu, to_dev, to_host
import oracle
from util import fitted_cb28

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _encode_both(W, b, cb):
    p_ref, n_ref = oracle.cq_encode(W, b, cb)
    p, n = cq.cq_encode(to_dev(W), b, cb)
    return p_ref, n_ref, to_host(p), to_host(n).view(np.uint16)


@pytest.mark.parametrize("b", [1, 2, 3, 4])
@pytest.mark.parametrize("shape,outl", [((37, 640), True), ((512, 512), False), ((1, 128), False)])
def test_encode_bit_exact(b, shape, outl):
    cb = fitted_cb28()
    W = synth.weights(*shape, seed=100 + b, outliers=outl)
    p_ref, n_ref, p, n = _encode_both(W, b, cb)
    assert np.array_equal(n, n_ref)
    assert np.array_equal(p, p_ref)


@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_encode_special_groups(b):
    cb = fitted_cb28()
    W = np.zeros((6, 256), np.float32)
    W[1, 0] = 0.5                      # rotated: all ones
    W[2, 129] = 3.0                    # alternating +-1
    W[3, 128] = W[3, 129] = 1.0        # exact zeros after rotation (ties)
    W[4] = synth.weights(1, 256, seed=5)[0] * np.float32(1e-6)   # subnormal fp16 norms
    W[5] = synth.weights(1, 256, seed=6)[0] * np.float32(3e5)    # norm overflows fp16 -> inf
    p_ref, n_ref, p, n = _encode_both(W, b, cb)
    assert np.array_equal(n, n_ref)
    assert np.array_equal(p, p_ref)
    assert n_ref[4, 0] < 0x0400 and n_ref[4, 0] > 0      # subnormal case really exercised
    assert n_ref[5, 0] == 0x7C00


def test_encode_full_size_sampled_rows():
    cb = fitted_cb28()
    N, K = 11008, 4096
    W = synth.weights(N, K, seed=synth.weight_seed(2, 1), outliers=True)
    p, n = cq.cq_encode(to_dev(W), 4, cb)
    p, n = to_host(p), to_host(n).view(np.uint16)
    rows = np.random.default_rng(0).choice(N, 48, replace=False)
    rows = np.concatenate([rows, [0, N - 1]])
    p_ref, n_ref = oracle.cq_encode(W[rows], 4, cb)
    assert np.array_equal(p[rows], p_ref)
    assert np.array_equal(n[rows], n_ref)


@pytest.mark.parametrize("B,K", [(1, 512), (3, 1), (16, 4096), (32, 28672), (5, 333)])
def test_a8_bit_exact(B, K):
    X = synth.activations(B, K, seed=K + B)
    if B > 2:
        X[1] = 0.0
    q_ref, s_ref = oracle.a8_quantize(X)
    q, s = cq.a8_quantize(to_dev(X))
    assert np.array_equal(to_host(s).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(to_host(q), q_ref)


@pytest.mark.parametrize("m", synth.MINUEZA_LAYER, ids=lambda m: m.name)
def test_q4_0_quantize_minueza_bit_exact(m):
    W = synth.weights(m.N, m.K, seed=synth.weight_seed(1, synth.MINUEZA_LAYER.index(m)))
    ref = oracle.q4_0_quantize(W)
    got = to_host(cq.q4_0_quantize(to_dev(W)))
    assert got.shape == ref.shape
    assert np.array_equal(got, ref)


def test_q4_0_quantize_edge_cases():
    W = np.zeros((4, 40), np.float32)
    W[1, 0], W[1, 1], W[1, 2], W[1, 3] = 0.8, -0.8, 0.31, -0.44
    W[2] = synth.weights(1, 40, seed=3)[0]
    W[3, 33] = -1e-30
    ref = oracle.q4_0_quantize(W)
    got = to_host(cq.q4_0_quantize(to_dev(W)))
    assert np.array_equal(got, ref)


def test_codebook_fit_matches_oracle():
    s = synth.gaussian_samples(synth.LLOYD_MAX_SAMPLES, seed=0)
    ds = to_dev(s)
    for L in (4, 8, 16):
        ref = oracle.lloyd_max_gaussian_fit(s, L, 200)
        got = to_host(cq.cq_codebook_fit(ds, L, 200))
        assert np.allclose(got, ref, rtol=1e-6, atol=1e-7), (L, got, ref)


@pytest.mark.parametrize("T,D,G", [(1, 32, 32), (7, 96, 32), (33, 512, 128), (5, 1024, 256),
                                   (300, 128, 32), (2, 4096, 64)])
def test_a8_groups_bit_exact(T, D, G):
    """Grouped A8 (per-head query / KV cache, .cact page §四): codes, scales and the
    fake-quant are bit-identical to the oracle, including zero groups and outliers."""
    X = synth.activations(T, D, seed=T * 7 + D)
    X[0, :G] = 0.0                                   # an all-zero group
    X[-1, -1] = 1e4                                  # an outlier in the last group
    codes, scales = cq.a8_quantize_groups(to_dev(X), G)
    fq = cq.a8_fake_quant_groups(to_dev(X), G)
    q_ref, s_ref = oracle.a8_quantize_groups(X, G)
    assert np.array_equal(to_host(codes), q_ref)
    assert np.array_equal(to_host(scales).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(to_host(fq).view(np.uint32), oracle.a8_fake_quant_groups(X, G).view(np.uint32))
