"""GPU parity of the decode GEMVs against the float64 oracle.

CQ: Needle .cact page §一 (reconstruction ``w_group = (cb[idx] * norm) @ H``) and §三
(GEMV along the [out, in] rows); Q4_0: Minueza -> KMCU page §2 and §3.  Tolerance: max
relative error (infinity norm per output vector) 1e-3 for the float32 accumulation.
The oracle encodes its own copy of the weights (bit-exact with the GPU encode, checked
in test_parity_quantize), so no oracle input comes from the CUDA path.
"""

import numpy as np
import pytest
import torch

import gemm_cq_gemv_gb300 as cq
from gemm_cq_gemv_gb300 import synth
from gpu_util import require_gpu, to_dev, to_host
import oracle
from util import fitted_cb28, max_rel_err

pytestmark = pytest.mark.gpu
TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _cq_case(N, K, b, B, wseed, xseed, outliers=False, rows=None):
    cb = fitted_cb28()
    W = synth.weights(N, K, seed=wseed, outliers=outliers)
    X = synth.activations(B, K, seed=xseed)
    dW = to_dev(W)
    packed, norms = cq.cq_encode(dW, b, cb)
    del dW
    q, s = cq.a8_quantize(to_dev(X))
    Y = to_host(cq.cq_gemv(packed, norms, N, K, b, cb, q, s))
    q_ref, s_ref = oracle.a8_quantize(X)
    if rows is None:
        p_ref, n_ref = oracle.cq_encode(W, b, cb)
        ref = oracle.cq_gemv_ref(p_ref, n_ref, b, cb, q_ref, s_ref)
        return Y, ref
    p_ref, n_ref = oracle.cq_encode(W[rows], b, cb)
    ref = oracle.cq_gemv_ref(p_ref, n_ref, b, cb, q_ref, s_ref)
    return Y[:, rows], ref


def test_cq_gemv_small_config():
    """512 x 512, 4-bit, batch 1 (the small CQ-W4A8 workload)."""
    Y, ref = _cq_case(512, 512, 4, 1, synth.weight_seed(0, 0), synth.activation_seed(0, 1))
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("b", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K,B", [(37, 640, 1), (300, 1536, 3), (8, 128, 2), (1, 2048, 1),
                                   (129, 1152, 5)])
def test_cq_gemv_ragged(b, N, K, B):
    Y, ref = _cq_case(N, K, b, B, 7 * N + b, 11 * K + B, outliers=True)
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("b", [1, 2, 3, 4])
@pytest.mark.parametrize("B", [1, 4, 16])
def test_cq_gemv_mixed_widths_4096(b, B):
    """[4096, 4096] of the mixed-width sweep, every width and batch, all rows."""
    Y, ref = _cq_case(4096, 4096, b, B, synth.weight_seed(2, 0), synth.activation_seed(2, B),
                      outliers=True)
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("b", [1, 4])
def test_cq_gemv_mixed_widths_11008_sampled(b):
    rows = np.sort(np.random.default_rng(b).choice(11008, 256, replace=False))
    rows[-1] = 11007
    Y, ref = _cq_case(11008, 4096, b, 16, synth.weight_seed(2, 1), synth.activation_seed(2, 16),
                      outliers=True, rows=rows)
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("m", synth.LARGE, ids=lambda m: m.name)
@pytest.mark.parametrize("B", [1, 32])
def test_cq_gemv_large_sampled(m, B):
    rows = np.sort(np.random.default_rng(m.N + B).choice(m.N, 128, replace=False))
    rows[0], rows[-1] = 0, m.N - 1
    Y, ref = _cq_case(m.N, m.K, 4, B, synth.weight_seed(4, synth.LARGE.index(m)),
                      synth.activation_seed(4, B), rows=rows)
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("b", [1, 2, 3])
@pytest.mark.parametrize("B", [1, 32])
def test_cq_gemv_large_widths_sampled(b, B):
    """1- to 3-bit rows on [8192, 28672]: the longest K of the large shapes (448 stages,
    K split in two on the tensor path at B = 32; two K segments per warp at B = 1)."""
    m = synth.LARGE[2]
    rows = np.sort(np.random.default_rng(b + B).choice(m.N, 128, replace=False))
    rows[0], rows[-1] = 0, m.N - 1
    Y, ref = _cq_case(m.N, m.K, b, B, synth.weight_seed(4, 2), synth.activation_seed(4, B),
                      outliers=True, rows=rows)
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("b", [4, 3, 2, 1])
@pytest.mark.parametrize("N,K,B", [(400, 1152, 3), (128, 8192, 8), (1040, 4096, 37), (16, 128, 5),
                                   (2048, 2048, 32)])
def test_cq_gemv_batched_tensor_path(N, K, B, b):
    """Batches of >= 3 tokens (rows a multiple of 16) run on the tensor cores with fp16
    operands and fp32 accumulation, every index width: ragged row tiles, ragged token
    tiles, long K, K split in two (128 x 8192)."""
    Y, ref = _cq_case(N, K, b, B, 5 * N + K + b, 13 * K + B, outliers=True)
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("b", [4, 3, 2, 1])
def test_cq_gemv_batched_tensor_path_deterministic(b):
    """The tensor-core batch with a two-way K split (few row tiles) reruns bit-identically."""
    cb = fitted_cb28()
    W = synth.weights(512, 4096, seed=41)
    X = synth.activations(8, 4096, seed=42)
    packed, norms = cq.cq_encode(to_dev(W), b, cb)
    q, s = cq.a8_quantize(to_dev(X))
    y0 = to_host(cq.cq_gemv(packed, norms, 512, 4096, b, cb, q, s))
    y1 = to_host(cq.cq_gemv(packed, norms, 512, 4096, b, cb, q, s))
    assert np.array_equal(y0, y1)


def test_cq_gemv_batch_consistency():
    """Each token of a batched call equals the same token alone (up to fp32 rounding)."""
    cb = fitted_cb28()
    W = synth.weights(333, 1024, seed=1)
    X = synth.activations(7, 1024, seed=2)
    packed, norms = cq.cq_encode(to_dev(W), 3, cb)
    q, s = cq.a8_quantize(to_dev(X))
    Yb = to_host(cq.cq_gemv(packed, norms, 333, 1024, 3, cb, q, s))
    for t in range(7):
        Y1 = to_host(cq.cq_gemv(packed, norms, 333, 1024, 3, cb, q[t:t + 1].clone(),
                                s[t:t + 1].clone()))
        assert np.allclose(Yb[t], Y1[0], rtol=1e-5, atol=1e-6 * np.abs(Y1).max())


def _q4_case(N, K, B, wseed, xseed, rows=None):
    W = synth.weights(N, K, seed=wseed)
    X = synth.activations(B, K, seed=xseed)
    blocks = cq.q4_0_quantize(to_dev(W))
    Y = to_host(cq.q4_0_gemv(blocks, N, K, to_dev(X)))
    if rows is None:
        ref = oracle.q4_0_gemv_ref(oracle.q4_0_quantize(W), K, X)
        return Y, ref
    ref = oracle.q4_0_gemv_ref(oracle.q4_0_quantize(W[rows]), K, X)
    return Y[:, rows], ref


@pytest.mark.parametrize("m", synth.MINUEZA_LAYER, ids=lambda m: m.name)
@pytest.mark.parametrize("B", [1, 2, 8, 32])
def test_q4_0_gemv_minueza(m, B):
    Y, ref = _q4_case(m.N, m.K, B, synth.weight_seed(1, synth.MINUEZA_LAYER.index(m)),
                      synth.activation_seed(1, B))
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("N,K,B", [(1, 1, 1), (3, 33, 2), (9, 1000, 3), (70, 2080, 1), (40, 2048, 3),
                                   (333, 8448, 1)])
def test_q4_0_gemv_ragged(N, K, B):
    Y, ref = _q4_case(N, K, B, N + K, K + B)
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("m", synth.LARGE, ids=lambda m: m.name)
@pytest.mark.parametrize("B", [1, 32])
def test_q4_0_gemv_large_sampled(m, B):
    rows = np.sort(np.random.default_rng(m.N - B).choice(m.N, 128, replace=False))
    rows[0], rows[-1] = 0, m.N - 1
    Y, ref = _q4_case(m.N, m.K, B, synth.weight_seed(4, 10 + synth.LARGE.index(m)),
                      synth.activation_seed(4, B), rows=rows)
    assert max_rel_err(Y, ref) < TOL
