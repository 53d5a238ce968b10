"""The degenerate inputs of the method through every decode and prefill product: an all-zero
token (per-token scale 1, every code 0: the A8 rule of the Needle .cact page, §一), an
all-zero weight row (norm 0 in every group, index 0 everywhere; Q4_0 blocks with d = 1 and
nibble 8, KMCU page §2) and a row with one zero group.  Outputs that the definition makes
zero must be exactly zero; the rest match the float64 oracle within the usual tolerance."""

import numpy as np
import pytest

import gemm_cq_gemv_gb300 as cq
from gemm_cq_gemv_gb300 import synth
from gpu_util import require_gpu, to_dev, to_host
import oracle
from util import fitted_cb28, max_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _inputs(N, K, B, seed):
    W = synth.weights(N, K, seed=seed, outliers=True)
    W[0] = 0.0                      # an all-zero row
    W[1, 128:256] = 0.0             # one zero group (CQ) / four zero blocks (Q4_0)
    X = synth.activations(B, K, seed=seed + 1)
    X[0] = 0.0                      # an all-zero token
    return W, X


def _check(Y, ref, tol):
    Y = np.asarray(Y, np.float64)
    assert not Y[0].any(), "zero token must give exact zeros"
    assert not Y[:, 0].any(), "zero row must give exact zeros"
    if Y.shape[0] > 1:   # with one token there is nothing left but the zero token
        assert max_rel_err(Y[1:], ref[1:]) < tol


@pytest.mark.parametrize("b", [4, 2, 1, cq.CQ_TERNARY])
@pytest.mark.parametrize("N,B", [(37, 2), (64, 2), (64, 5), (48, 7)])
def test_cq_gemv_zero_inputs(b, N, B):
    """CUDA-core passes (B <= 2, or rows not a multiple of 16) and the tensor-core batch."""
    cb = fitted_cb28()
    K = 1024
    W, X = _inputs(N, K, B, 300 + N + B + b)
    packed, norms = cq.cq_encode(to_dev(W), b, cb)
    q, s = cq.a8_quantize(to_dev(X))
    Y = to_host(cq.cq_gemv(packed, norms, N, K, b, cb, q, s))
    q_ref, s_ref = oracle.a8_quantize(X)
    assert s_ref[0] == 1.0 and not q_ref[0].any()
    p_ref, n_ref = oracle.cq_encode(W, b, cb)
    assert not n_ref[0].any() and n_ref[1, 1] == 0
    _check(Y, oracle.cq_gemv_ref(p_ref, n_ref, b, cb, q_ref, s_ref), 1e-3)


@pytest.mark.parametrize("b", [1, 2, cq.CQ_TERNARY])
def test_cq_gemv_lut_zero_inputs(b):
    cb = fitted_cb28()
    N, K, B = 40, 1024, 2
    W, X = _inputs(N, K, B, 320 + b)
    packed, norms = cq.cq_encode(to_dev(W), b, cb)
    q, s = cq.a8_quantize(to_dev(X))
    Y = to_host(cq.cq_gemv_lut(packed, norms, N, K, b, cb, q, s))
    q_ref, s_ref = oracle.a8_quantize(X)
    p_ref, n_ref = oracle.cq_encode(W, b, cb)
    _check(Y, oracle.cq_gemv_ref(p_ref, n_ref, b, cb, q_ref, s_ref), 1e-3)


def test_cq_gemm_zero_inputs():
    cb = fitted_cb28()
    N, K, M = 256, 512, 64
    W, X = _inputs(N, K, M, 330)
    packed, norms = cq.cq_encode(to_dev(W), 4, cb)
    q, s = cq.a8_quantize(to_dev(X))
    Y = to_host(cq.cq_gemm(packed, norms, N, K, 4, cb, q, s).float())
    q_ref, s_ref = oracle.a8_quantize(X)
    p_ref, n_ref = oracle.cq_encode(W, 4, cb)
    _check(Y, oracle.cq_gemm_ref(p_ref, n_ref, 4, cb, q_ref, s_ref), 1e-2)


@pytest.mark.parametrize("N,K,B", [(37, 312, 1), (37, 312, 2), (64, 1024, 2), (40, 1024, 3)])
def test_q4_0_gemv_zero_inputs(N, K, B):
    """Row-staged (K = 312) and ring-staged (K = 1024) kernels, one and two tokens per pass."""
    W, X = _inputs(N, K, B, 340 + N + B)
    blocks = cq.q4_0_quantize(to_dev(W))
    Y = to_host(cq.q4_0_gemv(blocks, N, K, to_dev(X)))
    b_ref = oracle.q4_0_quantize(W)
    _check(Y, oracle.q4_0_gemv_ref(b_ref, K, X), 1e-3)


def test_q4_0_gemm_zero_inputs():
    N, K, M = 128, 512, 8
    W, X = _inputs(N, K, M, 350)
    Y = to_host(cq.q4_0_gemm(cq.q4_0_quantize(to_dev(W)), N, K, to_dev(X)))
    _check(Y, oracle.q4_0_gemv_ref(oracle.q4_0_quantize(W), K, X), 1e-3)


@pytest.mark.parametrize("N,K,B", [(37, 312, 2), (64, 1024, 2), (40, 4096, 1)])
def test_q4_0_gemv_non_finite_activation(N, K, B):
    """A token with an infinite or NaN activation gets NaN outputs (every output row sums a
    block holding it; a float32 product would give inf or NaN there too); the other token
    is unaffected and matches the oracle."""
    W, X = _inputs(N, K, B, 360 + N + B)
    X = X.copy()
    X[0, K // 3] = np.inf if K % 2 else np.nan
    X[0, 5] = -np.inf
    blocks = cq.q4_0_quantize(to_dev(W))
    Y = to_host(cq.q4_0_gemv(blocks, N, K, to_dev(X)))
    assert np.isnan(Y[0]).all()
    if B > 1:
        ref = oracle.q4_0_gemv_ref(oracle.q4_0_quantize(W), K, X[1:])
        assert max_rel_err(Y[1:], ref) < 1e-3
