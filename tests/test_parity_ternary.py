"""GPU parity of the ternary CQ code (bits = 5, the fixed codebook {-c, 0, +c} of the Needle
mmap page, section "mmap 之下张量按偏移直读") against the oracle.

The encoding is the Needle .cact page's (§一: rotate each 128-group, nearest codeword,
fp16 L2 norm) with three levels, c the three-level Lloyd-Max Gaussian level, indices
0, 1, 2 in 2-bit fields.  Encode and pack are bit-exact; the decode products (the
CUDA-core GEMV at batches of 1 and 2 or ragged rows, the tensor-core pipeline for batches
of >= 3 tokens) are within max relative error 1e-3 of the float64 oracle, per output
vector.  The oracle encodes its own copy of the weights.
"""

import functools

import numpy as np
import pytest

import gemm_cq_gemv_gb300 as cq
from gemm_cq_gemv_gb300 import synth
from gpu_util import require_gpu, to_dev, to_host
import oracle
from util import fitted_cb28, max_rel_err

pytestmark = pytest.mark.gpu
TOL = 1e-3
TER = cq.CQ_TERNARY


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("shape,outl", [((37, 640), True), ((512, 512), False), ((1, 128), False),
                                        ((300, 4096), True)])
def test_ternary_encode_bit_exact(shape, outl):
    cb = fitted_cb28()
    W = synth.weights(*shape, seed=500 + shape[0], outliers=outl)
    p_ref, n_ref = oracle.cq_encode(W, TER, cb)
    p, n = cq.cq_encode(to_dev(W), TER, cb)
    p, n = to_host(p), to_host(n).view(np.uint16)
    assert p.shape == p_ref.shape == (shape[0], shape[1] // 128, 32)
    assert np.array_equal(n, n_ref)
    assert np.array_equal(p, p_ref)
    # every 2-bit field is 0, 1 or 2 (the value 3 is never written)
    assert oracle.unpack_indices(p, 2).max() <= 2


def test_ternary_encode_special_groups():
    """Zero groups (index 0 everywhere, +0 norm), exact zeros after the rotation (the zero
    level, index 1), subnormal and overflowing fp16 norms."""
    cb = fitted_cb28()
    W = np.zeros((6, 256), np.float32)
    W[1, 0] = 0.5                      # rotated: all ones -> +c
    W[2, 129] = 3.0                    # alternating +-1
    W[3, 128] = W[3, 129] = 1.0        # half the rotated coordinates exactly zero
    W[4] = synth.weights(1, 256, seed=5)[0] * np.float32(1e-6)
    W[5] = synth.weights(1, 256, seed=6)[0] * np.float32(3e5)
    p_ref, n_ref = oracle.cq_encode(W, TER, cb)
    p, n = cq.cq_encode(to_dev(W), TER, cb)
    p, n = to_host(p), to_host(n).view(np.uint16)
    assert np.array_equal(n, n_ref)
    assert np.array_equal(p, p_ref)
    idx = oracle.unpack_indices(p_ref, 2)
    assert not idx[0].any() and np.all(idx[1, 0] == 2)
    assert np.all(idx[3, 1, 1::2] == 1)


@functools.lru_cache(maxsize=1)
def _weights(N, K, seed, outliers):
    """Seeded weights, kept for the next case of the same shape (the large shape takes
    ~20 s to draw on the host)."""
    return synth.weights(N, K, seed=seed, outliers=outliers)


def _case(N, K, B, wseed, xseed, outliers=True, rows=None):
    cb = fitted_cb28()
    W = _weights(N, K, wseed, outliers)
    X = synth.activations(B, K, seed=xseed)
    packed, norms = cq.cq_encode(to_dev(W), TER, cb)
    q, s = cq.a8_quantize(to_dev(X))
    Y = to_host(cq.cq_gemv(packed, norms, N, K, TER, cb, q, s))
    q_ref, s_ref = oracle.a8_quantize(X)
    Wr = W if rows is None else W[rows]
    p_ref, n_ref = oracle.cq_encode(Wr, TER, cb)
    ref = oracle.cq_gemv_ref(p_ref, n_ref, TER, cb, q_ref, s_ref)
    return (Y if rows is None else Y[:, rows]), ref


@pytest.mark.parametrize("N,K,B", [(37, 640, 1), (8, 128, 2), (1, 2048, 1), (129, 1152, 5),
                                   (333, 8448, 2), (4096, 4096, 1)])
def test_ternary_gemv_cuda_cores(N, K, B):
    """Batches of 1 and 2 (rotation in the kernel's prologue) and ragged rows with several
    passes (rotation once into the workspace)."""
    Y, ref = _case(N, K, B, 3 * N + K, 17 * K + B)
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("N,K,B", [(400, 1152, 3), (128, 8192, 8), (1040, 4096, 37), (16, 128, 5),
                                   (2048, 2048, 32), (4096, 4096, 16)])
def test_ternary_gemv_tensor_path(N, K, B):
    """Batches of >= 3 tokens on the tensor cores (2-bit fields in the stage, fp16
    operands): ragged row and token tiles, long K, K split in two (128 x 8192)."""
    Y, ref = _case(N, K, B, 5 * N + K + 5, 13 * K + B)
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("B", [1, 32])
def test_ternary_gemv_large_sampled(B):
    """[8192, 28672], the longest K of the large shapes, 128 sampled rows."""
    m = synth.LARGE[2]
    rows = np.sort(np.random.default_rng(50 + B).choice(m.N, 128, replace=False))
    rows[0], rows[-1] = 0, m.N - 1
    Y, ref = _case(m.N, m.K, B, synth.weight_seed(4, 2), synth.activation_seed(4, B), rows=rows)
    assert max_rel_err(Y, ref) < TOL


def test_ternary_gemv_deterministic():
    cb = fitted_cb28()
    W = synth.weights(512, 4096, seed=43)
    X = synth.activations(8, 4096, seed=44)
    packed, norms = cq.cq_encode(to_dev(W), TER, cb)
    q, s = cq.a8_quantize(to_dev(X))
    y0 = to_host(cq.cq_gemv(packed, norms, 512, 4096, TER, cb, q, s))
    y1 = to_host(cq.cq_gemv(packed, norms, 512, 4096, TER, cb, q, s))
    assert np.array_equal(y0, y1)
