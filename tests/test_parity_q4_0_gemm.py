"""GPU parity of the Q4_0 tensor-core GEMM against the float64 oracle.

KMCU page §2 and §3 (Q4_0 blocks: d = amax / 8, nibbles q + 8, y = sum d * (nib - 8) * x).
The product runs with fp16 operands ((nib - 8) * d and x, each rounded once) and fp32
accumulation, so it meets the same bound as the fp32 GEMV: max relative error (infinity
norm per output vector) 1e-3.  The oracle quantizes its own copy of the weights
(bit-exact with the GPU quantizer, checked in test_parity_quantize).
"""

import numpy as np
import pytest

import gemm_cq_gemv_gb300 as cq
from gemm_cq_gemv_gb300 import synth
from gpu_util import require_gpu, to_dev, to_host
import oracle
from util import max_rel_err

pytestmark = pytest.mark.gpu
TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _case(N, K, M, wseed, xseed, rows=None, outliers=False):
    W = synth.weights(N, K, seed=wseed, outliers=outliers)
    X = synth.activations(M, K, seed=xseed)
    blocks = cq.q4_0_quantize(to_dev(W))
    Y = cq.q4_0_gemm(blocks, N, K, to_dev(X))
    cq.cq_device_error()
    Y = to_host(Y)
    sel = np.arange(N) if rows is None else rows
    ref = oracle.q4_0_gemv_ref(oracle.q4_0_quantize(W[sel]), K, X)
    return Y[:, sel], ref


@pytest.mark.parametrize("N,K,M", [
    (128, 256, 1),       # one tile, one slab, one token
    (300, 1000, 5),      # ragged rows, K padded to 1024 (32 blocks), narrow tiles
    (1040, 4096, 37),    # ragged rows, ragged 192-token tile
    (16, 256, 33),       # one partial row tile, the smallest wide tile
    (2048, 2048, 32),    # the largest narrow batch
    (200, 11008, 200),   # K of the mixed-width sweep: 344 blocks = 43 slabs
    (512, 512, 512),     # several token tiles
    (7, 8192, 3),        # fewer rows than one tile, long K
])
def test_q4_0_gemm(N, K, M):
    got, ref = _case(N, K, M, 3 * N + K, 5 * K + M, outliers=True)
    assert max_rel_err(got, ref) < TOL


@pytest.mark.parametrize("m", synth.LARGE, ids=lambda m: m.name)
@pytest.mark.parametrize("M", [32, 512])
def test_q4_0_gemm_large_sampled(m, M):
    rows = np.sort(np.random.default_rng(m.N + 3 * M).choice(m.N, 128, replace=False))
    rows[0], rows[-1] = 0, m.N - 1
    got, ref = _case(m.N, m.K, M, synth.weight_seed(4, 10 + synth.LARGE.index(m)),
                     synth.activation_seed(4, M), rows=rows)
    assert max_rel_err(got, ref) < TOL


def test_q4_0_gemm_matches_gemv_per_token():
    """The GEMM and the CUDA-core GEMV compute the same product: each token agrees to
    the fp16 operand rounding (both within 1e-3 of the oracle)."""
    N, K, M = 640, 2048, 9
    W = synth.weights(N, K, seed=21)
    X = synth.activations(M, K, seed=22)
    blocks = cq.q4_0_quantize(to_dev(W))
    Yg = to_host(cq.q4_0_gemm(blocks, N, K, to_dev(X)))
    Yv = to_host(cq.q4_0_gemv(blocks, N, K, to_dev(X)))
    assert max_rel_err(Yg, Yv) < TOL


@pytest.mark.parametrize("N,K,M", [(384, 1024, 40), (256, 2048, 8)])
def test_q4_0_gemm_deterministic(N, K, M):
    """Bit-identical reruns, including the two-way K split of small-token calls (two
    partials added onto a zeroed output in either order give the same sum)."""
    W = synth.weights(N, K, seed=31)
    X = to_dev(synth.activations(M, K, seed=32))
    blocks = cq.q4_0_quantize(to_dev(W))
    a = to_host(cq.q4_0_gemm(blocks, N, K, X))
    b = to_host(cq.q4_0_gemm(blocks, N, K, X))
    assert np.array_equal(a, b)
