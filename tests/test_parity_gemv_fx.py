"""GPU parity of the 4-bit CQ GEMV on 16-bit integer codewords (one and two tokens)
against the float64 oracle.

For 4-bit rows, one or two tokens, at least 16 rows and K a multiple of 1024, ``cq_gemv``
takes exact integer dot products on the codewords rounded to the 16-bit grid
``C = rint(cb * S)``, ``S = floor(32767 / max |cb|)``; everything else of the product
(Needle .cact page, section 一: ``w_group = (cb[idx] * norm / sqrt(128)) @ H``, with the
rotation applied to the activations instead) is float32 arithmetic.  The tolerance is the
float32-accumulation bound of the GEMV parity tests, 1e-3.
"""

import numpy as np
import pytest

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


def _case(N, K, B, seed, rows=None, cb=None):
    cb = fitted_cb28() if cb is None else cb
    W = synth.weights(N, K, seed=seed, outliers=True)
    X = synth.activations(B, K, seed=seed + 1)
    packed, norms = cq.cq_encode(to_dev(W), 4, cb)
    q, s = cq.a8_quantize(to_dev(X))
    Y = to_host(cq.cq_gemv(packed, norms, N, K, 4, cb, q, s))
    q_ref, s_ref = oracle.a8_quantize(X)
    Wr = W if rows is None else W[rows]
    p_ref, n_ref = oracle.cq_encode(Wr, 4, cb)
    ref = oracle.cq_gemv_ref(p_ref, n_ref, 4, cb, q_ref, s_ref)
    return (Y if rows is None else Y[:, rows]), ref, (packed, norms, q, s)


@pytest.mark.parametrize("B", [1, 2])
@pytest.mark.parametrize("N,K", [(16, 1024), (17, 2048), (1000, 3072), (4097, 1024), (600, 16384),
                                 (333, 28672), (130, 32768)])
def test_gemv_dp_ragged(N, K, B):
    """Ragged row tiles (N not a multiple of the tile), every segment count from 1 to 32
    (28 leaves warps idle), and the two-token pass (K <= 16384) against two passes."""
    Y, ref, _ = _case(N, K, B, 3 * N + K + B)
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("m", synth.LARGE, ids=lambda m: m.name)
def test_gemv_dp_large_two_tokens_sampled(m):
    rows = np.sort(np.random.default_rng(m.N).choice(m.N, 96, replace=False))
    rows[0], rows[-1] = 0, m.N - 1
    Y, ref, _ = _case(m.N, m.K, 2, synth.weight_seed(4, synth.LARGE.index(m)), rows=rows)
    assert max_rel_err(Y, ref) < TOL


def test_gemv_dp_deterministic():
    """A rerun is bit-identical (fixed-order sums and cross-warp reduction)."""
    cb = fitted_cb28()
    _, _, (packed, norms, q, s) = _case(2048, 4096, 1, 77)
    y0 = to_host(cq.cq_gemv(packed, norms, 2048, 4096, 4, cb, q, s))
    y1 = to_host(cq.cq_gemv(packed, norms, 2048, 4096, 4, cb, q, s))
    assert np.array_equal(y0, y1)


def test_gemv_dp_textbook_codebook():
    """Another 4-bit table (Max's printed levels): the 16-bit grid follows the table."""
    from util import textbook_cb28
    Y, ref, _ = _case(512, 2048, 1, 5, cb=textbook_cb28())
    assert max_rel_err(Y, ref) < TOL


def test_gemv_dp_two_tokens_equal_single_passes():
    """Each token of a two-token pass equals the same token alone (the integer sums are
    exact, and both kernels scale and reduce them in the same float32 order)."""
    cb = fitted_cb28()
    _, _, (packed, norms, q, s) = _case(777, 4096, 2, 91)
    y2 = to_host(cq.cq_gemv(packed, norms, 777, 4096, 4, cb, q, s))
    for t in range(2):
        y1 = to_host(cq.cq_gemv(packed, norms, 777, 4096, 4, cb, q[t:t + 1].clone(), s[t:t + 1].clone()))
        assert np.array_equal(y2[t], y1[0])
