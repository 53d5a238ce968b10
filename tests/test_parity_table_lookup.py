"""GPU parity of the table-lookup decode GEMV (``cq_gemv_lut``: 1-bit, 2-bit and ternary
codes) against the float64 oracle.

The product is the Needle .cact page's (§一 reconstruction, §三 rows along the reduction
axis); the kernel follows the smolmaxxing page's 1-bit lookup-table kernel (16-entry
tables of partial sums over 4 activations).  Tolerance: max relative error 1e-3 per
output vector, as for cq_gemv.  The oracle encodes its own copy of the weights.
"""

import functools

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
CODES = [1, 2, cq.CQ_TERNARY]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@functools.lru_cache(maxsize=1)
def _weights(N, K, seed, outliers):
    """Seeded weights, kept for the next case of the same shape (the large shape takes
    ~20 s to draw on the host)."""
    return synth.weights(N, K, seed=seed, outliers=outliers)


def _case(N, K, b, B, wseed, xseed, rows=None, outliers=True):
    cb = fitted_cb28()
    W = _weights(N, K, wseed, outliers)
    X = synth.activations(B, K, seed=xseed)
    packed, norms = cq.cq_encode(to_dev(W), b, cb)
    q, s = cq.a8_quantize(to_dev(X))
    Y = to_host(cq.cq_gemv_lut(packed, norms, N, K, b, cb, q, s))
    q_ref, s_ref = oracle.a8_quantize(X)
    Wr = W if rows is None else W[rows]
    p_ref, n_ref = oracle.cq_encode(Wr, b, cb)
    ref = oracle.cq_gemv_ref(p_ref, n_ref, b, cb, q_ref, s_ref)
    return (Y if rows is None else Y[:, rows]), ref


@pytest.mark.parametrize("b", CODES)
@pytest.mark.parametrize("N,K,B", [(37, 640, 1), (8, 128, 2), (1, 2048, 1), (129, 8448, 1),
                                   (300, 4096, 2), (16, 12288, 1)])
def test_lut_gemv_ragged(b, N, K, B):
    """Ragged rows and K: partial 512-byte pieces, one to six K ranges (8448 positions are
    two ranges at 1 bit and three at 2 bits), several tokens."""
    Y, ref = _case(N, K, b, B, 19 * N + K + b, 23 * K + B)
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("b", CODES)
def test_lut_gemv_mixed_widths_4096(b):
    """[4096, 4096] of the mixed-width sweep at batch 1, all rows."""
    Y, ref = _case(4096, 4096, b, 1, synth.weight_seed(2, 0), synth.activation_seed(2, 1))
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("b", CODES)
def test_lut_gemv_large_sampled(b):
    """[8192, 28672] (the longest K: 4 ranges at 1 bit, 7 at 2 bits), 128 sampled rows."""
    m = synth.LARGE[2]
    rows = np.sort(np.random.default_rng(70 + b).choice(m.N, 128, replace=False))
    rows[0], rows[-1] = 0, m.N - 1
    Y, ref = _case(m.N, m.K, b, 1, synth.weight_seed(4, 2), synth.activation_seed(4, 1), rows=rows)
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("b", [1, cq.CQ_TERNARY])
def test_lut_gemv_row_blocks(b):
    """Enough rows that every CTA holds more than one block of 256 row groups (one range):
    the rows around the blocks of several CTAs and a random sample are checked (row group
    j of 8 rows belongs to CTA j mod G)."""
    N, K = 320_000, 256
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ngroups = -(-N // 8)
    grid = min(sms, ngroups)
    assert -(-ngroups // grid) > 256
    rows = [0, N - 1]
    for c in (0, 1, grid // 2, grid - 1):
        for m in (0, 255, 256, 257):
            j = c + m * grid
            rows += [8 * j - 1, 8 * j, 8 * j + 7, 8 * j + 8]
    extra = np.random.default_rng(40 + b).choice(N, 100, replace=False)
    rows = np.unique(np.clip(np.array(rows + list(extra)), 0, N - 1))
    Y, ref = _case(N, K, b, 1, 31 + b, 37, rows=rows)
    assert max_rel_err(Y, ref) < TOL


@pytest.mark.parametrize("b", CODES)
def test_lut_gemv_matches_cq_gemv_and_is_deterministic(b):
    """Same inputs through both decode GEMVs: both within the tolerance of each other, and
    the table-lookup path reruns bit-identically."""
    cb = fitted_cb28()
    W = synth.weights(1000, 2048, seed=3 + b, outliers=True)
    X = synth.activations(1, 2048, seed=4 + b)
    packed, norms = cq.cq_encode(to_dev(W), b, cb)
    q, s = cq.a8_quantize(to_dev(X))
    y0 = to_host(cq.cq_gemv_lut(packed, norms, 1000, 2048, b, cb, q, s))
    y1 = to_host(cq.cq_gemv_lut(packed, norms, 1000, 2048, b, cb, q, s))
    yg = to_host(cq.cq_gemv(packed, norms, 1000, 2048, b, cb, q, s))
    assert np.array_equal(y0, y1)
    assert max_rel_err(y0, yg) < TOL


@pytest.mark.parametrize("b", [1, 2])
def test_lut_gemv_several_ranges_and_row_blocks(b):
    """Rows of several 512-byte ranges (K = 4224: two ranges at 1 bit, the second of four
    words; three at 2 bits) with more rows per CTA than one block of partial sums holds
    (2048): random packed indices and norms, checked against the oracle on rows at the
    block boundaries, the first and last rows and a random sample."""
    N, K = 312_000, 4224
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(90 + b)
    packed = rng.integers(0, 256, size=(N, K * b // 8), dtype=np.uint8)
    norms = rng.uniform(0.25, 2.0, size=(N, K // 128)).astype(np.float16).view(np.uint16)
    X = synth.activations(1, K, seed=91)
    cb = fitted_cb28()
    q, s = cq.a8_quantize(to_dev(X))
    Y = to_host(cq.cq_gemv_lut(to_dev(packed), to_dev(norms.view(np.int16)), N, K, b, cb, q, s))
    ngroups = -(-N // 8)
    grid = min(sms, ngroups)
    assert -(-ngroups // grid) > 256   # more than one block of 256 row groups per CTA
    rows = [0, N - 1]
    for c in (0, 1, grid // 2, grid - 1):
        for m in (255, 256, 257):
            j = c + m * grid
            rows += [8 * j, 8 * j + 7]
    rows = np.unique(np.clip(np.array(rows + list(rng.choice(N, 200, replace=False))), 0, N - 1))
    q_ref, s_ref = oracle.a8_quantize(X)
    ref = oracle.cq_gemv_ref(packed.reshape(N, K // 128, 16 * b), norms, b, cb, q_ref, s_ref, rows=rows)
    assert max_rel_err(Y[:, rows], ref) < TOL
