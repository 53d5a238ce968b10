"""GPU parity of the fused decode chain (one launch per layer) against the float64 oracle.

``cq_gemv_layer`` quantizes each problem's float32 activations per token (the A8 rule of
the Needle .cact page, section 一), rotates them and runs the CQ GEMV; ``q4_0_gemv_layer``
runs the Q4_0 GEMV (KMCU page, sections 2 and 3).  Every matrix of a layer is checked
against the oracle's product on the oracle's own encoding and quantization of the same
seeded inputs, within the float32-accumulation tolerance 1e-3 of the GEMV tests.
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


def _q4_layer(mats, B, seed, zero=False):
    """Q4_0 problems for ``mats`` (one activation per distinct K); returns problems, the
    host inputs and the output tensors."""
    xs, hostx, items, ref_in = {}, {}, [], []
    for i, m in enumerate(mats):
        W = synth.weights(m.N, m.K, seed=seed + i)
        if zero:
            W[0] = 0.0
        if m.K not in xs:
            X = synth.activations(B, m.K, seed=seed + 100 + m.K)
            if zero:
                X[0] = 0.0
            hostx[m.K] = X
            xs[m.K] = to_dev(X)
        Y = torch.full((B, m.N), float("nan"), dtype=torch.float32, device="cuda")
        items.append((cq.q4_0_quantize(to_dev(W)), m.N, m.K, xs[m.K], Y))
        ref_in.append((W, hostx[m.K]))
    return cq.make_q4_0_layer(items), items, ref_in


def _cq_layer(mats, b, B, seed, zero=False):
    cb = fitted_cb28()
    xs, hostx, items, ref_in = {}, {}, [], []
    for i, m in enumerate(mats):
        W = synth.weights(m.N, m.K, seed=seed + i, outliers=True)
        if zero:
            W[0] = 0.0
        if m.K not in xs:
            X = synth.activations(B, m.K, seed=seed + 100 + m.K)
            if zero:
                X[0] = 0.0
            hostx[m.K] = X
            xs[m.K] = to_dev(X)
        packed, norms = cq.cq_encode(to_dev(W), b, cb)
        Y = torch.full((B, m.N), float("nan"), dtype=torch.float32, device="cuda")
        items.append((packed, norms, m.N, m.K, xs[m.K], Y))
        ref_in.append((W, hostx[m.K]))
    return cq.make_gemv_layer(items), items, ref_in, cb


def _check_q4(items, ref_in, exact_zero=False):
    for (blocks, N, K, X, Y), (W, Xh) in zip(items, ref_in):
        got = to_host(Y)
        ref = oracle.q4_0_gemv_ref(oracle.q4_0_quantize(W), K, Xh)
        if exact_zero:
            assert not got[0].any() and not got[:, 0].any()
            if got.shape[0] > 1:
                assert max_rel_err(got[1:], ref[1:]) < TOL
        else:
            assert max_rel_err(got, ref) < TOL, (N, K)


def _check_cq(items, ref_in, b, cb, exact_zero=False):
    for (packed, norms, N, K, X, Y), (W, Xh) in zip(items, ref_in):
        got = to_host(Y)
        q_ref, s_ref = oracle.a8_quantize(Xh)
        p_ref, n_ref = oracle.cq_encode(W, b, cb)
        ref = oracle.cq_gemv_ref(p_ref, n_ref, b, cb, q_ref, s_ref)
        if exact_zero:
            assert not got[0].any() and not got[:, 0].any()
            if got.shape[0] > 1:
                assert max_rel_err(got[1:], ref[1:]) < TOL
        else:
            assert max_rel_err(got, ref) < TOL, (N, K, b)


@pytest.mark.parametrize("B", [1, 2])
def test_q4_0_layer_minueza(B):
    """One Minueza-32M layer with its tied lm_head (8 matrices, K = 312 and 1092, rows
    ragged against every block of rows) in one launch."""
    probs, items, ref_in = _q4_layer(synth.MINUEZA_LAYER, B, 7000 + B)
    cq.q4_0_gemv_layer(probs)
    _check_q4(items, ref_in)


@pytest.mark.parametrize("B", [1, 2])
@pytest.mark.parametrize("b", [4, 3, 2, 1, cq.CQ_TERNARY])
def test_cq_layer_45m(b, B):
    """One layer of the 45M-parameter model (q, k, v, o, up, down; K = 512 and 1536),
    every code."""
    probs, items, ref_in, cb = _cq_layer(synth.PREFILL_LAYER, b, B, 7100 + 10 * b + B)
    cq.cq_gemv_layer(probs, b, cb)
    _check_cq(items, ref_in, b, cb)


def test_cq_layer_small_config():
    """The CQ-W4A8 512 x 512 workload at batch 1 as a one-problem layer."""
    probs, items, ref_in, cb = _cq_layer(synth.CQ_SMALL, 4, 1, synth.weight_seed(0, 0))
    cq.cq_gemv_layer(probs, 4, cb)
    _check_cq(items, ref_in, 4, cb)


@pytest.mark.parametrize("B", [1, 2])
def test_layer_ragged_and_long(B):
    """Ragged rows (1 to 1000), K from one group to the 8192 limit, the 16-problem limit."""
    shapes = [(1, 128), (37, 640), (64, 8192), (300, 1152), (17, 4096), (2, 256), (129, 384),
              (1000, 512), (5, 2048), (33, 128), (16, 1024), (77, 896), (8, 3072), (250, 768),
              (3, 6144), (40, 1536)]
    assert len(shapes) == cq.LAYER_MAX_PROBLEMS
    mats = [synth.Mat(f"m{i}", N, K) for i, (N, K) in enumerate(shapes)]
    probs, items, ref_in, cb = _cq_layer(mats, 4, B, 7300 + B)
    cq.cq_gemv_layer(probs, 4, cb)
    _check_cq(items, ref_in, 4, cb)
    qshapes = [(1, 1), (3, 33), (9, 1000), (70, 2080), (40, 8192), (1000, 100)]
    qmats = [synth.Mat(f"q{i}", N, K) for i, (N, K) in enumerate(qshapes)]
    qprobs, qitems, qref = _q4_layer(qmats, B, 7400 + B)
    cq.q4_0_gemv_layer(qprobs)
    _check_q4(qitems, qref)


def test_layer_zero_inputs():
    """An all-zero token and an all-zero row give exact zeros (scale 1 and code 0; norm 0,
    or Q4_0 blocks of d = 1 and nibble 8)."""
    probs, items, ref_in, cb = _cq_layer(synth.PREFILL_LAYER[:2], 4, 2, 7500, zero=True)
    cq.cq_gemv_layer(probs, 4, cb)
    _check_cq(items, ref_in, 4, cb, exact_zero=True)
    qprobs, qitems, qref = _q4_layer(synth.MINUEZA_LAYER[:3], 2, 7600, zero=True)
    cq.q4_0_gemv_layer(qprobs)
    _check_q4(qitems, qref, exact_zero=True)


def test_layer_deterministic_and_consistent():
    """Reruns are bit-identical; the CQ chain agrees with a8_quantize followed by cq_gemv
    (the same quantization; the two products differ only in rounding)."""
    probs, items, ref_in, cb = _cq_layer(synth.PREFILL_LAYER, 4, 1, 7700)
    cq.cq_gemv_layer(probs, 4, cb)
    first = [to_host(it[5]).copy() for it in items]
    cq.cq_gemv_layer(probs, 4, cb)
    for it, f in zip(items, first):
        assert np.array_equal(to_host(it[5]), f)
    for packed, norms, N, K, X, Y in items:
        q, s = cq.a8_quantize(X)
        two = to_host(cq.cq_gemv(packed, norms, N, K, 4, cb, q, s))
        assert max_rel_err(to_host(Y), two) < 2e-4
    qprobs, qitems, _ = _q4_layer(synth.MINUEZA_LAYER, 1, 7800)
    cq.q4_0_gemv_layer(qprobs)
    qfirst = [to_host(it[4]).copy() for it in qitems]
    cq.q4_0_gemv_layer(qprobs)
    for it, f in zip(qitems, qfirst):
        assert np.array_equal(to_host(it[4]), f)
