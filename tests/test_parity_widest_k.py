"""GPU parity of the decode GEMVs at their largest reduction length, K = 32768: two
1024-position segments for every one of the 16 warps of a CTA (at K = 28672, the largest
of the workloads, four warps own only one).  The products are the Needle .cact page's (§一,
§三) and the KMCU page's (§2, §3); tolerance 1e-3 per output vector against the float64
oracle, which encodes its own copy of the weights."""

import numpy as np
import pytest

import gemm_cq_gemv_gb300 as cq
from gemm_cq_gemv_gb300 import synth
from gpu_util import require_gpu, to_dev, to_host
import oracle
from util import fitted_cb28, max_rel_err

pytestmark = pytest.mark.gpu
TOL = 1e-3
K_MAX = 32768


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("b", [4, 1])
@pytest.mark.parametrize("N,B", [(64, 1), (37, 2)])
def test_cq_gemv_max_k(b, N, B):
    cb = fitted_cb28()
    W = synth.weights(N, K_MAX, seed=900 + N + b, outliers=True)
    X = synth.activations(B, K_MAX, seed=901 + B)
    packed, norms = cq.cq_encode(to_dev(W), b, cb)
    q, s = cq.a8_quantize(to_dev(X))
    Y = to_host(cq.cq_gemv(packed, norms, N, K_MAX, b, cb, q, s))
    q_ref, s_ref = oracle.a8_quantize(X)
    p_ref, n_ref = oracle.cq_encode(W, b, cb)
    assert max_rel_err(Y, oracle.cq_gemv_ref(p_ref, n_ref, b, cb, q_ref, s_ref)) < TOL


@pytest.mark.parametrize("N,B", [(64, 1), (37, 2)])
def test_q4_0_gemv_max_k(N, B):
    W = synth.weights(N, K_MAX, seed=910 + N)
    X = synth.activations(B, K_MAX, seed=911 + B)
    blocks = cq.q4_0_quantize(to_dev(W))
    Y = to_host(cq.q4_0_gemv(blocks, N, K_MAX, to_dev(X)))
    ref = oracle.q4_0_gemv_ref(oracle.q4_0_quantize(W), K_MAX, X)
    assert max_rel_err(Y, ref) < TOL
