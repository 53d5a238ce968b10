"""GPU parity of the tcgen05 prefill GEMM against the float64 oracle.

Needle .cact page §三 (prefill GEMM over the [out, in] rows) and §一 (reconstruction);
the layer set is the synthetic 45M-parameter model (d_model 512, ffn 1536, kv width
128, 20 layers).  Tolerance: max relative error (infinity norm per output row of Y^T,
i.e. per token) 1e-2 for the bf16 tensor-core product with fp32 accumulation.
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
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _bf16_to_np(t):
    return t.float().cpu().numpy()


def _case(N, K, M, wseed, xseed, rows=None):
    cb = fitted_cb28()
    W = synth.weights(N, K, seed=wseed)
    X = synth.activations(M, K, seed=xseed)
    packed, norms = cq.cq_encode(to_dev(W), 4, cb)
    q, s = cq.a8_quantize(to_dev(X))
    Y = cq.cq_gemm(packed, norms, N, K, 4, cb, q, s)
    cq.cq_device_error()
    got = _bf16_to_np(Y)
    q_ref, s_ref = oracle.a8_quantize(X)
    sel = np.arange(N) if rows is None else rows
    p_ref, n_ref = oracle.cq_encode(W[sel], 4, cb)
    ref = oracle.cq_gemm_ref(p_ref, n_ref, 4, cb, q_ref, s_ref)
    return got[:, sel], ref


@pytest.mark.parametrize("N,K,M", [(256, 512, 256), (128, 512, 256), (512, 1536, 512),
                                   (1536, 512, 2048), (256, 128, 256)])
def test_gemm_single(N, K, M):
    got, ref = _case(N, K, M, N + K, M + K)
    assert max_rel_err(got, ref) < TOL


@pytest.mark.parametrize("N,K,M", [(144, 640, 300), (16, 256, 1), (400, 384, 129)])
def test_gemm_ragged(N, K, M):
    got, ref = _case(N, K, M, 3 * N + K, M + 7)
    assert max_rel_err(got, ref) < TOL


@pytest.mark.parametrize("M", synth.PREFILL_TOKENS)
def test_gemm_grouped_20_layer_model(M):
    """All 120 matrices of the 20-layer model in one grouped call (layer-major)."""
    cb = fitted_cb28()
    dev = torch.device("cuda:0")
    mats = synth.prefill_matrices()
    X = {K: synth.activations(M, K, seed=synth.activation_seed(3, M) + K) for K in (512, 1536)}
    act = {}
    for K, x in X.items():
        act[K] = cq.a8_quantize(to_dev(x))
    items, keep = [], []
    Ws = []
    for i, (layer, m) in enumerate(mats):
        W = synth.weights(m.N, m.K, seed=synth.weight_seed(3, i))
        Ws.append(W)
        packed, norms = cq.cq_encode(to_dev(W), 4, cb)
        Y = torch.empty((M, m.N), dtype=torch.bfloat16, device=dev)
        q, s = act[m.K]
        items.append((packed, norms, m.N, m.K, q, s, Y))
        keep.append(Y)
    probs = cq.make_gemm_problems(items)
    cq.cq_gemm_grouped(probs, M, 4, cb, device=dev)
    cq.cq_device_error()
    qs = {K: oracle.a8_quantize(x) for K, x in X.items()}
    for i, (layer, m) in enumerate(mats):
        got = _bf16_to_np(keep[i])
        p_ref, n_ref = oracle.cq_encode(Ws[i], 4, cb)
        q_ref, s_ref = qs[m.K]
        ref = oracle.cq_gemm_ref(p_ref, n_ref, 4, cb, q_ref, s_ref)
        err = max_rel_err(got, ref)
        assert err < TOL, (layer, m.name, err)
        if layer in (0, 7):
            # the grouped launch computes each tile exactly like a single-matrix call
            single = cq.cq_gemm(items[i][0], items[i][1], m.N, m.K, 4, cb, items[i][4],
                                items[i][5])
            assert torch.equal(single, keep[i])


def test_gemm_grouped_many_problems_and_activations():
    """More problems than one launch holds (130 > 120) and more distinct activations than
    one rotation launch or one GEMM launch takes (10 > 8): the call splits into several
    launches and every matrix still matches its own single-matrix call bit for bit and
    the oracle within the tolerance."""
    cb = fitted_cb28()
    dev = torch.device("cuda:0")
    M = 70
    Ks = [128, 256, 384, 512, 640, 768, 896, 1024, 1152, 1280]
    X = {K: synth.activations(M, K, seed=900 + K) for K in Ks}
    act = {K: cq.a8_quantize(to_dev(x)) for K, x in X.items()}
    items, Ws, shapes = [], [], []
    for i in range(130):
        K = Ks[i % len(Ks)]
        N = 16 * (1 + (i * 7) % 9)
        W = synth.weights(N, K, seed=5000 + i)
        Ws.append(W)
        shapes.append((N, K))
        packed, norms = cq.cq_encode(to_dev(W), 4, cb)
        q, s = act[K]
        items.append((packed, norms, N, K, q, s, torch.empty((M, N), dtype=torch.bfloat16, device=dev)))
    cq.cq_gemm_grouped(cq.make_gemm_problems(items), M, 4, cb, device=dev)
    cq.cq_device_error()
    qs = {K: oracle.a8_quantize(x) for K, x in X.items()}
    for i, (N, K) in enumerate(shapes):
        single = cq.cq_gemm(items[i][0], items[i][1], N, K, 4, cb, items[i][4], items[i][5])
        assert torch.equal(single, items[i][6]), i
        if i % 13 == 0:
            p_ref, n_ref = oracle.cq_encode(Ws[i], 4, cb)
            ref = oracle.cq_gemm_ref(p_ref, n_ref, 4, cb, *qs[K])
            assert max_rel_err(_bf16_to_np(items[i][6]), ref) < TOL, i
