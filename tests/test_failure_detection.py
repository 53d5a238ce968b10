"""Failure detection without a GPU fault: every wait in the GEMM pipeline and the GEMV
kernels is bounded; when one runs out the kernel raises its unit's device error word and
returns, and cq_device_error() reports CQ_ERR_DEVICE_TIMEOUT.  The probe kernels use the
same wait functions on a barrier phase that nothing completes (no fault, no hang)."""

import numpy as np
import pytest

import gemm_cq_gemv_gb300 as cq
from gemm_cq_gemv_gb300 import synth
from gpu_util import require_gpu, to_dev, to_host
import oracle
from util import fitted_cb28, max_rel_err


def test_probe_rejects_out_of_range_timeouts():
    lib = cq.lib()
    assert lib.cq_probe_bounded_wait(0, None) == 1
    assert lib.cq_probe_bounded_wait(20 * 10**9, None) == 1


@pytest.mark.gpu
def test_timed_out_wait_is_reported_and_context_survives():
    require_gpu()
    cq.cq_device_error()                      # start from cleared words
    cq.cq_probe_bounded_wait(20_000_000)      # 20 ms
    with pytest.raises(cq.CQError) as e:
        cq.cq_device_error()
    assert e.value.status == 5                # CQ_ERR_DEVICE_TIMEOUT
    cq.cq_device_error()                      # the report cleared the words
    # the context is still usable: a product right after is correct
    cb = fitted_cb28()
    W = synth.weights(256, 1024, seed=5)
    X = synth.activations(1, 1024, seed=6)
    packed, norms = cq.cq_encode(to_dev(W), 4, cb)
    q, s = cq.a8_quantize(to_dev(X))
    Y = to_host(cq.cq_gemv(packed, norms, 256, 1024, 4, cb, q, s))
    cq.cq_device_error()
    q_ref, s_ref = oracle.a8_quantize(X)
    p_ref, n_ref = oracle.cq_encode(W, 4, cb)
    assert max_rel_err(Y, oracle.cq_gemv_ref(p_ref, n_ref, 4, cb, q_ref, s_ref)) < 1e-3
