"""The allocation-free decode GEMV, ``cq_gemv_noalloc``, against ``cq_gemv``.

Callers that may not allocate device memory while they run (a plugin inside a host
framework that owns every allocation, an engine with a fixed memory budget) use
``cq_gemv_noalloc``: it keeps the rotated activations in the library's fixed 4 MiB
scratch array instead of a caller workspace.  This file is collected last so that a
run stopping at the first failure has already run every other test; it also passes
on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import gemm_cq_gemv_gb300 as cq
from gemm_cq_gemv_gb300 import build as build_mod
from gemm_cq_gemv_gb300 import synth
from util import fitted_cb28, max_rel_err

pytestmark = pytest.mark.gpu
TOL = 1e-3   # the float32-accumulation tolerance of the GEMV parity tests


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    build_mod.build()
    return cq.lib()


def _operands(N, K, B, b, seed, cbk):
    dev = torch.device("cuda:0")
    W = torch.from_numpy(synth.weights(N, K, seed=seed, outliers=True)).to(dev)
    X = torch.from_numpy(synth.activations(B, K, seed=seed + 1)).to(dev)
    packed, norms = cq.cq_encode(W, b, cbk)
    q, s = cq.a8_quantize(X)
    return packed, norms, q, s


def _call_noalloc(lib, packed, norms, N, K, b, cbk, q, s, Y):
    """Straight through the C ABI, on torch's current stream."""
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.cq_gemv_noalloc(packed.data_ptr(), norms.data_ptr(), N, K, 128, b,
                               ctypes.byref(cbk), q.data_ptr(), s.data_ptr(), q.shape[0],
                               Y.data_ptr(), st)


# (N, K, B, b, seed): the branches of the decode GEMV, in a sequence whose shapes change
# from call to call, so that each call reuses a scratch that still holds the previous
# call's activations:
#   * several CUDA-core passes sharing one rotation in the scratch (B = 3, N % 16 != 0);
#   * the same at another width and shape (2-bit, B = 5);
#   * the tensor-core batch, whose fp16 activations live in the scratch (B >= 3, N % 16 == 0);
#   * one fused pass, which rotates in its prologue and does not touch the scratch (B = 1);
#   * the tensor-core batch again, after the scratch was last written by another shape.
SEQUENCE = ((1000, 4096, 3, 4, 11), (257, 1536, 5, 2, 23), (1024, 4096, 8, 4, 31),
            (512, 2048, 1, 4, 37), (2048, 1024, 16, 4, 41))


def test_noalloc_matches_workspace_gemv_twice(lib):
    cbk = cq.make_codebook(fitted_cb28())
    for _ in range(2):   # the whole sequence twice in a row
        for (N, K, B, b, seed) in SEQUENCE:
            packed, norms, q, s = _operands(N, K, B, b, seed, cbk)
            ref = cq.cq_gemv(packed, norms, N, K, b, cbk, q, s)
            Y = torch.full((B, N), float("nan"), dtype=torch.float32, device=q.device)
            assert _call_noalloc(lib, packed, norms, N, K, b, cbk, q, s, Y) == 0
            torch.cuda.synchronize()
            got, want = Y.cpu().numpy(), ref.cpu().numpy()
            assert np.isfinite(got).all()
            assert max_rel_err(got, want) < TOL, (N, K, B, b)


def test_noalloc_rejects_sizes_beyond_the_scratch(lib):
    cbk = cq.make_codebook(fitted_cb28())
    limit = cq.NOALLOC_MAX_ELEMS
    K = 4096
    B = limit // K + 1                       # B * K just above the fixed scratch
    packed, norms, q, s = _operands(8, K, 1, 4, 5, cbk)
    qb = torch.zeros((B, K), dtype=torch.int8, device=q.device)
    sb = torch.ones((B,), dtype=torch.float32, device=q.device)
    Y = torch.zeros((B, 8), dtype=torch.float32, device=q.device)
    assert _call_noalloc(lib, packed, norms, 8, K, 4, cbk, qb, sb, Y) == 6   # CQ_ERR_WORKSPACE
    with pytest.raises(cq.CQError):
        cq.cq_gemv_noalloc(packed, norms, 8, K, 4, cbk, qb, sb, Y=Y)
