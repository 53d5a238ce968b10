"""Helpers for the GPU parity tests (device transfer only; no method arithmetic)."""

import numpy as np
import pytest
import torch

import gemm_cq_gemv_gb300 as cq


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    cq.lib()  # raises if the library was not built
    return torch.device("cuda:0")


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()
