"""The C-ABI library loads, exports every function ``include/*.h`` declares, and rejects
bad arguments on the host before launching anything (no GPU needed)."""

import ctypes
import glob
import os
import re

import pytest

import gemm_cq_gemv_gb300 as cq
from gemm_cq_gemv_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DECL = re.compile(r"^\s*(?:const\s+char\s*\*|cq_status|size_t|int)\s+(\w+)\s*\(", re.M)


def _declared():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        with open(h) as f:
            names += DECL.findall(f.read())
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return cq.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
        assert n in cq.SIGNATURES, f"binding lacks a signature for {n}"


def test_status_strings_and_version(lib):
    assert cq.cq_abi_version() == 1
    for code, name in [(0, "CQ_OK"), (1, "CQ_ERR_INVALID_ARG"), (2, "CQ_ERR_ALIGNMENT"),
                       (3, "CQ_ERR_UNSUPPORTED"), (4, "CQ_ERR_CUDA"), (5, "CQ_ERR_DEVICE_TIMEOUT"),
                       (6, "CQ_ERR_WORKSPACE")]:
        assert cq.cq_status_string(code) == name
    assert cq.cq_status_string(99) == "CQ_ERR_UNKNOWN"


def test_workspace_size_query(lib):
    assert cq.cq_gemv_workspace_bytes(1, 4096) == 4096 * 4
    assert cq.cq_gemv_workspace_bytes(0, 4096) == 0


# Host-side validation: fake (never dereferenced) pointers; every call below must return
# an error before any CUDA call is made.
A = 0x10000   # 16-byte aligned fake address
M = 0x10004   # misaligned fake address


def _cb():
    return ctypes.byref(cq.make_codebook([0.0] * 28))


def test_encode_validation(lib):
    INV, ALN = 1, 2
    assert lib.cq_encode(A, 4, 100, 128, 4, _cb(), A, A, None) == INV     # K % 128
    assert lib.cq_encode(A, 4, 128, 64, 4, _cb(), A, A, None) == INV      # g != 128
    assert lib.cq_encode(A, 4, 128, 128, 0, _cb(), A, A, None) == INV     # b = 0
    assert lib.cq_encode(A, 4, 128, 128, 6, _cb(), A, A, None) == INV     # b = 6 (5 is ternary)
    assert lib.cq_encode(M, 4, 128, 128, 5, _cb(), A, A, None) == ALN     # ternary accepted
    assert lib.cq_encode(None, 4, 128, 128, 4, _cb(), A, A, None) == INV  # NULL
    assert lib.cq_encode(A, 0, 128, 128, 4, _cb(), A, A, None) == INV     # N = 0
    assert lib.cq_encode(M, 4, 128, 128, 4, _cb(), A, A, None) == ALN


def test_a8_and_q4_validation(lib):
    INV, ALN = 1, 2
    assert lib.a8_quantize(A, 0, 16, A, A, None) == INV
    assert lib.a8_quantize(A, 1, 16, M, A, None) == ALN
    assert lib.q4_0_quantize(A, 1, 0, A, None) == INV
    assert lib.q4_0_quantize(M, 1, 32, A, None) == ALN
    assert lib.q4_0_gemv(A, 1, 0, A, 1, A, None) == INV
    assert lib.q4_0_gemv(A, 1, 32, A, 1, M, None) == ALN


def test_gemv_validation(lib):
    INV, ALN, WS = 1, 2, 6
    f = lib.cq_gemv
    assert f(A, A, 8, 100, 128, 4, _cb(), A, A, 1, A, A, 1 << 20, None) == INV
    assert f(A, A, 8, 128, 128, 7, _cb(), A, A, 1, A, A, 1 << 20, None) == INV
    assert f(A, A, 8, 128, 128, 6, _cb(), A, A, 1, A, A, 1 << 20, None) == INV
    assert f(A, A, 8, 128, 128, 5, _cb(), A, A, 1, M, A, 1 << 20, None) == ALN   # ternary accepted
    assert lib.cq_gemv_noalloc(A, A, 8, 128, 128, 6, _cb(), A, A, 1, A, None) == INV
    assert f(A, A, 8, 128, 128, 4, _cb(), A, A, 0, A, A, 1 << 20, None) == INV
    assert f(A, A, 8, 128, 128, 4, _cb(), A, A, 1, M, A, 1 << 20, None) == ALN
    assert f(A, A, 8, 128, 128, 4, _cb(), A, A, 2, A, A, 16, None) == WS
    assert f(A, A, 8, 128, 128, 4, _cb(), A, A, 2, A, None, 1 << 20, None) == WS
    UNS = 3
    assert f(A, A, 8, 128, 128, 4, _cb(), A, A, (1 << 30) + 1, A, A, 1 << 40, None) == UNS   # B
    # tensor-core path: ceil(B / 32) * ceil(N / 128) = 2^15 * 2^17 output tiles > 2^23
    assert f(A, A, 1 << 24, 128, 128, 2, _cb(), A, A, 1 << 20, A, A, 1 << 40, None) == UNS
    assert lib.q4_0_gemv(A, 1, 32, A, (1 << 30) + 1, A, None) == UNS
    # K beyond two 1024-position segments per warp (32768)
    assert f(A, A, 8, 32768 + 128, 128, 4, _cb(), A, A, 1, A, A, 1 << 40, None) == UNS
    assert lib.q4_0_gemv(A, 1, 32768 + 32, A, 1, A, None) == UNS


def test_gemv_lut_validation(lib):
    INV, ALN, UNS = 1, 2, 3
    f = lib.cq_gemv_lut
    assert f(A, A, 8, 128, 128, 4, _cb(), A, A, 1, A, None) == UNS    # 4-bit: use cq_gemv
    assert f(A, A, 8, 128, 128, 3, _cb(), A, A, 1, A, None) == UNS
    assert f(A, A, 8, 128, 128, 6, _cb(), A, A, 1, A, None) == INV
    assert f(A, A, 8, 100, 128, 1, _cb(), A, A, 1, A, None) == INV    # K % 128
    assert f(A, A, 8, 128, 64, 1, _cb(), A, A, 1, A, None) == INV     # g
    assert f(A, A, 0, 128, 128, 1, _cb(), A, A, 1, A, None) == INV    # N = 0
    assert f(A, A, 8, 128, 128, 2, None, A, A, 1, A, None) == INV     # no codebook
    assert f(A, None, 8, 128, 128, 1, _cb(), A, A, 1, A, None) == INV
    assert f(A, A, 8, 128, 128, 1, _cb(), A, A, 1, M, None) == ALN
    assert f(A, A, 8, 1 << 25, 128, 5, _cb(), A, A, 1, A, None) == UNS   # K above 2^24
    assert f(A, A, 1 << 31, 128, 128, 1, _cb(), A, A, 1, A, None) == UNS  # N: 32-bit copy rows


def test_codebook_fit_validation(lib):
    assert lib.cq_codebook_fit(A, 100, 1, 10, A, None) == 1
    assert lib.cq_codebook_fit(A, 100, 17, 10, A, None) == 1
    assert lib.cq_codebook_fit(None, 100, 4, 10, A, None) == 1


def test_gemm_validation(lib):
    INV, ALN, UNS, WS = 1, 2, 3, 6
    f = lib.cq_gemm
    big = 1 << 30
    assert f(A, A, 256, 512, 128, 3, _cb(), A, A, 256, A, A, big, None) == UNS   # only b = 4
    assert f(A, A, 256, 512, 128, 5, _cb(), A, A, 256, A, A, big, None) == UNS   # ternary
    assert f(A, A, 256, 512, 128, 6, _cb(), A, A, 256, A, A, big, None) == INV
    assert f(A, A, 250, 512, 128, 4, _cb(), A, A, 256, A, A, big, None) == INV   # N % 16
    assert f(A, A, 256, 500, 128, 4, _cb(), A, A, 256, A, A, big, None) == INV   # K % 128
    assert f(A, A, 256, 512, 128, 4, _cb(), A, A, 0, A, A, big, None) == INV     # M = 0
    assert f(A, A, 256, 512, 128, 4, _cb(), A, A, 256, M, A, big, None) == ALN
    assert f(A, A, 256, 512, 128, 4, _cb(), A, A, 256, A, A, 100, None) == WS
    # 2^24 rows x 2^30 tokens: far more than 2^23 output tiles
    assert f(A, A, 1 << 24, 128, 128, 4, _cb(), A, A, 1 << 30, A, A, 1 << 40, None) == UNS
    assert cq.cq_gemm_workspace_bytes(300, 512) == (300 * 512 * 2 + 255) // 256 * 256
    # grouped: problems sharing an activation count it once
    probs = (cq.cq_gemm_problem * 3)()
    for i, (n, k, x) in enumerate([(256, 512, A), (128, 512, A), (512, 1536, A + 4096)]):
        probs[i].packed, probs[i].norms, probs[i].N, probs[i].K = A, A, n, k
        probs[i].Xq, probs[i].scale, probs[i].Y = x, A, A
    assert lib.cq_gemm_grouped_workspace_bytes(probs, 3, 512) == 512 * 512 * 2 + 512 * 1536 * 2
    assert lib.cq_gemm_grouped(probs, 3, 512, 128, 4, _cb(), A, 1000, None) == WS
    probs[1].K = 1024   # same Xq with a different K is rejected
    assert lib.cq_gemm_grouped(probs, 3, 512, 128, 4, _cb(), A, big, None) == INV


def test_q4_0_gemm_validation(lib):
    INV, ALN, UNS, WS = 1, 2, 3, 6
    f = lib.q4_0_gemm
    big = 1 << 30
    assert f(A, 64, 256, A, 0, A, A, big, None) == INV      # M = 0
    assert f(None, 64, 256, A, 4, A, A, big, None) == INV   # NULL
    assert f(A, 64, 312, A, 4, A, A, big, None) == UNS      # 10 blocks: not whole slabs
    assert f(A, 64, 257, A, 4, A, A, big, None) == UNS      # 9 blocks
    assert f(A, 64, 256, M, 4, A, A, big, None) == ALN
    assert f(A, 64, 256, A, 4, A, A + 16, big, None) == ALN  # workspace 256-byte alignment
    assert f(A, 64, 256, A, 4, A, A, 100, None) == WS
    # K = 250 pads to 256 columns: 8 blocks
    assert cq.q4_0_gemm_workspace_bytes(3, 250) == (3 * 256 * 2 + 255) // 256 * 256
    assert cq.q4_0_gemm_workspace_bytes(0, 256) == 0


def test_a8_groups_validation(lib):
    INV, ALN = 1, 2
    assert lib.a8_quantize_groups(A, 4, 100, 32, A, A, None) == INV        # G does not divide D
    assert lib.a8_quantize_groups(A, 4, 96, 48, A, A, None) == INV         # G not a multiple of 32
    assert lib.a8_quantize_groups(A, 4, 512, 512, A, A, None) == INV       # G above 256
    assert lib.a8_quantize_groups(A, 0, 96, 32, A, A, None) == INV
    assert lib.a8_quantize_groups(M, 4, 96, 32, A, A, None) == ALN
    assert lib.a8_fake_quant_groups(A, 4, 96, 32, None, None) == INV
    assert lib.a8_fake_quant_groups(A, 4, 96, 32, M, None) == ALN


def test_kernel_level_tables_match_oracle(lib):
    """The level table every CQ kernel receives (cq_levels, host only) equals the oracle's
    codebook_levels bit for bit for every code, including the fixed 1-bit +-sqrt(2/pi) and
    the ternary {-c, 0, +c} of the Needle mmap page (c: the three-level Lloyd-Max level)."""
    import numpy as np
    import oracle
    from util import fitted_cb28
    cb = fitted_cb28()
    for b in (1, 2, 3, 4, 5):
        want = oracle.codebook_levels(cb, b)
        got = np.array(cq.cq_levels(b, cb), dtype=np.float32)
        L = want.shape[0]
        assert got[:L].view(np.uint32).tolist() == want.view(np.uint32).tolist(), b
        assert not got[L:].any(), b
    assert cq.cq_levels(5) == cq.cq_levels(5, cb)          # the fixed codes ignore the table
    assert lib.cq_levels(6, None, A) == 1
    assert lib.cq_levels(2, None, A) == 1                   # b = 2..4 need the caller's table
    assert lib.cq_levels(1, None, None) == 1


def test_header_is_plain_c():
    """include/cqgemv.h is a C ABI: it compiles as strict C99 on its own."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                            "-fsyntax-only", "-x", "c", h], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def _cq_layer(entries):
    arr = (cq.cq_gemv_problem * len(entries))()
    for i, (packed, norms, N, K, X, Y) in enumerate(entries):
        arr[i].packed, arr[i].norms, arr[i].N, arr[i].K, arr[i].X, arr[i].Y = packed, norms, N, K, X, Y
    return arr


def _q4_layer(entries):
    arr = (cq.q4_0_gemv_problem * len(entries))()
    for i, (blocks, N, K, X, Y) in enumerate(entries):
        arr[i].blocks, arr[i].N, arr[i].K, arr[i].X, arr[i].Y = blocks, N, K, X, Y
    return arr


def test_layer_validation(lib):
    """The fused decode chain rejects every bad argument on the host, before any launch."""
    INV, ALN, UNS = 1, 2, 3
    f, q = lib.cq_gemv_layer, lib.q4_0_gemv_layer
    ok = (A, A, 8, 512, A, A)
    assert f(_cq_layer([ok]), 0, 128, 4, _cb(), 1, None) == INV              # no problem
    assert f(None, 1, 128, 4, _cb(), 1, None) == INV
    assert f(_cq_layer([ok]), 1, 64, 4, _cb(), 1, None) == INV               # g
    assert f(_cq_layer([ok]), 1, 128, 6, _cb(), 1, None) == INV              # code
    assert f(_cq_layer([ok]), 1, 128, 4, None, 1, None) == INV               # codebook
    assert f(_cq_layer([ok]), 1, 128, 4, _cb(), 0, None) == INV              # B
    assert f(_cq_layer([ok]), 1, 128, 4, _cb(), 3, None) == UNS              # B above 2
    assert f(_cq_layer([ok, (A, A, 8, 500, A, A)]), 2, 128, 4, _cb(), 1, None) == INV   # K % 128
    assert f(_cq_layer([ok, (A, A, 0, 512, A, A)]), 2, 128, 4, _cb(), 1, None) == INV   # N
    assert f(_cq_layer([ok, (A, None, 8, 512, A, A)]), 2, 128, 4, _cb(), 1, None) == INV
    assert f(_cq_layer([ok, (A, A, 8, 512, M, A)]), 2, 128, 4, _cb(), 1, None) == ALN
    assert f(_cq_layer([(A, A, 8, cq.LAYER_MAX_K + 128, A, A)]), 1, 128, 4, _cb(), 1, None) == UNS
    many = _cq_layer([ok] * (cq.LAYER_MAX_PROBLEMS + 1))
    assert f(many, cq.LAYER_MAX_PROBLEMS + 1, 128, 4, _cb(), 1, None) == UNS
    okq = (A, 8, 312, A, A)
    assert q(_q4_layer([okq]), 0, 1, None) == INV
    assert q(_q4_layer([okq]), 1, 3, None) == UNS
    assert q(_q4_layer([okq, (A, 8, 0, A, A)]), 2, 1, None) == INV             # K
    assert q(_q4_layer([okq, (None, 8, 312, A, A)]), 2, 1, None) == INV
    assert q(_q4_layer([okq, (A, 8, 312, A, M)]), 2, 1, None) == ALN
    assert q(_q4_layer([(A, 8, cq.LAYER_MAX_K + 1, A, A)]), 1, 1, None) == UNS
