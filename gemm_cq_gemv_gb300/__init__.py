"""GB300 (sm_103a) low-bit GEMV / GEMM: CQ-WxA8 and Q4_0.

The compute lives in ``libcqgemv.so`` (hand-written CUDA, C ABI in
``include/cqgemv.h``); this package is a thin ctypes binding with the same function
names plus the seeded input generators in ``synth``.  Loading is lazy; the first call
raises if the shared library has not been built.
"""

from ._binding import (CQError, CQ_TERNARY, LIB_PATH, NOALLOC_MAX_ELEMS, SIGNATURES, a8_quantize, cq_abi_version,
                       cq_codebook, cq_codebook_fit, cq_encode, cq_gemv, cq_gemv_noalloc,
                       cq_gemv_workspace_bytes,
                       cq_status_string, lib, make_codebook, q4_0_gemv, q4_0_quantize,
                       cq_gemm, cq_gemm_grouped, cq_gemm_grouped_workspace_bytes,
                       cq_gemm_problem, cq_gemm_workspace_bytes, cq_device_error,
                       make_gemm_problems, q4_0_gemm, q4_0_gemm_workspace_bytes,
                       cq_probe_bounded_wait, a8_quantize_groups, a8_fake_quant_groups,
                       cq_field_bits, cq_levels, cq_gemv_lut, cq_gemv_problem, q4_0_gemv_problem,
                       make_gemv_layer, make_q4_0_layer, cq_gemv_layer, q4_0_gemv_layer,
                       LAYER_MAX_PROBLEMS, LAYER_MAX_K)

__all__ = ["CQError", "CQ_TERNARY", "LIB_PATH", "NOALLOC_MAX_ELEMS", "SIGNATURES", "a8_quantize", "cq_abi_version", "cq_codebook",
           "cq_codebook_fit", "cq_encode", "cq_gemv", "cq_gemv_noalloc", "cq_gemv_workspace_bytes",
           "cq_status_string", "lib", "make_codebook", "q4_0_gemv", "q4_0_quantize",
           "cq_gemm", "cq_gemm_grouped", "cq_gemm_grouped_workspace_bytes", "cq_gemm_problem",
           "cq_gemm_workspace_bytes", "cq_device_error", "make_gemm_problems", "q4_0_gemm",
           "q4_0_gemm_workspace_bytes", "cq_probe_bounded_wait", "a8_quantize_groups",
           "a8_fake_quant_groups", "cq_field_bits", "cq_levels", "cq_gemv_lut", "cq_gemv_problem",
           "q4_0_gemv_problem", "make_gemv_layer", "make_q4_0_layer", "cq_gemv_layer",
           "q4_0_gemv_layer", "LAYER_MAX_PROBLEMS", "LAYER_MAX_K"]
