"""CPU oracle for the CQ-WxA8 and Q4_0 low-bit GEMV / GEMM path.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
anything in this package.  The CUDA library (``gemm_cq_gemv_gb300``) never imports it,
and this package never imports the CUDA library: the two share no code, no tables and
no constant generators.  Seeded inputs come from ``gemm_cq_gemv_gb300.synth``, a module
that holds no arithmetic of the method.

Everything here is plain NumPy in float64 (float32 / float16 only where the pages fix
that precision: the fp16 group norm, the fp16 Q4_0 block scale, the fp32 int8 scale),
slow and written to be checked against the pages by eye.

Sources (cited by title and section; the pages are Chinese-language web articles):

* [CACT]  "14MB 装下 45M 参数：拆解 Needle 的 .cact 单文件与 W4A8 量化魔法",
          §一 (CQ codebook quantization: groups of 128, normalised Walsh-Hadamard
          rotation, nearest Lloyd-Max codeword, FP16 L2 norm, reconstruction
          ``w_group = (codebook_bits[idx] * norm) H``, 400k samples / 200 iterations,
          ``cb2[4] | cb3[8] | cb4[16]``, LSB-first nibble packing, low nibble = even
          column, ``WEIGHT_BITS 4 / ACT_BITS 8``), §三 (weights pre-transposed to
          ``[out, in]``) and §四 (int8 KV cache, per-head A8 query quantization and KV
          fake-quant, one 4-byte scale per ``KV_GROUP = 32`` values).
* [MMAP]  "免解析加载的秘诀：mmap 直读张量与 Needle 的秒级冷启动",
          section "mmap 之下张量按偏移直读" (groups of 128, the same reconstruction,
          the analytic 1-bit codebook ``{-sqrt(2/pi), +sqrt(2/pi)}`` and the ternary
          ``{-c, 0, c}`` of bits = 5, both hard-coded in the engine).
* [KMCU]  Minueza-32M -> KMCU v1 conversion page (pnsm.cn, MCU series),
          §1 (model shapes), §2 "Q4_0 量化" (32-weight blocks, fp16 ``d = max_abs/8``,
          ``q = clip(rint(w/d), -8, 7)``, nibble = q + 8, low nibble = even index,
          18 bytes / 32 weights) and §3 "行对齐到 32" (rows zero-padded to 32).

Where the pages are silent or garbled the reading taken is stated in the docstring of
the function that depends on it.

Parity pins: every function here is checked by ``tests/test_oracle_*.py`` against
values the pages or the mathematics fix (closed forms, textbook Lloyd-Max tables,
brute force, hand-worked fixtures in ``tests/golden/``), never against itself.
No function in this package is "parity unpinned".
"""

from .hadamard import sylvester_hadamard, fwht_butterfly
from .lloyd_max import (lloyd_max_gaussian_fit, gaussian_quantile_init, ONE_BIT_LEVEL,
                        TERNARY_LEVEL, ternary_gaussian_level)
from .cq import (
    GROUP,
    TERNARY,
    field_bits,
    codebook_levels,
    codebook_concat,
    pack_indices,
    unpack_indices,
    cq_encode,
    cq_reconstruct,
)
from .a8 import a8_quantize, a8_dequantize, a8_quantize_groups, a8_fake_quant_groups
from .q4_0 import q4_0_quantize, q4_0_dequantize, q4_0_row_bytes, Q4_0_BLOCK, Q4_0_BLOCK_BYTES
from .products import cq_gemv_ref, cq_gemm_ref, q4_0_gemv_ref

__all__ = [
    "sylvester_hadamard", "fwht_butterfly",
    "lloyd_max_gaussian_fit", "gaussian_quantile_init", "ONE_BIT_LEVEL",
    "TERNARY_LEVEL", "ternary_gaussian_level",
    "GROUP", "TERNARY", "field_bits", "codebook_levels", "codebook_concat", "pack_indices", "unpack_indices",
    "cq_encode", "cq_reconstruct",
    "a8_quantize", "a8_dequantize", "a8_quantize_groups", "a8_fake_quant_groups",
    "q4_0_quantize", "q4_0_dequantize", "q4_0_row_bytes", "Q4_0_BLOCK", "Q4_0_BLOCK_BYTES",
    "cq_gemv_ref", "cq_gemm_ref", "q4_0_gemv_ref",
]
