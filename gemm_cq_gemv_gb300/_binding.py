"""ctypes binding of ``libcqgemv.so`` (argument marshalling only).

Every function here has the name of the C entry point it calls (``include/cqgemv.h``),
takes CUDA tensors, checks dtype / device / contiguity / shape, passes raw device
pointers and sizes across the C ABI and raises ``CQError`` on a non-OK status.  All
arithmetic runs in the library's CUDA kernels; there is no fallback of any kind: if
the shared library is missing or does not load, every call raises.
"""

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcqgemv.so")

CQ_OK = 0
_STATUS = {0: "CQ_OK", 1: "CQ_ERR_INVALID_ARG", 2: "CQ_ERR_ALIGNMENT", 3: "CQ_ERR_UNSUPPORTED",
           4: "CQ_ERR_CUDA", 5: "CQ_ERR_DEVICE_TIMEOUT", 6: "CQ_ERR_WORKSPACE"}


class CQError(RuntimeError):
    def __init__(self, fn, status, cuda_err=0):
        name = _STATUS.get(status, f"status {status}")
        msg = f"{fn} failed: {name}"
        if status == 4:
            msg += f" (cudaError {cuda_err})"
        super().__init__(msg)
        self.status = status


class cq_codebook(ctypes.Structure):
    _fields_ = [("cb", ctypes.c_float * 28)]


class cq_gemm_problem(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("norms", ctypes.c_void_p), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("Xq", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("Y", ctypes.c_void_p)]


class cq_gemv_problem(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("norms", ctypes.c_void_p), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("X", ctypes.c_void_p), ("Y", ctypes.c_void_p)]


class q4_0_gemv_problem(ctypes.Structure):
    _fields_ = [("blocks", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("X", ctypes.c_void_p), ("Y", ctypes.c_void_p)]


LAYER_MAX_PROBLEMS = 16   # CQ_LAYER_MAX_PROBLEMS
LAYER_MAX_K = 8192        # CQ_LAYER_MAX_K

_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_SZ = ctypes.c_size_t

# name -> (restype, argtypes)
SIGNATURES = {
    "cq_status_string": (ctypes.c_char_p, [_INT]),
    "cq_last_cuda_error": (_INT, []),
    "cq_abi_version": (_INT, []),
    "cq_levels": (_INT, [_INT, ctypes.POINTER(cq_codebook), _P]),
    "cq_codebook_fit": (_INT, [_P, _I64, _INT, _INT, _P, _P]),
    "cq_encode": (_INT, [_P, _I64, _I64, _INT, _INT, ctypes.POINTER(cq_codebook), _P, _P, _P]),
    "a8_quantize": (_INT, [_P, _I64, _I64, _P, _P, _P]),
    "a8_quantize_groups": (_INT, [_P, _I64, _I64, _INT, _P, _P, _P]),
    "a8_fake_quant_groups": (_INT, [_P, _I64, _I64, _INT, _P, _P]),
    "cq_gemv_workspace_bytes": (_SZ, [_I64, _I64]),
    "cq_gemv": (_INT, [_P, _P, _I64, _I64, _INT, _INT, ctypes.POINTER(cq_codebook), _P, _P, _I64,
                       _P, _P, _SZ, _P]),
    "cq_gemv_noalloc": (_INT, [_P, _P, _I64, _I64, _INT, _INT, ctypes.POINTER(cq_codebook), _P,
                               _P, _I64, _P, _P]),
    "cq_gemv_lut": (_INT, [_P, _P, _I64, _I64, _INT, _INT, ctypes.POINTER(cq_codebook), _P, _P,
                           _I64, _P, _P]),
    "cq_gemm_workspace_bytes": (_SZ, [_I64, _I64]),
    "cq_gemm": (_INT, [_P, _P, _I64, _I64, _INT, _INT, ctypes.POINTER(cq_codebook), _P, _P, _I64,
                       _P, _P, _SZ, _P]),
    "cq_gemm_grouped_workspace_bytes": (_SZ, [ctypes.POINTER(cq_gemm_problem), _INT, _I64]),
    "cq_gemm_grouped": (_INT, [ctypes.POINTER(cq_gemm_problem), _INT, _I64, _INT, _INT,
                               ctypes.POINTER(cq_codebook), _P, _SZ, _P]),
    "cq_device_error": (_INT, [_P]),
    "cq_probe_bounded_wait": (_INT, [ctypes.c_uint64, _P]),
    "q4_0_quantize": (_INT, [_P, _I64, _I64, _P, _P]),
    "q4_0_gemv": (_INT, [_P, _I64, _I64, _P, _I64, _P, _P]),
    "q4_0_gemm_workspace_bytes": (_SZ, [_I64, _I64]),
    "q4_0_gemm": (_INT, [_P, _I64, _I64, _P, _I64, _P, _P, _SZ, _P]),
    "cq_gemv_layer": (_INT, [ctypes.POINTER(cq_gemv_problem), _INT, _INT, _INT,
                             ctypes.POINTER(cq_codebook), _I64, _P]),
    "q4_0_gemv_layer": (_INT, [ctypes.POINTER(q4_0_gemv_problem), _INT, _I64, _P]),
}


def lib():
    """Load ``libcqgemv.so`` (once).  Raises if it is missing: nothing runs without it."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                "g.build()\"` (nvcc, sm_103a). There is no fallback implementation.")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t, dtype, name, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")
    return ctypes.c_void_p(t.data_ptr())


def _check(fn, status):
    if status != CQ_OK:
        raise CQError(fn, status, lib().cq_last_cuda_error())


def make_codebook(cb28):
    """Build the C ``cq_codebook`` from 28 floats (``cb2 | cb3 | cb4``)."""
    vals = [float(v) for v in (cb28.tolist() if hasattr(cb28, "tolist") else cb28)]
    if len(vals) != 28:
        raise ValueError("codebook needs 28 floats (cb2[4] | cb3[8] | cb4[16])")
    c = cq_codebook()
    for i, v in enumerate(vals):
        c.cb[i] = v
    return c


def _cbk(cb):
    return cb if isinstance(cb, cq_codebook) else make_codebook(cb)


def cq_status_string(status: int) -> str:
    return lib().cq_status_string(status).decode()


def cq_abi_version() -> int:
    return lib().cq_abi_version()


def cq_levels(b, cb=None):
    """The 16-entry float32 level table the CQ kernels use for code ``b`` (host only), as a
    list of 16 Python floats (each exactly a float32 value)."""
    out = (ctypes.c_float * 16)()
    c = ctypes.byref(_cbk(cb)) if cb is not None else None
    _check("cq_levels", lib().cq_levels(b, c, ctypes.cast(out, ctypes.c_void_p)))
    return list(out)


def cq_codebook_fit(samples, L, iters=200, levels_out=None, stream=None):
    """A1: Lloyd-Max levels (float32 [L]) from float64 samples on the GPU."""
    s = _ptr(samples, torch.float64, "samples")
    if levels_out is None:
        levels_out = torch.empty(L, dtype=torch.float32, device=samples.device)
    _check("cq_codebook_fit", lib().cq_codebook_fit(s, samples.numel(), L, iters,
                                                     _ptr(levels_out, torch.float32, "levels_out"),
                                                     _stream(stream)))
    return levels_out


# CQ_TERNARY of the C header: bits = 5 selects the fixed codebook {-c, 0, +c}, whose
# indices are stored in 2-bit fields.
CQ_TERNARY = 5


def cq_field_bits(b: int) -> int:
    """Bits of one packed index field of code ``b`` (a group holds ``16 * field`` bytes)."""
    return 2 if b == CQ_TERNARY else b


def cq_encode(W, b, cb, packed=None, norms=None, g=128, stream=None):
    """A2: CQ-encode W [N, K] float32 -> (packed uint8 [N, K/128, 16 f], norms int16 [N, K/128]),
    f = ``cq_field_bits(b)``."""
    N, K = W.shape
    wp = _ptr(W, torch.float32, "W", 2)
    if packed is None:
        packed = torch.empty((N, K // 128, 16 * cq_field_bits(b)), dtype=torch.uint8, device=W.device)
    if norms is None:
        norms = torch.empty((N, K // 128), dtype=torch.int16, device=W.device)
    c = _cbk(cb)
    _check("cq_encode", lib().cq_encode(wp, N, K, g, b, ctypes.byref(c),
                                        _ptr(packed, torch.uint8, "packed"),
                                        _ptr(norms, torch.int16, "norms"), _stream(stream)))
    return packed, norms


def a8_quantize(X, Xq=None, scale=None, stream=None):
    """A3: X [B, K] float32 -> (Xq int8 [B, K], scale float32 [B])."""
    B, K = X.shape
    xp = _ptr(X, torch.float32, "X", 2)
    if Xq is None:
        Xq = torch.empty((B, K), dtype=torch.int8, device=X.device)
    if scale is None:
        scale = torch.empty((B,), dtype=torch.float32, device=X.device)
    _check("a8_quantize", lib().a8_quantize(xp, B, K, _ptr(Xq, torch.int8, "Xq"),
                                            _ptr(scale, torch.float32, "scale"), _stream(stream)))
    return Xq, scale


def a8_quantize_groups(X, G, codes=None, scales=None, stream=None):
    """Grouped A8: X [T, D] float32 -> (codes int8 [T, D], scales float32 [T, D/G])."""
    T, D = X.shape
    if codes is None:
        codes = torch.empty((T, D), dtype=torch.int8, device=X.device)
    if scales is None:
        scales = torch.empty((T, D // G), dtype=torch.float32, device=X.device)
    _check("a8_quantize_groups", lib().a8_quantize_groups(_ptr(X, torch.float32, "X", 2), T, D, G,
                                                          _ptr(codes, torch.int8, "codes"),
                                                          _ptr(scales, torch.float32, "scales"),
                                                          _stream(stream)))
    return codes, scales


def a8_fake_quant_groups(X, G, Y=None, stream=None):
    """Grouped A8 fake-quant: Y [T, D] float32 = q * s per group of G features."""
    T, D = X.shape
    if Y is None:
        Y = torch.empty((T, D), dtype=torch.float32, device=X.device)
    _check("a8_fake_quant_groups", lib().a8_fake_quant_groups(_ptr(X, torch.float32, "X", 2), T, D, G,
                                                              _ptr(Y, torch.float32, "Y"), _stream(stream)))
    return Y


def cq_gemv_workspace_bytes(B, K) -> int:
    return int(lib().cq_gemv_workspace_bytes(B, K))


def cq_gemv(packed, norms, N, K, b, cb, Xq, scale, Y=None, workspace=None, g=128, stream=None):
    """A4+A5: Y [B, N] float32 = decode GEMV of CQ weights with int8 activations."""
    B = Xq.shape[0]
    if Y is None:
        Y = torch.empty((B, N), dtype=torch.float32, device=Xq.device)
    need = cq_gemv_workspace_bytes(B, K)
    if workspace is None:
        workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=Xq.device)
    c = _cbk(cb)
    _check("cq_gemv", lib().cq_gemv(_ptr(packed, torch.uint8, "packed"),
                                    _ptr(norms, torch.int16, "norms"), N, K, g, b, ctypes.byref(c),
                                    _ptr(Xq, torch.int8, "Xq"), _ptr(scale, torch.float32, "scale"),
                                    B, _ptr(Y, torch.float32, "Y"),
                                    _ptr(workspace, torch.uint8, "workspace"),
                                    workspace.numel(), _stream(stream)))
    return Y


def cq_gemv_lut(packed, norms, N, K, b, cb, Xq, scale, Y=None, g=128, stream=None):
    """A4+A5 by table lookup (b = 1, 2 or ternary): Y [B, N] float32, no workspace."""
    B = Xq.shape[0]
    if Y is None:
        Y = torch.empty((B, N), dtype=torch.float32, device=Xq.device)
    c = _cbk(cb)
    _check("cq_gemv_lut", lib().cq_gemv_lut(_ptr(packed, torch.uint8, "packed"),
                                            _ptr(norms, torch.int16, "norms"), N, K, g, b,
                                            ctypes.byref(c), _ptr(Xq, torch.int8, "Xq"),
                                            _ptr(scale, torch.float32, "scale"), B,
                                            _ptr(Y, torch.float32, "Y"), _stream(stream)))
    return Y


def cq_gemm_workspace_bytes(M, K) -> int:
    return int(lib().cq_gemm_workspace_bytes(M, K))


def cq_gemm(packed, norms, N, K, b, cb, Xq, scale, Y=None, workspace=None, g=128, stream=None):
    """A4+A6: Y [M, N] bfloat16 = prefill GEMM of CQ weights with int8 activations."""
    M = Xq.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=Xq.device)
    need = cq_gemm_workspace_bytes(M, K)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=Xq.device)
    c = _cbk(cb)
    _check("cq_gemm", lib().cq_gemm(_ptr(packed, torch.uint8, "packed"),
                                    _ptr(norms, torch.int16, "norms"), N, K, g, b, ctypes.byref(c),
                                    _ptr(Xq, torch.int8, "Xq"), _ptr(scale, torch.float32, "scale"),
                                    M, _ptr(Y, torch.bfloat16, "Y"),
                                    _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
                                    _stream(stream)))
    return Y


def make_gemm_problems(items):
    """``items``: sequence of (packed, norms, N, K, Xq, scale, Y) tensors / ints."""
    arr = (cq_gemm_problem * len(items))()
    for i, (packed, norms, N, K, Xq, scale, Y) in enumerate(items):
        arr[i].packed = _ptr(packed, torch.uint8, "packed").value
        arr[i].norms = _ptr(norms, torch.int16, "norms").value
        arr[i].N, arr[i].K = N, K
        arr[i].Xq = _ptr(Xq, torch.int8, "Xq").value
        arr[i].scale = _ptr(scale, torch.float32, "scale").value
        arr[i].Y = _ptr(Y, torch.bfloat16, "Y").value
    return arr


def make_gemv_layer(items):
    """CQ layer problems from (packed, norms, N, K, X, Y) tuples: X [B][K] float32 and
    Y [B][N] float32 CUDA tensors.  The array keeps the tensors alive."""
    arr = (cq_gemv_problem * len(items))()
    for i, (packed, norms, N, K, X, Y) in enumerate(items):
        arr[i].packed = _ptr(packed, torch.uint8, "packed").value
        arr[i].norms = _ptr(norms, torch.int16, "norms").value
        arr[i].N, arr[i].K = N, K
        arr[i].X = _ptr(X, torch.float32, "X", 2).value
        arr[i].Y = _ptr(Y, torch.float32, "Y", 2).value
        if X.shape[1] != K or Y.shape != (X.shape[0], N):
            raise ValueError(f"problem {i}: X must be [B, {K}] and Y [B, {N}]")
    arr._keep = [t for it in items for t in it if isinstance(t, torch.Tensor)]
    arr._batch = items[0][4].shape[0]
    return arr


def make_q4_0_layer(items):
    """Q4_0 layer problems from (blocks, N, K, X, Y) tuples (X, Y as for make_gemv_layer)."""
    arr = (q4_0_gemv_problem * len(items))()
    for i, (blocks, N, K, X, Y) in enumerate(items):
        arr[i].blocks = _ptr(blocks, torch.uint8, "blocks").value
        arr[i].N, arr[i].K = N, K
        arr[i].X = _ptr(X, torch.float32, "X", 2).value
        arr[i].Y = _ptr(Y, torch.float32, "Y", 2).value
        if X.shape[1] != K or Y.shape != (X.shape[0], N):
            raise ValueError(f"problem {i}: X must be [B, {K}] and Y [B, {N}]")
    arr._keep = [t for it in items for t in it if isinstance(t, torch.Tensor)]
    arr._batch = items[0][3].shape[0]
    return arr


def cq_gemv_layer(problems, b, cb, g=128, stream=None):
    """Fused decode chain: a8 quantization, rotation and the CQ GEMV of every problem of a
    layer (an array from ``make_gemv_layer``) in one launch."""
    c = _cbk(cb)
    _check("cq_gemv_layer", lib().cq_gemv_layer(problems, len(problems), g, b, ctypes.byref(c),
                                                problems._batch, _stream(stream)))


def q4_0_gemv_layer(problems, stream=None):
    """Fused decode chain: the Q4_0 GEMV of every problem of a layer (an array from
    ``make_q4_0_layer``) in one launch."""
    _check("q4_0_gemv_layer", lib().q4_0_gemv_layer(problems, len(problems), problems._batch,
                                                    _stream(stream)))


def cq_gemm_grouped_workspace_bytes(problems, M) -> int:
    return int(lib().cq_gemm_grouped_workspace_bytes(problems, len(problems), M))


def cq_gemm_grouped(problems, M, b, cb, workspace=None, g=128, stream=None, device=None):
    """A6 grouped: every problem (a ``cq_gemm_problem`` array) in persistent launches."""
    need = cq_gemm_grouped_workspace_bytes(problems, M)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8,
                                device=device or torch.device("cuda"))
    c = _cbk(cb)
    _check("cq_gemm_grouped", lib().cq_gemm_grouped(problems, len(problems), M, g, b,
                                                    ctypes.byref(c),
                                                    _ptr(workspace, torch.uint8, "workspace"),
                                                    workspace.numel(), _stream(stream)))
    return workspace


def cq_device_error(stream=None):
    """Raise CQError(CQ_ERR_DEVICE_TIMEOUT) if a bounded device wait gave up (clears it)."""
    _check("cq_device_error", lib().cq_device_error(_stream(stream)))


def cq_probe_bounded_wait(timeout_ns=20_000_000, stream=None):
    """Enqueue the failure-detection probe (bounded waits that nothing completes)."""
    _check("cq_probe_bounded_wait", lib().cq_probe_bounded_wait(int(timeout_ns), _stream(stream)))


NOALLOC_MAX_ELEMS = 1 << 20   # CQ_GEMV_NOALLOC_MAX_ELEMS


def cq_gemv_noalloc(packed, norms, N, K, b, cb, Xq, scale, Y=None, g=128, stream=None):
    """``cq_gemv`` for callers that cannot allocate a workspace: the library's fixed
    4 MiB scratch holds the rotated activations (B * K <= 2**20).  Calls that overlap on
    the GPU share that scratch and race; the first call on a device must precede any
    stream capture.  ``Y`` may be passed preallocated."""
    B = Xq.shape[0]
    if Y is None:
        Y = torch.empty((B, N), dtype=torch.float32, device=Xq.device)
    c = _cbk(cb)
    _check("cq_gemv_noalloc", lib().cq_gemv_noalloc(
        _ptr(packed, torch.uint8, "packed"), _ptr(norms, torch.int16, "norms"), N, K, g, b,
        ctypes.byref(c), _ptr(Xq, torch.int8, "Xq"), _ptr(scale, torch.float32, "scale"), B,
        _ptr(Y, torch.float32, "Y"), _stream(stream)))
    return Y


def q4_0_quantize(W, blocks=None, stream=None):
    """A7: W [N, K] float32 -> Q4_0 blocks uint8 [N, ceil(K/32)*18]."""
    N, K = W.shape
    if blocks is None:
        blocks = torch.empty((N, ((K + 31) // 32) * 18), dtype=torch.uint8, device=W.device)
    _check("q4_0_quantize", lib().q4_0_quantize(_ptr(W, torch.float32, "W", 2), N, K,
                                                _ptr(blocks, torch.uint8, "blocks"), _stream(stream)))
    return blocks


def q4_0_gemv(blocks, N, K, X, Y=None, stream=None):
    """A8: Y [B, N] float32 = Q4_0 decode GEMV with float32 activations X [B, K]."""
    B = X.shape[0]
    if Y is None:
        Y = torch.empty((B, N), dtype=torch.float32, device=X.device)
    _check("q4_0_gemv", lib().q4_0_gemv(_ptr(blocks, torch.uint8, "blocks"), N, K,
                                        _ptr(X, torch.float32, "X"), B, _ptr(Y, torch.float32, "Y"),
                                        _stream(stream)))
    return Y


def q4_0_gemm_workspace_bytes(M, K) -> int:
    return int(lib().q4_0_gemm_workspace_bytes(M, K))


def q4_0_gemm(blocks, N, K, X, Y=None, workspace=None, stream=None):
    """Q4_0 GEMM on the tensor cores: Y [M, N] float32 for float32 activations X [M, K]
    (ceil(K/32) a multiple of 8)."""
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=X.device)
    need = q4_0_gemm_workspace_bytes(M, K)
    if workspace is None:
        workspace = torch.empty((max(need, 256),), dtype=torch.uint8, device=X.device)
    _check("q4_0_gemm", lib().q4_0_gemm(_ptr(blocks, torch.uint8, "blocks"), N, K,
                                        _ptr(X, torch.float32, "X"), M, _ptr(Y, torch.float32, "Y"),
                                        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
                                        _stream(stream)))
    return Y
