"""CQ ("Cactus Quant") weight encoding and reconstruction ([CACT] §一, §三; [MMAP]).

What the pages fix:
  * matmul weights are stored pre-transposed ``[out, in]``; quant groups of 128 run
    along ``in`` (the reduction axis);
  * each group is rotated by a normalised Walsh-Hadamard transform, every rotated
    coordinate is matched to the nearest Lloyd-Max Gaussian codeword, only the indices
    and the group's L2 norm (FP16) are kept;
  * reconstruction ``w_group = (codebook_bits[idx] * norm) @ H``, H the normalised WHT;
  * codebooks ``cb2[4] | cb3[8] | cb4[16]`` concatenated, indexed by bit width; the
    1-bit codebook is ``{-sqrt(2/pi), +sqrt(2/pi)}`` and the ternary one (bits = 5)
    ``{-c, 0, +c}``, both hard-coded, no table ([MMAP]);
  * indices are packed LSB-first, the low nibble holding the even column.

Readings taken (the pages are silent or inconsistent):
  * codewords are in N(0,1) units and the "unit sphere" scaling is a factor 1/sqrt(g)
    on the codewords, so ``W_hat_g = (cb[idx] * norm / sqrt(g)) @ (Hu / sqrt(g))``;
    this is the only reading under which "L2 norm stored", "scaled to the unit sphere"
    and the N(0,1)-unit 1-bit value +-sqrt(2/pi) all hold;
  * the encoder matches ``v = (Hu @ w) / ||w||`` against the codewords (the same
    comparison as ``H w / ||w||`` against ``cb / sqrt(g)``, with sqrt(g) removed from
    both sides);
  * decisions in IEEE float64 without fused multiply-add: ``Hu @ w`` by natural-order
    butterflies, ``||w||^2`` summed sequentially in index order, one correctly rounded
    square root, one division per coordinate, distances ``|v - cb[t]|``;
  * ties go to the lowest index; a zero group (norm 0) gets index 0 everywhere and a
    +0 norm;
  * norm rounding: float64 -> float16 in one round-to-nearest-even step;
  * packing for b < 4 (the pages only describe nibbles): a dense LSB-first bit stream
    per group, index i in bits [b*i, b*i + b) of the group's little-endian bytes, so a
    group is 16*b bytes; for b = 4 this is exactly "low nibble = even column";
  * norms are a separate ``[N, K/g]`` float16 array;
  * ternary (bits = 5): ``c`` is the three-level Lloyd-Max Gaussian level (see
    ``lloyd_max.ternary_gaussian_level``), the levels ``[-c, 0, +c]`` take indices
    0, 1, 2, and an index is stored in a 2-bit field of the same LSB-first stream (the
    smallest field that holds three values, and the ternary layout the smolmaxxing page
    chooses over base-3 packing for speed, kernel table E76/E77), so a group is 32 bytes.
"""

import numpy as np

from .hadamard import fwht_butterfly, sylvester_hadamard
from .lloyd_max import ONE_BIT_LEVEL, TERNARY_LEVEL

GROUP = 128  # [CACT] §一: "每个 group 默认 128 维"; [MMAP]: "按 128 的 group 切块"
TERNARY = 5  # [MMAP]: the bits value of the ternary codebook


def field_bits(b: int) -> int:
    """Bits of one packed index of code ``b``: ``b``, or 2 for the ternary code."""
    return 2 if b == TERNARY else b

_CB_OFFSETS = {2: (0, 4), 3: (4, 12), 4: (12, 28)}


def codebook_concat(cb2, cb3, cb4) -> np.ndarray:
    """The 28-float header table ``cb2[4] | cb3[8] | cb4[16]`` ([CACT] §一)."""
    out = np.concatenate([np.asarray(cb2, np.float32), np.asarray(cb3, np.float32),
                          np.asarray(cb4, np.float32)])
    if out.shape != (28,):
        raise ValueError("codebook table must hold 4 + 8 + 16 levels")
    return out


def codebook_levels(cb28: np.ndarray, b: int) -> np.ndarray:
    """Levels for bit width ``b`` as float32, ascending.

    b = 1 ignores the table and uses the analytic +-sqrt(2/pi); b = 5 (ternary) the
    fixed ``[-c, 0, +c]`` ([MMAP]).
    """
    if b == 1:
        c = np.float32(ONE_BIT_LEVEL)
        return np.array([-c, c], dtype=np.float32)
    if b == TERNARY:
        c = np.float32(TERNARY_LEVEL)
        return np.array([-c, 0.0, c], dtype=np.float32)
    if b not in _CB_OFFSETS:
        raise ValueError("CQ bit width must be 1..4, or 5 (ternary)")
    lo, hi = _CB_OFFSETS[b]
    return np.asarray(cb28, dtype=np.float32)[lo:hi].copy()


def pack_indices(idx: np.ndarray, b: int) -> np.ndarray:
    """Pack ``[..., 128]`` indices into ``[..., 16*b]`` bytes, LSB-first bit stream.

    Index i occupies bits [b*i, b*i + b) of the group's little-endian byte string.
    """
    idx = np.asarray(idx)
    g = idx.shape[-1]
    nbytes = g * b // 8
    lead = idx.shape[:-1]
    flat = idx.reshape(-1, g).astype(np.int64)
    out = np.zeros((flat.shape[0], nbytes), dtype=np.int64)
    for i in range(g):
        for bit in range(b):
            pos = b * i + bit
            out[:, pos // 8] |= ((flat[:, i] >> bit) & 1) << (pos % 8)
    return out.astype(np.uint8).reshape(lead + (nbytes,))


def unpack_indices(packed: np.ndarray, b: int, g: int = GROUP) -> np.ndarray:
    """Inverse of :func:`pack_indices`: ``[..., 16*b]`` bytes -> ``[..., g]`` indices."""
    packed = np.asarray(packed, dtype=np.uint8)
    lead = packed.shape[:-1]
    flat = packed.reshape(-1, packed.shape[-1]).astype(np.int64)
    out = np.zeros((flat.shape[0], g), dtype=np.int64)
    for i in range(g):
        for bit in range(b):
            pos = b * i + bit
            out[:, i] |= ((flat[:, pos // 8] >> (pos % 8)) & 1) << bit
    return out.reshape(lead + (g,))


def _encode_groups(wg: np.ndarray, levels: np.ndarray):
    """Encode rows of ``wg`` (``[G, 128]`` float32) -> (idx ``[G,128]``, norm f64 ``[G]``)."""
    w = wg.astype(np.float64)
    g = w.shape[1]
    # Rotation Hu @ w, natural-order butterflies in float64.
    r = fwht_butterfly(w)
    # ||w||^2 summed sequentially in index order, one rounding per multiply and add.
    acc = np.zeros(w.shape[0], dtype=np.float64)
    for i in range(g):
        sq = w[:, i] * w[:, i]
        acc = acc + sq
    n = np.sqrt(acc)
    idx = np.zeros(w.shape, dtype=np.int64)
    nz = n > 0.0
    if np.any(nz):
        v = r[nz] / n[nz][:, None]
        lv = levels.astype(np.float64)
        dist = np.abs(v[:, :, None] - lv[None, None, :])
        idx[nz] = np.argmin(dist, axis=2)  # first minimum = lowest index on ties
    return idx, n


def cq_encode(W: np.ndarray, b: int, cb28: np.ndarray, g: int = GROUP):
    """CQ-encode ``W`` (``[N, K]`` float32, ``[out, in]``) at ``b`` bits.

    Returns ``(packed, norms)``: ``packed`` uint8 ``[N, K/g, 16*f]`` (``f`` =
    ``field_bits(b)``) and ``norms`` uint16 ``[N, K/g]`` holding the IEEE float16 bits of
    each group's L2 norm.
    """
    W = np.asarray(W, dtype=np.float32)
    if g != GROUP:
        raise ValueError("group size is 128")
    N, K = W.shape
    if K % g != 0:
        raise ValueError("K must be a multiple of the group size")
    levels = codebook_levels(cb28, b)
    G = K // g
    flat = W.reshape(N * G, g)
    idx = np.empty((N * G, g), dtype=np.int64)
    n = np.empty(N * G, dtype=np.float64)
    for c0 in range(0, N * G, 8192):          # chunks only bound host memory
        idx[c0:c0 + 8192], n[c0:c0 + 8192] = _encode_groups(flat[c0:c0 + 8192], levels)
    norms16 = n.astype(np.float16).view(np.uint16).reshape(N, G)
    f = field_bits(b)
    packed = pack_indices(idx, f).reshape(N, G, 16 * f)
    return packed, norms16


def cq_reconstruct(packed: np.ndarray, norms16: np.ndarray, b: int, cb28: np.ndarray,
                   g: int = GROUP) -> np.ndarray:
    """Dequantised weights ``W_hat`` (``[N, K]`` float64) by the page's formula.

    Per group: ``w = (cb[idx] * norm / sqrt(g)) @ H`` with the dense normalised
    Sylvester ``H = Hu / sqrt(g)``.
    """
    packed = np.asarray(packed, dtype=np.uint8)
    N, G, _ = packed.shape
    levels = codebook_levels(cb28, b).astype(np.float64)
    idx = unpack_indices(packed, field_bits(b), g)             # [N, G, g]
    norm = np.asarray(norms16, dtype=np.uint16).view(np.float16).astype(np.float64)
    H = sylvester_hadamard(g) / np.sqrt(float(g))
    unit = levels[idx] / np.sqrt(float(g))                    # codewords on the unit sphere
    scaled = unit * norm[:, :, None]
    w = scaled.reshape(N * G, g) @ H
    return w.reshape(N, G * g)
