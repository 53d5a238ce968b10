"""Q4_0 flat-block quantization ([KMCU] §2 "Q4_0 量化", §3 "行对齐到 32").

What the page fixes: 32 weights per block; bytes [0, 2) hold the fp16 scale
``d = max_abs / 8``; bytes [2, 18) hold one 4-bit nibble per weight, ``q = round(w/d)``
clipped to [-8, 7], nibble = q + 8, the low nibble holding the even index; dequant
``w = (nibble - 8) * d``; 18 bytes per 32 weights = 4.5 bit/weight.  Each row is
zero-padded to a multiple of 32 before blocking, so a block never straddles two rows
and block (r, b) sits at index ``r * nblk + b`` with ``nblk = ceil(n_cols / 32)``.

Readings taken:
  * the garbled ``np.where(amax 0, amax / 8.0, 1.0)`` reads as ``amax > 0``;
  * quantization divides by the float32 ``d`` (NumPy float32 arithmetic); the block
    stores ``float16(d)`` (round to nearest even, little-endian); dequantization uses
    the stored float16 ``d``;
  * ``round`` is ``np.rint`` (half to even); padding zeros become nibble 8;
  * the even-index-in-low-nibble order is the page's (byte k = nib[2k] | nib[2k+1] << 4),
    not the j / j + 16 split of some other Q4_0 implementations.
"""

import numpy as np

Q4_0_BLOCK = 32
Q4_0_BLOCK_BYTES = 18


def q4_0_row_bytes(n_cols: int) -> int:
    """Bytes per row after padding to 32: ``ceil(n_cols / 32) * 18``."""
    return ((n_cols + Q4_0_BLOCK - 1) // Q4_0_BLOCK) * Q4_0_BLOCK_BYTES


def q4_0_quantize(W: np.ndarray) -> np.ndarray:
    """``W`` float32 ``[N, K]`` -> uint8 ``[N, ceil(K/32) * 18]`` Q4_0 blocks."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    nblk = (K + Q4_0_BLOCK - 1) // Q4_0_BLOCK
    padded = np.zeros((N, nblk * Q4_0_BLOCK), dtype=np.float32)
    padded[:, :K] = W
    blocks = padded.reshape(N * nblk, Q4_0_BLOCK)
    amax = np.abs(blocks).max(axis=1)
    d = np.where(amax > 0, amax / np.float32(8.0), np.float32(1.0)).astype(np.float32)
    q = np.clip(np.rint((blocks / d[:, None]).astype(np.float32)), -8, 7)
    nib = (q + 8).astype(np.uint8)
    out = np.zeros((N * nblk, Q4_0_BLOCK_BYTES), dtype=np.uint8)
    d16 = d.astype(np.float16).view(np.uint16)
    out[:, 0] = (d16 & 0xFF).astype(np.uint8)
    out[:, 1] = (d16 >> 8).astype(np.uint8)
    out[:, 2:] = nib[:, 0::2] | (nib[:, 1::2] << 4)
    return out.reshape(N, nblk * Q4_0_BLOCK_BYTES)


def q4_0_dequantize(blocks: np.ndarray, n_cols: int) -> np.ndarray:
    """Q4_0 bytes ``[N, nblk*18]`` -> ``W_hat`` float64 ``[N, n_cols]`` (padding dropped)."""
    blocks = np.asarray(blocks, dtype=np.uint8)
    N = blocks.shape[0]
    nblk = blocks.shape[1] // Q4_0_BLOCK_BYTES
    b = blocks.reshape(N * nblk, Q4_0_BLOCK_BYTES)
    d = (b[:, 0].astype(np.uint16) | (b[:, 1].astype(np.uint16) << 8)).view(np.float16)
    nib = np.empty((N * nblk, Q4_0_BLOCK), dtype=np.int64)
    nib[:, 0::2] = b[:, 2:] & 0x0F
    nib[:, 1::2] = b[:, 2:] >> 4
    w = (nib - 8).astype(np.float64) * d.astype(np.float64)[:, None]
    return w.reshape(N, nblk * Q4_0_BLOCK)[:, :n_cols]
