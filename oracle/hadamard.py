"""Walsh-Hadamard matrices for the CQ rotation ([CACT] §一; [MMAP] "mmap 之下张量按偏移直读").

The pages name a "normalised Walsh-Hadamard" rotation of each 128-wide group but give
no ordering.  Reading taken: Sylvester (natural) order, i.e. the matrix built by
repeated Kronecker products of [[1, 1], [1, -1]], which is also the order a radix-2
butterfly produces.  ``Hu`` below is unnormalised (entries +-1); the normalised
transform is ``H = Hu / sqrt(g)``, which is symmetric and its own inverse.

Two independent constructions are kept on purpose: the dense Kronecker matrix (used
by the reconstruction / product definitions) and the butterfly (used by the encoder,
whose fp64 rounding order it fixes).  Tests check them against each other and against
``scipy.linalg.hadamard``.
"""

import numpy as np


def sylvester_hadamard(g: int) -> np.ndarray:
    """Dense unnormalised Sylvester Hadamard matrix ``Hu`` of order ``g`` (float64).

    Built by Kronecker products: Hu_1 = [1], Hu_{2m} = [[Hu_m, Hu_m], [Hu_m, -Hu_m]].
    """
    if g < 1 or (g & (g - 1)) != 0:
        raise ValueError("Hadamard order must be a power of two")
    h = np.ones((1, 1), dtype=np.float64)
    base = np.array([[1.0, 1.0], [1.0, -1.0]], dtype=np.float64)
    while h.shape[0] < g:
        h = np.kron(base, h)
    return h


def fwht_butterfly(v: np.ndarray) -> np.ndarray:
    """Unnormalised fast Walsh-Hadamard transform along the last axis, in float64.

    Radix-2 butterflies in natural order: span h = 1, 2, 4, ..., n/2; each pair
    (a, b) = (v[i], v[i + h]) with i in a block of 2h becomes (a + b, a - b).
    Every add / subtract is one IEEE float64 operation (NumPy elementwise), so the
    rounding order of this function is the order the encoder's decisions depend on.
    Equals ``v @ sylvester_hadamard(n)`` (exactly, for small-integer inputs).
    """
    out = np.array(v, dtype=np.float64, copy=True)
    n = out.shape[-1]
    if n < 1 or (n & (n - 1)) != 0:
        raise ValueError("FWHT length must be a power of two")
    h = 1
    while h < n:
        shape = out.shape[:-1] + (n // (2 * h), 2, h)
        blk = out.reshape(shape)
        a = blk[..., 0, :].copy()
        b = blk[..., 1, :].copy()
        blk[..., 0, :] = a + b
        blk[..., 1, :] = a - b
        out = blk.reshape(out.shape)
        h *= 2
    return out
