"""Shared test helpers: codebook tables and tolerance metrics (no method arithmetic)."""

import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def textbook_cb28():
    """cb2 | cb3 | cb4 built from the printed Lloyd-Max Gaussian tables (Max 1960)."""
    with open(os.path.join(GOLDEN, "lloyd_max_gaussian_textbook.json")) as f:
        t = json.load(f)["levels_positive"]
    parts = []
    for b in ("2", "3", "4"):
        p = np.array(t[b], dtype=np.float64)
        parts.append(np.concatenate([-p[::-1], p]))
    return np.concatenate(parts).astype(np.float32)


def fitted_cb28():
    """The committed oracle fit (``codebook_seed0.json``), bit for bit."""
    with open(os.path.join(GOLDEN, "codebook_seed0.json")) as f:
        d = json.load(f)
    hexes = d["cb2_f32_hex"] + d["cb3_f32_hex"] + d["cb4_f32_hex"]
    return np.array([int(h, 16) for h in hexes], dtype=np.uint32).view(np.float32)


def max_rel_err(y, ref):
    """max_i |y_i - ref_i| / max_i |ref_i| per output vector (rows of a 2-D array)."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.ndim == 1:
        y, ref = y[None], ref[None]
    den = np.max(np.abs(ref), axis=1)
    den = np.where(den > 0, den, 1.0)
    return float(np.max(np.max(np.abs(y - ref), axis=1) / den))
