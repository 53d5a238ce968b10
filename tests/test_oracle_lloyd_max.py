"""Pins for the Lloyd-Max Gaussian codebooks (Needle .cact page §一; Needle mmap page).

The textbook table (Max 1960) in ``tests/golden/lloyd_max_gaussian_textbook.json`` is
first re-derived here by the closed-form Lloyd iteration on the exact N(0,1) density
(centroid of [a, b] = (phi(a) - phi(b)) / (Phi(b) - Phi(a))), independently of the
oracle; then the oracle's sampled fit (400k samples, 200 iterations) must land on it.
"""

import json
import math
import os

import numpy as np
import pytest

from gemm_cq_gemv_gb300.synth import gaussian_samples
from oracle import (ONE_BIT_LEVEL, TERNARY_LEVEL, gaussian_quantile_init, lloyd_max_gaussian_fit,
                    ternary_gaussian_level)


def _phi(x):
    return math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi) if math.isfinite(x) else 0.0


def _Phi(x):
    if x == math.inf:
        return 1.0
    if x == -math.inf:
        return 0.0
    return 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))


def _closed_form_lloyd(L, iters=5000):
    lv = [(-3.0 + 6.0 * (t + 0.5) / L) for t in range(L)]
    for _ in range(iters):
        thr = [-math.inf] + [(lv[i] + lv[i + 1]) / 2 for i in range(L - 1)] + [math.inf]
        lv = [(_phi(thr[i]) - _phi(thr[i + 1])) / (_Phi(thr[i + 1]) - _Phi(thr[i])) for i in range(L)]
    return lv


def _closed_form_mse(lv):
    L = len(lv)
    thr = [-math.inf] + [(lv[i] + lv[i + 1]) / 2 for i in range(L - 1)] + [math.inf]
    # E[(x - c)^2 on cell] = E[x^2] - 2c E[x] + c^2 P, each in closed form
    mse = 0.0
    for i in range(L):
        a, b, c = thr[i], thr[i + 1], lv[i]
        P = _Phi(b) - _Phi(a)
        m1 = _phi(a) - _phi(b)
        aphi = a * _phi(a) if math.isfinite(a) else 0.0
        bphi = b * _phi(b) if math.isfinite(b) else 0.0
        m2 = P + aphi - bphi
        mse += m2 - 2 * c * m1 + c * c * P
    return mse


@pytest.fixture(scope="module")
def textbook(golden_dir):
    with open(os.path.join(golden_dir, "lloyd_max_gaussian_textbook.json")) as f:
        return json.load(f)


@pytest.fixture(scope="module")
def fitted():
    s = gaussian_samples(400_000, seed=0)
    return s, {L: lloyd_max_gaussian_fit(s, L, 200) for L in (2, 4, 8, 16)}


@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_closed_form_reproduces_textbook(textbook, b):
    lv = _closed_form_lloyd(2 ** b)
    pos = sorted(v for v in lv if v > 0)
    ref = textbook["levels_positive"][str(b)]
    assert np.allclose(pos, ref, rtol=2e-3, atol=6e-4)
    assert abs(_closed_form_mse(lv) - textbook["mse"][str(b)]) < 2e-3 * textbook["mse"][str(b)] + 2e-5


def test_one_bit_level_is_sqrt_two_over_pi(textbook):
    assert ONE_BIT_LEVEL == math.sqrt(2.0 / math.pi)
    assert abs(ONE_BIT_LEVEL - textbook["levels_positive"]["1"][0]) < 2e-4  # printed to 4 figures
    # and it is E|X| for X ~ N(0,1), the 1-bit Lloyd-Max centroid
    assert abs(_closed_form_lloyd(2)[1] - ONE_BIT_LEVEL) < 1e-12


def test_quantile_init_is_symmetric_and_sorted():
    for L in (2, 4, 8, 16):
        lv = gaussian_quantile_init(L)
        assert np.all(np.diff(lv) > 0)
        assert np.allclose(lv, -lv[::-1], atol=1e-12)


@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_sampled_fit_lands_on_textbook(textbook, fitted, b):
    _, fits = fitted
    lv = fits[2 ** b].astype(np.float64)
    assert lv.dtype == np.float64 and fits[2 ** b].dtype == np.float32
    ref = np.array(textbook["levels_positive"][str(b)])
    full = np.concatenate([-ref[::-1], ref])
    assert np.all(np.diff(lv) > 0)
    assert np.max(np.abs(lv - full)) < 0.02
    assert np.max(np.abs(lv + lv[::-1])) < 0.02  # symmetric within 0.02


@pytest.mark.parametrize("L", [2, 4, 8, 16])
def test_sampled_fit_is_a_lloyd_fixed_point(fitted, L):
    s, fits = fitted
    lv = fits[L].astype(np.float64)
    thr = (lv[:-1] + lv[1:]) / 2
    cell = np.searchsorted(thr, s, side="left")
    for t in range(L):
        m = s[cell == t].mean()
        assert abs(m - lv[t]) < 1e-5, (t, m, lv[t])


@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_sampled_fit_mse(textbook, fitted, b):
    s, fits = fitted
    lv = fits[2 ** b].astype(np.float64)
    thr = (lv[:-1] + lv[1:]) / 2
    q = lv[np.searchsorted(thr, s, side="left")]
    mse = np.mean((s - q) ** 2)
    assert abs(mse - textbook["mse"][str(b)]) < 0.03 * textbook["mse"][str(b)]


def test_committed_codebook_matches_oracle_fit(golden_dir, fitted):
    _, fits = fitted
    with open(os.path.join(golden_dir, "codebook_seed0.json")) as f:
        cb = json.load(f)
    for b, L in ((2, 4), (3, 8), (4, 16)):
        hexes = [format(int(v), "08x") for v in fits[L].view(np.uint32)]
        assert hexes == cb[f"cb{b}_f32_hex"]


def test_ternary_level_matches_textbook(textbook):
    """The ternary c (mmap page, bits = 5; the page gives no value) is the three-level
    Lloyd-Max Gaussian level: Max's N = 3 row prints 0, +-1.224, thresholds +-0.6120 and
    MSE 0.1902 (4 figures)."""
    row = textbook["three_level"]
    c = TERNARY_LEVEL
    assert abs(c - row["levels_positive"][1]) < 5e-4
    assert abs(c / 2 - row["thresholds_positive"][0]) < 5e-4
    assert abs(_closed_form_mse([-c, 0.0, c]) - row["mse"]) < 5e-4


def test_ternary_level_is_the_three_level_lloyd_solution():
    """Against the general closed-form Lloyd iteration of this file (free middle level,
    asymmetric start): it converges to [-c, 0, c] with the oracle's c."""
    lv = _closed_form_lloyd(3)
    assert abs(lv[1]) < 1e-12 and abs(lv[0] + lv[2]) < 1e-12
    assert abs(lv[2] - TERNARY_LEVEL) < 1e-9
    assert ternary_gaussian_level() == TERNARY_LEVEL


def test_ternary_level_minimises_the_mse():
    """Among symmetric codebooks {-a, 0, a} with midpoint thresholds, a = c has the least
    mean-squared error (a wrong threshold or centroid rule would move the minimum)."""
    c = TERNARY_LEVEL
    best = _closed_form_mse([-c, 0.0, c])
    for d in (1e-3, -1e-3, 1e-2, -1e-2):
        assert _closed_form_mse([-(c + d), 0.0, c + d]) > best
