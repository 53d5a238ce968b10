"""Pins for the CQ encoder, packing and reconstruction (Needle .cact page §一;
Needle mmap page, section on tensors read by offset)."""

import json
import math
import os

import numpy as np
import pytest

from gemm_cq_gemv_gb300.synth import weights
from oracle import (GROUP, TERNARY, TERNARY_LEVEL, codebook_levels, cq_encode, cq_reconstruct,
                    field_bits, fwht_butterfly, pack_indices, sylvester_hadamard, unpack_indices)
from util import fitted_cb28, textbook_cb28

# Max 1960, Table I (4 figures); 5 = the ternary code, the table's three-level row
TEXTBOOK_MSE = {1: 0.3634, 2: 0.1175, 3: 0.03454, 4: 0.009497, 5: 0.1902}


def test_pack_examples(golden_dir):
    with open(os.path.join(golden_dir, "cq_pack_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        b = c["b"]
        idx = np.zeros(128, dtype=np.int64)
        idx[: len(c["idx_prefix"])] = c["idx_prefix"]
        f = field_bits(b)
        packed = pack_indices(idx, f)
        assert packed.shape == (16 * f,)
        want = bytes.fromhex(c["bytes_prefix_hex"])
        assert bytes(packed[: len(want)]) == want
        assert not packed[len(want):].any()


@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_pack_round_trip(b):
    rng = np.random.default_rng(b)
    idx = rng.integers(0, 2 ** b, size=(7, 3, 128))
    p = pack_indices(idx, b)
    assert p.shape == (7, 3, 16 * b)
    assert np.array_equal(unpack_indices(p, b), idx)


def test_ternary_packs_in_two_bit_fields():
    rng = np.random.default_rng(11)
    idx = rng.integers(0, 3, size=(5, 2, 128))
    W = rng.standard_normal((5, 256)).astype(np.float32)
    packed, _ = cq_encode(W, TERNARY, textbook_cb28())
    assert packed.shape == (5, 2, 32)
    p = pack_indices(idx, field_bits(TERNARY))
    assert p.shape == (5, 2, 32)
    assert np.array_equal(unpack_indices(p, 2), idx)
    # every stored field of an encoding is 0, 1 or 2
    assert unpack_indices(packed, 2).max() <= 2


def test_four_bit_layout_is_low_nibble_even_column():
    rng = np.random.default_rng(9)
    idx = rng.integers(0, 16, size=128)
    p = pack_indices(idx, 4)
    assert np.array_equal(p & 0x0F, idx[0::2])
    assert np.array_equal(p >> 4, idx[1::2])


def test_codebook_levels_indexing():
    cb = textbook_cb28()
    assert np.array_equal(codebook_levels(cb, 2), cb[0:4])
    assert np.array_equal(codebook_levels(cb, 3), cb[4:12])
    assert np.array_equal(codebook_levels(cb, 4), cb[12:28])
    one = codebook_levels(cb, 1)
    assert one[1] == np.float32(math.sqrt(2 / math.pi)) and one[0] == -one[1]
    ter = codebook_levels(cb, TERNARY)
    assert ter.tolist() == [-np.float32(TERNARY_LEVEL), 0.0, np.float32(TERNARY_LEVEL)]
    with pytest.raises(ValueError):
        codebook_levels(cb, 6)


@pytest.mark.parametrize("cbname", ["textbook", "fitted"])
def test_encode_known_answers(golden_dir, cbname):
    cb = textbook_cb28() if cbname == "textbook" else fitted_cb28()
    with open(os.path.join(golden_dir, "cq_encode_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        W = np.zeros((1, 128), dtype=np.float32)
        if c["w"] == "0.5 * e_0":
            W[0, 0] = 0.5
        else:
            W[0, 1] = 3.0
        packed, norms = cq_encode(W, c["b"], cb)
        idx = unpack_indices(packed, field_bits(c["b"]))[0, 0]
        if "all_idx" in c:
            assert np.all(idx == c["all_idx"]), (c, idx[:8])
        else:
            assert np.all(idx[0::2] == c["even_idx"]) and np.all(idx[1::2] == c["odd_idx"]), c
        assert format(int(norms[0, 0]), "04x") == c["norm_f16_hex"]


@pytest.mark.parametrize("b", [1, 2, 3, 4, 5])
def test_encode_brute_force_nearest(b):
    """Every chosen codeword is a nearest one, recomputed with the dense matrix."""
    cb = fitted_cb28()
    W = weights(8, 4 * 128, seed=77, outliers=True)
    packed, norms = cq_encode(W, b, cb)
    idx = unpack_indices(packed, field_bits(b))               # [8, 4, 128]
    lv = codebook_levels(cb, b).astype(np.float64)
    Hu = sylvester_hadamard(128)
    for o in range(8):
        for j in range(4):
            w = W[o, j * 128:(j + 1) * 128].astype(np.float64)
            v = (Hu @ w) / np.linalg.norm(w)
            d = np.abs(v[:, None] - lv[None, :])
            chosen = d[np.arange(128), idx[o, j]]
            assert np.all(chosen <= d.min(axis=1) + 1e-12)
            assert abs(np.float16(norms[o, j].view(np.float16)) - np.linalg.norm(w)) <= \
                np.linalg.norm(w) * 2 ** -11 * 1.0001


def test_zero_group_and_one_bit_tie():
    cb = fitted_cb28()
    W = np.zeros((2, 256), dtype=np.float32)
    W[1, 128] = 1.0
    W[1, 129] = 1.0            # rotated: [2, 0, 2, 0, ...] -> every odd coordinate is 0
    packed, norms = cq_encode(W, 1, cb)
    idx = unpack_indices(packed, 1)
    assert not idx[0].any() and norms[0, 0] == 0 and norms[0, 1] == 0 and norms[1, 0] == 0
    assert np.all(idx[1, 1, 0::2] == 1)  # +sqrt(2) -> +c
    assert np.all(idx[1, 1, 1::2] == 0)  # exact tie at 0 -> lowest index
    assert np.all(idx[1, 0] == 0)
    # ternary: the zero coordinates take the zero level (index 1), sqrt(2) takes +c
    packed, norms = cq_encode(W, TERNARY, cb)
    idx = unpack_indices(packed, 2)
    assert not idx[0].any() and not idx[1, 0].any()
    assert np.all(idx[1, 1, 0::2] == 2) and np.all(idx[1, 1, 1::2] == 1)


@pytest.mark.parametrize("b", [1, 2, 3, 4, 5])
def test_reconstruction_error_matches_lloyd_max_mse(b):
    """||w - w_hat||^2 / ||w||^2 = ||v - cb[idx]||^2 / g, i.e. the quantizer's MSE
    (rotated coordinates of a Gaussian group are ~N(0,1) after dividing by the norm).
    A wrong normalisation (1/sqrt(g) vs 1/g), sign or transposition breaks this."""
    cb = textbook_cb28()
    W = weights(64, 1024, seed=5)
    packed, norms = cq_encode(W, b, cb)
    W_hat = cq_reconstruct(packed, norms, b, cb)
    err = np.sum((W_hat - W) ** 2) / np.sum(W.astype(np.float64) ** 2)
    assert abs(err - TEXTBOOK_MSE[b]) < 0.08 * TEXTBOOK_MSE[b], err


def test_reconstruction_norm_identity_and_fwht_route():
    cb = fitted_cb28()
    W = weights(16, 512, seed=3, outliers=True)
    for b in (1, 2, 3, 4, 5):
        packed, norms = cq_encode(W, b, cb)
        W_hat = cq_reconstruct(packed, norms, b, cb).reshape(16, 4, 128)
        idx = unpack_indices(packed, field_bits(b))
        lv = codebook_levels(cb, b).astype(np.float64)
        nrm = norms.view(np.float16).astype(np.float64)
        # ||w_hat_g|| = norm / sqrt(g) * ||cb[idx]||  (H is orthonormal)
        lhs = np.linalg.norm(W_hat, axis=2)
        rhs = nrm / math.sqrt(128) * np.linalg.norm(lv[idx], axis=2)
        assert np.allclose(lhs, rhs, rtol=1e-12)
        # same result by the butterfly: w_hat_g = (norm / g) * Hu @ cb[idx]
        alt = (nrm[:, :, None] / 128.0) * fwht_butterfly(lv[idx])
        assert np.allclose(W_hat, alt, rtol=1e-12, atol=1e-15)


def test_encode_rejects_bad_shapes():
    cb = fitted_cb28()
    with pytest.raises(ValueError):
        cq_encode(np.zeros((2, 100), np.float32), 4, cb)
    with pytest.raises(ValueError):
        cq_encode(np.zeros((2, 128), np.float32), 6, cb)   # 5 is the ternary code
    assert GROUP == 128
