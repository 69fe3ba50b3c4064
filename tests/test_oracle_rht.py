"""Pins of the oracle's transposed random-Hadamard amax (NVFP4 backward,
[MoE-Fusion] "Fusing MXFP8 and NVFP4 quantisation"): a library routine, the
transform's algebra, closed forms and an independent fast transform."""
import numpy as np
import pytest

from oracle import moe_oracle as O

scipy_linalg = pytest.importorskip("scipy.linalg")


def test_hadamard16_is_the_sylvester_matrix():
    assert np.array_equal(O.hadamard16(), scipy_linalg.hadamard(16).astype(np.float64))


@pytest.mark.parametrize("mask", [0, 0xFFFF, 0xA5C3, 0x0001])
def test_rotation_is_orthonormal(mask):
    M = O.hadamard16() * O.rht_signs(mask)[None, :] / 4.0
    assert np.allclose(M @ M.T, np.eye(16), atol=1e-15)


def test_signs_follow_the_mask_bits():
    s = O.rht_signs(0b1000000000000101)
    assert list(np.nonzero(s < 0)[0]) == [0, 2, 15]


def test_norm_is_kept_per_block_column():
    rng = np.random.default_rng(3)
    y = O.bf16_round(rng.standard_normal((64, 5)))
    Z = O.rht_transposed(y, 0x3C5A)
    for b in range(4):
        for c in range(5):
            assert np.isclose(np.linalg.norm(Z[16 * b:16 * b + 16, c]), np.linalg.norm(y[16 * b:16 * b + 16, c]))


def test_single_spike_spreads_to_a_quarter():
    y = np.zeros((32, 3))
    y[21, 1] = -6.5            # row 5 of the second block
    Z = O.rht_transposed(y, 0x1234)
    assert np.allclose(np.abs(Z[16:, 1]), 6.5 / 4)
    assert np.all(Z[:16] == 0) and np.all(Z[:, [0, 2]] == 0)
    assert O.rht_transposed_amax(y, 0x1234) == 6.5 / 4


def test_signs_matched_constant_concentrates():
    mask = 0x9B21
    y = np.zeros((16, 2))
    y[:, 0] = 0.75 * O.rht_signs(mask)    # diag(s) y = 0.75 * ones
    Z = O.rht_transposed(y, mask)
    assert Z[0, 0] == 3.0 and np.all(Z[1:, 0] == 0)
    assert O.rht_transposed_amax(y, mask) == 3.0


def _fwht(v):
    """Iterative fast Walsh-Hadamard transform (butterflies), unnormalised."""
    v = np.array(v, dtype=np.float64)
    h = 1
    while h < len(v):
        for i in range(0, len(v), 2 * h):
            a, b = v[i:i + h].copy(), v[i + h:i + 2 * h].copy()
            v[i:i + h], v[i + h:i + 2 * h] = a + b, a - b
        h *= 2
    return v


def test_matches_a_fast_transform_brute_force():
    rng = np.random.default_rng(11)
    y = rng.standard_normal((48, 7)) * 3.0
    mask = 0x5AA5
    Z = O.rht_transposed(y, mask)
    yb = O.bf16_round(y)
    s = O.rht_signs(mask)
    for b in range(3):
        for c in range(7):
            ref = _fwht(s * yb[16 * b:16 * b + 16, c]) / 4.0
            assert np.allclose(Z[16 * b:16 * b + 16, c], ref, rtol=0, atol=1e-12)
    assert np.isclose(O.rht_transposed_amax(y, mask),
                      max(np.max(np.abs(_fwht(s * yb[16 * b:16 * b + 16, c]) / 4.0)) for b in range(3)
                          for c in range(7)))


def test_input_is_rounded_to_bf16_first():
    y = np.zeros((16, 1))
    y[0, 0] = 1.0 + 2.0 ** -9      # a quarter of a bf16 ulp above 1.0: rounds to 1.0
    assert O.rht_transposed_amax(y, 0) == 0.25
