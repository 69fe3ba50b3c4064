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


def test_rotation_leaves_the_weight_gradient_unchanged():
    """H16 diag(s) / 4 is orthonormal, so rotating both operands of the weight
    gradient along the contracted rows (16-row blocks inside each expert's
    32-row-padded segment) leaves D_e = A_e B_e^T unchanged: the reason the
    backward may quantise rotated operands."""
    rng = np.random.default_rng(31)
    idx = np.repeat(np.arange(3), [40, 0, 70])[:, None]
    rt = O.route(idx, 0, 3)
    A = O.bf16_round(rng.standard_normal((rt.R_pad, 24)))
    B = O.bf16_round(rng.standard_normal((rt.R_pad, 20)))
    A[rt.tok_of < 0] = 0
    B[rt.tok_of < 0] = 0
    ref = O.grouped_wgrad(A.T, B.T, rt)
    rot = O.grouped_wgrad(O.rht_transposed(A, 0x5A3C).T, O.rht_transposed(B, 0x5A3C).T, rt)
    assert np.allclose(rot, ref, rtol=1e-12, atol=1e-12)
    # a different sign draw on one operand does not cancel
    bad = O.grouped_wgrad(O.rht_transposed(A, 0x5A3C).T, O.rht_transposed(B, 0x0001).T, rt)
    assert not np.allclose(bad, ref, rtol=1e-3, atol=1e-3)


def test_nvfp4_rht_cast_cols_closed_form():
    """A column that is one constant c over a 16-row block rotates to a single
    non-zero entry (row 0 of the block under all-plus signs: sum of the 16 values
    / 4 = 4c), so with c = 0.375 and s_g = 448 * 6 / 1.5 the block's codes are one
    6 (code 7) in row 0 and zeros, block scale E4M3(1.5 / 6 * 1792) = 448 (0x7E)."""
    y = np.zeros((16, 1))
    y[:, 0] = 0.375
    sg = O.nvfp4_global_scale(1.5)
    q, sb = O.nvfp4_rht_cast_cols(y, 0, sg)
    assert q.shape == (1, 8) and sb.shape == (1, 1)
    assert sb[0, 0] == 0x7E
    assert q[0, 0] == 0x07 and np.all(q[0, 1:] == 0)
    assert np.isclose(O.rht_transposed_amax(y, 0), 1.5)


def test_grouped_wgrad_nvfp4_closed_form():
    """Column-wise NVFP4 operands of all 1.0 (code 2, scale 0x7E, s_g 448) and
    0.5: each expert's D_e is its padded segment length (real rows only hold
    data here: pad rows carry code 0) times 0.5."""
    idx = np.repeat(np.arange(2), [20, 40])[:, None]
    rt = O.route(idx, 0, 2)
    R = rt.R_pad
    real = (rt.tok_of >= 0).astype(np.uint8)
    codes_a = np.where(real, 2, 0).astype(np.uint8)
    codes_b = np.where(real, 1, 0).astype(np.uint8)
    pack = lambda c: (c[0::2] | (c[1::2] << 4)).astype(np.uint8)
    Aq = np.tile(pack(codes_a), (3, 1))
    Bq = np.tile(pack(codes_b), (5, 1))
    As = np.full((3, R // 16), 0x7E, dtype=np.uint8)
    Bs = np.full((5, R // 16), 0x7E, dtype=np.uint8)
    D = O.grouped_wgrad_nvfp4(Aq, As, 448.0, Bq, Bs, 448.0, rt)
    assert D.shape == (2, 3, 5)
    assert np.all(D[0] == 20 * 0.5) and np.all(D[1] == 40 * 0.5)
