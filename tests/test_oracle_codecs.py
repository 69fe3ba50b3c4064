"""Pins of the oracle's number formats against hand-worked examples, the
format definitions and torch's own float8/bfloat16 conversions."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = O.e4m3_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok])


def test_e4m3_round_trip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(O.e4m3_encode(O.e4m3_decode(codes)), codes)


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.normal(0, 30, 20000), rng.uniform(-448, 448, 20000),
                        rng.normal(0, 1e-2, 5000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(x), ref)


def test_e4m3_saturates():
    assert O.e4m3_encode(np.array([1e6, -1e6, 470.0]))[0] == 0x7E
    assert O.e4m3_encode(np.array([-1e6]))[0] == 0xFE
    assert O.e4m3_encode(np.array([np.nan]))[0] == 0x7F


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(2)
    x = (rng.normal(0, 1, 50000) * np.exp2(rng.integers(-20, 20, 50000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_round(x), ref)


@pytest.mark.parametrize("case", _load("mxfp8_hand_examples.json")["cases"])
def test_mxfp8_hand_examples(case):
    blk = np.array([float(v) for v in case["block"]], dtype=np.float32)
    v = np.zeros(32, dtype=np.float32)
    v[: len(blk)] = blk
    q, s = O.mx_quantize_rows(v[None, :])
    assert int(s[0, 0]) == case["scale"], case["why"]
    if case["codes"] is not None:
        assert [int(c) for c in q[0, : len(blk)]] == case["codes"], case["why"]


def test_mx_scale_invariant_random():
    """For a normal, finite, non-zero amax, amax * 2^-e lies in [256, 512)
    (E4M3 emax = 8), and every dequantised element is within half an E4M3
    step of its value unless saturated."""
    rng = np.random.default_rng(3)
    v = (rng.normal(0, 1, (64, 256)) * np.exp2(rng.integers(-30, 30, (64, 1)))).astype(np.float32)
    q, s = O.mx_quantize_rows(v)
    blocks = v.reshape(64, 8, 32).astype(np.float64)
    amax = np.abs(blocks).max(-1)
    scaled = amax * np.exp2(127.0 - s)
    assert np.all((scaled >= 256) & (scaled < 512))
    deq = O.mx_dequantize(q, s).reshape(64, 8, 32)
    scale = np.exp2(s - 127.0)[..., None]
    x = blocks / scale                       # exact
    absx = np.abs(x)
    e = np.floor(np.log2(np.maximum(absx, 2.0 ** -6)))
    half_step = np.exp2(e - 3) / 2
    err = np.abs(deq / scale - x)
    sat = absx > 448
    assert np.all(err[~sat] <= half_step[~sat] + 1e-12)
    assert np.all(np.abs(deq / scale)[sat] == 448)


def test_mx_cols_is_rows_of_transpose():
    rng = np.random.default_rng(4)
    v = rng.normal(0, 1, (64, 32)).astype(np.float32)
    qc, sc = O.mx_quantize_cols(v)
    assert qc.shape == (32, 64) and sc.shape == (32, 2)
    # column 5, rows 32..63 form one block: its scale is the rule applied to that block
    blk = v[32:64, 5]
    assert sc[5, 1] == O.mx_scale_byte(np.abs(blk).max())
    assert qc[5, 40] == O.e4m3_encode(v[40, 5] * 2.0 ** (127 - int(sc[5, 1])))


def test_e2m1_and_nvfp4_hand_examples():
    g = _load("nvfp4_hand_examples.json")
    for x, code in g["e2m1_ties"]:
        assert int(O.e2m1_encode(np.array([x]))[0]) == code, x
    assert float(O.nvfp4_global_scale(g["tensor_amax"])) == g["global_scale"]
    for blk in g["blocks"]:
        v = np.zeros((1, 16), dtype=np.float32)
        v[0, : len(blk["values"])] = blk["values"]
        packed, sc = O.nvfp4_quantize_rows(v, np.float32(g["global_scale"]))
        assert int(sc[0, 0]) == blk["scale_code"], blk["why"]
        codes = [int(packed[0, i // 2] >> (4 * (i % 2))) & 0xF for i in range(len(blk["values"]))]
        assert codes == blk["codes"], blk["why"]


def test_e2m1_decode_all_codes():
    assert list(O.e2m1_decode(np.arange(16))) == [0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3, -4, -6]


def test_nvfp4_error_bound_random():
    """Dequantised NVFP4 stays within half an E2M1 step (in block units) plus
    the block-scale rounding of the block maximum."""
    rng = np.random.default_rng(5)
    v = rng.normal(0, 1, (32, 64)).astype(np.float32)
    amax = float(np.abs(v).max())
    sg = O.nvfp4_global_scale(amax)
    packed, sc = O.nvfp4_quantize_rows(v, sg)
    deq = O.nvfp4_dequantize(packed, sc, sg)
    sb = O.e4m3_decode(sc) / float(sg)            # block unit
    err = np.abs(deq - v).reshape(32, 4, 16) / sb[..., None]
    # magnitudes up to 6 units: largest E2M1 gap is 2 (4 -> 6), so half-step <= 1;
    # the block scale itself is rounded (<= 1/16 relative), values may saturate by that much
    assert np.all(err <= 1.0 + 6 * 0.0625 + 1e-6)
    assert math.isclose(float(sg), 2688.0 / np.float32(amax), rel_tol=1e-6)


def test_nvfp4_cols_hand_worked():
    """Column-wise NVFP4 with amax_tensor 6: s_g = 448 * 6 / 6 = 448; column 0
    holds 6, 3, 0, ... (block amax 6 -> s_b = E4M3(6 / 6 * 448) = 448, code
    0x7E; elements E2M1(v * 448 / 448): 6 -> 7, 3 -> 5, 0 -> 0, so the first
    byte is 7 | 5 << 4 = 0x57); column 1 holds -0.5 in row 15 only (block amax
    0.5 -> s_b = E4M3(0.5 / 6 * 448) = E4M3(37.33) = 36 = 1.125 * 2^5 (code 0x61, the
    nearer of 36 and 40), element
    E2M1(-0.5 * 448 / 36) = E2M1(-6.22) = -6 saturated (code 0xF), the high
    nibble of byte 7)."""
    v = np.zeros((16, 2))
    v[0, 0], v[1, 0] = 6.0, 3.0
    v[15, 1] = -0.5
    sg = O.nvfp4_global_scale(6.0)
    assert float(sg) == 448.0
    q, sb = O.nvfp4_quantize_cols(v, sg)
    assert q.shape == (2, 8) and sb.shape == (2, 1)
    assert sb[0, 0] == 0x7E and q[0, 0] == 0x57 and np.all(q[0, 1:] == 0)
    assert sb[1, 0] == 0x61 and q[1, 7] == 0xF0 and np.all(q[1, :7] == 0)


def test_grouped_gemm_nvfp4_closed_form():
    """A = E2M1 1.0 (code 2) and B = 0.5 (code 1) everywhere, block scales 448
    (0x7E) and per-tensor scales 448: both dequantise exactly (1.0 and 0.5),
    so every real output is K * 0.5 and pad rows are 0."""
    K, N = 64, 16
    idx = np.repeat(np.arange(2), [5, 33])[:, None]
    rt = O.route(idx, 0, 2)
    Aq = np.full((rt.R_pad, K // 2), 0x22, dtype=np.uint8)
    As = np.full((rt.R_pad, K // 16), 0x7E, dtype=np.uint8)
    Bq = np.full((2, N, K // 2), 0x11, dtype=np.uint8)
    Bs = np.full((2, N, K // 16), 0x7E, dtype=np.uint8)
    y = O.grouped_gemm_nvfp4(Aq, As, 448.0, Bq, Bs, 448.0, rt)
    real = rt.tok_of >= 0
    assert y.dtype == np.float32
    assert np.all(y[real] == K * 0.5) and np.all(y[~real] == 0)
