"""Pins of the oracle's activation functions: library routines (torch), closed
forms, and central finite differences for every derivative."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

from oracle import moe_oracle as O

RNG = np.random.default_rng(7)
U = RNG.normal(0, 2, 4000)
G = RNG.normal(0, 3, 4000)


def _t(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


def test_swiglu_matches_torch_silu():
    ref = (_t(U) * Fn.silu(_t(G))).numpy()
    assert np.allclose(O.act_fwd(U, G, O.ActParams(O.ACT_SWIGLU)), ref, rtol=1e-13, atol=1e-13)


def test_geglu_matches_torch_gelu():
    ref = (_t(U) * Fn.gelu(_t(G))).numpy()
    assert np.allclose(O.act_fwd(U, G, O.ActParams(O.ACT_GEGLU)), ref, rtol=1e-12, atol=1e-13)
    ref_t = (_t(U) * Fn.gelu(_t(G), approximate="tanh")).numpy()
    assert np.allclose(O.act_fwd(U, G, O.ActParams(O.ACT_GEGLU_TANH)), ref_t, rtol=1e-12, atol=1e-13)


def test_srelu_matches_torch_relu_squared():
    assert np.allclose(O.act_fwd(U, None, O.ActParams(O.ACT_SRELU)), (Fn.relu(_t(U)) ** 2).numpy())


def test_swiglu_closed_forms_at_zero_gate():
    u = np.array([1.5, -2.0, 3.25])
    y = O.act_fwd(u, np.zeros(3), O.ActParams(O.ACT_SWIGLU))
    assert np.all(y == 0)
    du, dg = O.act_bwd(u, np.zeros(3), np.ones(3), O.ActParams(O.ACT_SWIGLU))
    assert np.allclose(dg, u / 2) and np.all(du == 0)
    # GeGLU at g = 0: gelu(0) = 0, gelu'(0) = Phi(0) = 1/2
    du, dg = O.act_bwd(u, np.zeros(3), np.ones(3), O.ActParams(O.ACT_GEGLU))
    assert np.allclose(dg, u / 2) and np.all(du == 0)
    # GeGLU at g = 1: gelu(1) = Phi(1) = 0.5 (1 + erf(1/sqrt 2))
    y = O.act_fwd(np.ones(1), np.ones(1), O.ActParams(O.ACT_GEGLU))
    assert math.isclose(float(y[0]), 0.5 * (1 + math.erf(1 / math.sqrt(2))), rel_tol=1e-14)


GPT_OSS = O.ActParams(O.ACT_SWIGLU, alpha=1.702, up_offset=1.0, gate_lo=-7.0, gate_hi=7.0)
PARAMS = [O.ActParams(O.ACT_SWIGLU), O.ActParams(O.ACT_GEGLU), O.ActParams(O.ACT_GEGLU_TANH),
          O.ActParams(O.ACT_SREGLU), GPT_OSS,
          O.ActParams(O.ACT_SWIGLU, alpha=1.702, up_offset=1.0, gate_lo=-7, gate_hi=7, up_lo=-7, up_hi=7)]


@pytest.mark.parametrize("prm", PARAMS, ids=lambda p: f"act{p.act}_a{p.alpha}_c{p.up_offset}_{p.gate_hi}_{p.up_hi}")
def test_gated_grad_finite_difference(prm):
    u = RNG.normal(0, 3, 3000)
    g = RNG.normal(0, 4, 3000)
    dy = RNG.normal(0, 1, 3000)
    h = 1e-6
    # stay away from the clamp corners and relu kink where the derivative jumps
    ok = (np.abs(np.abs(g) - 7) > 1e-3) & (np.abs(np.abs(u) - 7) > 1e-3) & (np.abs(g) > 1e-3)
    du, dg = O.act_bwd(u, g, dy, prm)
    fd_u = dy * (O.act_fwd(u + h, g, prm) - O.act_fwd(u - h, g, prm)) / (2 * h)
    fd_g = dy * (O.act_fwd(u, g + h, prm) - O.act_fwd(u, g - h, prm)) / (2 * h)
    assert np.allclose(du[ok], fd_u[ok], rtol=1e-6, atol=1e-6)
    assert np.allclose(dg[ok], fd_g[ok], rtol=1e-6, atol=1e-6)


def test_srelu_grad_finite_difference():
    x = RNG.normal(0, 2, 3000)
    x = x[np.abs(x) > 1e-3]
    dy = RNG.normal(0, 1, x.size)
    h = 1e-6
    prm = O.ActParams(O.ACT_SRELU)
    dx, none = O.act_bwd(x, None, dy, prm)
    fd = dy * (O.act_fwd(x + h, None, prm) - O.act_fwd(x - h, None, prm)) / (2 * h)
    assert none is None and np.allclose(dx, fd, rtol=1e-6, atol=1e-6)


def test_gpt_oss_variant_special_values():
    # reduces to plain SwiGLU when alpha = 1, no offset, no clamp
    assert np.allclose(O.act_fwd(U, G, O.ActParams(O.ACT_SWIGLU, alpha=1.0)), (_t(U) * Fn.silu(_t(G))).numpy())
    # alpha scales the sigmoid's argument: alpha*g'*sigmoid(alpha*g') = silu(alpha*g')
    g = np.clip(G, -7, 7)
    ref = ((_t(U) + 1) * Fn.silu(1.702 * _t(g)) / 1.702).numpy()
    assert np.allclose(O.act_fwd(U, G, GPT_OSS), ref, rtol=1e-12, atol=1e-12)
    # above the gate clamp the output is flat and the gate gradient vanishes
    u = np.array([0.5, -2.0])
    big = np.array([9.0, 30.0])
    assert np.allclose(O.act_fwd(u, big, GPT_OSS), O.act_fwd(u, np.full(2, 7.0), GPT_OSS))
    _, dg = O.act_bwd(u, big, np.ones(2), GPT_OSS)
    assert np.all(dg == 0)


def test_phi_cdf_negative_tail_relative_precision():
    """The normal CDF keeps its relative precision deep in the negative tail,
    where (1 + erf) would cancel to 0: tabulated values of Phi and the
    Mills-ratio asymptote Phi(z) ~ phi(z) / |z| (1 - 1/z^2 + 3/z^4)."""
    assert math.isclose(float(O._phi_cdf(-10.0)), 7.619853024160527e-24, rel_tol=1e-12)
    assert math.isclose(float(O._phi_cdf(-5.0)), 2.866515718791939e-07, rel_tol=1e-12)
    for z in (-12.0, -20.0, -30.0):
        pdf = math.exp(-0.5 * z * z) / math.sqrt(2 * math.pi)
        approx = pdf / abs(z) * (1 - 1 / z ** 2 + 3 / z ** 4)
        assert math.isclose(float(O._phi_cdf(z)), approx, rel_tol=15 / z ** 6)
    # GeGLU of a deep-tail gate is tiny but not zero, and so is its derivative
    prm = O.ActParams(O.ACT_GEGLU)
    y = O.act_fwd(np.array([2.0]), np.array([-9.0]), prm)
    assert y[0] < 0 and abs(y[0]) > 1e-18
