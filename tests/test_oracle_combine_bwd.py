"""Pins of the oracle's combine and permute backward ([MegaMoE] §2.1,
y = sum_{i in top-k} p_i E_i(x)): central finite differences of the forward
definitions (unpermute_combine, permute) and torch autograd of the same
forward written with library gathers, plus the special cases (dropped
assignments, tokens without a local expert, duplicate-free rows)."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O


def _routing(seed, T=7, k=3, E=4, n_experts=6):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(n_experts, size=k, replace=False) for _ in range(T)]).astype(np.int64)
    rt = O.route(idx, 1, E)   # experts 1..4 local, 0 and 5 dropped
    p = rng.random((T, k))
    return rt, idx, p


def test_combine_bwd_matches_finite_differences():
    rt, idx, p = _routing(1)
    T, k = p.shape
    H = 5
    rng = np.random.default_rng(2)
    y = rng.standard_normal((rt.R_pad, H))
    y[rt.tok_of < 0] = 0
    g = rng.standard_normal((T, H))
    f = lambda pp, yy: float(np.sum(g * O.unpermute_combine(yy, rt.row_of, pp)))
    dY, dprob = O.combine_bwd(g, y, rt.row_of, p, rt.R_pad)
    eps = 1e-6
    for t in range(T):
        for j in range(k):
            e = np.zeros_like(p); e[t, j] = eps
            fd = (f(p + e, y) - f(p - e, y)) / (2 * eps)
            assert abs(fd - dprob[t, j]) < 1e-6, (t, j)
    for row in range(rt.R_pad):
        for h in range(H):
            e = np.zeros_like(y); e[row, h] = eps
            fd = (f(p, y + e) - f(p, y - e)) / (2 * eps)
            assert abs(fd - dY[row, h]) < 1e-6, (row, h)


def test_combine_bwd_matches_autograd_and_special_cases():
    rt, idx, p = _routing(3, T=9, k=4, E=3)
    T, k = p.shape
    H = 6
    rng = np.random.default_rng(4)
    y = rng.standard_normal((rt.R_pad, H))
    g = rng.standard_normal((T, H))
    yt = torch.tensor(y, requires_grad=True)
    pt = torch.tensor(p, requires_grad=True)
    rows = torch.tensor(rt.row_of.reshape(T, k))
    keep = (rows >= 0).double()
    gathered = yt[rows.clamp(min=0)] * keep[..., None]            # [T, k, H]
    out = (pt[..., None] * gathered).sum(1)
    (out * torch.tensor(g)).sum().backward()
    dY, dprob = O.combine_bwd(g, y, rt.row_of, p, rt.R_pad)
    np.testing.assert_allclose(dY, yt.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dprob, (pt.grad * keep).numpy(), rtol=0, atol=1e-12)
    dropped = rt.row_of.reshape(T, k) < 0
    assert dropped.any() and np.all(dprob[dropped] == 0)
    assert np.all(dY[rt.tok_of < 0] == 0)       # pad rows receive nothing


def test_permute_bwd_matches_finite_differences_and_autograd():
    rt, idx, p = _routing(5, T=8, k=3, E=4)
    T, k = p.shape
    H = 4
    rng = np.random.default_rng(6)
    x = rng.standard_normal((T, H))
    G = rng.standard_normal((rt.R_pad, H))
    f = lambda xx: float(np.sum(G * O.permute(xx, rt)))
    dx = O.permute_bwd(G, rt.row_of, T, k)
    eps = 1e-6
    for t in range(T):
        for h in range(H):
            e = np.zeros_like(x); e[t, h] = eps
            assert abs((f(x + e) - f(x - e)) / (2 * eps) - dx[t, h]) < 1e-6
    xt = torch.tensor(x, requires_grad=True)
    tok = torch.tensor(rt.tok_of)
    xp = xt[tok.clamp(min=0)] * (tok >= 0).double()[:, None]
    (xp * torch.tensor(G)).sum().backward()
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=0, atol=1e-12)
    none_local = np.all(rt.row_of.reshape(T, k) < 0, axis=1)
    assert np.all(dx[none_local] == 0)


def test_no_local_tokens_give_zero_gradients():
    idx = np.array([[0, 5], [5, 0]], dtype=np.int64)   # nothing in experts 1..4
    rt = O.route(idx, 1, 4)
    p = np.array([[0.6, 0.4], [0.7, 0.3]])
    g = np.ones((2, 3))
    dY, dprob = O.combine_bwd(g, np.zeros((rt.R_pad, 3)), rt.row_of, p, rt.R_pad)
    assert rt.R_pad == 0 and dY.shape == (0, 3) and np.all(dprob == 0)
    assert np.all(O.permute_bwd(np.zeros((0, 3)), rt.row_of, 2, 2) == 0)
