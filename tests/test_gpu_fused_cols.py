"""GPU parity of the column-wise MXFP8 copies made inside the gather and the
combine backward ([MoE-Fusion] "Fusing MXFP8 and NVFP4 quantisation": MXFP8
= row-wise output plus a transposed copy; the weight gradients read the
transposed copies of x_perm and dY_perm).  The fused outputs are compared
with the oracle's column cast of the same rows, bit for bit, and the rows,
tok_of, prob_perm, dY_perm and dprob with the plain kernels' (which the route
and combine-backward tests compare with the oracle)."""
import numpy as np
import pytest
import torch

from grouped_gemm_glu_gb300 import ops, synth
from oracle import moe_oracle as O
from parity import assert_exact, np_

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _case(T, H, k, E, n_experts, begin, seed, nan_token=None):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(n_experts, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    prob = rng.random((T, k), dtype=np.float32)
    xf = rng.standard_normal((T, H), dtype=np.float32) * np.exp2(rng.integers(-6, 6, (1, H)))
    if nan_token is not None:
        xf[nan_token, 3] = np.nan
        xf[nan_token, 5] = np.inf
    x = synth._bf16(xf)
    R_cap = ((T * k + 31 * E) + 127) // 128 * 128
    return idx, prob, x, R_cap


def _check_cols(q, s, rows, R, what):
    qr, sr = O.mx_quantize_cols(rows)
    assert_exact(np_(q)[:, :R], qr, f"{what} codes")
    assert_exact(np_(s)[:, : R // 32], sr, f"{what} scales")


# H = 520 and 1000: a partial last chunk of 512 columns; H = 7168 with 32 of
# 256 experts and top-8 is the DeepSeek-V3-shaped shard
@pytest.mark.parametrize("T,H,k,E,n_experts,begin", [(300, 256, 4, 6, 16, 3), (1000, 1000, 2, 8, 8, 0),
                                                       (77, 520, 8, 5, 64, 60), (8192, 7168, 8, 32, 256, 0)])
def test_gather_column_cast(T, H, k, E, n_experts, begin):
    idx, prob, x, R_cap = _case(T, H, k, E, n_experts, begin, seed=T + H, nan_token=T // 2)
    args = (x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(prob).to(DEV), E, R_cap, begin)
    g = ops.route_permute(*args, with_col=True)
    ref = ops.route_permute(*args)
    torch.cuda.synchronize()
    assert ops.read_status(g["status"]) == 0
    rt = O.route(idx, begin, E)
    R = rt.R_pad
    for n in ("counts", "offsets", "row_of"):
        assert torch.equal(g[n], ref[n]), n
    for n in ("tok_of", "prob_perm"):
        assert torch.equal(g[n][:R], ref[n][:R]), n
    assert torch.equal(g["x_perm"][:R].view(torch.int16), ref["x_perm"][:R].view(torch.int16)), "x_perm"
    xp = O.permute(np_(x), rt)
    np.testing.assert_array_equal(np_(g["x_perm"])[:R], xp, "x_perm")  # NaN positions equal too
    _check_cols(g["x_qc"], g["x_sc"], xp, R, "x_perm column cast")
    # blocks at or past offsets[E] are untouched (the buffers start as zeros)
    assert np.all(np_(g["x_qc"])[:, R:] == 0) and np.all(np_(g["x_sc"])[:, R // 32:] == 0)


@pytest.mark.parametrize("T,H,k,E,n_experts,begin", [(300, 256, 4, 6, 16, 3), (77, 520, 8, 5, 64, 60),
                                                       (8192, 7168, 8, 32, 256, 0)])
def test_combine_bwd_column_cast(T, H, k, E, n_experts, begin):
    idx, prob, x, R_cap = _case(T, H, k, E, n_experts, begin, seed=2 * T + H)
    rng = np.random.default_rng(T)
    doutf = rng.standard_normal((T, H), dtype=np.float32)
    doutf[T // 3, 7] = np.nan
    dout = synth._bf16(doutf).to(DEV)
    y_perm = synth._bf16(rng.standard_normal((R_cap, H), dtype=np.float32)).to(DEV)
    g = ops.route_permute(x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(prob).to(DEV), E, R_cap, begin)
    q = torch.zeros(H, R_cap, dtype=torch.uint8, device=DEV)
    s = torch.zeros(H, R_cap // 32, dtype=torch.uint8, device=DEV)
    dY, dprob = ops.combine_bwd(dout, y_perm, g, k, col=(q, s))
    dY0, dprob0 = ops.combine_bwd(dout, y_perm, g, k)
    torch.cuda.synchronize()
    assert ops.read_status(g["status"]) == 0
    R = int(g["offsets"][-1].item())
    assert torch.equal(dY[:R].view(torch.int16), dY0[:R].view(torch.int16)), "dY_perm"
    assert torch.equal(torch.nan_to_num(dprob, nan=7.0), torch.nan_to_num(dprob0, nan=7.0)), "dprob"
    _check_cols(q, s, np_(dY)[:R], R, "dY_perm column cast")
    assert np.all(np_(q)[:, R:] == 0) and np.all(np_(s)[:, R // 32:] == 0)
