"""GPU parity of the combine backward (dY_perm, dprob) and the permute
backward (dx) against the oracle's chain rule ([MegaMoE] §2.1 differentiated).

Tolerances, from the arithmetic: dY_perm = bf16(fp32(p * dout)) rounds twice
(fp32, then bf16) where the oracle rounds the exact product once, so a value
may sit one bf16 step away when the fp32 product lands on a bf16 tie; dprob is
an fp32 dot over H terms (per-lane fma chains, then a 5-level butterfly), so
its error is below ~(H/256 + 5) * 2^-24 * sum|dout * y|, bounded here by
1e-5 * sum|dout * y|; dx sums at most k bf16 values in fp32 before one bf16
rounding (again at most one bf16 step)."""
import numpy as np
import pytest
import torch

from grouped_gemm_glu_gb300 import ops, synth
from oracle import moe_oracle as O
from parity import np_

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _bf16_step_close(gpu, ref, what, exact_frac=0.999):
    g, r = np.asarray(gpu, np.float64), np.asarray(ref, np.float64)
    assert g.shape == r.shape, what
    step = np.exp2(np.floor(np.log2(np.maximum(np.abs(r), 1e-38))) - 7)   # one bf16 ulp at |ref|
    d = np.abs(g - r)
    assert np.all(d <= step * 1.0000001), f"{what}: {np.sum(d > step)} values beyond one bf16 step"
    assert np.mean(d == 0) >= exact_frac, f"{what}: only {np.mean(d == 0):.5f} bit-identical"


def _case(T, H, k, E, n_experts, expert_begin, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(n_experts, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    prob = rng.random((T, k), dtype=np.float32)
    x = synth._bf16(rng.standard_normal((T, H), dtype=np.float32))
    dout = synth._bf16(rng.standard_normal((T, H), dtype=np.float32))
    R_cap = ((T * k + 31 * E) + 127) // 128 * 128
    y_perm = synth._bf16(rng.standard_normal((R_cap, H), dtype=np.float32))
    dxp = synth._bf16(rng.standard_normal((R_cap, H), dtype=np.float32))
    g = ops.route_permute(x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(prob).to(DEV), E, R_cap,
                          expert_begin)
    rt = O.route(idx, expert_begin, E)
    return rt, g, prob, dout, y_perm, dxp, R_cap


@pytest.mark.parametrize("T,H,k,E,n_experts,begin", [(300, 256, 4, 6, 16, 3), (1000, 64, 2, 8, 8, 0),
                                                       (77, 520, 8, 5, 64, 60)])
def test_combine_and_permute_bwd_match_oracle(T, H, k, E, n_experts, begin):
    rt, g, prob, dout, y_perm, dxp, R_cap = _case(T, H, k, E, n_experts, begin, seed=T + H)
    yd = y_perm.to(DEV)
    dY, dprob = ops.combine_bwd(dout.to(DEV), yd, g, k)
    dx = ops.permute_bwd(dxp.to(DEV), g["row_of"], T, k, status=g["status"])
    torch.cuda.synchronize()
    assert ops.read_status(g["status"]) == 0
    R = rt.R_pad
    yv = np_(y_perm)[:R].copy()
    ref_dY, ref_dprob = O.combine_bwd(np_(dout), yv, rt.row_of, prob, R)
    _bf16_step_close(np_(dY)[:R], O.bf16_round(ref_dY), "dY_perm")
    assert np.all(np_(dY)[:R][rt.tok_of < 0] == 0), "pad rows of dY_perm"
    rows = rt.row_of.reshape(T, k)
    mag = np.zeros((T, k))
    for j in range(k):
        ok = rows[:, j] >= 0
        mag[ok, j] = np.sum(np.abs(np_(dout)[ok] * yv[rows[ok, j]]), axis=1)
    err = np.abs(np_(dprob).astype(np.float64) - ref_dprob)
    assert np.all(err <= 1e-5 * mag + 1e-30), f"dprob: worst {err.max():.3g}"
    assert np.all(np_(dprob)[rows < 0] == 0), "dprob of dropped slots"
    xv = np_(dxp)[:R].copy()
    _bf16_step_close(np_(dx), O.bf16_round(O.permute_bwd(xv, rt.row_of, T, k)), "dx")
    none_local = np.all(rows < 0, axis=1)
    assert np.all(np_(dx)[none_local] == 0)


def test_combine_bwd_dsv3_shape_sampled_tokens():
    """Full DeepSeek-V3 shard sizes (T 8192, H 7168, top-8 of 256, experts
    0..31 local); the oracle checks 48 sampled tokens, every slot of which is
    either local (dY row, dprob) or dropped (dprob 0)."""
    w = synth.WORKLOADS["dsv3"]
    rs = synth._streams(31, 4)
    idx, prob = synth.router_inputs(w, rs[0])
    T, H, k, E = w.T, w.H, w.k, w.E
    R_cap = w.R_cap
    x = synth._bf16(rs[1].standard_normal((T, H), dtype=np.float32))
    dout = synth._bf16(rs[2].standard_normal((T, H), dtype=np.float32))
    y_perm = synth._bf16(rs[3].standard_normal((R_cap, H), dtype=np.float32))
    g = ops.route_permute(x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(prob).to(DEV), E, R_cap,
                          w.expert_begin)
    dY, dprob = ops.combine_bwd(dout.to(DEV), y_perm.to(DEV), g, k)
    dx = ops.permute_bwd(y_perm.to(DEV), g["row_of"], T, k, status=g["status"])
    torch.cuda.synchronize()
    assert ops.read_status(g["status"]) == 0
    rt = O.route(idx, w.expert_begin, E)
    rows = rt.row_of.reshape(T, k)
    toks = np.random.default_rng(8).choice(T, 48, replace=False)
    dYn, dpn, dxn = np_(dY), np_(dprob), np_(dx)
    yv, gv = np_(y_perm), np_(dout)
    for t in toks:
        for j in range(k):
            r = rows[t, j]
            if r < 0:
                assert dpn[t, j] == 0
                continue
            ref = O.bf16_round(float(prob[t, j]) * gv[t].astype(np.float64))
            _bf16_step_close(dYn[r], ref, f"dY row {r}", exact_frac=0.99)
            dot = float(np.dot(gv[t].astype(np.float64), yv[r].astype(np.float64)))
            assert abs(dpn[t, j] - dot) <= 1e-5 * float(np.sum(np.abs(gv[t] * yv[r]))), (t, j)
        ref_dx = O.bf16_round(sum(yv[r].astype(np.float64) for r in rows[t] if r >= 0) if (rows[t] >= 0).any()
                              else np.zeros(H))
        _bf16_step_close(dxn[t], ref_dx, f"dx token {t}", exact_frac=0.99)
    assert np.all(dpn[rows < 0] == 0)
    assert np.all(dYn[:rt.R_pad][rt.tok_of < 0] == 0)
