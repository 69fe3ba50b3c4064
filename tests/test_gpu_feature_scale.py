"""GPU parity of feature scaling ([MoE-Fusion] "clamping and scaling";
reading: the router probability multiplied into the FC1 output, a = p *
act(pre)): the forward epilogue's row scale, the backward epilogue's scaled
dActivation, and the feature-scale gradient dL/dp = sum_c da * act(pre) that
the backward epilogue writes as per-row partials and moe_feature_scale_grad
maps onto the routed slots.

dprob tolerance, from the arithmetic: da comes from an fp32 tensor-core
accumulation, act from fp32 transcendental approximations, and the sum over F
columns is fp32, so |dprob - oracle| <= 1e-3 * sum_c |da * act| + 1e-6."""
import numpy as np
import pytest
import torch

from grouped_gemm_glu_gb300 import lib as L
from grouped_gemm_glu_gb300 import ops, synth
from oracle import moe_oracle as O
from parity import assert_bf16_close, assert_mx_close, np_

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _params(w):
    if w.gpt_oss:
        return (L.glu_params("swiglu", alpha=1.702, up_offset=1.0, gate_lo=-7.0, gate_hi=7.0),
                O.ActParams(O.ACT_SWIGLU, alpha=1.702, up_offset=1.0, gate_lo=-7.0, gate_hi=7.0))
    m = {"swiglu": O.ACT_SWIGLU, "geglu": O.ACT_GEGLU, "srelu": O.ACT_SRELU}
    return L.glu_params(w.act), O.ActParams(m[w.act])


def _setup(w, seed):
    inp = synth.make_inputs(w, seed)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    r = ops.route_permute(g["x"], g["topk_idx"], g["topk_prob"], w.E, w.R_cap, w.expert_begin)
    rt = O.route(inp["topk_idx"].numpy(), w.expert_begin, w.E)
    p_rows = O.permute_probs(inp["topk_prob"].numpy(), rt).astype(np.float32)
    return inp, g, r, rt, p_rows


def test_fc1_forward_row_scale_tiny():
    w = synth.WORKLOADS["tiny"]
    inp, g, r, rt, p_rows = _setup(w, 41)
    gp, op = _params(w)
    W1p = ops.repack_fc1(g["W1"])
    o = ops.fc1_fwd(r["x_perm"], W1p, r["counts"], r["offsets"], w.F, gp, L.OUT_MXFP8, row_scale=r["prob_perm"])
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    R = rt.R_pad
    assert np.array_equal(np_(r["prob_perm"])[:R], p_rows)
    fo = O.fc1_glu_fwd(O.permute(np_(inp["x"]), rt), O.repack_fc1(np_(inp["W1"])), None, rt, op,
                       row_scale=p_rows.astype(np.float64))
    assert_bf16_close(np_(o["pre"])[:R], fo.pre_bf16, "pre (unscaled)")
    q, s = O.mx_quantize_rows(fo.y)
    assert_mx_close(np_(o["q_row"])[:R], np_(o["s_row"])[:R], q, s, fo.y, "scaled row-wise")
    qc, sc = O.mx_quantize_cols(fo.y)
    assert_mx_close(np_(o["q_col"])[:, :R], np_(o["s_col"])[:, :R // 32], qc, sc, fo.y.T, "scaled col-wise")


def _dprob_check(got, rows_ok, dY, W2, pre, rt, op, w, rows):
    """Oracle feature-scale gradient of the given rows, one at a time."""
    for r in rows:
        if rt.tok_of[r] < 0:
            continue
        e = int(rt.expert_of_row[r])
        da = dY[r].astype(np.float64) @ W2[e].T.astype(np.float64)
        pr = pre[r].astype(np.float64)[None]
        if w.gated:
            u, gg = O.unpack_glu_cols(pr)
            act = O.act_fwd(u, gg, op)[0]
        else:
            act = O.act_fwd(pr, None, op)[0]
        ref = float(np.sum(da * act))
        mag = float(np.sum(np.abs(da * act)))
        assert abs(got[r] - ref) <= 1e-3 * mag + 1e-6, (r, got[r], ref)


@pytest.mark.parametrize("name", ["tiny", "gptoss", "skew_srelu"])
def test_dglu_row_scale_and_feature_scale_grad(name):
    w = synth.WORKLOADS[name]
    if name != "tiny":
        w = synth.scaled(w, T=512, H=512)
    inp, g, r, rt, p_rows = _setup(w, 42)
    gp, op = _params(w)
    rng = np.random.default_rng(43)
    pre = synth._bf16(rng.standard_normal((w.R_cap, w.N1), dtype=np.float32) * 2.0)
    o = ops.dglu_bwd(g["dY"], g["W2"], pre.to(DEV), r["counts"], r["offsets"], w.F, gp, L.OUT_BF16,
                     row_scale=r["prob_perm"], row_dot=True, status=r["status"])
    dprob = ops.feature_scale_grad(o["row_dot"], r["row_of"], w.T, w.k)
    torch.cuda.synchronize()
    assert ops.read_status(r["status"]) == 0
    assert o["row_dot"].shape[1] == 2 * ((w.F + 255) // 256)
    R = rt.R_pad
    dY = np_(inp["dY"])[:R].copy()
    dY[rt.tok_of < 0] = 0
    d = O.dglu_bwd(dY, np_(inp["W2"]), np_(pre)[:R], rt, op, row_scale=p_rows.astype(np.float64))
    assert_bf16_close(np_(o["y"])[:R], O.bf16_round(d), f"{name} scaled dFC1")
    row_sum = np_(o["row_dot"]).astype(np.float64).sum(axis=1)
    _dprob_check(row_sum, None, dY, np_(inp["W2"]), np_(pre), rt, op, w, range(R))
    # slot mapping: every routed slot gets its row's partials added in order in
    # fp32 (emulated exactly here), dropped slots 0
    rows = rt.row_of.reshape(w.T, w.k)
    got = np_(dprob)
    ok = rows >= 0
    assert np.all(got[~ok] == 0)
    parts = np_(o["row_dot"])
    acc = np.zeros(parts.shape[0], dtype=np.float32)
    for q in range(parts.shape[1]):
        acc = (acc + parts[:, q]).astype(np.float32)
    assert np.array_equal(got[ok], acc[rows[ok]])


def test_feature_scale_grad_dsv3_shape_sampled():
    """DeepSeek-V3 shard sizes: partials of every sampled row against the
    oracle, computed row by row."""
    w = synth.WORKLOADS["dsv3"]
    inp, g, r, rt, p_rows = _setup(w, 44)
    gp, op = _params(w)
    pre = synth._bf16(np.random.default_rng(45).standard_normal((w.R_cap, w.N1), dtype=np.float32))
    o = ops.dglu_bwd(g["dY"], g["W2"], pre.to(DEV), r["counts"], r["offsets"], w.F, gp, L.OUT_MXFP8,
                     row_scale=r["prob_perm"], row_dot=True, status=r["status"])
    dprob = ops.feature_scale_grad(o["row_dot"], r["row_of"], w.T, w.k)
    torch.cuda.synchronize()
    assert ops.read_status(r["status"]) == 0
    row_sum = np_(o["row_dot"]).astype(np.float64).sum(axis=1)
    rows = np.sort(np.random.default_rng(46).choice(rt.R_pad, 96, replace=False))
    dY = np_(inp["dY"])
    _dprob_check(row_sum, None, dY, np_(inp["W2"]), np_(pre), rt, op, w, rows)
    got = np_(dprob)
    ro = rt.row_of.reshape(w.T, w.k)
    assert np.all(got[ro < 0] == 0)
