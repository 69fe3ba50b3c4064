"""A whole layer step (forward + backward) through the C ABI against the
oracle's chain, and its capture as one CUDA graph: replaying the graph on new
routing (new counts, no re-capture, no host sync) gives the eager results."""
import numpy as np
import pytest
import torch

from grouped_gemm_glu_gb300 import lib as L
from grouped_gemm_glu_gb300 import ops, synth
from grouped_gemm_glu_gb300.layer import MoeLayer
from oracle import moe_oracle as O
from parity import assert_bf16_close, assert_chain_close, assert_exact, np_, untile_weight_scales

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _acts(w):
    """(kernel parameters, oracle parameters) of the workload's activation."""
    if w.gpt_oss:
        return (L.glu_params("swiglu", alpha=1.702, up_offset=1.0, gate_lo=-7.0, gate_hi=7.0),
                O.ActParams(O.ACT_SWIGLU, alpha=1.702, up_offset=1.0, gate_lo=-7.0, gate_hi=7.0))
    return L.glu_params("swiglu"), O.ActParams(O.ACT_SWIGLU)


def oracle_chain(inp, w):
    """float64 oracle of the whole step with the same MXFP8 casts."""
    f64 = lambda t: np_(t)
    prm = _acts(w)[1]
    rt = O.route(inp["topk_idx"].numpy(), 0, w.E)
    Rp = rt.R_pad
    xp = O.permute(f64(inp["x"]), rt)
    W1p = O.repack_fc1(f64(inp["W1"]))
    W2 = f64(inp["W2"])
    b1p = None if inp.get("b1") is None else O.repack_fc1(f64(inp["b1"])[..., None])[..., 0]
    fo = O.fc1_glu_fwd(xp, W1p, b1p, rt, prm)
    a = O.mx_dequantize(*O.mx_quantize_rows(fo.y))
    W2d = np.stack([O.mx_dequantize(*O.mx_quantize_cols(W2[e])) for e in range(w.E)])
    y = O.bf16_round(O.grouped_gemm_rows(a, W2d, rt))
    out = O.bf16_round(O.unpermute_combine(y, rt.row_of, inp["topk_prob"].numpy()))
    dY, dprob = O.combine_bwd(f64(inp["dOut"]), y, rt.row_of, inp["topk_prob"].numpy(), Rp)
    dY = O.bf16_round(dY)
    d = O.dglu_bwd(dY, W2, fo.pre_bf16, rt, prm)
    W1q = np.stack([O.mx_dequantize(*O.mx_quantize_cols(W1p[e])) for e in range(w.E)])
    dX = O.bf16_round(O.grouped_gemm_rows(O.mx_dequantize(*O.mx_quantize_rows(d)), W1q, rt))
    dW1 = O.bf16_round(O.grouped_wgrad(O.mx_dequantize(*O.mx_quantize_cols(d)),
                                       O.mx_dequantize(*O.mx_quantize_cols(xp)), rt))
    dW2 = O.bf16_round(O.grouped_wgrad(O.mx_dequantize(*O.mx_quantize_cols(fo.y)),
                                       O.mx_dequantize(*O.mx_quantize_cols(dY)), rt))
    dx = O.bf16_round(O.permute_bwd(dX, rt.row_of, w.T, w.k))
    return rt, out, dX, dW1, dW2, dprob, dx


def _layer(w, inp):
    g = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    layer = MoeLayer(g["W1"], g["W2"], w.T, w.k, w.R_cap, _acts(w)[0], b1=g.get("b1"))
    return layer, g


def _check_stagewise(layer, rt):
    """The backward GEMMs against the oracle fed the layer's own quantized
    operands (each GEMM on its exact inputs; no upstream rounding involved)."""
    Rp = rt.R_pad
    deq = lambda q, s_: O.mx_dequantize(np_(q), np_(s_))
    dW2 = O.grouped_wgrad(deq(layer.a_qc, layer.a_sc)[:, :Rp], deq(layer.dy_qc, layer.dy_sc)[:, :Rp], rt)
    assert_bf16_close(np_(layer.dW2), O.bf16_round(dW2), "dW2 on the layer's operands")
    dW1 = O.grouped_wgrad(deq(layer.d_qc, layer.d_sc)[:, :Rp], deq(layer.x_qc, layer.x_sc)[:, :Rp], rt)
    assert_bf16_close(np_(layer.dW1), O.bf16_round(dW1), "dW1 on the layer's operands")
    W1s = (np_(layer.W1s_p) if layer.fc1_mxfp8 else
           untile_weight_scales(np_(layer.W1s), rt.E, layer.N1, layer.H))
    W1q = np.stack([O.mx_dequantize(np_(layer.W1q[e]), W1s[e]) for e in range(rt.E)])
    dX = O.grouped_gemm_rows(deq(layer.d_q, layer.d_s)[:Rp], W1q, rt)
    real = rt.tok_of >= 0
    assert_bf16_close(np_(layer.dX_perm)[:Rp][real], O.bf16_round(dX)[real], "dX on the layer's operands")


def _check(layer, inp, w, dprob_frac=0.999, wgrad_chain_bound=0.02):
    rt, out, dX, dW1, dW2, dprob, dx = oracle_chain(inp, w)
    Rp = rt.R_pad
    assert_chain_close(np_(layer.out), out, "layer output")
    real = rt.tok_of >= 0
    # dprob = <dOut, y_perm> over H: on the layer's own y_perm it is an fp32 dot
    # (tight); against the oracle chain it inherits every upstream rounding
    _, dprob_own = O.combine_bwd(np_(inp["dOut"]), np_(layer.y_perm)[:Rp], rt.row_of, inp["topk_prob"].numpy(), Rp)
    assert np.allclose(np_(layer.dprob), dprob_own, rtol=1e-4, atol=1e-4), "dprob on the layer's y_perm"
    assert_chain_close(np_(layer.dprob), dprob, "dprob", frac=dprob_frac)
    assert_chain_close(np_(layer.dX_perm)[:Rp][real], dX[real], "dX_perm")
    assert_chain_close(np_(layer.dx), dx, "dx")
    assert_chain_close(np_(layer.dW1), dW1, "dW1 (packed rows)", max_frac=wgrad_chain_bound)
    assert_chain_close(np_(layer.dW2), dW2, "dW2", max_frac=wgrad_chain_bound)


def test_layer_step_matches_oracle():
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w, seed=21)
    layer, g = _layer(w, inp)
    layer.step(g["x"], g["topk_idx"], g["topk_prob"], g["dOut"])
    torch.cuda.synchronize()
    assert ops.read_status(layer.status) == 0
    _check(layer, inp, w)


def test_layer_step_gptoss_shapes():
    """A whole step at the GPT-OSS-shaped layer's widths (H = F = 2880, not
    multiples of 128: partial last k-blocks and column tiles in FC2, dX and
    the weight gradients), with its bias, clamp, alpha and (up + 1).  Fewer
    tokens and 4 experts (every token reaches all of them: 256 rows each, as
    many as in the DeepSeek-V3 shard) so that the float64 oracle chain stays
    quick while each weight-gradient element still sums 256 products."""
    w = synth.scaled(synth.WORKLOADS["gptoss"], T=256, E=4, n_experts=4)
    inp = synth.make_inputs(w, seed=23)
    layer, g = _layer(w, inp)
    layer.step(g["x"], g["topk_idx"], g["topk_prob"], g["dOut"])
    torch.cuda.synchronize()
    assert ops.read_status(layer.status) == 0
    # Each GEMM is first checked on the layer's own quantized operands (tight).
    # Against the float64 chain, dprob sums 2880 products whose y factors carry
    # the chain's MXFP8 code flips (one E4M3 step on <= 0.1% of codes, allowed
    # per element), and the weight gradients sum 256 products of operands
    # re-quantized after two such stages, where a scale one step apart (allowed
    # near a power of two) moves a whole 32-row block of codes together: the
    # chain rule takes 99% for dprob and 5% of the max for dW1 / dW2.
    _check_stagewise(layer, O.route(inp["topk_idx"].numpy(), 0, w.E))
    _check(layer, inp, w, dprob_frac=0.99, wgrad_chain_bound=0.05)


def test_layer_graph_replay_new_routing():
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w, seed=22)
    layer, g = _layer(w, inp)
    graph = layer.capture(g["x"], g["topk_idx"], g["topk_prob"], g["dOut"])
    # new batch: different tokens, routing and counts, copied into the captured buffers
    new = synth.make_inputs(synth.scaled(w), seed=23)
    new["W1"], new["W2"] = inp["W1"], inp["W2"]
    for k in ("x", "topk_idx", "topk_prob", "dOut"):
        g[k].copy_(new[k].to(DEV))
    graph.replay()
    torch.cuda.synchronize()
    assert ops.read_status(layer.status) == 0
    got = {k: getattr(layer, k).clone() for k in ("out", "dprob", "dX_perm", "dx", "dW1", "dW2", "counts")}
    assert not torch.equal(got["counts"].cpu(), torch.from_numpy(O.route(inp["topk_idx"].numpy(), 0, w.E)
                                                                 .counts.astype(np.int32)))
    _check(layer, new, w)
    # eager step on the same inputs gives identical bits (deterministic kernels)
    layer.step(g["x"], g["topk_idx"], g["topk_prob"], g["dOut"])
    torch.cuda.synchronize()
    for k in ("out", "dprob", "dX_perm", "dx", "dW1", "dW2"):
        assert torch.equal(getattr(layer, k), got[k]), k


def test_unfused_path_matches_oracle():
    """The ablation baseline (bf16 GEMM -> activation -> quantize kernels,
    forward and backward) against the oracle with the same rounding points:
    the unfused path rounds the GEMM output to bf16, applies the activation
    to that, rounds again to bf16 and quantises the bf16 tensor."""
    from parity import assert_mx_close
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w, seed=24)
    layer, g = _layer(w, inp)
    layer.step(g["x"], g["topk_idx"], g["topk_prob"], g["dOut"])
    layer.run(layer.forward_unfused_calls())
    layer.run(layer.backward_unfused_calls(g["dY"]))
    torch.cuda.synchronize()
    assert ops.read_status(layer.status) == 0
    u = layer._u
    prm = O.ActParams(O.ACT_SWIGLU)
    rt = O.route(inp["topk_idx"].numpy(), 0, w.E)
    R = rt.R_pad
    real = rt.tok_of >= 0
    fo = O.fc1_glu_fwd(O.permute(np_(inp["x"]), rt), O.repack_fc1(np_(inp["W1"])), None, rt, prm)
    assert_bf16_close(np_(u["pre"])[:R], fo.pre_bf16, "unfused pre")
    y = O.act_fwd(*O.unpack_glu_cols(fo.pre_bf16), prm)
    y[~real] = 0
    yb = O.bf16_round(y).astype(np.float32)
    assert_bf16_close(np_(u["y"])[:R], yb, "unfused y")
    band = 2.0 ** -7   # the bf16 roundings before the quantiser can move a block max by one bf16 step
    q, s_ = O.mx_quantize_rows(yb)
    assert_mx_close(np_(u["a_q"])[:R], np_(u["a_s"])[:R], q, s_, yb, "unfused a rows", rel_band=band)
    qc, sc = O.mx_quantize_cols(yb)
    assert_mx_close(np_(u["a_qc"])[:, :R], np_(u["a_sc"])[:, :R // 32], qc, sc, yb.T, "unfused a cols", rel_band=band)
    dY = np_(inp["dY"])[:R].copy()
    da = O.bf16_round(O.grouped_gemm_rows(dY, np_(inp["W2"]), rt))
    assert_bf16_close(np_(u["da"])[:R], da, "unfused da")
    du, dg = O.act_bwd(*O.unpack_glu_cols(fo.pre_bf16), da, prm)
    d = O.pack_glu_cols(du, dg)
    d[~real] = 0
    db = O.bf16_round(d).astype(np.float32)
    assert_bf16_close(np_(u["d"])[:R], db, "unfused dFC1")
    q, s_ = O.mx_quantize_rows(db)
    assert_mx_close(np_(u["d_q"])[:R], np_(u["d_s"])[:R], q, s_, db, "unfused dFC1 rows", rel_band=band)


def test_dense_mode_single_expert():
    """Dense MLP / shared expert: one local expert that every token uses
    (E = 1, top-1), through the same layer step and kernels."""
    w = synth.Workload("dense", 640, 256, 1, 1, 1, 512, "swiglu", "mxfp8", "normal")
    inp = synth.make_inputs(w, seed=25)
    assert int((inp["topk_idx"] == 0).sum()) == w.T
    layer, g = _layer(w, inp)
    layer.step(g["x"], g["topk_idx"], g["topk_prob"], g["dOut"])
    torch.cuda.synchronize()
    assert ops.read_status(layer.status) == 0
    assert int(layer.counts[0]) == w.T
    _check(layer, inp, w)


def test_layer_step_mxfp8_fc1():
    """The layer with the MXFP8-input FC1: both MXFP8 copies of W1 from one
    read (bit-exact against the oracle's two casts), the row-wise cast of
    x_perm (bit-exact), FC1's saved pre-activations against the oracle FC1 on
    the dequantised operands, the backward GEMMs on the layer's own operands,
    and one captured graph replaying to the eager results."""
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w, seed=24)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    kp, prm = _acts(w)
    layer = MoeLayer(g["W1"], g["W2"], w.T, w.k, w.R_cap, kp, fc1_mxfp8=True)
    args = (g["x"], g["topk_idx"], g["topk_prob"], g["dOut"])
    layer.step(*args)
    torch.cuda.synchronize()
    assert ops.read_status(layer.status) == 0
    names = [n for n, _ in layer.step_calls(*args)]
    assert "quant_w1_dual" in names and "fc1_mxfp8" in names and "quant_w1" not in names
    rt = O.route(inp["topk_idx"].numpy(), 0, w.E)
    Rp = rt.R_pad
    W1p = O.repack_fc1(np_(inp["W1"]))
    for e in range(w.E):
        q, s_ = O.mx_quantize_rows(W1p[e])
        assert_exact(np_(layer.W1qr[e]), q, "W1 rows codes")
        assert_exact(np_(layer.W1sr[e]), s_, "W1 rows scales")
        q, s_ = O.mx_quantize_cols(W1p[e])
        assert_exact(np_(layer.W1q[e]), q, "W1 columns codes")
        assert_exact(np_(layer.W1s_p[e]), s_, "W1 columns scales")
    xp = O.permute(np_(inp["x"]), rt)
    xq, xs = O.mx_quantize_rows(xp)
    assert_exact(np_(layer.x_qr)[:Rp], xq, "x_perm rows codes")
    assert_exact(np_(layer.x_sr)[:Rp], xs, "x_perm rows scales")
    fo = O.fc1_glu_fwd(O.mx_dequantize(xq, xs), np.stack([O.mx_dequantize(*O.mx_quantize_rows(W1p[e]))
                                                          for e in range(w.E)]), None, rt, prm)
    assert_bf16_close(np_(layer.pre)[:Rp], fo.pre_bf16, "FC1 pre-activations")
    _check_stagewise(layer, rt)
    eager = {k: getattr(layer, k).clone() for k in ("out", "dx", "dW1", "dW2", "dprob")}
    graph = layer.capture(*args)
    for t in eager:
        getattr(layer, t).zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert ops.read_status(layer.status) == 0
    for t, v in eager.items():
        assert torch.equal(getattr(layer, t), v), f"graph replay differs from eager: {t}"
