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
from parity import assert_bf16_close, assert_chain_close, np_

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def oracle_chain(inp, w):
    """float64 oracle of the whole step with the same MXFP8 casts."""
    f64 = lambda t: np_(t)
    prm = O.ActParams(O.ACT_SWIGLU)
    rt = O.route(inp["topk_idx"].numpy(), 0, w.E)
    Rp = rt.R_pad
    xp = O.permute(f64(inp["x"]), rt)
    W1p = O.repack_fc1(f64(inp["W1"]))
    W2 = f64(inp["W2"])
    fo = O.fc1_glu_fwd(xp, W1p, None, rt, prm)
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
    layer = MoeLayer(g["W1"], g["W2"], w.T, w.k, w.R_cap, L.glu_params("swiglu"))
    return layer, g


def _check(layer, inp, w):
    rt, out, dX, dW1, dW2, dprob, dx = oracle_chain(inp, w)
    Rp = rt.R_pad
    assert_chain_close(np_(layer.out), out, "layer output")
    real = rt.tok_of >= 0
    assert_chain_close(np_(layer.dprob), dprob, "dprob")
    assert_chain_close(np_(layer.dX_perm)[:Rp][real], dX[real], "dX_perm")
    assert_chain_close(np_(layer.dx), dx, "dx")
    assert_chain_close(np_(layer.dW1), dW1, "dW1 (packed rows)")
    assert_chain_close(np_(layer.dW2), dW2, "dW2")


def test_layer_step_matches_oracle():
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w, seed=21)
    layer, g = _layer(w, inp)
    layer.step(g["x"], g["topk_idx"], g["topk_prob"], g["dOut"])
    torch.cuda.synchronize()
    assert ops.read_status(layer.status) == 0
    _check(layer, inp, w)


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
