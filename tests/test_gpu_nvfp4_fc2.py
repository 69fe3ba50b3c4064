"""GPU parity of the NVFP4 consumer ([MoE-Fusion] "Fusing MXFP8 and NVFP4
quantisation"): the block-scaled FC2 on NVFP4 operands (kind::mxf4nvf4, E4M3
scales per 16 elements, per-tensor scales), the column-wise NVFP4 weight cast
and the per-tensor amax, and the forward chain FC1 (NVFP4 mode: bf16 + amax)
-> NVFP4 cast -> NVFP4 FC2 against the oracle's own chain."""
import numpy as np
import pytest
import torch

from grouped_gemm_glu_gb300 import lib as L
from grouped_gemm_glu_gb300 import ops, synth
from oracle import moe_oracle as O
from parity import assert_bf16_close, assert_chain_close, assert_exact, np_

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _routing(counts, seed):
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).astype(np.int32)
    np.random.default_rng(seed).shuffle(ids)
    rt = O.route(ids.reshape(-1, 1), 0, len(counts))
    R_cap = (sum(counts) + 31 * len(counts) + 127) // 128 * 128
    cnt = torch.from_numpy(rt.counts.astype(np.int32)).to(DEV)
    off = torch.from_numpy(rt.offsets.astype(np.int32)).to(DEV)
    return rt, R_cap, cnt, off


def _nvfp4_operand(rows, K, seed, scale=1.0):
    """Random values quantised by the oracle: (codes, block scales, s_g)."""
    v = np.random.default_rng(seed).standard_normal((rows, K)).astype(np.float32) * scale
    sg = O.nvfp4_global_scale(float(np.max(np.abs(v))))
    q, s = O.nvfp4_quantize_rows(v, sg)
    return q, s, sg


@pytest.mark.parametrize("K,N", [(256, 256), (192, 320), (1536, 512), (2880, 288)])
def test_nvfp4_fc2_edge_counts(K, N):
    """Experts of 0, 1, 33, 128, 129 and 300 rows; K = 192 and 2880 leave a
    partial 256-element k-block, N = 320 and 288 a partial column tile."""
    counts = [0, 1, 33, 128, 129, 300]
    E = len(counts)
    rt, R_cap, cnt, off = _routing(counts, 1)
    Aq, As, sgA = _nvfp4_operand(R_cap, K, 2)
    Wq, Ws, sgW = _nvfp4_operand(E * N, K, 3, scale=1.0 / np.sqrt(K))
    Wq, Ws = Wq.reshape(E, N, K // 2), Ws.reshape(E, N, K // 16)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    sga, sgw = torch.tensor([float(sgA)], device=DEV), torch.tensor([float(sgW)], device=DEV)
    st = ops.new_status(DEV)
    y = ops.fc2_fwd_nvfp4(t(Aq), t(As), sga, t(Wq), t(Ws), sgw, cnt, off, status=st)
    torch.cuda.synchronize()
    assert ops.read_status(st) == 0
    ref = O.grouped_gemm_nvfp4(Aq[: rt.R_pad], As[: rt.R_pad], sgA, Wq, Ws, sgW, rt)
    assert_bf16_close(np_(y)[: rt.R_pad], O.bf16_round(ref), f"nvfp4 fc2 K={K} N={N}")


@pytest.mark.parametrize("R", [64, 48, 1536])
def test_nvfp4_weight_cast_and_amax_bit_exact(R):
    """The column-wise NVFP4 cast of a bf16 weight [E, F, H] and its per-tensor
    amax against the oracle on the same bf16 values: codes, scales and s_g
    bit-exact (R a multiple of 64: four blocks per thread; R = 48: one)."""
    rng = np.random.default_rng(4)
    W = synth._bf16(rng.standard_normal((3, R, 96), dtype=np.float32) * np.exp2(rng.integers(-4, 4, (3, 1, 96))))
    Wd = W.to(DEV)
    am = ops.amax_bf16(Wd)
    q, s, sg = ops.nvfp4_cast_cols(Wd, am)
    torch.cuda.synchronize()
    Wn = np_(W)
    assert float(am.item()) == float(np.max(np.abs(Wn)))
    sg_ref = O.nvfp4_global_scale(float(np.max(np.abs(Wn))))
    assert float(sg.item()) == float(sg_ref)
    for e in range(3):
        qr, sr = O.nvfp4_quantize_cols(Wn[e], sg_ref)
        assert_exact(np_(q[e]), qr, f"codes expert {e}")
        assert_exact(np_(s[e]), sr, f"scales expert {e}")


@pytest.mark.parametrize("act", ["geglu", "srelu"])
def test_nvfp4_forward_chain(act):
    """Skewed-config forward at a small size (T 1024, H 512, 64 experts with
    the Zipf routing, F 1536): FC1 in NVFP4 mode -> NVFP4 cast -> W2 amax and
    column-wise NVFP4 cast -> NVFP4 FC2, against the oracle's chain on the
    same inputs (each side rounds and quantises its own intermediates)."""
    w = synth.scaled(synth.WORKLOADS["skew" if act == "geglu" else "skew_srelu"], T=1024, H=512)
    inp = synth.make_inputs(w, 0)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    r = ops.route_permute(g["x"], g["topk_idx"], g["topk_prob"], w.E, w.R_cap)
    W1p = ops.repack_fc1(g["W1"]) if w.gated else g["W1"]
    fo = ops.fc1_fwd(r["x_perm"], W1p, r["counts"], r["offsets"], w.F, L.glu_params(act), L.OUT_NVFP4)
    aq, asc, sga = ops.nvfp4_cast(fo["y"], fo["amax"], r["counts"], r["offsets"])
    W2t = g["W2"]  # [E][F][H]: contraction of FC2 runs along F (its rows)
    wq, wsc, sgw = ops.nvfp4_cast_cols(W2t, ops.amax_bf16(W2t))
    st = ops.new_status(DEV)
    y = ops.fc2_fwd_nvfp4(aq, asc, sga, wq, wsc, sgw, r["counts"], r["offsets"], status=st)
    torch.cuda.synchronize()
    assert ops.read_status(st) == 0 and ops.read_status(fo["status"]) == 0
    rt = O.route(inp["topk_idx"].numpy(), 0, w.E)
    op = O.ActParams({"geglu": O.ACT_GEGLU, "srelu": O.ACT_SRELU}[act])
    W1 = np_(inp["W1"])
    ref1 = O.fc1_glu_fwd(O.permute(np_(inp["x"]), rt), O.repack_fc1(W1) if w.gated else W1, None, rt, op)
    yb = O.bf16_round(ref1.y)
    # the per-tensor amax of the NVFP4 mode is taken on the fp32 activation (Fc1Out.amax)
    sa_ref = O.nvfp4_global_scale(ref1.amax)
    qa, sa = O.nvfp4_quantize_rows(yb, sa_ref)
    W2 = np_(inp["W2"])
    sw_ref = O.nvfp4_global_scale(float(np.max(np.abs(W2))))
    qw = np.stack([O.nvfp4_quantize_cols(W2[e], sw_ref)[0] for e in range(w.E)])
    sw = np.stack([O.nvfp4_quantize_cols(W2[e], sw_ref)[1] for e in range(w.E)])
    ref = O.grouped_gemm_nvfp4(qa, sa, sa_ref, qw, sw, sw_ref, rt)
    assert_chain_close(np_(y)[: rt.R_pad], O.bf16_round(ref), f"nvfp4 chain {act}")


def test_layer_nvfp4_forward_step_and_graph():
    """MoeLayer with the NVFP4 forward on the skewed config (small T and H):
    the layer output against the oracle's NVFP4 chain, the FC2 weight gradient
    on the layer's own operands (the MXFP8 column cast of the bf16 FC1
    output), and one captured graph replaying to the eager results."""
    from grouped_gemm_glu_gb300.layer import MoeLayer
    w = synth.scaled(synth.WORKLOADS["skew"], T=1024, H=512)
    inp = synth.make_inputs(w, 3)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    layer = MoeLayer(g["W1"], g["W2"], w.T, w.k, w.R_cap, L.glu_params("geglu"), nvfp4_fwd=True)
    args = (g["x"], g["topk_idx"], g["topk_prob"], g["dOut"])
    layer.step(*args)
    torch.cuda.synchronize()
    assert ops.read_status(layer.status) == 0
    rt = O.route(inp["topk_idx"].numpy(), 0, w.E)
    Rp = rt.R_pad
    fo = O.fc1_glu_fwd(O.permute(np_(inp["x"]), rt), O.repack_fc1(np_(inp["W1"])), None, rt, O.ActParams(O.ACT_GEGLU))
    sa = O.nvfp4_global_scale(fo.amax)
    qa, sba = O.nvfp4_quantize_rows(O.bf16_round(fo.y), sa)
    W2 = np_(inp["W2"])
    sw = O.nvfp4_global_scale(float(np.max(np.abs(W2))))
    cols = [O.nvfp4_quantize_cols(W2[e], sw) for e in range(w.E)]
    y = O.bf16_round(O.grouped_gemm_nvfp4(qa, sba, sa, np.stack([c[0] for c in cols]),
                                          np.stack([c[1] for c in cols]), sw, rt))
    out = O.bf16_round(O.unpermute_combine(y, rt.row_of, inp["topk_prob"].numpy()))
    assert_chain_close(np_(layer.out), out, "NVFP4 layer output")
    deq = lambda q, s_: O.mx_dequantize(np_(q), np_(s_))
    qc, sc = O.mx_quantize_cols(np_(layer.a_y)[:Rp])   # the layer's bf16 FC1 output, cast by the oracle
    assert_exact(np_(layer.a_qc)[:, :Rp], qc, "column cast of the bf16 FC1 output")
    assert_exact(np_(layer.a_sc)[:, :Rp // 32], sc, "its scales")
    dW2 = O.grouped_wgrad(deq(layer.a_qc, layer.a_sc)[:, :Rp], deq(layer.dy_qc, layer.dy_sc)[:, :Rp], rt)
    assert_bf16_close(np_(layer.dW2), O.bf16_round(dW2), "dW2 on the layer's operands")
    eager = {k: getattr(layer, k).clone() for k in ("out", "dx", "dW1", "dW2", "dprob")}
    graph = layer.capture(*args)
    for t in eager:
        getattr(layer, t).zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert ops.read_status(layer.status) == 0
    for t, v in eager.items():
        assert torch.equal(getattr(layer, t), v), f"graph replay differs from eager: {t}"
