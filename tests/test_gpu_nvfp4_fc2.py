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
from parity import (assert_bf16_close, assert_chain_close, assert_exact, np_, nvfp4_tiled_pad,
                    untile_nvfp4_weight_scales)

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


@pytest.mark.parametrize("R,C", [(64, 96), (48, 96), (1536, 96), (64, 45), (48, 45)])
def test_nvfp4_weight_cast_and_amax_bit_exact(R, C):
    """The column-wise NVFP4 cast of a bf16 weight [E, F, H] and its per-tensor
    amax against the oracle on the same bf16 values: codes, scales and s_g
    bit-exact.  R = 1536, C = 96: 128 x 128 tiles staged through shared
    memory (a partial column tile); otherwise the direct kernels: R a
    multiple of 64 four blocks per thread, R = 48 one; C even two columns
    per thread, C odd one."""
    rng = np.random.default_rng(4)
    W = synth._bf16(rng.standard_normal((3, R, C), dtype=np.float32) * np.exp2(rng.integers(-4, 4, (3, 1, C))))
    Wd = W.to(DEV)
    am = ops.amax_bf16(Wd)
    st = ops.new_status(DEV)
    q, s, sg = ops.nvfp4_cast_cols(Wd, am, status=st)
    torch.cuda.synchronize()
    assert ops.read_status(st) == 0
    Wn = np_(W)
    assert float(am.item()) == float(np.max(np.abs(Wn)))
    sg_ref = O.nvfp4_global_scale(float(np.max(np.abs(Wn))))
    assert float(sg.item()) == float(sg_ref)
    for e in range(3):
        qr, sr = O.nvfp4_quantize_cols(Wn[e], sg_ref)
        assert_exact(np_(q[e]), qr, f"codes expert {e}")
        assert_exact(np_(s[e]), sr, f"scales expert {e}")


@pytest.mark.parametrize("R,C", [(1536, 512), (384, 264), (640, 392)])
def test_nvfp4_tiled_weight_scales(R, C):
    """moe_nvfp4_cast_cols_tiled: the same codes and (after un-permuting the
    tensor-core order) the same scales as the plain cast, bit for bit, with
    zero scales past R and C in a buffer that started as 0xAA.  R = 384 and
    640 end in half a 256-row k-block; C = 264 ends in the first half of a
    256-column tile (its second half is written as zeros), C = 392 inside a
    second half."""
    E = 3
    rng = np.random.default_rng(R + C)
    W = synth._bf16(rng.standard_normal((E, R, C), dtype=np.float32) * np.exp2(rng.integers(-4, 4, (E, 1, C))))
    Wd = W.to(DEV)
    am = ops.amax_bf16(Wd)
    q0, s0, sg0 = ops.nvfp4_cast_cols(Wd, am)
    lib = L.load()
    q = torch.full((E, C, R // 2), 0xAA, dtype=torch.uint8, device=DEV)
    s = torch.full((lib.moe_nvfp4_tiled_scale_bytes(E, R, C),), 0xAA, dtype=torch.uint8, device=DEV)
    sg = torch.zeros(1, dtype=torch.float32, device=DEV)
    st = ops.new_status(DEV)
    ops.nvfp4_cast_cols(Wd, am, status=st, tiled=True, out=(q, s, sg))
    torch.cuda.synchronize()
    assert ops.read_status(st) == 0
    assert float(sg.item()) == float(sg0.item())
    assert torch.equal(q, q0), "codes"
    assert_exact(untile_nvfp4_weight_scales(np_(s), E, R, C), np_(s0), "scales")
    assert not nvfp4_tiled_pad(np_(s), E, R, C).any(), "pad scales"


@pytest.mark.parametrize("K,N", [(1536, 512), (384, 288)])
def test_nvfp4_fc2_tiled_weight_bit_identical(K, N):
    """FC2 on an NVFP4 weight cast with tiled scales (MOE_IN_NVFP4_TILED, no
    weight-scale re-tiling in the call) returns the same bits as on the plain
    cast of the same weight.  K = 384 ends in half a k-block, N = 288 in a
    partial column tile whose missing half holds zero scales."""
    counts = [0, 1, 33, 128, 129, 300]
    E = len(counts)
    rt, R_cap, cnt, off = _routing(counts, 5)
    Aq, As, sgA = _nvfp4_operand(R_cap, K, 6)
    rng = np.random.default_rng(7)
    W = synth._bf16(rng.standard_normal((E, K, N), dtype=np.float32) / np.sqrt(K)).to(DEV)  # [E][K][N]
    am = ops.amax_bf16(W)
    wq, ws, sgw = ops.nvfp4_cast_cols(W, am)
    wq_t, ws_t, sgw_t = ops.nvfp4_cast_cols(W, am, tiled=True)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    sga = torch.tensor([float(sgA)], device=DEV)
    st = ops.new_status(DEV)
    y0 = ops.fc2_fwd_nvfp4(t(Aq), t(As), sga, wq, ws, sgw, cnt, off, status=st)
    y1 = ops.fc2_fwd_nvfp4(t(Aq), t(As), sga, wq_t, ws_t, sgw_t, cnt, off, status=st, w_tiled=True)
    torch.cuda.synchronize()
    assert ops.read_status(st) == 0
    Rp = rt.R_pad
    assert torch.equal(y0[:Rp].view(torch.int16), y1[:Rp].view(torch.int16))
    ref = O.grouped_gemm_nvfp4(Aq[:Rp], As[:Rp], sgA, np_(wq), np_(ws), float(sgw.item()), rt)
    assert_bf16_close(np_(y1)[:Rp], O.bf16_round(ref), f"nvfp4 fc2 tiled weight K={K} N={N}")


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


def _zero_codes_as_one(q):
    """E2M1 codes 0x0 and 0x8 (+0, -0) both mean zero; map -0 to +0 in both nibbles."""
    lo, hi = q & 0xF, q >> 4
    return (np.where(lo == 8, 0, lo) | (np.where(hi == 8, 0, hi) << 4)).astype(np.uint8)


def _assert_rot_cast(q, s, sg, v, signs, what):
    """A rotated column-wise NVFP4 cast of the layer's bf16 tensor v [Rp, C]
    against the oracle's cast of the same tensor under the same s_g: codes and
    scales equal on >= 99.9% (a rotated value the fp32 butterfly and the
    float64 oracle round differently may cross an E2M1 / E4M3 boundary), the
    dequantised values within two E2M1 steps of their block everywhere."""
    Rp = v.shape[0]
    qr, sr = O.nvfp4_rht_cast_cols(v, signs, sg)
    qg, sgc = np_(q)[:, : Rp // 2], np_(s)[:, : Rp // 16]
    assert (_zero_codes_as_one(qg) == _zero_codes_as_one(qr)).mean() >= 0.999, what
    assert (sgc == sr).mean() >= 0.999, what
    dg, dr = O.nvfp4_dequantize(qg, sgc, sg), O.nvfp4_dequantize(qr, sr, sg)
    blk = np.repeat(np.maximum(O.e4m3_decode(sgc), O.e4m3_decode(sr)), 16, axis=1) / float(sg)
    assert np.all(np.abs(dg - dr) <= 2.0 * blk * (1 + 1e-6)), what


SIGNS = 0x6A5D


@pytest.mark.parametrize("F", [1536, 1600])
def test_layer_nvfp4_step_and_graph(F):
    """MoeLayer in NVFP4 mode on the skewed config (small T and H; F = 1536
    casts the weights with their scales in the tensor-core order, F = 1600 (F
    % 128 = 64) with the plain scale layout and the direct column cast of W2,
    a k-block of 256 ending half full).  Forward:
    the layer output against the oracle's NVFP4 chain.  Backward: dFC1 and its
    two amaxes against the oracle's dGLU on the layer's dY and saved pre; every
    NVFP4 cast against the oracle's cast of the layer's own bf16 tensor; dX,
    dW1 and dW2 against the oracle's GEMMs on the layer's own NVFP4 operands;
    dx through the permute backward.  Then one captured graph replays to the
    eager results."""
    from grouped_gemm_glu_gb300.layer import MoeLayer
    w = synth.scaled(synth.WORKLOADS["skew"], T=1024, H=512, F=F)
    inp = synth.make_inputs(w, 3)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    prm = O.ActParams(O.ACT_GEGLU)
    layer = MoeLayer(g["W1"], g["W2"], w.T, w.k, w.R_cap, L.glu_params("geglu"), nvfp4=True, rht_signs=SIGNS)
    args = (g["x"], g["topk_idx"], g["topk_prob"], g["dOut"])
    layer.step(*args)
    torch.cuda.synchronize()
    assert ops.read_status(layer.status) == 0
    assert layer.w4_tiled == (F % 128 == 0)
    rt = O.route(inp["topk_idx"].numpy(), 0, w.E)
    Rp = rt.R_pad
    fo = O.fc1_glu_fwd(O.permute(np_(inp["x"]), rt), O.repack_fc1(np_(inp["W1"])), None, rt, prm)
    sa = O.nvfp4_global_scale(fo.amax)
    qa, sba = O.nvfp4_quantize_rows(O.bf16_round(fo.y), sa)
    W2 = np_(inp["W2"])
    sw = O.nvfp4_global_scale(float(np.max(np.abs(W2))))
    cols = [O.nvfp4_quantize_cols(W2[e], sw) for e in range(w.E)]
    y = O.bf16_round(O.grouped_gemm_nvfp4(qa, sba, sa, np.stack([c[0] for c in cols]),
                                          np.stack([c[1] for c in cols]), sw, rt))
    out = O.bf16_round(O.unpermute_combine(y, rt.row_of, inp["topk_prob"].numpy()))
    assert_chain_close(np_(layer.out), out, "NVFP4 layer output")

    # dFC1 from the layer's own dY and saved pre; its amax and rotated amax (fp32, before bf16)
    d_ref = O.dglu_bwd(np_(layer.dY_perm)[:Rp], W2, np_(layer.pre)[:Rp], rt, prm)
    d = np_(layer.d_y)[:Rp]
    assert_bf16_close(d, O.bf16_round(d_ref), "dFC1")
    assert abs(float(layer.d_amax.item()) / np.max(np.abs(d_ref)) - 1) < 1e-2
    assert abs(float(layer.d_rht.item()) / O.rht_transposed_amax(d_ref, SIGNS) - 1) < 1e-2
    # NVFP4 rows of dFC1 and W1 along 2F: the data gradient's operands
    sd = O.nvfp4_global_scale(float(layer.d_amax.item()))
    assert float(layer.d_sg.item()) == float(sd)
    qd, sbd = O.nvfp4_quantize_rows(d, sd)
    assert_exact(_zero_codes_as_one(np_(layer.d_q4)[:Rp]), _zero_codes_as_one(qd), "dFC1 NVFP4 codes")
    assert_exact(np_(layer.d_s4)[:Rp], sbd, "dFC1 NVFP4 scales")
    W1p = np_(layer.W1p)
    s1 = O.nvfp4_global_scale(float(np.max(np.abs(W1p))))
    assert float(layer.w1_sg.item()) == float(s1)
    c1 = [O.nvfp4_quantize_cols(W1p[e], s1) for e in range(w.E)]
    assert_exact(np_(layer.W1q4), np.stack([c[0] for c in c1]), "W1 NVFP4 codes (along 2F)")
    W1s4 = np_(layer.W1s4)
    if layer.w4_tiled:  # scales in the tensor-core order: un-permute them
        W1s4 = untile_nvfp4_weight_scales(W1s4, w.E, W1p.shape[1], W1p.shape[2])
    assert_exact(W1s4, np.stack([c[1] for c in c1]), "W1 NVFP4 scales")
    dX = O.grouped_gemm_nvfp4(np_(layer.d_q4)[:Rp], np_(layer.d_s4)[:Rp], float(layer.d_sg.item()),
                              np_(layer.W1q4), W1s4, float(layer.w1_sg.item()), rt)
    assert_bf16_close(np_(layer.dX_perm)[:Rp], O.bf16_round(dX), "NVFP4 dX on the layer's operands")
    dx = O.permute_bwd(np_(layer.dX_perm)[:Rp], rt.row_of, w.T, w.k)
    assert_bf16_close(np_(layer.dx), O.bf16_round(dx), "dx")

    # rotated column-wise casts and the weight gradients
    rot = {"d": (d, layer.d_rht), "x": (np_(layer.x_perm)[:Rp], layer.x_ramax),
           "a": (np_(layer.a_y)[:Rp], layer.a_ramax), "dy": (np_(layer.dY_perm)[:Rp], layer.dy_ramax)}
    for n, (v, am) in rot.items():
        if n != "d":
            assert abs(float(am.item()) / O.rht_transposed_amax(v, SIGNS) - 1) < 1e-6, n
        sg = getattr(layer, f"{n}_rsg")
        assert abs(float(sg.item()) / float(O.nvfp4_global_scale(float(am.item()))) - 1) < 1e-6, n
        _assert_rot_cast(getattr(layer, f"{n}_rq"), getattr(layer, f"{n}_rs"), float(sg.item()), v, SIGNS,
                         f"rotated cast of {n}")
    op = lambda n: (np_(getattr(layer, f"{n}_rq"))[:, : Rp // 2], np_(getattr(layer, f"{n}_rs"))[:, : Rp // 16],
                    float(getattr(layer, f"{n}_rsg").item()))
    dW1 = O.grouped_wgrad_nvfp4(*op("d"), *op("x"), rt)
    assert_bf16_close(np_(layer.dW1), O.bf16_round(dW1), "NVFP4 dW1 on the layer's operands")
    dW2 = O.grouped_wgrad_nvfp4(*op("a"), *op("dy"), rt)
    assert_bf16_close(np_(layer.dW2), O.bf16_round(dW2), "NVFP4 dW2 on the layer's operands")

    eager = {k: getattr(layer, k).clone() for k in ("out", "dx", "dW1", "dW2", "dprob")}
    graph = layer.capture(*args)
    for t in eager:
        getattr(layer, t).zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert ops.read_status(layer.status) == 0
    for t, v in eager.items():
        assert torch.equal(getattr(layer, t), v), f"graph replay differs from eager: {t}"
