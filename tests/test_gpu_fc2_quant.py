"""GPU parity of GroupGemm + Quantize (moe_grouped_fc2_fwd with MXFP8 or bf16
operands, bf16 / MXFP8 row + column / NVFP4 outputs) and of the FC1 bias
gradient written by the fused dGLU backward, against the oracle."""
import math

import numpy as np
import pytest
import torch

from grouped_gemm_glu_gb300 import lib as L
from grouped_gemm_glu_gb300 import ops, synth
from oracle import moe_oracle as O
from parity import assert_bf16_close, assert_exact, assert_mx_close, np_, untile_weight_scales

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


def _operands(E, K, N, R_cap, seed, mx):
    if mx:
        Aq, As = synth.random_mxfp8(R_cap, K, seed + 1)
        Wq, Ws = synth.random_mxfp8(E * N, K, seed + 2)
        Wq, Ws = Wq.view(E, N, K), Ws.view(E, N, K // 32)
        A = O.mx_dequantize(Aq.numpy(), As.numpy())
        W = O.mx_dequantize(Wq.numpy(), Ws.numpy())
        return (Aq.to(DEV), As.to(DEV), Wq.to(DEV), Ws.to(DEV)), A, W
    rng = np.random.default_rng(seed)
    Ab = synth._bf16(rng.standard_normal((R_cap, K), dtype=np.float32))
    Wb = synth._bf16(rng.standard_normal((E, N, K), dtype=np.float32) / np.sqrt(K))
    return (Ab.to(DEV), None, Wb.to(DEV), None), np_(Ab), np_(Wb)


def _check(o, out_mode, y, rt, cols=None, what=""):
    """y: oracle float32 [R_pad, N] (pad rows 0); cols: sampled 32-column blocks."""
    R = rt.R_pad
    cs = np.arange(y.shape[1]) if cols is None else np.concatenate([np.arange(c, c + 32) for c in cols])
    yv = y[:, cs]
    if out_mode == L.OUT_BF16:
        assert_bf16_close(np_(o)[:R][:, cs], O.bf16_round(yv), what + " y")
        return
    if out_mode == L.OUT_NVFP4:
        assert_bf16_close(np_(o["y"])[:R][:, cs], O.bf16_round(yv), what + " y")
        if cols is None:
            assert math.isclose(float(o["amax"].item()), float(np.max(np.abs(y))), rel_tol=1e-3)
        return
    q, s = O.mx_quantize_rows(yv)
    sb = (cs[::32] // 32)
    assert_mx_close(np_(o["q_row"])[:R][:, cs], np_(o["s_row"])[:R][:, sb], q, s, yv, what + " row-wise")
    if "q_col" in o:
        qc, sc = O.mx_quantize_cols(yv)
        assert_mx_close(np_(o["q_col"])[cs][:, :R], np_(o["s_col"])[cs][:, :R // 32], qc, sc, yv.T,
                        what + " col-wise")


@pytest.mark.parametrize("mx", [True, False])
@pytest.mark.parametrize("out_mode", [L.OUT_MXFP8, L.OUT_BF16, L.OUT_NVFP4])
def test_fc2_quant_edge_counts(mx, out_mode):
    """Experts of 0, 1, 33, 128, 129 and 300 rows; K = 256, N = 320 (the last
    256-wide column tile is partial)."""
    counts = [0, 1, 33, 128, 129, 300]
    E, K, N = len(counts), 256, 320
    rt, R_cap, cnt, off = _routing(counts, 1)
    (a, a_s, w, w_s), A, W = _operands(E, K, N, R_cap, 5, mx)
    o = ops.fc2_fwd(a, a_s, w, w_s, cnt, off, out_mode=out_mode)
    torch.cuda.synchronize()
    if out_mode != L.OUT_BF16:
        assert ops.read_status(o["status"]) == 0
    y = O.grouped_gemm_quant_fwd(A[: rt.R_pad], W, rt)
    _check(o, out_mode, y, rt, what=f"mx={mx}")


@pytest.mark.parametrize("mx", [True, False])
def test_fc2_quant_dsv3_shape_sampled(mx):
    """FC2 of the DeepSeek-V3 shard (K = F = 2048, N = H = 7168, 32 experts
    of ~256 rows) with MXFP8 row + column outputs; three experts in full
    over 24 sampled 32-column blocks."""
    counts = list(np.random.default_rng(2).integers(200, 320, 32))
    E, K, N = 32, 2048, 7168
    rt, R_cap, cnt, off = _routing(counts, 2)
    (a, a_s, w, w_s), A, W = _operands(E, K, N, R_cap, 7, mx)
    o = ops.fc2_fwd(a, a_s, w, w_s, cnt, off, out_mode=L.OUT_MXFP8)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    cols = sorted(np.random.default_rng(3).choice(N // 32, 24, replace=False) * 32)
    cs = np.concatenate([np.arange(c, c + 32) for c in cols])
    rows = np.concatenate([np.arange(int(rt.offsets[e]), int(rt.offsets[e + 1])) for e in (0, 13, 31)])
    y = np.zeros((rt.R_pad, len(cs)), dtype=np.float32)
    for e in (0, 13, 31):
        r0, n = int(rt.offsets[e]), int(rt.counts[e])
        y[r0:r0 + n] = (A[r0:r0 + n] @ W[e][cs].T).astype(np.float32)
    yv = y[rows]
    q, s = O.mx_quantize_rows(yv)
    assert_mx_close(np_(o["q_row"])[rows][:, cs], np_(o["s_row"])[rows][:, cs[::32] // 32], q, s, yv,
                    f"dsv3 mx={mx} row-wise")
    qc, sc = O.mx_quantize_cols(yv)
    assert_mx_close(np_(o["q_col"])[cs][:, rows], np_(o["s_col"])[cs][:, rows[::32] // 32], qc, sc, yv.T,
                    f"dsv3 mx={mx} col-wise")


def test_fc2_bf16_operands_match_mxfp8_path_on_exact_values():
    """bf16 and MXFP8 operands that hold the same values (E4M3 codes with
    scale 2^0 are exact in bf16) give the same bf16 result."""
    counts = [5, 70, 0, 200]
    E, K, N = len(counts), 192, 256
    rt, R_cap, cnt, off = _routing(counts, 4)
    Aq, _ = synth.random_mxfp8(R_cap, K, 11)
    Wq, _ = synth.random_mxfp8(E * N, K, 12)
    As = torch.full((R_cap, K // 32), 127, dtype=torch.uint8)
    Ws = torch.full((E * N, K // 32), 127, dtype=torch.uint8)
    A = torch.from_numpy(O.mx_dequantize(Aq.numpy(), As.numpy()).astype(np.float32)).to(torch.bfloat16)
    W = torch.from_numpy(O.mx_dequantize(Wq.numpy(), Ws.numpy()).astype(np.float32)).to(torch.bfloat16)
    y_mx = ops.fc2_fwd(Aq.to(DEV), As.to(DEV), Wq.view(E, N, K).to(DEV), Ws.view(E, N, K // 32).to(DEV), cnt, off)
    y_bf = ops.fc2_fwd(A.to(DEV), None, W.view(E, N, K).to(DEV), None, cnt, off)
    torch.cuda.synchronize()
    R = rt.R_pad
    assert_bf16_close(np_(y_bf)[:R], np_(y_mx)[:R], "bf16 vs mxfp8 operands", rtol=1e-2, atol=1e-3)


def _dbias_case(w, seed=0, experts=None):
    rt = O.route(synth.router_inputs(w, synth._streams(seed, 1)[0])[0], w.expert_begin, w.E)
    cnt = torch.from_numpy(rt.counts.astype(np.int32)).to(DEV)
    off = torch.from_numpy(rt.offsets.astype(np.int32)).to(DEV)
    inp = synth.make_inputs(w, seed)
    rng = np.random.default_rng(seed + 100)
    pre = synth._bf16(rng.standard_normal((w.R_cap, w.N1), dtype=np.float32) * 2.0)
    prm_c = L.glu_params("swiglu", alpha=1.702, up_offset=1.0, gate_lo=-7.0, gate_hi=7.0)
    prm = O.ActParams(O.ACT_SWIGLU, alpha=1.702, up_offset=1.0, gate_lo=-7.0, gate_hi=7.0)
    o = ops.dglu_bwd(inp["dY"].to(DEV), inp["W2"].to(DEV), pre.to(DEV), cnt, off, w.F, prm_c, L.OUT_MXFP8,
                     dbias=True)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    got = np_(o["dbias"])
    dY, W2, pr = np_(inp["dY"]), np_(inp["W2"]), np_(pre)
    for e in (range(w.E) if experts is None else experts):
        r0, n = int(rt.offsets[e]), int(rt.counts[e])
        if n == 0:
            assert np.all(got[e] == 0)
            continue
        da = dY[r0:r0 + n] @ W2[e].T
        u, g = O.unpack_glu_cols(pr[r0:r0 + n])
        du, dg = O.act_bwd(u, g, da, prm)
        d = O.pack_glu_cols(du, dg).astype(np.float32)
        ref = d.astype(np.float64).sum(axis=0)
        lim = 1e-3 * np.abs(d).astype(np.float64).sum(axis=0) + 1e-6
        err = np.abs(got[e] - ref)
        assert np.all(err <= lim), f"expert {e}: {np.sum(err > lim)} columns off, worst {err.max():.3g}"


def test_dbias_gptoss_tail():
    """FC1 bias gradient with the GPT-OSS SwiGLU (gate clamp, alpha, +1) on a
    small batch of the GPT-OSS shape (F 2880: a half-full last N tile)."""
    _dbias_case(synth.scaled(synth.WORKLOADS["gptoss"], T=512))


def test_dbias_edge_counts():
    """Experts of 0, 1, 31, 33, 129 rows (and an empty last one)."""
    w = synth.Workload("edge", 1, 128, 6, 6, 1, 96, "swiglu", "mxfp8", "normal", bias=True, gpt_oss=True)
    counts = [0, 1, 31, 33, 129, 0]
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).astype(np.int32)
    np.random.default_rng(8).shuffle(ids)
    w = synth.scaled(w, T=ids.size)
    rt = O.route(ids.reshape(-1, 1), 0, w.E)
    cnt = torch.from_numpy(rt.counts.astype(np.int32)).to(DEV)
    off = torch.from_numpy(rt.offsets.astype(np.int32)).to(DEV)
    inp = synth.make_inputs(w, 3)
    pre = synth._bf16(np.random.default_rng(9).standard_normal((w.R_cap, w.N1), dtype=np.float32) * 3.0)
    prm_c = L.glu_params("swiglu", alpha=1.702, up_offset=1.0, gate_lo=-7.0, gate_hi=7.0)
    prm = O.ActParams(O.ACT_SWIGLU, alpha=1.702, up_offset=1.0, gate_lo=-7.0, gate_hi=7.0)
    o = ops.dglu_bwd(inp["dY"].to(DEV), inp["W2"].to(DEV), pre.to(DEV), cnt, off, w.F, prm_c, L.OUT_BF16,
                     dbias=True)
    torch.cuda.synchronize()
    R = rt.R_pad
    d = O.dglu_bwd(np_(inp["dY"])[:R], np_(inp["W2"]), np_(pre)[:R], rt, prm)
    ref = O.fc1_bias_grad(d, rt)
    lim = 1e-3 * O.fc1_bias_grad(np.abs(d), rt) + 1e-6
    got = np_(o["dbias"])
    assert np.all(np.abs(got - ref) <= lim)
    assert np.all(got[[0, 5]] == 0)


def test_dbias_gptoss_full_size_sampled_experts():
    """GPT-OSS-shaped backward at full size (T 16384, 32 experts of ~2048
    rows): the bias gradient of four experts, each summed over ~64 blocks."""
    _dbias_case(synth.WORKLOADS["gptoss"], experts=(0, 9, 22, 31))


@pytest.mark.parametrize("E,K,N", [(3, 160, 384), (2, 4096, 2880), (4, 2048, 7168)])
def test_tiled_weight_scales(E, K, N):
    """A weight cast with its scales written in the tensor-core order
    (moe_quantize_mxfp8 col = 2): the same codes as the plain column cast and
    the same scales once un-permuted (K = 160: a partial last k-block; N =
    384 and 2880: an odd number of 128-row groups); the FC2 on that operand
    (MXFP8_TILED, no re-tiling of its scales) gives the same bits as on the
    plain one."""
    rng = np.random.default_rng(E * K + N)
    Wsrc = synth._bf16(rng.standard_normal((E, K, N), dtype=np.float32)
                       * np.exp2(rng.integers(-6, 6, (E, 1, N)))).to(DEV)   # [E][K][N]: cast along K
    st = ops.new_status(DEV)
    q_t, s_t = ops.quantize_mxfp8(Wsrc, col=True, tiled=True, status=st)
    q_p, s_p = ops.quantize_mxfp8(Wsrc, col=True, status=st)
    torch.cuda.synchronize()
    assert ops.read_status(st) == 0
    assert torch.equal(q_t, q_p)
    assert_exact(untile_weight_scales(np_(s_t), E, K, N), np_(s_p), "un-permuted tiled scales")
    counts = [0, 33, 300, 129][:E] + [0] * max(0, E - 4)
    rt, R_cap, cnt, off = _routing(counts, 11)
    Aq, As = synth.random_mxfp8(R_cap, K, 12)
    Aq, As = Aq.to(DEV), As.to(DEV)
    y_t = ops.fc2_fwd(Aq, As, q_t, s_t, cnt, off, status=st, w_tiled=True)
    y_p = ops.fc2_fwd(Aq, As, q_p, s_p, cnt, off, status=st)
    torch.cuda.synchronize()
    assert ops.read_status(st) == 0
    R = rt.R_pad
    assert torch.equal(y_t[:R], y_p[:R]), "FC2 on tiled vs plain weight scales"
