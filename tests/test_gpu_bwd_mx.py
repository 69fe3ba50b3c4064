"""GPU parity of the fused backward GroupGemm + dActivation + Quantize/Transpose
and of the block-scaled MXFP8 grouped GEMMs (FC2 forward, data gradient,
weight gradient) against the oracle, each fed the same synthetic inputs."""
import math
import sys

import numpy as np
import pytest
import torch

from grouped_gemm_glu_gb300 import lib as L
from grouped_gemm_glu_gb300 import ops, synth
from oracle import moe_oracle as O
from parity import assert_bf16_close, assert_mx_close, np_

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _routing(w, seed=0, counts=None):
    if counts is not None:
        ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).astype(np.int32)
        np.random.default_rng(seed).shuffle(ids)
        idx = ids.reshape(-1, 1)
    else:
        idx, _ = synth.router_inputs(w, synth._streams(seed, 1)[0])
    rt = O.route(idx, w.expert_begin, w.E)
    cnt = torch.from_numpy(rt.counts.astype(np.int32)).to(DEV)
    off = torch.from_numpy(rt.offsets.astype(np.int32)).to(DEV)
    return rt, cnt, off


def _act(w):
    if w.gpt_oss:
        return (L.glu_params("swiglu", alpha=1.702, up_offset=1.0, gate_lo=-7.0, gate_hi=7.0),
                O.ActParams(O.ACT_SWIGLU, alpha=1.702, up_offset=1.0, gate_lo=-7.0, gate_hi=7.0))
    m = {"swiglu": O.ACT_SWIGLU, "geglu": O.ACT_GEGLU, "srelu": O.ACT_SRELU}
    return L.glu_params(w.act), O.ActParams(m[w.act])


def _dglu_case(w, rows=None, counts=None, seed=0, out_mode=L.OUT_MXFP8):
    rt, cnt, off = _routing(w, seed, counts)
    inp = synth.make_inputs(w, seed)
    rng = np.random.default_rng(seed + 100)
    pre = synth._bf16(rng.standard_normal((w.R_cap, w.N1), dtype=np.float32) * 2.0)
    gp, op = _act(w)
    o = ops.dglu_bwd(inp["dY"].to(DEV), inp["W2"].to(DEV), pre.to(DEV), cnt, off, w.F, gp, out_mode)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    dY, W2, pr = inp["dY"], inp["W2"], np_(pre)
    w2_cache = {}
    blocks = rows if rows is not None else list(range(0, rt.R_pad, 32))
    acc = {k: [] for k in ("qg", "sg", "qr", "sr", "v", "qcg", "scg", "qcr", "scr", "vc")}
    for r0 in blocks:
        rr = np.arange(r0, r0 + 32)
        e = int(rt.expert_of_row[r0])
        real = rt.tok_of[rr] >= 0
        if e not in w2_cache:
            w2_cache = {e: np_(W2[e])}
        da = np_(dY[r0:r0 + 32]) @ w2_cache[e].T
        if w.gated:
            u, g = O.unpack_glu_cols(pr[rr])
            du, dg = O.act_bwd(u, g, da, op)
            d = O.pack_glu_cols(du, dg)
        else:
            d, _ = O.act_bwd(pr[rr], None, da, op)
        d[~real] = 0
        d = d.astype(np.float32)
        if out_mode == L.OUT_BF16:
            assert_bf16_close(np_(o["y"][r0:r0 + 32]), O.bf16_round(d), f"dFC1 rows {r0}")
            continue
        q, s = O.mx_quantize_rows(d)
        qc, sc = O.mx_quantize_cols(d)
        acc["qg"].append(np_(o["q_row"][r0:r0 + 32]))
        acc["sg"].append(np_(o["s_row"][r0:r0 + 32]))
        acc["qr"].append(q)
        acc["sr"].append(s)
        acc["v"].append(d)
        acc["qcg"].append(np_(o["q_col"][:, r0:r0 + 32]))
        acc["scg"].append(np_(o["s_col"][:, r0 // 32:r0 // 32 + 1]))
        acc["qcr"].append(qc)
        acc["scr"].append(sc)
        acc["vc"].append(d.T)
    if out_mode == L.OUT_MXFP8:
        cat = {k: np.concatenate(v) for k, v in acc.items()}
        assert_mx_close(cat["qg"], cat["sg"], cat["qr"], cat["sr"], cat["v"], f"{w.name} dFC1 row-wise")
        assert_mx_close(cat["qcg"], cat["scg"], cat["qcr"], cat["scr"], cat["vc"], f"{w.name} dFC1 col-wise")


@pytest.mark.parametrize("out_mode", [L.OUT_MXFP8, L.OUT_BF16])
def test_dglu_tiny_full(out_mode):
    _dglu_case(synth.WORKLOADS["tiny"], out_mode=out_mode)


def test_dglu_swiglu_alpha_offset_unclamped(monkeypatch):
    """dSwiGLU with alpha = 1.702 and (up + 1) but no clamp: the epilogue's
    short derivative form with non-default alpha and offset."""
    monkeypatch.setattr(sys.modules[__name__], "_act", lambda w: (
        L.glu_params("swiglu", alpha=1.702, up_offset=1.0), O.ActParams(O.ACT_SWIGLU, alpha=1.702, up_offset=1.0)))
    _dglu_case(synth.WORKLOADS["tiny"], out_mode=L.OUT_MXFP8)


@pytest.mark.parametrize("name", ["tiny", "skew_srelu"])
def test_dglu_nvfp4_rotated_amax(name):
    """NVFP4 backward ([MoE-Fusion] "Fusing MXFP8 and NVFP4 quantisation"):
    the epilogue writes dFC1 in bf16, max |dFC1| and the amax of dFC1's
    transposed random Hadamard rotation.  The rotated amax is checked on the
    kernel's own bf16 output (the transform alone, fp32 sums) and against the
    oracle's dFC1 (the whole path)."""
    w = synth.WORKLOADS[name]
    if name != "tiny":
        w = synth.scaled(w, T=512, H=512)
    rt, cnt, off = _routing(w, 0, None)
    inp = synth.make_inputs(w, 0)
    rng = np.random.default_rng(100)
    pre = synth._bf16(rng.standard_normal((w.R_cap, w.N1), dtype=np.float32) * 2.0)
    gp, op = _act(w)
    mask = 0xB3C5
    o = ops.dglu_bwd(inp["dY"].to(DEV), inp["W2"].to(DEV), pre.to(DEV), cnt, off, w.F, gp, L.OUT_NVFP4,
                     rht_signs=mask)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    R = rt.R_pad
    y = np_(o["y"])[:R].astype(np.float64)
    got = float(o["rht_amax"].item())
    assert math.isclose(got, O.rht_transposed_amax(y, mask), rel_tol=1e-5)
    d = O.dglu_bwd(np_(inp["dY"])[:R], np_(inp["W2"]), np_(pre)[:R], rt, op)
    assert math.isclose(got, O.rht_transposed_amax(d, mask), rel_tol=2e-2)
    assert math.isclose(float(o["amax"].item()), float(np.max(np.abs(d))), rel_tol=2e-2)
    # a different sign draw gives a different rotation (the signs reach the kernel)
    o2 = ops.dglu_bwd(inp["dY"].to(DEV), inp["W2"].to(DEV), pre.to(DEV), cnt, off, w.F, gp, L.OUT_NVFP4,
                      rht_signs=0x0001)
    torch.cuda.synchronize()
    assert math.isclose(float(o2["rht_amax"].item()), O.rht_transposed_amax(y, 0x0001), rel_tol=1e-5)


def test_dglu_single_cta_kernel():
    """The single-CTA variant of the bf16 GEMM (CTA pairs switched off)."""
    lib = L.load()
    lib.moe_set_cta_pairs(0)
    try:
        _dglu_case(synth.WORKLOADS["tiny"], out_mode=L.OUT_MXFP8)
    finally:
        lib.moe_set_cta_pairs(1)


def test_dglu_edge_counts():
    counts = [0, 1, 31, 32, 33, 127, 128, 129, 255, 256, 257, 0]
    w = synth.Workload("edge", sum(counts), 128, len(counts), len(counts), 1, 96, "swiglu", "mxfp8", "normal")
    _dglu_case(w, counts=counts)


def test_dglu_gptoss_tail():
    w = synth.scaled(synth.WORKLOADS["gptoss"], T=512)
    _dglu_case(w)


def test_dglu_geglu_tiny():
    """GeGLU (exact erf): the epilogue's short GeGLU derivative."""
    _dglu_case(synth.scaled(synth.WORKLOADS["tiny"], act="geglu"), out_mode=L.OUT_MXFP8)


def test_dglu_srelu():
    w = synth.scaled(synth.WORKLOADS["skew_srelu"], T=512, H=512)
    _dglu_case(w)


def _sampled_blocks(rt, n_random, seed):
    """Every expert's first and last 32-row block plus n_random blocks drawn
    uniformly over the padded rows (interior blocks of the long segments)."""
    blocks = {int(rt.offsets[e]) for e in range(rt.E) if rt.counts[e]} | \
             {int(rt.offsets[e + 1]) - 32 for e in range(rt.E) if rt.counts[e]}
    if rt.R_pad:
        blocks |= {int(b) * 32 for b in np.random.default_rng(seed).integers(0, rt.R_pad // 32, n_random)}
    return sorted(blocks)


def test_dglu_dsv3_full_size_sampled():
    """DeepSeek-V3 shard backward at full size: every expert's first and last
    block and 16 random interior blocks."""
    w = synth.WORKLOADS["dsv3"]
    rt, _, _ = _routing(w)
    _dglu_case(w, rows=_sampled_blocks(rt, 16, 21))


@pytest.mark.parametrize("name", ["skew", "skew_srelu"])
def test_dglu_skew_full_size_sampled(name):
    """Skewed 64-expert config at full size (T 32768, H 4096, F 1536, top-6,
    Zipf routing: one expert holds ~97% of the tokens, 8 hold none): GeGLU
    (gated, N1 = 2F) and sReLU (not gated, N1 = F) derivatives, MXFP8 row
    and column outputs, on sampled blocks."""
    w = synth.WORKLOADS[name]
    rt, _, _ = _routing(w)
    _dglu_case(w, rows=_sampled_blocks(rt, 12, 22))


def test_dglu_gptoss_full_size_sampled():
    """GPT-OSS-shaped backward at full size (clamped SwiGLU derivative, F 2880
    with a half-full last N tile); every expert's first and last 32-row block
    and random interior blocks."""
    w = synth.WORKLOADS["gptoss"]
    rt, _, _ = _routing(w)
    _dglu_case(w, rows=_sampled_blocks(rt, 8, 23))


def _fc2_case(E, K, N, counts, seed, experts=None, n_cols=None):
    """Block-scaled grouped GEMM on random MXFP8 operands; the oracle
    dequantises (exact) and multiplies in float64.  experts / n_cols limit
    the comparison to some experts and a random subset of columns."""
    w = synth.Workload("fc2", sum(counts), 64, E, E, 1, 64, "swiglu", "mxfp8", "normal")
    rt, cnt, off = _routing(w, seed, counts)
    R_cap = w.R_cap
    Aq, As = synth.random_mxfp8(R_cap, K, seed + 1)
    Wq, Ws = synth.random_mxfp8(E * N, K, seed + 2)
    Wq, Ws = Wq.view(E, N, K), Ws.view(E, N, K // 32)
    y = ops.fc2_fwd(Aq.to(DEV), As.to(DEV), Wq.to(DEV), Ws.to(DEV), cnt, off)
    torch.cuda.synchronize()
    yg = np_(y)
    cols = np.arange(N) if n_cols is None else np.sort(np.random.default_rng(seed).choice(N, n_cols, replace=False))
    for e in (range(E) if experts is None else experts):
        r0, n, r1 = int(rt.offsets[e]), int(rt.counts[e]), int(rt.offsets[e + 1])
        A = O.mx_dequantize(Aq[r0:r0 + n].numpy(), As[r0:r0 + n].numpy())
        W = O.mx_dequantize(Wq[e][cols].numpy(), Ws[e][cols].numpy())
        assert_bf16_close(yg[r0:r0 + n][:, cols], O.bf16_round(A @ W.T), f"fc2 expert {e}")
        assert np.all(yg[r0 + n:r1] == 0), "pad rows must be zero"


def test_fc2_block_scaled_edge_counts():
    _fc2_case(6, 256, 256, [0, 1, 33, 128, 129, 300], 1)


def test_fc2_dsv3_shape():
    # FC2 of the DeepSeek-V3 shard: K = F = 2048, N = H = 7168, ~256 rows per expert
    _fc2_case(32, 2048, 7168, list(np.random.default_rng(2).integers(200, 320, 32)), 2,
              experts=(0, 13, 31), n_cols=512)


def test_dx_shape():
    # data gradient dX = dFC1 . W1p: K = 2F = 4096
    _fc2_case(4, 4096, 1024, [100, 0, 257, 64], 3)


@pytest.mark.parametrize("out_f32", [True, False])
def test_wgrad_edge_counts(out_f32):
    counts = [0, 1, 31, 32, 33, 127, 128, 129, 200, 0]
    E, M, N = len(counts), 256, 384
    w = synth.Workload("wg", sum(counts), 64, E, E, 1, 64, "swiglu", "mxfp8", "normal")
    rt, cnt, off = _routing(w, 4, counts)
    R_cap = w.R_cap
    Aq, As = synth.random_mxfp8(M, R_cap, 5)
    Bq, Bs = synth.random_mxfp8(N, R_cap, 6)
    D = ops.wgrad(Aq.to(DEV), As.to(DEV), Bq.to(DEV), Bs.to(DEV), cnt, off, out_f32=out_f32)
    torch.cuda.synchronize()
    ref = O.grouped_wgrad(O.mx_dequantize(Aq.numpy(), As.numpy()), O.mx_dequantize(Bq.numpy(), Bs.numpy()), rt)
    got = np_(D)
    assert_bf16_close(got, ref if out_f32 else O.bf16_round(ref), "wgrad")
    for e, c in enumerate(counts):
        if c == 0:
            assert np.all(got[e] == 0)


@pytest.mark.parametrize("K,N", [(2880, 2880), (5760, 2880), (96, 160)])
def test_fc2_partial_k_block_and_column_tile(K, N):
    """K and N multiples of 32 but not of 128 / 256 (the GPT-OSS FC2 K = N =
    2880, its dX K = 5760, N = 2880, and a small odd case): the last k-block
    and the last column tile are partial."""
    counts = [3, 40, 0, 129] if K > 200 else [1, 33, 0, 70, 5]
    _fc2_case(len(counts), K, N, counts, seed=7, n_cols=min(N, 200))


@pytest.mark.parametrize("M,N", [(2880, 2880), (5760, 2880), (96, 160)])
def test_wgrad_partial_row_and_column_tiles(M, N):
    """M and N multiples of 32 but not of 128 / 256 (GPT-OSS dW2 and dW1
    shapes): the last row tile and column tile of every expert are partial."""
    counts = [0, 1, 31, 33, 129, 0]
    E = len(counts)
    w = synth.Workload("wg", sum(counts), 64, E, E, 1, 64, "swiglu", "mxfp8", "normal")
    rt, cnt, off = _routing(w, 9, counts)
    R_cap = w.R_cap
    Aq, As = synth.random_mxfp8(M, R_cap, 10)
    Bq, Bs = synth.random_mxfp8(N, R_cap, 11)
    D = ops.wgrad(Aq.to(DEV), As.to(DEV), Bq.to(DEV), Bs.to(DEV), cnt, off, out_f32=False)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(12).choice(M, min(M, 96), replace=False))
    ref = O.grouped_wgrad(O.mx_dequantize(Aq.numpy()[rows], As.numpy()[rows]),
                          O.mx_dequantize(Bq.numpy(), Bs.numpy()), rt)
    got = np_(D)
    assert_bf16_close(got[:, rows], O.bf16_round(ref), "wgrad")
    assert np.all(got[[0, 5]] == 0)


def test_wgrad_dsv3_dw2_shape_sampled_experts():
    # dW2 of the DeepSeek-V3 shard: [E, F=2048, H=7168], K = rows of each expert
    w = synth.WORKLOADS["dsv3"]
    rt, cnt, off = _routing(w)
    F, H = 2048, 7168
    Aq, As = synth.random_mxfp8(F, w.R_cap, 7)
    Bq, Bs = synth.random_mxfp8(H, w.R_cap, 8)
    D = ops.wgrad(Aq.to(DEV), As.to(DEV), Bq.to(DEV), Bs.to(DEV), cnt, off, out_f32=False)
    torch.cuda.synchronize()
    Aq, As, Bq, Bs = Aq.numpy(), As.numpy(), Bq.numpy(), Bs.numpy()
    for e in (0, 7, 31):
        r0, r1 = int(rt.offsets[e]), int(rt.offsets[e + 1])
        sl = np.random.default_rng(e).choice(F, 64, replace=False)
        A = O.mx_dequantize(Aq[sl][:, r0:r1], As[sl][:, r0 // 32:r1 // 32])
        B = O.mx_dequantize(Bq[:, r0:r1], Bs[:, r0 // 32:r1 // 32])
        ref = A @ B.T
        assert_bf16_close(np_(D[e])[sl], O.bf16_round(ref), f"dW2 expert {e}")
