"""GPU parity of the MXFP8-input FC1 (GroupGemm + Activation +
Quantize/Transpose on the block-scaled product of the row-wise MXFP8 x_perm
and packed W1): the oracle quantises the same bf16 inputs itself, multiplies
the dequantised operands in float64 and applies the same activation and
output quantisation."""
import numpy as np
import pytest
import torch

import test_gpu_fc1 as F
from grouped_gemm_glu_gb300 import lib as L
from grouped_gemm_glu_gb300 import ops, synth
from oracle import moe_oracle as O
from parity import assert_bf16_close, assert_exact, assert_mx_close, np_

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run(case, out_mode, row_scale=None):
    w = case.w
    gp, _ = F.act_params(w)
    xq, xs = ops.quantize_mxfp8(case.r["x_perm"], col=False, counts=case.r["counts"], offsets=case.r["offsets"])
    W1q, W1s = ops.quantize_mxfp8(case.W1p, col=False)
    o = ops.fc1_fwd_mxfp8(xq, xs, W1q, W1s, case.r["counts"], case.r["offsets"], w.F, gp, out_mode,
                          b1p=case.b1p, row_scale=row_scale)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    return o


def _oracle_operands(case):
    """The oracle's own MXFP8 rounding of x_perm and W1p, dequantised."""
    rt = case.rt
    xp = O.permute(np_(case.inp["x"]), rt)
    xd = O.mx_dequantize(*O.mx_quantize_rows(xp))
    Wd = O.mx_dequantize(*O.mx_quantize_rows(case.W1p_np))
    return xd, Wd


@pytest.mark.parametrize("name,out_mode", [("tiny", L.OUT_MXFP8), ("tiny", L.OUT_BF16), ("geglu", L.OUT_NVFP4),
                                           ("srelu", L.OUT_MXFP8)])
def test_fc1_mxfp8_tiny_full(name, out_mode):
    w = synth.WORKLOADS["tiny"] if name == "tiny" else synth.scaled(synth.WORKLOADS["tiny"], act=name)
    case = F.Case(w)
    o = _run(case, out_mode)
    _, op = F.act_params(w)
    xd, Wd = _oracle_operands(case)
    rt = case.rt
    fo = O.fc1_glu_fwd(xd, Wd, None, rt, op)
    R = rt.R_pad
    assert_bf16_close(np_(o["pre"])[:R], fo.pre_bf16, "pre")
    if out_mode == L.OUT_MXFP8:
        q, s = O.mx_quantize_rows(fo.y)
        assert_mx_close(np_(o["q_row"])[:R], np_(o["s_row"])[:R], q, s, fo.y, "row-wise")
        qc, sc = O.mx_quantize_cols(fo.y)
        assert_mx_close(np_(o["q_col"])[:, :R], np_(o["s_col"])[:, :R // 32], qc, sc, fo.y.T, "col-wise")
    else:
        assert_bf16_close(np_(o["y"])[:R], O.bf16_round(fo.y), "y")
        if out_mode == L.OUT_NVFP4:
            assert abs(float(o["amax"].item()) - fo.amax) <= 1e-3 * fo.amax


def test_fc1_mxfp8_edge_counts_gptoss_bias_rowscale():
    """Experts of 0 .. 257 rows, the GPT-OSS activation with bias, a row scale."""
    counts = [0, 1, 31, 32, 33, 127, 128, 129, 255, 256, 257, 0]
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).astype(np.int32)
    np.random.default_rng(3).shuffle(ids)
    w = synth.Workload("edge", ids.size, 128, len(counts), len(counts), 1, 96, "swiglu", "mxfp8", "normal",
                       bias=True, gpt_oss=True)
    case = F.Case(w, idx=ids.reshape(-1, 1))
    rs = torch.rand(w.R_cap, generator=torch.Generator().manual_seed(5)) + 0.5
    o = _run(case, L.OUT_MXFP8, row_scale=rs.to(DEV))
    _, op = F.act_params(w)
    xd, Wd = _oracle_operands(case)
    rt = case.rt
    fo = O.fc1_glu_fwd(xd, Wd, case.b1p_np, rt, op, row_scale=np_(rs)[: rt.R_pad])
    R = rt.R_pad
    assert_bf16_close(np_(o["pre"])[:R], fo.pre_bf16, "pre")
    q, s = O.mx_quantize_rows(fo.y)
    assert_mx_close(np_(o["q_row"])[:R], np_(o["s_row"])[:R], q, s, fo.y, "row-wise")
    qc, sc = O.mx_quantize_cols(fo.y)
    assert_mx_close(np_(o["q_col"])[:, :R], np_(o["s_col"])[:, :R // 32], qc, sc, fo.y.T, "col-wise")


def test_fc1_mxfp8_dsv3_full_size_sampled():
    """DeepSeek-V3 shard at full size (K = H = 7168, N1 = 4096): sampled
    32-row blocks (every expert's first and last plus random ones)."""
    case = F.Case(synth.WORKLOADS["dsv3"])
    o = _run(case, L.OUT_MXFP8)
    _, op = F.act_params(case.w)
    rt = case.rt
    x = np_(case.inp["x"])
    Wd = {}
    acc = {k: [] for k in ("qg", "sg", "qr", "sr", "v")}
    for r0 in F.sample_blocks(rt, 16, 2):
        rows = np.arange(r0, r0 + 32)
        e = int(rt.expert_of_row[r0])
        if e not in Wd:
            Wd = {e: O.mx_dequantize(*O.mx_quantize_rows(case.W1p_np[e]))}
        real = rt.tok_of[rows] >= 0
        xb = np.zeros((32, x.shape[1]))
        xb[real] = x[rt.tok_of[rows][real]]
        pre = O.mx_dequantize(*O.mx_quantize_rows(xb)) @ Wd[e].T
        pre[~real] = 0
        u, g = O.unpack_glu_cols(pre)
        y = O.act_fwd(u, g, op)
        y[~real] = 0
        y = y.astype(np.float32)
        assert_bf16_close(np_(o["pre"][r0:r0 + 32]), O.bf16_round(pre), f"pre rows {r0}")
        q, s = O.mx_quantize_rows(y)
        acc["qg"].append(np_(o["q_row"][r0:r0 + 32]))
        acc["sg"].append(np_(o["s_row"][r0:r0 + 32]))
        acc["qr"].append(q)
        acc["sr"].append(s)
        acc["v"].append(y)
    cat = {k: np.concatenate(v) for k, v in acc.items()}
    assert_mx_close(cat["qg"], cat["sg"], cat["qr"], cat["sr"], cat["v"], "dsv3 mxfp8 FC1 row-wise")


@pytest.mark.parametrize("G,R,C", [(3, 96, 160), (2, 256, 256), (1, 4096, 448)])
def test_weight_dual_cast_bit_exact(G, R, C):
    """Both MXFP8 copies of a weight from one read (row-wise along C for the
    MXFP8-input FC1, column-wise along R for the data gradient): bit-exact
    against the oracle's two casts, with partial tiles (R 96, C 160), a NaN
    and an Inf (scale 0xFF, codes 0x7F for their blocks) and exponents spread
    over 2^-8 .. 2^8 per column."""
    rng = np.random.default_rng(G * R + C)
    Wf = rng.standard_normal((G, R, C), dtype=np.float32) * np.exp2(rng.integers(-8, 8, (G, 1, C)))
    Wf[0, 5, 7] = np.nan
    Wf[G - 1, R - 1, C - 1] = np.inf
    W = synth._bf16(Wf)
    st = ops.new_status(DEV)
    qr, sr, qc, sc = ops.quantize_mxfp8_dual(W.to(DEV), status=st)
    torch.cuda.synchronize()
    assert ops.read_status(st) == 0
    Wn = np_(W)
    for g in range(G):
        q_ref, s_ref = O.mx_quantize_rows(Wn[g])
        assert_exact(np_(qr[g]), q_ref, f"row codes {g}")
        assert_exact(np_(sr[g]), s_ref, f"row scales {g}")
        q_ref, s_ref = O.mx_quantize_cols(Wn[g])
        assert_exact(np_(qc[g]), q_ref, f"column codes {g}")
        assert_exact(np_(sc[g]), s_ref, f"column scales {g}")
