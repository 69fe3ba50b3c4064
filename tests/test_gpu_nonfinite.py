"""Non-finite inputs through the fused epilogues (MXFP8 rule: a block holding
a NaN or an infinity gets the NaN scale byte 0xFF and every one of its codes
is the E4M3 NaN 0x7F), and the NVFP4 forward's per-tensor amax against the
oracle on a case small enough to evaluate in full."""
import math

import numpy as np
import pytest
import torch

from grouped_gemm_glu_gb300 import lib as L
from grouped_gemm_glu_gb300 import ops, synth
from oracle import moe_oracle as O
from parity import assert_bf16_close, assert_mx_close, np_

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _assert_nan_blocks(q_gpu, s_gpu, s_ref, what):
    """Blocks the oracle marks non-finite: scale 0xFF and all 32 codes 0x7F on
    the GPU too (the value comparison of assert_mx_close skips them)."""
    q, s, sr = np.asarray(q_gpu), np.asarray(s_gpu), np.asarray(s_ref)
    bad = sr == 255
    assert bad.any(), f"{what}: the case has no non-finite block"
    assert np.all(s[bad] == 255), f"{what}: {np.sum(s[bad] != 255)} non-finite blocks without the NaN scale"
    qb = q.reshape(*s.shape, 32)
    assert np.all(qb[bad] == 0x7F), f"{what}: codes of non-finite blocks are not all 0x7F"


def test_fc1_nan_inf_tokens():
    """Tiny forward with one token's x holding a NaN and another's a +Inf:
    every row those tokens were routed to is non-finite after the GEMM, so its
    row-wise blocks and the column-wise blocks that contain it are NaN blocks;
    everything else matches the oracle as usual."""
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w, 0)
    x = inp["x"].clone()
    x[7, 3] = float("nan")
    x[100, 17] = float("inf")
    rt = O.route(inp["topk_idx"].numpy(), 0, w.E)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    r = ops.route_permute(x.to(DEV), g["topk_idx"], g["topk_prob"], w.E, w.R_cap)
    W1p = ops.repack_fc1(g["W1"])
    o = ops.fc1_fwd(r["x_perm"], W1p, r["counts"], r["offsets"], w.F, L.glu_params("swiglu"), L.OUT_MXFP8)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    with np.errstate(all="ignore"):
        fo = O.fc1_glu_fwd(O.permute(np_(x), rt), O.repack_fc1(np_(inp["W1"])), None, rt,
                           O.ActParams(O.ACT_SWIGLU))
        q, s = O.mx_quantize_rows(fo.y)
        qc, sc = O.mx_quantize_cols(fo.y)
    R = rt.R_pad
    assert_bf16_close(np_(o["pre"])[:R], fo.pre_bf16, "pre")
    assert_mx_close(np_(o["q_row"])[:R], np_(o["s_row"])[:R], q, s, fo.y, "row-wise")
    assert_mx_close(np_(o["q_col"])[:, :R], np_(o["s_col"])[:, :R // 32], qc, sc, fo.y.T, "col-wise")
    _assert_nan_blocks(np_(o["q_row"])[:R], np_(o["s_row"])[:R], s, "row-wise")
    _assert_nan_blocks(np_(o["q_col"])[:, :R], np_(o["s_col"])[:, :R // 32], sc, "col-wise")
    # the non-finite rows are exactly the rows of tokens 7 and 100
    rows = {int(v) for v in rt.row_of.reshape(w.T, w.k)[[7, 100]].ravel() if v >= 0}
    bad_rows = set(np.nonzero((np_(o["s_row"])[:R] == 255).any(axis=1))[0].tolist())
    assert bad_rows == rows


def test_dglu_nan_inf_rows():
    """Tiny backward with a NaN in one permuted row of dY and a +Inf in another:
    the dFC1 blocks of those rows (row-wise) and the column blocks containing
    them are NaN blocks; everything else matches the oracle."""
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w, 0)
    rt = O.route(inp["topk_idx"].numpy(), 0, w.E)
    cnt = torch.from_numpy(rt.counts.astype(np.int32)).to(DEV)
    off = torch.from_numpy(rt.offsets.astype(np.int32)).to(DEV)
    dY = inp["dY"].clone()
    r_nan, r_inf = int(rt.row_of[5]), int(rt.row_of[301])
    dY[r_nan, 11] = float("nan")
    dY[r_inf, 200] = float("inf")
    rng = np.random.default_rng(100)
    pre = synth._bf16(rng.standard_normal((w.R_cap, w.N1), dtype=np.float32) * 2.0)
    o = ops.dglu_bwd(dY.to(DEV), inp["W2"].to(DEV), pre.to(DEV), cnt, off, w.F, L.glu_params("swiglu"),
                     L.OUT_MXFP8)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    R = rt.R_pad
    with np.errstate(all="ignore"):
        d = O.dglu_bwd(np_(dY)[:R], np_(inp["W2"]), np_(pre)[:R], rt, O.ActParams(O.ACT_SWIGLU))
        q, s = O.mx_quantize_rows(d)
        qc, sc = O.mx_quantize_cols(d)
    assert_mx_close(np_(o["q_row"])[:R], np_(o["s_row"])[:R], q, s, d, "dFC1 row-wise")
    assert_mx_close(np_(o["q_col"])[:, :R], np_(o["s_col"])[:, :R // 32], qc, sc, d.T, "dFC1 col-wise")
    _assert_nan_blocks(np_(o["q_row"])[:R], np_(o["s_row"])[:R], s, "dFC1 row-wise")
    _assert_nan_blocks(np_(o["q_col"])[:, :R], np_(o["s_col"])[:, :R // 32], sc, "dFC1 col-wise")
    bad_rows = set(np.nonzero((np_(o["s_row"])[:R] == 255).any(axis=1))[0].tolist())
    assert bad_rows == {r_nan, r_inf}


@pytest.mark.parametrize("act", ["geglu", "srelu"])
def test_fc1_nvfp4_amax_tiny_full(act):
    """NVFP4 forward mode on the tiny config in full: bf16 y against the
    oracle's activation and the per-tensor amax against the oracle's
    Fc1Out.amax (max |y| over every real row, float32)."""
    w = synth.scaled(synth.WORKLOADS["tiny"], act=act)
    inp = synth.make_inputs(w, 0)
    rt = O.route(inp["topk_idx"].numpy(), 0, w.E)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    r = ops.route_permute(g["x"], g["topk_idx"], g["topk_prob"], w.E, w.R_cap)
    W1p = ops.repack_fc1(g["W1"]) if w.gated else g["W1"]
    o = ops.fc1_fwd(r["x_perm"], W1p, r["counts"], r["offsets"], w.F, L.glu_params(act), L.OUT_NVFP4)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    W1 = np_(inp["W1"])
    op = O.ActParams({"geglu": O.ACT_GEGLU, "srelu": O.ACT_SRELU}[act])
    fo = O.fc1_glu_fwd(O.permute(np_(inp["x"]), rt), O.repack_fc1(W1) if w.gated else W1, None, rt, op)
    R = rt.R_pad
    assert_bf16_close(np_(o["y"])[:R], O.bf16_round(fo.y), "y")
    assert fo.amax > 0
    assert math.isclose(float(o["amax"].item()), fo.amax, rel_tol=1e-3)
