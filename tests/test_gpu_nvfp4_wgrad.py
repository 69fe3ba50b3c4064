"""GPU parity of the NVFP4 weight gradient ([MoE-Fusion] "Fusing MXFP8 and
NVFP4 quantisation": the backward's NVFP4 operands are the transposed tensors
after a random Hadamard rotation, whose amax the dGLU epilogue computes): the
rotated column-wise cast and its amax, the K-grouped kind::mxf4nvf4 GEMM on
oracle-made operands (expert segments whose last MMA covers 32 of its 64
rows), and the chain dGLU (NVFP4 mode) -> rotated casts -> dW1."""
import math

import numpy as np
import pytest
import torch

from grouped_gemm_glu_gb300 import lib as L
from grouped_gemm_glu_gb300 import ops, synth
from oracle import moe_oracle as O
from parity import assert_bf16_close, assert_chain_close, np_

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SIGNS = 0xB3C5


def _routing(counts, seed):
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).astype(np.int32)
    np.random.default_rng(seed).shuffle(ids)
    rt = O.route(ids.reshape(-1, 1), 0, len(counts))
    R_cap = (sum(counts) + 31 * len(counts) + 127) // 128 * 128
    cnt = torch.from_numpy(rt.counts.astype(np.int32)).to(DEV)
    off = torch.from_numpy(rt.offsets.astype(np.int32)).to(DEV)
    return rt, R_cap, cnt, off


def _rot_operand(rt, R_cap, cols, seed):
    """A bf16 activation [R_cap, cols] (pad rows 0) and its rotated NVFP4 cast by the oracle."""
    v = np.random.default_rng(seed).standard_normal((R_cap, cols)).astype(np.float32)
    v[: rt.R_pad][rt.tok_of < 0] = 0
    v[rt.R_pad:] = 0
    vb = O.bf16_round(v)
    sg = O.nvfp4_global_scale(O.rht_transposed_amax(vb[: rt.R_pad], SIGNS))
    q, s = O.nvfp4_rht_cast_cols(vb[: rt.R_pad], SIGNS, sg)
    qf = np.zeros((cols, R_cap // 2), dtype=np.uint8)
    sf = np.zeros((cols, R_cap // 16), dtype=np.uint8)
    qf[:, : rt.R_pad // 2], sf[:, : rt.R_pad // 16] = q, s
    return vb, qf, sf, sg


def _zero_codes_as_one(q):
    lo, hi = q & 0xF, q >> 4
    return (np.where(lo == 8, 0, lo) | (np.where(hi == 8, 0, hi) << 4)).astype(np.uint8)


@pytest.mark.parametrize("M,N", [(256, 384), (96, 160), (2880, 288)])
def test_nvfp4_wgrad_edge_counts(M, N):
    counts = [0, 1, 31, 33, 129, 300, 0]
    rt, R_cap, cnt, off = _routing(counts, 2)
    _, Aq, As, sgA = _rot_operand(rt, R_cap, M, 3)
    _, Bq, Bs, sgB = _rot_operand(rt, R_cap, N, 4)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    st = ops.new_status(DEV)
    D = ops.wgrad_nvfp4(t(Aq), t(As), torch.tensor([float(sgA)], device=DEV), t(Bq), t(Bs),
                        torch.tensor([float(sgB)], device=DEV), cnt, off, out_f32=True, status=st)
    torch.cuda.synchronize()
    assert ops.read_status(st) == 0
    R = rt.R_pad
    ref = O.grouped_wgrad_nvfp4(Aq[:, : R // 2], As[:, : R // 16], sgA, Bq[:, : R // 2], Bs[:, : R // 16], sgB, rt)
    assert_bf16_close(np_(D), ref, f"NVFP4 wgrad M={M} N={N}", rtol=1e-3, atol=1e-3)
    assert np.all(np_(D)[[0, 6]] == 0)


@pytest.mark.parametrize("C", [200, 46, 45])
def test_rotated_cast_and_amax(C):
    """The rotated amax to fp32 rounding, and the rotated NVFP4 codes / scales:
    equal to the oracle's on >= 99.9% (a rotated value the two sides round
    differently in its last bit may cross an E2M1 or E4M3 boundary) and the
    dequantised values within two E2M1 steps everywhere.  C = 200: tiles
    staged through shared memory (a partial column tile, and a partial row
    tile at offsets[E]); C = 46: the direct kernels on column pairs; C = 45:
    one column per thread."""
    counts = [5, 40, 0, 300, 64]
    rt, R_cap, cnt, off = _routing(counts, 5)
    v, q_ref, s_ref, sg_ref = _rot_operand(rt, R_cap, C, 6)
    vd = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).to(DEV)
    st = ops.new_status(DEV)
    am = ops.rht_amax_cols(vd, off, SIGNS, status=st)
    q, s, sg = ops.nvfp4_rht_cast_cols(vd, off, am, SIGNS, status=st)
    torch.cuda.synchronize()
    assert ops.read_status(st) == 0
    R = rt.R_pad
    assert math.isclose(float(am.item()), O.rht_transposed_amax(v[:R], SIGNS), rel_tol=1e-6)
    assert math.isclose(float(sg.item()), float(sg_ref), rel_tol=1e-6)
    qg, sgc = np_(q)[:, : R // 2], np_(s)[:, : R // 16]
    # a rotated value that is exactly zero (blocks of pad rows) comes out as +0 or -0
    # depending on the order of the sums (fp32 butterfly vs float64): E2M1 codes 0x0 and
    # 0x8 both mean 0, so the two zero codes are identified before comparing
    assert (_zero_codes_as_one(qg) == _zero_codes_as_one(q_ref[:, : R // 2])).mean() >= 0.999
    assert (sgc == s_ref[:, : R // 16]).mean() >= 0.999
    dg = O.nvfp4_dequantize(qg, sgc, float(sg.item()))
    dr = O.nvfp4_dequantize(q_ref[:, : R // 2], s_ref[:, : R // 16], sg_ref)
    blk = np.repeat(np.maximum(O.e4m3_decode(sgc), O.e4m3_decode(s_ref[:, : R // 16])), 16, axis=1) / float(sg_ref)
    assert np.all(np.abs(dg - dr) <= 2.0 * blk * (1 + 1e-6))


def test_nvfp4_dw1_chain():
    """dW1 through the NVFP4 backward: the fused dGLU in NVFP4 mode writes bf16
    dFC1 and its rotated amax; x_perm gets its rotated amax; both are cast
    rotated and column-wise to NVFP4 and the K-grouped NVFP4 GEMM forms
    dW1[e] = dFC1^T x.  Against the oracle's chain on the same inputs."""
    w = synth.scaled(synth.WORKLOADS["skew"], T=512, H=512)
    inp = synth.make_inputs(w, 0)
    g = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    r = ops.route_permute(g["x"], g["topk_idx"], g["topk_prob"], w.E, w.R_cap)
    rt = O.route(inp["topk_idx"].numpy(), 0, w.E)
    pre = synth._bf16(np.random.default_rng(100).standard_normal((w.R_cap, w.N1), dtype=np.float32))
    o = ops.dglu_bwd(g["dY"], g["W2"], pre.to(DEV), r["counts"], r["offsets"], w.F, L.glu_params("geglu"),
                     L.OUT_NVFP4, rht_signs=SIGNS)
    aq, asc, sga = ops.nvfp4_rht_cast_cols(o["y"], r["offsets"], o["rht_amax"], SIGNS)
    xam = ops.rht_amax_cols(r["x_perm"], r["offsets"], SIGNS)
    xq, xs, sgx = ops.nvfp4_rht_cast_cols(r["x_perm"], r["offsets"], xam, SIGNS)
    st = ops.new_status(DEV)
    D = ops.wgrad_nvfp4(aq, asc, sga, xq, xs, sgx, r["counts"], r["offsets"], status=st)
    torch.cuda.synchronize()
    assert ops.read_status(st) == 0 and ops.read_status(o["status"]) == 0
    R = rt.R_pad
    d = O.bf16_round(O.dglu_bwd(np_(inp["dY"])[:R], np_(inp["W2"]), np_(pre)[:R], rt, O.ActParams(O.ACT_GEGLU)))
    xp = O.permute(np_(inp["x"]), rt)
    sa = O.nvfp4_global_scale(O.rht_transposed_amax(d, SIGNS))
    sx = O.nvfp4_global_scale(O.rht_transposed_amax(xp, SIGNS))
    qa, sb_a = O.nvfp4_rht_cast_cols(d, SIGNS, sa)
    qx, sb_x = O.nvfp4_rht_cast_cols(xp, SIGNS, sx)
    ref = O.bf16_round(O.grouped_wgrad_nvfp4(qa, sb_a, sa, qx, sb_x, sx, rt))
    # The GEMM and the casts are checked tightly above.  Along the chain both sides
    # round their own dFC1 to bf16; where the two differ by one step, the rotation
    # spreads it over 16 values and an E2M1 code may flip.  One flip moves one
    # product term by up to the 4 <-> 6 step of E2M1, a third of its block's
    # largest magnitude: about 1/sqrt(K) ~ 4% of an output that sums K ~ 500
    # tokens (the hottest expert of this batch).  So: the bf16 rule on 99.9% of
    # the elements and every element within 5% of the output's largest magnitude.
    assert_chain_close(np_(D), ref, "NVFP4 dW1", max_frac=0.05)
