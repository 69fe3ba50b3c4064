"""GPU parity of the fused forward GroupGemm + Activation + Quantize/Transpose
(and of the standalone quantize / NVFP4 / activation kernels) against the
oracle.  Small workloads are compared in full; the full-size ones on sampled
32-row blocks (every expert's first and last block plus random ones), which
the oracle evaluates one by one."""
import math

import sys

import numpy as np
import pytest
import torch

from grouped_gemm_glu_gb300 import lib as L
from grouped_gemm_glu_gb300 import ops, synth
from oracle import moe_oracle as O
from parity import assert_bf16_close, assert_exact, assert_mx_close, np_

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

ORACLE_ACT = {"swiglu": O.ACT_SWIGLU, "geglu": O.ACT_GEGLU, "srelu": O.ACT_SRELU}


def act_params(w):
    if w.gpt_oss:
        return (L.glu_params("swiglu", alpha=1.702, up_offset=1.0, gate_lo=-7.0, gate_hi=7.0),
                O.ActParams(O.ACT_SWIGLU, alpha=1.702, up_offset=1.0, gate_lo=-7.0, gate_hi=7.0))
    return L.glu_params(w.act), O.ActParams(ORACLE_ACT[w.act])


class Case:
    """Inputs on both sides plus the GPU routing / repack results."""

    def __init__(self, w, seed=0, idx=None):
        self.w = w
        self.inp = synth.make_inputs(w, seed)
        if idx is not None:
            self.inp["topk_idx"] = torch.from_numpy(idx)
            self.inp["topk_prob"] = torch.rand(idx.shape, generator=torch.Generator().manual_seed(seed))
        self.rt = O.route(self.inp["topk_idx"].numpy(), w.expert_begin, w.E)
        g = {k: (v.to(DEV) if v is not None else None) for k, v in self.inp.items()}
        self.g = g
        self.r = ops.route_permute(g["x"], g["topk_idx"], g["topk_prob"], w.E, w.R_cap, w.expert_begin)
        self.W1p = ops.repack_fc1(g["W1"]) if w.gated else g["W1"]
        self.b1p = None
        if g["b1"] is not None:
            self.b1p = (ops.repack_fc1(g["b1"].unsqueeze(-1)).squeeze(-1) if w.gated else g["b1"])
        self.W1_np = np_(self.inp["W1"])
        self.W1p_np = O.repack_fc1(self.W1_np) if w.gated else self.W1_np
        b = self.inp["b1"]
        self.b1p_np = None if b is None else (O.repack_fc1(np_(b)[..., None])[..., 0] if w.gated else np_(b))

    def oracle_rows(self, rows, prm):
        """Oracle pre-activation (bf16) and activation (float32) of the given
        permuted rows (all of one 32-row block)."""
        rt = self.rt
        e = int(rt.expert_of_row[rows[0]])
        x = np_(self.inp["x"])
        real = rt.tok_of[rows] >= 0
        xb = np.zeros((len(rows), x.shape[1]))
        xb[real] = x[rt.tok_of[rows][real]]
        pre = xb @ self.W1p_np[e].T
        if self.b1p_np is not None:
            pre[real] += self.b1p_np[e]
        pre[~real] = 0
        if self.w.gated:
            u, g = O.unpack_glu_cols(pre)
            y = O.act_fwd(u, g, prm)
        else:
            y = O.act_fwd(pre, None, prm)
        y[~real] = 0
        return O.bf16_round(pre), y.astype(np.float32)


def run_fc1(case, out_mode, save_pre=True):
    w = case.w
    gp, _ = act_params(w)
    return ops.fc1_fwd(case.r["x_perm"], case.W1p, case.r["counts"], case.r["offsets"], w.F, gp, out_mode,
                       b1p=case.b1p, save_pre=save_pre)


def sample_blocks(rt, n_random, seed):
    blocks = set()
    for e in range(rt.E):
        if rt.counts[e]:
            blocks.add(int(rt.offsets[e]))
            blocks.add(int(rt.offsets[e + 1]) - 32)
    rng = np.random.default_rng(seed)
    if rt.R_pad:
        blocks.update(int(b) * 32 for b in rng.integers(0, rt.R_pad // 32, n_random))
    return sorted(blocks)


def check_blocks(case, o, blocks, out_mode):
    """Compares the sampled 32-row blocks; the MXFP8 rule is applied to all
    sampled elements together."""
    w = case.w
    _, op = act_params(w)
    pre_g = np_(o["pre"]) if "pre" in o else None
    acc = {k: [] for k in ("qg", "sg", "qr", "sr", "v", "qcg", "scg", "qcr", "scr", "vc")}
    for r0 in blocks:
        rows = np.arange(r0, r0 + 32)
        pre_ref, y_ref = case.oracle_rows(rows, op)
        tag = f"{w.name} rows {r0}"
        if pre_g is not None:
            assert_bf16_close(pre_g[rows], pre_ref, tag + " pre")
        if out_mode == L.OUT_MXFP8:
            q_ref, s_ref = O.mx_quantize_rows(y_ref)
            acc["qg"].append(np_(o["q_row"][r0:r0 + 32]))
            acc["sg"].append(np_(o["s_row"][r0:r0 + 32]))
            acc["qr"].append(q_ref)
            acc["sr"].append(s_ref)
            acc["v"].append(y_ref)
            qc_ref, sc_ref = O.mx_quantize_cols(y_ref)
            acc["qcg"].append(np_(o["q_col"][:, r0:r0 + 32]))
            acc["scg"].append(np_(o["s_col"][:, r0 // 32:r0 // 32 + 1]))
            acc["qcr"].append(qc_ref)
            acc["scr"].append(sc_ref)
            acc["vc"].append(y_ref.T)
        else:
            assert_bf16_close(np_(o["y"][r0:r0 + 32]), O.bf16_round(y_ref), tag + " y")
    if out_mode == L.OUT_MXFP8:
        cat = {k: np.concatenate(v, axis=0) for k, v in acc.items() if v}
        assert_mx_close(cat["qg"], cat["sg"], cat["qr"], cat["sr"], cat["v"], f"{w.name} row-wise")
        assert_mx_close(cat["qcg"], cat["scg"], cat["qcr"], cat["scr"], cat["vc"], f"{w.name} col-wise")


def test_repack_matches_oracle():
    case = Case(synth.WORKLOADS["tiny"])
    assert_exact(np_(case.W1p), case.W1p_np, "W1p")
    back = ops.repack_fc1(case.W1p, inverse=True)
    assert torch.equal(back, case.g["W1"])


@pytest.mark.parametrize("out_mode", [L.OUT_MXFP8, L.OUT_BF16])
def test_fc1_tiny_full(out_mode):
    case = Case(synth.WORKLOADS["tiny"])
    o = run_fc1(case, out_mode)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    rt = case.rt
    _, op = act_params(case.w)
    fo = O.fc1_glu_fwd(O.permute(np_(case.inp["x"]), rt), case.W1p_np, None, rt, op)
    R = rt.R_pad
    assert_bf16_close(np_(o["pre"])[:R], fo.pre_bf16, "pre")
    if out_mode == L.OUT_MXFP8:
        q, s = O.mx_quantize_rows(fo.y)
        assert_mx_close(np_(o["q_row"])[:R], np_(o["s_row"])[:R], q, s, fo.y, "row-wise")
        qc, sc = O.mx_quantize_cols(fo.y)
        assert_mx_close(np_(o["q_col"])[:, :R], np_(o["s_col"])[:, :R // 32], qc, sc, fo.y.T, "col-wise")
    else:
        assert_bf16_close(np_(o["y"])[:R], O.bf16_round(fo.y), "y")


def test_fc1_swiglu_alpha_offset_unclamped(monkeypatch):
    """SwiGLU with alpha = 1.702 and (up + 1) but every clamp bound infinite:
    the epilogue's short SwiGLU form with non-default alpha and offset."""
    monkeypatch.setattr(sys.modules[__name__], "act_params", lambda w: (
        L.glu_params("swiglu", alpha=1.702, up_offset=1.0), O.ActParams(O.ACT_SWIGLU, alpha=1.702, up_offset=1.0)))
    case = Case(synth.WORKLOADS["tiny"])
    o = run_fc1(case, L.OUT_MXFP8)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    check_blocks(case, o, list(range(0, case.rt.R_pad, 32)), L.OUT_MXFP8)


def test_fc1_geglu_tiny_full():
    """GeGLU (exact erf) forward: the epilogue's short GeGLU form, every block."""
    case = Case(synth.scaled(synth.WORKLOADS["tiny"], act="geglu"))
    o = run_fc1(case, L.OUT_MXFP8)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    check_blocks(case, o, list(range(0, case.rt.R_pad, 32)), L.OUT_MXFP8)


def test_fc1_single_cta_kernel():
    """The single-CTA variant of the bf16 GEMM (CTA pairs switched off)."""
    lib = L.load()
    lib.moe_set_cta_pairs(0)
    try:
        case = Case(synth.WORKLOADS["tiny"])
        o = run_fc1(case, L.OUT_MXFP8)
        torch.cuda.synchronize()
        assert ops.read_status(o["status"]) == 0
        check_blocks(case, o, list(range(0, case.rt.R_pad, 32)), L.OUT_MXFP8)
    finally:
        lib.moe_set_cta_pairs(1)


def test_fc1_edge_counts():
    """Experts with 0, 1, 31, 32, 33, 127, 128, 129, 255, 256, 257 rows."""
    counts = [0, 1, 31, 32, 33, 127, 128, 129, 255, 256, 257, 0]
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).astype(np.int32)
    np.random.default_rng(3).shuffle(ids)
    w = synth.Workload("edge", ids.size, 128, len(counts), len(counts), 1, 96, "swiglu", "mxfp8", "normal")
    case = Case(w, idx=ids.reshape(-1, 1))
    o = run_fc1(case, L.OUT_MXFP8)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    check_blocks(case, o, list(range(0, case.rt.R_pad, 32)), L.OUT_MXFP8)


def test_fc1_gptoss_tail_bias_clamp():
    """F = 2880: the last N tile is half full; bias, gate clamp, alpha, +1."""
    w = synth.scaled(synth.WORKLOADS["gptoss"], T=1024)
    case = Case(w)
    o = run_fc1(case, L.OUT_MXFP8)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    check_blocks(case, o, sample_blocks(case.rt, 8, 1), L.OUT_MXFP8)


def test_fc1_dsv3_full_size_sampled():
    case = Case(synth.WORKLOADS["dsv3"])
    o = run_fc1(case, L.OUT_MXFP8)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    check_blocks(case, o, sample_blocks(case.rt, 16, 2), L.OUT_MXFP8)


def test_fc1_gptoss_full_size_sampled():
    """GPT-OSS-shaped layer at full size (T 16384, H 2880, 32 experts, top-4,
    F 2880: N1 = 5760, the last N tile half full), bias, gate clamp +-7,
    alpha 1.702, (up + 1), uniform router logits; sampled 32-row blocks."""
    case = Case(synth.WORKLOADS["gptoss"])
    o = run_fc1(case, L.OUT_MXFP8)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    check_blocks(case, o, sample_blocks(case.rt, 8, 5), L.OUT_MXFP8)


@pytest.mark.parametrize("name", ["skew", "skew_srelu"])
def test_fc1_skew_nvfp4_mode_sampled(name):
    case = Case(synth.WORKLOADS[name])
    o = run_fc1(case, L.OUT_NVFP4)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    check_blocks(case, o, sample_blocks(case.rt, 8, 3), L.OUT_NVFP4)
    # the per-tensor amax is the max |y| over every real row: bounded below
    # by the sampled rows and equal to the max of the bf16 output's magnitude
    y = o["y"][: int(case.rt.R_pad)].float()
    assert math.isclose(float(o["amax"]), float(y.abs().max()), rel_tol=1e-2)


def test_quantize_kernels_bit_exact():
    """Same bf16 input on both sides: codes and scales must be identical."""
    rng = np.random.default_rng(11)
    src = synth._bf16(rng.standard_normal((3, 96, 320), dtype=np.float32) * np.exp2(rng.integers(-8, 8, (3, 96, 1))))
    src[1, 5, 7] = float("nan")
    g = src.to(DEV)
    q, s = ops.quantize_mxfp8(g, col=False)
    qr, sr = O.mx_quantize_rows(np_(src))
    assert_exact(np_(q), qr, "rows q")
    assert_exact(np_(s), sr, "rows s")
    qc, sc = ops.quantize_mxfp8(g, col=True)
    qcr, scr = O.mx_quantize_rows(np.transpose(np_(src), (0, 2, 1)))
    assert_exact(np_(sc), scr, "cols s")
    assert_exact(np_(qc), qcr, "cols q")


def test_quantize_kernels_ragged_shapes():
    """Flat row streaming with a partial last warp task (672 blocks) and column
    tiles cut by C = 200 (not a multiple of the 64-column tile) and R = 96."""
    rng = np.random.default_rng(14)
    src = synth._bf16(rng.standard_normal((1, 96, 224), dtype=np.float32) * 5)
    q, s = ops.quantize_mxfp8(src.to(DEV), col=False)
    qr, sr = O.mx_quantize_rows(np_(src))
    assert_exact(np_(q), qr, "rows q")
    assert_exact(np_(s), sr, "rows s")
    src = synth._bf16(rng.standard_normal((2, 96, 200), dtype=np.float32))
    st = ops.new_status(DEV)
    qc, sc = ops.quantize_mxfp8(src.to(DEV), col=True, status=st)
    qcr, scr = O.mx_quantize_rows(np.transpose(np_(src), (0, 2, 1)))
    assert ops.read_status(st) == 0
    assert_exact(np_(sc), scr, "cols s")
    assert_exact(np_(qc), qcr, "cols q")


def test_quantize_grouped_rows_masks_pad():
    counts = [5, 0, 40, 64]
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).astype(np.int32)
    rt = O.route(ids.reshape(-1, 1), 0, len(counts))
    R_cap = 256
    rng = np.random.default_rng(12)
    src = synth._bf16(rng.standard_normal((R_cap, 64), dtype=np.float32))
    cnt = torch.from_numpy(rt.counts.astype(np.int32)).to(DEV)
    off = torch.from_numpy(rt.offsets.astype(np.int32)).to(DEV)
    masked = np_(src).copy()
    masked[: rt.R_pad][rt.tok_of < 0] = 0
    q, s = ops.quantize_mxfp8(src.to(DEV), col=True, counts=cnt, offsets=off)
    qr, sr = O.mx_quantize_cols(masked[: rt.R_pad])
    assert_exact(np_(q)[:, : rt.R_pad], qr, "grouped cols q")
    assert_exact(np_(s)[:, : rt.R_pad // 32], sr, "grouped cols s")
    q, s = ops.quantize_mxfp8(src.to(DEV), col=False, counts=cnt, offsets=off)
    qr, sr = O.mx_quantize_rows(masked[: rt.R_pad])
    assert_exact(np_(q)[: rt.R_pad], qr, "grouped rows q")
    assert_exact(np_(s)[: rt.R_pad], sr, "grouped rows s")


def test_nvfp4_cast_bit_exact():
    rng = np.random.default_rng(13)
    R, N = 96, 256
    y = synth._bf16(rng.standard_normal((R, N), dtype=np.float32) * 3)
    amax = float(np_(y).__abs__().max())
    offsets = torch.tensor([0, 64, 96], dtype=torch.int32, device=DEV)
    counts = torch.tensor([64, 32], dtype=torch.int32, device=DEV)
    q, s, sg = ops.nvfp4_cast(y.to(DEV), torch.tensor([amax], device=DEV), counts, offsets)
    sg_ref = O.nvfp4_global_scale(amax)
    assert float(sg) == float(sg_ref)
    qr, sr = O.nvfp4_quantize_rows(np_(y), sg_ref)
    assert_exact(np_(s), sr, "nvfp4 scales")
    assert_exact(np_(q), qr, "nvfp4 codes")


# Every activation form the unfused kernels are instantiated for: plain
# SwiGLU, clamped GPT-OSS SwiGLU with alpha and the +1 offset, GeGLU with an
# offset on the linear half, the general forms (sReGLU), and sReLU without a
# gate.
UNFUSED_ACTS = {
    "swiglu": ({}, O.ACT_SWIGLU),
    "swiglu_oss": ({"alpha": 1.702, "up_offset": 1.0, "gate_lo": -7.0, "gate_hi": 7.0, "up_lo": -7.0, "up_hi": 7.0},
                   O.ACT_SWIGLU),
    "geglu": ({"up_offset": 0.5}, O.ACT_GEGLU),
    "sreglu": ({}, O.ACT_SREGLU),
    "srelu": ({}, O.ACT_SRELU),
}


def _unfused_params(name):
    kw, oact = UNFUSED_ACTS[name]
    act = {O.ACT_SWIGLU: "swiglu", O.ACT_GEGLU: "geglu", O.ACT_SREGLU: "sreglu", O.ACT_SRELU: "srelu"}[oact]
    return L.glu_params(act, **kw), O.ActParams(oact, **kw)


@pytest.mark.parametrize("name", list(UNFUSED_ACTS))
def test_unfused_glu_act(name):
    rng = np.random.default_rng(14)
    F, R = 128, 96
    prm_c, prm = _unfused_params(name)
    N1 = F if prm.act == O.ACT_SRELU else 2 * F
    pre = synth._bf16(rng.standard_normal((R, N1), dtype=np.float32) * 4)
    # rows past offsets[E] are not processed and stay as they were
    offsets = torch.tensor([0, 32, 80], dtype=torch.int32, device=DEV)
    counts = torch.tensor([32, 48], dtype=torch.int32, device=DEV)
    y = ops.glu_act(pre.to(DEV), counts, offsets, F, prm_c)
    p = np_(pre)[:80]
    ref = O.act_fwd(p, None, prm) if prm.act == O.ACT_SRELU else O.act_fwd(*O.unpack_glu_cols(p), prm)
    assert_bf16_close(np_(y)[:80], O.bf16_round(ref), "glu_act")


@pytest.mark.parametrize("name", list(UNFUSED_ACTS))
def test_unfused_dglu_act(name):
    rng = np.random.default_rng(15)
    F, R = 128, 96
    prm_c, prm = _unfused_params(name)
    N1 = F if prm.act == O.ACT_SRELU else 2 * F
    pre = synth._bf16(rng.standard_normal((R, N1), dtype=np.float32) * 4)
    da = synth._bf16(rng.standard_normal((R, F), dtype=np.float32))
    offsets = torch.tensor([0, 32, 80], dtype=torch.int32, device=DEV)
    counts = torch.tensor([32, 48], dtype=torch.int32, device=DEV)
    d = ops.dglu_act(da.to(DEV), pre.to(DEV), counts, offsets, F, prm_c)
    p, dy = np_(pre)[:80], np_(da)[:80]
    if prm.act == O.ACT_SRELU:
        ref, _ = O.act_bwd(p, None, dy, prm)
    else:
        du, dg = O.act_bwd(*O.unpack_glu_cols(p), dy, prm)
        ref = O.pack_glu_cols(du, dg)
    assert_bf16_close(np_(d)[:80], O.bf16_round(ref), "dglu_act")
