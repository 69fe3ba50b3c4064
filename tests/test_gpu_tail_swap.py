"""Swapped tail tiles of the CTA-pair bf16 GEMMs (an expert's last, thin
256-row pair tile computed with the weights as the M operand and its rows as
N): every output mode and epilogue form against the oracle with the swap
off and at each allowed threshold, on expert counts that put tails of 1..257
rows in the swapped and in the regular path."""
import math

import numpy as np
import pytest
import torch

import test_gpu_bwd_mx as B
import test_gpu_fc1 as F
from grouped_gemm_glu_gb300 import lib as L
from grouped_gemm_glu_gb300 import ops, synth
from oracle import moe_oracle as O
from parity import assert_bf16_close, np_

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
COUNTS = [0, 1, 31, 32, 33, 63, 64, 65, 96, 127, 128, 129, 255, 256, 257, 300, 0]


@pytest.fixture(params=[0, 32, 64, 128], ids=lambda v: f"swap{v}")
def swap(request):
    lib = L.load()
    assert lib.moe_set_tail_swap(request.param) == 0
    yield request.param
    lib.moe_set_tail_swap(32)


def _edge_ids():
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(COUNTS)]).astype(np.int32)
    np.random.default_rng(3).shuffle(ids)
    return ids.reshape(-1, 1)


def test_threshold_validation():
    lib = L.load()
    for bad in (-32, 16, 160, 256):
        assert lib.moe_set_tail_swap(bad) == L.MOE_ERR_ARG
    assert lib.moe_set_tail_swap(32) == 0


@pytest.mark.parametrize("act", ["swiglu", "geglu", "srelu"])
@pytest.mark.parametrize("out_mode", [L.OUT_MXFP8, L.OUT_BF16])
def test_fc1_swapped_tails(swap, act, out_mode):
    ids = _edge_ids()
    w = synth.Workload("edge", ids.size, 128, len(COUNTS), len(COUNTS), 1, 96, act, "mxfp8", "normal")
    case = F.Case(w, idx=ids)
    o = F.run_fc1(case, out_mode)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    F.check_blocks(case, o, list(range(0, case.rt.R_pad, 32)), out_mode)


def test_fc1_swapped_tails_gptoss_bias_rowscale(swap):
    """GPT-OSS activation with bias and a per-row scale on tails of every size."""
    ids = _edge_ids()
    w = synth.Workload("edge", ids.size, 128, len(COUNTS), len(COUNTS), 1, 96, "swiglu", "mxfp8", "normal",
                       bias=True, gpt_oss=True)
    case = F.Case(w, idx=ids)
    gp, op = F.act_params(w)
    rs = torch.rand(w.R_cap, generator=torch.Generator().manual_seed(4)) + 0.5
    o = ops.fc1_fwd(case.r["x_perm"], case.W1p, case.r["counts"], case.r["offsets"], w.F, gp, L.OUT_BF16,
                    b1p=case.b1p, row_scale=rs.to(DEV))
    torch.cuda.synchronize()
    rt = case.rt
    x = O.permute(np_(case.inp["x"]), rt)
    fo = O.fc1_glu_fwd(x, case.W1p_np, case.b1p_np, rt, op, row_scale=np_(rs)[: rt.R_pad])
    R = rt.R_pad
    assert_bf16_close(np_(o["y"])[:R], O.bf16_round(fo.y), "y")
    assert_bf16_close(np_(o["pre"])[:R], fo.pre_bf16, "pre")


@pytest.mark.parametrize("act", ["swiglu", "geglu", "srelu"])
def test_dglu_swapped_tails(swap, act):
    w = synth.Workload("edge", sum(COUNTS), 128, len(COUNTS), len(COUNTS), 1, 96, act, "mxfp8", "normal")
    B._dglu_case(w, counts=COUNTS)
    B._dglu_case(w, counts=COUNTS, out_mode=L.OUT_BF16)


def test_dglu_swapped_tails_nvfp4_rht_and_dbias(swap):
    """NVFP4 backward (bf16 dFC1, max |dFC1|, rotated transposed amax) and the
    bias gradient, both of which the swapped tiles compute in their own
    (transposed) layout."""
    w = synth.Workload("edge", sum(COUNTS), 128, len(COUNTS), len(COUNTS), 1, 96, "swiglu", "mxfp8", "normal",
                       bias=True, gpt_oss=True)
    rt, cnt, off = B._routing(w, 0, COUNTS)
    inp = synth.make_inputs(w, 0)
    pre = synth._bf16(np.random.default_rng(100).standard_normal((w.R_cap, w.N1), dtype=np.float32) * 2.0)
    gp, op = B._act(w)
    o = ops.dglu_bwd(inp["dY"].to(DEV), inp["W2"].to(DEV), pre.to(DEV), cnt, off, w.F, gp, L.OUT_NVFP4,
                     rht_signs=0xB3C5, dbias=True)
    torch.cuda.synchronize()
    assert ops.read_status(o["status"]) == 0
    R = rt.R_pad
    d = O.dglu_bwd(np_(inp["dY"])[:R], np_(inp["W2"]), np_(pre)[:R], rt, op)
    y = np_(o["y"])[:R]
    assert_bf16_close(y, O.bf16_round(d), "dFC1 bf16")
    assert math.isclose(float(o["rht_amax"].item()), O.rht_transposed_amax(y, 0xB3C5), rel_tol=1e-5)
    assert math.isclose(float(o["amax"].item()), float(np.max(np.abs(d))), rel_tol=2e-2)
    ref = O.fc1_bias_grad(d, rt)
    lim = 1e-3 * O.fc1_bias_grad(np.abs(d), rt) + 1e-6
    assert np.all(np.abs(np_(o["dbias"]) - ref) <= lim)


def test_plain_gemm_swapped_tails(swap):
    """The plain bf16 grouped GEMM (GroupGemm + Quantize with bf16 operands,
    and the unfused path's pre-activation GEMM) on the same tails."""
    E, K, N = len(COUNTS), 128, 320
    w = synth.Workload("edge", sum(COUNTS), K, E, E, 1, 64, "swiglu", "mxfp8", "normal")
    rt, cnt, off = B._routing(w, 0, COUNTS)
    rng = np.random.default_rng(6)
    A = synth._bf16(rng.standard_normal((w.R_cap, K), dtype=np.float32))
    W = synth._bf16(rng.standard_normal((E, N, K), dtype=np.float32) / np.sqrt(K))
    y = ops.fc2_fwd(A.to(DEV), None, W.to(DEV), None, cnt, off)
    torch.cuda.synchronize()
    ref = O.grouped_gemm_quant_fwd(np_(A)[: rt.R_pad], np_(W), rt)
    assert_bf16_close(np_(y)[: rt.R_pad], O.bf16_round(ref), "plain gemm")
    pre = ops.fc1_fwd(A.to(DEV), W.to(DEV), cnt, off, N, L.glu_params("none"), L.OUT_BF16)["pre"]
    torch.cuda.synchronize()
    assert_bf16_close(np_(pre)[: rt.R_pad], O.bf16_round(ref), "unfused pre-activation gemm")
