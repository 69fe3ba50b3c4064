"""Dynamic tile scheduler of the CTA-pair bf16 GEMMs ([MoE-Fusion]: dynamic
scheduling, so that the grouped kernels share the GPU with concurrent
kernels): the clusters take tiles from an atomic counter, so which cluster
computes a tile depends on timing, but every tile is computed the same way.
Outputs must be bit-identical to the static schedule's, alone, next to a
kernel that occupies SMs on another stream, and with two calls in flight on
two streams with their own workspaces."""
import numpy as np
import pytest
import torch

import test_gpu_fc1 as F
from grouped_gemm_glu_gb300 import lib as L
from grouped_gemm_glu_gb300 import ops, synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
KEYS = ("q_row", "s_row", "q_col", "s_col", "y", "pre", "amax", "dbias")


def _same(a, b, what, R):
    """Outputs are defined on the rows of the padded segments (R = offsets[E])."""
    view = {"q_row": lambda t: t[:R], "s_row": lambda t: t[:R], "y": lambda t: t[:R], "pre": lambda t: t[:R],
            "q_col": lambda t: t[:, :R], "s_col": lambda t: t[:, :R // 32]}
    for k in KEYS:
        if k in a or k in b:
            f = view.get(k, lambda t: t)
            assert torch.equal(f(a[k]), f(b[k])), f"{what}: {k} differs between schedules"


def _case(name):
    if name == "edge":
        counts = [0, 1, 31, 32, 33, 127, 128, 129, 255, 256, 257, 300, 0, 511, 512, 513]
        ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).astype(np.int32)
        np.random.default_rng(7).shuffle(ids)
        w = synth.Workload("edge", ids.size, 256, len(counts), len(counts), 1, 160, "swiglu", "mxfp8", "normal",
                           bias=True, gpt_oss=True)
        return F.Case(w, idx=ids.reshape(-1, 1))
    return F.Case(synth.scaled(synth.WORKLOADS["gptoss"], T=2048))


@pytest.mark.parametrize("name", ["edge", "gptoss"])
@pytest.mark.parametrize("out_mode", [L.OUT_MXFP8, L.OUT_NVFP4])
def test_dynamic_matches_static(name, out_mode):
    case = _case(name)
    w = case.w
    gp, _ = F.act_params(w)
    args = (case.r["x_perm"], case.W1p, case.r["counts"], case.r["offsets"], w.F, gp, out_mode)
    fs = ops.fc1_fwd(*args, b1p=case.b1p, dynamic=False)
    fd = ops.fc1_fwd(*args, b1p=case.b1p, dynamic=True)
    torch.cuda.synchronize()
    assert ops.read_status(fd["status"]) == 0
    _same(fs, fd, "FC1", case.rt.R_pad)
    dY = case.inp["dY"].to(DEV)
    W2 = case.g["W2"]
    bs = ops.dglu_bwd(dY, W2, fs["pre"], case.r["counts"], case.r["offsets"], w.F, gp, out_mode, dbias=True,
                      dynamic=False)
    bd = ops.dglu_bwd(dY, W2, fs["pre"], case.r["counts"], case.r["offsets"], w.F, gp, out_mode, dbias=True,
                      dynamic=True)
    torch.cuda.synchronize()
    assert ops.read_status(bd["status"]) == 0
    _same(bs, bd, "dGLU", case.rt.R_pad)


def test_dynamic_with_a_concurrent_kernel_and_sm_margin():
    """FC1 and dGLU on one stream with sm_margin = 16 while another stream
    keeps SMs busy with a long elementwise loop: same results as alone."""
    case = _case("gptoss")
    w = case.w
    gp, _ = F.act_params(w)
    args = (case.r["x_perm"], case.W1p, case.r["counts"], case.r["offsets"], w.F, gp, L.OUT_MXFP8)
    ref = ops.fc1_fwd(*args, b1p=case.b1p, dynamic=False)
    torch.cuda.synchronize()
    busy = torch.randn(1 << 26, device=DEV)
    other = torch.cuda.Stream()
    mine = torch.cuda.Stream()
    start = torch.cuda.Event()
    start.record()
    other.wait_event(start)
    mine.wait_event(start)
    with torch.cuda.stream(other):
        for _ in range(20):
            busy.mul_(1.0000001).add_(1e-7)
    with torch.cuda.stream(mine):
        outs = [ops.fc1_fwd(*args, b1p=case.b1p, dynamic=True, sm_margin=16) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs:
        assert ops.read_status(o["status"]) == 0
        _same(ref, o, "FC1 next to a concurrent kernel", case.rt.R_pad)


def test_two_calls_in_flight_on_two_streams():
    """Two FC1 calls running at the same time, each with its own workspace."""
    case = _case("edge")
    w = case.w
    gp, _ = F.act_params(w)
    args = (case.r["x_perm"], case.W1p, case.r["counts"], case.r["offsets"], w.F, gp, L.OUT_MXFP8)
    ref = ops.fc1_fwd(*args, b1p=case.b1p, dynamic=False)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ev = torch.cuda.Event()
    ev.record()
    s1.wait_event(ev)
    s2.wait_event(ev)
    with torch.cuda.stream(s1):
        o1 = ops.fc1_fwd(*args, b1p=case.b1p, dynamic=True, sm_margin=76)
    with torch.cuda.stream(s2):
        o2 = ops.fc1_fwd(*args, b1p=case.b1p, dynamic=True, sm_margin=76)
    torch.cuda.synchronize()
    _same(ref, o1, "stream 1", case.rt.R_pad)
    _same(ref, o2, "stream 2", case.rt.R_pad)
