"""The allocation-free routing entry point against the regular one.

moe_route_permute_noalloc serves callers that cannot allocate device memory
while they route (a runtime that owns all GPU memory in its own pool, code
running where cudaMalloc is not allowed): its scratch is a fixed array inside
the library.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes on its own in a
fresh process."""
import ctypes as C

import numpy as np
import pytest
import torch

from grouped_gemm_glu_gb300 import lib as L
from grouped_gemm_glu_gb300 import ops, synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
P = lambda t: C.c_void_p(t.data_ptr())


def _outputs(T, H, k, E, R_cap):
    return {
        "x_perm": torch.zeros(R_cap, H, dtype=torch.bfloat16, device=DEV),
        "row_of": torch.zeros(T * k, dtype=torch.int32, device=DEV),
        "tok_of": torch.zeros(R_cap, dtype=torch.int32, device=DEV),
        "prob_perm": torch.zeros(R_cap, dtype=torch.float32, device=DEV),
        "counts": torch.zeros(E, dtype=torch.int32, device=DEV),
        "offsets": torch.zeros(E + 1, dtype=torch.int32, device=DEV),
        "status": torch.zeros(1, dtype=torch.int32, device=DEV),
    }


def _noalloc(x, idx, prob, E, R_cap, expert_begin=0):
    lib = L.load()
    T, H = x.shape
    k = idx.shape[1]
    o = _outputs(T, H, k, E, R_cap)
    rc = lib.moe_route_permute_noalloc(P(x), P(idx), P(prob), T, H, k, expert_begin, E, R_cap, P(o["x_perm"]),
                                       P(o["row_of"]), P(o["tok_of"]), P(o["prob_perm"]), P(o["counts"]),
                                       P(o["offsets"]), None, None, P(o["status"]),
                                       C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == L.MOE_OK
    return o


def _compare(x, idx, prob, E, R_cap, expert_begin=0):
    ref = ops.route_permute(x, idx, prob, E, R_cap, expert_begin)
    got = _noalloc(x, idx, prob, E, R_cap, expert_begin)
    torch.cuda.synchronize()
    assert ops.read_status(got["status"]) == ops.read_status(ref["status"]) == 0
    R = int(ref["offsets"][-1])
    for key in ("counts", "offsets", "row_of"):
        assert torch.equal(got[key], ref[key]), key
    for key in ("tok_of", "prob_perm", "x_perm"):
        assert torch.equal(got[key][:R], ref[key][:R]), key


def _inputs(name, seed, H=256):
    w = synth.scaled(synth.WORKLOADS[name], H=H)
    idx, prob = synth.router_inputs(w, np.random.default_rng(seed))
    x = synth._bf16(np.random.default_rng(seed + 1).standard_normal((w.T, w.H), dtype=np.float32))
    return w, x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(prob).to(DEV)


def test_noalloc_matches_route_permute_two_calls_in_a_row():
    # two different routings back to back through the same fixed scratch
    w, x, idx, prob = _inputs("dsv3", 1)
    _compare(x, idx, prob, w.E, w.capped_R(2.0))
    w2, x2, idx2, prob2 = _inputs("skew", 2, H=128)
    _compare(x2, idx2, prob2, w2.E, w2.R_cap)


def test_noalloc_repeated_calls_same_input():
    w, x, idx, prob = _inputs("tiny", 3)
    _compare(x, idx, prob, w.E, w.R_cap)
    _compare(x, idx, prob, w.E, w.R_cap)


def test_noalloc_rejects_routing_beyond_its_scratch():
    lib = L.load()
    cap = lib.moe_route_noalloc_max_scratch_bytes()
    assert cap == 1 << 20
    T, k, E = 1 << 16, 8, 1024      # 256 chunks x 1024 experts of bases: 1 MiB + flag
    assert lib.moe_route_workspace_size(T, k, E) > cap
    x = torch.zeros(T, 8, dtype=torch.bfloat16, device=DEV)
    idx = torch.zeros(T, k, dtype=torch.int32, device=DEV)
    prob = torch.zeros(T, k, dtype=torch.float32, device=DEV)
    o = _outputs(T, 8, k, E, 128)
    rc = lib.moe_route_permute_noalloc(P(x), P(idx), P(prob), T, 8, k, 0, E, 128, P(o["x_perm"]), P(o["row_of"]),
                                       P(o["tok_of"]), P(o["prob_perm"]), P(o["counts"]), P(o["offsets"]),
                                       None, None, P(o["status"]), None)
    assert rc == L.MOE_ERR_ARG
