"""GPU parity of routing, permutation and combine against the oracle
(bit-exact integers and copies; combine within the bf16 rule)."""
import numpy as np
import pytest
import torch

from grouped_gemm_glu_gb300 import ops, synth
from grouped_gemm_glu_gb300 import lib as L
from oracle import moe_oracle as O
from parity import assert_bf16_close, assert_exact, np_

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _check_route(x, idx, prob, E, R_cap, expert_begin=0):
    g = ops.route_permute(x.to(DEV), idx.to(DEV), prob.to(DEV), E, R_cap, expert_begin)
    torch.cuda.synchronize()
    assert ops.read_status(g["status"]) == 0
    rt = O.route(idx.numpy(), expert_begin, E)
    assert_exact(np_(g["counts"]), rt.counts, "counts")
    assert_exact(np_(g["offsets"]), rt.offsets, "offsets")
    assert_exact(np_(g["row_of"]), rt.row_of, "row_of")
    R = rt.R_pad
    assert_exact(np_(g["tok_of"])[:R], rt.tok_of, "tok_of")
    assert_exact(np_(g["prob_perm"])[:R], O.permute_probs(prob.numpy(), rt).astype(np.float32), "prob_perm")
    xp = np_(g["x_perm"])[:R]
    assert_exact(xp, O.permute(np_(x), rt), "x_perm")
    return g, rt


@pytest.mark.parametrize("name", ["tiny", "dsv3", "gptoss", "skew"])
def test_route_permute_workloads(name):
    w = synth.WORKLOADS[name]
    if name in ("gptoss", "skew"):
        w = synth.scaled(w, H=256)       # routing does not depend on H; keep the copy small
    rs = synth._streams(3, 2)
    idx, prob = synth.router_inputs(w, rs[0])
    x = synth._bf16(rs[1].standard_normal((w.T, w.H), dtype=np.float32))
    _check_route(x, torch.from_numpy(idx), torch.from_numpy(prob), w.E, w.R_cap, w.expert_begin)


def test_route_edge_cases():
    # counts 0, 1, 31, 32, 33, 127, 128, 129, 0 (last expert empty), all with k = 1
    counts = [0, 1, 31, 32, 33, 127, 128, 129, 0]
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)])
    rng = np.random.default_rng(5)
    rng.shuffle(ids)
    T, H = ids.size, 64
    x = synth._bf16(rng.standard_normal((T, H), dtype=np.float32))
    prob = torch.from_numpy(rng.random((T, 1), dtype=np.float32))
    E = len(counts)
    R_cap = ((T + 31 * E) + 127) // 128 * 128
    _check_route(x, torch.from_numpy(ids.reshape(T, 1).astype(np.int32)), prob, E, R_cap)


def test_route_drops_non_local_experts_and_all_on_one():
    rng = np.random.default_rng(6)
    T, k, H = 3000, 3, 32
    idx = np.stack([rng.permutation(12)[:k] for _ in range(T)]).astype(np.int32)
    x = synth._bf16(rng.standard_normal((T, H), dtype=np.float32))
    prob = torch.from_numpy(rng.random((T, k), dtype=np.float32))
    _check_route(x, torch.from_numpy(idx), prob, 5, ((T * k + 31 * 5) + 127) // 128 * 128, expert_begin=4)
    one = np.full((T, 1), 2, dtype=np.int32)
    _check_route(x, torch.from_numpy(one), prob[:, :1].contiguous(), 4, ((T + 31 * 4) + 127) // 128 * 128)


def test_route_capacity_overflow_sets_status():
    rng = np.random.default_rng(7)
    T, H = 1000, 32
    idx = torch.from_numpy(rng.integers(0, 4, size=(T, 2)).astype(np.int32))
    x = synth._bf16(rng.standard_normal((T, H), dtype=np.float32)).to(DEV)
    prob = torch.from_numpy(rng.random((T, 2), dtype=np.float32)).to(DEV)
    g = ops.route_permute(x, idx.to(DEV), prob, 4, 512)
    st = ops.read_status(g["status"])
    assert st & L.MOE_ERR_CAPACITY
    assert int(g["offsets"][-1]) > 512
    assert bool((g["row_of"] == -1).all())


def test_combine_matches_oracle():
    w = synth.WORKLOADS["tiny"]
    rng = np.random.default_rng(8)
    idx, prob = synth.router_inputs(w, rng)
    rt = O.route(idx, 0, w.E)
    y = synth._bf16(rng.standard_normal((w.R_cap, w.H), dtype=np.float32))
    out = ops.unpermute_combine(y.to(DEV), torch.from_numpy(rt.row_of.astype(np.int32)).to(DEV),
                                torch.from_numpy(prob).to(DEV))
    ref = O.bf16_round(O.unpermute_combine(np_(y), rt.row_of, prob))
    assert_bf16_close(np_(out), ref, "combine")


def test_combine_dsv3_shape_with_dropped_assignments():
    w = synth.WORKLOADS["dsv3"]
    rng = np.random.default_rng(9)
    idx, prob = synth.router_inputs(w, rng)
    rt = O.route(idx, 0, w.E)
    y = synth._bf16(rng.standard_normal((rt.R_pad, w.H), dtype=np.float32))
    out = ops.unpermute_combine(y.to(DEV), torch.from_numpy(rt.row_of.astype(np.int32)).to(DEV),
                                torch.from_numpy(prob).to(DEV))
    sel = rng.choice(w.T, 256, replace=False)
    ref = O.bf16_round(O.unpermute_combine(np_(y), rt.row_of.reshape(w.T, w.k)[sel].reshape(-1), prob[sel]))
    assert_bf16_close(np_(out)[sel], ref, "combine dsv3")


def test_permute_unpermute_round_trip_identity():
    rng = np.random.default_rng(10)
    T, H, E = 777, 128, 6
    idx = torch.from_numpy(rng.integers(0, E, size=(T, 1)).astype(np.int32))
    x = synth._bf16(rng.standard_normal((T, H), dtype=np.float32)).to(DEV)
    ones = torch.ones(T, 1, dtype=torch.float32, device=DEV)
    g = ops.route_permute(x, idx.to(DEV), ones, E, ((T + 31 * E) + 127) // 128 * 128)
    out = ops.unpermute_combine(g["x_perm"], g["row_of"], ones)
    assert torch.equal(out, x)


@pytest.mark.parametrize("k,H", [(3, 2880), (6, 4096), (12, 2880), (32, 256)])
def test_combine_and_permute_bwd_warp_per_token_k(k, H):
    """Top-k other than 4 and 8 runs the one-warp-per-token kernel: a row
    width that is not a multiple of the warp's 128-chunk step (H = 2880), and
    a shard that sees only some of each token's experts (dropped slots)."""
    rng = np.random.default_rng(20 + k)
    T, n_experts, E, begin = 1024, 64, 16, 8
    idx = np.stack([rng.permutation(n_experts)[:k] for _ in range(T)]).astype(np.int32)
    prob = rng.random((T, k), dtype=np.float32)
    rt = O.route(idx, begin, E)
    R = int(rt.R_pad)
    y = synth._bf16(rng.standard_normal((R, H), dtype=np.float32))
    row_of = torch.from_numpy(rt.row_of.astype(np.int32)).to(DEV)
    out = ops.unpermute_combine(y.to(DEV), row_of, torch.from_numpy(prob).to(DEV))
    ref = O.bf16_round(O.unpermute_combine(np_(y), rt.row_of, prob))
    assert_bf16_close(np_(out), ref, f"combine k={k}")
    dx = ops.permute_bwd(y.to(DEV), row_of, T, k)
    ref = O.bf16_round(O.permute_bwd(np_(y), rt.row_of, T, k))
    assert_bf16_close(np_(dx), ref, f"permute bwd k={k}")
