"""Multi-rank (gloo, CPU) test of the expert-parallel shard logic: ranks
route the same batch on their own expert ranges; together they keep every
assignment exactly once, and each rank's kept set is what a single shard of
that range would keep."""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from grouped_gemm_glu_gb300 import shard, synth
from oracle import moe_oracle as O


def _worker(rank, world, port, E, n_experts, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.scaled(synth.WORKLOADS["dsv3"], T=2048, n_experts=n_experts, E=E)
        idx, _ = synth.router_inputs(w, np.random.default_rng(5))       # same batch on every rank
        eb = shard.shard_expert_begin(rank, E, n_experts)
        rt = O.route(idx, eb, E)
        kept = torch.from_numpy((rt.row_of >= 0).astype(np.int64))
        counts = torch.from_numpy(rt.counts.astype(np.int64))
        allk = [torch.zeros_like(kept) for _ in range(world)]
        dist.all_gather(allk, kept)
        allc = [torch.zeros_like(counts) for _ in range(world)]
        dist.all_gather(allc, counts)
        if rank == 0:
            total = torch.stack(allk).sum(0)
            q.put((int(total.min()), int(total.max()), int(torch.stack(allc).sum()), idx.size))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,E,n_experts", [(2, 16, 32), (2, 4, 8)])
def test_two_rank_shards_partition_assignments(world, E, n_experts):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, world, port, E, n_experts, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    lo, hi, n_kept, n_assign = q.get(timeout=10)
    assert lo == 1 and hi == 1          # every assignment kept by exactly one rank
    assert n_kept == n_assign
    assert shard.shards_cover(world, E, n_experts)


def test_shard_begin_wraps_and_validates():
    assert [shard.shard_expert_begin(r, 32, 256) for r in range(9)] == [0, 32, 64, 96, 128, 160, 192, 224, 0]
    assert not shard.shards_cover(4, 32, 256)
    with pytest.raises(ValueError):
        shard.shard_expert_begin(0, 0, 8)
