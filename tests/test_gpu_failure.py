"""Failure detection without a GPU fault: the bounded wait behind every
pipeline wait of the persistent kernels gives up after its limit, records
MOE_ERR_TIMEOUT in the status word and returns, and the context stays
usable.  The wait that runs out is one on an mbarrier nothing arrives at."""
import numpy as np
import pytest
import torch

from grouped_gemm_glu_gb300 import lib as L
from grouped_gemm_glu_gb300 import ops
from oracle import moe_oracle as O

DEV = "cuda:0"
LIMIT_NS = 2_000_000
DEFAULT_LIMIT_NS = 2_000_000_000


@pytest.mark.gpu
def test_bounded_wait_gives_up_and_context_stays_usable():
    lib = L.load()
    lib.moe_set_wait_limit_ns(LIMIT_NS)
    try:
        st, waited = ops.wait_selftest(False, DEV)
        assert st & L.MOE_ERR_TIMEOUT, st
        assert st == L.MOE_ERR_TIMEOUT, st
        # the guard reads the clock every 64 polls: it stops soon after the limit
        assert LIMIT_NS <= waited < LIMIT_NS + 20_000_000, waited
        # a wait whose barrier completes is not flagged
        st, waited = ops.wait_selftest(True, DEV)
        assert st == L.MOE_OK, st
        assert waited < LIMIT_NS, waited
    finally:
        lib.moe_set_wait_limit_ns(DEFAULT_LIMIT_NS)
    # the context still runs the library's kernels correctly
    rng = np.random.default_rng(3)
    T, H, k, E = 64, 256, 2, 4
    idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
    idx[:, 1] = (idx[:, 0] + 1) % E
    prob = rng.random((T, k), dtype=np.float32)
    x = torch.randn(T, H, dtype=torch.bfloat16)
    R_cap = 256  # >= T*k + 31*E, a multiple of 32
    r = ops.route_permute(x.to(DEV), torch.from_numpy(idx).to(DEV), torch.from_numpy(prob).to(DEV), E, R_cap)
    ref = O.route(idx, 0, E)
    assert np.array_equal(r["counts"].cpu().numpy(), ref.counts)
    assert ops.read_status(r["status"]) == L.MOE_OK
