"""Seeded synthetic inputs for the MoE MLP hot path.

This module only draws random inputs of the right shapes, value
distributions and routing structure.  It computes none of the method's
steps: the router (softmax and top-k over logits) is the caller's business
and is drawn here as input, exactly as a training framework would hand it
over.  Both the CUDA library's tests/bench and the CPU oracle's tests consume
what it returns; it imports neither.

Workloads (names used across tests, bench and docs):
  tiny    T=512,   H=256,  4 experts of 4,   top-2, F=512,  SwiGLU, bf16 out
  dsv3    T=8192,  H=7168, 32 experts of 256 (one expert-parallel shard),
          top-8, F=2048, SwiGLU, MXFP8 out + transposed copy (and its
          backward: dY ~ N(0,1) over the routed rows)
  gptoss  T=16384, H=2880, 32 experts, top-4, F=2880, SwiGLU with gate clamp
          +-7, alpha 1.702, (up + 1), FC1 bias ~ N(0, 0.02^2), MXFP8 out
  skew    T=32768, H=4096, 64 experts, top-6, F=1536, logits + Zipf(1.2)
          expert bias (8 experts never chosen), GeGLU or sReLU, NVFP4 out
Weights are N(0, 1/H) (variance) for both FC1 and FC2; x ~ N(0, 1).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int               # local experts (this shard)
    n_experts: int       # experts the router chooses among
    k: int
    F: int
    act: str             # "swiglu" | "geglu" | "srelu"
    out: str             # "bf16" | "mxfp8" | "nvfp4"
    router: str          # "normal" | "uniform" | "zipf"
    bias: bool = False
    gpt_oss: bool = False
    expert_begin: int = 0

    @property
    def gated(self) -> bool:
        return self.act != "srelu"

    @property
    def N1(self) -> int:
        """FC1 output width: 2F when gated (input | gate), F otherwise."""
        return 2 * self.F if self.gated else self.F

    @property
    def R_cap(self) -> int:
        """Capacity of the permuted buffers: every assignment local plus
        up to 31 pad rows per expert, rounded up to a multiple of 128."""
        r = self.T * min(self.k, self.E) + self.E * 31
        return (r + 127) // 128 * 128

    def capped_R(self, factor: float) -> int:
        """A smaller capacity for an expert-parallel shard: `factor` times the
        expected number of local rows plus the padding (routing reports
        MOE_ERR_CAPACITY if a batch ever exceeds it)."""
        expect = self.T * self.k * self.E / self.n_experts
        r = min(int(factor * expect), self.T * min(self.k, self.E)) + self.E * 31
        return (r + 127) // 128 * 128


WORKLOADS = {
    "tiny": Workload("tiny", 512, 256, 4, 4, 2, 512, "swiglu", "bf16", "normal"),
    "dsv3": Workload("dsv3", 8192, 7168, 32, 256, 8, 2048, "swiglu", "mxfp8", "normal"),
    "gptoss": Workload("gptoss", 16384, 2880, 32, 32, 4, 2880, "swiglu", "mxfp8", "uniform",
                       bias=True, gpt_oss=True),
    "skew": Workload("skew", 32768, 4096, 64, 64, 6, 1536, "geglu", "nvfp4", "zipf"),
    "skew_srelu": Workload("skew_srelu", 32768, 4096, 64, 64, 6, 1536, "srelu", "nvfp4", "zipf"),
}


def scaled(w: Workload, **kw) -> Workload:
    """A copy of a workload with some sizes replaced (smaller parity cases)."""
    d = dict(w.__dict__)
    d.update(kw)
    return Workload(**d)


def _streams(seed: int, n: int):
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


_CHUNK = 1 << 22


def _normal(ss: np.random.SeedSequence, shape, scale: float = 1.0) -> np.ndarray:
    """float32 N(0, scale^2) of the given shape, filled in fixed chunks of 4M
    values, each from its own child seed (so the values do not depend on the
    number of threads that fill them)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    nch = (n + _CHUNK - 1) // _CHUNK
    seeds = ss.spawn(nch)

    def fill(i):
        seg = out[i * _CHUNK:min(n, (i + 1) * _CHUNK)]
        np.random.default_rng(seeds[i]).standard_normal(seg.shape[0], dtype=np.float32, out=seg)
        if scale != 1.0:
            seg *= np.float32(scale)

    with ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as ex:
        list(ex.map(fill, range(nch)))
    return out.reshape(shape)


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def router_inputs(w: Workload, rng: np.random.Generator):
    """Top-k expert ids (int32 [T, k]) and their router probabilities
    (float32 [T, k]) drawn from synthetic logits.  Ties go to the lower
    expert id; probabilities are the softmax values, not renormalised."""
    T, n = w.T, w.n_experts
    if w.router == "normal":
        logits = rng.standard_normal((T, n), dtype=np.float32)
    elif w.router == "uniform":
        logits = rng.random((T, n), dtype=np.float32)
    elif w.router == "zipf":
        # Zipf(s=1.2) popularity as a log-bias over a seeded ranking of the
        # experts; the 8 lowest-ranked experts are never chosen.  The hottest
        # expert is then picked by ~97% of tokens (~10x the mean load, close
        # to the most a top-6 router with distinct experts allows).
        rank = rng.permutation(n) + 1
        bias = -1.2 * np.log(rank.astype(np.float64))
        dead = rank > n - 8
        bias[dead] = -np.inf
        logits = (rng.standard_normal((T, n)) + bias[None, :]).astype(np.float32)
    else:
        raise ValueError(w.router)
    lg = logits.astype(np.float64)
    m = np.max(lg, axis=1, keepdims=True)
    ex = np.exp(lg - m)
    prob = ex / ex.sum(axis=1, keepdims=True)
    order = np.argsort(-lg, axis=1, kind="stable")[:, : w.k]
    idx = order.astype(np.int32)
    p = np.take_along_axis(prob, order, axis=1).astype(np.float32)
    return idx, p


def make_inputs(w: Workload, seed: int = 0, R_cap: int | None = None) -> dict:
    """All inputs of one forward + backward step as CPU torch tensors.

    x bf16 [T, H]; topk_idx int32 [T, k]; topk_prob f32 [T, k];
    W1 bf16 [E, N1, H] in logical order (rows [0, F) input, [F, 2F) gate);
    b1 bf16 [E, N1] or None; W2 bf16 [E, F, H] (y = a @ W2_e);
    dY bf16 [R_cap, H] (a gradient at the FC2 output, per permuted row, for
    calls that start there; rows that turn out to be padding are ignored);
    dOut bf16 [T, H] (the gradient arriving at the layer output)."""
    ss = np.random.SeedSequence(seed).spawn(7)
    sd = 1.0 / np.sqrt(w.H)
    out = {}
    out["x"] = _bf16(_normal(ss[0], (w.T, w.H)))
    idx, p = router_inputs(w, np.random.default_rng(ss[1]))
    out["topk_idx"] = torch.from_numpy(idx)
    out["topk_prob"] = torch.from_numpy(p)
    out["W1"] = _bf16(_normal(ss[2], (w.E, w.N1, w.H), sd))
    out["W2"] = _bf16(_normal(ss[3], (w.E, w.F, w.H), sd))
    out["b1"] = _bf16(_normal(ss[4], (w.E, w.N1), 0.02)) if w.bias else None
    out["dY"] = _bf16(_normal(ss[5], (R_cap or w.R_cap, w.H)))
    out["dOut"] = _bf16(_normal(ss[6], (w.T, w.H)))
    return out


def random_mxfp8(rows: int, cols: int, seed: int, scale_lo: int = 123, scale_hi: int = 125,
                 exp_lo: int = 5, exp_hi: int = 9):
    """Random MXFP8 operand: E4M3 codes with a random sign, exponent field in
    [exp_lo, exp_hi) (magnitudes 2^(exp_lo-7) .. 2^(exp_hi-7), never the NaN
    code) and random mantissa, plus E8M0 scales drawn from [scale_lo,
    scale_hi].  The defaults keep a K ~ 2000 contraction of two such
    operands near unit magnitude."""
    rng = np.random.default_rng(seed)
    sign = rng.integers(0, 2, size=(rows, cols), dtype=np.uint8) << 7
    ex = rng.integers(exp_lo, exp_hi, size=(rows, cols), dtype=np.uint8) << 3
    man = rng.integers(0, 8, size=(rows, cols), dtype=np.uint8)
    q = (sign | ex | man).astype(np.uint8)
    s = rng.integers(scale_lo, scale_hi + 1, size=(rows, cols // 32), dtype=np.uint8)
    return torch.from_numpy(q), torch.from_numpy(s)
