"""Comparison rules shared by the GPU parity tests.

  * integers (counts, offsets, permutation, tok_of): bit-exact;
  * bf16 outputs: |gpu - ref| <= 1e-2 + 2e-2 |ref| elementwise;
  * MXFP8: E8M0 scales equal, except that a scale may differ by one step
    where the block's amax lies within the accumulation-error band of a
    power of two (the GPU decides from its fp32 accumulator, the oracle
    from the float64 value rounded to float32; fp32 accumulation over K
    products is off by at most ~K * 2^-24 relative, so the band is
    REL_BAND = 1e-3, and such blocks must stay rare: <= 0.1%);
    dequantised elements within 1 E4M3 step on >= 99.9% of elements and
    within 4 steps everywhere (a wrong code, sign or scale breaks both);
  * outputs of a chain of kernels that re-quantise intermediate results
    (a whole layer step): both sides round their own intermediate values,
    which differ in the last fp32 bits, so a small fraction of intermediate
    MXFP8 codes land one step apart and each such flip moves a downstream
    sum by one E4M3 step (2^-3 relative) of one term.  The bf16 rule must
    hold on >= 99.9% of elements and every element must lie within 2% of
    the output's largest magnitude (a wrong tile, row or sign breaks both).
"""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import moe_oracle as O

REL_BAND = 1e-3


def np_(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.to(torch.float64)
    return t.numpy()


def assert_exact(gpu, ref, what=""):
    g, r = np.asarray(gpu), np.asarray(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    bad = np.nonzero(g != r)
    assert bad[0].size == 0, f"{what}: {bad[0].size} mismatches, first at {tuple(b[0] for b in bad)}: " \
                             f"{g[tuple(b[0] for b in bad)]} vs {r[tuple(b[0] for b in bad)]}"


def assert_bf16_close(gpu, ref, what="", rtol=2e-2, atol=1e-2):
    g, r = np.asarray(gpu, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    err = np.abs(g - r)
    lim = atol + rtol * np.abs(r)
    bad = err > lim
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst |d|={err.max():.4g} " \
                          f"at {np.unravel_index(np.argmax(err - lim), err.shape)}"


def _near_pow2(a: np.ndarray, band: float = REL_BAND) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        p2 = np.exp2(np.round(np.log2(a)))
        return (a > 0) & (np.abs(a - p2) <= band * p2)


def e4m3_step(x_scaled: np.ndarray) -> np.ndarray:
    """Spacing of E4M3 values at |x| (in block units)."""
    ax = np.abs(x_scaled)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.maximum(ax, 2.0 ** -6)))
    return np.exp2(e - 3)


def assert_mx_close(q_gpu, s_gpu, q_ref, s_ref, v_ref, what="", frac=0.999, rel_band=REL_BAND):
    """q [..., N] codes, s [..., N/32] scales, v_ref the oracle's float32
    values that were quantised (used for the amax band).  rel_band widens
    the power-of-two band when both sides round to bf16 before quantising
    (one bf16 step, 2^-7 relative)."""
    qg, sg = np.asarray(q_gpu), np.asarray(s_gpu).astype(np.int64)
    qr, sr = np.asarray(q_ref), np.asarray(s_ref).astype(np.int64)
    assert qg.shape == qr.shape and sg.shape == sr.shape, (what, qg.shape, qr.shape, sg.shape, sr.shape)
    v = np.asarray(v_ref, dtype=np.float32).reshape(*qr.shape[:-1], -1, 32).astype(np.float64)
    amax = np.abs(v).max(-1)
    diff = sg != sr
    if diff.any():
        ok = (np.abs(sg - sr) == 1) & _near_pow2(amax, rel_band)
        assert np.all(ok[diff]), f"{what}: scale mismatch off the power-of-two band: " \
                                 f"{np.sum(diff & ~ok)} blocks, e.g. gpu {sg[diff & ~ok][:4]} ref {sr[diff & ~ok][:4]} " \
                                 f"amax {amax[diff & ~ok][:4]}"
        # a block maximum falls in the band with probability ~ band / ln 2 (log-uniform
        # mantissas): 1.4e-3 for the accumulation band, 1.1e-2 for one bf16 step
        cap = max(1e-3, rel_band / math.log(2.0))
        assert diff.mean() <= cap, f"{what}: {diff.sum()} of {diff.size} scales differ"
    finite = (sr != 255)[..., None]
    dg = O.mx_dequantize(qg, sg.astype(np.uint8)).reshape(v.shape)
    dr = O.mx_dequantize(qr, sr.astype(np.uint8)).reshape(v.shape)
    S = np.exp2(np.maximum(sg, sr) - 127.0)[..., None]
    step = np.maximum(e4m3_step(dr / S), e4m3_step(dg / S)) * S
    err = np.abs(dg - dr)
    fin = np.broadcast_to(finite, err.shape)
    within1 = (err <= step * (1 + 1e-9)) | ~fin
    within4 = (err <= 4 * step * (1 + 1e-9)) | ~fin
    assert within4.all(), f"{what}: {np.sum(~within4)} elements beyond 4 E4M3 steps"
    assert within1.mean() >= frac, f"{what}: only {within1.mean():.5f} within 1 E4M3 step"


def assert_chain_close(gpu, ref, what="", frac=0.999, max_frac=0.02):
    g, r = np.asarray(gpu, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    err = np.abs(g - r)
    ok = err <= 1e-2 + 2e-2 * np.abs(r)
    assert ok.mean() >= frac, f"{what}: only {ok.mean():.5f} of elements within the bf16 rule"
    bound = max_frac * np.abs(r).max()
    assert err.max() <= bound, f"{what}: worst |d|={err.max():.4g} above {100 * max_frac:g}% of max |ref| ({bound:.4g})"


def untile_weight_scales(s_tiled, G: int, R: int, C: int) -> np.ndarray:
    """The plain column-wise scale layout [G][C][R/32] of scales written in
    the tensor-core order (moe_quantize_mxfp8 with col = 2): the 512 bytes of
    (128-row group of C, 128-element k-block of R) hold at byte 16 l + 4 j + i
    the scale of row 32 j + l of the group, sub-block i of the k-block."""
    nt, kbs = (C + 255) // 256, (R + 127) // 128
    t = np.asarray(s_tiled, dtype=np.uint8).reshape(G, nt, kbs, 2, 32, 4, 4)   # g, ntile, kb, half, l, j, i
    t = t.transpose(0, 1, 3, 5, 4, 2, 6).reshape(G, nt * 256, kbs * 4)          # g, c, sub-block
    return t[:, :C, : R // 32]


def untile_nvfp4_weight_scales(s_tiled, G: int, R: int, C: int) -> np.ndarray:
    """The plain column-wise NVFP4 scale layout [G][C][R/16] of scales written
    in the tensor-core order (moe_nvfp4_cast_cols_tiled): the 512 bytes of
    (256-column tile, 64-row group of R, 128-column half) hold at byte
    16 l + 4 j + i the scale of column 32 j + l of the half, 16-row sub-block
    i of the group."""
    nt, kgs = (C + 255) // 256, 4 * ((R + 255) // 256)
    t = np.asarray(s_tiled, dtype=np.uint8).reshape(G, nt, kgs, 2, 32, 4, 4)   # g, ntile, group, half, l, j, i
    t = t.transpose(0, 1, 3, 5, 4, 2, 6).reshape(G, nt * 256, kgs * 4)          # g, c, sub-block
    return t[:, :C, : R // 16]


def nvfp4_tiled_pad(s_tiled, G: int, R: int, C: int) -> np.ndarray:
    """The scale bytes of a tiled NVFP4 weight layout that lie past R or C
    (groups after the last row, columns after the last one), which the cast
    writes as zeros."""
    nt, kgs = (C + 255) // 256, 4 * ((R + 255) // 256)
    t = np.asarray(s_tiled, dtype=np.uint8).reshape(G, nt, kgs, 2, 32, 4, 4)
    t = t.transpose(0, 1, 3, 5, 4, 2, 6).reshape(G, nt * 256, kgs * 4)
    return np.concatenate([t[:, C:, :].ravel(), t[:, :C, R // 16:].ravel()])
