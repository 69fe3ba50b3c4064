"""CPU oracle for the fused MoE grouped GEMM + GLU + MXFP8/NVFP4 path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use it.  It shares no code, table or constant
generator with the CUDA library (``grouped_gemm_glu_gb300/csrc``), and it never
imports that package.

Every function is the plain definition of one step, written in float64 numpy
(a library matmul, sort or erf may serve as a step; there is no blocking,
fusion or reordering).  Where a quantised code is decided, the decision is
taken in float32, the precision of the kernel's accumulator, as the value
handed to the quantiser is a float32 on the GPU as well.

Sources (titles of the pages; sections named on them):
  [MoE-Fusion]  "Boosting MoE Training Throughput with Advanced Fusion Kernels"
                (NVIDIA technical blog, 2026-06-15, Spanish rewrite): sections
                "Optimizing GLU via fused GEMM epilogues" (Fig. 2),
                "Eliminating host-device synchronisation",
                "Fusing MXFP8 and NVFP4 quantisation".
  [MegaMoE]     hnwysp.cn article on the MegaMoE math model and DeepGEMM:
                §2.1 (routing and combine formula), §2.3 (FP8 formats and
                per-block scales), §4.3 (grouped GEMM on contiguous expert
                rows), §5.3 (tail rows).
Readings taken where the pages are silent are stated beside each function.

Parity status: every function below is pinned by tests/test_oracle_*.py
against closed forms, finite differences, library routines (torch, scipy),
hand-worked codec examples (tests/golden/) or brute force.  None is
"parity unpinned".
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# Rows of one expert's segment are padded to a multiple of ALIGN.  Reading:
# the pages do not give the padding; 32 is the MX block, so a column-wise MX
# block (32 consecutive permuted rows) never straddles two experts.
ALIGN = 32
MX_BLOCK = 32          # MXFP8 block size along the quantised dimension
NVFP4_BLOCK = 16       # NVFP4 block size


# ---------------------------------------------------------------------------
# Number formats.  [MegaMoE] §2.3: E4M3 = 1 sign, 4 exponent, 3 mantissa bits.
# OCP MX: a block of 32 values shares one power-of-two scale stored as E8M0.
# ---------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """E4M3 byte -> float64.  Bias 7; exponent field 0 is subnormal
    (m * 2^-9); 0x7F / 0xFF are NaN; there is no infinity."""
    c = np.asarray(codes, dtype=np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return s * mag


# the 127 non-negative finite E4M3 values, indexed by code 0x00..0x7E
_E4M3_POS = e4m3_decode(np.arange(0x7F))
E4M3_MAX = 448.0


def _nearest_even(x_abs: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the grid value nearest to x_abs (grid sorted ascending, index
    = code); a tie goes to the even code.  Values above the top of the grid
    saturate to it (the 'satfinite' rule)."""
    x_abs = np.minimum(x_abs, grid[-1])
    hi = np.searchsorted(grid, x_abs, side="left")          # grid[hi] >= x
    hi = np.clip(hi, 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    d_lo = x_abs - grid[lo]
    d_hi = grid[hi] - x_abs
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    return np.where(pick_hi, hi, lo)


def e4m3_encode(x) -> np.ndarray:
    """float -> E4M3 byte, round to nearest even, saturating to +-448
    (no overflow to NaN); NaN -> 0x7F.  The sign bit is kept for values that
    round to zero."""
    x = np.asarray(x, dtype=np.float64)
    code = _nearest_even(np.abs(np.nan_to_num(x, nan=0.0, posinf=E4M3_MAX, neginf=-E4M3_MAX)), _E4M3_POS)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


_E2M1_POS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_decode(codes) -> np.ndarray:
    """E2M1 nibble -> float64 (bit 3 = sign; magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6)."""
    c = np.asarray(codes, dtype=np.int64)
    return np.where(c & 0x8, -1.0, 1.0) * _E2M1_POS[c & 0x7]


def e2m1_encode(x) -> np.ndarray:
    """float -> E2M1 nibble, nearest even code, saturating to +-6."""
    x = np.asarray(x, dtype=np.float64)
    code = _nearest_even(np.abs(np.nan_to_num(x, nan=0.0)), _E2M1_POS)
    return (code | np.where(np.signbit(x), 0x8, 0)).astype(np.uint8)


def e8m0_decode(byte) -> np.ndarray:
    """E8M0 scale byte -> 2^(byte-127); 0xFF is NaN."""
    b = np.asarray(byte, dtype=np.float64)
    return np.where(b == 255, np.nan, np.exp2(b - 127.0))


def _floor_log2(a: np.ndarray) -> np.ndarray:
    """floor(log2 a) for finite a > 0, exact (frexp gives a = m 2^e, m in [.5,1))."""
    _, ex = np.frexp(a)
    return ex.astype(np.int64) - 1


def mx_scale_byte(amax_f32) -> np.ndarray:
    """E8M0 shared scale of one MX block from its float32 amax.

    OCP MX rule: shared exponent = floor(log2 amax) - emax(E4M3), emax = 8,
    clamped to the E8M0 range [-127, 127]; byte = exponent + 127.
    Reading: amax = 0 gives the clamp floor (byte 0x00, all elements 0);
    a block holding NaN or +-Inf gets byte 0xFF (NaN)."""
    a = np.asarray(amax_f32, dtype=np.float32).astype(np.float64)
    finite = np.isfinite(a)
    pos = finite & (a > 0)
    e = np.full(a.shape, -127, dtype=np.int64)
    e[pos] = _floor_log2(a[pos]) - 8
    e = np.clip(e, -127, 127)
    return np.where(finite, e + 127, 255).astype(np.uint8)


def mx_quantize_rows(v) -> tuple[np.ndarray, np.ndarray]:
    """MXFP8 (E4M3 + E8M0) quantisation along the last axis in blocks of 32.

    v: [..., N] (N % 32 == 0), converted to float32 first (the decision is
    taken in the kernel's precision).  Returns (codes uint8 [..., N],
    scales uint8 [..., N/32]).  Element = RNE_E4M3_satfinite(v * 2^-e); the
    multiply by a power of two is exact.  Elements of a NaN-scale block are
    0x7F."""
    v32 = np.asarray(v, dtype=np.float32)
    assert v32.shape[-1] % MX_BLOCK == 0
    blocks = v32.reshape(*v32.shape[:-1], v32.shape[-1] // MX_BLOCK, MX_BLOCK).astype(np.float64)
    with np.errstate(invalid="ignore"):
        amax = np.max(np.abs(blocks), axis=-1)
    amax = np.where(np.isnan(blocks).any(axis=-1), np.nan, amax)
    s = mx_scale_byte(amax)
    mult = np.exp2(127.0 - s.astype(np.float64))[..., None]
    with np.errstate(invalid="ignore", over="ignore"):
        q = e4m3_encode(blocks * mult)
    q = np.where((s == 255)[..., None], np.uint8(0x7F), q)
    return q.reshape(v32.shape), s


def mx_quantize_cols(v) -> tuple[np.ndarray, np.ndarray]:
    """Column-wise MXFP8 of v [R, N]: blocks of 32 consecutive rows of one
    column.  Returned transposed, the layout a GEMM that contracts over R
    reads: codes [N, R], scales [N, R/32]  ([MoE-Fusion], "Fusing MXFP8 and
    NVFP4 quantisation": the MXFP8 output plus a transposed copy)."""
    return mx_quantize_rows(np.asarray(v).T)


def mx_dequantize(q, s) -> np.ndarray:
    """codes [..., N], scales [..., N/32] -> float64 values."""
    q = np.asarray(q)
    vals = e4m3_decode(q).reshape(*q.shape[:-1], q.shape[-1] // MX_BLOCK, MX_BLOCK)
    return (vals * e8m0_decode(s)[..., None]).reshape(q.shape)


# NVFP4.  [MoE-Fusion], "Fusing MXFP8 and NVFP4 quantisation": for NVFP4 the
# forward kernel emits BF16 plus the per-tensor amax.  Reading of the cast
# that follows (the pages do not spell it out): the two-level NVFP4 recipe,
#   s_g = 448 * 6 / amax_tensor            (1 when amax_tensor == 0)
#   s_b = E4M3_RNE_sat(fp32(fp32(amax_b / 6) * s_g))      per block of 16
#   q   = E2M1_RNE_sat(fp32(v * fp32(s_g / s_b)))         (0 when s_b == 0)
#   v ~= q * s_b / s_g.
# Each step is one float32 operation in the order written, so that both
# sides decide the codes in the same precision.

def nvfp4_global_scale(amax_tensor) -> np.float32:
    a = np.float32(amax_tensor)
    if a == 0 or not np.isfinite(a):
        return np.float32(1.0)
    return np.float32(np.float32(448.0 * 6.0) / a)


def nvfp4_quantize_rows(v, s_g) -> tuple[np.ndarray, np.ndarray]:
    """v [R, N] (N % 16 == 0) -> (packed codes uint8 [R, N/2] with element 2i
    in the low nibble, block scales E4M3 uint8 [R, N/16])."""
    v32 = np.asarray(v, dtype=np.float32)
    R, N = v32.shape
    b = v32.reshape(R, N // NVFP4_BLOCK, NVFP4_BLOCK)
    amax_b = np.max(np.abs(b), axis=-1).astype(np.float32)
    sb_f = (amax_b / np.float32(6.0)).astype(np.float32)
    sb_f = (sb_f * np.float32(s_g)).astype(np.float32)
    sb_code = e4m3_encode(sb_f)
    sb_val = e4m3_decode(sb_code).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.where(sb_val > 0, np.float32(s_g) / np.where(sb_val > 0, sb_val, 1), 0).astype(np.float32)
    x = (b * inv[..., None]).astype(np.float32)
    q = e2m1_encode(x).reshape(R, N)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return packed, sb_code


def nvfp4_dequantize(packed, sb_code, s_g) -> np.ndarray:
    lo = packed & 0xF
    hi = packed >> 4
    q = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.uint8)
    q[:, 0::2] = lo
    q[:, 1::2] = hi
    vals = e2m1_decode(q).reshape(q.shape[0], -1, NVFP4_BLOCK)
    return (vals * (e4m3_decode(sb_code) / float(s_g))[..., None]).reshape(q.shape)


def nvfp4_quantize_cols(v, s_g) -> tuple[np.ndarray, np.ndarray]:
    """Column-wise NVFP4 of v [R, N] (R % 16 == 0): blocks of 16 consecutive
    rows of one column, under the per-tensor scale s_g.  Returned transposed,
    the K-major layout a GEMM contracting over R reads: packed codes
    [N, R/2] (element 2i in the low nibble) and E4M3 block scales [N, R/16]."""
    return nvfp4_quantize_rows(np.asarray(v, dtype=np.float32).T, s_g)


def grouped_gemm_nvfp4(Aq, As, sgA, Bq, Bs, sgB, rt: "Routing") -> np.ndarray:
    """Grouped GEMM on NVFP4 operands ([MoE-Fusion], "Fusing MXFP8 and NVFP4
    quantisation": the NVFP4 recipe, E2M1 values with an E4M3 scale per 16
    elements and a per-tensor float32 scale).  Each operand is dequantised
    (v = e2m1(q) * e4m3(s_b) / s_g, exact in float64) and multiplied:
    y[rows of e] = A[rows] @ B[e]^T for the expert's count rows, pad rows 0.
    Aq [R, K/2], As [R, K/16]; Bq [E, N, K/2], Bs [E, N, K/16]; returns the
    float32 value handed to the output rounding."""
    A = nvfp4_dequantize(np.asarray(Aq), np.asarray(As), sgA)
    B = np.stack([nvfp4_dequantize(np.asarray(Bq[e]), np.asarray(Bs[e]), sgB) for e in range(rt.E)])
    return grouped_gemm_rows(A, B, rt).astype(np.float32)


def bf16_round(x) -> np.ndarray:
    """float -> nearest bfloat16 (ties to even), via float32 (the kernel's
    value is a float32), returned as float64."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    r = np.where(nan, np.uint64(0x7FC00000), r).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Routing.  [MegaMoE] §2.1: y = sum_{i in topk} p_i E_i(x).  §4.3: tokens of
# one expert are laid out contiguously so that its rows form one GEMM problem.
# [MoE-Fusion], "Eliminating host-device synchronisation": the per-group token
# counts live in device memory.
# Readings: flat assignment index i = t*k + j; an expert's rows are ordered
# by ascending i (a stable counting sort); each segment is padded to ALIGN;
# assignments to experts outside [expert_begin, expert_begin + E) are
# dropped (row_of = -1).
# ---------------------------------------------------------------------------

@dataclass
class Routing:
    counts: np.ndarray       # int64 [E]
    offsets: np.ndarray      # int64 [E+1], padded exclusive prefix sum
    row_of: np.ndarray       # int64 [T*k], -1 if dropped
    tok_of: np.ndarray       # int64 [R_pad], -1 on pad rows
    slot_of: np.ndarray      # int64 [R_pad], flat index t*k+j, -1 on pad rows
    E: int = 0
    R_pad: int = 0
    expert_of_row: np.ndarray = field(default=None)  # int64 [R_pad]


def route(topk_idx, expert_begin: int, E: int, align: int = ALIGN) -> Routing:
    idx = np.asarray(topk_idx, dtype=np.int64)
    T, k = idx.shape
    e = idx.reshape(-1) - expert_begin
    local = (e >= 0) & (e < E)
    counts = np.bincount(e[local], minlength=E).astype(np.int64)
    padded = (counts + align - 1) // align * align
    offsets = np.concatenate([[0], np.cumsum(padded)]).astype(np.int64)
    R_pad = int(offsets[-1])
    # stable sort by expert (a library sort as one step); dropped entries last
    key = np.where(local, e, E)
    order = np.argsort(key, kind="stable")
    sorted_e = key[order]
    first = np.searchsorted(sorted_e, np.arange(E + 1), side="left")
    rank = np.arange(T * k) - first[sorted_e]
    row_of = np.full(T * k, -1, dtype=np.int64)
    keep = sorted_e < E
    row_of[order[keep]] = offsets[sorted_e[keep]] + rank[keep]
    tok_of = np.full(R_pad, -1, dtype=np.int64)
    slot_of = np.full(R_pad, -1, dtype=np.int64)
    flat = np.nonzero(row_of >= 0)[0]
    tok_of[row_of[flat]] = flat // k
    slot_of[row_of[flat]] = flat
    expert_of_row = np.repeat(np.arange(E), padded)
    return Routing(counts, offsets, row_of, tok_of, slot_of, E, R_pad, expert_of_row)


def permute(x, rt: Routing) -> np.ndarray:
    """x_perm[row] = x[tok_of[row]]; pad rows are zero.  [R_pad, H] float64."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros((rt.R_pad, x.shape[1]))
    real = rt.tok_of >= 0
    out[real] = x[rt.tok_of[real]]
    return out


def permute_probs(topk_prob, rt: Routing) -> np.ndarray:
    """prob_perm[row] = p[t, j] for the assignment (t, j) placed at that row
    (the router weight of [MegaMoE] §2.1 carried along with the permuted
    row, so that a per-row factor can be applied to it); pad rows 0.
    float64 [R_pad]."""
    p = np.asarray(topk_prob, dtype=np.float64).reshape(-1)
    out = np.zeros(rt.R_pad)
    real = rt.slot_of >= 0
    out[real] = p[rt.slot_of[real]]
    return out


def unpermute_combine(y_perm, row_of, topk_prob) -> np.ndarray:
    """[MegaMoE] §2.1: out[t] = sum_j p[t,j] * y_perm[row_of[t*k+j]] over the
    assignments kept on this shard (0 if none).  float64 [T, H]."""
    y = np.asarray(y_perm, dtype=np.float64)
    p = np.asarray(topk_prob, dtype=np.float64)
    T, k = p.shape
    r = np.asarray(row_of, dtype=np.int64).reshape(T, k)
    out = np.zeros((T, y.shape[1]))
    for j in range(k):
        ok = r[:, j] >= 0
        out[ok] += p[ok, j][:, None] * y[r[ok, j]]
    return out


def combine_bwd(dout, y_perm, row_of, topk_prob, R_rows: int) -> tuple[np.ndarray, np.ndarray]:
    """Gradient of the combine of [MegaMoE] §2.1 (out[t] = sum_j p[t,j] *
    y_perm[row_of[t*k+j]]) for an upstream gradient dout [T, H]; the chain
    rule on that sum, written out:
      dY_perm[row_of[t*k+j]] = p[t,j] * dout[t]          (float64 [R_rows, H];
                                                          rows no assignment
                                                          maps to stay 0)
      dprob[t, j]            = <dout[t], y_perm[row_of[t*k+j]]>  (0 if dropped)
    """
    g = np.asarray(dout, dtype=np.float64)
    y = np.asarray(y_perm, dtype=np.float64)
    p = np.asarray(topk_prob, dtype=np.float64)
    T, k = p.shape
    r = np.asarray(row_of, dtype=np.int64).reshape(T, k)
    dY = np.zeros((R_rows, g.shape[1]))
    dprob = np.zeros((T, k))
    for t in range(T):
        for j in range(k):
            row = r[t, j]
            if row < 0:
                continue
            dY[row] = p[t, j] * g[t]
            dprob[t, j] = float(np.dot(g[t], y[row]))
    return dY, dprob


def permute_bwd(dx_perm, row_of, T: int, k: int) -> np.ndarray:
    """Gradient of the permute (x_perm[row_of[t*k+j]] = x[t]): every token
    collects the gradients of the rows it was copied to, summed in j order.
    float64 [T, H]; 0 for a token with no local assignment."""
    d = np.asarray(dx_perm, dtype=np.float64)
    r = np.asarray(row_of, dtype=np.int64).reshape(T, k)
    dx = np.zeros((T, d.shape[1]))
    for j in range(k):
        ok = r[:, j] >= 0
        dx[ok] += d[r[ok, j]]
    return dx


# ---------------------------------------------------------------------------
# FC1 weight repack.  [MoE-Fusion], "Optimizing GLU via fused GEMM epilogues"
# (Fig. 2): the weights are repacked into input and gate columns so one
# thread block holds half a tile of input columns and half of gate columns.
# Logical W1 [E][2F][H]: rows [0, F) input, [F, 2F) gate.  Packed row p:
# block b = p // 2G, o = p % 2G; o < G -> input row b*G + o, else gate row
# F + b*G + (o - G).  Reading: granularity G (default 32) must divide F.
# ---------------------------------------------------------------------------

def packed_to_logical(F: int, G: int) -> np.ndarray:
    assert F % G == 0
    p = np.arange(2 * F)
    b, o = p // (2 * G), p % (2 * G)
    return np.where(o < G, b * G + o, F + b * G + (o - G))


def repack_fc1(W1, G: int = 32) -> np.ndarray:
    """W1 [..., 2F, H] (logical input|gate rows) -> packed rows."""
    W1 = np.asarray(W1)
    F = W1.shape[-2] // 2
    return W1[..., packed_to_logical(F, G), :]


def unpack_fc1(W1p, G: int = 32) -> np.ndarray:
    W1p = np.asarray(W1p)
    F = W1p.shape[-2] // 2
    out = np.empty_like(W1p)
    out[..., packed_to_logical(F, G), :] = W1p
    return out


# ---------------------------------------------------------------------------
# Activations.  [MoE-Fusion]: SwiGLU, GeGLU and sReLU, with clamping, feature
# scaling and bias.  The pages name them without formulas; these are the
# textbook definitions (readings):
#   SwiGLU  y = (u' + c) * g' * sigmoid(alpha g')      (alpha = 1, c = 0 plain)
#   GeGLU   y = (u' + c) * gelu(g'), gelu(z) = z Phi(z) (erf form; tanh form
#           as an option)
#   sReLU   y = max(x, 0)^2, not gated (FC1 width F)
#   sReGLU  y = (u' + c) * max(g', 0)^2 (gated variant)
# with g' = clamp(g, gate_lo, gate_hi), u' = clamp(u, up_lo, up_hi) and the
# clamp's derivative taken as 1 inside the closed interval, 0 outside.
# Feature scaling: an optional per-row factor s multiplies y.
# ---------------------------------------------------------------------------

ACT_SWIGLU, ACT_GEGLU, ACT_GEGLU_TANH, ACT_SRELU, ACT_SREGLU = 0, 1, 2, 3, 4
GATED = {ACT_SWIGLU: True, ACT_GEGLU: True, ACT_GEGLU_TANH: True, ACT_SRELU: False, ACT_SREGLU: True}


@dataclass
class ActParams:
    act: int = ACT_SWIGLU
    alpha: float = 1.0
    up_offset: float = 0.0
    gate_lo: float = -math.inf
    gate_hi: float = math.inf
    up_lo: float = -math.inf
    up_hi: float = math.inf


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def _phi_cdf(z):
    """Standard normal CDF, Phi(z) = erfc(-z / sqrt 2) / 2 (the same function
    as (1 + erf(z / sqrt 2)) / 2, written with erfc so that the negative tail
    keeps full relative precision instead of cancelling against 1)."""
    from scipy.special import erfc
    return 0.5 * erfc(-np.asarray(z, dtype=np.float64) / math.sqrt(2.0))


def _phi_pdf(z):
    return np.exp(-0.5 * z * z) / math.sqrt(2.0 * math.pi)


_K_TANH = math.sqrt(2.0 / math.pi)


def _gelu_tanh(z):
    return 0.5 * z * (1.0 + np.tanh(_K_TANH * (z + 0.044715 * z ** 3)))


def _gelu_tanh_grad(z):
    t = np.tanh(_K_TANH * (z + 0.044715 * z ** 3))
    return 0.5 * (1.0 + t) + 0.5 * z * (1.0 - t * t) * _K_TANH * (1.0 + 3 * 0.044715 * z * z)


def act_fwd(u, g, prm: ActParams):
    """u, g float64 arrays (bias already added).  For sReLU, g is ignored and
    u is the FC1 output."""
    u = np.asarray(u, dtype=np.float64)
    if prm.act == ACT_SRELU:
        return np.maximum(u, 0.0) ** 2
    g = np.asarray(g, dtype=np.float64)
    gc = np.clip(g, prm.gate_lo, prm.gate_hi)
    uc = np.clip(u, prm.up_lo, prm.up_hi) + prm.up_offset
    if prm.act == ACT_SWIGLU:
        return uc * gc * _sigmoid(prm.alpha * gc)
    if prm.act == ACT_GEGLU:
        return uc * gc * _phi_cdf(gc)
    if prm.act == ACT_GEGLU_TANH:
        return uc * _gelu_tanh(gc)
    if prm.act == ACT_SREGLU:
        return uc * np.maximum(gc, 0.0) ** 2
    raise ValueError(prm.act)


def act_bwd(u, g, dy, prm: ActParams):
    """Returns (du, dg) = (dy * dy/du, dy * dy/dg); dg is None for sReLU."""
    u = np.asarray(u, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    if prm.act == ACT_SRELU:
        return dy * 2.0 * np.maximum(u, 0.0), None
    g = np.asarray(g, dtype=np.float64)
    gc = np.clip(g, prm.gate_lo, prm.gate_hi)
    uc = np.clip(u, prm.up_lo, prm.up_hi) + prm.up_offset
    mg = ((g >= prm.gate_lo) & (g <= prm.gate_hi)).astype(np.float64)
    mu = ((u >= prm.up_lo) & (u <= prm.up_hi)).astype(np.float64)
    if prm.act == ACT_SWIGLU:
        s = _sigmoid(prm.alpha * gc)
        f, df = gc * s, s * (1.0 + prm.alpha * gc * (1.0 - s))
    elif prm.act == ACT_GEGLU:
        f, df = gc * _phi_cdf(gc), _phi_cdf(gc) + gc * _phi_pdf(gc)
    elif prm.act == ACT_GEGLU_TANH:
        f, df = _gelu_tanh(gc), _gelu_tanh_grad(gc)
    elif prm.act == ACT_SREGLU:
        f, df = np.maximum(gc, 0.0) ** 2, 2.0 * np.maximum(gc, 0.0)
    else:
        raise ValueError(prm.act)
    return dy * f * mu, dy * uc * df * mg


# ---------------------------------------------------------------------------
# Grouped GEMMs.  [MegaMoE] §4.3: one launch, one problem per expert, each
# expert's rows contiguous; §5.3: rows past an expert's count are masked.
# Plain definition per expert: C_e = A_e @ B_e^T (B stored with the
# contraction dimension last).  float64.
# ---------------------------------------------------------------------------

def grouped_gemm_rows(A, B, rt: Routing) -> np.ndarray:
    """A [R_pad, K], B [E, N, K] -> C [R_pad, N] with C[rows of e] = A[rows of
    e] @ B[e]^T for the count_e real rows; pad rows 0."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    C = np.zeros((rt.R_pad, B.shape[1]))
    for e in range(rt.E):
        r0, n = int(rt.offsets[e]), int(rt.counts[e])
        if n:
            C[r0:r0 + n] = A[r0:r0 + n] @ B[e].T
    return C


def unpack_glu_cols(pre, G: int = 32):
    """pre [R, 2F] in packed column order -> (u, g) each [R, F] logical."""
    pre = np.asarray(pre)
    F = pre.shape[1] // 2
    log = packed_to_logical(F, G)
    u = np.empty((pre.shape[0], F), dtype=pre.dtype)
    g = np.empty_like(u)
    is_in = log < F
    u[:, log[is_in]] = pre[:, is_in]
    g[:, log[~is_in] - F] = pre[:, ~is_in]
    return u, g


def pack_glu_cols(du, dg, G: int = 32):
    """(du, dg) each [R, F] -> [R, 2F] in packed column order."""
    F = du.shape[1]
    log = packed_to_logical(F, G)
    full = np.concatenate([du, dg], axis=1)
    return full[:, log]


@dataclass
class Fc1Out:
    pre_bf16: np.ndarray     # [R_pad, N1] packed order, bf16 values (float64)
    y: np.ndarray            # [R_pad, F]  float32 activation values
    q_row: np.ndarray = None
    s_row: np.ndarray = None
    q_col: np.ndarray = None
    s_col: np.ndarray = None
    amax: float = 0.0


def fc1_glu_fwd(x_perm, W1p, b1p, rt: Routing, prm: ActParams, G: int = 32,
                row_scale=None) -> Fc1Out:
    """GroupGemm + Activation + Quantize/Transpose ([MoE-Fusion], kernel
    family; "Optimizing GLU via fused GEMM epilogues").

    pre = x_perm @ W1p_e^T + b1p_e (float64), saved as bf16; activation on
    the unrounded pre-activation; y rounded to float32 (the kernel's
    precision); pad rows 0.  Quantised outputs are derived by the caller with
    mx_quantize_rows / mx_quantize_cols / NVFP4 from ``y``."""
    pre = grouped_gemm_rows(x_perm, W1p, rt)
    if b1p is not None:
        b = np.asarray(b1p, dtype=np.float64)
        for e in range(rt.E):
            r0, n = int(rt.offsets[e]), int(rt.counts[e])
            pre[r0:r0 + n] += b[e][None, :]
    if GATED[prm.act]:
        u, g = unpack_glu_cols(pre, G)
        y = act_fwd(u, g, prm)
    else:
        y = act_fwd(pre, None, prm)
    if row_scale is not None:
        y = y * np.asarray(row_scale, dtype=np.float64)[:, None]
    y = _zero_pad_rows(y, rt)
    pre = _zero_pad_rows(pre, rt)
    return Fc1Out(pre_bf16=bf16_round(pre), y=y.astype(np.float32), amax=float(np.max(np.abs(y.astype(np.float32)), initial=0.0)))


def _zero_pad_rows(M, rt: Routing):
    M = np.array(M, dtype=np.float64, copy=True)
    M[rt.tok_of < 0] = 0.0
    return M


def dglu_bwd(dY_perm, W2, pre_bf16, rt: Routing, prm: ActParams, G: int = 32,
             row_scale=None) -> np.ndarray:
    """GroupGemm + dActivation ([MoE-Fusion]: in the backward the epilogue
    reads the GEMM output, computes dSwiGLU, quantises and writes).

    da = dY_perm @ W2_e^T with W2 [E, F, H]; the saved bf16 pre-activation
    gives (u, g); returns dFC1 [R_pad, N1] float32 in packed column order
    (quantise it with mx_quantize_rows / mx_quantize_cols)."""
    da = grouped_gemm_rows(dY_perm, W2, rt)
    if row_scale is not None:
        da = da * np.asarray(row_scale, dtype=np.float64)[:, None]
    pre = np.asarray(pre_bf16, dtype=np.float64)
    if GATED[prm.act]:
        u, g = unpack_glu_cols(pre, G)
        du, dg = act_bwd(u, g, da, prm)
        d = pack_glu_cols(du, dg, G)
    else:
        d, _ = act_bwd(pre, None, da, prm)
    return _zero_pad_rows(d, rt).astype(np.float32)


def dglu_row_prob_grad(dY_perm, W2, pre_bf16, rt: Routing, prm: ActParams, G: int = 32) -> np.ndarray:
    """Gradient of the per-row "feature scaling" factor ([MoE-Fusion],
    "clamping and scaling"; reading: the router probability p multiplied into
    the FC1 output, a = p * act(pre)): dL/dp[r] = sum_c da[r, c] * act(pre)[r, c]
    with da = dY_perm @ W2_e^T, the activation taken on the saved bf16 pre.
    float64 [R_pad]; pad rows 0."""
    da = grouped_gemm_rows(dY_perm, W2, rt)
    pre = np.asarray(pre_bf16, dtype=np.float64)
    if GATED[prm.act]:
        u, g = unpack_glu_cols(pre, G)
        act = act_fwd(u, g, prm)
    else:
        act = act_fwd(pre, None, prm)
    out = np.sum(da * act, axis=1)
    out[rt.tok_of < 0] = 0.0
    return out


def fc1_bias_grad(dfc1, rt: Routing) -> np.ndarray:
    """Gradient of the FC1 bias ([MoE-Fusion], "clamping and scaling": the
    GLU's bias vector b_e added to every row of expert e; the chain rule on
    pre = x_perm W1p_e^T + b1p_e): dbias[e] = sum over the expert's rows of
    dL/dpre = dFC1 (the values before any quantisation; pad rows hold 0).
    dfc1 [R_pad, N1] -> float64 [E, N1], in dfc1's column order."""
    d = np.asarray(dfc1, dtype=np.float64)
    out = np.zeros((rt.E, d.shape[1]))
    for e in range(rt.E):
        r0, n = int(rt.offsets[e]), int(rt.counts[e])
        out[e] = d[r0:r0 + n].sum(axis=0)
    return out


def grouped_gemm_quant_fwd(A, B, rt: Routing) -> np.ndarray:
    """GroupGemm + Quantize ([MoE-Fusion], the first kernel of the fused
    family: a grouped GEMM whose output is quantised in its epilogue).
    y = A_e @ B_e^T per expert (pad rows 0) as handed to the quantiser: the
    float32 value of the accumulator (quantise with mx_quantize_rows /
    mx_quantize_cols; the bf16 output mode is bf16_round of the same y)."""
    return grouped_gemm_rows(A, B, rt).astype(np.float32)


def rows_to_slots(row_values, row_of, T: int, k: int) -> np.ndarray:
    """[T, k]: the value of the row each (token, slot) was routed to; 0 for
    dropped slots."""
    v = np.asarray(row_values, dtype=np.float64)
    r = np.asarray(row_of, dtype=np.int64).reshape(T, k)
    out = np.zeros((T, k))
    ok = r >= 0
    out[ok] = v[r[ok]]
    return out


def grouped_wgrad(A_col, B_col, rt: Routing) -> np.ndarray:
    """Weight gradient per expert, contraction over that expert's padded row
    segment: D_e = A_col[:, seg_e] @ B_col[:, seg_e]^T.  A_col [M, R_pad],
    B_col [N, R_pad] -> [E, M, N] float64 (pad rows are zero in the inputs)."""
    A = np.asarray(A_col, dtype=np.float64)
    B = np.asarray(B_col, dtype=np.float64)
    out = np.zeros((rt.E, A.shape[0], B.shape[0]))
    for e in range(rt.E):
        r0, r1 = int(rt.offsets[e]), int(rt.offsets[e + 1])
        if r1 > r0:
            out[e] = A[:, r0:r1] @ B[:, r0:r1].T
    return out


# ---------------------------------------------------------------------------
# NVFP4 backward.  [MoE-Fusion], "Fusing MXFP8 and NVFP4 quantisation": for
# NVFP4 the backward kernel also computes the amax of the transposed Hadamard
# rotation of its output, which removes the separate pass over the tensor
# that this per-tensor amax would otherwise need.
# Readings (the page gives neither the size of the transform nor its signs):
#  - the rotation acts along the rows of the output (the token dimension,
#    which is the contraction dimension of the weight-gradient GEMM that reads
#    the transposed tensor) on blocks of 16 consecutive rows; expert segments
#    are padded to 32 rows, so no block straddles two experts;
#  - it is the orthonormal random Hadamard transform H16 diag(s) / 4 with H16
#    the 16 x 16 Sylvester-Hadamard matrix (H[i][j] = (-1)^popcount(i & j))
#    and s 16 random signs drawn by the caller and passed in (bit i of
#    `sign_mask` set: s_i = -1);
#  - it is applied to the bf16 tensor the kernel writes (what a separate pass
#    would read); pad rows are zero.
# The amax does not depend on the row order of H16.
# ---------------------------------------------------------------------------
RHT_BLOCK = 16


def hadamard16() -> np.ndarray:
    """H16[i][j] = (-1)^popcount(i & j) (Sylvester order), float64."""
    i = np.arange(RHT_BLOCK)
    ones = np.array([[bin(int(a) & int(b)).count("1") for b in i] for a in i])
    return np.where(ones % 2 == 0, 1.0, -1.0)


def rht_signs(sign_mask: int) -> np.ndarray:
    """The diagonal s of the rotation: -1 where bit i of the mask is set."""
    return np.array([-1.0 if (int(sign_mask) >> i) & 1 else 1.0 for i in range(RHT_BLOCK)])


def rht_transposed(y, sign_mask: int) -> np.ndarray:
    """Z [R, C] with Z[16b:16b+16, c] = H16 diag(s) bf16(y)[16b:16b+16, c] / 4
    for every 16-row block b and column c (R % 16 == 0), float64."""
    Y = bf16_round(y)
    R, C = Y.shape
    if R % RHT_BLOCK:
        raise ValueError("rows must be a multiple of 16")
    M = hadamard16() * rht_signs(sign_mask)[None, :] / 4.0
    Z = np.einsum("ij,bjc->bic", M, Y.reshape(R // RHT_BLOCK, RHT_BLOCK, C))
    return Z.reshape(R, C)


def nvfp4_rht_cast_cols(y, sign_mask: int, s_g) -> tuple[np.ndarray, np.ndarray]:
    """NVFP4 operand of the weight-gradient GEMM ([MoE-Fusion], "Fusing MXFP8
    and NVFP4 quantisation": the backward's NVFP4 operands are the transposed
    tensors after a random Hadamard rotation): y [R, C] is rotated along its
    rows (rht_transposed: 16-row blocks, H16 diag(s) / 4 on the bf16 values)
    and cast column-wise to NVFP4 under s_g, whose blocks of 16 rows are the
    rotation's blocks.  Returns codes [C, R/2] and scales [C, R/16]."""
    return nvfp4_quantize_cols(rht_transposed(y, sign_mask), s_g)


def grouped_wgrad_nvfp4(Aq, As, sgA, Bq, Bs, sgB, rt: "Routing") -> np.ndarray:
    """Weight gradient on column-wise NVFP4 operands: each operand [M, R/2] /
    [M, R/16] is dequantised (e2m1 * s_b / s_g) and D_e = A[:, seg_e] @
    B[:, seg_e]^T over the expert's padded row segment (grouped_wgrad).
    float64 [E, M, N]."""
    A = nvfp4_dequantize(np.asarray(Aq), np.asarray(As), sgA)
    B = nvfp4_dequantize(np.asarray(Bq), np.asarray(Bs), sgB)
    return grouped_wgrad(A, B, rt)


def rht_transposed_amax(y, sign_mask: int) -> float:
    """Per-tensor amax of the rotated transposed output (0 for an empty tensor)."""
    Z = rht_transposed(y, sign_mask)
    return float(np.max(np.abs(Z))) if Z.size else 0.0
