"""torch-facing wrappers of the C ABI: allocate outputs with torch (device
memory and streams only) and pass raw pointers to libmoeglu.  No step of the
method is computed here."""
from __future__ import annotations

import ctypes as C

import torch

from . import lib as L


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _s(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _dev(t):
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    return t.device


def new_status(device) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def read_status(status: torch.Tensor) -> int:
    out = C.c_int32(0)
    L.check(L.load().moe_get_status(_p(status), C.byref(out), _s()), "moe_get_status")
    return out.value


def wait_selftest(arrive: bool, device="cuda") -> tuple[int, int]:
    """Runs the bounded-wait self-test; returns (status word, ns waited)."""
    status = new_status(device)
    waited = torch.zeros(1, dtype=torch.int64, device=device)
    L.check(L.load().moe_wait_selftest(1 if arrive else 0, _p(status), _p(waited), _s()), "moe_wait_selftest")
    return read_status(status), int(waited.item())


def repack_fc1(W1: torch.Tensor, inverse: bool = False) -> torch.Tensor:
    """[E, 2F, H] logical input|gate rows <-> packed rows (bf16)."""
    lib = L.load()
    E, N1, H = W1.shape
    out = torch.empty_like(W1)
    L.check(lib.moe_repack_fc1(_p(W1), _p(out), E, N1 // 2, H, int(inverse), _s()), "moe_repack_fc1")
    return out


def route_permute(x, topk_idx, topk_prob, E: int, R_cap: int, expert_begin: int = 0, status=None,
                  with_col: bool = False) -> dict:
    """Routing + gather; with_col also returns the column-wise MXFP8 copy of
    x_perm made during the gather (x_qc [H, R_cap], x_sc [H, R_cap/32])."""
    lib = L.load()
    dev = _dev(x)
    T, H = x.shape
    k = topk_idx.shape[1]
    o = {
        "x_perm": torch.empty(R_cap, H, dtype=torch.bfloat16, device=dev),
        "row_of": torch.empty(T * k, dtype=torch.int32, device=dev),
        "tok_of": torch.empty(R_cap, dtype=torch.int32, device=dev),
        "prob_perm": torch.empty(R_cap, dtype=torch.float32, device=dev),
        "counts": torch.empty(E, dtype=torch.int32, device=dev),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
    }
    if with_col:
        o["x_qc"] = torch.zeros(H, R_cap, dtype=torch.uint8, device=dev)
        o["x_sc"] = torch.zeros(H, R_cap // 32, dtype=torch.uint8, device=dev)
    ws_bytes = lib.moe_route_workspace_size(T, k, E)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    st = status if status is not None else new_status(dev)
    L.check(lib.moe_route_permute(_p(x), _p(topk_idx), _p(topk_prob), T, H, k, expert_begin, E, R_cap,
                                  _p(o["x_perm"]), _p(o["row_of"]), _p(o["tok_of"]), _p(o["prob_perm"]),
                                  _p(o["counts"]), _p(o["offsets"]), _p(o.get("x_qc")), _p(o.get("x_sc")), _p(ws),
                                  ws_bytes, _p(st), _s()),
            "moe_route_permute")
    o["status"] = st
    return o


def _act_out(q_row=None, s_row=None, q_col=None, s_col=None, y=None, amax=None, pre=None) -> L.ActOut:
    return L.ActOut(*(None if t is None else t.data_ptr() for t in (q_row, s_row, q_col, s_col, y, amax, pre)))


def fc1_fwd(x_perm, W1p, counts, offsets, F: int, params: L.GluParams, out_mode: int = L.OUT_MXFP8,
            b1p=None, row_scale=None, save_pre: bool = True, with_col: bool = True, sm_margin: int = 0,
            status=None, out: dict | None = None, dynamic: bool = True) -> dict:
    """GroupGemm + Activation + Quantize/Transpose.  Returns the output tensors
    ({q_row, s_row, q_col, s_col} | {y[, amax]}, and pre when saved).
    dynamic=False runs the static tile schedule (no workspace)."""
    lib = L.load()
    dev = _dev(x_perm)
    R_cap, H = x_perm.shape
    E = counts.shape[0]
    gated = params.act in (L.ACT["swiglu"], L.ACT["geglu"], L.ACT["geglu_tanh"], L.ACT["sreglu"])
    N1 = 2 * F if gated else F
    o = out if out is not None else {}
    if params.act == L.ACT["none"]:
        o.setdefault("pre", torch.empty(R_cap, F, dtype=torch.bfloat16, device=dev))
    else:
        if out_mode == L.OUT_MXFP8:
            o.setdefault("q_row", torch.empty(R_cap, F, dtype=torch.uint8, device=dev))
            o.setdefault("s_row", torch.empty(R_cap, F // 32, dtype=torch.uint8, device=dev))
            if with_col:
                o.setdefault("q_col", torch.empty(F, R_cap, dtype=torch.uint8, device=dev))
                o.setdefault("s_col", torch.empty(F, R_cap // 32, dtype=torch.uint8, device=dev))
        else:
            o.setdefault("y", torch.empty(R_cap, F, dtype=torch.bfloat16, device=dev))
            if out_mode == L.OUT_NVFP4:
                o.setdefault("amax", torch.zeros(1, dtype=torch.float32, device=dev))
        if save_pre:
            o.setdefault("pre", torch.empty(R_cap, N1, dtype=torch.bfloat16, device=dev))
    st = status if status is not None else new_status(dev)
    ao = _act_out(o.get("q_row"), o.get("s_row"), o.get("q_col"), o.get("s_col"), o.get("y"), o.get("amax"),
                  o.get("pre"))
    ws_bytes = lib.moe_grouped_fc1_workspace_size(E, N1, R_cap) if dynamic else 0
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if dynamic else None
    L.check(lib.moe_grouped_fc1_glu_quant_fwd(_p(x_perm), _p(W1p), _p(b1p), _p(row_scale), _p(counts),
                                              _p(offsets), E, H, F, R_cap, C.byref(params), out_mode,
                                              C.byref(ao), _p(ws), ws_bytes, sm_margin, _p(st), _s()),
            "moe_grouped_fc1_glu_quant_fwd")
    o["status"] = st
    return o


def fc1_fwd_mxfp8(xq, xs, W1q, W1s, counts, offsets, F: int, params: L.GluParams, out_mode: int = L.OUT_MXFP8,
                  b1p=None, row_scale=None, save_pre: bool = True, with_col: bool = True, sm_margin: int = 0,
                  status=None) -> dict:
    """GroupGemm + Activation + Quantize/Transpose on MXFP8 operands: xq/xs
    [R_cap, H] (+ /32) the row-wise MXFP8 of x_perm, W1q/W1s [E, N1, H]
    (+ /32) the row-wise MXFP8 of the packed W1p.  Same outputs as fc1_fwd."""
    lib = L.load()
    dev = _dev(xq)
    R_cap, H = xq.shape
    E, N1, _ = W1q.shape
    o = {}
    if out_mode == L.OUT_MXFP8:
        o["q_row"] = torch.empty(R_cap, F, dtype=torch.uint8, device=dev)
        o["s_row"] = torch.empty(R_cap, F // 32, dtype=torch.uint8, device=dev)
        if with_col:
            o["q_col"] = torch.empty(F, R_cap, dtype=torch.uint8, device=dev)
            o["s_col"] = torch.empty(F, R_cap // 32, dtype=torch.uint8, device=dev)
    else:
        o["y"] = torch.empty(R_cap, F, dtype=torch.bfloat16, device=dev)
        if out_mode == L.OUT_NVFP4:
            o["amax"] = torch.zeros(1, dtype=torch.float32, device=dev)
    if save_pre:
        o["pre"] = torch.empty(R_cap, N1, dtype=torch.bfloat16, device=dev)
    st = status if status is not None else new_status(dev)
    ws_bytes = lib.moe_grouped_fc2_workspace_size(E, H, N1, R_cap)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ao = _act_out(o.get("q_row"), o.get("s_row"), o.get("q_col"), o.get("s_col"), o.get("y"), o.get("amax"),
                  o.get("pre"))
    L.check(lib.moe_grouped_fc1_glu_quant_fwd_mxfp8(_p(xq), _p(xs), _p(W1q), _p(W1s), _p(b1p), _p(row_scale),
                                                    _p(counts), _p(offsets), E, H, F, R_cap, C.byref(params),
                                                    out_mode, C.byref(ao), _p(ws), ws_bytes, sm_margin, _p(st),
                                                    _s()), "moe_grouped_fc1_glu_quant_fwd_mxfp8")
    o["status"] = st
    return o


def dglu_bwd(dY_perm, W2, pre, counts, offsets, F: int, params: L.GluParams, out_mode: int = L.OUT_MXFP8,
             row_scale=None, with_col: bool = True, sm_margin: int = 0, status=None,
             out: dict | None = None, row_dot: bool = False, rht_signs: int | None = None,
             dbias: bool = False, dynamic: bool = True) -> dict:
    """GroupGemm + dActivation + Quantize/Transpose.  dFC1 in packed order;
    row_dot=True also returns o["row_dot"], the per-row partials of the
    feature-scale gradient (reduce with feature_scale_grad).  NVFP4 mode
    returns y and amax (max |y|); with rht_signs (16-bit mask) also
    o["rht_amax"], the amax of y's transposed random Hadamard rotation.
    dbias=True also returns o["dbias"] [E, N1] f32, the FC1 bias gradient
    (packed column order)."""
    lib = L.load()
    dev = _dev(dY_perm)
    R_cap, H = dY_perm.shape
    E = counts.shape[0]
    N1 = pre.shape[1]
    o = out if out is not None else {}
    if out_mode == L.OUT_MXFP8:
        o.setdefault("q_row", torch.empty(R_cap, N1, dtype=torch.uint8, device=dev))
        o.setdefault("s_row", torch.empty(R_cap, N1 // 32, dtype=torch.uint8, device=dev))
        if with_col:
            o.setdefault("q_col", torch.empty(N1, R_cap, dtype=torch.uint8, device=dev))
            o.setdefault("s_col", torch.empty(N1, R_cap // 32, dtype=torch.uint8, device=dev))
    else:
        o.setdefault("y", torch.empty(R_cap, N1, dtype=torch.bfloat16, device=dev))
        if out_mode == L.OUT_NVFP4:
            o.setdefault("amax", torch.zeros(1, dtype=torch.float32, device=dev))
            if rht_signs is not None:
                o.setdefault("rht_amax", torch.zeros(1, dtype=torch.float32, device=dev))
    if row_dot:
        o.setdefault("row_dot", torch.empty(R_cap, lib.moe_dglu_row_dot_parts(F), dtype=torch.float32, device=dev))
    st = status if status is not None else new_status(dev)
    ao = _act_out(o.get("q_row"), o.get("s_row"), o.get("q_col"), o.get("s_col"), o.get("y"), o.get("amax"))
    ao.row_dot = o["row_dot"].data_ptr() if "row_dot" in o else None
    if "rht_amax" in o:
        ao.rht_amax, ao.rht_signs = o["rht_amax"].data_ptr(), int(rht_signs) & 0xFFFF
    ws_bytes, ws = 0, None
    if dbias:
        o.setdefault("dbias", torch.empty(E, N1, dtype=torch.float32, device=dev))
    if dbias or dynamic:
        ws_bytes = lib.moe_grouped_dglu_workspace_size(N1, R_cap) if dbias else lib.moe_grouped_dglu_workspace_size(0, 0)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    L.check(lib.moe_grouped_dglu_quant_bwd(_p(dY_perm), _p(W2), _p(pre), _p(row_scale), _p(counts), _p(offsets),
                                           E, H, F, R_cap, C.byref(params), out_mode, C.byref(ao), _p(o.get("dbias")),
                                           _p(ws), ws_bytes, sm_margin, _p(st), _s()),
            "moe_grouped_dglu_quant_bwd")
    o["status"] = st
    return o


def quantize_mxfp8(src, col: bool = False, counts=None, offsets=None, out=None, status=None, tiled: bool = False):
    """src [R, C] or [G, R, C] bf16 -> (q, s); col=True gives the transposed
    column-wise copy; tiled (with col) writes the scales in the tensor-core
    order of a GEMM weight operand (flat uint8 [moe_mxfp8_tiled_scale_bytes])."""
    lib = L.load()
    dev = _dev(src)
    s3 = src if src.dim() == 3 else src.unsqueeze(0)
    G, R, Cc = s3.shape
    if col and tiled:
        q = torch.empty(G, Cc, R, dtype=torch.uint8, device=dev) if out is None else out[0]
        s = (torch.empty(lib.moe_mxfp8_tiled_scale_bytes(G, R, Cc), dtype=torch.uint8, device=dev)
             if out is None else out[1])
        L.check(lib.moe_quantize_mxfp8(_p(s3), G, R, Cc, 2, None, None, 0, _p(q), _p(s), _p(status), _s()),
                "moe_quantize_mxfp8")
        return (q[0] if src.dim() == 2 and out is None else q), s
    if col:
        q = torch.empty(G, Cc, R, dtype=torch.uint8, device=dev) if out is None else out[0]
        s = torch.empty(G, Cc, R // 32, dtype=torch.uint8, device=dev) if out is None else out[1]
    else:
        q = torch.empty(G, R, Cc, dtype=torch.uint8, device=dev) if out is None else out[0]
        s = torch.empty(G, R, Cc // 32, dtype=torch.uint8, device=dev) if out is None else out[1]
    E = 0 if counts is None else counts.shape[0]
    L.check(lib.moe_quantize_mxfp8(_p(s3), G, R, Cc, int(col), _p(counts), _p(offsets), E, _p(q), _p(s),
                                   _p(status), _s()), "moe_quantize_mxfp8")
    if src.dim() == 2 and out is None:
        return q[0], s[0]
    return q, s


def quantize_mxfp8_dual(src, status=None):
    """src [G, R, C] (or [R, C]) bf16 read once -> (q_row [G, R, C],
    s_row [G, R, C/32], q_col [G, C, R], s_col [G, C, R/32])."""
    lib = L.load()
    dev = _dev(src)
    s3 = src if src.dim() == 3 else src.unsqueeze(0)
    G, R, Cc = s3.shape
    qr = torch.empty(G, R, Cc, dtype=torch.uint8, device=dev)
    sr = torch.empty(G, R, Cc // 32, dtype=torch.uint8, device=dev)
    qc = torch.empty(G, Cc, R, dtype=torch.uint8, device=dev)
    sc = torch.empty(G, Cc, R // 32, dtype=torch.uint8, device=dev)
    L.check(lib.moe_quantize_mxfp8_dual(_p(s3), G, R, Cc, _p(qr), _p(sr), _p(qc), _p(sc), _p(status), _s()),
            "moe_quantize_mxfp8_dual")
    return qr, sr, qc, sc


def fc2_fwd(Aq, As, Wq, Ws, counts, offsets, sm_margin: int = 0, status=None, out=None,
            out_mode: int = L.OUT_BF16, with_col: bool = True, w_tiled: bool = False):
    """GroupGemm (+ Quantize): y [R_cap, N] = A [R_cap, K] . W[e]^T per expert
    with W [E, N, K].  MXFP8 operands (codes Aq/Wq with E8M0 scales As/Ws),
    or bf16 operands when As and Ws are None.  out_mode OUT_BF16 returns the
    bf16 tensor y; OUT_MXFP8 returns {q_row, s_row[, q_col, s_col]};
    OUT_NVFP4 returns {y, amax}.  w_tiled: Ws is in the tensor-core order
    (quantize_mxfp8(..., col=True, tiled=True))."""
    lib = L.load()
    dev = _dev(Aq)
    R_cap, K = Aq.shape
    E, N, _ = Wq.shape
    if (As is None) != (Ws is None):
        raise ValueError("both operands bf16 (no scales) or both MXFP8")
    o = {}
    if out_mode == L.OUT_BF16:
        o["y"] = out if out is not None else torch.empty(R_cap, N, dtype=torch.bfloat16, device=dev)
    elif out_mode == L.OUT_MXFP8:
        o["q_row"] = torch.empty(R_cap, N, dtype=torch.uint8, device=dev)
        o["s_row"] = torch.empty(R_cap, N // 32, dtype=torch.uint8, device=dev)
        if with_col:
            o["q_col"] = torch.empty(N, R_cap, dtype=torch.uint8, device=dev)
            o["s_col"] = torch.empty(N, R_cap // 32, dtype=torch.uint8, device=dev)
    else:
        o["y"] = torch.empty(R_cap, N, dtype=torch.bfloat16, device=dev)
        o["amax"] = torch.zeros(1, dtype=torch.float32, device=dev)
    st = status if status is not None else new_status(dev)
    a_in = L.in_operand(Aq.data_ptr(), None if As is None else As.data_ptr())
    w_in = L.in_operand(Wq.data_ptr(), None if Ws is None else Ws.data_ptr(), tiled=w_tiled)
    ws_bytes = lib.moe_grouped_fc2_workspace_size(E, K, N, R_cap) if As is not None else 0
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    ao = _act_out(o.get("q_row"), o.get("s_row"), o.get("q_col"), o.get("s_col"), o.get("y"), o.get("amax"))
    L.check(lib.moe_grouped_fc2_fwd(C.byref(a_in), C.byref(w_in), _p(counts), _p(offsets), E, K, N, R_cap, out_mode,
                                    C.byref(ao), _p(ws), ws_bytes, sm_margin, _p(st), _s()), "moe_grouped_fc2_fwd")
    o["status"] = st
    return o["y"] if out_mode == L.OUT_BF16 else o


def fc2_fwd_nvfp4(Aq, As, sgA, Wq, Ws, sgW, counts, offsets, sm_margin: int = 0, status=None, out=None,
                  w_tiled: bool = False):
    """GroupGemm on NVFP4 operands: y [R_cap, N] bf16 = A . W[e]^T with
    A = packed E2M1 [R_cap, K/2] + E4M3 scales [R_cap, K/16] + per-tensor
    scale sgA (device float [1]), W [E, N, K/2] + [E, N, K/16] + sgW
    (w_tiled: Ws in the tensor-core order, nvfp4_cast_cols(..., tiled=True))."""
    lib = L.load()
    dev = _dev(Aq)
    R_cap, K2 = Aq.shape
    K = 2 * K2
    E, N, _ = Wq.shape
    y = out if out is not None else torch.empty(R_cap, N, dtype=torch.bfloat16, device=dev)
    st = status if status is not None else new_status(dev)
    a_in = L.in_operand(Aq.data_ptr(), As.data_ptr(), sgA.data_ptr())
    w_in = L.in_operand(Wq.data_ptr(), Ws.data_ptr(), sgW.data_ptr(), tiled=w_tiled)
    ws_bytes = lib.moe_grouped_fc2_workspace_size(E, K, N, R_cap)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ao = _act_out(y=y)
    L.check(lib.moe_grouped_fc2_fwd(C.byref(a_in), C.byref(w_in), _p(counts), _p(offsets), E, K, N, R_cap,
                                    L.OUT_BF16, C.byref(ao), _p(ws), ws_bytes, sm_margin, _p(st), _s()),
            "moe_grouped_fc2_fwd (NVFP4)")
    return y


def amax_bf16(x):
    """max |x| of a bf16 tensor as a device float [1]."""
    lib = L.load()
    a = torch.empty(1, dtype=torch.float32, device=_dev(x))
    L.check(lib.moe_amax_bf16(_p(x), x.numel(), _p(a), _s()), "moe_amax_bf16")
    return a


def nvfp4_cast_cols(src, amax, status=None, tiled: bool = False, out=None):
    """Column-wise NVFP4 of src [G, R, C] (or [R, C]) bf16: (q [G, C, R/2],
    s [G, C, R/16], s_global [1]); tiled: s in the tensor-core order of a
    GEMM weight operand (flat uint8 [moe_nvfp4_tiled_scale_bytes]).  out:
    optional (q, s, s_global) to write into."""
    lib = L.load()
    dev = _dev(src)
    s3 = src if src.dim() == 3 else src.unsqueeze(0)
    G, R, Cc = s3.shape
    if out is not None:
        q, s, sg = out
    else:
        q = torch.empty(G, Cc, R // 2, dtype=torch.uint8, device=dev)
        s = (torch.empty(lib.moe_nvfp4_tiled_scale_bytes(G, R, Cc), dtype=torch.uint8, device=dev) if tiled
             else torch.empty(G, Cc, R // 16, dtype=torch.uint8, device=dev))
        sg = torch.empty(1, dtype=torch.float32, device=dev)
    fn = lib.moe_nvfp4_cast_cols_tiled if tiled else lib.moe_nvfp4_cast_cols
    L.check(fn(_p(s3), G, R, Cc, _p(amax), _p(q), _p(s), _p(sg), _p(status), _s()),
            "moe_nvfp4_cast_cols_tiled" if tiled else "moe_nvfp4_cast_cols")
    return q, s, sg


def wgrad(Aq_col, As_col, Bq_col, Bs_col, counts, offsets, out_f32: bool = False, sm_margin: int = 0,
          status=None, out=None):
    """D [E, M, N] = per-expert contraction over the expert's rows of the
    column-wise MXFP8 copies A [M, R_cap] and B [N, R_cap]."""
    lib = L.load()
    dev = _dev(Aq_col)
    M, R_cap = Aq_col.shape
    N = Bq_col.shape[0]
    E = counts.shape[0]
    D = out if out is not None else torch.empty(E, M, N, dtype=torch.float32 if out_f32 else torch.bfloat16,
                                                device=dev)
    st = status if status is not None else new_status(dev)
    ws_bytes = lib.moe_grouped_wgrad_workspace_size(E, M, N, R_cap)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    L.check(lib.moe_grouped_wgrad(_p(Aq_col), _p(As_col), _p(Bq_col), _p(Bs_col), _p(counts), _p(offsets), E, M,
                                  N, R_cap, _p(D), int(out_f32), _p(ws), ws_bytes, sm_margin, _p(st), _s()),
            "moe_grouped_wgrad")
    return D


def rht_amax_cols(src, offsets, signs: int, status=None):
    """max |rotated value| of src [R_cap, C] (16-row Hadamard blocks below
    offsets[E]) as a device float [1]."""
    lib = L.load()
    R_cap, Cc = src.shape
    a = torch.empty(1, dtype=torch.float32, device=_dev(src))
    L.check(lib.moe_rht_amax_cols(_p(src), R_cap, Cc, _p(offsets), offsets.shape[0] - 1, int(signs) & 0xFFFF, _p(a),
                                  _p(status), _s()), "moe_rht_amax_cols")
    return a


def nvfp4_rht_cast_cols(src, offsets, amax, signs: int, status=None):
    """Rotated column-wise NVFP4 of src [R_cap, C]: (q [C, R_cap/2],
    s [C, R_cap/16], s_global [1])."""
    lib = L.load()
    dev = _dev(src)
    R_cap, Cc = src.shape
    q = torch.empty(Cc, R_cap // 2, dtype=torch.uint8, device=dev)
    s = torch.empty(Cc, R_cap // 16, dtype=torch.uint8, device=dev)
    sg = torch.empty(1, dtype=torch.float32, device=dev)
    L.check(lib.moe_nvfp4_rht_cast_cols(_p(src), R_cap, Cc, _p(offsets), offsets.shape[0] - 1, _p(amax),
                                        int(signs) & 0xFFFF, _p(q), _p(s), _p(sg), _p(status), _s()),
            "moe_nvfp4_rht_cast_cols")
    return q, s, sg


def wgrad_nvfp4(Aq, As, sgA, Bq, Bs, sgB, counts, offsets, out_f32: bool = False, sm_margin: int = 0, status=None):
    """D [E, M, N] = per-expert contraction over the expert's rows of the
    column-wise NVFP4 operands A [M, R_cap/2] and B [N, R_cap/2]."""
    lib = L.load()
    dev = _dev(Aq)
    M, R2 = Aq.shape
    R_cap = 2 * R2
    N = Bq.shape[0]
    E = counts.shape[0]
    D = torch.empty(E, M, N, dtype=torch.float32 if out_f32 else torch.bfloat16, device=dev)
    st = status if status is not None else new_status(dev)
    ws_bytes = lib.moe_grouped_wgrad_workspace_size(E, M, N, R_cap)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    L.check(lib.moe_grouped_wgrad_nvfp4(_p(Aq), _p(As), _p(sgA), _p(Bq), _p(Bs), _p(sgB), _p(counts), _p(offsets), E,
                                        M, N, R_cap, _p(D), int(out_f32), _p(ws), ws_bytes, sm_margin, _p(st), _s()),
            "moe_grouped_wgrad_nvfp4")
    return D


def unpermute_combine(y_perm, row_of, topk_prob, status=None, out=None):
    lib = L.load()
    dev = _dev(y_perm)
    T, k = topk_prob.shape
    H = y_perm.shape[1]
    o = out if out is not None else torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    L.check(lib.moe_unpermute_combine(_p(y_perm), _p(row_of), _p(topk_prob), T, H, k, _p(o), _p(status), _s()),
            "moe_unpermute_combine")
    return o


def combine_bwd(dout, y_perm, route: dict, k: int, status=None, out=None, col=None):
    """Gradient of the combine for dout [T, H]: (dY_perm [R_cap, H] bf16,
    dprob [T, k] f32); route = the dict of route_permute.  col = (q [H, R_cap],
    s [H, R_cap/32]) uint8 tensors: also the column-wise MXFP8 of dY_perm."""
    lib = L.load()
    dev = _dev(dout)
    T, H = dout.shape
    R_cap = y_perm.shape[0]
    E = route["counts"].shape[0]
    dY = out[0] if out is not None else torch.empty(R_cap, H, dtype=torch.bfloat16, device=dev)
    dprob = out[1] if out is not None else torch.empty(T, k, dtype=torch.float32, device=dev)
    st = status if status is not None else route.get("status")
    L.check(lib.moe_combine_bwd(_p(dout), _p(y_perm), _p(route["row_of"]), _p(route["tok_of"]),
                                _p(route["prob_perm"]), _p(route["offsets"]), T, H, k, E, R_cap, _p(dY),
                                _p(dprob), _p(col[0] if col else None), _p(col[1] if col else None), _p(st),
                                _s()), "moe_combine_bwd")
    return dY, dprob


def feature_scale_grad(row_dot, row_of, T: int, k: int, out=None):
    """dprob [T, k] f32 from the dGLU epilogue's per-row partials."""
    lib = L.load()
    o = out if out is not None else torch.empty(T, k, dtype=torch.float32, device=row_dot.device)
    L.check(lib.moe_feature_scale_grad(_p(row_dot), row_dot.shape[1], _p(row_of), T, k, _p(o), _s()),
            "moe_feature_scale_grad")
    return o


def permute_bwd(dx_perm, row_of, T: int, k: int, status=None, out=None):
    """Gradient of the permute: dx [T, H] bf16 from dx_perm [R_cap, H]."""
    lib = L.load()
    dev = _dev(dx_perm)
    H = dx_perm.shape[1]
    o = out if out is not None else torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    L.check(lib.moe_permute_bwd(_p(dx_perm), _p(row_of), T, H, k, _p(o), _p(status), _s()), "moe_permute_bwd")
    return o


def nvfp4_cast(y, amax, counts, offsets):
    lib = L.load()
    dev = _dev(y)
    R_cap, N = y.shape
    q = torch.empty(R_cap, N // 2, dtype=torch.uint8, device=dev)
    s = torch.empty(R_cap, N // 16, dtype=torch.uint8, device=dev)
    sg = torch.empty(1, dtype=torch.float32, device=dev)
    L.check(lib.moe_nvfp4_cast(_p(y), _p(amax), _p(counts), _p(offsets), counts.shape[0], N, R_cap, _p(q), _p(s),
                               _p(sg), _s()), "moe_nvfp4_cast")
    return q, s, sg


def glu_act(pre, counts, offsets, F: int, params: L.GluParams):
    lib = L.load()
    dev = _dev(pre)
    R_cap = pre.shape[0]
    y = torch.empty(R_cap, F, dtype=torch.bfloat16, device=dev)
    L.check(lib.moe_glu_act(_p(pre), _p(counts), _p(offsets), counts.shape[0], F, R_cap, C.byref(params), _p(y),
                            _s()), "moe_glu_act")
    return y


def dglu_act(da, pre, counts, offsets, F: int, params: L.GluParams):
    """Unfused backward activation: da [R, F] and pre [R, N1] -> dFC1 [R, N1]."""
    lib = L.load()
    dev = _dev(da)
    R_cap, N1 = pre.shape
    d = torch.empty(R_cap, N1, dtype=torch.bfloat16, device=dev)
    L.check(lib.moe_dglu_act(_p(da), _p(pre), _p(counts), _p(offsets), counts.shape[0], F, R_cap, C.byref(params),
                             _p(d), _s()), "moe_dglu_act")
    return d
