"""One MoE MLP layer step (forward + backward) as a fixed sequence of C-ABI
calls over preallocated device buffers.  Nothing here reads device data on
the host, so the whole step captures into one CUDA graph.

Forward:  route+permute -> FC1 GroupGemm+Activation+Quantize/Transpose
          -> MXFP8 cast of W2 -> FC2 block-scaled GroupGemm -> unpermute+combine
Backward: (from dOut, the gradient at the layer output)
          combine backward (dY_perm = p * dOut[tok], dprob = <dOut, y_perm>)
          -> FC2-data-grad GroupGemm+dActivation+Quantize/Transpose (dFC1)
          -> MXFP8 cast of W1p (transposed) -> dX_perm = dFC1 . W1p
          -> column-wise MXFP8 of x_perm and dY_perm
          -> weight gradients dW1p = dFC1^T x, dW2 = a^T dY (per expert),
             and the FC1 bias gradient db1 (per expert column sums of dFC1)
          -> permute backward (dx[t] = sum of its rows of dX_perm)

Weight layouts: W1 [E][2F][H] (rows: input | gate; repacked once into W1p),
W2 [E][F][H] (y = a . W2[e]); gradients come out in the same layouts
(dW1 in packed row order).
"""
from __future__ import annotations

import ctypes as C

import torch

from . import lib as L
from .ops import _p, _s


class MoeLayer:
    def __init__(self, W1, W2, T: int, k: int, R_cap: int, params: L.GluParams, b1=None,
                 expert_begin: int = 0, sm_margin: int = 0, gated: bool = True, dynamic: bool = True,
                 nvfp4: bool = False, rht_signs: int = 0x6A5D, fused_col_casts: bool = True,
                 fc1_mxfp8: bool = False):
        """dynamic: the bf16 grouped GEMMs take their tiles from the dynamic
        scheduler (each call site has its own counter workspace); False runs
        the static schedule.  nvfp4: the step runs the NVFP4 recipe.  Forward:
        FC1 epilogue in NVFP4 mode (bf16 + amax) -> NVFP4 casts of its output
        and of W2 -> NVFP4 FC2.  Backward: the dGLU epilogue in NVFP4 mode (bf16
        dFC1, its amax and the amax of its transposed random Hadamard rotation
        with the 16 signs rht_signs) -> NVFP4 dFC1 and W1 (along 2F) -> NVFP4
        dX; the weight gradients on the rotated column-wise NVFP4 casts of
        dFC1, x, the FC1 output and dY (the same signs on both operands of a
        product, so the rotation cancels).  fused_col_casts (MXFP8 recipe):
        the column-wise MXFP8 copies of x_perm and dY_perm that the weight
        gradients read are made by the gather and by the combine backward
        themselves; False runs them as separate quantize calls.  fc1_mxfp8
        (MXFP8 recipe): FC1 contracts MXFP8 x_perm (row-wise cast after the
        gather) with MXFP8 W1, whose two copies (along H for FC1, along 2F for
        the data gradient) come from one read of W1 in the forward; the
        backward then has no W1 cast of its own."""
        self.lib = L.load()
        dev = W1.device
        self.dev = dev
        E, N1, H = W1.shape
        F = W2.shape[1]
        self.E, self.N1, self.H, self.F, self.T, self.k, self.R_cap = E, N1, H, F, T, k, R_cap
        self.params = params
        self.expert_begin = expert_begin
        self.sm_margin = sm_margin
        self.gated = gated
        self.W2 = W2
        u8, bf = torch.uint8, torch.bfloat16
        z = lambda *s, dt=bf: torch.empty(*s, dtype=dt, device=dev)
        if gated:
            self.W1p = z(E, N1, H)
            L.check(self.lib.moe_repack_fc1(_p(W1), _p(self.W1p), E, F, H, 0, _s()), "repack")
            self.b1p = None
            if b1 is not None:
                self.b1p = z(E, N1)
                L.check(self.lib.moe_repack_fc1(_p(b1), _p(self.b1p), E, F, 1, 0, _s()), "repack bias")
        else:
            self.W1p, self.b1p = W1, b1
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        # routing
        self.x_perm = z(R_cap, H)
        self.row_of = z(T * k, dt=torch.int32)
        self.tok_of = z(R_cap, dt=torch.int32)
        self.prob_perm = z(R_cap, dt=torch.float32)
        self.counts = z(E, dt=torch.int32)
        self.offsets = z(E + 1, dt=torch.int32)
        self.ws_bytes = self.lib.moe_route_workspace_size(T, k, E)
        self.ws = z(self.ws_bytes, dt=u8)
        # forward
        self.a_q, self.a_s = z(R_cap, F, dt=u8), z(R_cap, F // 32, dt=u8)
        self.a_qc, self.a_sc = z(F, R_cap, dt=u8), z(F, R_cap // 32, dt=u8)
        self.pre = z(R_cap, N1)
        # weight copies for FC2 / dX (MXFP8, transposed), scales in the tensor-core order
        self.W2q = z(E, H, F, dt=u8)
        self.W2s = z(self.lib.moe_mxfp8_tiled_scale_bytes(E, F, H), dt=u8)
        self.y_perm = z(R_cap, H)
        self.out = z(T, H)
        # backward
        self.d_q, self.d_s = z(R_cap, N1, dt=u8), z(R_cap, N1 // 32, dt=u8)
        self.d_qc, self.d_sc = z(N1, R_cap, dt=u8), z(N1, R_cap // 32, dt=u8)
        self.W1q = z(E, H, N1, dt=u8)
        self.W1s = z(self.lib.moe_mxfp8_tiled_scale_bytes(E, N1, H), dt=u8)
        self.dY_perm = z(R_cap, H)
        self.dprob = z(T, k, dt=torch.float32)
        self.dX_perm = z(R_cap, H)
        self.dx = z(T, H)
        self.x_qc, self.x_sc = z(H, R_cap, dt=u8), z(H, R_cap // 32, dt=u8)
        self.dy_qc, self.dy_sc = z(H, R_cap, dt=u8), z(H, R_cap // 32, dt=u8)
        self.dW1 = z(E, N1, H)
        self.dW2 = z(E, F, H)
        # scale re-tiling workspaces of the block-scaled GEMMs (one per call
        # site, so that no two calls of one step share one)
        lib = self.lib
        ws = lambda n: z(max(n, 256), dt=u8)
        self.ws_fc2 = ws(lib.moe_grouped_fc2_workspace_size(E, F, H, R_cap))
        self.ws_dx = ws(lib.moe_grouped_fc2_workspace_size(E, N1, H, R_cap))
        self.ws_wg1 = ws(lib.moe_grouped_wgrad_workspace_size(E, N1, H, R_cap))
        self.ws_wg2 = ws(lib.moe_grouped_wgrad_workspace_size(E, F, H, R_cap))
        # scheduler counters of the bf16 GEMMs, and the FC1 bias gradient
        # (packed order, like b1p) with its partial sums when the layer has a bias
        self.ws_fc1 = self.ws_fc1u = None
        self.ws_fc1_bytes = 0
        self.db1, self.ws_db, self.ws_db_bytes = None, None, 0
        if dynamic:
            self.ws_fc1_bytes = lib.moe_grouped_fc1_workspace_size(E, N1, R_cap)
            self.ws_fc1, self.ws_fc1u = z(self.ws_fc1_bytes, dt=u8), z(self.ws_fc1_bytes, dt=u8)
            self.ws_db_bytes = lib.moe_grouped_dglu_workspace_size(0, 0)
        if self.b1p is not None:
            self.db1 = z(E, N1, dt=torch.float32)
            self.ws_db_bytes = lib.moe_grouped_dglu_workspace_size(N1, R_cap)
        if self.ws_db_bytes:
            self.ws_db = z(self.ws_db_bytes, dt=u8)
        self.nvfp4 = nvfp4
        self.fused_cols = fused_col_casts and not nvfp4
        self.fc1_mxfp8 = fc1_mxfp8 and not nvfp4
        if self.fc1_mxfp8:
            self.x_qr, self.x_sr = z(R_cap, H, dt=u8), z(R_cap, H // 32, dt=u8)
            self.W1qr, self.W1sr = z(E, N1, H, dt=u8), z(E, N1, H // 32, dt=u8)
            self.W1s_p = z(E, H, N1 // 32, dt=u8)  # the dual cast's column scales (plain layout)
            self.ws_fc1mx = ws(lib.moe_grouped_fc2_workspace_size(E, H, N1, R_cap))
        if nvfp4:
            f32 = torch.float32
            self.a_y, self.a_amax = z(R_cap, F), z(1, dt=f32)
            self.a_q4, self.a_s4, self.a_sg = z(R_cap, F // 2, dt=u8), z(R_cap, F // 16, dt=u8), z(1, dt=f32)
            self.w2_amax = z(1, dt=f32)
            # weight casts write their scales in the tensor-core order when the
            # staged cast takes the shapes (F % 128 == 0, H % 8 == 0)
            self.w4_tiled = F % 128 == 0 and H % 8 == 0
            w4s = (lambda R_, C_: z(lib.moe_nvfp4_tiled_scale_bytes(E, R_, C_), dt=u8)) if self.w4_tiled else \
                (lambda R_, C_: z(E, C_, R_ // 16, dt=u8))
            self.cast_w4 = lib.moe_nvfp4_cast_cols_tiled if self.w4_tiled else lib.moe_nvfp4_cast_cols
            self.W2q4, self.W2s4, self.w2_sg = z(E, H, F // 2, dt=u8), w4s(F, H), z(1, dt=f32)
            self.fc1_out4 = L.ActOut(None, None, None, None, self.a_y.data_ptr(), self.a_amax.data_ptr(),
                                     self.pre.data_ptr())
            self.fc2_a4 = L.in_operand(self.a_q4.data_ptr(), self.a_s4.data_ptr(), self.a_sg.data_ptr())
            self.fc2_w4 = L.in_operand(self.W2q4.data_ptr(), self.W2s4.data_ptr(), self.w2_sg.data_ptr(),
                                       tiled=self.w4_tiled)
            # backward: bf16 dFC1 with its amaxes; NVFP4 rows of dFC1 and W1 (along 2F) for dX;
            # rotated column-wise NVFP4 of dFC1, x, a and dY for the weight gradients
            self.rht_signs = int(rht_signs) & 0xFFFF
            one = lambda: z(1, dt=f32)
            self.d_y, self.d_amax, self.d_rht = z(R_cap, N1), one(), one()
            self.d_q4, self.d_s4, self.d_sg = z(R_cap, N1 // 2, dt=u8), z(R_cap, N1 // 16, dt=u8), one()
            self.w1_amax, self.w1_sg = one(), one()
            self.W1q4, self.W1s4 = z(E, H, N1 // 2, dt=u8), w4s(N1, H)
            rot = lambda C_: (z(C_, R_cap // 2, dt=u8), z(C_, R_cap // 16, dt=u8), one(), one())
            self.d_rq, self.d_rs, self.d_rsg, _ = rot(N1)
            self.x_rq, self.x_rs, self.x_rsg, self.x_ramax = rot(H)
            self.dy_rq, self.dy_rs, self.dy_rsg, self.dy_ramax = rot(H)
            self.a_rq, self.a_rs, self.a_rsg, self.a_ramax = rot(F)
            self.bwd_out4 = L.ActOut(None, None, None, None, self.d_y.data_ptr(), self.d_amax.data_ptr(), None,
                                     None, self.d_rht.data_ptr(), self.rht_signs)
            self.dx_a4 = L.in_operand(self.d_q4.data_ptr(), self.d_s4.data_ptr(), self.d_sg.data_ptr())
            self.dx_w4 = L.in_operand(self.W1q4.data_ptr(), self.W1s4.data_ptr(), self.w1_sg.data_ptr(),
                                      tiled=self.w4_tiled)
        # operands and outputs of the two block-scaled M-grouped GEMMs
        self.fc2_a = L.in_operand(self.a_q.data_ptr(), self.a_s.data_ptr())
        self.fc2_w = L.in_operand(self.W2q.data_ptr(), self.W2s.data_ptr(), tiled=True)
        self.fc2_out = L.ActOut(None, None, None, None, self.y_perm.data_ptr(), None, None)
        self.dx_a = L.in_operand(self.d_q.data_ptr(), self.d_s.data_ptr())
        self.dx_w = (L.in_operand(self.W1q.data_ptr(), self.W1s_p.data_ptr()) if self.fc1_mxfp8
                     else L.in_operand(self.W1q.data_ptr(), self.W1s.data_ptr(), tiled=True))
        self.dx_out = L.ActOut(None, None, None, None, self.dX_perm.data_ptr(), None, None)
        self.fc1_out = L.ActOut(self.a_q.data_ptr(), self.a_s.data_ptr(), self.a_qc.data_ptr(),
                                self.a_sc.data_ptr(), None, None, self.pre.data_ptr())
        self.bwd_out = L.ActOut(self.d_q.data_ptr(), self.d_s.data_ptr(), self.d_qc.data_ptr(),
                                self.d_sc.data_ptr(), None, None, None)

    # each entry: (name, callable issuing exactly one C-ABI call)
    def forward_calls(self, x, topk_idx, topk_prob):
        lib, s = self.lib, _s()
        E, N1, H, F, T, k, R = self.E, self.N1, self.H, self.F, self.T, self.k, self.R_cap
        st = _p(self.status)
        if self.nvfp4:
            return self._forward_calls_nvfp4(x, topk_idx, topk_prob)
        xq, xs = (_p(self.x_qc), _p(self.x_sc)) if self.fused_cols else (None, None)
        fc1 = [("fc1_glu_quant", self.fc1_mxfp8_call())]
        if self.fc1_mxfp8:
            fc1 = [
                ("quant_x_rows", lambda: lib.moe_quantize_mxfp8(
                    _p(self.x_perm), 1, R, H, 0, _p(self.counts), _p(self.offsets), E, _p(self.x_qr), _p(self.x_sr),
                    st, s)),
                ("quant_w1_dual", lambda: lib.moe_quantize_mxfp8_dual(
                    _p(self.W1p), E, N1, H, _p(self.W1qr), _p(self.W1sr), _p(self.W1q), _p(self.W1s_p), st, s)),
                ("fc1_mxfp8", lambda: lib.moe_grouped_fc1_glu_quant_fwd_mxfp8(
                    _p(self.x_qr), _p(self.x_sr), _p(self.W1qr), _p(self.W1sr), _p(self.b1p), None, _p(self.counts),
                    _p(self.offsets), E, H, F, R, C.byref(self.params), L.OUT_MXFP8, C.byref(self.fc1_out),
                    _p(self.ws_fc1mx), self.ws_fc1mx.numel(), self.sm_margin, st, s)),
            ]
        return [
            ("route_permute_qcol" if self.fused_cols else "route_permute", lambda: lib.moe_route_permute(
                _p(x), _p(topk_idx), _p(topk_prob), T, H, k, self.expert_begin, E, R, _p(self.x_perm),
                _p(self.row_of), _p(self.tok_of), _p(self.prob_perm), _p(self.counts), _p(self.offsets), xq, xs,
                _p(self.ws), self.ws_bytes, st, s)),
            *fc1,
            ("quant_w2", lambda: lib.moe_quantize_mxfp8(
                _p(self.W2), E, F, H, 2, None, None, 0, _p(self.W2q), _p(self.W2s), st, s)),
            ("fc2", lambda: lib.moe_grouped_fc2_fwd(
                C.byref(self.fc2_a), C.byref(self.fc2_w), _p(self.counts), _p(self.offsets), E, F, H, R,
                L.OUT_BF16, C.byref(self.fc2_out), _p(self.ws_fc2), self.ws_fc2.numel(), self.sm_margin, st, s)),
            ("combine", lambda: lib.moe_unpermute_combine(
                _p(self.y_perm), _p(self.row_of), _p(topk_prob), T, H, k, _p(self.out), st, s)),
        ]

    def fc1_mxfp8_call(self):
        """The fused FC1 with MXFP8 row + column outputs (the MXFP8 forward's
        FC1 call; also the fused side of the forward ablation)."""
        lib, s = self.lib, _s()
        E, H, F, R = self.E, self.H, self.F, self.R_cap
        st = _p(self.status)
        return lambda: lib.moe_grouped_fc1_glu_quant_fwd(
            _p(self.x_perm), _p(self.W1p), _p(self.b1p), None, _p(self.counts), _p(self.offsets), E, H, F, R,
            C.byref(self.params), L.OUT_MXFP8, C.byref(self.fc1_out), _p(self.ws_fc1), self.ws_fc1_bytes,
            self.sm_margin, st, s)

    def dglu_mxfp8_call(self):
        """The fused dGLU with MXFP8 row + column outputs (the MXFP8 backward's
        dGLU call; also the fused side of the backward ablation)."""
        lib, s = self.lib, _s()
        E, H, F, R = self.E, self.H, self.F, self.R_cap
        return lambda: lib.moe_grouped_dglu_quant_bwd(
            _p(self.dY_perm), _p(self.W2), _p(self.pre), None, _p(self.counts), _p(self.offsets), E, H, F, R,
            C.byref(self.params), L.OUT_MXFP8, C.byref(self.bwd_out), _p(self.db1), _p(self.ws_db),
            self.ws_db_bytes, self.sm_margin, _p(self.status), s)

    def _forward_calls_nvfp4(self, x, topk_idx, topk_prob):
        lib, s = self.lib, _s()
        E, N1, H, F, T, k, R = self.E, self.N1, self.H, self.F, self.T, self.k, self.R_cap
        st = _p(self.status)
        return [
            ("route_permute", lambda: lib.moe_route_permute(
                _p(x), _p(topk_idx), _p(topk_prob), T, H, k, self.expert_begin, E, R, _p(self.x_perm),
                _p(self.row_of), _p(self.tok_of), _p(self.prob_perm), _p(self.counts), _p(self.offsets), None,
                None, _p(self.ws), self.ws_bytes, st, s)),
            ("fc1_glu_nvfp4", lambda: lib.moe_grouped_fc1_glu_quant_fwd(
                _p(self.x_perm), _p(self.W1p), _p(self.b1p), None, _p(self.counts), _p(self.offsets), E, H, F, R,
                C.byref(self.params), L.OUT_NVFP4, C.byref(self.fc1_out4), _p(self.ws_fc1), self.ws_fc1_bytes,
                self.sm_margin, st, s)),
            ("quant_a_nvfp4", lambda: lib.moe_nvfp4_cast(
                _p(self.a_y), _p(self.a_amax), _p(self.counts), _p(self.offsets), E, F, R, _p(self.a_q4),
                _p(self.a_s4), _p(self.a_sg), s)),
            ("amax_w2", lambda: lib.moe_amax_bf16(_p(self.W2), self.W2.numel(), _p(self.w2_amax), s)),
            ("quant_w2_nvfp4", lambda: self.cast_w4(
                _p(self.W2), E, F, H, _p(self.w2_amax), _p(self.W2q4), _p(self.W2s4), _p(self.w2_sg), st, s)),
            ("fc2_nvfp4", lambda: lib.moe_grouped_fc2_fwd(
                C.byref(self.fc2_a4), C.byref(self.fc2_w4), _p(self.counts), _p(self.offsets), E, F, H, R,
                L.OUT_BF16, C.byref(self.fc2_out), _p(self.ws_fc2), self.ws_fc2.numel(), self.sm_margin, st, s)),
            ("combine", lambda: lib.moe_unpermute_combine(
                _p(self.y_perm), _p(self.row_of), _p(topk_prob), T, H, k, _p(self.out), st, s)),
        ]

    def backward_calls(self, dOut):
        lib, s = self.lib, _s()
        E, N1, H, F, T, k, R = self.E, self.N1, self.H, self.F, self.T, self.k, self.R_cap
        st = _p(self.status)
        dY_perm = self.dY_perm
        if self.nvfp4:
            return self._backward_calls_nvfp4(dOut)
        dq, ds = (_p(self.dy_qc), _p(self.dy_sc)) if self.fused_cols else (None, None)
        col_casts = [] if self.fused_cols else [
            ("quant_x_col", lambda: lib.moe_quantize_mxfp8(
                _p(self.x_perm), 1, R, H, 1, _p(self.counts), _p(self.offsets), E, _p(self.x_qc), _p(self.x_sc), st, s)),
            ("quant_dy_col", lambda: lib.moe_quantize_mxfp8(
                _p(dY_perm), 1, R, H, 1, _p(self.counts), _p(self.offsets), E, _p(self.dy_qc), _p(self.dy_sc), st, s)),
        ]
        return [
            ("combine_bwd_qcol" if self.fused_cols else "combine_bwd", lambda: lib.moe_combine_bwd(
                _p(dOut), _p(self.y_perm), _p(self.row_of), _p(self.tok_of), _p(self.prob_perm), _p(self.offsets),
                T, H, k, E, R, _p(dY_perm), _p(self.dprob), dq, ds, st, s)),
            ("dglu_quant", self.dglu_mxfp8_call()),
            *([] if self.fc1_mxfp8 else [("quant_w1", lambda: lib.moe_quantize_mxfp8(
                _p(self.W1p), E, N1, H, 2, None, None, 0, _p(self.W1q), _p(self.W1s), st, s))]),
            ("dx", lambda: lib.moe_grouped_fc2_fwd(
                C.byref(self.dx_a), C.byref(self.dx_w), _p(self.counts), _p(self.offsets), E, N1, H, R,
                L.OUT_BF16, C.byref(self.dx_out), _p(self.ws_dx), self.ws_dx.numel(), self.sm_margin, st, s)),
            *col_casts,
            ("wgrad_w1", lambda: lib.moe_grouped_wgrad(
                _p(self.d_qc), _p(self.d_sc), _p(self.x_qc), _p(self.x_sc), _p(self.counts), _p(self.offsets), E,
                N1, H, R, _p(self.dW1), 0, _p(self.ws_wg1), self.ws_wg1.numel(), self.sm_margin, st, s)),
            ("wgrad_w2", lambda: lib.moe_grouped_wgrad(
                _p(self.a_qc), _p(self.a_sc), _p(self.dy_qc), _p(self.dy_sc), _p(self.counts), _p(self.offsets),
                E, F, H, R, _p(self.dW2), 0, _p(self.ws_wg2), self.ws_wg2.numel(), self.sm_margin, st, s)),
            ("permute_bwd", lambda: lib.moe_permute_bwd(
                _p(self.dX_perm), _p(self.row_of), T, H, k, _p(self.dx), st, s)),
        ]

    def _backward_calls_nvfp4(self, dOut):
        lib, s = self.lib, _s()
        E, N1, H, F, T, k, R = self.E, self.N1, self.H, self.F, self.T, self.k, self.R_cap
        st, cnt, off = _p(self.status), _p(self.counts), _p(self.offsets)
        sig = self.rht_signs

        def rot_cast(name, src, C_, ramax, q, sc, sg, amax_call=True):
            calls = []
            if amax_call:
                calls.append((f"rht_amax_{name}", lambda: lib.moe_rht_amax_cols(_p(src), R, C_, off, E, sig, _p(ramax),
                                                                                 st, s)))
            calls.append((f"quant_{name}_rht", lambda: lib.moe_nvfp4_rht_cast_cols(_p(src), R, C_, off, E, _p(ramax),
                                                                                    sig, _p(q), _p(sc), _p(sg), st, s)))
            return calls

        return [
            ("combine_bwd", lambda: lib.moe_combine_bwd(
                _p(dOut), _p(self.y_perm), _p(self.row_of), _p(self.tok_of), _p(self.prob_perm), off,
                T, H, k, E, R, _p(self.dY_perm), _p(self.dprob), None, None, st, s)),
            ("dglu_nvfp4", lambda: lib.moe_grouped_dglu_quant_bwd(
                _p(self.dY_perm), _p(self.W2), _p(self.pre), None, cnt, off, E, H, F, R, C.byref(self.params),
                L.OUT_NVFP4, C.byref(self.bwd_out4), _p(self.db1), _p(self.ws_db), self.ws_db_bytes,
                self.sm_margin, st, s)),
            ("quant_d_nvfp4", lambda: lib.moe_nvfp4_cast(
                _p(self.d_y), _p(self.d_amax), cnt, off, E, N1, R, _p(self.d_q4), _p(self.d_s4), _p(self.d_sg), s)),
            ("amax_w1", lambda: lib.moe_amax_bf16(_p(self.W1p), self.W1p.numel(), _p(self.w1_amax), s)),
            ("quant_w1_nvfp4", lambda: self.cast_w4(
                _p(self.W1p), E, N1, H, _p(self.w1_amax), _p(self.W1q4), _p(self.W1s4), _p(self.w1_sg), st, s)),
            ("dx_nvfp4", lambda: lib.moe_grouped_fc2_fwd(
                C.byref(self.dx_a4), C.byref(self.dx_w4), cnt, off, E, N1, H, R, L.OUT_BF16, C.byref(self.dx_out),
                _p(self.ws_dx), self.ws_dx.numel(), self.sm_margin, st, s)),
            *rot_cast("d", self.d_y, N1, self.d_rht, self.d_rq, self.d_rs, self.d_rsg, amax_call=False),
            *rot_cast("x", self.x_perm, H, self.x_ramax, self.x_rq, self.x_rs, self.x_rsg),
            ("wgrad_w1_nvfp4", lambda: lib.moe_grouped_wgrad_nvfp4(
                _p(self.d_rq), _p(self.d_rs), _p(self.d_rsg), _p(self.x_rq), _p(self.x_rs), _p(self.x_rsg), cnt, off,
                E, N1, H, R, _p(self.dW1), 0, _p(self.ws_wg1), self.ws_wg1.numel(), self.sm_margin, st, s)),
            *rot_cast("a", self.a_y, F, self.a_ramax, self.a_rq, self.a_rs, self.a_rsg),
            *rot_cast("dy", self.dY_perm, H, self.dy_ramax, self.dy_rq, self.dy_rs, self.dy_rsg),
            ("wgrad_w2_nvfp4", lambda: lib.moe_grouped_wgrad_nvfp4(
                _p(self.a_rq), _p(self.a_rs), _p(self.a_rsg), _p(self.dy_rq), _p(self.dy_rs), _p(self.dy_rsg), cnt,
                off, E, F, H, R, _p(self.dW2), 0, _p(self.ws_wg2), self.ws_wg2.numel(), self.sm_margin, st, s)),
            ("permute_bwd", lambda: lib.moe_permute_bwd(
                _p(self.dX_perm), _p(self.row_of), T, H, k, _p(self.dx), st, s)),
        ]

    # ---- unfused path (the ablation baseline): the same tcgen05 GEMM writing
    # bf16, then a separate activation kernel and separate quantize kernels
    def _unfused_buffers(self):
        if getattr(self, "_u", None) is None:
            z = lambda *sh, dt=torch.bfloat16: torch.empty(*sh, dtype=dt, device=self.dev)
            E, N1, H, F, R = self.E, self.N1, self.H, self.F, self.R_cap
            u8 = torch.uint8
            self._u = {
                "pre": z(R, N1), "y": z(R, F), "a_q": z(R, F, dt=u8), "a_s": z(R, F // 32, dt=u8),
                "a_qc": z(F, R, dt=u8), "a_sc": z(F, R // 32, dt=u8), "da": z(R, F), "d": z(R, N1),
                "d_q": z(R, N1, dt=u8), "d_s": z(R, N1 // 32, dt=u8), "d_qc": z(N1, R, dt=u8),
                "d_sc": z(N1, R // 32, dt=u8),
            }
            self._u_none = L.glu_params("none")
            self._u_fwd_out = L.ActOut(None, None, None, None, None, None, self._u["pre"].data_ptr())
            self._u_bwd_out = L.ActOut(None, None, None, None, None, None, self._u["da"].data_ptr())
        return self._u

    def forward_unfused_calls(self):
        """GEMM (+bias) -> bf16 pre; activation -> bf16 y; MXFP8 rows; MXFP8 columns."""
        u = self._unfused_buffers()
        lib, s = self.lib, _s()
        E, N1, H, F, R = self.E, self.N1, self.H, self.F, self.R_cap
        st, cnt, off = _p(self.status), _p(self.counts), _p(self.offsets)
        return [
            ("gemm", lambda: lib.moe_grouped_fc1_glu_quant_fwd(
                _p(self.x_perm), _p(self.W1p), _p(self.b1p), None, cnt, off, E, H, N1, R, C.byref(self._u_none),
                L.OUT_BF16, C.byref(self._u_fwd_out), _p(self.ws_fc1u), self.ws_fc1_bytes, self.sm_margin, st, s)),
            ("act", lambda: lib.moe_glu_act(_p(u["pre"]), cnt, off, E, F, R, C.byref(self.params), _p(u["y"]), s)),
            ("quant_rows", lambda: lib.moe_quantize_mxfp8(_p(u["y"]), 1, R, F, 0, cnt, off, E, _p(u["a_q"]),
                                                          _p(u["a_s"]), st, s)),
            ("quant_cols", lambda: lib.moe_quantize_mxfp8(_p(u["y"]), 1, R, F, 1, cnt, off, E, _p(u["a_qc"]),
                                                          _p(u["a_sc"]), st, s)),
        ]

    def backward_unfused_calls(self, dY_perm):
        """GEMM dY . W2^T -> bf16 da; dActivation -> bf16 dFC1; MXFP8 rows; columns."""
        u = self._unfused_buffers()
        lib, s = self.lib, _s()
        E, N1, H, F, R = self.E, self.N1, self.H, self.F, self.R_cap
        st, cnt, off = _p(self.status), _p(self.counts), _p(self.offsets)
        return [
            ("gemm", lambda: lib.moe_grouped_fc1_glu_quant_fwd(
                _p(dY_perm), _p(self.W2), None, None, cnt, off, E, H, F, R, C.byref(self._u_none), L.OUT_BF16,
                C.byref(self._u_bwd_out), _p(self.ws_fc1u), self.ws_fc1_bytes, self.sm_margin, st, s)),
            ("dact", lambda: lib.moe_dglu_act(_p(u["da"]), _p(self.pre), cnt, off, E, F, R, C.byref(self.params),
                                              _p(u["d"]), s)),
            ("quant_rows", lambda: lib.moe_quantize_mxfp8(_p(u["d"]), 1, R, N1, 0, cnt, off, E, _p(u["d_q"]),
                                                          _p(u["d_s"]), st, s)),
            ("quant_cols", lambda: lib.moe_quantize_mxfp8(_p(u["d"]), 1, R, N1, 1, cnt, off, E, _p(u["d_qc"]),
                                                          _p(u["d_sc"]), st, s)),
        ]

    def step_calls(self, x, topk_idx, topk_prob, dOut):
        return self.forward_calls(x, topk_idx, topk_prob) + self.backward_calls(dOut)

    def run(self, calls, events=None):
        """Issues the calls on the current stream; optional events[i] are
        recorded before call i and events[-1] after the last one."""
        for i, (name, fn) in enumerate(calls):
            if events is not None:
                events[i].record()
            L.check(fn(), name)
        if events is not None:
            events[len(calls)].record()

    def step(self, x, topk_idx, topk_prob, dOut):
        self.run(self.step_calls(x, topk_idx, topk_prob, dOut))

    def capture(self, x, topk_idx, topk_prob, dOut) -> torch.cuda.CUDAGraph:
        """Captures one forward + backward step into a CUDA graph (global
        capture mode: any host synchronisation inside would fail it)."""
        calls = self.step_calls(x, topk_idx, topk_prob, dOut)
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.run(calls)  # warm-up outside capture (sets kernel attributes)
            torch.cuda.synchronize()
            n0 = self.lib.moe_launch_count()
            with torch.cuda.graph(g, stream=s, capture_error_mode="global"):
                self.run(self.step_calls(x, topk_idx, topk_prob, dOut))
            # kernel launches recorded into the graph (one per library launch)
            self.graph_launches = int(self.lib.moe_launch_count() - n0)
        torch.cuda.current_stream().wait_stream(s)
        return g
