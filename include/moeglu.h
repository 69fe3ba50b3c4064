/*
 * moeglu.h — C ABI of libmoeglu.so: the sync-free MoE MLP hot path for
 * GB300 (sm_103a).  Grouped GEMM with the GLU activation fused into its
 * epilogue and MXFP8 / NVFP4 quantisation (plus the transposed copy) fused
 * after it, forward and backward, with the permute and combine around it.
 *
 * Sources (page titles; sections named on them):
 *   [MoE-Fusion] "Boosting MoE Training Throughput with Advanced Fusion
 *                Kernels" (NVIDIA technical blog, 2026-06-15): the
 *                three-kernel family GroupGemm + Quantize,
 *                GroupGemm + Activation + Quantize/Transpose,
 *                GroupGemm + dActivation + Quantize/Transpose; sections
 *                "Optimizing GLU via fused GEMM epilogues" (Fig. 2),
 *                "Eliminating host-device synchronisation",
 *                "Fusing MXFP8 and NVFP4 quantisation", and the list of
 *                end-to-end features (dynamic scheduling, cluster margin).
 *   [MegaMoE]    hnwysp.cn article on the MegaMoE math model and DeepGEMM:
 *                §2.1 (routing, combine), §2.3 (FP8 formats, block scales),
 *                §4.3 (grouped GEMM over contiguous expert rows), §5.3 (tails).
 *
 * Conventions for every call
 *   - All tensor pointers are caller-owned DEVICE memory, row-major, dense
 *     (the leading dimension is the row length given).  The library never
 *     allocates device memory, never synchronises the stream and never reads
 *     device data on the host: per-expert counts stay on the device, so a
 *     whole layer can be captured in one CUDA graph.
 *   - Arguments are validated on the host; a bad argument returns
 *     MOE_ERR_ARG and launches nothing.  A launch failure returns
 *     MOE_ERR_CUDA.  Errors found on the device (capacity overflow, a
 *     pipeline wait that timed out) are OR-ed into the caller's int32
 *     `status` word (device memory, zero it before use) and read with
 *     moe_get_status() outside any capture.
 *   - Shapes: T tokens, H hidden, k top-k, E local experts, F expert FFN
 *     width, N1 = 2F (gated activations) or F (sReLU).  Permuted buffers
 *     have R_cap rows (a multiple of 128, >= T*min(k,E) + 31*E is always
 *     enough).  Rows of one expert are contiguous, start at offsets[e]
 *     (a multiple of 32) and are followed by pad rows up to the next
 *     multiple of 32; only rows < offsets[E] are defined.
 *   - bf16 means IEEE bfloat16 (uint16 storage); MXFP8 tensors are E4M3
 *     codes (uint8) with one E8M0 scale byte per 32 consecutive elements
 *     along the contiguous dimension.
 *   - `stream` is a cudaStream_t (0 = legacy default stream).
 *   - `sm_margin` leaves that many SMs free for concurrent kernels
 *     ([MoE-Fusion]: configurable cluster margin); the persistent GEMMs
 *     launch one CTA per remaining SM.
 */
#ifndef MOEGLU_H
#define MOEGLU_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef void* moe_stream_t; /* cudaStream_t */
typedef uint16_t moe_bf16;  /* bfloat16 storage */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_ARG = 1,         /* invalid argument (host check) */
  MOE_ERR_CUDA = 2,        /* CUDA runtime / launch error */
  MOE_ERR_CAPACITY = 4,    /* device: routed rows exceed R_cap */
  MOE_ERR_TIMEOUT = 8,     /* device: a pipeline wait gave up */
  MOE_ERR_UNSUPPORTED = 16 /* shape/option this build does not handle */
} moe_status_t;

/* Activation of the FC1 epilogue.  [MoE-Fusion] names SwiGLU, GeGLU and
 * sReLU; formulas (textbook readings): SwiGLU (u'+c) g' sigmoid(alpha g');
 * GeGLU (u'+c) g' Phi(g') (erf form) or its tanh approximation; sReLU
 * max(x,0)^2 (not gated, N1 = F); sReGLU (u'+c) max(g',0)^2. */
typedef enum {
  MOE_ACT_SWIGLU = 0,
  MOE_ACT_GEGLU = 1,
  MOE_ACT_GEGLU_TANH = 2,
  MOE_ACT_SRELU = 3,
  MOE_ACT_SREGLU = 4,
  MOE_ACT_NONE = 5 /* FC1 only: plain grouped GEMM writing the bf16 pre-activation (out->pre),
                      no activation, for the unfused path; here F is the full GEMM width N1 */
} moe_act_t;

/* Epilogue options ([MoE-Fusion]: clamping, feature scaling, bias).
 * g' = clamp(gate, gate_lo, gate_hi), u' = clamp(up, up_lo, up_hi); the
 * clamp's derivative is 1 inside the closed interval and 0 outside.  Use
 * +-INFINITY to disable a bound.  c = up_offset (GPT-OSS uses 1). */
typedef struct {
  int32_t act;       /* moe_act_t */
  float alpha;       /* SwiGLU sigmoid slope (1 = plain, 1.702 GPT-OSS) */
  float up_offset;   /* c */
  float gate_lo, gate_hi;
  float up_lo, up_hi;
} moe_glu_params_t;

/* Output quantisation of a fused epilogue. */
typedef enum {
  MOE_OUT_BF16 = 0,  /* y bf16 [R_cap][N] */
  MOE_OUT_MXFP8 = 1, /* q_row/s_row (+ q_col/s_col when non-null) */
  MOE_OUT_NVFP4 = 2  /* y bf16 + per-tensor amax (cast with moe_nvfp4_cast) */
} moe_out_mode_t;

/* Outputs of a fused activation epilogue (N = F for the forward, N = N1 for
 * the backward).  Unused pointers may be NULL. */
typedef struct {
  uint8_t* q_row;    /* MXFP8 codes   [R_cap][N]      */
  uint8_t* s_row;    /* E8M0 scales   [R_cap][N/32]   */
  uint8_t* q_col;    /* transposed    [N][R_cap]      (column-wise blocks of 32 rows) */
  uint8_t* s_col;    /*               [N][R_cap/32]   */
  moe_bf16* y;       /* bf16 output   [R_cap][N]      (BF16 / NVFP4 modes) */
  float* amax;       /* one float: max |y| over all real rows (NVFP4 mode; the call zeroes it first) */
  moe_bf16* pre;     /* forward only: saved pre-activation [R_cap][N1] (bias added), for the backward */
  float* row_dot;    /* backward only, may be NULL: per-row partial sums of da * act(pre) (the
                      * gradient of a per-row feature scale), [R_cap][moe_dglu_row_dot_parts(F)]
                      * f32; reduce them with moe_feature_scale_grad */
  float* rht_amax;   /* backward NVFP4 mode only, may be NULL: one float, the amax of the
                      * transposed random Hadamard rotation of y ([MoE-Fusion] "Fusing MXFP8 and
                      * NVFP4 quantisation"): over every 16-row block of the padded segments and
                      * every column, max |H16 diag(s) bf16(y)[block, c]| / 4, H16 the Sylvester
                      * Hadamard matrix; the call zeroes it first.  Must be NULL in the forward. */
  uint32_t rht_signs;/*   the 16 signs s of that rotation: bit i set -> s_i = -1 (drawn by the caller) */
} moe_act_out_t;

/* Operand of a grouped GEMM that takes either precision. */
typedef enum {
  MOE_IN_BF16 = 0,        /* bf16 values */
  MOE_IN_MXFP8 = 1,       /* E4M3 codes with E8M0 scales, one per 32 elements along K */
  MOE_IN_NVFP4 = 2,       /* packed E2M1 codes (element 2i in the low nibble of byte i) with E4M3
                             scales, one per 16 elements along K, and one fp32 per-tensor scale
                             s_g: value = e2m1 * s_b / s_g (moe_nvfp4_cast, moe_nvfp4_cast_cols) */
  MOE_IN_MXFP8_TILED = 3, /* an MXFP8 weight (the W operand of moe_grouped_fc2_fwd, next to an
                             MXFP8 A) whose scales are already in the order the tensor cores copy
                             them, as written by moe_quantize_mxfp8 with col = 2: the call skips
                             their re-tiling.  Scales 16-byte aligned. */
  MOE_IN_NVFP4_TILED = 4  /* the same for an NVFP4 weight next to an NVFP4 A: scales as written by
                             moe_nvfp4_cast_cols_tiled.  Scales 16-byte aligned. */
} moe_in_dtype_t;

typedef struct {
  int32_t dtype;              /* moe_in_dtype_t */
  const void* data;           /* the values (bf16) or codes (E4M3, packed E2M1) */
  const uint8_t* scale;       /* MXFP8: the E8M0 scales; NVFP4: the E4M3 block scales */
  const float* global_scale;  /* NVFP4 only: device pointer to s_g */
} moe_in_t;

/* ---------------------------------------------------------------------- */

/* FC1 weight repack ([MoE-Fusion], "Optimizing GLU via fused GEMM
 * epilogues", Fig. 2: input and gate columns repacked so one thread block
 * owns matching halves; done once at checkpoint load).
 * W1 [E][2F][H] bf16, rows [0,F) input, [F,2F) gate  ->  W1p [E][2F][H]:
 * packed row p, block b = p/64, o = p%64: o < 32 -> input row 32b+o,
 * else gate row F+32b+o-32.  Also repacks a bias [E][2F] when H == 1.
 * F % 32 == 0.  inverse != 0 performs the inverse permutation. */
MOE_API moe_status_t moe_repack_fc1(const moe_bf16* W1, moe_bf16* W1p, int E, int F, int H,
                            int inverse, moe_stream_t stream);

/* Bytes of device workspace moe_route_permute needs. */
MOE_API size_t moe_route_workspace_size(int T, int k, int E);

/* Routing + permutation ([MegaMoE] §2.1, §4.3; [MoE-Fusion],
 * "Eliminating host-device synchronisation": counts stay on the device).
 * In:  x [T][H] bf16, topk_idx [T][k] int32 (global expert ids),
 *      topk_prob [T][k] f32.  Experts [expert_begin, expert_begin+E) are
 *      local; other assignments are dropped (row_of = -1).
 * Out: counts [E], offsets [E+1] (exclusive prefix of counts rounded up to
 *      32), row_of [T*k] (permuted row of assignment t*k+j, rows of one
 *      expert in ascending t*k+j), tok_of [R_cap] (token of each row, -1
 *      on pad rows), prob_perm [R_cap] (0 on pad rows), x_perm [R_cap][H]
 *      (pad rows zero).  ws: moe_route_workspace_size() bytes.
 *      offsets[E] > R_cap sets MOE_ERR_CAPACITY in *status and writes no rows.
 * xq_col / xs_col (both or neither; xq_col 16-byte aligned): also the
 *      column-wise MXFP8 copy of x_perm that the FC1 weight gradient reads
 *      ([MoE-Fusion] "Fusing MXFP8 and NVFP4 quantisation": MXFP8 = row-wise
 *      output plus a transposed copy), made while the rows are gathered:
 *      xq_col [H][R_cap] E4M3 codes, xs_col [H][R_cap/32] E8M0 scales, one
 *      block per 32 rows (the same values as moe_quantize_mxfp8 with col = 1
 *      on x_perm and the counts); blocks at or past offsets[E] untouched. */
MOE_API moe_status_t moe_route_permute(const moe_bf16* x, const int32_t* topk_idx, const float* topk_prob,
                               int T, int H, int k, int expert_begin, int E, int R_cap,
                               moe_bf16* x_perm, int32_t* row_of, int32_t* tok_of, float* prob_perm,
                               int32_t* counts, int32_t* offsets, uint8_t* xq_col, uint8_t* xs_col,
                               void* ws, size_t ws_bytes, int32_t* status, moe_stream_t stream);

/* GroupGemm + Activation + Quantize/Transpose, forward ([MoE-Fusion]).
 * pre = x_perm[rows of e] . W1p[e]^T + b1p[e]  (bf16 in, fp32 accumulate in
 * tensor memory); the epilogue pairs input/gate columns of the packed tile,
 * applies the activation, multiplies by row_scale[row] when non-NULL
 * (feature scaling), and writes per out_mode.  Pad rows are written as 0.
 * x_perm [R_cap][H], W1p [E][N1][H] (packed when gated), b1p [E][N1] or
 * NULL, row_scale [R_cap] f32 or NULL.  H % 64 == 0, F % 32 == 0.
 * ws (nullable, moe_grouped_fc1_workspace_size() bytes, 16-byte aligned):
 * the dynamic tile scheduler's counter; NULL runs the static schedule. */
MOE_API moe_status_t moe_grouped_fc1_glu_quant_fwd(const moe_bf16* x_perm, const moe_bf16* W1p,
                                           const moe_bf16* b1p, const float* row_scale,
                                           const int32_t* counts, const int32_t* offsets,
                                           int E, int H, int F, int R_cap,
                                           const moe_glu_params_t* params, int out_mode,
                                           const moe_act_out_t* out, void* ws, size_t ws_bytes,
                                           int sm_margin, int32_t* status, moe_stream_t stream);

/* Bytes of device workspace of moe_grouped_fc1_glu_quant_fwd: the counter of
 * the dynamic tile scheduler ([MoE-Fusion]: dynamic scheduling, so that the
 * grouped kernels share the GPU with concurrent work).  With ws the CTA
 * pairs take tiles from an atomic counter (zeroed by the call itself, in
 * stream order) instead of a fixed stride; results are the same either way.
 * Calls that may run at the same time need separate workspaces. */
MOE_API size_t moe_grouped_fc1_workspace_size(int E, int N1, int R_cap);

/* GroupGemm + dActivation + Quantize/Transpose, backward ([MoE-Fusion]: the
 * epilogue reads the GEMM output, computes dSwiGLU, quantises and writes).
 * da = dY_perm[rows of e] . W2[e]^T with W2 [E][F][H] (the forward is
 * y = a . W2[e]); (du, dg) from the saved bf16 pre [R_cap][N1]; times
 * row_scale when non-NULL; written as dFC1 [R_cap][N1] in packed column
 * order per out_mode (MXFP8 row + column-wise, or bf16; NVFP4: bf16 plus
 * max |dFC1| and, with dfc1->rht_amax set, the amax of dFC1's transposed
 * random Hadamard rotation, so that no separate pass computes it).  When
 * dfc1->row_dot is non-NULL the epilogue also writes, for every row of the
 * padded segments, partial sums of da * act(pre) over disjoint column
 * ranges (fp32, each slot written once: deterministic), the ingredients of
 * the feature-scale gradient ([MoE-Fusion] "clamping and scaling").
 * dbias (nullable, f32 [E][N1], packed column order like b1p): the gradient
 * of the FC1 bias ([MoE-Fusion] "clamping and scaling": the bias vector of
 * the GLU), dbias[e][c] = sum over the expert's rows of dFC1[r][c] taken on
 * the fp32 values before quantisation.  The epilogue writes one column-sum
 * line per 32-row block into ws and a second kernel adds each expert's lines
 * in block order (deterministic; 0 for an expert without rows).
 * ws (moe_grouped_dglu_workspace_size(N1, R_cap) bytes, 16-byte aligned;
 * required with dbias, else nullable): its first 256 bytes are the dynamic
 * tile scheduler's counter (as for the forward; NULL runs the static
 * schedule), the rest the bias-gradient lines.
 * H % 64 == 0. */
MOE_API moe_status_t moe_grouped_dglu_quant_bwd(const moe_bf16* dY_perm, const moe_bf16* W2,
                                        const moe_bf16* pre, const float* row_scale,
                                        const int32_t* counts, const int32_t* offsets,
                                        int E, int H, int F, int R_cap,
                                        const moe_glu_params_t* params, int out_mode,
                                        const moe_act_out_t* dfc1, float* dbias,
                                        void* ws, size_t ws_bytes, int sm_margin,
                                        int32_t* status, moe_stream_t stream);

/* Bytes of device workspace moe_grouped_dglu_quant_bwd needs for the bias
 * gradient (N1 = 2F gated, F for sReLU). */
MOE_API size_t moe_grouped_dglu_workspace_size(int N1, int R_cap);

/* MXFP8 quantisation of a bf16 tensor (the standalone quantize/transpose
 * kernel of the unfused path, and the weight cast).  src [G][R][C] bf16,
 * 16-byte aligned.
 * col == 0: q [G][R][C], s [G][R][C/32] (blocks along C); C % 32 == 0.
 * col == 1: q [G][C][R], s [G][C][R/32] (blocks of 32 rows; transposed);
 *           R % 32 == 0, C % 8 == 0; the tiles are staged by TMA.
 * col == 2: as col == 1, with the scales written in the order the
 *           block-scaled GEMM's tensor-core copies read them when the
 *           result is its N x K weight (N = C, K = R; an MXFP8_TILED
 *           operand of moe_grouped_fc2_fwd):
 *           s [G][ceil(C/256)][ceil(R/128)][2][512] bytes, byte 16 l + 4 j + i
 *           of the 512 of (128-row group g of C, k-block b of R) = the scale
 *           of row 128 g + 32 j + l, rows 128 b + 32 i .. + 31 of R
 *           (moe_mxfp8_tiled_scale_bytes); no counts; s 16-byte aligned.
 * counts/offsets (G == 1 only, may be NULL): rows of the permuted layout
 * outside [offsets[e], offsets[e]+counts[e]) are treated as zero; results
 * for rows >= offsets[E] are unspecified (their scales are not written).
 * status (nullable): device word that receives MOE_ERR_TIMEOUT if a staged
 * tile never arrives (the column kernel then stops early). */
MOE_API moe_status_t moe_quantize_mxfp8(const moe_bf16* src, int G, int R, int C, int col,
                                const int32_t* counts, const int32_t* offsets, int E,
                                uint8_t* q, uint8_t* s, int32_t* status, moe_stream_t stream);

/* Bytes of the col == 2 scale layout of moe_quantize_mxfp8 for src [G][R][C]. */
MOE_API size_t moe_mxfp8_tiled_scale_bytes(int G, int R, int C);

/* Both MXFP8 copies of a weight in one pass ([MoE-Fusion] "Fusing MXFP8 and
 * NVFP4 quantisation": a row-wise output plus a transposed copy): src
 * [G][R][C] bf16 is read once and written as
 *   q_row [G][R][C], s_row [G][R][C/32]  (blocks along C, as col == 0), and
 *   q_col [G][C][R], s_col [G][C][R/32]  (blocks along R, as col != 0),
 * the same bytes as the two moe_quantize_mxfp8 calls.  For W1p [E][2F][H]
 * the first feeds an MXFP8-input FC1 (contraction over H), the second the
 * data gradient (contraction over 2F).  R % 32 == 0, C % 32 == 0; src and
 * q_col 16-byte, q_row 8-byte aligned.  status (nullable) as above. */
MOE_API moe_status_t moe_quantize_mxfp8_dual(const moe_bf16* src, int G, int R, int C, uint8_t* q_row,
                                             uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, int32_t* status,
                                             moe_stream_t stream);

/* Bytes of device workspace moe_grouped_fc2_fwd needs with block-scaled
 * (MXFP8 or NVFP4) operands: the scales of the visited tiles, rewritten in the
 * order the tensor cores read them (enough for either type); bf16 operands
 * need none. */
MOE_API size_t moe_grouped_fc2_workspace_size(int E, int K, int N, int R_cap);

/* GroupGemm + Quantize ([MoE-Fusion] "Boosting MoE Training Throughput with
 * Advanced Fusion Kernels": the first of the three fused kernels, a grouped
 * GEMM whose epilogue quantises its output; [MegaMoE] §2.3: block-scaled
 * FP8, C ~ (A_q/s_A)(B_q/s_B)).
 * y[rows of e] = A[rows] . W[e]^T, fp32 accumulate, pad rows 0, written per
 * out_mode from the fp32 accumulator: MOE_OUT_BF16 (out->y), MOE_OUT_MXFP8
 * (out->q_row/s_row, plus the column-wise copy out->q_col/s_col when
 * non-NULL: blocks of 32 rows of one column, as for the fused FC1), or
 * MOE_OUT_NVFP4 (out->y bf16 and out->amax, which the call zeroes first).
 * out->pre, row_dot and rht_amax must be NULL.
 * Serves FC2 (K = F, N = H) and the data-gradient GEMM dX = dFC1 . W1p
 * (K = N1, N = H).
 * Operands: A [R_cap][K], W [E][N][K] (K contiguous in both), the same
 * dtype for both (the tensor cores take one operand type per MMA; a W of
 * MOE_IN_MXFP8_TILED / MOE_IN_NVFP4_TILED counts as MXFP8 / NVFP4 and
 * carries its scales in the tensor-core order):
 *   MOE_IN_MXFP8: E4M3 codes, scale = E8M0 [R_cap][K/32] / [E][N][K/32]
 *                 (4-byte aligned); block-scaled MMA (kind::mxf8f6f4);
 *                 ws = moe_grouped_fc2_workspace_size() bytes, 256-byte
 *                 aligned.  K % 32 == 0, N % 32 == 0 (a partial last
 *                 128-wide k-block or 256-wide column tile is handled).
 *   MOE_IN_NVFP4: packed E2M1 A [R_cap][K/2], W [E][N][K/2], E4M3 block
 *                 scales [R_cap][K/16] / [E][N][K/16] (4-byte aligned) and
 *                 the per-tensor scales; block-scaled MMA (kind::mxf4nvf4,
 *                 16-element blocks); the product is divided by both s_g in
 *                 the epilogue.  ws as for MXFP8.  K % 64 == 0, N % 32 == 0;
 *                 out_mode must be MOE_OUT_BF16 (else MOE_ERR_UNSUPPORTED).
 *                 ([MoE-Fusion] "Fusing MXFP8 and NVFP4 quantisation": the
 *                 consumer of the forward's NVFP4 cast.)
 *   MOE_IN_BF16:  bf16, scale unused; kind::f16 MMA on CTA pairs; ws
 *                 nullable: with >= 256 bytes (16-byte aligned) it holds the
 *                 dynamic tile scheduler's counter, as for the fused FC1.
 *                 K % 64 == 0, N % 32 == 0. */
MOE_API moe_status_t moe_grouped_fc2_fwd(const moe_in_t* A, const moe_in_t* W,
                                 const int32_t* counts, const int32_t* offsets,
                                 int E, int K, int N, int R_cap, int out_mode,
                                 const moe_act_out_t* out, void* ws, size_t ws_bytes,
                                 int sm_margin, int32_t* status, moe_stream_t stream);

/* GroupGemm + Activation + Quantize/Transpose on MXFP8 operands ([MoE-Fusion]
 * "Boosting MoE Training Throughput with Advanced Fusion Kernels": the fused
 * MLP kernels serve the dense and MoE paths in BF16 and MXFP8 recipes; the
 * FC1 input x is quantised to MXFP8 before the GEMM).  The same epilogue as
 * moe_grouped_fc1_glu_quant_fwd (bias, activation, row scale, saved bf16
 * pre-activation, MXFP8 row + column-wise / bf16 / NVFP4 outputs) on the
 * block-scaled product
 *   pre[rows of e] = dequant(xq, xs)[rows] . dequant(W1q[e], W1s[e])^T + b1p[e]
 * xq [R_cap][H] E4M3 with xs [R_cap][H/32] E8M0 (the row-wise MXFP8 of x_perm,
 * e.g. moe_quantize_mxfp8 with col = 0 and the routing's counts/offsets);
 * W1q [E][N1][H] with W1s [E][N1][H/32] (the row-wise MXFP8 of the packed W1p,
 * blocks along H).  ws: moe_grouped_fc2_workspace_size(E, H, N1, R_cap)
 * bytes, 256-byte aligned.  H % 32 == 0, F % 32 == 0; out->row_dot and
 * out->rht_amax must be NULL. */
MOE_API moe_status_t moe_grouped_fc1_glu_quant_fwd_mxfp8(const uint8_t* xq, const uint8_t* xs,
                                                 const uint8_t* W1q, const uint8_t* W1s,
                                                 const moe_bf16* b1p, const float* row_scale,
                                                 const int32_t* counts, const int32_t* offsets,
                                                 int E, int H, int F, int R_cap,
                                                 const moe_glu_params_t* params, int out_mode,
                                                 const moe_act_out_t* out, void* ws, size_t ws_bytes,
                                                 int sm_margin, int32_t* status, moe_stream_t stream);

/* Bytes of device workspace moe_grouped_wgrad (and moe_grouped_wgrad_nvfp4) needs. */
MOE_API size_t moe_grouped_wgrad_workspace_size(int E, int M, int N, int R_cap);

/* Weight-gradient grouped GEMM, contraction over each expert's rows
 * (variable K = the expert's padded row count).  Inputs are the
 * column-wise (transposed) MXFP8 copies: Aq [M][R_cap], As [M][R_cap/32],
 * Bq [N][R_cap], Bs [N][R_cap/32].  D[e] = A[:, seg e] . B[:, seg e]^T,
 * written as f32 (out_f32 != 0) or bf16 into D [E][M][N].
 * dW1p = wgrad(dFC1 col, x col); dW2 = wgrad(a col, dY col).
 * ws: moe_grouped_wgrad_workspace_size() bytes, 256-byte aligned.
 * Pad rows of each segment must hold zero codes (the quantizers write them).
 * M % 32 == 0, N % 32 == 0. */
MOE_API moe_status_t moe_grouped_wgrad(const uint8_t* Aq, const uint8_t* As,
                               const uint8_t* Bq, const uint8_t* Bs,
                               const int32_t* counts, const int32_t* offsets,
                               int E, int M, int N, int R_cap,
                               void* D, int out_f32, void* ws, size_t ws_bytes,
                               int sm_margin, int32_t* status, moe_stream_t stream);

/* Weight-gradient grouped GEMM on NVFP4 operands (kind::mxf4nvf4, E4M3
 * scales per 16 rows): the NVFP4 form of moe_grouped_wgrad.  Aq [M][R_cap/2],
 * As [M][R_cap/16], Bq [N][R_cap/2], Bs [N][R_cap/16] as written by
 * moe_nvfp4_rht_cast_cols (rotated along the rows, which leaves the product
 * unchanged), sgA / sgB their per-tensor scales (device floats).
 * D[e] = dequant(A)[:, seg e] . dequant(B)[:, seg e]^T over the expert's
 * padded row segment (contraction in MMAs of 64 rows; a segment's last MMA
 * may cover 32 of its rows, the rest weighted 0), written as f32
 * (out_f32 != 0) or bf16 into D [E][M][N]; 0 for an expert without rows.
 * ws: moe_grouped_wgrad_workspace_size() bytes, 256-byte aligned.
 * M % 32 == 0, N % 32 == 0. */
MOE_API moe_status_t moe_grouped_wgrad_nvfp4(const uint8_t* Aq, const uint8_t* As, const float* sgA,
                                     const uint8_t* Bq, const uint8_t* Bs, const float* sgB,
                                     const int32_t* counts, const int32_t* offsets,
                                     int E, int M, int N, int R_cap,
                                     void* D, int out_f32, void* ws, size_t ws_bytes,
                                     int sm_margin, int32_t* status, moe_stream_t stream);

/* Unpermute + combine ([MegaMoE] §2.1: y = sum_{i in topk} p_i E_i(x)).
 * out[t] = bf16( sum_j topk_prob[t][j] * y_perm[row_of[t*k+j]] ) over
 * j with row_of >= 0, summed in fp32 in j order; 0 when none is local.
 * H % 8 == 0. */
MOE_API moe_status_t moe_unpermute_combine(const moe_bf16* y_perm, const int32_t* row_of,
                                   const float* topk_prob, int T, int H, int k,
                                   moe_bf16* out, int32_t* status, moe_stream_t stream);

/* Number of partial-sum slots per row that moe_grouped_dglu_quant_bwd writes
 * to dfc1->row_dot for FFN width F (host arithmetic). */
MOE_API int moe_dglu_row_dot_parts(int F);

/* Feature-scale gradient per routed slot: dprob[t*k+j] = sum of the `parts`
 * partials of row row_of[t*k+j] in row_dot (added in slot order, fp32;
 * 0 for row_of < 0).  With a = p * act(pre) in the forward (row_scale =
 * prob_perm), this is dL/dp for the slot's router probability. */
MOE_API moe_status_t moe_feature_scale_grad(const float* row_dot, int parts, const int32_t* row_of,
                                    int T, int k, float* dprob, moe_stream_t stream);

/* Combine backward: the chain rule on the combine above ([MegaMoE] §2.1),
 * for the gradient dout [T][H] bf16 arriving at the layer output.  For every
 * permuted row r < offsets[E] with t = tok_of[r] >= 0:
 *   dY_perm[r] = bf16(prob_perm[r] * dout[t])                 [R_cap][H]
 *   dprob[t*k + j] = <dout[t], y_perm[r]>  (fp32) for the slot with
 *                    row_of[t*k + j] == r                       [T*k] f32
 * Pad rows (tok_of < 0) of dY_perm are written as 0, slots with row_of < 0
 * get dprob 0, rows >= offsets[E] are untouched.  row_of / tok_of /
 * prob_perm / offsets as written by moe_route_permute.  H % 8 == 0,
 * 1 <= k <= 32, 16-byte aligned bf16 buffers.  offsets[E] > R_cap records
 * MOE_ERR_CAPACITY in status and writes nothing else.
 * dyq_col / dys_col (both or neither; dyq_col 16-byte aligned, R_cap % 32
 * == 0): also the column-wise MXFP8 copy of dY_perm that the FC2 weight
 * gradient reads, made while the rows are written: dyq_col [H][R_cap],
 * dys_col [H][R_cap/32], as moe_quantize_mxfp8 with col = 1 on dY_perm. */
MOE_API moe_status_t moe_combine_bwd(const moe_bf16* dout, const moe_bf16* y_perm, const int32_t* row_of,
                             const int32_t* tok_of, const float* prob_perm, const int32_t* offsets,
                             int T, int H, int k, int E, int R_cap, moe_bf16* dY_perm, float* dprob,
                             uint8_t* dyq_col, uint8_t* dys_col, int32_t* status, moe_stream_t stream);

/* Permute backward: dx[t] = bf16( sum_j dx_perm[row_of[t*k+j]] ) over the
 * slots with row_of >= 0, summed in fp32 in j order (the gradient of the
 * gather x_perm[row] = x[tok_of[row]]); 0 for a token with no local
 * assignment.  dx_perm [R_cap][H], dx [T][H] bf16, H % 8 == 0. */
MOE_API moe_status_t moe_permute_bwd(const moe_bf16* dx_perm, const int32_t* row_of, int T, int H, int k,
                             moe_bf16* dx, int32_t* status, moe_stream_t stream);

/* NVFP4 cast of the forward's bf16 output ([MoE-Fusion], "Fusing MXFP8 and
 * NVFP4 quantisation": the fused kernel emits BF16 + per-tensor amax).
 * s_g = 2688 / amax (1 if amax == 0) written to *s_global; per 16
 * elements s_b = E4M3(fp32(amax_b/6) * s_g); q = E2M1(v * fp32(s_g/s_b)).
 * y [R_cap][N] bf16 -> q [R_cap][N/2] (element 2i low nibble),
 * s [R_cap][N/16] E4M3.  Rows >= offsets[E] are not written; pad rows
 * give zeros.  N % 16 == 0. */
MOE_API moe_status_t moe_nvfp4_cast(const moe_bf16* y, const float* amax,
                            const int32_t* counts, const int32_t* offsets, int E,
                            int N, int R_cap, uint8_t* q, uint8_t* s, float* s_global,
                            moe_stream_t stream);

/* max |x| over n bf16 values (n % 8 == 0, x 16-byte aligned) into *amax
 * (device float; overwritten): the per-tensor amax an NVFP4 weight cast
 * needs. */
MOE_API moe_status_t moe_amax_bf16(const moe_bf16* x, size_t n, float* amax, moe_stream_t stream);

/* Column-wise (transposed) NVFP4 cast of a weight whose contraction runs
 * along its rows ([MoE-Fusion] "Fusing MXFP8 and NVFP4 quantisation"; e.g.
 * W2 [E][F][H] for an NVFP4 FC2, K = F): src [G][R][C] bf16 -> q [G][C][R/2]
 * (element 2i in the low nibble), s [G][C][R/16] E4M3, with the same
 * two-level rule as moe_nvfp4_cast under s_g = 2688 / amax (1 if 0 or not
 * finite), written to *s_global.  amax: device float (moe_amax_bf16).
 * R % 16 == 0, q 8-byte aligned.  With src 16-byte aligned, C % 8 == 0,
 * R % 128 == 0, q 16- and s 8-byte aligned the cast streams 128 x 128 tiles
 * through shared memory by TMA; its pipeline waits are bounded and a wait
 * that gives up ORs MOE_ERR_TIMEOUT into *status (device int32, may be
 * NULL).  Other shapes take a direct kernel without waits. */
MOE_API moe_status_t moe_nvfp4_cast_cols(const moe_bf16* src, int G, int R, int C, const float* amax,
                                         uint8_t* q, uint8_t* s, float* s_global, int32_t* status,
                                         moe_stream_t stream);

/* moe_nvfp4_cast_cols with the scales written in the order the block-scaled
 * GEMM's tensor-core copies read them when the result is its N x K weight
 * operand (N = C, K = R; W of moe_grouped_fc2_fwd as MOE_IN_NVFP4_TILED), so
 * that the GEMM call re-tiles no weight scales:
 * s [G][ceil(C/256)][4 ceil(R/256)][2][512 bytes]; the 512 bytes of (256-
 * column tile n, 64-row group k of R, 128-column half h) hold at byte
 * 16 l + 4 j + i the scale of column 256 n + 128 h + 32 j + l, rows
 * 64 k + 16 i .. + 15 of R.  Groups past R and columns past C hold zero
 * scales.  Codes and scale values equal moe_nvfp4_cast_cols's.  Staged form
 * only: src and q 16-byte aligned, s 16-byte aligned, C % 8 == 0,
 * R % 128 == 0, else MOE_ERR_ARG.  s holds moe_nvfp4_tiled_scale_bytes(G, R,
 * C) bytes. */
MOE_API moe_status_t moe_nvfp4_cast_cols_tiled(const moe_bf16* src, int G, int R, int C, const float* amax,
                                               uint8_t* q, uint8_t* s, float* s_global, int32_t* status,
                                               moe_stream_t stream);
MOE_API size_t moe_nvfp4_tiled_scale_bytes(int G, int R, int C);

/* NVFP4 backward operands ([MoE-Fusion] "Fusing MXFP8 and NVFP4
 * quantisation": the weight-gradient GEMM reads the transposed tensors after
 * a random Hadamard rotation, whose per-tensor amax the dGLU epilogue writes
 * for dFC1).  For src [R_cap][C] bf16 in the permuted layout (dFC1, x_perm;
 * rows >= offsets[E] are not read) every 16-row block of every column is
 * rotated, z = H16 diag(s) v / 4 (H16 the Sylvester Hadamard matrix, bit i of
 * signs set -> s_i = -1, the same rotation as moe_act_out_t.rht_amax), and:
 *   moe_rht_amax_cols   writes max |z| to *amax (device float, overwritten);
 *   moe_nvfp4_rht_cast_cols casts z column-wise to NVFP4 under
 *       s_g = 2688 / amax (amax = that rotated amax), written to *s_global:
 *       q [C][R_cap/2] (element 2i in the low nibble), s [C][R_cap/16] E4M3;
 *       blocks at or past offsets[E] are not written.
 * The rotation is orthonormal, so rotating both operands of the weight
 * gradient along its contracted rows leaves the product unchanged.
 * R_cap % 128 == 0; q 16-byte and s 4-byte aligned.  With src 16-byte
 * aligned, C % 8 == 0 (and s 8-byte aligned for the cast) both stream
 * 128 x 128 tiles through shared memory by TMA, with bounded waits that OR
 * MOE_ERR_TIMEOUT into *status (device int32, may be NULL) when they give
 * up; other shapes take direct kernels. */
MOE_API moe_status_t moe_rht_amax_cols(const moe_bf16* src, int R_cap, int C, const int32_t* offsets, int E,
                                       uint32_t signs, float* amax, int32_t* status, moe_stream_t stream);
MOE_API moe_status_t moe_nvfp4_rht_cast_cols(const moe_bf16* src, int R_cap, int C, const int32_t* offsets, int E,
                                             const float* amax, uint32_t signs, uint8_t* q, uint8_t* s,
                                             float* s_global, int32_t* status, moe_stream_t stream);

/* Standalone activation of the unfused path: pre [R][N1] bf16 -> y [R][F]
 * bf16 (rows >= offsets[E] untouched, pad rows 0).  F % 32 == 0; pre and y
 * 16-byte aligned, else MOE_ERR_ARG.  Evaluates the same activation forms
 * as the fused epilogue of moe_grouped_fc1_glu_quant_fwd. */
MOE_API moe_status_t moe_glu_act(const moe_bf16* pre, const int32_t* counts, const int32_t* offsets,
                         int E, int F, int R_cap, const moe_glu_params_t* params,
                         moe_bf16* y, moe_stream_t stream);

/* moe_route_permute without a workspace argument and without any device
 * allocation, for callers that cannot allocate device memory when they route
 * (a runtime that owns all GPU memory in its own pool, or code running where
 * cudaMalloc is not allowed).  The pages describe no such entry point: it is
 * a convenience of this library, not part of the method.
 * Same arguments, results and status semantics as moe_route_permute minus
 * ws/ws_bytes.  Its scratch is a fixed 1 MiB array inside the library
 * (moe_route_noalloc_max_scratch_bytes()).  The array comes into being on a
 * GPU when the library's device code is first loaded there (with CUDA's lazy
 * module loading: the first kernel launch or the address look-up below) and
 * stays until the process exits; a routing whose scratch
 * (moe_route_workspace_size(T, k, E)) exceeds it returns MOE_ERR_ARG.
 * The first call on each device looks up that array's device address
 * (cudaGetSymbolAddress) with the device current and keeps it; make that
 * first call before any stream capture.  After cudaDeviceReset the kept
 * address is stale: do not call this entry point on a device that has been
 * reset in this process.  All calls share the one array: calls that
 * may run at the same time on the GPU (different streams, or several host
 * threads) race on it and must be serialised by the caller.  Nothing in the
 * array needs to start at zero: each call writes every entry it reads. */
MOE_API moe_status_t moe_route_permute_noalloc(const moe_bf16* x, const int32_t* topk_idx, const float* topk_prob,
                                               int T, int H, int k, int expert_begin, int E, int R_cap,
                                               moe_bf16* x_perm, int32_t* row_of, int32_t* tok_of,
                                               float* prob_perm, int32_t* counts, int32_t* offsets,
                                               uint8_t* xq_col, uint8_t* xs_col, int32_t* status,
                                               moe_stream_t stream);

/* Size in bytes of the fixed scratch array used by moe_route_permute_noalloc. */
MOE_API size_t moe_route_noalloc_max_scratch_bytes(void);

/* Standalone backward activation of the unfused path: da [R][F] bf16 (the
 * data-gradient GEMM output, computed e.g. by moe_grouped_fc1_glu_quant_fwd
 * with MOE_ACT_NONE on dY_perm and W2) and the saved pre [R][N1] bf16 ->
 * dFC1 [R][N1] bf16 in packed column order (rows >= offsets[E] untouched).
 * F % 32 == 0; da, pre and dfc1 16-byte aligned, else MOE_ERR_ARG.
 * Evaluates the same forms as the fused epilogue of moe_grouped_dglu_quant_bwd. */
MOE_API moe_status_t moe_dglu_act(const moe_bf16* da, const moe_bf16* pre, const int32_t* counts,
                                  const int32_t* offsets, int E, int F, int R_cap,
                                  const moe_glu_params_t* params, moe_bf16* dfc1, moe_stream_t stream);

/* Copies the device status word to *host_out (synchronises `stream`; not
 * for use inside a graph capture). */
MOE_API moe_status_t moe_get_status(const int32_t* status, int32_t* host_out, moe_stream_t stream);

/* Pipeline wait limit in nanoseconds for the persistent GEMMs (default 2e9);
 * after it a wait gives up, sets MOE_ERR_TIMEOUT and the kernel returns. */
MOE_API void moe_set_wait_limit_ns(uint64_t ns);

/* Self-test of the bounded wait behind every pipeline wait of the
 * persistent kernels (failure detection without a GPU fault).  One thread
 * waits for an mbarrier phase through the same guard the GEMMs use, with the
 * limit set by moe_set_wait_limit_ns.  arrive != 0: the barrier is arrived
 * at first, the wait succeeds and *status is not touched.  arrive == 0:
 * nothing arrives, the wait gives up after the limit and ORs MOE_ERR_TIMEOUT
 * into *status; the kernel then returns normally.  *waited_ns (device
 * uint64) receives the time the wait took.  status and waited_ns are device
 * pointers; NULL returns MOE_ERR_ARG. */
MOE_API moe_status_t moe_wait_selftest(int arrive, int32_t* status, uint64_t* waited_ns, moe_stream_t stream);

/* Tile configuration of the bf16 grouped GEMMs (FC1 forward, dGLU
 * backward): enable != 0 (default) runs them on CTA pairs (256 x 256 tiles,
 * tcgen05 cta_group::2, 32 KB per SM per pipeline stage); 0 runs one CTA per
 * 128 x 256 tile.  Both compute the same results.  Process-wide. */
MOE_API void moe_set_cta_pairs(int enable);

/* Tail tiles of the CTA-pair bf16 GEMMs (FC1 forward, dGLU backward, the
 * bf16 case of moe_grouped_fc2_fwd): an expert whose last 256-row pair tile
 * holds at most max_rows rows computes that tile transposed (the weights as
 * the M = 256 operand, the tile's rows rounded up to 32 as N), so the
 * tensor cores do not multiply the empty rows of a mostly empty tile.  The
 * results are the same as the regular tile's (the bias-gradient partials
 * add their 32 rows in another order).  max_rows in {0 (off), 32, 64, 96,
 * 128}, default 32; anything else returns MOE_ERR_ARG.  Process-wide. */
MOE_API moe_status_t moe_set_tail_swap(int max_rows);

/* Cumulative number of kernels this library has launched in this process
 * (launch accounting for benchmarks). */
MOE_API uint64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MOEGLU_H */
