// Output stage shared by the fused epilogues of the grouped GEMMs: one
// 32-column block of fp32 results of one accumulator row (one thread = one
// row, a warp = 32 consecutive rows) becomes MXFP8 row-wise codes and scale,
// the column-wise (transposed) MXFP8 copy, bf16, or bf16 plus the NVFP4
// amaxes ([MoE-Fusion] "Boosting MoE Training Throughput with Advanced Fusion
// Kernels", "Fusing MXFP8 and NVFP4 quantisation": quantisation and the
// transposed copy happen inside the GEMM kernel, on the fp32 accumulator
// values).  The argument struct `Out` of emit_block provides out_mode, out_N
// (row length of the outputs), R_cap, q_row, s_row, q_col, s_col, y,
// rht_amax and rht_signs.
#pragma once

#include "common.cuh"

namespace moeglu {

// Running per-thread maxima of the NVFP4 mode (float bits of |v|, v >= 0):
// plain = max |y|, rht = max |rotated y| (backward, when requested).
struct Amax {
  uint32_t plain, rht;
};

// One 32-column block of activation results of one row -> its outputs.
// y: 32 fp32 values (0 on pad rows).  col0: first output column (multiple
// of 32).  row_ok: this thread's row lies inside the padded segment.
// The column-wise MXFP8 path needs the whole warp (the warp's 32 rows are
// one column block).
template <class Out>
__device__ __forceinline__ void emit_block(const Out& a, const float* y, int col0, int row, int rb, bool row_ok,
                                           uint8_t* scratch, int lane, Amax& amax_bits) {
  const int N = a.out_N;
  if (a.out_mode == MOE_OUT_MXFP8) {
    uint32_t codes[8];
    const uint32_t sb = mx_quant_block32(y, codes);
    if (row_ok) {
      uint4* dst = reinterpret_cast<uint4*>(a.q_row + (size_t)row * N + col0);
      dst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
      dst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
      a.s_row[(size_t)row * (N / 32) + col0 / 32] = (uint8_t)sb;
    }
    if (a.q_col != nullptr) {
      // Column blocks (one column, the warp's 32 rows), eight columns at a
      // time through the warp's 1 KB of shared memory: row r's eight floats
      // go to slot s(r) (r with its low two bits rotated by r / 8) with the
      // two 16-byte halves swapped when bit 2 of the slot is set, so both the
      // row-wise 16-byte writes and the column reads below hit 32 distinct
      // banks.  Lane l then takes column l % 8, rows 8 (l / 8) .. +7: amax
      // over its eight values and the three other lanes of the column, then
      // eight codes as one 8-byte store (the column's 32 codes are one sector).
      float* sf = reinterpret_cast<float*>(scratch);
      const uint32_t r_w = (uint32_t)lane;
      const uint32_t slot_w = (r_w & ~3u) | ((r_w + (r_w >> 3)) & 3u);
      const uint32_t half_w = (slot_w >> 2) & 1u;
      const int cc = lane & 7, rg = lane >> 3;
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        float4* dst = reinterpret_cast<float4*>(sf + slot_w * 8);
        dst[half_w] = make_float4(y[8 * c8 + 0], y[8 * c8 + 1], y[8 * c8 + 2], y[8 * c8 + 3]);
        dst[half_w ^ 1u] = make_float4(y[8 * c8 + 4], y[8 * c8 + 5], y[8 * c8 + 6], y[8 * c8 + 7]);
        __syncwarp();
        float v[8];
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t r = (uint32_t)(8 * rg + i);
          const uint32_t sr = (r & ~3u) | ((r + (r >> 3)) & 3u);
          v[i] = sf[sr * 8 + ((uint32_t)cc ^ (((sr >> 2) & 1u) << 2))];
          m = max(m, abs_bits(v[i]));
        }
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
        const uint32_t sb = e8m0_from_amax_bits(m);
        uint32_t w0 = 0x7F7F7F7Fu, w1 = 0x7F7F7F7Fu;
        if (sb != 0xFFu) {
          const float inv = mx_inv_scale(sb);
          w0 = e4m3x2(v[0] * inv, v[1] * inv) | (e4m3x2(v[2] * inv, v[3] * inv) << 16);
          w1 = e4m3x2(v[4] * inv, v[5] * inv) | (e4m3x2(v[6] * inv, v[7] * inv) << 16);
        }
        const size_t col = (size_t)(col0 + 8 * c8 + cc);
        *reinterpret_cast<uint2*>(a.q_col + col * a.R_cap + rb + 8 * rg) = make_uint2(w0, w1);
        if (rg == 0) a.s_col[col * (a.R_cap / 32) + rb / 32] = (uint8_t)sb;
        __syncwarp();
      }
    }
  } else {
    if (row_ok) {
      uint4* dst = reinterpret_cast<uint4*>(a.y + (size_t)row * N + col0);
#pragma unroll
      for (int w = 0; w < 4; ++w)
        dst[w] = make_uint4(pack_bf16x2(y[8 * w], y[8 * w + 1]), pack_bf16x2(y[8 * w + 2], y[8 * w + 3]),
                            pack_bf16x2(y[8 * w + 4], y[8 * w + 5]), pack_bf16x2(y[8 * w + 6], y[8 * w + 7]));
    }
    if (a.out_mode == MOE_OUT_NVFP4) {
#pragma unroll
      for (int i = 0; i < 32; ++i) amax_bits.plain = max(amax_bits.plain, abs_bits(y[i]));
      if (a.rht_amax != nullptr) {
        // Transposed random Hadamard rotation of the bf16 values written: the
        // warp's rows are its lanes and a 16-row block is lanes 0-15 or 16-31,
        // so H16 diag(s) per column is four xor-butterflies across the lanes
        // (Sylvester order), then the 1/4 normalisation.
        const float sg = ((a.rht_signs >> (lane & 15)) & 1u) ? -1.0f : 1.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float x = __bfloat162float(__float2bfloat16_rn(y[i])) * sg;
#pragma unroll
          for (int m = 1; m < 16; m <<= 1) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, x, m);
            x = (lane & m) ? (o - x) : (x + o);
          }
          amax_bits.rht = max(amax_bits.rht, abs_bits(x * 0.25f));
        }
      }
    }
  }
}

__device__ __forceinline__ void load_bf16x32(const uint16_t* p, float* v) {
  const uint4* s = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint4 q = __ldg(s + w);
    v[8 * w + 0] = bf16_lo(q.x);
    v[8 * w + 1] = bf16_hi(q.x);
    v[8 * w + 2] = bf16_lo(q.y);
    v[8 * w + 3] = bf16_hi(q.y);
    v[8 * w + 4] = bf16_lo(q.z);
    v[8 * w + 5] = bf16_hi(q.z);
    v[8 * w + 6] = bf16_lo(q.w);
    v[8 * w + 7] = bf16_hi(q.w);
  }
}

__device__ __forceinline__ void store_bf16x32(uint16_t* p, const float* v, bool zero) {
  uint4* d = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    if (zero) {
      d[w] = make_uint4(0, 0, 0, 0);
    } else {
      d[w] = make_uint4(pack_bf16x2(v[8 * w], v[8 * w + 1]), pack_bf16x2(v[8 * w + 2], v[8 * w + 3]),
                        pack_bf16x2(v[8 * w + 4], v[8 * w + 5]), pack_bf16x2(v[8 * w + 6], v[8 * w + 7]));
    }
  }
}

// Transposed output stage, for tiles whose accumulator holds one output
// column per thread and 32 consecutive rows rb .. rb+31 in c[0..31] (the
// lanes of the warp are 32 consecutive columns, col - lane .. col - lane + 31).
// Row-wise MXFP8 blocks are the warp's 32 columns of one row (amax by a warp
// max), column-wise blocks are the thread's own 32 values.  The outputs are
// the same as emit_block's for the same values (codes decided from fp32 with
// the same scale rule); rows rb .. rb+31 must lie inside the padded segment.
template <class Out>
__device__ __forceinline__ void emit_block_t(const Out& a, const float* c, int col, int rb, int lane, Amax& amax_bits) {
  const int N = a.out_N;
  if (a.out_mode == MOE_OUT_MXFP8) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, abs_bits(c[j]));
      const uint32_t sb = e8m0_from_amax_bits(m);
      const uint32_t code = sb == 0xFFu ? 0x7Fu : (e4m3x2(c[j] * mx_inv_scale(sb), 0.0f) & 0xFFu);
      a.q_row[(size_t)(rb + j) * N + col] = (uint8_t)code;
      if (lane == 0) a.s_row[(size_t)(rb + j) * (N / 32) + (col - lane) / 32] = (uint8_t)sb;
    }
    if (a.q_col != nullptr) {
      uint32_t codes[8];
      const uint32_t sb = mx_quant_block32(c, codes);
      uint4* dst = reinterpret_cast<uint4*>(a.q_col + (size_t)col * a.R_cap + rb);
      dst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
      dst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
      a.s_col[(size_t)col * (a.R_cap / 32) + rb / 32] = (uint8_t)sb;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      a.y[(size_t)(rb + j) * N + col] = __bfloat16_as_ushort(__float2bfloat16_rn(c[j]));
    if (a.out_mode == MOE_OUT_NVFP4) {
#pragma unroll
      for (int j = 0; j < 32; ++j) amax_bits.plain = max(amax_bits.plain, abs_bits(c[j]));
      if (a.rht_amax != nullptr) {
        // transposed random Hadamard rotation of the bf16 values written:
        // the 16-row blocks are this thread's c[0..15] and c[16..31], so
        // H16 diag(s) is an in-register butterfly (Sylvester order), then /4
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          float x[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            x[i] = __bfloat162float(__float2bfloat16_rn(c[16 * b + i])) * (((a.rht_signs >> i) & 1u) ? -1.0f : 1.0f);
#pragma unroll
          for (int m = 1; m < 16; m <<= 1) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              if (i & m) continue;
              const float lo = x[i], hi = x[i + m];
              x[i] = lo + hi;
              x[i + m] = lo - hi;
            }
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) amax_bits.rht = max(amax_bits.rht, abs_bits(x[i] * 0.25f));
        }
      }
    }
  }
}

// Column sums of a warp's 32 x 32 block (lane = row, x[c] = column c of the
// lane's row): returns, in lane c, the sum over the 32 rows of column c.  A
// reduce-scatter by halving (the lanes that differ in bit m swap the halves
// they do not keep), so every addition happens in a fixed order and the
// result is deterministic; 31 shuffles per block.
__device__ __forceinline__ float warp_column_sum32(const float* x, int lane) {
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = x[i];
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < m; ++i) {
      const float keep = up ? v[i + m] : v[i];
      const float send = up ? v[i] : v[i + m];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, m);
    }
  }
  return v[0];
}

}  // namespace moeglu
