// Standalone memory-bound kernels around the fused GEMMs:
//   k_quant_rows / k_quant_cols  MXFP8 quantisation of a bf16 tensor along its
//                                rows or (transposed) columns: the weight
//                                casts, the column-wise copies the weight-
//                                gradient GEMMs read, and the quantize step
//                                of the unfused path
//   k_nvfp4_cast                 NVFP4 cast after the forward's bf16 + amax
//                                output
//   k_glu_act                    activation of the unfused path
// ([MoE-Fusion] "Boosting MoE Training Throughput with Advanced Fusion
// Kernels", "Fusing MXFP8 and NVFP4 quantisation": MXFP8 = row-wise output
// plus a transposed copy; NVFP4 = bf16 output plus per-tensor amax.
// [MegaMoE] §2.3: E4M3 elements with per-block scales.)
#include "common.cuh"
#include "host_common.h"

namespace moeglu {

constexpr int QE_MAX = 1024;

// Number of real rows (0..32) of the 32-row block starting at r0, given the
// expert segment map in shared memory; -1 if r0 >= offsets[E].
__device__ __forceinline__ int block_real_rows(int r0, const int32_t* s_off, const int32_t* s_cnt, int E) {
  if (r0 >= s_off[E]) return -1;
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_off[mid] <= r0) lo = mid; else hi = mid - 1;
  }
  return max(0, min(32, s_off[lo] + s_cnt[lo] - r0));
}

__device__ __forceinline__ void load_seg(const int32_t* counts, const int32_t* offsets, int E, int32_t* s_off,
                                         int32_t* s_cnt) {
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    s_off[e] = offsets[e];
    if (e < E) s_cnt[e] = counts[e];
  }
  __syncthreads();
}

// Row-wise.  The blocks of src [G][R][C] are contiguous runs of 32 elements,
// so the tensor is streamed flat: a warp task is QR_TASK consecutive blocks;
// in each of its QR_TASK / 8 loads a lane holds 8 elements (16 bytes) of
// block 8u + lane / 4, the 4 lanes of a block combine their amax with two
// shuffles, and every load and store instruction of the warp covers
// contiguous memory (512 bytes in, 256 bytes of codes out).  Rows >=
// offsets[E] are untouched; rows of an expert past its count quantise as 0.
constexpr int QR_TASK = 64;
constexpr int QR_LOADS = QR_TASK / 8;

__global__ void __launch_bounds__(256, 1) k_quant_rows(const uint16_t* __restrict__ src, int G, int R, int Cc,
                                                    const int32_t* __restrict__ counts,
                                                    const int32_t* __restrict__ offsets, int E,
                                                    uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
  extern __shared__ int32_t seg[];  // s_off [E + 1], s_cnt [E]
  int32_t* s_off = seg;
  int32_t* s_cnt = seg + E + 1;
  if (E > 0) load_seg(counts, offsets, E, s_off, s_cnt);
  const int lane = threadIdx.x & 31, quarter = lane & 3;
  const int nb = Cc / 32;
  const size_t nblocks = (size_t)G * R * nb;
  const size_t tasks = (nblocks + QR_TASK - 1) / QR_TASK;
  const size_t nwarps = ((size_t)gridDim.x * blockDim.x) >> 5;
  for (size_t task = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; task < tasks; task += nwarps) {
    uint4 x[QR_LOADS];
    bool keep[QR_LOADS];
#pragma unroll
    for (int u = 0; u < QR_LOADS; ++u) {
      const size_t blk = task * QR_TASK + 8 * u + (lane >> 2);
      keep[u] = blk < nblocks;
      bool zero = false;
      if (E > 0 && keep[u]) {
        const int r = (int)(blk / nb);
        const int real = block_real_rows(r & ~31, s_off, s_cnt, E);
        keep[u] = real >= 0;
        zero = (r & 31) >= real;
      }
      x[u] = make_uint4(0, 0, 0, 0);
      if (keep[u] && !zero) x[u] = __ldg(reinterpret_cast<const uint4*>(src + blk * 32 + quarter * 8));
    }
#pragma unroll
    for (int u = 0; u < QR_LOADS; ++u) {
      const float v[8] = {bf16_lo(x[u].x), bf16_hi(x[u].x), bf16_lo(x[u].y), bf16_hi(x[u].y),
                          bf16_lo(x[u].z), bf16_hi(x[u].z), bf16_lo(x[u].w), bf16_hi(x[u].w)};
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = max(m, abs_bits(v[i]));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      const uint32_t sb = e8m0_from_amax_bits(m);
      uint2 c = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
      if (sb != 0xFFu) {
        const float inv = mx_inv_scale(sb);
        c.x = e4m3x2(v[0] * inv, v[1] * inv) | (e4m3x2(v[2] * inv, v[3] * inv) << 16);
        c.y = e4m3x2(v[4] * inv, v[5] * inv) | (e4m3x2(v[6] * inv, v[7] * inv) << 16);
      }
      if (keep[u]) {
        const size_t blk = task * QR_TASK + 8 * u + (lane >> 2);
        *reinterpret_cast<uint2*>(q + blk * 32 + quarter * 8) = c;
        if (quarter == 0) s[blk] = (uint8_t)sb;
      }
    }
  }
}

// Column-wise (transposed).  A CTA streams tiles of 128 rows (four MX blocks
// along R) x 128 columns through a ring of QC_STAGES shared-memory buffers
// filled by TMA (thread 0 issues; completion on one mbarrier per buffer):
//   1. thread (column pair c, c + 1, block b) reads the two columns in rows
//      32b..32b+31 of the staged tile as one 32-bit word per row (consecutive
//      lanes read consecutive words: no bank conflicts), takes both amaxes at
//      once as a packed 16-bit max of the bf16 magnitudes (the float amax is
//      that value shifted left by 16), quantises both columns and writes
//      their 32 + 32 codes into a [128][128]-byte code tile;
//   2. the buffer is refilled with the tile QC_STAGES steps ahead;
//   3. each column's 128 codes leave as one full 128-byte line (8 lanes x 16
//      bytes, 4 columns per warp instruction), its 4 scales as bytes.
// Rows past R or columns past C arrive as zeros from TMA and are not stored.
constexpr int QC_ROWS = 128, QC_COLS = 128, QC_STAGES = 2;
constexpr int QC_TILE = QC_ROWS * QC_COLS * 2;  // bytes of one staged bf16 tile (128-byte rows)
constexpr int QC_CODE_ROW = QC_ROWS + 16;       // padded bytes per staged code column
constexpr int QC_OFF_CODE = QC_STAGES * QC_TILE;
constexpr int QC_OFF_SCALE = QC_OFF_CODE + QC_COLS * QC_CODE_ROW;
constexpr int QC_OFF_BARS = QC_OFF_SCALE + QC_COLS * 4;
constexpr int QC_OFF_MISC = QC_OFF_BARS + QC_STAGES * 8;  // real_rows[2][4], abort flag
constexpr int QC_OFF_SEG = QC_OFF_MISC + 48;
constexpr int QC_SMEM_BASE = QC_OFF_SEG;                  // + (2E + 1) ints of expert map

// ROWS: the same pass also writes the row-wise copy (q_row [G][R][C],
// s_row [G][R][C/32]) from the staged tile: four lanes per 32-element block,
// 8 elements (one 16-byte shared-memory load) each, two rows per warp
// instruction (512 contiguous bytes: no bank conflicts), 8-byte code stores
// that join into whole 128-byte lines.  One read of a weight then feeds both
// of its MXFP8 copies (along C for one GEMM, along R for another).
// s_tiled: the scales leave in the order the block-scaled GEMM's tensor-core
// copies read them when this tensor is its N x K weight operand (N = C, K =
// R): [G][ceil(C/256)][ceil(R/128)][2][512 bytes], the 512 bytes of one
// (128-row group of C, 128-element k-block of R) holding at byte
// 16 l + 4 j + i the scale of row 32 j + l of the group, sub-block i.  A
// staged tile is exactly one such block.
template <bool ROWS>
__global__ void __launch_bounds__(256) k_quant_cols(const __grid_constant__ CUtensorMap tm, int G, int R, int Cc,
                                                    const int32_t* __restrict__ counts,
                                                    const int32_t* __restrict__ offsets, int E,
                                                    uint8_t* __restrict__ q, uint8_t* __restrict__ s,
                                                    uint8_t* __restrict__ q_row, uint8_t* __restrict__ s_row,
                                                    int s_tiled, int32_t* status, uint64_t wait_ns) {
  extern __shared__ __align__(128) uint8_t qsm[];
  uint8_t* tin = qsm;
  uint8_t* tcode = qsm + QC_OFF_CODE;
  uint8_t* tscale = qsm + QC_OFF_SCALE;
  uint64_t* full = reinterpret_cast<uint64_t*>(qsm + QC_OFF_BARS);
  int* real_rows = reinterpret_cast<int*>(qsm + QC_OFF_MISC);  // [2][4]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(qsm + QC_OFF_MISC + 32);
  int32_t* s_off = reinterpret_cast<int32_t*>(qsm + QC_OFF_SEG);
  int32_t* s_cnt = s_off + E + 1;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (t == 0) {
    for (int st = 0; st < QC_STAGES; ++st) mbar_init(full + st, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm);
  }
  if (E > 0) load_seg(counts, offsets, E, s_off, s_cnt);  // (ends with a barrier)
  __syncthreads();
  const int col_tiles = (Cc + QC_COLS - 1) / QC_COLS;
  // grouped rows: only the tiles that hold rows < offsets[E]
  const int rows_used = E > 0 ? max(0, min(R, s_off[E])) : R;
  const int row_tiles = (rows_used + QC_ROWS - 1) / QC_ROWS;
  const int total = G * row_tiles * col_tiles;
  const int nblk = R / 32;
  auto block_real = [&](int rb) -> int {  // real rows of the 32-row block at rb; -1: none stored
    int real = rb < R ? 32 : -1;
    if (E > 0 && real >= 0) real = block_real_rows(rb, s_off, s_cnt, E);
    return real;
  };
  auto coords = [&](int i, int& g, int& r0, int& c0) {
    const int ct = i % col_tiles;
    const int rest = i / col_tiles;
    r0 = (rest % row_tiles) * QC_ROWS;
    g = rest / row_tiles;
    c0 = ct * QC_COLS;
  };
  auto issue = [&](int i, int st) {
    int g, r0, c0;
    coords(i, g, r0, c0);
    mbar_arrive_expect_tx(full + st, QC_TILE);
    tma_load_3d(tin + st * QC_TILE, &tm, full + st, c0, r0, g);
  };
  // step j of this CTA handles tile blockIdx.x + j * gridDim.x in buffer j % QC_STAGES;
  // its load is issued at step j - QC_STAGES (steps 0..QC_STAGES-1: here)
  if (t == 0) {
#pragma unroll
    for (int st = 0; st < QC_STAGES; ++st) {
      const int i = blockIdx.x + st * gridDim.x;
      if (i < total) issue(i, st);
    }
  }
  WaitGuard guard{abort_flag, status, wait_ns};
  int k = 0;
  for (int i = blockIdx.x; i < total; i += gridDim.x, ++k) {
    const int st = k % QC_STAGES;
    const uint32_t ph = (uint32_t)(k / QC_STAGES) & 1u;
    int g, r0, c0;
    coords(i, g, r0, c0);
    int* rr = real_rows + 4 * (k & 1);
    if (t < 4) rr[t] = block_real(r0 + 32 * t);
    const bool ok = mbar_wait(full + st, ph, guard);
    if (__syncthreads_or(ok ? 0 : 1)) break;
    // 1. quantise: warp w -> block b = w / 2, columns 2p, 2p + 1 with
    //    p = (w % 2) * 32 + lane
    {
      const int b = warp >> 1;
      const int p = (warp & 1) * 32 + lane;
      const int real = rr[b];
      const uint8_t* src = tin + st * QC_TILE + (32 * b) * (QC_COLS * 2) + p * 4;
      uint32_t w[32];
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        w[j] = j < real ? *reinterpret_cast<const uint32_t*>(src + j * QC_COLS * 2) : 0u;
        m = __vmaxu2(m, w[j] & 0x7FFF7FFFu);
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        // column 2p + half: the low (half 0) or high bf16 of each word
        const uint32_t sb = e8m0_from_amax_bits(half ? (m & 0xFFFF0000u) : (m << 16));
        uint32_t codes[8];
        if (sb == 0xFFu) {
#pragma unroll
          for (int k8 = 0; k8 < 8; ++k8) codes[k8] = 0x7F7F7F7Fu;
        } else {
          const float inv = mx_inv_scale(sb);
#pragma unroll
          for (int k8 = 0; k8 < 8; ++k8) {
            float v4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t x = w[4 * k8 + e];
              v4[e] = __uint_as_float(half ? (x & 0xFFFF0000u) : (x << 16));
            }
            codes[k8] = e4m3x2(v4[0] * inv, v4[1] * inv) | (e4m3x2(v4[2] * inv, v4[3] * inv) << 16);
          }
        }
        const int cl = 2 * p + half;
        uint4* dc = reinterpret_cast<uint4*>(tcode + cl * QC_CODE_ROW + 32 * b);
        dc[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
        dc[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
        tscale[cl * 4 + b] = (uint8_t)sb;
      }
    }
    // 1b. row-wise copy (ROWS): warp w, pass it -> rows 2 (8 it + w) + (lane / 16),
    //     block (lane / 4) % 4, elements 8 (lane % 4) .. + 8 of it
    if constexpr (ROWS) {
      const int rsub = lane >> 4, blk = (lane >> 2) & 3, part = lane & 3;
#pragma unroll 2
      for (int it = 0; it < QC_ROWS / 16; ++it) {
        const int lr = 2 * (8 * it + warp) + rsub;
        const uint4 x = *reinterpret_cast<const uint4*>(tin + st * QC_TILE + lr * (QC_COLS * 2) + 64 * blk + 16 * part);
        uint32_t m = __vmaxu2(__vmaxu2(x.x & 0x7FFF7FFFu, x.y & 0x7FFF7FFFu), __vmaxu2(x.z & 0x7FFF7FFFu, x.w & 0x7FFF7FFFu));
        m = max(m & 0xFFFFu, m >> 16);
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        const uint32_t sb = e8m0_from_amax_bits(m << 16);
        uint2 c = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
        if (sb != 0xFFu) {
          const float inv = mx_inv_scale(sb);
          c.x = e4m3x2(bf16_lo(x.x) * inv, bf16_hi(x.x) * inv) | (e4m3x2(bf16_lo(x.y) * inv, bf16_hi(x.y) * inv) << 16);
          c.y = e4m3x2(bf16_lo(x.z) * inv, bf16_hi(x.z) * inv) | (e4m3x2(bf16_lo(x.w) * inv, bf16_hi(x.w) * inv) << 16);
        }
        const int row = r0 + lr, col = c0 + 32 * blk;
        if (row < R && col < Cc) {
          const size_t rr = (size_t)g * R + row;
          *reinterpret_cast<uint2*>(q_row + rr * Cc + col + 8 * part) = c;
          if (part == 0) s_row[rr * (Cc / 32) + col / 32] = (uint8_t)sb;
        }
      }
    }
    __syncthreads();
    // 2. the buffer is free again: fetch the tile QC_STAGES steps ahead
    if (t == 0) {
      const int nxt = i + QC_STAGES * gridDim.x;
      if (nxt < total) issue(nxt, st);
    }
    // 3. store: lane group of 8 -> one column's 128 bytes; 4 columns per warp pass
    {
      const int sub = lane >> 3, part = lane & 7;
      const bool whole = r0 + QC_ROWS <= R;
#pragma unroll
      for (int h = 0; h < QC_COLS / 32; ++h) {
        const int cl = warp * (QC_COLS / 8) + h * 4 + sub;
        const int c = c0 + cl;
        if (c < Cc) {
          const uint4 val = *reinterpret_cast<const uint4*>(tcode + cl * QC_CODE_ROW + part * 16);
          uint8_t* dst = q + ((size_t)g * Cc + c) * R + r0 + part * 16;
          if (whole || r0 + part * 16 < R) *reinterpret_cast<uint4*>(dst) = val;
          if (!s_tiled && part < 4 && rr[part] >= 0)
            s[((size_t)g * Cc + c) * nblk + (r0 >> 5) + part] = tscale[cl * 4 + part];
        }
      }
      if (s_tiled && warp == 0) {  // the tile's 512-byte block: lane l writes bytes 16 l .. 16 l + 15
        const int nt = (Cc + 255) / 256, kbs = (R + 127) / 128, gi = c0 / QC_COLS;
        const uint32_t* ts = reinterpret_cast<const uint32_t*>(tscale);
        uint8_t* dst = s + ((((size_t)g * nt + (gi >> 1)) * kbs + r0 / QC_ROWS) * 2 + (gi & 1)) * 512;
        reinterpret_cast<uint4*>(dst)[lane] = make_uint4(ts[lane], ts[32 + lane], ts[64 + lane], ts[96 + lane]);
      }
    }
  }
  // after a timeout at step k: the loads of steps k .. k + QC_STAGES - 1 were
  // issued and not consumed; let them land before the CTA exits
  if (t == 0 && *abort_flag) {
    volatile int never = 0;
    WaitGuard drain{&never, status, 100000000ull};
    for (int j = k; j < k + QC_STAGES; ++j)
      if (blockIdx.x + j * gridDim.x < total) mbar_wait(full + j % QC_STAGES, (uint32_t)(j / QC_STAGES) & 1u, drain);
  }
}

// Eight fp32 values (a.x, a.y, b.x, ... d.y) to E2M1, round to nearest even
// with saturation, packed element 2i in the low nibble of byte i: each
// cvt...e2m1x2 puts its first source operand in the high nibble, and the
// four bytes are joined by one vector move.
__device__ __forceinline__ uint32_t e2m1x8(float2 a, float2 b, float2 c, float2 d) {
  uint32_t r;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(r)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y), "f"(d.x), "f"(d.y));
  return r;
}

// One NVFP4 block of 16 values under the per-tensor scale sg: returns the
// E4M3 block-scale byte and writes the 16 E2M1 codes (element 2i in the low
// nibble of byte i) to w[0..1].  s_b = E4M3(fp32(amax_b / 6) * sg),
// q = E2M1(fp32(v * fp32(sg / s_b))), each step one fp32 operation.  The
// block is pre * v[0..15] with pre a power of two (the 1/4 of the Hadamard
// rotation): scaling by it is exact, so it is applied to the block amax and
// to the quantisation multiplier instead of to each value.
// inv_tab (optional): the multiplier of every scale code, inv_tab[c] =
// fp32(sg / s_b(c)) * pre (0 where s_b(c) is 0 or NaN), made once per CTA by
// nvfp4_inv_table; the same values as computed here, without a divide per block.
__device__ __forceinline__ uint32_t nvfp4_block16(const float* v, float sg, uint32_t* w, float pre = 1.0f,
                                                  const float* inv_tab = nullptr) {
  float ab = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) ab = fmaxf(ab, fabsf(v[j]));
  ab *= pre;
  const float sbf = (ab / 6.0f) * sg;
  const __nv_fp8_storage_t sc = __nv_cvt_float_to_fp8(sbf, __NV_SATFINITE, __NV_E4M3);
  float inv;
  if (inv_tab != nullptr) {
    inv = inv_tab[sc & 0x7Fu];
  } else {
    const float sbv = __half2float(__half(__nv_cvt_fp8_to_halfraw(sc, __NV_E4M3)));
    inv = (sbv > 0.0f ? sg / sbv : 0.0f) * pre;
  }
  float2 x[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) x[k] = __fmul2_rn(make_float2(v[2 * k], v[2 * k + 1]), make_float2(inv, inv));
  w[0] = e2m1x8(x[0], x[1], x[2], x[3]);
  w[1] = e2m1x8(x[4], x[5], x[6], x[7]);
  return (uint32_t)sc;
}

__device__ __forceinline__ float nvfp4_global_scale(float am) {
  return (am > 0.0f && am <= 3.402823466e38f) ? 2688.0f / am : 1.0f;
}

// The quantisation multiplier of each of the 128 non-negative E4M3 scale
// codes (the block amax is never negative, so the sign bit stays clear):
// tab[c] = fp32(sg / s_b(c)) * pre, 0 for s_b(c) = 0 and for the NaN code.
// Filled by threads 0..127 of the CTA; the caller synchronises after.
__device__ __forceinline__ void nvfp4_inv_table(float* tab, float sg, float pre) {
  if (threadIdx.x < 128) {
    const float sbv = __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)threadIdx.x, __NV_E4M3)));
    tab[threadIdx.x] = (sbv > 0.0f ? sg / sbv : 0.0f) * pre;
  }
}

// Rows [row0, row0 + 16) of CPT adjacent columns c, c + 1, ... of src [.][C]
// bf16 as fp32.  CPT = 2 (c and C even, src 4-byte aligned): one 32-bit load
// per row, so a warp's loads of one row cover 128 contiguous bytes.
template <int CPT>
__device__ __forceinline__ void load_cols16(const uint16_t* __restrict__ src, int C, size_t row0, int c,
                                            float (&v)[CPT][16]) {
  const uint16_t* p = src + row0 * C + c;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if constexpr (CPT == 2) {
      const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(p + (size_t)j * C));
      v[0][j] = __uint_as_float(w << 16);
      v[1][j] = __uint_as_float(w & 0xFFFF0000u);
    } else {
      v[0][j] = __uint_as_float((uint32_t)__ldg(p + (size_t)j * C) << 16);
    }
  }
}

// BPT blocks' codes (8 bytes each) and scales of one column at q_col / s_col
// (the column's rows of q [.][R/2] and s [.][R/16], offset to the first block).
template <int BPT>
__device__ __forceinline__ void store_col_blocks(uint8_t* q_col, uint8_t* s_col, const uint32_t* w, uint32_t sc4,
                                                 int nblk) {
  if (BPT == 4 && nblk == 4) {
    reinterpret_cast<uint4*>(q_col)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(q_col)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    *reinterpret_cast<uint32_t*>(s_col) = sc4;
  } else {
    for (int b = 0; b < nblk; ++b) {
      *reinterpret_cast<uint2*>(q_col + 8 * b) = make_uint2(w[2 * b], w[2 * b + 1]);
      s_col[b] = (uint8_t)(sc4 >> (8 * b));
    }
  }
}

// Column-wise NVFP4 (the K-major copy of a weight whose contraction runs
// along its rows): src [G][R][C] bf16 -> q [G][C][R/2], s [G][C][R/16].  One
// thread per (g, BPT consecutive 16-row blocks, CPT adjacent columns);
// neighbouring threads take neighbouring columns, so each row load is
// coalesced, and with BPT = 4 a thread's codes of a column are one whole
// 32-byte sector of its output row.
template <int BPT, int CPT>
__global__ void __launch_bounds__(256) k_nvfp4_cast_cols(const uint16_t* __restrict__ src, int G, int R, int C,
                                                         const float* __restrict__ amax, uint8_t* __restrict__ q,
                                                         uint8_t* __restrict__ s, float* __restrict__ s_global) {
  const float sg = nvfp4_global_scale(*amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) *s_global = sg;
  const int nb = R / 16, ng = nb / BPT, ncp = C / CPT;
  const size_t total = (size_t)G * ng * ncp;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % ncp) * CPT;
    const size_t rest = i / ncp;
    const int rg = (int)(rest % ng);
    const int g = (int)(rest / ng);
    uint32_t w[CPT][2 * BPT];
    uint32_t sc4[CPT];
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) sc4[cc] = 0;
#pragma unroll
    for (int b = 0; b < BPT; ++b) {
      float v[CPT][16];
      load_cols16<CPT>(src + (size_t)g * R * C, C, (size_t)(rg * BPT + b) * 16, c, v);
#pragma unroll
      for (int cc = 0; cc < CPT; ++cc) sc4[cc] |= nvfp4_block16(v[cc], sg, w[cc] + 2 * b) << (8 * b);
    }
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) {
      const size_t col = (size_t)g * C + c + cc;
      store_col_blocks<BPT>(q + col * (R / 2) + (size_t)rg * BPT * 8, s + col * nb + (size_t)rg * BPT, w[cc],
                            sc4[cc], BPT);
    }
  }
}

// Transposed random Hadamard rotation of one 16-row block of one column, in
// place: v <- H16 diag(s) v / 4 (s_i = -1 where bit i of signs is set;
// Sylvester order), on fp32 values of bf16 inputs.  The same butterfly as
// the dGLU epilogue's rotated amax.
__device__ __forceinline__ void hadamard16_unscaled(float* v) {  // v <- H16 v
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & m) continue;
      const float lo = v[i], hi = v[i + m];
      v[i] = lo + hi;
      v[i + m] = lo - hi;
    }
  }
}

// The same butterfly on two columns at once (v[j] = row j of both), with the
// packed two-lane fp32 add; lo - hi as fma(hi, -1, lo), rounded once like
// the subtraction.
__device__ __forceinline__ void hadamard16_unscaled_x2(float2* v) {
  const float2 neg1 = make_float2(-1.0f, -1.0f);
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & m) continue;
      const float2 lo = v[i], hi = v[i + m];
      v[i] = __fadd2_rn(lo, hi);
      v[i + m] = __ffma2_rn(hi, neg1, lo);
    }
  }
}

__device__ __forceinline__ void rht16(float* v, uint32_t signs) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if ((signs >> i) & 1u) v[i] = -v[i];
  hadamard16_unscaled(v);
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] *= 0.25f;
}

// NVFP4 operand of the weight gradient: the rows of src [R_cap][C] (an
// activation or its gradient in the permuted layout) below offsets[E],
// rotated in 16-row blocks and cast column-wise: q [C][R_cap/2],
// s [C][R_cap/16] under s_g = 2688 / amax (amax = the rotated amax).  One
// thread per (4 consecutive 16-row blocks, CPT adjacent columns); blocks at
// or past offsets[E] are not written.
template <int CPT>
__global__ void __launch_bounds__(256) k_nvfp4_rht_cast_cols(const uint16_t* __restrict__ src, int R_cap, int C,
                                                             const int32_t* __restrict__ offsets, int E,
                                                             const float* __restrict__ amax, uint32_t signs,
                                                             uint8_t* __restrict__ q, uint8_t* __restrict__ s,
                                                             float* __restrict__ s_global) {
  const float sg = nvfp4_global_scale(*amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) *s_global = sg;
  const int R = min(__ldg(offsets + E), R_cap);
  const int nb = (R + 15) / 16, ng = (nb + 3) / 4, ncp = C / CPT;
  const size_t total = (size_t)ng * ncp;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % ncp) * CPT;
    const int rg = (int)(i / ncp);
    uint32_t w[CPT][8];
    uint32_t sc4[CPT];
    const int nblk = min(4, nb - rg * 4);
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) sc4[cc] = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      if (b < nblk) {
        float v[CPT][16];
        load_cols16<CPT>(src, C, (size_t)(rg * 4 + b) * 16, c, v);
#pragma unroll
        for (int cc = 0; cc < CPT; ++cc) {
          rht16(v[cc], signs);
          sc4[cc] |= nvfp4_block16(v[cc], sg, w[cc] + 2 * b) << (8 * b);
        }
      } else {
#pragma unroll
        for (int cc = 0; cc < CPT; ++cc) w[cc][2 * b] = w[cc][2 * b + 1] = 0;
      }
    }
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc)
      store_col_blocks<4>(q + (size_t)(c + cc) * (R_cap / 2) + (size_t)rg * 32,
                          s + (size_t)(c + cc) * (R_cap / 16) + (size_t)rg * 4, w[cc], sc4[cc], nblk);
  }
}

// max |rotated value| over the 16-row blocks below offsets[E] of every column
// (the per-tensor amax of k_nvfp4_rht_cast_cols' input), as ordered float
// bits.  One thread per (16-row block, CPT adjacent columns).
template <int CPT>
__global__ void __launch_bounds__(256) k_rht_amax_cols(const uint16_t* __restrict__ src, int R_cap, int C,
                                                       const int32_t* __restrict__ offsets, int E, uint32_t signs,
                                                       float* __restrict__ amax) {
  const int R = min(__ldg(offsets + E), R_cap);
  const int nb = (R + 15) / 16, ncp = C / CPT;
  const size_t total = (size_t)nb * ncp;
  uint32_t m = 0;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    float v[CPT][16];
    load_cols16<CPT>(src, C, (size_t)(i / ncp) * 16, (int)(i % ncp) * CPT, v);
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) {
      rht16(v[cc], signs);
#pragma unroll
      for (int j = 0; j < 16; ++j) m = max(m, __float_as_uint(v[cc][j]) & 0x7FFFFFFFu);
    }
  }
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if ((threadIdx.x & 31) == 0 && m != 0) atomicMax(reinterpret_cast<int*>(amax), (int)m);
}

// Column-wise NVFP4 through shared memory: the weight casts (NC_CAST) and
// the rotated operands of the weight gradient (NC_RHT_CAST, and their
// rotated amax, NC_RHT_AMAX).  A CTA streams tiles of 128 rows (eight 16-row
// blocks) x NC_COLS columns of src [G][R][C] through a ring of NC_STAGES
// buffers filled by TMA (thread 0 issues; one mbarrier per buffer); two
// independent (block, pair) items per thread give the ALU-heavy rotation and
// cast the instruction-level parallelism that hides their latencies:
//   1. thread (column pair p, block b) reads its two columns in the 16 rows
//      of a block as one 32-bit word per row (consecutive lanes read
//      consecutive words: no bank conflicts), rotates both columns (rotated
//      modes, both at once with packed two-lane fp32 adds) and casts them
//      into a [NC_COLS][64]-byte code tile and a [NC_COLS][8] scale tile,
//      or folds them into its amax (NC_RHT_AMAX);
//   2. the buffer is refilled with the tile NC_STAGES steps ahead;
//   3. each column's 64 code bytes leave as 4 x 16 bytes (8 columns per warp
//      instruction) and its 8 scales as one 8-byte word, or (TILED, weight
//      casts) the tile's scales as two 512-byte blocks in the order the
//      block-scaled GEMM's tensor-core copies read them, so that its call
//      has no weight scales to re-tile.
// Only the blocks below rows_valid (R, or offsets[E] for the permuted
// operands: a multiple of 32) are read into a result or stored; columns
// past C arrive as zeros from TMA and are not stored.  R % 128 == 0.
enum { NC_CAST = 0, NC_RHT_CAST = 1, NC_RHT_AMAX = 2 };
constexpr int NC_ROWS = 128, NC_COLS = 128, NC_STAGES = 3, NC_THREADS = 256, NC_CTAS_PER_SM = 2;
constexpr int NC_PAIRS = NC_COLS / 2;                          // column pairs of a tile row
constexpr int NC_ITEMS = (NC_ROWS / 16) * NC_PAIRS / NC_THREADS;  // (block, pair) items per thread
constexpr int NC_WARPS = NC_THREADS / 32;
constexpr int NC_TILE = NC_ROWS * NC_COLS * 2;   // bytes of one staged bf16 tile
constexpr int NC_CODE_ROW = NC_ROWS / 2 + 16;    // padded bytes per staged code column
constexpr int NC_OFF_CODE = NC_STAGES * NC_TILE;
constexpr int NC_OFF_SCALE = NC_OFF_CODE + NC_COLS * NC_CODE_ROW;
constexpr int NC_OFF_BARS = NC_OFF_SCALE + NC_COLS * 8;
constexpr int NC_OFF_MISC = NC_OFF_BARS + NC_STAGES * 8;  // abort flag
constexpr int NC_OFF_TAB = NC_OFF_MISC + 16;               // float [128]: nvfp4_inv_table
constexpr int NC_SMEM = NC_OFF_TAB + 128 * 4;

template <int MODE, bool TILED = false>
__global__ void __launch_bounds__(NC_THREADS, NC_CTAS_PER_SM) k_nvfp4_cols_tma(const __grid_constant__ CUtensorMap tm, int G, int R, int C,
                                                        const int32_t* __restrict__ offsets, int E,
                                                        const float* __restrict__ amax, uint32_t signs,
                                                        uint8_t* __restrict__ q, uint8_t* __restrict__ s,
                                                        float* __restrict__ s_global, float* __restrict__ amax_out,
                                                        int32_t* status, uint64_t wait_ns) {
  extern __shared__ __align__(128) uint8_t nsm[];
  uint8_t* tin = nsm;
  uint8_t* tcode = nsm + NC_OFF_CODE;
  uint8_t* tscale = nsm + NC_OFF_SCALE;
  uint64_t* full = reinterpret_cast<uint64_t*>(nsm + NC_OFF_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(nsm + NC_OFF_MISC);
  float* inv_tab = reinterpret_cast<float*>(nsm + NC_OFF_TAB);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  constexpr float pre = MODE == NC_CAST ? 1.0f : 0.25f;
  float sg = 1.0f;
  if constexpr (MODE != NC_RHT_AMAX) {
    sg = nvfp4_global_scale(*amax);
    if (blockIdx.x == 0 && t == 0) *s_global = sg;
    nvfp4_inv_table(inv_tab, sg, pre);
  }
  if (t == 0) {
    for (int st = 0; st < NC_STAGES; ++st) mbar_init(full + st, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm);
  }
  __syncthreads();
  const int rows_valid = offsets ? max(0, min(__ldg(offsets + E), R)) : R;
  const int col_tiles = (C + NC_COLS - 1) / NC_COLS;
  const int row_tiles = (rows_valid + NC_ROWS - 1) / NC_ROWS;
  const int total = G * row_tiles * col_tiles;
  auto coords = [&](int i, int& g, int& r0, int& c0) {
    c0 = (i % col_tiles) * NC_COLS;
    const int rest = i / col_tiles;
    r0 = (rest % row_tiles) * NC_ROWS;
    g = rest / row_tiles;
  };
  auto issue = [&](int i, int st) {
    int g, r0, c0;
    coords(i, g, r0, c0);
    mbar_arrive_expect_tx(full + st, NC_TILE);
    tma_load_3d(tin + st * NC_TILE, &tm, full + st, c0, r0, g);
  };
  if (t == 0) {
#pragma unroll
    for (int st = 0; st < NC_STAGES; ++st) {
      const int i = blockIdx.x + st * gridDim.x;
      if (i < total) issue(i, st);
    }
  }
  WaitGuard guard{abort_flag, status, wait_ns};
  const int p = t % NC_PAIRS, bq = t / NC_PAIRS;  // column pair; blocks bq + (NC_THREADS / NC_PAIRS) h
  // rotated modes: the sign of row j of a block flips both bf16 of the
  // packed word (s_j = -1 -> XOR 0x80008000); the butterfly then runs
  // without its 1/4, which is folded into the cast or the amax (exact)
  uint32_t smask[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) smask[j] = (MODE != NC_CAST && ((signs >> j) & 1u)) ? 0x80008000u : 0u;
  uint32_t m_abs = 0;
  int k = 0;
  for (int i = blockIdx.x; i < total; i += gridDim.x, ++k) {
    const int st = k % NC_STAGES;
    const uint32_t ph = (uint32_t)(k / NC_STAGES) & 1u;
    int g, r0, c0;
    coords(i, g, r0, c0);
    const int nvalid = min(8, (rows_valid - r0 + 15) / 16);
    const bool ok = mbar_wait(full + st, ph, guard);
    if (__syncthreads_or(ok ? 0 : 1)) break;
#pragma unroll
    for (int h = 0; h < NC_ITEMS; ++h) {
      const int b = bq + (NC_THREADS / NC_PAIRS) * h;
      if (b < nvalid) {
        const uint8_t* src = tin + st * NC_TILE + (16 * b) * (NC_COLS * 2) + p * 4;
        float2 v2[16];  // row j of the block: (column 2p, column 2p + 1)
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(src + j * NC_COLS * 2) ^ smask[j];
          v2[j] = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
        }
        if constexpr (MODE != NC_CAST) hadamard16_unscaled_x2(v2);
        float v[2][16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          v[0][j] = v2[j].x;
          v[1][j] = v2[j].y;
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          if constexpr (MODE == NC_RHT_AMAX) {
#pragma unroll
            for (int j = 0; j < 16; ++j) m_abs = max(m_abs, __float_as_uint(v[cc][j]) & 0x7FFFFFFFu);
          } else {
            uint32_t w2[2];
            const uint32_t sc = nvfp4_block16(v[cc], sg, w2, pre, inv_tab);
            const int cl = 2 * p + cc;
            *reinterpret_cast<uint2*>(tcode + cl * NC_CODE_ROW + 8 * b) = make_uint2(w2[0], w2[1]);
            tscale[cl * 8 + b] = (uint8_t)sc;
          }
        }
      }
    }
    __syncthreads();
    // 2. the buffer is free again: fetch the tile NC_STAGES steps ahead
    if (t == 0) {
      const int nxt = i + NC_STAGES * gridDim.x;
      if (nxt < total) issue(nxt, st);
    }
    // 3. store: lane group of 4 -> one column's 64 code bytes; 8 columns per warp pass
    if constexpr (MODE != NC_RHT_AMAX) {
      const int sub = lane >> 2, part = lane & 3;
#pragma unroll
      for (int h2 = 0; h2 < NC_COLS / (8 * NC_WARPS); ++h2) {
        const int cl = warp * (NC_COLS / NC_WARPS) + h2 * 8 + sub;
        const int c = c0 + cl;
        if (c < C) {
          const size_t col = (size_t)g * C + c;
          if (2 * part < nvalid)
            *reinterpret_cast<uint4*>(q + col * (R / 2) + r0 / 2 + part * 16) =
                *reinterpret_cast<const uint4*>(tcode + cl * NC_CODE_ROW + part * 16);
          if (part == 0 && !TILED) {
            uint8_t* sd = s + col * (R / 16) + r0 / 16;
            if (nvalid == 8)
              *reinterpret_cast<uint2*>(sd) = *reinterpret_cast<const uint2*>(tscale + cl * 8);
            else
              for (int b = 0; b < nvalid; ++b) sd[b] = tscale[cl * 8 + b];
          }
        }
      }
      if (TILED && warp == 0) {
        // the tile's scales in the block-scaled GEMM's order (rows R = K,
        // all valid): one 512-byte block per 64-row group of R, lane l
        // writing bytes 16 l .. 16 l + 15, byte 16 l + 4 j + i = the scale
        // of column 32 j + l of the 128-column group, sub-block i (column
        // cl's scales 4 q .. 4 q + 3 are 32-bit word 2 cl + q of tscale)
        const int nt = (C + 255) / 256, kgs = 4 * ((R + 255) / 256), gi = c0 / NC_COLS;
        const uint32_t* ts = reinterpret_cast<const uint32_t*>(tscale);
        uint8_t* base = s + ((size_t)g * nt + (gi >> 1)) * kgs * 1024 + (gi & 1) * 512;
        // groups past R in the last k-block of 256 and the missing half of a
        // last 256-column tile hold zero scales (their codes are zero too)
        const bool r_tail = r0 + NC_ROWS == R && (R % 256) != 0;
        const bool c_tail = (gi & 1) == 0 && c0 + NC_COLS >= C;
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q >= 2 && !r_tail) break;
          uint8_t* dst = base + (size_t)(r0 / 64 + q) * 1024;
          const uint4 v = q < 2 ? make_uint4(ts[2 * lane + q], ts[2 * (32 + lane) + q], ts[2 * (64 + lane) + q],
                                             ts[2 * (96 + lane) + q])
                                : zero;
          reinterpret_cast<uint4*>(dst)[lane] = v;
          if (c_tail) reinterpret_cast<uint4*>(dst + 512)[lane] = zero;
        }
      }
    }
  }
  if constexpr (MODE == NC_RHT_AMAX) {
    m_abs = __reduce_max_sync(0xFFFFFFFFu, m_abs);
    // the 1/4 of the rotation (exact; a NaN stays NaN, inf stays inf)
    m_abs = __float_as_uint(__uint_as_float(m_abs) * 0.25f);
    if (lane == 0 && m_abs != 0) atomicMax(reinterpret_cast<int*>(amax_out), (int)m_abs);
  }
  // after a timeout at step k: the loads of steps k .. k + NC_STAGES - 1 were
  // issued and not consumed; let them land before the CTA exits
  if (t == 0 && *abort_flag) {
    volatile int never = 0;
    WaitGuard drain{&never, status, 100000000ull};
    for (int j = k; j < k + NC_STAGES; ++j)
      if (blockIdx.x + j * gridDim.x < total) mbar_wait(full + j % NC_STAGES, (uint32_t)(j / NC_STAGES) & 1u, drain);
  }
}

// max |x| over a bf16 tensor of n8 16-byte words (x 16-byte aligned) into
// *amax as ordered float bits (the caller's call zeroes it first).
__global__ void __launch_bounds__(256, 1) k_amax_bf16(const uint4* __restrict__ x, size_t n8, float* __restrict__ amax) {
  uint32_t m = 0;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const uint4 w = __ldg(x + i);
    // magnitudes of the eight bf16 values, each half of a word on its own
    const uint32_t wv[4] = {w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu, w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu};
#pragma unroll
    for (int h = 0; h < 4; ++h) m = max(m, max(wv[h] & 0xFFFFu, wv[h] >> 16));
  }
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if ((threadIdx.x & 31) == 0 && m != 0) atomicMax(reinterpret_cast<int*>(amax), (int)(m << 16));
}

// NVFP4: one thread per 16-element block of a row < offsets[E].
__global__ void __launch_bounds__(256) k_nvfp4_cast(const uint16_t* __restrict__ y, const float* __restrict__ amax,
                                                    const int32_t* __restrict__ offsets, int E, int N,
                                                    uint8_t* __restrict__ q, uint8_t* __restrict__ s,
                                                    float* __restrict__ s_global) {
  const float sg = nvfp4_global_scale(*amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) *s_global = sg;
  const int R = __ldg(offsets + E);
  const int nb = N / 16;
  const size_t total = (size_t)R * nb;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const uint4* p = reinterpret_cast<const uint4*>(y + i * 16);
    const uint4 a = __ldg(p), b = __ldg(p + 1);
    float v[16] = {bf16_lo(a.x), bf16_hi(a.x), bf16_lo(a.y), bf16_hi(a.y), bf16_lo(a.z), bf16_hi(a.z),
                   bf16_lo(a.w), bf16_hi(a.w), bf16_lo(b.x), bf16_hi(b.x), bf16_lo(b.y), bf16_hi(b.y),
                   bf16_lo(b.z), bf16_hi(b.z), bf16_lo(b.w), bf16_hi(b.w)};
    uint32_t w[2];
    const uint32_t sc = nvfp4_block16(v, sg, w);
    *reinterpret_cast<uint2*>(q + i * 8) = make_uint2(w[0], w[1]);
    s[i] = (uint8_t)sc;
  }
}

// Eight bf16 values of one 16-byte word, widened to fp32.
__device__ __forceinline__ void unpack8(const uint4 w, float* v) {
  v[0] = bf16_lo(w.x);
  v[1] = bf16_hi(w.x);
  v[2] = bf16_lo(w.y);
  v[3] = bf16_hi(w.y);
  v[4] = bf16_lo(w.z);
  v[5] = bf16_hi(w.z);
  v[6] = bf16_lo(w.w);
  v[7] = bf16_hi(w.w);
}

// The activation forms the unfused kernels are instantiated for; LEAN follows
// GluParams::lean, so the two paths evaluate the same expressions.
template <int LEAN>
__device__ __forceinline__ float glu_fwd_form(const GluParams& p, float u, float g) {
  if constexpr (LEAN == 1) return swiglu_fwd_lean(p, u, g);
  else if constexpr (LEAN == 2) return swiglu_fwd_lean_clamped(p, u, g);
  else if constexpr (LEAN == 3) return geglu_fwd_lean(p, u, g);
  else return act_fwd(p, u, g);
}
template <int LEAN>
__device__ __forceinline__ void glu_bwd_form(const GluParams& p, float u, float g, float dy, float& du, float& dg) {
  if constexpr (LEAN == 1) swiglu_bwd_lean(p, u, g, dy, du, dg);
  else if constexpr (LEAN == 2) swiglu_bwd_lean_clamped(p, u, g, dy, du, dg);
  else if constexpr (LEAN == 3) geglu_bwd_lean(p, u, g, dy, du, dg);
  else act_bwd(p, u, g, dy, du, dg);
}

// Unfused activation: pre [R][N1] bf16 -> y [R][F] bf16, one thread per 32
// output columns of a row < offsets[E], 16-byte loads and stores.
template <int LEAN>
__global__ void __launch_bounds__(256) k_glu_act(const uint16_t* __restrict__ pre, const int32_t* __restrict__ offsets,
                                                 int E, int F, int N1, GluParams prm, uint16_t* __restrict__ y) {
  const int R = __ldg(offsets + E);
  const int nb = F / 32;
  const bool gated = N1 == 2 * F;
  const size_t total = (size_t)R * nb;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / nb;
    const int b = (int)(i - r * nb);
    const uint4* pr = reinterpret_cast<const uint4*>(pre + r * N1 + (gated ? b * 64 : b * 32));
    uint4 wu[4], wg[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) wu[w] = __ldg(pr + w);
    if (gated) {
#pragma unroll
      for (int w = 0; w < 4; ++w) wg[w] = __ldg(pr + 4 + w);
    } else {
#pragma unroll
      for (int w = 0; w < 4; ++w) wg[w] = make_uint4(0, 0, 0, 0);
    }
    uint4* d = reinterpret_cast<uint4*>(y + r * F + (size_t)b * 32);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float u[8], g[8], o[8];
      unpack8(wu[w], u);
      unpack8(wg[w], g);
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j] = glu_fwd_form<LEAN>(prm, u[j], g[j]);
      d[w] = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                        pack_bf16x2(o[6], o[7]));
    }
  }
}

// Unfused backward activation: da [R][F] bf16 (the data-gradient GEMM's
// output) and the saved pre-activation [R][N1] bf16 -> dFC1 [R][N1] bf16 in
// packed column order.  One thread per 32 columns of da of a row < offsets[E].
template <int LEAN>
__global__ void __launch_bounds__(256) k_dglu_act(const uint16_t* __restrict__ da, const uint16_t* __restrict__ pre,
                                                  const int32_t* __restrict__ offsets, int E, int F, int N1,
                                                  GluParams prm, uint16_t* __restrict__ d) {
  const int R = __ldg(offsets + E);
  const int nb = F / 32;
  const bool gated = N1 == 2 * F;
  const size_t total = (size_t)R * nb;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / nb;
    const int b = (int)(i - r * nb);
    const int pu = gated ? b * 64 : b * 32;
    const uint4* pr = reinterpret_cast<const uint4*>(pre + r * N1 + pu);
    const uint4* dr = reinterpret_cast<const uint4*>(da + r * F + (size_t)b * 32);
    uint4 wu[4], wg[4], wd[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      wu[w] = __ldg(pr + w);
      wd[w] = __ldg(dr + w);
    }
    if (gated) {
#pragma unroll
      for (int w = 0; w < 4; ++w) wg[w] = __ldg(pr + 4 + w);
    } else {
#pragma unroll
      for (int w = 0; w < 4; ++w) wg[w] = make_uint4(0, 0, 0, 0);
    }
    uint4 ou[4], og[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float u[8], g[8], dy[8], du[8], dg[8];
      unpack8(wu[w], u);
      unpack8(wg[w], g);
      unpack8(wd[w], dy);
#pragma unroll
      for (int j = 0; j < 8; ++j) glu_bwd_form<LEAN>(prm, u[j], g[j], dy[j], du[j], dg[j]);
      ou[w] = make_uint4(pack_bf16x2(du[0], du[1]), pack_bf16x2(du[2], du[3]), pack_bf16x2(du[4], du[5]),
                         pack_bf16x2(du[6], du[7]));
      og[w] = make_uint4(pack_bf16x2(dg[0], dg[1]), pack_bf16x2(dg[2], dg[3]), pack_bf16x2(dg[4], dg[5]),
                         pack_bf16x2(dg[6], dg[7]));
    }
    uint4* o = reinterpret_cast<uint4*>(d + r * N1 + pu);
#pragma unroll
    for (int w = 0; w < 4; ++w) o[w] = ou[w];
    if (gated) {
#pragma unroll
      for (int w = 0; w < 4; ++w) o[4 + w] = og[w];
    }
  }
}

static int grid_for(size_t items, int per_block) {
  const size_t g = (items + per_block - 1) / per_block;
  const size_t cap = (size_t)sm_count() * 16;
  return (int)(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace moeglu

using namespace moeglu;

extern "C" moe_status_t moe_quantize_mxfp8(const moe_bf16* src, int G, int R, int Cc, int col, const int32_t* counts,
                                           const int32_t* offsets, int E, uint8_t* q, uint8_t* s, int32_t* status,
                                           moe_stream_t stream) {
  if (!src || !q || !s || G <= 0 || R <= 0 || Cc <= 0) return MOE_ERR_ARG;
  if ((counts == nullptr) != (offsets == nullptr)) return MOE_ERR_ARG;
  if (counts && (G != 1 || E <= 0 || E > QE_MAX || (R % 32))) return MOE_ERR_ARG;
  if (!counts) E = 0;
  if (!aligned16(src) || !aligned16(q)) return MOE_ERR_ARG;
  cudaStream_t st = as_stream(stream);
  const int sms = sm_count();
  if (!col) {
    if (Cc % 32) return MOE_ERR_ARG;
    const int smem = E > 0 ? (2 * E + 1) * 4 : 0;
    const size_t tasks = ((size_t)G * R * (Cc / 32) + QR_TASK - 1) / QR_TASK;
    const int occ = max(1, max_active_blocks((const void*)k_quant_rows, 256, 2 * QE_MAX * 4 + 4));
    size_t grid = (tasks + 7) / 8;
    if (grid > (size_t)sms * occ) grid = (size_t)sms * occ;
    k_quant_rows<<<(int)(grid < 1 ? 1 : grid), 256, smem, st>>>(src, G, R, Cc, counts, offsets, E, q, s);
  } else {
    if ((R % 32) || (Cc % 8)) return MOE_ERR_ARG;
    if (col == 2 && (E > 0 || (reinterpret_cast<uintptr_t>(s) & 15))) return MOE_ERR_ARG;  // weights only
    const size_t tiles = (size_t)G * ((R + QC_ROWS - 1) / QC_ROWS) * ((Cc + QC_COLS - 1) / QC_COLS);
    if (tiles > (size_t)INT32_MAX) return MOE_ERR_ARG;
    CUtensorMap tm;
    const uint64_t dims[3] = {(uint64_t)Cc, (uint64_t)R, (uint64_t)G};
    const uint64_t strides[2] = {(uint64_t)Cc * 2, (uint64_t)R * Cc * 2};
    const uint32_t box[3] = {QC_COLS, QC_ROWS, 1};
    if (!encode_tmap(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, src, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return MOE_ERR_CUDA;
    const int smem = QC_SMEM_BASE + (2 * E + 1) * 4;
    const int smem_max = QC_SMEM_BASE + (2 * QE_MAX + 1) * 4;
    if (!set_smem_limit((const void*)k_quant_cols<false>, smem_max)) return MOE_ERR_CUDA;
    const int occ = max(1, max_active_blocks((const void*)k_quant_cols<false>, 256, smem_max));
    size_t grid = tiles;
    if (grid > (size_t)sms * occ) grid = (size_t)sms * occ;
    k_quant_cols<false><<<(int)(grid < 1 ? 1 : grid), 256, smem, st>>>(tm, G, R, Cc, counts, offsets, E, q, s,
                                                                      nullptr, nullptr, col == 2 ? 1 : 0, status,
                                                                      g_wait_limit_ns.load());
  }
  count_launch();
  return launch_status();
}

extern "C" size_t moe_mxfp8_tiled_scale_bytes(int G, int R, int C) {
  if (G <= 0 || R <= 0 || C <= 0) return 0;
  return (size_t)G * ((C + 255) / 256) * ((R + 127) / 128) * 1024;
}

extern "C" moe_status_t moe_quantize_mxfp8_dual(const moe_bf16* src, int G, int R, int Cc, uint8_t* q_row,
                                                uint8_t* s_row, uint8_t* q_col, uint8_t* s_col, int32_t* status,
                                                moe_stream_t stream) {
  if (!src || !q_row || !s_row || !q_col || !s_col || G <= 0 || R <= 0 || Cc <= 0) return MOE_ERR_ARG;
  if ((R % 32) || (Cc % 32) || !aligned16(src) || !aligned16(q_col) || (reinterpret_cast<uintptr_t>(q_row) & 7))
    return MOE_ERR_ARG;
  const size_t tiles = (size_t)G * ((R + QC_ROWS - 1) / QC_ROWS) * ((Cc + QC_COLS - 1) / QC_COLS);
  if (tiles > (size_t)INT32_MAX) return MOE_ERR_ARG;
  CUtensorMap tm;
  const uint64_t dims[3] = {(uint64_t)Cc, (uint64_t)R, (uint64_t)G};
  const uint64_t strides[2] = {(uint64_t)Cc * 2, (uint64_t)R * Cc * 2};
  const uint32_t box[3] = {QC_COLS, QC_ROWS, 1};
  if (!encode_tmap(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, src, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
    return MOE_ERR_CUDA;
  const int smem = QC_SMEM_BASE + 4;
  if (!set_smem_limit((const void*)k_quant_cols<true>, smem)) return MOE_ERR_CUDA;
  const int occ = max(1, max_active_blocks((const void*)k_quant_cols<true>, 256, smem));
  size_t grid = tiles;
  if (grid > (size_t)sm_count() * occ) grid = (size_t)sm_count() * occ;
  k_quant_cols<true><<<(int)(grid < 1 ? 1 : grid), 256, smem, as_stream(stream)>>>(
      tm, G, R, Cc, nullptr, nullptr, 0, q_col, s_col, q_row, s_row, 0, status, g_wait_limit_ns.load());
  count_launch();
  return launch_status();
}

extern "C" moe_status_t moe_nvfp4_cast(const moe_bf16* y, const float* amax, const int32_t* counts,
                                       const int32_t* offsets, int E, int N, int R_cap, uint8_t* q, uint8_t* s,
                                       float* s_global, moe_stream_t stream) {
  (void)counts;
  if (!y || !amax || !offsets || !q || !s || !s_global || E <= 0 || N <= 0 || (N % 16) || R_cap <= 0)
    return MOE_ERR_ARG;
  if (!aligned16(y) || (reinterpret_cast<uintptr_t>(q) & 7)) return MOE_ERR_ARG;
  k_nvfp4_cast<<<grid_for((size_t)R_cap * (N / 16), 256), 256, 0, as_stream(stream)>>>(y, amax, offsets, E, N, q, s,
                                                                                      s_global);
  count_launch();
  return launch_status();
}

extern "C" moe_status_t moe_amax_bf16(const moe_bf16* x, size_t n, float* amax, moe_stream_t stream) {
  if (!x || !amax || n == 0 || (n % 8) || !aligned16(x)) return MOE_ERR_ARG;
  cudaStream_t st = as_stream(stream);
  if (cudaMemsetAsync(amax, 0, sizeof(float), st) != cudaSuccess) return MOE_ERR_CUDA;
  k_amax_bf16<<<grid_for(n / 8, 256), 256, 0, st>>>(reinterpret_cast<const uint4*>(x), n / 8, amax);
  count_launch();
  return launch_status();
}

template <int MODE, bool TILED = false>
static moe_status_t launch_nvfp4_cols_tma(const moe_bf16* src, int G, int R, int C, const int32_t* offsets, int E,
                                          const float* amax, uint32_t signs, uint8_t* q, uint8_t* s, float* s_global,
                                          float* amax_out, int32_t* status, cudaStream_t st) {
  const size_t tiles = (size_t)G * ((R + NC_ROWS - 1) / NC_ROWS) * ((C + NC_COLS - 1) / NC_COLS);
  if (tiles > (size_t)INT32_MAX) return MOE_ERR_ARG;
  CUtensorMap tm;
  const uint64_t dims[3] = {(uint64_t)C, (uint64_t)R, (uint64_t)G};
  const uint64_t strides[2] = {(uint64_t)C * 2, (uint64_t)R * C * 2};
  const uint32_t box[3] = {NC_COLS, NC_ROWS, 1};
  if (!encode_tmap(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, src, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
    return MOE_ERR_CUDA;
  const void* fn = (const void*)k_nvfp4_cols_tma<MODE, TILED>;
  if (!set_smem_limit(fn, NC_SMEM)) return MOE_ERR_CUDA;
  const int occ = max(1, max_active_blocks(fn, NC_THREADS, NC_SMEM));
  size_t grid = tiles;
  if (grid > (size_t)sm_count() * occ) grid = (size_t)sm_count() * occ;
  k_nvfp4_cols_tma<MODE, TILED><<<(int)(grid < 1 ? 1 : grid), NC_THREADS, NC_SMEM, st>>>(
      tm, G, R, C, offsets, E, amax, signs, q, s, s_global, amax_out, status, g_wait_limit_ns.load());
  count_launch();
  return launch_status();
}

// The staged (TMA) form needs 16-byte rows and 128-row tiles; other shapes
// take the direct kernels (two adjacent columns per thread when C is even).
static bool nvfp4_cols_staged(const void* src, int R, int C) { return aligned16(src) && (C % 8) == 0 && (R % 128) == 0; }

extern "C" moe_status_t moe_nvfp4_cast_cols(const moe_bf16* src, int G, int R, int C, const float* amax, uint8_t* q,
                                            uint8_t* s, float* s_global, int32_t* status, moe_stream_t stream) {
  if (!src || !amax || !q || !s || !s_global || G <= 0 || R <= 0 || (R % 16) || C <= 0) return MOE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(q) & 7)) return MOE_ERR_ARG;
  cudaStream_t st = as_stream(stream);
  if (nvfp4_cols_staged(src, R, C) && aligned16(q) && (reinterpret_cast<uintptr_t>(s) & 7) == 0)
    return launch_nvfp4_cols_tma<NC_CAST>(src, G, R, C, nullptr, 0, amax, 0u, q, s, s_global, nullptr, status, st);
  // four blocks per thread (32-byte code stores, 4-byte scale stores) when
  // the rows come in 64s and the outputs are aligned for it
  const bool wide = (R % 64) == 0 && aligned16(q) && (reinterpret_cast<uintptr_t>(s) & 3) == 0;
  // two adjacent columns per thread (32-bit row loads) when C is even
  const bool pair = (C % 2) == 0 && (reinterpret_cast<uintptr_t>(src) & 3) == 0;
  const uint16_t* src16 = reinterpret_cast<const uint16_t*>(src);
  const size_t units = (size_t)G * (R / (wide ? 64 : 16)) * (C / (pair ? 2 : 1));
  if (wide && pair)
    k_nvfp4_cast_cols<4, 2><<<grid_for(units, 256), 256, 0, st>>>(src16, G, R, C, amax, q, s, s_global);
  else if (wide)
    k_nvfp4_cast_cols<4, 1><<<grid_for(units, 256), 256, 0, st>>>(src16, G, R, C, amax, q, s, s_global);
  else if (pair)
    k_nvfp4_cast_cols<1, 2><<<grid_for(units, 256), 256, 0, st>>>(src16, G, R, C, amax, q, s, s_global);
  else
    k_nvfp4_cast_cols<1, 1><<<grid_for(units, 256), 256, 0, st>>>(src16, G, R, C, amax, q, s, s_global);
  count_launch();
  return launch_status();
}

extern "C" size_t moe_nvfp4_tiled_scale_bytes(int G, int R, int C) {
  if (G <= 0 || R <= 0 || C <= 0) return 0;
  return (size_t)G * ((C + 255) / 256) * ((R + 255) / 256) * 4096;
}

extern "C" moe_status_t moe_nvfp4_cast_cols_tiled(const moe_bf16* src, int G, int R, int C, const float* amax,
                                                  uint8_t* q, uint8_t* s, float* s_global, int32_t* status,
                                                  moe_stream_t stream) {
  if (!src || !amax || !q || !s || !s_global || G <= 0 || R <= 0 || C <= 0) return MOE_ERR_ARG;
  if (!nvfp4_cols_staged(src, R, C) || !aligned16(q) || !aligned16(s)) return MOE_ERR_ARG;
  return launch_nvfp4_cols_tma<NC_CAST, true>(src, G, R, C, nullptr, 0, amax, 0u, q, s, s_global, nullptr, status,
                                              as_stream(stream));
}

extern "C" moe_status_t moe_rht_amax_cols(const moe_bf16* src, int R_cap, int C, const int32_t* offsets, int E,
                                          uint32_t signs, float* amax, int32_t* status, moe_stream_t stream) {
  if (!src || !offsets || !amax || R_cap <= 0 || (R_cap % 128) || C <= 0 || E <= 0) return MOE_ERR_ARG;
  cudaStream_t st = as_stream(stream);
  if (cudaMemsetAsync(amax, 0, sizeof(float), st) != cudaSuccess) return MOE_ERR_CUDA;
  if (nvfp4_cols_staged(src, R_cap, C))
    return launch_nvfp4_cols_tma<NC_RHT_AMAX>(src, 1, R_cap, C, offsets, E, nullptr, signs & 0xFFFFu, nullptr,
                                              nullptr, nullptr, amax, status, st);
  const uint16_t* src16 = reinterpret_cast<const uint16_t*>(src);
  if ((C % 2) == 0 && (reinterpret_cast<uintptr_t>(src) & 3) == 0)
    k_rht_amax_cols<2><<<grid_for((size_t)(R_cap / 16) * (C / 2), 256), 256, 0, st>>>(src16, R_cap, C, offsets, E,
                                                                                      signs & 0xFFFFu, amax);
  else
    k_rht_amax_cols<1><<<grid_for((size_t)(R_cap / 16) * C, 256), 256, 0, st>>>(src16, R_cap, C, offsets, E,
                                                                                signs & 0xFFFFu, amax);
  count_launch();
  return launch_status();
}

extern "C" moe_status_t moe_nvfp4_rht_cast_cols(const moe_bf16* src, int R_cap, int C, const int32_t* offsets, int E,
                                                const float* amax, uint32_t signs, uint8_t* q, uint8_t* s,
                                                float* s_global, int32_t* status, moe_stream_t stream) {
  if (!src || !offsets || !amax || !q || !s || !s_global || R_cap <= 0 || (R_cap % 128) || C <= 0 || E <= 0)
    return MOE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(s) & 3)) return MOE_ERR_ARG;
  cudaStream_t st = as_stream(stream);
  if (nvfp4_cols_staged(src, R_cap, C) && (reinterpret_cast<uintptr_t>(s) & 7) == 0)
    return launch_nvfp4_cols_tma<NC_RHT_CAST>(src, 1, R_cap, C, offsets, E, amax, signs & 0xFFFFu, q, s, s_global,
                                              nullptr, status, st);
  const uint16_t* src16 = reinterpret_cast<const uint16_t*>(src);
  if ((C % 2) == 0 && (reinterpret_cast<uintptr_t>(src) & 3) == 0)
    k_nvfp4_rht_cast_cols<2><<<grid_for((size_t)(R_cap / 64) * (C / 2), 256), 256, 0, st>>>(
        src16, R_cap, C, offsets, E, amax, signs & 0xFFFFu, q, s, s_global);
  else
    k_nvfp4_rht_cast_cols<1><<<grid_for((size_t)(R_cap / 64) * C, 256), 256, 0, st>>>(
        src16, R_cap, C, offsets, E, amax, signs & 0xFFFFu, q, s, s_global);
  count_launch();
  return launch_status();
}

extern "C" moe_status_t moe_glu_act(const moe_bf16* pre, const int32_t* counts, const int32_t* offsets, int E, int F,
                                    int R_cap, const moe_glu_params_t* params, moe_bf16* y, moe_stream_t stream) {
  (void)counts;
  if (!pre || !offsets || !params || !y || E <= 0 || F <= 0 || (F % 32) || R_cap <= 0) return MOE_ERR_ARG;
  if (!aligned16(y) || !aligned16(pre)) return MOE_ERR_ARG;
  const int act = params->act;
  if (act < MOE_ACT_SWIGLU || act > MOE_ACT_SREGLU) return MOE_ERR_ARG;
  GluParams g;
  g.act = act;
  g.alpha = params->alpha;
  g.up_offset = params->up_offset;
  g.gate_lo = params->gate_lo;
  g.gate_hi = params->gate_hi;
  g.up_lo = params->up_lo;
  g.up_hi = params->up_hi;
  g.lean = glu_lean_kind(params);
  g.nk = -params->alpha * 1.4426950408889634f;
  const int N1 = act == MOE_ACT_SRELU ? F : 2 * F;
  const int grid = grid_for((size_t)R_cap * (F / 32), 256);
  cudaStream_t st = as_stream(stream);
  if (g.lean == 1) k_glu_act<1><<<grid, 256, 0, st>>>(pre, offsets, E, F, N1, g, y);
  else if (g.lean == 2) k_glu_act<2><<<grid, 256, 0, st>>>(pre, offsets, E, F, N1, g, y);
  else if (g.lean == 3) k_glu_act<3><<<grid, 256, 0, st>>>(pre, offsets, E, F, N1, g, y);
  else k_glu_act<0><<<grid, 256, 0, st>>>(pre, offsets, E, F, N1, g, y);
  count_launch();
  return launch_status();
}

extern "C" moe_status_t moe_dglu_act(const moe_bf16* da, const moe_bf16* pre, const int32_t* counts,
                                     const int32_t* offsets, int E, int F, int R_cap, const moe_glu_params_t* params,
                                     moe_bf16* dfc1, moe_stream_t stream) {
  (void)counts;
  if (!da || !pre || !offsets || !params || !dfc1 || E <= 0 || F <= 0 || (F % 32) || R_cap <= 0) return MOE_ERR_ARG;
  if (!aligned16(dfc1) || !aligned16(pre) || !aligned16(da)) return MOE_ERR_ARG;
  const int act = params->act;
  if (act < MOE_ACT_SWIGLU || act > MOE_ACT_SREGLU) return MOE_ERR_ARG;
  GluParams g;
  g.act = act;
  g.alpha = params->alpha;
  g.up_offset = params->up_offset;
  g.gate_lo = params->gate_lo;
  g.gate_hi = params->gate_hi;
  g.up_lo = params->up_lo;
  g.up_hi = params->up_hi;
  g.lean = glu_lean_kind(params);
  g.nk = -params->alpha * 1.4426950408889634f;
  const int N1 = act == MOE_ACT_SRELU ? F : 2 * F;
  const int grid = grid_for((size_t)R_cap * (F / 32), 256);
  cudaStream_t st = as_stream(stream);
  if (g.lean == 1) k_dglu_act<1><<<grid, 256, 0, st>>>(da, pre, offsets, E, F, N1, g, dfc1);
  else if (g.lean == 2) k_dglu_act<2><<<grid, 256, 0, st>>>(da, pre, offsets, E, F, N1, g, dfc1);
  else if (g.lean == 3) k_dglu_act<3><<<grid, 256, 0, st>>>(da, pre, offsets, E, F, N1, g, dfc1);
  else k_dglu_act<0><<<grid, 256, 0, st>>>(da, pre, offsets, E, F, N1, g, dfc1);
  count_launch();
  return launch_status();
}
