// Block-scaled MXFP8 grouped GEMMs on tcgen05 (kind::mxf8f6f4, E4M3 x E4M3,
// E8M0 scale per 32 elements of K, fp32 accumulators in tensor memory):
//   M-grouped (FC2 forward, data gradient):  y[rows of e] = A[rows] . W[e]^T
//   K-grouped (weight gradient):             D[e] = A[:, rows of e] . B[:, rows of e]^T
// ([MoE-Fusion] "Boosting MoE Training Throughput with Advanced Fusion
// Kernels": GroupGemm + Quantize family and the sync-free grouped GEMM whose
// per-group counts stay in device memory; [MegaMoE] §2.3: C ~ (A_q / s_A)
// (B_q / s_B) with fine-grained per-block scales folded into the GEMM;
// §4.3: grouped problems over contiguous expert rows.)
//
// Two launches per call:
//   k_sf_tile     rewrites the row-major E8M0 scales of the tiles the GEMM
//                 will visit into the order tcgen05.cp consumes: for every
//                 (128-row tile, 128-element k-block) 512 contiguous bytes,
//                 byte 16*l + 4*j + i = scale of row 32*j + l, k sub-block i
//                 (a gather done by thousands of warps in parallel)
//   k_grouped_mx  persistent GEMM, 10 warps, one CTA per SM, 128 x 256 tiles:
//     warps 0-7  epilogue: warp w reads TMEM lane quarter w % 4 and columns
//                128 * (w / 4) .. +128 with one wait, releases the
//                accumulator, then either stages 8 rows at a time in shared
//                memory and stores full 128-byte lines (FC2, dX), or (weight
//                gradients) stages its whole 32 x 128 block in the 128-byte
//                swizzled layout and writes it with two TMA stores that
//                stream while the next tile computes (bf16 / fp32)
//     warp  8    TMA producer: A (128 x 128 bytes) and B (256 x 128 bytes)
//                tiles with the 128-byte swizzle, and the scale blocks (512 +
//                1024 bytes, 1-D bulk copies), all completing on the stage's
//                mbarrier; 4 stages (3 for the weight gradients)
//     warp  9    TMEM owner + MMA issuer: tcgen05.cp of the scale blocks into
//                tensor memory, then 4 MMAs of K = 32 (M = 128, N = 256)
//                selecting scale byte k of each 32-bit column
// The 256-wide tile halves the shared-memory traffic per FLOP of a 128-wide
// one (each stage is written once by TMA and read once by the tensor core).
// Every wait is bounded (MOE_ERR_TIMEOUT + early exit, never a trap).
#include "common.cuh"
#include "epilogue.cuh"
#include "host_common.h"

namespace moeglu {
namespace gmx {

constexpr int BM = 128, BN = 256, BK = 128;
constexpr int EPI_WARPS = 8;
constexpr int PRODUCER_WARP = 8, MMA_WARP = 9;
constexpr int THREADS = 10 * 32;
constexpr int A_TILE = BM * BK;
constexpr int B_TILE = BN * BK;
constexpr int STAGE_BYTES = A_TILE + B_TILE;
constexpr int SF_BLOCK = 512;             // one (128-row group, k-block) of scales
constexpr int SFB_BYTES = 2 * SF_BLOCK;   // the B tile's two 128-row groups
constexpr int SF_STAGE = SF_BLOCK + SFB_BYTES;
constexpr uint32_t TMEM_COLS = 512;
// accumulator: columns 0..255 (one buffer); scales of A: 4 columns; of B: 8
constexpr uint32_t SFA_COL = BN, SFB_COL = BN + 4;
// NVFP4: the four MMAs of a k-block each read their own scale columns (4 for
// the 128 rows of A, 8 for the 256 rows of B)
constexpr uint32_t SFA4_COL = BN, SFB4_COL = BN + 16;
constexpr int E_MAX = 1024;
constexpr int EPI_ROW_BYTES = 256 + 16;   // staged output row (64 words + pad)
constexpr int EPI_ROWS = 8;               // rows staged per pass
constexpr int TS_SUB = 32 * 128;          // TMA-store staging: one 32-row x 128-byte swizzled sub-tile

// Shared-memory layout of the two instantiations.  TS = false (FC2, dX): 4
// stages, 8-row staged line stores.  TS = true (weight gradients, whose K per
// tile is one expert's rows and whose output tile is the bulk of the
// traffic): 3 stages and a whole 32 x 128-column block per epilogue warp
// staged for two asynchronous TMA stores, so the stores stream while the
// next tile's MMAs run.
// NV4 (NVFP4 operands): the same 128-byte k-blocks now hold 256 E2M1
// elements and 16 E4M3 scales per row (four 512-byte scale blocks per
// 128-row group, one per MMA), so a stage carries 4x the scales; 3 stages.
template <bool TS, bool NV4 = false>
struct Lay {
  static constexpr int STAGES = TS ? (NV4 ? 2 : 3) : (NV4 ? 3 : 4);
  static constexpr int SF_ST = NV4 ? 4 * SF_STAGE : SF_STAGE;
  static constexpr int EPI_WARP_BYTES = TS ? 2 * TS_SUB : EPI_ROWS * EPI_ROW_BYTES;
  static constexpr int OFF_SF = STAGES * STAGE_BYTES;
  static constexpr int OFF_EPI = (OFF_SF + STAGES * SF_ST + 1023) / 1024 * 1024;
  static constexpr int OFF_PREF = OFF_EPI + EPI_WARPS * EPI_WARP_BYTES;
  static constexpr int OFF_BARS = OFF_PREF + (E_MAX + 2) * 4;
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  static constexpr int OFF_MISC = OFF_BARS + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = 1024 + OFF_MISC + 64;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct Args {
  const int32_t* counts;
  const int32_t* offsets;
  int E, M, N, K, R_cap;   // K: fixed contraction (M-grouped); M: rows of A (K-grouped)
  int kgrouped;            // 0: FC2 / dX, 1: weight gradient
  int b_pretiled;          // M-grouped: Bs is already in the tensor-core order (sfb_t = Bs; nothing to re-tile)
  int n_tiles_n, m_tiles;  // tiles along N; along M (K-grouped)
  int KB;                  // M-grouped: k-blocks per row tile (K / 128)
  int KG;                  // K-grouped: stride of the k-block axis of the tiled scales
  const uint8_t* As;       // scales, row-major (input of k_sf_tile)
  const uint8_t* Bs;
  uint8_t* sfa_t;          // scales in MMA order (output of k_sf_tile)
  uint8_t* sfb_t;
  void* out;               // bf16 [R_cap][N] or D [E][M][N] (f32 or bf16)
  int out_f32;
  int32_t* status;
  uint64_t wait_ns;
  // M-grouped quantised outputs (GroupGemm + Quantize), read by emit_block:
  // out_mode MOE_OUT_MXFP8 writes q_row/s_row (+ q_col/s_col), MOE_OUT_NVFP4
  // writes y (bf16) and the amax; MOE_OUT_BF16 keeps the staged bf16 path
  int out_mode, out_N;
  uint8_t* q_row;
  uint8_t* s_row;
  uint8_t* q_col;
  uint8_t* s_col;
  uint16_t* y;
  float* amax;
  float* rht_amax;         // always null here (the rotated amax belongs to the dGLU backward)
  uint32_t rht_signs;
  // MXFP8-input FC1 (EPI_GLU*, EPI_ELT): N = N1 GEMM columns (packed when
  // gated), out_N = F outputs
  const uint16_t* bias;    // [E][N1] bf16 or null
  const float* row_scale;  // [R_cap] or null
  uint16_t* pre_out;       // [R_cap][N1] bf16 or null
  GluParams prm;
  // M-grouped: real k-blocks per tile (KB counts 4-scale groups of the tiled
  // scales: KB = KBr for MXFP8, 4 * KBr for NVFP4) and scale bytes per row
  int KBr, sf_ks;
  int nv4;                 // NVFP4 operands (the EPI_NV4 instantiations)
  const float* sg_a;       // NVFP4: per-tensor scales of A and B (the product is divided by both)
  const float* sg_b;
};

// Prefix in shared memory: M-grouped -> 128-row tiles per expert (from
// counts); K-grouped -> 128-row k-blocks per expert (from the padded
// segment lengths).  pref[0..E], exclusive.  Uses all threads of the CTA.
__device__ __forceinline__ void build_prefix(const Args& a, int32_t* pref, int nthreads) {
  const int E = a.E;
  for (int e = threadIdx.x; e < E; e += nthreads) {
    int v;
    if (!a.kgrouped) {
      v = (__ldg(a.counts + e) + BM - 1) / BM;
    } else {
      const int seg = __ldg(a.offsets + e + 1) - __ldg(a.offsets + e);
      // 4-scale groups of the tiled scales: one per 128-row k-block (MXFP8),
      // four per 256-row k-block (NVFP4)
      v = seg > 0 ? (a.nv4 ? 4 * ((seg + 2 * BK - 1) / (2 * BK)) : (seg + BK - 1) / BK) : 0;
    }
    pref[e + 1] = max(v, 0);
  }
  if (threadIdx.x == 0) pref[0] = 0;
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (E + 31) / 32;
    const int beg = 1 + lane * per, end = min(E + 1, beg + per);
    int s = 0;
    for (int i = beg; i < end; ++i) s += pref[i];
    int incl = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - s;
    for (int i = beg; i < end; ++i) {
      run += pref[i];
      pref[i] = run;
    }
  }
  __syncthreads();
}

__device__ __forceinline__ int find_group(const int32_t* pref, int E, int x) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct Tile {
  int e, m0, n0;             // expert, first A row (M-grouped: permuted row), first column
  int rows_valid, rows_pad;  // M-grouped row masks
  int kseg0, kseg;           // contraction start (K-grouped: segment's first row) and length
  int num_kb;
  size_t sfa, sfb;           // byte offsets of the tile's first scale blocks
};

__device__ __forceinline__ Tile decode(int t, const int32_t* pref, const Args& a) {
  Tile ti;
  if (!a.kgrouped) {
    int lo = 0, hi = a.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pref[mid] * a.n_tiles_n <= t) lo = mid; else hi = mid - 1;
    }
    ti.e = lo;
    const int mt = pref[lo + 1] - pref[lo];
    const int local = t - pref[lo] * a.n_tiles_n;
    const int n_idx = local / mt;
    const int m_idx = local - n_idx * mt;
    const int cnt = __ldg(a.counts + lo);
    ti.m0 = __ldg(a.offsets + lo) + m_idx * BM;
    ti.n0 = n_idx * BN;
    ti.rows_valid = min(BM, cnt - m_idx * BM);
    ti.rows_pad = min(BM, ((cnt + 31) & ~31) - m_idx * BM);
    ti.rows_pad = ti.m0 < 0 ? 0 : max(0, min(ti.rows_pad, a.R_cap - ti.m0));
    ti.rows_valid = min(ti.rows_valid, ti.rows_pad);
    ti.kseg0 = 0;
    ti.kseg = a.K;
    ti.num_kb = a.KBr;  // the last k-block may be partial (MXFP8: K % 128 == 32, 64 or 96)
    ti.sfa = (size_t)(pref[lo] + m_idx) * a.KB * SF_BLOCK;
    ti.sfb = ((size_t)lo * a.n_tiles_n + n_idx) * a.KB * SFB_BYTES;
  } else {
    const int per_e = a.m_tiles * a.n_tiles_n;
    ti.e = t / per_e;
    const int local = t - ti.e * per_e;
    const int m_idx = local / a.n_tiles_n;
    const int n_idx = local - m_idx * a.n_tiles_n;
    ti.m0 = m_idx * BM;
    ti.n0 = n_idx * BN;
    ti.rows_valid = ti.rows_pad = min(BM, a.M - ti.m0);  // the last M tile may be partial (M % 32 == 0)
    const int o0 = __ldg(a.offsets + ti.e), o1 = __ldg(a.offsets + ti.e + 1);
    ti.kseg0 = o0;
    ti.kseg = (o0 < 0 || o1 > a.R_cap || o1 < o0) ? 0 : o1 - o0;
    ti.num_kb = a.nv4 ? (ti.kseg + 2 * BK - 1) / (2 * BK) : (ti.kseg + BK - 1) / BK;
    ti.sfa = ((size_t)m_idx * a.KG + pref[ti.e]) * SF_BLOCK;
    ti.sfb = ((size_t)n_idx * a.KG + pref[ti.e]) * SFB_BYTES;
  }
  return ti;
}

// ---------------------------------------------------------------------------
// Scale re-tiling.  One warp per 512-byte block (128 rows of A, or one of
// the two 128-row halves of a 256-row B tile); lane l gathers the 4 scale
// bytes of rows 32j + l (j = 0..3) and writes its 16 bytes.  Rows past the
// operand's end read as 0.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t load4_unaligned(const uint8_t* row, int kbyte, int ks) {
  // bytes row[kbyte .. kbyte+3]; bytes at or past ks read as 0.  ks % 4 == 0.
  const int w0 = kbyte & ~3, sh = (kbyte & 3) * 8;
  const uint32_t lo = w0 < ks ? __ldg(reinterpret_cast<const uint32_t*>(row + w0)) : 0u;
  const uint32_t hi = (sh != 0 && w0 + 4 < ks) ? __ldg(reinterpret_cast<const uint32_t*>(row + w0 + 4)) : 0u;
  return sh == 0 ? lo : __funnelshift_r(lo, hi, sh);
}

// Scale bytes kbyte .. kbyte+3 of one row of ks bytes (kbyte % 4 == 0);
// bytes at or past ks read as 0.  Rows of a K that is not a multiple of 128
// are not 4-byte aligned, so they are read bytewise.
__device__ __forceinline__ uint32_t load_scale4(const uint8_t* row, int kbyte, int ks) {
  if ((ks & 3) == 0) return kbyte < ks ? __ldg(reinterpret_cast<const uint32_t*>(row + kbyte)) : 0u;
  uint32_t v = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (kbyte + i < ks) v |= (uint32_t)__ldg(row + kbyte + i) << (8 * i);
  return v;
}

__global__ void __launch_bounds__(256) k_sf_tile(const Args a) {
  __shared__ int32_t pref[E_MAX + 2];
  build_prefix(a, pref, blockDim.x);
  if (__ldg(a.offsets + a.E) > a.R_cap) return;
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int bgroups = a.n_tiles_n * 2;  // 128-row groups of B (the last may pass N)
  size_t nA, nB;
  int ktot = 0;
  if (!a.kgrouped) {
    const int mt_cap = a.R_cap / BM + a.E;
    nA = (size_t)min(pref[a.E], mt_cap) * a.KB;
    nB = a.b_pretiled ? 0 : (size_t)a.E * bgroups * a.KB;
  } else {
    ktot = min(pref[a.E], a.KG);
    nA = (size_t)a.m_tiles * ktot;
    nB = (size_t)bgroups * ktot;
  }
  const size_t total = nA + nB;
  for (size_t it = (size_t)blockIdx.x * warps + (threadIdx.x >> 5); it < total; it += (size_t)gridDim.x * warps) {
    uint32_t v[4];
    uint8_t* dst;
    if (!a.kgrouped) {
      const int ks = a.sf_ks;
      if (it < nA) {
        const int mt = (int)(it / a.KB), kb = (int)(it % a.KB);
        const int e = find_group(pref, a.E, mt);
        const int m0 = __ldg(a.offsets + e) + (mt - pref[e]) * BM;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = m0 + 32 * j + lane;
          v[j] = (r >= 0 && r < a.R_cap) ? load_scale4(a.As + (size_t)r * ks, kb * 4, ks) : 0u;
        }
        dst = a.sfa_t + it * SF_BLOCK;
      } else {
        const size_t jb = it - nA;
        const int kb = (int)(jb % a.KB);
        const size_t rest = jb / a.KB;
        const int g = (int)(rest % bgroups), e = (int)(rest / bgroups);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int n = g * 128 + 32 * j + lane;
          v[j] = n < a.N ? load_scale4(a.Bs + ((size_t)e * a.N + n) * ks, kb * 4, ks) : 0u;
        }
        // [expert][n tile][k-block][half of the tile][512 bytes]
        dst = a.sfb_t + ((((size_t)e * a.n_tiles_n + (g >> 1)) * a.KB + kb) * 2 + (g & 1)) * SF_BLOCK;
      }
    } else {
      const int ks = a.sf_ks;  // scale bytes per operand row: R_cap / 32 (MXFP8) or R_cap / 16 (NVFP4)
      const int rpb = a.nv4 ? 16 : 32;  // rows per scale byte
      const bool isA = it < nA;
      const size_t jb = isA ? it : it - nA;
      const int rt = (int)(jb / ktot), kg = (int)(jb % ktot);
      const int e = find_group(pref, a.E, kg);
      const int kbyte = __ldg(a.offsets + e) / rpb + (kg - pref[e]) * 4;
      // bytes past the expert's segment are zero, so a partial last MMA adds
      // nothing from the next expert's rows
      const int kend = __ldg(a.offsets + e + 1) / rpb;
      const uint8_t* base = isA ? a.As : a.Bs;
      const int rows = isA ? a.M : a.N;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = rt * 128 + 32 * j + lane;
        uint32_t w4 = r < rows ? load4_unaligned(base + (size_t)r * ks, kbyte, ks) : 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (kbyte + i >= kend) w4 &= ~(0xFFu << (8 * i));
        v[j] = w4;
      }
      // A: [m tile][k-block][512]; B: [n tile][k-block][half][512]
      dst = isA ? a.sfa_t + ((size_t)rt * a.KG + kg) * SF_BLOCK
                : a.sfb_t + (((size_t)(rt >> 1) * a.KG + kg) * 2 + (rt & 1)) * SF_BLOCK;
    }
    reinterpret_cast<uint4*>(dst)[lane] = make_uint4(v[0], v[1], v[2], v[3]);
  }
}

// Epilogue pass over this warp's 32 accumulator rows and its 128 columns
// 128 * h .. (v[] holds them): fp32 goes out in two passes of 64 columns
// (P = 0, 64), bf16 in one pass of 128.  Rows are staged 8 at a time in
// shared memory (256 bytes each) and stored two rows per instruction as full
// 128-byte lines; columns at or past N are not stored.
template <bool F32, int P>
__device__ __forceinline__ void store_pass(const Args& a, const Tile& ti, const float* v, uint8_t* stg, int q, int h,
                                           int lane) {
  const int es = F32 ? 4 : 2;
  const int half = lane >> 4, ch = lane & 15;
  const int col0 = ti.n0 + h * 128 + P;             // first column of this pass
  const bool ch_ok = col0 + ch * (16 / es) < a.N;  // this lane's 16-byte chunk exists
#pragma unroll
  for (int g = 0; g < 32 / EPI_ROWS; ++g) {
    if ((lane >> 3) == g) {
      const int srow = lane & 7;
      if (F32) {
        float4* d = reinterpret_cast<float4*>(stg + srow * EPI_ROW_BYTES);
#pragma unroll
        for (int w = 0; w < 16; ++w)
          d[w] = make_float4(v[P + 4 * w], v[P + 4 * w + 1], v[P + 4 * w + 2], v[P + 4 * w + 3]);
      } else {
        uint4* d = reinterpret_cast<uint4*>(stg + srow * EPI_ROW_BYTES);
#pragma unroll
        for (int w = 0; w < 16; ++w)
          d[w] = make_uint4(pack_bf16x2(v[8 * w], v[8 * w + 1]), pack_bf16x2(v[8 * w + 2], v[8 * w + 3]),
                            pack_bf16x2(v[8 * w + 4], v[8 * w + 5]), pack_bf16x2(v[8 * w + 6], v[8 * w + 7]));
      }
    }
    __syncwarp();
#pragma unroll
    for (int rr = 0; rr < EPI_ROWS; rr += 2) {
      const int srow = rr + half;
      const int r_local = q * 32 + g * EPI_ROWS + srow;
      if (r_local < ti.rows_pad && ch_ok) {
        const uint4 val = *reinterpret_cast<const uint4*>(stg + srow * EPI_ROW_BYTES + ch * 16);
        uint8_t* gp;
        if (!a.kgrouped)
          gp = reinterpret_cast<uint8_t*>(a.out) + ((size_t)(ti.m0 + r_local) * a.N + col0) * es;
        else
          gp = reinterpret_cast<uint8_t*>(a.out) + (((size_t)ti.e * a.M + ti.m0 + r_local) * a.N + col0) * es;
        *reinterpret_cast<uint4*>(gp + ch * 16) = val;
      }
    }
    __syncwarp();
  }
}

// Weight-gradient epilogue pass: this warp's 32 rows x 128 bf16 columns (or
// 64 fp32 columns starting at P) as two 32 x 128-byte sub-tiles in the
// 128-byte swizzled layout (16-byte chunk c of row r at chunk c ^ (r % 8):
// the lanes of a quarter-warp hit distinct banks), then two TMA stores of
// D[e] issued by lane 0.  The buffer is reused only after the previous
// stores have read it.  The tensor map clips boxes that reach past M or N
// (M, N multiples of 32); boxes that start past N are not issued.
template <bool F32, int P>
__device__ __forceinline__ void store_pass_tma(const CUtensorMap* tmO, const Tile& ti, const float* v, uint8_t* stg,
                                               int q, int h, int lane, int N) {
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
  const int sw = lane & 7;
#pragma unroll
  for (int w = 0; w < 16; ++w) {
    uint4* d = reinterpret_cast<uint4*>(stg + (w >> 3) * TS_SUB + lane * 128 + (((w & 7) ^ sw) << 4));
    if (F32)
      *d = make_uint4(__float_as_uint(v[P + 4 * w]), __float_as_uint(v[P + 4 * w + 1]),
                      __float_as_uint(v[P + 4 * w + 2]), __float_as_uint(v[P + 4 * w + 3]));
    else
      *d = make_uint4(pack_bf16x2(v[8 * w], v[8 * w + 1]), pack_bf16x2(v[8 * w + 2], v[8 * w + 3]),
                      pack_bf16x2(v[8 * w + 4], v[8 * w + 5]), pack_bf16x2(v[8 * w + 6], v[8 * w + 7]));
  }
  fence_async_shared();
  __syncwarp();
  if (lane == 0) {
    constexpr int SUB_COLS = F32 ? 32 : 64;
    const int col0 = ti.n0 + h * 128 + P;
    const int row = ti.m0 + q * 32;
    // boxes reaching past N or M are clipped by the tensor map; one that
    // starts at or past N (N % 128 != 0) is not issued
    if (col0 < N) tma_store_3d(tmO, stg, col0, row, ti.e);
    if (col0 + SUB_COLS < N) tma_store_3d(tmO, stg + TS_SUB, col0 + SUB_COLS, row, ti.e);
    bulk_commit();
  }
}

// ---------------------------------------------------------------------------
// The GEMM
// ---------------------------------------------------------------------------
// Epilogue kinds of the M-grouped instantiations (TS = false): plain bf16
// rows, the quantising output stage (GroupGemm + Quantize), and the fused
// activation of the MXFP8-input FC1 (GroupGemm + Activation +
// Quantize/Transpose) with the activation forms of the bf16 kernel.
enum Epi { EPI_BF16 = 0, EPI_QUANT = 1, EPI_GLU = 2, EPI_GLU_L1 = 3, EPI_GLU_L2 = 4, EPI_GLU_L3 = 5, EPI_ELT = 6,
           // NVFP4 operands (kind::mxf4nvf4, E4M3 scales per 16 elements), bf16 rows divided by
           // the two per-tensor scales
           EPI_NV4 = 7 };
__host__ __device__ constexpr bool epi_glu(int k) { return k >= EPI_GLU && k <= EPI_GLU_L3; }

template <bool TS, int EPI>
__global__ void __launch_bounds__(THREADS, 1)
    k_grouped_mx(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmO, const Args a) {
  constexpr bool NV4 = EPI == EPI_NV4;
  using L = Lay<TS, NV4>;
  constexpr int SF_ST = L::SF_ST;
  constexpr int SF_MUL = NV4 ? 4 : 1;  // 512-byte scale blocks per 128-row group and k-block
  constexpr int STAGES = L::STAGES;
  constexpr int OFF_SF = L::OFF_SF, OFF_EPI = L::OFF_EPI, OFF_PREF = L::OFF_PREF, OFF_BARS = L::OFF_BARS,
                OFF_MISC = L::OFF_MISC, EPI_WARP_BYTES = L::EPI_WARP_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;
  uint8_t* sf = smem + OFF_SF;
  uint8_t* epi_all = smem + OFF_EPI;
  int32_t* pref = reinterpret_cast<int32_t*>(smem + OFF_PREF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BARS);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E;

  if (warp == PRODUCER_WARP && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full + b, 1);
      mbar_init(acc_empty + b, EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_async_shared();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (TS) tma_prefetch_desc(&tmO);
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  build_prefix(a, pref, THREADS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool over = __ldg(a.offsets + E) > a.R_cap;
  if (over && threadIdx.x == 0) set_status(a.status, MOE_ERR_CAPACITY);
  int total = 0;
  if (!over) total = a.kgrouped ? E * a.m_tiles * a.n_tiles_n : pref[E] * a.n_tiles_n;
  const uint32_t tmem_base = *tmem_slot;
  WaitGuard guard{abort_flag, a.status, a.wait_ns};

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_parity = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const Tile ti = decode(t, pref, a);
        bool ok = true;
        for (int kb = 0; kb < ti.num_kb; ++kb) {
          if (!mbar_wait(empty + stage, phase ^ 1u, guard)) {
            ok = false;
            break;
          }
          uint8_t* dst = tiles + stage * STAGE_BYTES;
          uint8_t* sdst = sf + stage * SF_ST;
          mbar_arrive_expect_tx(full + stage, STAGE_BYTES + SF_ST);
          if (!a.kgrouped) {
            tma_load_2d(dst, &tmA, full + stage, kb * BK, ti.m0);
            tma_load_3d(dst + A_TILE, &tmB, full + stage, kb * BK, ti.n0, ti.e);
          } else {
            // the contraction runs along the operands' rows of tokens: one byte
            // per token (MXFP8) or per two tokens (packed NVFP4)
            const int kx = NV4 ? ti.kseg0 / 2 + kb * BK : ti.kseg0 + kb * BK;
            tma_load_2d(dst, &tmA, full + stage, kx, ti.m0);
            tma_load_2d(dst + A_TILE, &tmB, full + stage, kx, ti.n0);
          }
          bulk_load(sdst, a.sfa_t + ti.sfa + (size_t)kb * SF_MUL * SF_BLOCK, SF_MUL * SF_BLOCK, full + stage);
          bulk_load(sdst + SF_MUL * SF_BLOCK, a.sfb_t + ti.sfb + (size_t)kb * SF_MUL * SFB_BYTES, SF_MUL * SFB_BYTES,
                    full + stage);
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (*abort_flag) {
        volatile int never = 0;
        WaitGuard drain{&never, a.status, 100000000ull};
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s)) mbar_wait(full + s, (issued_parity >> s) & 1u, drain);
      }
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      const uint32_t idesc = NV4 ? idesc_nvf4_e4m3(BM, BN) : idesc_mxf8_e8m0(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int lt = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x, ++lt) {
        const Tile ti = decode(t, pref, a);
        const int buf = 0;  // one accumulator: the epilogue frees it as soon as it has read it
        const uint32_t aph = (uint32_t)lt & 1u;
        if (!mbar_wait(acc_empty + buf, aph ^ 1u, guard)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base;
        bool ok = true;
        for (int kb = 0; kb < ti.num_kb; ++kb) {
          if (!mbar_wait(full + stage, phase, guard)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(tiles + stage * STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_TILE;
          const uint32_t sf_addr = smem_u32(sf + stage * SF_ST);
          if (NV4) {
            // four MMAs of K = 64 E2M1 elements (32 bytes of the 128-byte
            // rows), each with its own 4 scale bytes per row: MMA k's block
            // of A scales goes to columns SFA4 + 4k, its two blocks of B
            // scales to SFB4 + 8k (rows 0..127) and SFB4 + 8k + 4
            // MMAs of 64 elements; a weight gradient's last one may cover 32
            // rows of its segment (the scales of the rest are zero)
            const int nsub = min(4, (ti.kseg - kb * 2 * BK + 63) / 64);
            for (int k = 0; k < nsub; ++k) {
              tc_cp_32x128b_x4(tmem_base + SFA4_COL + 4 * k, sdesc_noswizzle(sf_addr + k * SF_BLOCK, 128));
              tc_cp_32x128b_x4(tmem_base + SFB4_COL + 8 * k,
                               sdesc_noswizzle(sf_addr + 4 * SF_BLOCK + k * SFB_BYTES, 128));
              tc_cp_32x128b_x4(tmem_base + SFB4_COL + 8 * k + 4,
                               sdesc_noswizzle(sf_addr + 4 * SF_BLOCK + k * SFB_BYTES + SF_BLOCK, 128));
            }
            for (int k = 0; k < nsub; ++k) {
              umma_nvf4(d_tmem, sdesc_kmajor_sw128(a_addr + k * 32), sdesc_kmajor_sw128(b_addr + k * 32), idesc,
                        tmem_base + SFA4_COL + 4 * k, tmem_base + SFB4_COL + 8 * k, (kb | k) != 0 ? 1u : 0u);
            }
          } else {
            tc_cp_32x128b_x4(tmem_base + SFA_COL, sdesc_noswizzle(sf_addr, 128));
            tc_cp_32x128b_x4(tmem_base + SFB_COL, sdesc_noswizzle(sf_addr + SF_BLOCK, 128));
            tc_cp_32x128b_x4(tmem_base + SFB_COL + 4, sdesc_noswizzle(sf_addr + 2 * SF_BLOCK, 128));
            // descriptors of the stage computed once; a step of 32 bytes along
            // K is +2 in the descriptor's 16-byte address field
            const int nsub = min(4, (ti.kseg - kb * BK) / 32);
            const uint64_t ad = sdesc_kmajor_sw128(a_addr), bd = sdesc_kmajor_sw128(b_addr);
            if (nsub == 4) {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                umma_mxf8(d_tmem, ad + 2 * k, bd + 2 * k, idesc_with_sf_ids(idesc, (uint32_t)k, (uint32_t)k),
                          tmem_base + SFA_COL, tmem_base + SFB_COL, (kb | k) != 0 ? 1u : 0u);
            } else {
              for (int k = 0; k < nsub; ++k)
                umma_mxf8(d_tmem, ad + 2 * k, bd + 2 * k, idesc_with_sf_ids(idesc, (uint32_t)k, (uint32_t)k),
                          tmem_base + SFA_COL, tmem_base + SFB_COL, (kb | k) != 0 ? 1u : 0u);
            }
          }
          tc_commit(empty + stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(acc_full + buf);
      }
      tc_commit(mma_done);
      volatile int never = 0;
      WaitGuard drain{&never, a.status, 100000000ull};
      mbar_wait(mma_done, 0, drain);
    }
  } else {
    const int q = warp & 3, h = warp >> 2;
    uint8_t* stg = epi_all + warp * EPI_WARP_BYTES;
    const int out_es = (a.kgrouped && a.out_f32) ? 4 : 2;  // output element size
    Amax amax_bits{0u, 0u};
    int lt = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++lt) {
      const int buf = 0;
      const uint32_t aph = (uint32_t)lt & 1u;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(acc_full + buf, aph, guard) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const Tile ti = decode(t, pref, a);
      const bool live = q * 32 < ti.rows_pad && ti.n0 + h * 128 < a.N;
      const bool real = q * 32 + lane < ti.rows_valid;
      if (EPI == EPI_QUANT) {
        // GroupGemm + Quantize (M-grouped only): the thread's row, 32 columns
        // at a time, as MXFP8 row-wise codes (+ the column-wise copy through
        // the warp's staging buffer) or bf16 plus the NVFP4 amax.  The 128
        // columns are drained in two halves of 64 (the epilogue warps have
        // 168 registers), and the accumulator is released once the second
        // half is in registers.
        const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * 128);
        const int r_local = q * 32 + lane;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[64];
          if (live) {
            tmem_ld32(tbase + half * 64, v);
            tmem_ld32(tbase + half * 64 + 32, v + 32);
          }
          if (half == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty + buf);
          }
          if (!live) continue;
          if (!real) {
#pragma unroll
            for (int i = 0; i < 64; ++i) v[i] = 0.0f;
          }
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int col0 = ti.n0 + h * 128 + half * 64 + 32 * j;
            if (col0 < a.N)
              emit_block(a, v + 32 * j, col0, ti.m0 + r_local, ti.m0 + q * 32, r_local < ti.rows_pad, stg, lane,
                         amax_bits);
          }
        }
        continue;
      }
      if (epi_glu(EPI) || EPI == EPI_ELT) {
        // FC1 on MXFP8 operands: the warp's 128 accumulator columns are two
        // packed 64-column blocks (32 input + 32 gate columns each; or 64
        // plain columns without a gate), drained one block at a time; bias,
        // saved bf16 pre-activation, activation (times the row scale), then
        // the output stage on the fp32 results.  The accumulator is released
        // once the second block is in registers.
        const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * 128);
        const int r_local = q * 32 + lane;
        const int row = ti.m0 + r_local;
        const bool row_ok = r_local < ti.rows_pad;
        const float rs = (a.row_scale != nullptr && real) ? __ldg(a.row_scale + row) : 1.0f;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          float v[64];
          if (live) {
            tmem_ld32(tbase + half * 64, v);
            tmem_ld32(tbase + half * 64 + 32, v + 32);
          }
          if (half == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty + buf);
          }
          const int p0 = ti.n0 + h * 128 + half * 64;  // first GEMM column of the block
          if (!live || p0 >= a.N) continue;
          if (a.bias != nullptr) {
            float b[32];
            const uint16_t* bp = a.bias + (size_t)ti.e * a.N + p0;
            load_bf16x32(bp, b);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] += b[i];
            load_bf16x32(bp + 32, b);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[32 + i] += b[i];
          }
          if (a.pre_out != nullptr && row_ok) {
            uint16_t* pp = a.pre_out + (size_t)row * a.N + p0;
            store_bf16x32(pp, v, !real);
            store_bf16x32(pp + 32, v + 32, !real);
          }
          if (epi_glu(EPI)) {
            float yv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              float y;
              if (EPI == EPI_GLU_L1)
                y = swiglu_fwd_lean(a.prm, v[i], v[32 + i]);
              else if (EPI == EPI_GLU_L2)
                y = swiglu_fwd_lean_clamped(a.prm, v[i], v[32 + i]);
              else if (EPI == EPI_GLU_L3)
                y = geglu_fwd_lean(a.prm, v[i], v[32 + i]);
              else
                y = act_fwd(a.prm, v[i], v[32 + i]);
              yv[i] = real ? y * rs : 0.0f;
            }
            emit_block(a, yv, p0 / 2, row, ti.m0 + q * 32, row_ok, stg, lane, amax_bits);
          } else {
#pragma unroll
            for (int bk = 0; bk < 2; ++bk) {
              float yv[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) yv[i] = real ? act_fwd(a.prm, v[32 * bk + i], 0.0f) * rs : 0.0f;
              emit_block(a, yv, p0 + 32 * bk, row, ti.m0 + q * 32, row_ok, stg, lane, amax_bits);
            }
          }
        }
        continue;
      }
      float v[128];
      if (live && ti.num_kb > 0)
        tmem_ld128(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * 128), v);
      // the accumulator is in registers: hand the buffer back to the MMA
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + buf);
      if (!live) continue;
      if (ti.num_kb == 0 || !real) {
#pragma unroll
        for (int i = 0; i < 128; ++i) v[i] = 0.0f;
      }
      if (NV4) {
        // NVFP4 values are e2m1 * s_b / s_g: the MMA applied the block scales,
        // the two per-tensor scales divide the product here
        const float g = 1.0f / (__ldg(a.sg_a) * __ldg(a.sg_b));
#pragma unroll
        for (int i = 0; i < 128; ++i) v[i] *= g;
      }
      if (TS) {
        if (out_es == 4) {
          store_pass_tma<true, 0>(&tmO, ti, v, stg, q, h, lane, a.N);
          store_pass_tma<true, 64>(&tmO, ti, v, stg, q, h, lane, a.N);
        } else {
          store_pass_tma<false, 0>(&tmO, ti, v, stg, q, h, lane, a.N);
        }
      } else if (out_es == 4) {
        store_pass<true, 0>(a, ti, v, stg, q, h, lane);
        store_pass<true, 64>(a, ti, v, stg, q, h, lane);
      } else {
        store_pass<false, 0>(a, ti, v, stg, q, h, lane);
      }
    }
    if (TS && lane == 0) bulk_wait_all();
    if (EPI != EPI_BF16 && a.out_mode == MOE_OUT_NVFP4 && a.amax != nullptr) {
      const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, amax_bits.plain);
      if (lane == 0 && m != 0) atomicMax(reinterpret_cast<int*>(a.amax), (int)m);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <bool TS, int EPI>
static void launch_kernel(int grid, int smem, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmO,
                          const Args& a, cudaStream_t stream) {
  k_grouped_mx<TS, EPI><<<grid, THREADS, smem, stream>>>(tmA, tmB, tmO, a);
}

// epi: the epilogue kind (Epi) of an M-grouped call; the weight gradient
// (tmO != null) always takes the TMA-store epilogue
static moe_status_t launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap* tmO, const Args& a,
                           long long tiles_bound, long long sf_items, int sm_margin, cudaStream_t stream,
                           int epi = -1) {
  const bool ts = tmO != nullptr;
  if (epi < 0) epi = (!ts && a.out_mode != MOE_OUT_BF16) ? EPI_QUANT : EPI_BF16;
  if (!ts && a.out_mode == MOE_OUT_NVFP4 && a.amax &&
      cudaMemsetAsync(a.amax, 0, sizeof(float), stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  const void* kfn = ts ? (epi == EPI_NV4 ? (const void*)k_grouped_mx<true, EPI_NV4>
                                         : (const void*)k_grouped_mx<true, EPI_BF16>)
                    : epi == EPI_QUANT  ? (const void*)k_grouped_mx<false, EPI_QUANT>
                    : epi == EPI_GLU    ? (const void*)k_grouped_mx<false, EPI_GLU>
                    : epi == EPI_GLU_L1 ? (const void*)k_grouped_mx<false, EPI_GLU_L1>
                    : epi == EPI_GLU_L2 ? (const void*)k_grouped_mx<false, EPI_GLU_L2>
                    : epi == EPI_GLU_L3 ? (const void*)k_grouped_mx<false, EPI_GLU_L3>
                    : epi == EPI_ELT    ? (const void*)k_grouped_mx<false, EPI_ELT>
                    : epi == EPI_NV4    ? (const void*)k_grouped_mx<false, EPI_NV4>
                                        : (const void*)k_grouped_mx<false, EPI_BF16>;
  const int smem = ts ? (epi == EPI_NV4 ? Lay<true, true>::SMEM_BYTES : Lay<true>::SMEM_BYTES)
                      : (epi == EPI_NV4 ? Lay<false, true>::SMEM_BYTES : Lay<false>::SMEM_BYTES);
  if (!set_smem_limit(kfn, smem)) return MOE_ERR_CUDA;
  const int sms = sm_count();
  long long sgrid = (sf_items + 7) / 8;
  if (sgrid > (long long)sms * 8) sgrid = (long long)sms * 8;
  if (sgrid < 1) sgrid = 1;
  k_sf_tile<<<(int)sgrid, 256, 0, stream>>>(a);
  int grid = sms - sm_margin;
  if (grid > tiles_bound) grid = (int)tiles_bound;
  if (grid < 1) grid = 1;
  if (ts && epi == EPI_NV4)
    launch_kernel<true, EPI_NV4>(grid, smem, tmA, tmB, *tmO, a, stream);
  else if (ts)
    launch_kernel<true, EPI_BF16>(grid, smem, tmA, tmB, *tmO, a, stream);
  else if (epi == EPI_QUANT)
    launch_kernel<false, EPI_QUANT>(grid, smem, tmA, tmB, tmA, a, stream);
  else if (epi == EPI_GLU)
    launch_kernel<false, EPI_GLU>(grid, smem, tmA, tmB, tmA, a, stream);
  else if (epi == EPI_GLU_L1)
    launch_kernel<false, EPI_GLU_L1>(grid, smem, tmA, tmB, tmA, a, stream);
  else if (epi == EPI_GLU_L2)
    launch_kernel<false, EPI_GLU_L2>(grid, smem, tmA, tmB, tmA, a, stream);
  else if (epi == EPI_GLU_L3)
    launch_kernel<false, EPI_GLU_L3>(grid, smem, tmA, tmB, tmA, a, stream);
  else if (epi == EPI_ELT)
    launch_kernel<false, EPI_ELT>(grid, smem, tmA, tmB, tmA, a, stream);
  else if (epi == EPI_NV4)
    launch_kernel<false, EPI_NV4>(grid, smem, tmA, tmB, tmA, a, stream);
  else
    launch_kernel<false, EPI_BF16>(grid, smem, tmA, tmB, tmA, a, stream);
  count_launch(2);
  return launch_status();
}

static size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

static int n_tiles(int N) { return (N + BN - 1) / BN; }
static int k_blocks(int K) { return (K + BK - 1) / BK; }
static int m_tiles_of(int M) { return (M + BM - 1) / BM; }

// Tiled-scale workspace of an M-grouped call: MXFP8 has one 512-byte block per
// (128-row group, 128-element k-block); NVFP4 four per 256-element k-block.
static size_t sf_kblocks(int K, bool nv4) { return nv4 ? 4 * (size_t)((K + 255) / 256) : (size_t)k_blocks(K); }

static void fc2_ws_parts(int E, int K, int N, int R_cap, size_t* a_bytes, size_t* b_bytes, bool nv4 = false) {
  const size_t KB = sf_kblocks(K, nv4);
  *a_bytes = align_up(((size_t)R_cap / BM + E) * KB * SF_BLOCK);
  *b_bytes = align_up((size_t)E * n_tiles(N) * KB * SFB_BYTES);
}

// 4-scale groups a weight gradient's tiled scales hold per row tile (the
// stride of the group axis): MXFP8 one per 128 rows of each segment, NVFP4
// four per 256 rows
static size_t wgrad_kg(int E, int R_cap, bool nv4) {
  return nv4 ? (size_t)R_cap / 64 + 4 * (size_t)E : (size_t)R_cap / BK + E;
}

static void wgrad_ws_parts(int E, int M, int N, int R_cap, size_t* a_bytes, size_t* b_bytes, bool nv4 = false) {
  const size_t KG = wgrad_kg(E, R_cap, nv4);
  *a_bytes = align_up((size_t)m_tiles_of(M) * KG * SF_BLOCK);
  *b_bytes = align_up((size_t)n_tiles(N) * KG * SFB_BYTES);
}

}  // namespace gmx
}  // namespace moeglu

using namespace moeglu;

extern "C" size_t moe_grouped_fc2_workspace_size(int E, int K, int N, int R_cap) {
  if (E <= 0 || K <= 0 || N <= 0 || R_cap <= 0) return 0;
  size_t a, b, a4, b4;
  gmx::fc2_ws_parts(E, K, N, R_cap, &a, &b);
  gmx::fc2_ws_parts(E, K, N, R_cap, &a4, &b4, true);
  return a + b > a4 + b4 ? a + b : a4 + b4;  // enough for either block-scaled operand type
}

extern "C" size_t moe_grouped_wgrad_workspace_size(int E, int M, int N, int R_cap) {
  if (E <= 0 || M <= 0 || N <= 0 || R_cap <= 0) return 0;
  size_t a, b, a4, b4;
  gmx::wgrad_ws_parts(E, M, N, R_cap, &a, &b);
  gmx::wgrad_ws_parts(E, M, N, R_cap, &a4, &b4, true);
  return a + b > a4 + b4 ? a + b : a4 + b4;  // enough for MXFP8 or NVFP4 operands
}

extern "C" moe_status_t moe_grouped_fc2_fwd(const moe_in_t* A, const moe_in_t* W, const int32_t* counts,
                                            const int32_t* offsets, int E, int K, int N, int R_cap, int out_mode,
                                            const moe_act_out_t* out, void* ws, size_t ws_bytes, int sm_margin,
                                            int32_t* status, moe_stream_t stream) {
  using namespace gmx;
  if (!A || !W || !A->data || !W->data || !counts || !offsets || !out) return MOE_ERR_ARG;
  if (E <= 0 || E > E_MAX || K <= 0 || (K % 32) || N <= 0 || (N % 32) || R_cap <= 0 || (R_cap % BM))
    return MOE_ERR_ARG;
  // one operand type per MMA (an MXFP8 or NVFP4 weight may carry pre-tiled scales)
  const bool w_tiled = (A->dtype == MOE_IN_MXFP8 && W->dtype == MOE_IN_MXFP8_TILED) ||
                       (A->dtype == MOE_IN_NVFP4 && W->dtype == MOE_IN_NVFP4_TILED);
  if (sm_margin < 0 || (A->dtype != W->dtype && !w_tiled)) return MOE_ERR_ARG;
  if (out_mode != MOE_OUT_BF16 && out_mode != MOE_OUT_MXFP8 && out_mode != MOE_OUT_NVFP4) return MOE_ERR_ARG;
  if (out->pre || out->row_dot || out->rht_amax) return MOE_ERR_ARG;
  if (A->dtype == MOE_IN_BF16)
    return grouped_gemm_bf16_out(A->data, W->data, counts, offsets, E, K, N, R_cap, out_mode, out, ws, ws_bytes,
                                 sm_margin, status, as_stream(stream));
  if (A->dtype == MOE_IN_NVFP4) {
    // NVFP4 operands: packed E2M1 (K/2 bytes per row), E4M3 scales per 16
    // elements (K/16 bytes per row), per-tensor scales; bf16 output only
    const uint8_t* Aq4 = static_cast<const uint8_t*>(A->data);
    const uint8_t* Wq4 = static_cast<const uint8_t*>(W->data);
    if (!A->scale || !W->scale || !A->global_scale || !W->global_scale || !ws) return MOE_ERR_ARG;
    if (K % 64) return MOE_ERR_ARG;
    if (out_mode != MOE_OUT_BF16) return MOE_ERR_UNSUPPORTED;
    if (!out->y || !aligned16(out->y) || !aligned16(Aq4) || !aligned16(Wq4) ||
        (reinterpret_cast<uintptr_t>(A->scale) & 3) || (reinterpret_cast<uintptr_t>(W->scale) & 3) ||
        (reinterpret_cast<uintptr_t>(ws) & 255))
      return MOE_ERR_ARG;
    if (w_tiled && (reinterpret_cast<uintptr_t>(W->scale) & 15)) return MOE_ERR_ARG;  // 16-byte bulk copies
    size_t a4, b4;
    fc2_ws_parts(E, K, N, R_cap, &a4, &b4, true);
    if (ws_bytes < a4 + b4) return MOE_ERR_ARG;
    CUtensorMap tA, tB;
    {
      const uint64_t dims[2] = {(uint64_t)K / 2, (uint64_t)R_cap};
      const uint64_t strides[1] = {(uint64_t)K / 2};
      const uint32_t box[2] = {BK, BM};
      if (!encode_tmap(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, Aq4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return MOE_ERR_CUDA;
    }
    {
      const uint64_t dims[3] = {(uint64_t)K / 2, (uint64_t)N, (uint64_t)E};
      const uint64_t strides[2] = {(uint64_t)K / 2, (uint64_t)N * (K / 2)};
      const uint32_t box[3] = {BK, BN, 1};
      if (!encode_tmap(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, Wq4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return MOE_ERR_CUDA;
    }
    Args a{};
    a.counts = counts;
    a.offsets = offsets;
    a.E = E;
    a.N = N;
    a.K = K;
    a.R_cap = R_cap;
    a.n_tiles_n = n_tiles(N);
    a.KB = (int)sf_kblocks(K, true);
    a.KBr = (K + 255) / 256;
    a.nv4 = 1;
    a.sf_ks = K / 16;
    a.As = A->scale;
    a.Bs = W->scale;
    a.sfa_t = static_cast<uint8_t*>(ws);
    a.sfb_t = w_tiled ? const_cast<uint8_t*>(W->scale) : static_cast<uint8_t*>(ws) + a4;
    a.b_pretiled = w_tiled ? 1 : 0;
    a.out = out->y;
    a.status = status;
    a.wait_ns = g_wait_limit_ns.load();
    a.out_mode = MOE_OUT_BF16;
    a.out_N = N;
    a.sg_a = A->global_scale;
    a.sg_b = W->global_scale;
    const long long mt_bound = (long long)R_cap / BM + E;
    const long long bound = mt_bound * a.n_tiles_n;
    const long long sf_items = mt_bound * a.KB + (w_tiled ? 0 : (long long)E * 2 * a.n_tiles_n * a.KB);
    return launch(tA, tB, nullptr, a, bound, sf_items, sm_margin, as_stream(stream), EPI_NV4);
  }
  if (A->dtype != MOE_IN_MXFP8) return MOE_ERR_ARG;
  const uint8_t* Aq = static_cast<const uint8_t*>(A->data);
  const uint8_t* Wq = static_cast<const uint8_t*>(W->data);
  const uint8_t* As = A->scale;
  const uint8_t* Ws = W->scale;
  if (!As || !Ws || !ws) return MOE_ERR_ARG;
  if (!aligned16(Aq) || !aligned16(Wq) || (reinterpret_cast<uintptr_t>(As) & 3) ||
      (reinterpret_cast<uintptr_t>(Ws) & 3) || (reinterpret_cast<uintptr_t>(ws) & 255))
    return MOE_ERR_ARG;
  if (w_tiled && (reinterpret_cast<uintptr_t>(Ws) & 15)) return MOE_ERR_ARG;  // 16-byte bulk copies
  if (out_mode == MOE_OUT_MXFP8) {
    if (!out->q_row || !out->s_row || (out->q_col == nullptr) != (out->s_col == nullptr)) return MOE_ERR_ARG;
    if (!aligned16(out->q_row) || (out->q_col && !aligned16(out->q_col))) return MOE_ERR_ARG;
  } else {
    if (!out->y || !aligned16(out->y)) return MOE_ERR_ARG;
    if (out_mode == MOE_OUT_NVFP4 && !out->amax) return MOE_ERR_ARG;
  }
  size_t a_bytes, b_bytes;
  fc2_ws_parts(E, K, N, R_cap, &a_bytes, &b_bytes);
  if (ws_bytes < a_bytes + b_bytes) return MOE_ERR_ARG;
  CUtensorMap tmA, tmB;
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)R_cap};
    const uint64_t strides[1] = {(uint64_t)K};
    const uint32_t box[2] = {BK, BM};
    if (!encode_tmap(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, Aq, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {(uint64_t)K, (uint64_t)N, (uint64_t)E};
    const uint64_t strides[2] = {(uint64_t)K, (uint64_t)N * K};
    const uint32_t box[3] = {BK, BN, 1};
    if (!encode_tmap(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, Wq, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  Args a{};
  a.counts = counts;
  a.offsets = offsets;
  a.E = E;
  a.M = 0;
  a.N = N;
  a.K = K;
  a.R_cap = R_cap;
  a.kgrouped = 0;
  a.n_tiles_n = n_tiles(N);
  a.m_tiles = 0;
  a.KB = k_blocks(K);
  a.KBr = a.KB;
  a.sf_ks = K / 32;
  a.KG = 0;
  a.As = As;
  a.Bs = Ws;
  a.sfa_t = static_cast<uint8_t*>(ws);
  a.sfb_t = w_tiled ? const_cast<uint8_t*>(Ws) : static_cast<uint8_t*>(ws) + a_bytes;
  a.b_pretiled = w_tiled ? 1 : 0;
  a.out = out->y;
  a.out_f32 = 0;
  a.status = status;
  a.wait_ns = g_wait_limit_ns.load();
  a.out_mode = out_mode;
  a.out_N = N;
  a.q_row = out->q_row;
  a.s_row = out->s_row;
  a.q_col = out->q_col;
  a.s_col = out->s_col;
  a.y = reinterpret_cast<uint16_t*>(out->y);
  a.amax = out->amax;
  const long long mt_bound = (long long)R_cap / BM + E;
  const long long bound = mt_bound * a.n_tiles_n;
  const long long sf_items = mt_bound * a.KB + (w_tiled ? 0 : (long long)E * 2 * a.n_tiles_n * a.KB);
  return launch(tmA, tmB, nullptr, a, bound, sf_items, sm_margin, as_stream(stream));
}

extern "C" moe_status_t moe_grouped_fc1_glu_quant_fwd_mxfp8(
    const uint8_t* xq, const uint8_t* xs, const uint8_t* W1q, const uint8_t* W1s, const moe_bf16* b1p,
    const float* row_scale, const int32_t* counts, const int32_t* offsets, int E, int H, int F, int R_cap,
    const moe_glu_params_t* params, int out_mode, const moe_act_out_t* out, void* ws, size_t ws_bytes, int sm_margin,
    int32_t* status, moe_stream_t stream) {
  using namespace gmx;
  if (!xq || !xs || !W1q || !W1s || !counts || !offsets || !params || !out || !ws) return MOE_ERR_ARG;
  if (E <= 0 || E > E_MAX || H <= 0 || (H % 32) || F <= 0 || (F % 32) || R_cap <= 0 || (R_cap % BM) || sm_margin < 0)
    return MOE_ERR_ARG;
  const int act = params->act;
  if (act < MOE_ACT_SWIGLU || act > MOE_ACT_SREGLU) return MOE_ERR_ARG;
  const bool gated = act != MOE_ACT_SRELU;
  const int N1 = gated ? 2 * F : F;
  if (!aligned16(xq) || !aligned16(W1q) || (reinterpret_cast<uintptr_t>(xs) & 3) ||
      (reinterpret_cast<uintptr_t>(W1s) & 3) || (reinterpret_cast<uintptr_t>(ws) & 255) || (b1p && !aligned16(b1p)))
    return MOE_ERR_ARG;
  if (out->row_dot || out->rht_amax) return MOE_ERR_ARG;
  if (out->pre && !aligned16(out->pre)) return MOE_ERR_ARG;
  if (out_mode == MOE_OUT_MXFP8) {
    if (!out->q_row || !out->s_row || (out->q_col == nullptr) != (out->s_col == nullptr)) return MOE_ERR_ARG;
    if (!aligned16(out->q_row) || (out->q_col && !aligned16(out->q_col))) return MOE_ERR_ARG;
  } else if (out_mode == MOE_OUT_BF16 || out_mode == MOE_OUT_NVFP4) {
    if (!out->y || !aligned16(out->y)) return MOE_ERR_ARG;
    if (out_mode == MOE_OUT_NVFP4 && !out->amax) return MOE_ERR_ARG;
  } else {
    return MOE_ERR_ARG;
  }
  size_t a_bytes, b_bytes;
  fc2_ws_parts(E, H, N1, R_cap, &a_bytes, &b_bytes);
  if (ws_bytes < a_bytes + b_bytes) return MOE_ERR_ARG;
  CUtensorMap tmA, tmB;
  {
    const uint64_t dims[2] = {(uint64_t)H, (uint64_t)R_cap};
    const uint64_t strides[1] = {(uint64_t)H};
    const uint32_t box[2] = {BK, BM};
    if (!encode_tmap(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, xq, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {(uint64_t)H, (uint64_t)N1, (uint64_t)E};
    const uint64_t strides[2] = {(uint64_t)H, (uint64_t)N1 * H};
    const uint32_t box[3] = {BK, BN, 1};
    if (!encode_tmap(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, W1q, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  Args a{};
  a.counts = counts;
  a.offsets = offsets;
  a.E = E;
  a.N = N1;
  a.K = H;
  a.R_cap = R_cap;
  a.kgrouped = 0;
  a.n_tiles_n = n_tiles(N1);
  a.KB = k_blocks(H);
  a.KBr = a.KB;
  a.sf_ks = H / 32;
  a.As = xs;
  a.Bs = W1s;
  a.sfa_t = static_cast<uint8_t*>(ws);
  a.sfb_t = static_cast<uint8_t*>(ws) + a_bytes;
  a.status = status;
  a.wait_ns = g_wait_limit_ns.load();
  a.out_mode = out_mode;
  a.out_N = F;
  a.q_row = out->q_row;
  a.s_row = out->s_row;
  a.q_col = out->q_col;
  a.s_col = out->s_col;
  a.y = reinterpret_cast<uint16_t*>(out->y);
  a.amax = out->amax;
  a.bias = reinterpret_cast<const uint16_t*>(b1p);
  a.row_scale = row_scale;
  a.pre_out = reinterpret_cast<uint16_t*>(out->pre);
  a.prm = GluParams{params->act,    params->alpha, params->up_offset, params->gate_lo, params->gate_hi,
                    params->up_lo,  params->up_hi, glu_lean_kind(params), -params->alpha * 1.4426950408889634f};
  int epi = EPI_ELT;
  if (gated) {
    const int lean = glu_lean_kind(params);
    epi = lean == 1 ? EPI_GLU_L1 : lean == 2 ? EPI_GLU_L2 : lean == 3 ? EPI_GLU_L3 : EPI_GLU;
  }
  const long long mt_bound = (long long)R_cap / BM + E;
  const long long bound = mt_bound * a.n_tiles_n;
  const long long sf_items = mt_bound * a.KB + (long long)E * 2 * a.n_tiles_n * a.KB;
  return launch(tmA, tmB, nullptr, a, bound, sf_items, sm_margin, as_stream(stream), epi);
}

extern "C" moe_status_t moe_grouped_wgrad(const uint8_t* Aq, const uint8_t* As, const uint8_t* Bq, const uint8_t* Bs,
                                          const int32_t* counts, const int32_t* offsets, int E, int M, int N,
                                          int R_cap, void* D, int out_f32, void* ws, size_t ws_bytes, int sm_margin,
                                          int32_t* status, moe_stream_t stream) {
  using namespace gmx;
  if (!Aq || !As || !Bq || !Bs || !counts || !offsets || !D || !ws) return MOE_ERR_ARG;
  if (E <= 0 || E > E_MAX || M <= 0 || (M % 32) || N <= 0 || (N % 32) || R_cap <= 0 || (R_cap % BM))
    return MOE_ERR_ARG;
  if (!aligned16(Aq) || !aligned16(Bq) || !aligned16(D) || (reinterpret_cast<uintptr_t>(As) & 3) ||
      (reinterpret_cast<uintptr_t>(Bs) & 3) || (reinterpret_cast<uintptr_t>(ws) & 255) || sm_margin < 0)
    return MOE_ERR_ARG;
  size_t a_bytes, b_bytes;
  wgrad_ws_parts(E, M, N, R_cap, &a_bytes, &b_bytes);
  if (ws_bytes < a_bytes + b_bytes) return MOE_ERR_ARG;
  CUtensorMap tmA, tmB;
  {
    const uint64_t dims[2] = {(uint64_t)R_cap, (uint64_t)M};
    const uint64_t strides[1] = {(uint64_t)R_cap};
    const uint32_t box[2] = {BK, BM};
    if (!encode_tmap(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, Aq, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {(uint64_t)R_cap, (uint64_t)N};
    const uint64_t strides[1] = {(uint64_t)R_cap};
    const uint32_t box[2] = {BK, BN};
    if (!encode_tmap(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, Bq, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  Args a{};
  a.counts = counts;
  a.offsets = offsets;
  a.E = E;
  a.M = M;
  a.N = N;
  a.K = 0;
  a.R_cap = R_cap;
  a.kgrouped = 1;
  a.n_tiles_n = n_tiles(N);
  a.m_tiles = m_tiles_of(M);
  a.KB = 0;
  a.KG = R_cap / BK + E;
  a.sf_ks = R_cap / 32;
  a.As = As;
  a.Bs = Bs;
  a.sfa_t = static_cast<uint8_t*>(ws);
  a.sfb_t = static_cast<uint8_t*>(ws) + a_bytes;
  a.out = D;
  a.out_f32 = out_f32 ? 1 : 0;
  a.status = status;
  a.wait_ns = g_wait_limit_ns.load();
  CUtensorMap tmO;
  {
    const uint64_t es = out_f32 ? 4 : 2;
    const uint64_t dims[3] = {(uint64_t)N, (uint64_t)M, (uint64_t)E};
    const uint64_t strides[2] = {(uint64_t)N * es, (uint64_t)M * N * es};
    const uint32_t box[3] = {out_f32 ? 32u : 64u, 32, 1};
    if (!encode_tmap(&tmO, out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, D, dims,
                     strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  const long long bound = (long long)E * a.m_tiles * a.n_tiles_n;
  const long long sf_items = (long long)(a.m_tiles + 2 * a.n_tiles_n) * a.KG;
  return launch(tmA, tmB, &tmO, a, bound, sf_items, sm_margin, as_stream(stream));
}

extern "C" moe_status_t moe_grouped_wgrad_nvfp4(const uint8_t* Aq, const uint8_t* As, const float* sgA,
                                                const uint8_t* Bq, const uint8_t* Bs, const float* sgB,
                                                const int32_t* counts, const int32_t* offsets, int E, int M, int N,
                                                int R_cap, void* D, int out_f32, void* ws, size_t ws_bytes,
                                                int sm_margin, int32_t* status, moe_stream_t stream) {
  using namespace gmx;
  if (!Aq || !As || !sgA || !Bq || !Bs || !sgB || !counts || !offsets || !D || !ws) return MOE_ERR_ARG;
  if (E <= 0 || E > E_MAX || M <= 0 || (M % 32) || N <= 0 || (N % 32) || R_cap <= 0 || (R_cap % BM))
    return MOE_ERR_ARG;
  if (!aligned16(Aq) || !aligned16(Bq) || !aligned16(D) || (reinterpret_cast<uintptr_t>(As) & 3) ||
      (reinterpret_cast<uintptr_t>(Bs) & 3) || (reinterpret_cast<uintptr_t>(ws) & 255) || sm_margin < 0)
    return MOE_ERR_ARG;
  size_t a_bytes, b_bytes;
  wgrad_ws_parts(E, M, N, R_cap, &a_bytes, &b_bytes, true);
  if (ws_bytes < a_bytes + b_bytes) return MOE_ERR_ARG;
  CUtensorMap tmA, tmB, tmO;
  {
    const uint64_t dims[2] = {(uint64_t)R_cap / 2, (uint64_t)M};
    const uint64_t strides[1] = {(uint64_t)R_cap / 2};
    const uint32_t box[2] = {BK, BM};
    if (!encode_tmap(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, Aq, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {(uint64_t)R_cap / 2, (uint64_t)N};
    const uint64_t strides[1] = {(uint64_t)R_cap / 2};
    const uint32_t box[2] = {BK, BN};
    if (!encode_tmap(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, Bq, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  {
    const uint64_t es = out_f32 ? 4 : 2;
    const uint64_t dims[3] = {(uint64_t)N, (uint64_t)M, (uint64_t)E};
    const uint64_t strides[2] = {(uint64_t)N * es, (uint64_t)M * N * es};
    const uint32_t box[3] = {out_f32 ? 32u : 64u, 32, 1};
    if (!encode_tmap(&tmO, out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, D, dims,
                     strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  Args a{};
  a.counts = counts;
  a.offsets = offsets;
  a.E = E;
  a.M = M;
  a.N = N;
  a.R_cap = R_cap;
  a.kgrouped = 1;
  a.n_tiles_n = n_tiles(N);
  a.m_tiles = m_tiles_of(M);
  a.KG = (int)wgrad_kg(E, R_cap, true);
  a.sf_ks = R_cap / 16;
  a.nv4 = 1;
  a.As = As;
  a.Bs = Bs;
  a.sfa_t = static_cast<uint8_t*>(ws);
  a.sfb_t = static_cast<uint8_t*>(ws) + a_bytes;
  a.out = D;
  a.out_f32 = out_f32 ? 1 : 0;
  a.status = status;
  a.wait_ns = g_wait_limit_ns.load();
  a.sg_a = sgA;
  a.sg_b = sgB;
  const long long bound = (long long)E * a.m_tiles * a.n_tiles_n;
  const long long sf_items = (long long)(a.m_tiles + 2 * a.n_tiles_n) * a.KG;
  return launch(tmA, tmB, &tmO, a, bound, sf_items, sm_margin, as_stream(stream), EPI_NV4);
}
