// Persistent grouped GEMM on the 5th-generation tensor cores (tcgen05) with
// bf16 operands and the activation fused into the epilogue:
//   forward  GroupGemm + Activation + Quantize/Transpose
//   backward GroupGemm + dActivation + Quantize/Transpose
// ([MoE-Fusion] "Boosting MoE Training Throughput with Advanced Fusion
// Kernels": the three-kernel family; "Optimizing GLU via fused GEMM
// epilogues" (Fig. 2): repacked weights put matching input and gate columns
// in one tile, so the epilogue combines them without a global round trip;
// "Fusing MXFP8 and NVFP4 quantisation": the MXFP8 output and its transposed
// copy are produced inside the GEMM kernel; "Eliminating host-device
// synchronisation": the per-expert row counts are read from device memory by
// the kernel's own tile scheduler.  [MegaMoE] §4.2: producer / consumer warp
// specialisation over a multi-stage shared-memory ring; §5.3: tails masked.)
//
// Two variants share the warp roles and the epilogue.  CTA = 10 warps, one
// CTA per SM, persistent over tiles (ordered expert-major, then N, then M so
// that the CTAs working at one time share weight tiles in L2):
//   warps 0-7  epilogue: warp w reads TMEM lane quarter w % 4 (one thread =
//              one accumulator row) and column half w / 4 of the tile; bias,
//              activation (or its derivative from the saved pre-activation),
//              MXFP8 row + column quantisation (or bf16 / NVFP4), stores
//   warp  8    TMA producer (one thread): 128-byte-swizzled boxes of A
//              (activations [rows][K], 64 columns of K) and B (weights
//              [E][N][K]) into a multi-stage ring of full/empty mbarriers
//   warp  9    TMEM owner + MMA issuer (one thread): tcgen05.mma kind::f16,
//              K = 16 per instruction, fp32 accumulators double-buffered in
//              TMEM (2 x 256 of the 512 columns); tcgen05.commit frees smem
//              stages and hands finished accumulators to the epilogue
// Default (k_grouped_bf16_pair): clusters of 2 CTAs run 256 x 256 tiles with
// tcgen05 cta_group::2 (M = 256 issued by the even CTA, each CTA holding 128
// rows of A and half of B per stage, 6 stages); moe_set_cta_pairs(0) selects
// k_grouped_bf16, one CTA per 128 x 256 tile with 4 stages.  The pair
// kernel takes its tiles from an atomic counter in the call's workspace (the
// leader's producer hands each tile to both CTAs through a 4-slot queue) and
// computes an expert's thin last tile transposed (weights as M = 256, the
// rows as N).
// Every wait is bounded (MOE_ERR_TIMEOUT + early exit, never a trap).
#include <cmath>

#include "common.cuh"
#include "epilogue.cuh"
#include "host_common.h"

namespace moeglu {
namespace g16 {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
// 8 epilogue warps: warp w reads TMEM lane quarter w % 4 and handles half
// w / 4 of the tile's accumulator columns
constexpr int EPI_WARPS = 8;
constexpr int THREADS = (EPI_WARPS + 2) * 32;
constexpr int PRODUCER_WARP = 8, MMA_WARP = 9;
constexpr int A_TILE = BM * BK * 2;
constexpr int B_TILE = BN * BK * 2;
constexpr int STAGE_BYTES = A_TILE + B_TILE;
constexpr uint32_t TMEM_COLS = 512;
constexpr int E_MAX = 1024;
constexpr int SCRATCH_PER_WARP = 1024;
constexpr int OFF_SCRATCH = STAGES * STAGE_BYTES;
constexpr int OFF_PREF = OFF_SCRATCH + EPI_WARPS * SCRATCH_PER_WARP;
constexpr int OFF_BARS = OFF_PREF + (E_MAX + 2) * 4;
constexpr int NUM_BARS = 2 * STAGES + 5;
constexpr int OFF_MISC = OFF_BARS + NUM_BARS * 8;
constexpr int SMEM_BYTES = 1024 + OFF_MISC + 64;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// BWD_*_DOT: the backward modes that also write the feature-scale partials
// (separate instantiations, so the plain backward carries no extra code)
enum Mode { FWD_GLU = 0, FWD_ELT = 1, FWD_PRE = 2, BWD_GLU = 3, BWD_ELT = 4, BWD_GLU_DOT = 5, BWD_ELT_DOT = 6,
            // SwiGLU with its short activation forms (GluParams::lean 1: no clamp, 2: clamped), each
            // its own instantiation so that a kernel carries only the activation code it runs
            FWD_GLU_L1 = 7, FWD_GLU_L2 = 8, BWD_GLU_L1 = 9, BWD_GLU_L2 = 10, FWD_GLU_L3 = 11, BWD_GLU_L3 = 12,
            // plain grouped GEMM whose fp32 result goes through the output stage
            // (GroupGemm + Quantize with bf16 operands)
            FWD_ID = 13 };
__host__ __device__ constexpr bool is_fwd_glu(int m) {
  return m == FWD_GLU || m == FWD_GLU_L1 || m == FWD_GLU_L2 || m == FWD_GLU_L3;
}
__host__ __device__ constexpr bool is_bwd_glu(int m) {
  return m == BWD_GLU || m == BWD_GLU_DOT || m == BWD_GLU_L1 || m == BWD_GLU_L2 || m == BWD_GLU_L3;
}
__host__ __device__ constexpr int lean_of(int m) {
  return (m == FWD_GLU_L1 || m == BWD_GLU_L1)   ? 1
         : (m == FWD_GLU_L2 || m == BWD_GLU_L2) ? 2
         : (m == FWD_GLU_L3 || m == BWD_GLU_L3) ? 3
                                                : 0;
}

struct Args {
  const int32_t* counts;
  const int32_t* offsets;
  int E, K, N_gemm, F, N1, R_cap, n_tiles_n, out_N;
  const uint16_t* bias;    // [E][N1] (forward), may be null
  const float* row_scale;  // [R_cap], may be null
  const uint16_t* pre_in;  // backward: saved pre-activation [R_cap][N1]
  GluParams prm;
  int out_mode;
  uint8_t* q_row;
  uint8_t* s_row;
  uint8_t* q_col;
  uint8_t* s_col;
  uint16_t* y;
  float* amax;
  uint16_t* pre_out;
  float* row_dot;          // backward: [R_cap][2 * n_tiles_n] partials of da * act(pre), may be null
  float* db_parts;         // backward: [R_cap / 32][N1] column sums of dFC1 per 32-row block (bias gradient), may be null
  int swap_max;            // pair kernel: an expert's last pair tile with at most this many rows runs swapped (0: never)
  int* sched;              // pair kernel: tile counter of the dynamic scheduler (zeroed before the launch), or null
  float* rht_amax;         // backward NVFP4: amax of the transposed random Hadamard rotation, may be null
  uint32_t rht_signs;      //   its 16 signs (bit i set: -1)
  int32_t* status;
  uint64_t wait_ns;
};

struct Tile {
  int e, m_idx, n_idx, row0, rows_valid, rows_pad;
  // swapped tail tile (CTA-pair kernel): the expert's last pair tile holds at
  // most Args::swap_max rows, so it is computed transposed, weights as the
  // M = 256 operand and its nt (a multiple of 32) rows as N
  int swap, nt, tail0, tail_valid;
};

__device__ __forceinline__ Tile decode_tile(int t, const int32_t* pref, int E, int n_tiles_n,
                                            const int32_t* counts, const int32_t* offsets, int R_cap) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] * n_tiles_n <= t) lo = mid; else hi = mid - 1;
  }
  Tile ti;
  ti.e = lo;
  const int mt = pref[lo + 1] - pref[lo];
  const int local = t - pref[lo] * n_tiles_n;
  ti.n_idx = local / mt;
  ti.m_idx = local - ti.n_idx * mt;
  const int cnt = __ldg(counts + lo);
  ti.row0 = __ldg(offsets + lo) + ti.m_idx * BM;
  ti.rows_valid = min(BM, cnt - ti.m_idx * BM);
  ti.rows_pad = min(BM, ((cnt + 31) & ~31) - ti.m_idx * BM);
  // never touch rows at or past R_cap, whatever counts/offsets hold
  ti.rows_pad = ti.row0 < 0 ? 0 : max(0, min(ti.rows_pad, R_cap - ti.row0));
  ti.rows_valid = min(ti.rows_valid, ti.rows_pad);
  ti.swap = ti.nt = ti.tail0 = ti.tail_valid = 0;
  return ti;
}

template <int MODE>
__device__ __forceinline__ void epilogue_tile(const Args& a, const Tile& ti, uint32_t tacc, int q, int h, int lane,
                                              uint8_t* scratch, Amax& amax_bits) {
  if (q * 32 >= ti.rows_pad) return;  // no row of this warp lies in the padded segment
  const int r_local = q * 32 + lane;
  const bool real = r_local < ti.rows_valid;
  const bool row_ok = r_local < ti.rows_pad;  // always true here, kept for clarity
  const int row = ti.row0 + r_local;
  const int rb = ti.row0 + q * 32;
  const float rs = (a.row_scale != nullptr && real) ? __ldg(a.row_scale + row) : 1.0f;

  if (is_fwd_glu(MODE)) {
#pragma unroll 1
    for (int j = h * (BN / 128); j < (h + 1) * (BN / 128); ++j) {
      const int f0 = ti.n_idx * (BN / 2) + j * 32;
      if (f0 >= a.F) break;
      const int p0 = ti.n_idx * BN + j * 64;
      float v[64];
      tmem_ld32(tacc + j * 64, v);
      tmem_ld32(tacc + j * 64 + 32, v + 32);
      if (a.bias != nullptr) {
        float b[32];
        const uint16_t* bp = a.bias + (size_t)ti.e * a.N1 + p0;
        load_bf16x32(bp, b);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += b[i];
        load_bf16x32(bp + 32, b);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[32 + i] += b[i];
      }
      if (a.pre_out != nullptr && row_ok) {
        uint16_t* pp = a.pre_out + (size_t)row * a.N1 + p0;
        store_bf16x32(pp, v, !real);
        store_bf16x32(pp + 32, v + 32, !real);
      }
      float yv[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) yv[i] = 0.0f;
      if (real) {
        if (lean_of(MODE) == 1) {
#pragma unroll
          for (int i = 0; i < 32; ++i) yv[i] = swiglu_fwd_lean(a.prm, v[i], v[32 + i]) * rs;
        } else if (lean_of(MODE) == 2) {
#pragma unroll
          for (int i = 0; i < 32; ++i) yv[i] = swiglu_fwd_lean_clamped(a.prm, v[i], v[32 + i]) * rs;
        } else if (lean_of(MODE) == 3) {
#pragma unroll
          for (int i = 0; i < 32; ++i) yv[i] = geglu_fwd_lean(a.prm, v[i], v[32 + i]) * rs;
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) yv[i] = act_fwd(a.prm, v[i], v[32 + i]) * rs;
        }
      }
      emit_block(a, yv, f0, row, rb, row_ok, scratch, lane, amax_bits);
    }
  } else if (MODE == FWD_ELT || MODE == FWD_PRE || MODE == FWD_ID) {
#pragma unroll 1
    for (int j = h * (BN / 64); j < (h + 1) * (BN / 64); ++j) {
      const int c0 = ti.n_idx * BN + j * 32;
      if (c0 >= a.N_gemm) break;
      float v[32];
      tmem_ld32(tacc + j * 32, v);
      if (a.bias != nullptr) {
        float b[32];
        load_bf16x32(a.bias + (size_t)ti.e * a.N1 + c0, b);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += b[i];
      }
      if (a.pre_out != nullptr && row_ok) store_bf16x32(a.pre_out + (size_t)row * a.N1 + c0, v, !real);
      if (MODE == FWD_ELT) {
        float yv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) yv[i] = real ? act_fwd(a.prm, v[i], 0.0f) * rs : 0.0f;
        emit_block(a, yv, c0, row, rb, row_ok, scratch, lane, amax_bits);
      } else if (MODE == FWD_ID) {
        if (!real) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.0f;
        }
        emit_block(a, v, c0, row, rb, row_ok, scratch, lane, amax_bits);
      }
    }
  } else if (is_bwd_glu(MODE)) {
    constexpr bool DOT = MODE == BWD_GLU_DOT;
    float dot = 0.0f;  // this warp half's share of sum_c da * act(pre) (feature-scale gradient)
    // the saved pre-activations of the next 32-column block (128 contiguous
    // bytes of the row, one L1 line) are prefetched while this one is processed
    const int j_end = (h + 1) * (BN / 64);
#pragma unroll 1
    for (int j = h * (BN / 64); j < j_end; ++j) {
      const int f0 = ti.n_idx * BN + j * 32;
      if (f0 >= a.F) break;
      const int p0 = (f0 / 32) * 64;
      if (real && j + 1 < j_end && f0 + 32 < a.F)
        prefetch_l1(a.pre_in + (size_t)row * a.N1 + p0 + 64);
      float d[32], u[32], g[32];
      tmem_ld32(tacc + j * 32, d);
      if (real) {
        load_bf16x32(a.pre_in + (size_t)row * a.N1 + p0, u);
        load_bf16x32(a.pre_in + (size_t)row * a.N1 + p0 + 32, g);
        if (DOT) {
#pragma unroll
          for (int i = 0; i < 32; ++i) dot = fmaf(d[i], act_fwd(a.prm, u[i], g[i]), dot);
        }
        if (lean_of(MODE) == 1) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float du, dg;
            swiglu_bwd_lean(a.prm, u[i], g[i], d[i] * rs, du, dg);
            u[i] = du;
            g[i] = dg;
          }
        } else if (lean_of(MODE) == 2) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float du, dg;
            swiglu_bwd_lean_clamped(a.prm, u[i], g[i], d[i] * rs, du, dg);
            u[i] = du;
            g[i] = dg;
          }
        } else if (lean_of(MODE) == 3) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float du, dg;
            geglu_bwd_lean(a.prm, u[i], g[i], d[i] * rs, du, dg);
            u[i] = du;
            g[i] = dg;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float du, dg;
            act_bwd(a.prm, u[i], g[i], d[i] * rs, du, dg);
            u[i] = du;
            g[i] = dg;
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) u[i] = g[i] = 0.0f;
      }
      if (a.db_parts != nullptr) {
        // bias gradient: this block's column sums over the warp's 32 rows
        // (pad rows hold 0), one coalesced line per 32 columns
        float* dst = a.db_parts + (size_t)(rb / 32) * a.N1 + p0 + lane;
        dst[0] = warp_column_sum32(u, lane);
        dst[32] = warp_column_sum32(g, lane);
      }
      emit_block(a, u, p0, row, rb, row_ok, scratch, lane, amax_bits);
      emit_block(a, g, p0 + 32, row, rb, row_ok, scratch, lane, amax_bits);
    }
    if (DOT) a.row_dot[(size_t)row * (2 * a.n_tiles_n) + ti.n_idx * 2 + h] = dot;
  } else {  // BWD_ELT, BWD_ELT_DOT
    constexpr bool DOT = MODE == BWD_ELT_DOT;
    float dot = 0.0f;
#pragma unroll 1
    for (int j = h * (BN / 64); j < (h + 1) * (BN / 64); ++j) {
      const int f0 = ti.n_idx * BN + j * 32;
      if (f0 >= a.F) break;
      float d[32], x[32];
      tmem_ld32(tacc + j * 32, d);
      if (real) {
        load_bf16x32(a.pre_in + (size_t)row * a.N1 + f0, x);
        if (DOT) {
#pragma unroll
          for (int i = 0; i < 32; ++i) dot = fmaf(d[i], act_fwd(a.prm, x[i], 0.0f), dot);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float du, dg;
          act_bwd(a.prm, x[i], 0.0f, d[i] * rs, du, dg);
          x[i] = du;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = 0.0f;
      }
      if (a.db_parts != nullptr) a.db_parts[(size_t)(rb / 32) * a.N1 + f0 + lane] = warp_column_sum32(x, lane);
      emit_block(a, x, f0, row, rb, row_ok, scratch, lane, amax_bits);
    }
    if (DOT) a.row_dot[(size_t)row * (2 * a.n_tiles_n) + ti.n_idx * 2 + h] = dot;
  }
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    k_grouped_bf16(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;
  uint8_t* scratch_all = smem + OFF_SCRATCH;
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
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  // m-tiles per expert -> exclusive prefix pref[0..E]
  for (int e = threadIdx.x; e < E; e += THREADS) pref[e + 1] = (__ldg(a.counts + e) + BM - 1) / BM;
  if (threadIdx.x == 0) pref[0] = 0;
  __syncthreads();
  if (warp == 0) {
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // capacity guard: a routing that overflowed R_cap produces no tiles
  const bool over = __ldg(a.offsets + E) > a.R_cap;
  if (over && threadIdx.x == 0) set_status(a.status, MOE_ERR_CAPACITY);
  const int total = over ? 0 : pref[E] * a.n_tiles_n;
  const int num_kb = a.K / BK;
  WaitGuard guard{abort_flag, a.status, a.wait_ns};

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;  // per stage: armed and its parity
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const Tile ti = decode_tile(t, pref, E, a.n_tiles_n, a.counts, a.offsets, a.R_cap);
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(empty + stage, phase ^ 1u, guard)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = tiles + stage * STAGE_BYTES;
          mbar_arrive_expect_tx(full + stage, STAGE_BYTES);
          tma_load_2d(a_dst, &tmA, full + stage, kb * BK, ti.row0);
          tma_load_3d(a_dst + A_TILE, &tmB, full + stage, kb * BK, ti.n_idx * BN, ti.e);
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
        // give the copies already in flight a bounded chance to land
        volatile int never = 0;
        WaitGuard drain{&never, a.status, 100000000ull};
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s)) mbar_wait(full + s, (issued_parity >> s) & 1u, drain);
      }
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int lt = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x, ++lt) {
        const int buf = lt & 1;
        const uint32_t aph = (uint32_t)(lt >> 1) & 1u;
        if (!mbar_wait(acc_empty + buf, aph ^ 1u, guard)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(full + stage, phase, guard)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(tiles + stage * STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_TILE;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            umma_bf16(d_tmem, sdesc_kmajor_sw128(a_addr + k * 32), sdesc_kmajor_sw128(b_addr + k * 32), idesc,
                      (kb | k) != 0 ? 1u : 0u);
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
      // all MMAs issued by this thread have completed once this arrives
      tc_commit(mma_done);
      volatile int never = 0;
      WaitGuard drain{&never, a.status, 100000000ull};
      mbar_wait(mma_done, 0, drain);
    }
  } else {
    // epilogue warps 0..3: warp q reads TMEM lanes 32q..32q+31
    const int q = warp & 3, h = warp >> 2;
    uint8_t* scratch = scratch_all + warp * SCRATCH_PER_WARP;
    Amax amax_bits{0u, 0u};
    int lt = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++lt) {
      const int buf = lt & 1;
      const uint32_t aph = (uint32_t)(lt >> 1) & 1u;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(acc_full + buf, aph, guard) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const Tile ti = decode_tile(t, pref, E, a.n_tiles_n, a.counts, a.offsets, a.R_cap);
      const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
      epilogue_tile<MODE>(a, ti, tacc, q, h, lane, scratch, amax_bits);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + buf);
    }
    if (a.out_mode == MOE_OUT_NVFP4 && a.amax != nullptr) {
      const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, amax_bits.plain);
      if (lane == 0 && m != 0) atomicMax(reinterpret_cast<int*>(a.amax), (int)m);
    }
    if (a.out_mode == MOE_OUT_NVFP4 && a.rht_amax != nullptr) {
      const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, amax_bits.rht);
      if (lane == 0 && m != 0) atomicMax(reinterpret_cast<int*>(a.rht_amax), (int)m);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// CTA-pair variant (clusters of 2, tcgen05 cta_group::2).  The pair computes
// a 256 x 256 tile: each CTA holds 128 rows of A and 128 of the 256 B rows
// in its own shared memory (32 KB per stage, 6 stages) and receives its 128
// accumulator rows in its own tensor memory.  The even CTA issues the MMAs
// (M = 256) and its commits are multicast to both CTAs; both CTAs' TMA loads
// complete on the even CTA's stage barrier; the odd CTA's epilogue releases
// accumulators through the even CTA's barrier.  Per SM this fetches 32 KB
// per 128x256x64 step instead of 48 KB.
// ---------------------------------------------------------------------------
namespace pair {
constexpr int STAGES = 6;
constexpr int THREADS = (EPI_WARPS + 2) * 32;
constexpr int B_HALF = (BN / 2) * BK * 2;
constexpr int STAGE_BYTES = A_TILE + B_HALF;
constexpr int OFF_SCRATCH = STAGES * STAGE_BYTES;
constexpr int OFF_PREF = OFF_SCRATCH + EPI_WARPS * SCRATCH_PER_WARP;
constexpr int OFF_BARS = OFF_PREF + (E_MAX + 2) * 4;
// tile queue: TQ slots of tile indices handed from the leader's producer to
// every other role of both CTAs, with a full and an empty barrier per slot
constexpr int TQ = 4;
constexpr int NUM_BARS = 2 * STAGES + 5 + 2 * TQ;
constexpr int OFF_MISC = OFF_BARS + NUM_BARS * 8;
constexpr int SMEM_BYTES = 1024 + OFF_MISC + 64;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
// consumers that release a queue slot: the leader's MMA thread and both
// CTAs' epilogue warps and the peer's producer
constexpr int TQ_CONSUMERS = 1 + 2 * EPI_WARPS + 1;
}  // namespace pair

// Tile t of the pair sequence: expert e, N tile, 256-row pair tile mp; this
// CTA's half starts 128 * rank rows further.
__device__ __forceinline__ Tile decode_pair(int t, const int32_t* pref, int E, int n_tiles_n, const int32_t* counts,
                                            const int32_t* offsets, int R_cap, int rank, int swap_max) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] * n_tiles_n <= t) lo = mid; else hi = mid - 1;
  }
  Tile ti;
  ti.e = lo;
  const int mt = pref[lo + 1] - pref[lo];
  const int local = t - pref[lo] * n_tiles_n;
  ti.n_idx = local / mt;
  ti.m_idx = local - ti.n_idx * mt;
  const int cnt = __ldg(counts + lo);
  const int base = ti.m_idx * 2 * BM + rank * BM;
  ti.row0 = __ldg(offsets + lo) + base;
  ti.rows_valid = max(0, min(BM, cnt - base));
  ti.rows_pad = max(0, min(BM, ((cnt + 31) & ~31) - base));
  ti.rows_pad = ti.row0 < 0 ? 0 : max(0, min(ti.rows_pad, R_cap - ti.row0));
  ti.rows_valid = min(ti.rows_valid, ti.rows_pad);
  // the expert's last pair tile, when thin, runs swapped: its rows become
  // the N operand (nt = rows rounded up to 32, inside the padded segment)
  const int tail = cnt - ti.m_idx * 2 * BM;
  ti.tail0 = __ldg(offsets + lo) + ti.m_idx * 2 * BM;
  ti.tail_valid = max(0, min(tail, 2 * BM));
  ti.nt = min((ti.tail_valid + 31) & ~31, ti.tail0 < 0 ? 0 : (R_cap - ti.tail0) & ~31);
  ti.swap = (tail > 0 && tail <= swap_max && ti.nt >= 32) ? 1 : 0;
  return ti;
}

// Named barrier of the two epilogue warps (lane quarters q and q + 1 of one
// column half) that share a swapped forward tile's input and gate columns.
__device__ __forceinline__ void pair_warps_sync(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }

// Epilogue of a swapped tail tile.  This CTA's accumulator lane i holds GEMM
// column n_idx * BN + rank * BN/2 + i, and accumulator column j holds row
// tail0 + j (j < nt).  Warp (q, h) takes the columns of lane quarter q and
// the 32-row groups h, h + 2, ...; each thread then owns one column and 32
// consecutive rows, emitted through the transposed output stage.  Forward
// GLU: lane quarters 2i (input) and 2i + 1 (gate) hold the two halves of one
// packed 64-column block, so the gate warp hands its values to the input
// warp through their shared 2 KB of scratch.
template <int MODE>
__device__ __forceinline__ void epilogue_swapped(const Args& a, const Tile& ti, uint32_t tacc, int q, int h, int lane,
                                                 int rank, uint8_t* pair_scratch, Amax& amax_bits) {
  const int colbase = ti.n_idx * BN + rank * (BN / 2) + q * 32;  // first GEMM column of this warp
  const int ngroups = ti.nt / 32;
  if (colbase >= a.N_gemm) return;  // a multiple of 64 (gated) or 32: whole warp pairs drop out together
  const int col = colbase + lane;
  if (is_fwd_glu(MODE)) {
    const bool gate_warp = (q & 1) != 0;
    const int bar_id = 1 + h * 2 + (q >> 1);
    const float bias = a.bias != nullptr ? bf16_lo(__ldg(a.bias + (size_t)ti.e * a.N1 + col)) : 0.0f;
    float* xs = reinterpret_cast<float*>(pair_scratch);  // 16 rows x 32 lanes
    const int f = (colbase / 64) * 32 + lane;           // output column (input warp)
#pragma unroll 1
    for (int tg = h; tg < ngroups; tg += 2) {
      const int rb = ti.tail0 + tg * 32;
      const int nvalid = min(32, ti.tail_valid - tg * 32);
      float v[32];
      tmem_ld32(tacc + tg * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = j < nvalid ? v[j] + bias : 0.0f;
      if (a.pre_out != nullptr) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          a.pre_out[(size_t)(rb + j) * a.N1 + col] = __bfloat16_as_ushort(__float2bfloat16_rn(v[j]));
      }
      float g[32];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        pair_warps_sync(bar_id);  // the input warp has read the previous half
        if (gate_warp) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) xs[jj * 32 + lane] = v[16 * hf + jj];
        }
        pair_warps_sync(bar_id);
        if (!gate_warp) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) g[16 * hf + jj] = xs[jj * 32 + lane];
        }
      }
      if (gate_warp) continue;
#pragma unroll
      for (int j = 0; j < 32; ++j) {  // the activation in place of the input half
        const float rs = (a.row_scale != nullptr && j < nvalid) ? __ldg(a.row_scale + rb + j) : 1.0f;
        float yy;
        if (lean_of(MODE) == 1)
          yy = swiglu_fwd_lean(a.prm, v[j], g[j]);
        else if (lean_of(MODE) == 2)
          yy = swiglu_fwd_lean_clamped(a.prm, v[j], g[j]);
        else if (lean_of(MODE) == 3)
          yy = geglu_fwd_lean(a.prm, v[j], g[j]);
        else
          yy = act_fwd(a.prm, v[j], g[j]);
        v[j] = j < nvalid ? yy * rs : 0.0f;
      }
      emit_block_t(a, v, f, rb, lane, amax_bits);
    }
    // the scratch goes back to the two warps' own use only after the input
    // warp has read the last half
    pair_warps_sync(bar_id);
  } else if (MODE == FWD_ELT || MODE == FWD_PRE || MODE == FWD_ID) {
    const float bias = a.bias != nullptr ? bf16_lo(__ldg(a.bias + (size_t)ti.e * a.N1 + col)) : 0.0f;
#pragma unroll 1
    for (int tg = h; tg < ngroups; tg += 2) {
      const int rb = ti.tail0 + tg * 32;
      const int nvalid = min(32, ti.tail_valid - tg * 32);
      float v[32];
      tmem_ld32(tacc + tg * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = j < nvalid ? v[j] + bias : 0.0f;
      if (a.pre_out != nullptr) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          a.pre_out[(size_t)(rb + j) * a.N1 + col] = __bfloat16_as_ushort(__float2bfloat16_rn(v[j]));
      }
      if (MODE == FWD_ELT) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float rs = (a.row_scale != nullptr && j < nvalid) ? __ldg(a.row_scale + rb + j) : 1.0f;
          v[j] = j < nvalid ? act_fwd(a.prm, v[j], 0.0f) * rs : 0.0f;
        }
      }
      if (MODE != FWD_PRE) emit_block_t(a, v, col, rb, lane, amax_bits);
    }
  } else {  // backward (the DOT instantiations never run swapped)
    const bool gated = is_bwd_glu(MODE);
    const int pu = gated ? (colbase / 32) * 64 + lane : col;  // packed input column (or the column itself)
#pragma unroll 1
    for (int tg = h; tg < ngroups; tg += 2) {
      const int rb = ti.tail0 + tg * 32;
      const int nvalid = min(32, ti.tail_valid - tg * 32);
      float u[32], g[32];  // u: da on load, then d(input) in place
      tmem_ld32(tacc + tg * 32, u);
      const uint16_t* pp = a.pre_in + (size_t)rb * a.N1 + pu;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float dj = u[j];
        u[j] = g[j] = 0.0f;
        if (j < nvalid) {
          const float rs = a.row_scale != nullptr ? __ldg(a.row_scale + rb + j) : 1.0f;
          const float dy = dj * rs;
          const float uu = __uint_as_float((uint32_t)__ldg(pp + (size_t)j * a.N1) << 16);
          float du, dg;
          if (gated) {
            const float gg = __uint_as_float((uint32_t)__ldg(pp + (size_t)j * a.N1 + 32) << 16);
            if (lean_of(MODE) == 1)
              swiglu_bwd_lean(a.prm, uu, gg, dy, du, dg);
            else if (lean_of(MODE) == 2)
              swiglu_bwd_lean_clamped(a.prm, uu, gg, dy, du, dg);
            else if (lean_of(MODE) == 3)
              geglu_bwd_lean(a.prm, uu, gg, dy, du, dg);
            else
              act_bwd(a.prm, uu, gg, dy, du, dg);
          } else {
            act_bwd(a.prm, uu, 0.0f, dy, du, dg);
          }
          u[j] = du;
          g[j] = dg;
        }
      }
      if (a.db_parts != nullptr) {
        float su = 0.0f, sg = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          su += u[j];
          sg += g[j];
        }
        float* dst = a.db_parts + (size_t)(rb / 32) * a.N1 + pu;
        dst[0] = su;
        if (gated) dst[32] = sg;
      }
      emit_block_t(a, u, pu, rb, lane, amax_bits);
      if (gated) emit_block_t(a, g, pu + 32, rb, lane, amax_bits);
    }
  }
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair::THREADS, 1)
    k_grouped_bf16_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA32,
                        const __grid_constant__ CUtensorMap tmA16, const __grid_constant__ CUtensorMap tmB,
                        const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;
  uint8_t* scratch_all = smem + pair::OFF_SCRATCH;
  int32_t* pref = reinterpret_cast<int32_t*>(smem + pair::OFF_PREF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + pair::OFF_BARS);
  uint64_t* full = bars;
  uint64_t* empty = bars + pair::STAGES;
  uint64_t* acc_full = bars + 2 * pair::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_empty + 2;
  uint64_t* tq_full = mma_done + 1;
  uint64_t* tq_empty = tq_full + pair::TQ;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + pair::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + pair::OFF_MISC + 4);
  volatile int32_t* tq = reinterpret_cast<volatile int32_t*>(smem + pair::OFF_MISC + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E;
  const uint32_t rank = cluster_ctarank();
  const int cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;

  if (warp == PRODUCER_WARP && lane == 0) {
    for (int s = 0; s < pair::STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full + b, 1);
      mbar_init(acc_empty + b, 2 * EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    for (int i = 0; i < pair::TQ; ++i) {
      mbar_init(tq_full + i, 1);
      mbar_init(tq_empty + i, pair::TQ_CONSUMERS);
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_async_shared();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmA32);
    tma_prefetch_desc(&tmA16);
    tma_prefetch_desc(&tmB);
  }
  if (warp == MMA_WARP) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  // 256-row pair tiles per expert -> exclusive prefix pref[0..E]
  for (int e = threadIdx.x; e < E; e += pair::THREADS) pref[e + 1] = (__ldg(a.counts + e) + 2 * BM - 1) / (2 * BM);
  if (threadIdx.x == 0) pref[0] = 0;
  __syncthreads();
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int beg = 1 + lane * per, end = min(E + 1, beg + per);
    int sum = 0;
    for (int i = beg; i < end; ++i) sum += pref[i];
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= d) incl += v;
    }
    int run = incl - sum;
    for (int i = beg; i < end; ++i) {
      run += pref[i];
      pref[i] = run;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers and tensor memory exist before any cross-CTA use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const bool over = __ldg(a.offsets + E) > a.R_cap;
  if (over && threadIdx.x == 0) set_status(a.status, MOE_ERR_CAPACITY);
  const int total = over ? 0 : pref[E] * a.n_tiles_n;
  const int num_kb = a.K / BK;
  WaitGuard guard{abort_flag, a.status, a.wait_ns};

  // Tile sequence of this cluster.  The leader's producer takes the next
  // tile (the scheduler's atomic counter when a.sched is set: clusters that
  // finish early take more tiles, whatever else shares the SMs; otherwise the
  // static stride cl, cl + ncl, ...), publishes it in queue slot i % TQ of
  // both CTAs and ends the sequence with -1.  Every other role reads the
  // slots in order and releases each one on the leader.
  auto tq_next = [&](int i, bool own_cta_release, int& t) -> bool {
    const int slot = i % pair::TQ;
    const uint32_t ph = (uint32_t)(i / pair::TQ) & 1u;
    if (!mbar_wait_cluster(tq_full + slot, ph, guard)) return false;
    t = tq[slot];
    if (own_cta_release)
      mbar_arrive(tq_empty + slot);
    else
      mbar_arrive_cluster(mapa_shared(smem_u32(tq_empty + slot), 0));
    return true;
  };

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int i = 0;; ++i) {
        int t;
        if (rank == 0) {
          const int slot = i % pair::TQ;
          if (!mbar_wait(tq_empty + slot, ((uint32_t)(i / pair::TQ) & 1u) ^ 1u, guard)) break;
          t = a.sched != nullptr ? atomicAdd(a.sched, 1) : cl + i * ncl;
          if (t >= total) t = -1;
          tq[slot] = t;
          st_shared_cluster(mapa_shared(smem_u32((const void*)(tq + slot)), 1), t);
          mbar_arrive(tq_full + slot);
          mbar_arrive_cluster(mapa_shared(smem_u32(tq_full + slot), 1));
        } else if (!tq_next(i, false, t)) {
          break;
        }
        if (t < 0) break;
        const Tile ti = decode_pair(t, pref, E, a.n_tiles_n, a.counts, a.offsets, a.R_cap, (int)rank, a.swap_max);
        // Only the 32-row blocks of A inside the expert's padded segment are
        // fetched: the rows past it (the second half of an expert's last pair
        // tile, mostly) feed accumulator rows the epilogue never reads.  A
        // swapped tile loads this CTA's 128 weight rows into the A slot and
        // its half of the tile's nt rows (16-row boxes) into the B slot.  The
        // leader's barrier expects both CTAs' bytes.
        const int a_blk = (ti.rows_pad + 31) / 32;
        uint32_t tx = 0;
        if (rank == 0) {
          if (ti.swap) {
            tx = 2u * pair::B_HALF + (uint32_t)ti.nt * (BK * 2);
          } else {
            const Tile tp = decode_pair(t, pref, E, a.n_tiles_n, a.counts, a.offsets, a.R_cap, 1, a.swap_max);
            tx = (uint32_t)(a_blk + (tp.rows_pad + 31) / 32) * (32 * BK * 2) + 2u * pair::B_HALF;
          }
        }
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          const int s = stage;
          if (!mbar_wait(empty + s, phase ^ 1u, guard)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = tiles + s * pair::STAGE_BYTES;
          const uint32_t bar_lead = mapa_shared(smem_u32(full + s), 0);
          if (rank == 0) mbar_arrive_expect_tx(full + s, tx);
          if (ti.swap) {
            tma_load_3d_pair(a_dst, &tmB, bar_lead, kb * BK, ti.n_idx * BN + (int)rank * (BN / 2), ti.e);
            const int half = ti.nt / 2;
            for (int i = 0; i < half / 16; ++i)
              tma_load_2d_pair(a_dst + A_TILE + i * (16 * BK * 2), &tmA16, bar_lead, kb * BK,
                               ti.tail0 + (int)rank * half + 16 * i);
          } else {
            if (a_blk == BM / 32) {
              tma_load_2d_pair(a_dst, &tmA, bar_lead, kb * BK, ti.row0);
            } else {
              for (int i = 0; i < a_blk; ++i)
                tma_load_2d_pair(a_dst + i * (32 * BK * 2), &tmA32, bar_lead, kb * BK, ti.row0 + 32 * i);
            }
            tma_load_3d_pair(a_dst + A_TILE, &tmB, bar_lead, kb * BK, ti.n_idx * BN + (int)rank * (BN / 2), ti.e);
          }
          if (++stage == pair::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0 && rank == 0) {
      const uint32_t idesc = idesc_bf16_f32(2 * BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int lt = 0;
      for (;; ++lt) {
        int t;
        if (!tq_next(lt, true, t) || t < 0) break;
        const int buf = lt & 1;
        const uint32_t aph = (uint32_t)(lt >> 1) & 1u;
        // a swapped tile multiplies the weight rows (A slot) by its nt rows
        // (B slot): M = 256, N = nt
        const Tile ti = decode_pair(t, pref, E, a.n_tiles_n, a.counts, a.offsets, a.R_cap, 0, a.swap_max);
        const uint32_t id_t = ti.swap ? idesc_bf16_f32(2 * BM, ti.nt) : idesc;
        if (!mbar_wait(acc_empty + buf, aph ^ 1u, guard)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(full + stage, phase, guard)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(tiles + stage * pair::STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_TILE;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            umma_bf16_pair(d_tmem, sdesc_kmajor_sw128(a_addr + k * 32), sdesc_kmajor_sw128(b_addr + k * 32), id_t,
                           (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit_pair_mc(empty + stage, 0x3);
          if (++stage == pair::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(acc_full + buf, 0x3);
      }
      tc_commit_pair_mc(mma_done, 0x1);
      volatile int never = 0;
      WaitGuard drain{&never, a.status, 100000000ull};
      mbar_wait(mma_done, 0, drain);
    }
  } else {
    const int q = warp & 3, h = warp >> 2;
    uint8_t* scratch = scratch_all + warp * SCRATCH_PER_WARP;
    Amax amax_bits{0u, 0u};
    int lt = 0;
    for (;; ++lt) {
      int t = -1, ok = 1;
      if (lane == 0) ok = tq_next(lt, rank == 0, t) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      t = __shfl_sync(0xFFFFFFFFu, t, 0);
      if (!ok || t < 0) break;
      const int buf = lt & 1;
      const uint32_t aph = (uint32_t)(lt >> 1) & 1u;
      if (lane == 0) ok = mbar_wait(acc_full + buf, aph, guard) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const Tile ti = decode_pair(t, pref, E, a.n_tiles_n, a.counts, a.offsets, a.R_cap, (int)rank, a.swap_max);
      const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
      if (ti.swap)
        epilogue_swapped<MODE>(a, ti, tacc, q, h, lane, (int)rank, scratch_all + (warp & ~1) * SCRATCH_PER_WARP,
                               amax_bits);
      else
        epilogue_tile<MODE>(a, ti, tacc, q, h, lane, scratch, amax_bits);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(acc_empty + buf), 0));
    }
    if (a.out_mode == MOE_OUT_NVFP4 && a.amax != nullptr) {
      const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, amax_bits.plain);
      if (lane == 0 && m != 0) atomicMax(reinterpret_cast<int*>(a.amax), (int)m);
    }
    if (a.out_mode == MOE_OUT_NVFP4 && a.rht_amax != nullptr) {
      const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, amax_bits.rht);
      if (lane == 0 && m != 0) atomicMax(reinterpret_cast<int*>(a.rht_amax), (int)m);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still touch its memory
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <int MODE>
static moe_status_t launch_pair(const void* A, const void* B, const Args& args, int sm_margin, cudaStream_t stream) {
  CUtensorMap tmA, tmA32, tmA16, tmB;
  {
    const uint64_t dims[2] = {(uint64_t)args.K, (uint64_t)args.R_cap};
    const uint64_t strides[1] = {(uint64_t)args.K * 2};
    const uint32_t box[2] = {BK, BM};
    if (!encode_tmap(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
    const uint32_t box32[2] = {BK, 32};
    if (!encode_tmap(&tmA32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, dims, strides, box32,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
    const uint32_t box16[2] = {BK, 16};
    if (!encode_tmap(&tmA16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, dims, strides, box16,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {(uint64_t)args.K, (uint64_t)args.N_gemm, (uint64_t)args.E};
    const uint64_t strides[2] = {(uint64_t)args.K * 2, (uint64_t)args.N_gemm * args.K * 2};
    const uint32_t box[3] = {BK, BN / 2, 1};
    if (!encode_tmap(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, B, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  const void* kfn = (const void*)k_grouped_bf16_pair<MODE>;
  if (!set_smem_limit(kfn, pair::SMEM_BYTES)) return MOE_ERR_CUDA;
  int clusters = max_active_pairs(kfn, pair::THREADS, pair::SMEM_BYTES);
  if (clusters <= 0) return MOE_ERR_CUDA;
  const int by_margin = (sm_count() - sm_margin) / 2;
  if (clusters > by_margin) clusters = by_margin;
  const long long tiles_bound = ((long long)args.R_cap / (2 * BM) + args.E) * args.n_tiles_n;
  if (clusters > tiles_bound) clusters = (int)tiles_bound;
  if (clusters < 1) clusters = 1;
  // thin expert tails run swapped, except in the feature-scale modes (their
  // per-row partials are laid out for the regular tile)
  Args a2 = args;
  a2.swap_max = (MODE == BWD_GLU_DOT || MODE == BWD_ELT_DOT) ? 0 : g_tail_swap_rows.load();
  if (a2.sched != nullptr && cudaMemsetAsync(a2.sched, 0, sizeof(int), stream) != cudaSuccess) return MOE_ERR_CUDA;
  k_grouped_bf16_pair<MODE><<<2 * clusters, pair::THREADS, pair::SMEM_BYTES, stream>>>(tmA, tmA32, tmA16, tmB, a2);
  count_launch();
  return launch_status();
}

template <int MODE>
static moe_status_t launch(const void* A, const void* B, const Args& args, int sm_margin, cudaStream_t stream) {
  // the NVFP4 amaxes are maxima over this call's tiles: they start from zero
  // (memset nodes in stream order, so a captured step needs no other kernel)
  if (args.out_mode == MOE_OUT_NVFP4) {
    if (args.amax && cudaMemsetAsync(args.amax, 0, sizeof(float), stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (args.rht_amax && cudaMemsetAsync(args.rht_amax, 0, sizeof(float), stream) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (g_cta_pairs.load()) return launch_pair<MODE>(A, B, args, sm_margin, stream);
  CUtensorMap tmA, tmB;
  {
    const uint64_t dims[2] = {(uint64_t)args.K, (uint64_t)args.R_cap};
    const uint64_t strides[1] = {(uint64_t)args.K * 2};
    const uint32_t box[2] = {BK, BM};
    if (!encode_tmap(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {(uint64_t)args.K, (uint64_t)args.N_gemm, (uint64_t)args.E};
    const uint64_t strides[2] = {(uint64_t)args.K * 2, (uint64_t)args.N_gemm * args.K * 2};
    const uint32_t box[3] = {BK, BN, 1};
    if (!encode_tmap(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, B, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return MOE_ERR_CUDA;
  }
  const void* kfn = (const void*)k_grouped_bf16<MODE>;
  if (!set_smem_limit(kfn, SMEM_BYTES)) return MOE_ERR_CUDA;
  const int sms = sm_count();
  int grid = sms - sm_margin;
  const long long tiles_bound = ((long long)args.R_cap / BM + args.E) * args.n_tiles_n;
  if (grid > tiles_bound) grid = (int)tiles_bound;
  if (grid < 1) grid = 1;
  k_grouped_bf16<MODE><<<grid, THREADS, SMEM_BYTES, stream>>>(tmA, tmB, args);
  count_launch();
  return launch_status();
}

static GluParams to_glu(const moe_glu_params_t* p) {
  GluParams g;
  g.act = p->act;
  g.alpha = p->alpha;
  g.up_offset = p->up_offset;
  g.gate_lo = p->gate_lo;
  g.gate_hi = p->gate_hi;
  g.up_lo = p->up_lo;
  g.up_hi = p->up_hi;
  const bool unclamped = std::isinf(p->gate_lo) && std::isinf(p->gate_hi) && std::isinf(p->up_lo) && std::isinf(p->up_hi);
  if (p->act == MOE_ACT_SWIGLU)
    g.lean = unclamped ? 1 : 2;
  else if (p->act == MOE_ACT_GEGLU && unclamped)
    g.lean = 3;
  else
    g.lean = 0;
  g.nk = -p->alpha * 1.4426950408889634f;
  return g;
}

static bool out_ok(int out_mode, const moe_act_out_t* o) {
  if (!o) return false;
  if (out_mode == MOE_OUT_MXFP8) {
    if (!o->q_row || !o->s_row) return false;
    if ((o->q_col == nullptr) != (o->s_col == nullptr)) return false;
    if (!aligned16(o->q_row) || (o->q_col && !aligned16(o->q_col))) return false;
    return true;
  }
  if (out_mode == MOE_OUT_BF16) return o->y && aligned16(o->y);
  if (out_mode == MOE_OUT_NVFP4) return o->y && aligned16(o->y) && o->amax;
  return false;
}

}  // namespace g16
}  // namespace moeglu

using namespace moeglu;

// Workspace of the bf16 grouped GEMMs: the dynamic scheduler's tile counter
// in its first 256 bytes, then (backward with a bias gradient) one column-sum
// line per 32-row block.
static constexpr size_t SCHED_BYTES = 256;
static constexpr size_t g16_sched_bytes() { return SCHED_BYTES; }

extern "C" size_t moe_grouped_fc1_workspace_size(int E, int N1, int R_cap) {
  (void)E;
  (void)N1;
  (void)R_cap;
  return SCHED_BYTES;
}

extern "C" moe_status_t moe_grouped_fc1_glu_quant_fwd(const moe_bf16* x_perm, const moe_bf16* W1p,
                                                      const moe_bf16* b1p, const float* row_scale,
                                                      const int32_t* counts, const int32_t* offsets, int E, int H,
                                                      int F, int R_cap, const moe_glu_params_t* params,
                                                      int out_mode, const moe_act_out_t* out, void* ws,
                                                      size_t ws_bytes, int sm_margin, int32_t* status,
                                                      moe_stream_t stream) {
  using namespace g16;
  if (!x_perm || !W1p || !counts || !offsets || !params || !out) return MOE_ERR_ARG;
  if (E <= 0 || E > E_MAX || H <= 0 || (H % BK) || F <= 0 || (F % 32) || R_cap <= 0 || (R_cap % BM)) return MOE_ERR_ARG;
  if (!aligned16(x_perm) || !aligned16(W1p) || (b1p && !aligned16(b1p))) return MOE_ERR_ARG;
  if (sm_margin < 0) return MOE_ERR_ARG;
  const int act = params->act;
  if (act < MOE_ACT_SWIGLU || act > MOE_ACT_NONE) return MOE_ERR_ARG;
  const bool gated = act == MOE_ACT_SWIGLU || act == MOE_ACT_GEGLU || act == MOE_ACT_GEGLU_TANH || act == MOE_ACT_SREGLU;
  const bool none = act == MOE_ACT_NONE;
  Args a{};
  a.counts = counts;
  a.offsets = offsets;
  a.E = E;
  a.K = H;
  a.F = F;
  a.R_cap = R_cap;
  a.bias = b1p;
  a.row_scale = row_scale;
  a.prm = to_glu(params);
  a.out_mode = out_mode;
  a.status = status;
  a.wait_ns = g_wait_limit_ns.load();
  if (ws != nullptr) {
    if (ws_bytes < SCHED_BYTES || (reinterpret_cast<uintptr_t>(ws) & 15)) return MOE_ERR_ARG;
    a.sched = static_cast<int*>(ws);
  }
  if (none) {
    // unfused path: the GEMM writes the bf16 pre-activation of all N1 = F columns given
    if (!out->pre || !aligned16(out->pre)) return MOE_ERR_ARG;
    a.N1 = F;  // for MOE_ACT_NONE, F is the full GEMM width
    a.N_gemm = F;
    a.out_N = F;
    a.out_mode = MOE_OUT_BF16;
    a.pre_out = reinterpret_cast<uint16_t*>(out->pre);
    a.n_tiles_n = (F + BN - 1) / BN;
    return launch<FWD_PRE>(x_perm, W1p, a, sm_margin, as_stream(stream));
  }
  if (!out_ok(out_mode, out)) return MOE_ERR_ARG;
  if (out->pre && !aligned16(out->pre)) return MOE_ERR_ARG;
  a.q_row = out->q_row;
  a.s_row = out->s_row;
  a.q_col = out->q_col;
  a.s_col = out->s_col;
  a.y = reinterpret_cast<uint16_t*>(out->y);
  a.amax = out->amax;
  if (out->rht_amax != nullptr) return MOE_ERR_ARG;  // the rotated amax belongs to the backward
  a.pre_out = reinterpret_cast<uint16_t*>(out->pre);
  a.out_N = F;
  if (gated) {
    a.N1 = 2 * F;
    a.N_gemm = 2 * F;
    a.n_tiles_n = (2 * F + BN - 1) / BN;
    if (a.prm.lean == 1) return launch<FWD_GLU_L1>(x_perm, W1p, a, sm_margin, as_stream(stream));
    if (a.prm.lean == 2) return launch<FWD_GLU_L2>(x_perm, W1p, a, sm_margin, as_stream(stream));
    if (a.prm.lean == 3) return launch<FWD_GLU_L3>(x_perm, W1p, a, sm_margin, as_stream(stream));
    return launch<FWD_GLU>(x_perm, W1p, a, sm_margin, as_stream(stream));
  }
  a.N1 = F;
  a.N_gemm = F;
  a.n_tiles_n = (F + BN - 1) / BN;
  return launch<FWD_ELT>(x_perm, W1p, a, sm_margin, as_stream(stream));
}

namespace moeglu {
// Bias gradient from the dGLU epilogue's partials: dbias[e][c] = sum over the
// expert's 32-row blocks, in block order, of parts[block][c] (fp32; 0 for an
// expert without rows).  One thread per (expert, column); a routing that
// overflowed R_cap (no GEMM tile ran) gives zeros.
__global__ void __launch_bounds__(256) k_bias_grad(const float* __restrict__ parts, const int32_t* __restrict__ offsets,
                                                   int E, int N1, int R_cap, float* __restrict__ dbias) {
  const bool over = __ldg(offsets + E) > R_cap;
  const long long n = (long long)E * N1;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int e = (int)(i / N1), c = (int)(i - (long long)e * N1);
    float s = 0.0f;
    if (!over) {
      const int b0 = __ldg(offsets + e) / 32, b1 = __ldg(offsets + e + 1) / 32;
      for (int b = b0; b < b1; ++b) s += __ldg(parts + (size_t)b * N1 + c);
    }
    dbias[i] = s;
  }
}
}  // namespace moeglu

extern "C" size_t moe_grouped_dglu_workspace_size(int N1, int R_cap) {
  if (N1 <= 0 || R_cap <= 0) return g16_sched_bytes();
  return g16_sched_bytes() + (((size_t)(R_cap / 32) * N1 * sizeof(float) + 255) & ~(size_t)255);
}

extern "C" moe_status_t moe_grouped_dglu_quant_bwd(const moe_bf16* dY_perm, const moe_bf16* W2, const moe_bf16* pre,
                                                   const float* row_scale, const int32_t* counts,
                                                   const int32_t* offsets, int E, int H, int F, int R_cap,
                                                   const moe_glu_params_t* params, int out_mode,
                                                   const moe_act_out_t* dfc1, float* dbias, void* ws,
                                                   size_t ws_bytes, int sm_margin, int32_t* status,
                                                   moe_stream_t stream) {
  using namespace g16;
  if (!dY_perm || !W2 || !pre || !counts || !offsets || !params || !dfc1) return MOE_ERR_ARG;
  if (E <= 0 || E > E_MAX || H <= 0 || (H % BK) || F <= 0 || (F % 32) || R_cap <= 0 || (R_cap % BM)) return MOE_ERR_ARG;
  if (!aligned16(dY_perm) || !aligned16(W2) || !aligned16(pre)) return MOE_ERR_ARG;
  if (sm_margin < 0) return MOE_ERR_ARG;
  const int act = params->act;
  if (act < MOE_ACT_SWIGLU || act > MOE_ACT_SREGLU) return MOE_ERR_ARG;
  if (!out_ok(out_mode, dfc1)) return MOE_ERR_ARG;
  const bool gated = act != MOE_ACT_SRELU;
  Args a{};
  a.counts = counts;
  a.offsets = offsets;
  a.E = E;
  a.K = H;
  a.F = F;
  a.R_cap = R_cap;
  a.N_gemm = F;
  a.N1 = gated ? 2 * F : F;
  a.n_tiles_n = (F + BN - 1) / BN;
  a.out_N = a.N1;
  a.row_scale = row_scale;
  a.pre_in = reinterpret_cast<const uint16_t*>(pre);
  a.prm = to_glu(params);
  a.out_mode = out_mode;
  a.q_row = dfc1->q_row;
  a.s_row = dfc1->s_row;
  a.q_col = dfc1->q_col;
  a.s_col = dfc1->s_col;
  a.y = reinterpret_cast<uint16_t*>(dfc1->y);
  a.row_dot = dfc1->row_dot;
  // NVFP4 mode: max |dFC1| and, when asked for, the amax of its transposed
  // random Hadamard rotation (what the NVFP4 cast of the transposed operand needs)
  if ((dfc1->amax != nullptr || dfc1->rht_amax != nullptr) && out_mode != MOE_OUT_NVFP4) return MOE_ERR_ARG;
  a.amax = dfc1->amax;
  a.rht_amax = dfc1->rht_amax;
  a.rht_signs = dfc1->rht_signs;
  a.status = status;
  a.wait_ns = g_wait_limit_ns.load();
  if (ws != nullptr) {
    // the scheduler's counter, then (bias gradient) one column-sum line per 32-row block
    if (ws_bytes < g16_sched_bytes() || (reinterpret_cast<uintptr_t>(ws) & 15)) return MOE_ERR_ARG;
    a.sched = static_cast<int*>(ws);
  }
  if (dbias != nullptr) {
    if (!ws || ws_bytes < moe_grouped_dglu_workspace_size(a.N1, R_cap)) return MOE_ERR_ARG;
    a.db_parts = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + g16_sched_bytes());
  }
  cudaStream_t st = as_stream(stream);
  moe_status_t rc;
  if (a.row_dot != nullptr)
    rc = gated ? launch<BWD_GLU_DOT>(dY_perm, W2, a, sm_margin, st) : launch<BWD_ELT_DOT>(dY_perm, W2, a, sm_margin, st);
  else if (gated && a.prm.lean == 1)
    rc = launch<BWD_GLU_L1>(dY_perm, W2, a, sm_margin, st);
  else if (gated && a.prm.lean == 2)
    rc = launch<BWD_GLU_L2>(dY_perm, W2, a, sm_margin, st);
  else if (gated && a.prm.lean == 3)
    rc = launch<BWD_GLU_L3>(dY_perm, W2, a, sm_margin, st);
  else
    rc = gated ? launch<BWD_GLU>(dY_perm, W2, a, sm_margin, st) : launch<BWD_ELT>(dY_perm, W2, a, sm_margin, st);
  if (rc != MOE_OK || dbias == nullptr) return rc;
  const long long n = (long long)E * a.N1;
  long long grid = (n + 255) / 256;
  if (grid > (long long)sm_count() * 8) grid = (long long)sm_count() * 8;
  k_bias_grad<<<(int)grid, 256, 0, st>>>(a.db_parts, offsets, E, a.N1, R_cap, dbias);
  count_launch();
  return launch_status();
}

// Plain grouped GEMM y[rows of e] = A[rows] . W[e]^T with bf16 operands
// (A [R_cap][K], W [E][N][K]) through the fused output stage (bf16, MXFP8
// row + column-wise, or bf16 + NVFP4 amax); the bf16 case of
// moe_grouped_fc2_fwd.  Arguments are checked by the caller except the ones
// this kernel adds (K % 64).
moe_status_t moeglu::grouped_gemm_bf16_out(const void* A, const void* W, const int32_t* counts, const int32_t* offsets,
                                           int E, int K, int N, int R_cap, int out_mode, const moe_act_out_t* out,
                                           void* ws, size_t ws_bytes, int sm_margin, int32_t* status,
                                           cudaStream_t stream) {
  using namespace g16;
  if (E > E_MAX || (K % BK) || (R_cap % BM)) return MOE_ERR_ARG;
  if (!aligned16(A) || !aligned16(W)) return MOE_ERR_ARG;
  if (!out_ok(out_mode, out) || out->rht_amax != nullptr || out->pre != nullptr || out->row_dot != nullptr)
    return MOE_ERR_ARG;
  Args a{};
  a.counts = counts;
  a.offsets = offsets;
  a.E = E;
  a.K = K;
  a.F = N;
  a.N1 = N;
  a.N_gemm = N;
  a.R_cap = R_cap;
  a.n_tiles_n = (N + BN - 1) / BN;
  a.out_N = N;
  a.prm = GluParams{};
  a.out_mode = out_mode;
  a.q_row = out->q_row;
  a.s_row = out->s_row;
  a.q_col = out->q_col;
  a.s_col = out->s_col;
  a.y = reinterpret_cast<uint16_t*>(out->y);
  a.amax = out->amax;
  a.status = status;
  a.wait_ns = g_wait_limit_ns.load();
  if (ws != nullptr && ws_bytes >= 256 && (reinterpret_cast<uintptr_t>(ws) & 15) == 0) a.sched = static_cast<int*>(ws);
  return launch<FWD_ID>(A, W, a, sm_margin, stream);
}

extern "C" int moe_dglu_row_dot_parts(int F) { return F > 0 ? 2 * ((F + g16::BN - 1) / g16::BN) : 0; }

namespace moeglu {
// One thread per routed slot: the row's partials added in slot order.
__global__ void __launch_bounds__(256) k_feature_scale_grad(const float* __restrict__ row_dot, int parts,
                                                            const int32_t* __restrict__ row_of, int n,
                                                            float* __restrict__ dprob) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int r = __ldg(row_of + i);
    float s = 0.0f;
    if (r >= 0) {
      const float* p = row_dot + (size_t)r * parts;
      for (int q = 0; q < parts; ++q) s += __ldg(p + q);
    }
    dprob[i] = s;
  }
}
}  // namespace moeglu

extern "C" moe_status_t moe_feature_scale_grad(const float* row_dot, int parts, const int32_t* row_of, int T, int k,
                                               float* dprob, moe_stream_t stream) {
  if (!row_dot || !row_of || !dprob || parts <= 0 || T <= 0 || k <= 0) return MOE_ERR_ARG;
  const long long n = (long long)T * k;
  if (n > (1ll << 31) - 1) return MOE_ERR_ARG;
  long long grid = (n + 255) / 256;
  const long long cap = (long long)sm_count() * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  k_feature_scale_grad<<<(int)grid, 256, 0, as_stream(stream)>>>(row_dot, parts, row_of, (int)n, dprob);
  count_launch();
  return launch_status();
}
