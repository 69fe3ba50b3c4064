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
// CTA = 7 warps, one per SM, persistent over tiles t = blockIdx.x + i*gridDim.x:
//   warps 0-3  epilogue (thread = accumulator row): fp32 -> bf16 / fp32 stores
//   warp  4    TMA producer: A and B tiles of 128 x 128 bytes, 128-byte swizzle
//   warp  5    TMEM owner + MMA issuer: per k-block, tcgen05.cp of the A and
//              B scale tiles into tensor memory, then 4 MMAs of K = 32
//              (M=128, N=128) selecting scale byte k of each 32-bit column
//   warp  6    scale loader: gathers the 4 scale bytes of each of the 128 A
//              rows and 128 B rows of the k-block into shared memory in the
//              order tcgen05.cp expects (16-byte row r holds rows r, r+32,
//              r+64, r+96), fences it to the async proxy and arrives
// Every wait is bounded (MOE_ERR_TIMEOUT + early exit, never a trap).
#include "common.cuh"
#include "host_common.h"

namespace moeglu {
namespace gmx {

constexpr int BM = 128, BN = 128, BK = 128, STAGES = 5;
constexpr int EPI_WARPS = 4;
constexpr int PRODUCER_WARP = 4, MMA_WARP = 5, SF_WARP = 6;
constexpr int THREADS = 7 * 32;
constexpr int A_TILE = BM * BK;
constexpr int B_TILE = BN * BK;
constexpr int STAGE_BYTES = A_TILE + B_TILE;
constexpr int SF_STAGE = 1024;  // 512 bytes of A scales + 512 of B scales
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SFA_COL = 2 * BN, SFB_COL = 2 * BN + 4;
constexpr int E_MAX = 1024;
constexpr int SF_PREFETCH = 4;                   // stages the scale loader runs ahead
constexpr int EPI_ROW_BYTES = 256 + 16;          // staged output row (64 words + pad)
constexpr int EPI_WARP_BYTES = 32 * EPI_ROW_BYTES;
constexpr int OFF_SF = STAGES * STAGE_BYTES;
constexpr int OFF_EPI = OFF_SF + STAGES * SF_STAGE;
constexpr int OFF_PREF = OFF_EPI + EPI_WARPS * EPI_WARP_BYTES;
constexpr int OFF_BARS = OFF_PREF + (E_MAX + 2) * 4;
constexpr int NUM_BARS = 2 * STAGES + 5;
constexpr int OFF_MISC = OFF_BARS + NUM_BARS * 8;
constexpr int SMEM_BYTES = 1024 + OFF_MISC + 64;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

struct Args {
  const int32_t* counts;
  const int32_t* offsets;
  int E, M, N, K, R_cap;   // K: fixed contraction (M-grouped); M: rows of A (K-grouped)
  int kgrouped;            // 0: FC2 / dX, 1: weight gradient
  int n_tiles_n, m_tiles;  // tiles along N; along M (K-grouped only)
  const uint8_t* As;       // A scales
  const uint8_t* Bs;       // B scales
  void* out;               // bf16 [R_cap][N] or D [E][M][N] (f32 or bf16)
  int out_f32;
  int32_t* status;
  uint64_t wait_ns;
};

struct Tile {
  int e, m0, n0;           // expert, first A row (M-grouped: permuted row), first column
  int rows_valid, rows_pad;  // M-grouped row masks
  int kseg0, kseg;         // K-grouped: first row of the expert segment and its padded length
  int num_kb;
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
    ti.num_kb = a.K / BK;
  } else {
    const int per_e = a.m_tiles * a.n_tiles_n;
    ti.e = t / per_e;
    const int local = t - ti.e * per_e;
    const int m_idx = local / a.n_tiles_n;
    ti.m0 = m_idx * BM;
    ti.n0 = (local - m_idx * a.n_tiles_n) * BN;
    ti.rows_valid = ti.rows_pad = BM;
    const int o0 = __ldg(a.offsets + ti.e), o1 = __ldg(a.offsets + ti.e + 1);
    ti.kseg0 = o0;
    ti.kseg = (o0 < 0 || o1 > a.R_cap || o1 < o0) ? 0 : o1 - o0;
    ti.num_kb = (ti.kseg + BK - 1) / BK;
  }
  return ti;
}

// Walks the (tile, k-block) stages of this CTA in the order the producer and
// the MMA issuer consume them (tiles without k-blocks contribute none).
struct StageIter {
  int t, kb, total;
  Tile ti;
  bool valid;
};

__device__ __forceinline__ void stage_iter_settle(StageIter& it, const int32_t* pref, const Args& a) {
  while (it.t < it.total) {
    it.ti = decode(it.t, pref, a);
    if (it.ti.num_kb > 0) {
      it.valid = true;
      return;
    }
    it.t += gridDim.x;
  }
  it.valid = false;
}

__device__ __forceinline__ void stage_iter_init(StageIter& it, int total, const int32_t* pref, const Args& a) {
  it.t = blockIdx.x;
  it.kb = 0;
  it.total = total;
  stage_iter_settle(it, pref, a);
}

__device__ __forceinline__ void stage_iter_next(StageIter& it, const int32_t* pref, const Args& a) {
  if (++it.kb < it.ti.num_kb) return;
  it.kb = 0;
  it.t += gridDim.x;
  stage_iter_settle(it, pref, a);
}

// The 4 scale bytes (k sub-blocks 0..3 of k-block kb) of A rows
// m0+32j+lane and B rows n0+32j+lane, j = 0..3.
__device__ __forceinline__ void load_scales(const StageIter& it, const Args& a, int lane, uint32_t* v) {
  const Tile& ti = it.ti;
  if (!a.kgrouped) {
    const int ks = a.K / 32;
    const int kbyte = it.kb * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = ti.m0 + 32 * j + lane;
      v[j] = (r < a.R_cap) ? __ldg(reinterpret_cast<const uint32_t*>(a.As + (size_t)r * ks + kbyte)) : 0u;
      const int n = ti.n0 + 32 * j + lane;
      v[4 + j] = __ldg(reinterpret_cast<const uint32_t*>(a.Bs + ((size_t)ti.e * a.N + n) * ks + kbyte));
    }
  } else {
    const int ks = a.R_cap / 32;
    const int kbyte = ti.kseg0 / 32 + it.kb * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint8_t* pa = a.As + (size_t)(ti.m0 + 32 * j + lane) * ks;
      const uint8_t* pb = a.Bs + (size_t)(ti.n0 + 32 * j + lane) * ks;
      uint32_t x = 0, y = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (kbyte + i < ks) {
          x |= (uint32_t)__ldg(pa + kbyte + i) << (8 * i);
          y |= (uint32_t)__ldg(pb + kbyte + i) << (8 * i);
        }
      }
      v[j] = x;
      v[4 + j] = y;
    }
  }
}

__global__ void __launch_bounds__(THREADS, 1)
    k_grouped_mx(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Args a) {
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
      mbar_init(full + s, 2);   // TMA transaction arrival + scale loader
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
  int total = 0;
  bool over = false;
  if (!a.kgrouped) {
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  over = __ldg(a.offsets + E) > a.R_cap;
  if (over && threadIdx.x == 0) set_status(a.status, MOE_ERR_CAPACITY);
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
          mbar_arrive_expect_tx(full + stage, STAGE_BYTES);
          if (!a.kgrouped) {
            tma_load_2d(dst, &tmA, full + stage, kb * BK, ti.m0);
            tma_load_3d(dst + A_TILE, &tmB, full + stage, kb * BK, ti.n0, ti.e);
          } else {
            tma_load_2d(dst, &tmA, full + stage, ti.kseg0 + kb * BK, ti.m0);
            tma_load_2d(dst + A_TILE, &tmB, full + stage, ti.kseg0 + kb * BK, ti.n0);
          }
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
  } else if (warp == SF_WARP) {
    // Scale loader: global loads run SF_PREFETCH stages ahead of the
    // shared-memory writes, so their latency overlaps the pipeline.
    StageIter cs, pf;
    stage_iter_init(cs, total, pref, a);
    pf = cs;
    uint32_t ring[SF_PREFETCH][8];
#pragma unroll
    for (int d = 0; d < SF_PREFETCH; ++d) {
      if (pf.valid) {
        load_scales(pf, a, lane, ring[d]);
        stage_iter_next(pf, pref, a);
      }
    }
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    while (cs.valid && ok) {
#pragma unroll
      for (int d = 0; d < SF_PREFETCH; ++d) {
        if (!cs.valid) break;
        int w = 1;
        if (lane == 0) w = mbar_wait(empty + stage, phase ^ 1u, guard) ? 1 : 0;
        w = __shfl_sync(0xFFFFFFFFu, w, 0);
        if (!w) {
          ok = false;
          break;
        }
        uint4* dsa = reinterpret_cast<uint4*>(sf + stage * SF_STAGE);
        dsa[lane] = make_uint4(ring[d][0], ring[d][1], ring[d][2], ring[d][3]);
        dsa[32 + lane] = make_uint4(ring[d][4], ring[d][5], ring[d][6], ring[d][7]);
        fence_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(full + stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        stage_iter_next(cs, pref, a);
        if (pf.valid) {
          load_scales(pf, a, lane, ring[d]);
          stage_iter_next(pf, pref, a);
        }
      }
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      const uint32_t idesc = idesc_mxf8_e8m0(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int lt = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x, ++lt) {
        const Tile ti = decode(t, pref, a);
        const int buf = lt & 1;
        const uint32_t aph = (uint32_t)(lt >> 1) & 1u;
        if (!mbar_wait(acc_empty + buf, aph ^ 1u, guard)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
        bool ok = true;
        for (int kb = 0; kb < ti.num_kb; ++kb) {
          if (!mbar_wait(full + stage, phase, guard)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(tiles + stage * STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_TILE;
          const uint32_t sf_addr = smem_u32(sf + stage * SF_STAGE);
          tc_cp_32x128b_x4(tmem_base + SFA_COL, sdesc_noswizzle(sf_addr, 128));
          tc_cp_32x128b_x4(tmem_base + SFB_COL, sdesc_noswizzle(sf_addr + 512, 128));
          const int nsub = min(4, (ti.kseg - kb * BK) / 32);
          for (int k = 0; k < nsub; ++k) {
            umma_mxf8(d_tmem, sdesc_kmajor_sw128(a_addr + k * 32), sdesc_kmajor_sw128(b_addr + k * 32),
                      idesc_with_sf_ids(idesc, (uint32_t)k, (uint32_t)k), tmem_base + SFA_COL, tmem_base + SFB_COL,
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
      tc_commit(mma_done);
      volatile int never = 0;
      WaitGuard drain{&never, a.status, 100000000ull};
      mbar_wait(mma_done, 0, drain);
    }
  } else {
    const int q = warp;
    int lt = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++lt) {
      const int buf = lt & 1;
      const uint32_t aph = (uint32_t)(lt >> 1) & 1u;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(acc_full + buf, aph, guard) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const Tile ti = decode(t, pref, a);
      const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
      if (q * 32 < ti.rows_pad) {
        const bool real = q * 32 + lane < ti.rows_valid;
        const bool empty_k = ti.num_kb == 0;
        uint8_t* stg = epi_all + q * EPI_WARP_BYTES;
        const int out_es = (a.kgrouped && a.out_f32) ? 4 : 2;      // output element size
        const int chunk_cols = 256 / out_es;                        // columns per staged pass
        // each pass stages 32 rows x 256 bytes, then stores them row by row
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += chunk_cols) {
#pragma unroll 1
          for (int c = c0; c < c0 + chunk_cols; c += 32) {
            float v[32];
            if (!empty_k) tmem_ld32(tacc + c, v);
            if (empty_k || !real) {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = 0.0f;
            }
            uint8_t* dst = stg + lane * EPI_ROW_BYTES + (c - c0) * out_es;
            if (out_es == 4) {
#pragma unroll
              for (int w = 0; w < 8; ++w)
                reinterpret_cast<float4*>(dst)[w] = make_float4(v[4 * w], v[4 * w + 1], v[4 * w + 2], v[4 * w + 3]);
            } else {
#pragma unroll
              for (int w = 0; w < 4; ++w)
                reinterpret_cast<uint4*>(dst)[w] =
                    make_uint4(pack_bf16x2(v[8 * w], v[8 * w + 1]), pack_bf16x2(v[8 * w + 2], v[8 * w + 3]),
                               pack_bf16x2(v[8 * w + 4], v[8 * w + 5]), pack_bf16x2(v[8 * w + 6], v[8 * w + 7]));
            }
          }
          __syncwarp();
          // 2 rows per instruction, 16 lanes x 16 bytes each: full 128-byte lines
          const int half = lane >> 4, ch = lane & 15;
#pragma unroll 4
          for (int rr = 0; rr < 32; rr += 2) {
            const int row = rr + half;
            const int r_local = q * 32 + row;
            if (r_local < ti.rows_pad) {
              const uint4 val = *reinterpret_cast<const uint4*>(stg + row * EPI_ROW_BYTES + ch * 16);
              uint8_t* g;
              if (!a.kgrouped)
                g = reinterpret_cast<uint8_t*>(a.out) +
                    ((size_t)(ti.m0 + r_local) * a.N + ti.n0 + c0) * 2;
              else
                g = reinterpret_cast<uint8_t*>(a.out) +
                    (((size_t)ti.e * a.M + ti.m0 + r_local) * a.N + ti.n0 + c0) * out_es;
              *reinterpret_cast<uint4*>(g + ch * 16) = val;
            }
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + buf);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

static moe_status_t launch(const CUtensorMap& tmA, const CUtensorMap& tmB, const Args& a, long long tiles_bound,
                           int sm_margin, cudaStream_t stream) {
  if (!set_smem_limit((const void*)k_grouped_mx, SMEM_BYTES)) return MOE_ERR_CUDA;
  int grid = sm_count() - sm_margin;
  if (grid > tiles_bound) grid = (int)tiles_bound;
  if (grid < 1) grid = 1;
  k_grouped_mx<<<grid, THREADS, SMEM_BYTES, stream>>>(tmA, tmB, a);
  count_launch();
  return launch_status();
}

}  // namespace gmx
}  // namespace moeglu

using namespace moeglu;

extern "C" moe_status_t moe_grouped_fc2_fwd(const uint8_t* Aq, const uint8_t* As, const uint8_t* Wq,
                                            const uint8_t* Ws, const int32_t* counts, const int32_t* offsets, int E,
                                            int K, int N, int R_cap, moe_bf16* y, int sm_margin, int32_t* status,
                                            moe_stream_t stream) {
  using namespace gmx;
  if (!Aq || !As || !Wq || !Ws || !counts || !offsets || !y) return MOE_ERR_ARG;
  if (E <= 0 || E > E_MAX || K <= 0 || (K % BK) || N <= 0 || (N % BN) || R_cap <= 0 || (R_cap % BM))
    return MOE_ERR_ARG;
  if (!aligned16(Aq) || !aligned16(Wq) || !aligned16(y) || (reinterpret_cast<uintptr_t>(As) & 3) ||
      (reinterpret_cast<uintptr_t>(Ws) & 3) || sm_margin < 0)
    return MOE_ERR_ARG;
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
  a.n_tiles_n = N / BN;
  a.m_tiles = 0;
  a.As = As;
  a.Bs = Ws;
  a.out = y;
  a.out_f32 = 0;
  a.status = status;
  a.wait_ns = g_wait_limit_ns.load();
  const long long bound = ((long long)R_cap / BM + E) * (N / BN);
  return launch(tmA, tmB, a, bound, sm_margin, as_stream(stream));
}

extern "C" moe_status_t moe_grouped_wgrad(const uint8_t* Aq, const uint8_t* As, const uint8_t* Bq, const uint8_t* Bs,
                                          const int32_t* counts, const int32_t* offsets, int E, int M, int N,
                                          int R_cap, void* D, int out_f32, int sm_margin, int32_t* status,
                                          moe_stream_t stream) {
  using namespace gmx;
  if (!Aq || !As || !Bq || !Bs || !counts || !offsets || !D) return MOE_ERR_ARG;
  if (E <= 0 || E > E_MAX || M <= 0 || (M % BM) || N <= 0 || (N % BN) || R_cap <= 0 || (R_cap % BM))
    return MOE_ERR_ARG;
  if (!aligned16(Aq) || !aligned16(Bq) || !aligned16(D) || sm_margin < 0) return MOE_ERR_ARG;
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
  a.n_tiles_n = N / BN;
  a.m_tiles = M / BM;
  a.As = As;
  a.Bs = Bs;
  a.out = D;
  a.out_f32 = out_f32 ? 1 : 0;
  a.status = status;
  a.wait_ns = g_wait_limit_ns.load();
  const long long bound = (long long)E * (M / BM) * (N / BN);
  return launch(tmA, tmB, a, bound, sm_margin, as_stream(stream));
}
