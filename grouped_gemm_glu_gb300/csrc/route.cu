// Routing, permutation, unpermute-combine and FC1 weight repack.
//
// Sources: [MegaMoE] (hnwysp.cn article on the MegaMoE math model and
// DeepGEMM) §2.1 — y = sum over the top-k experts of p_i E_i(x) — and §4.3 —
// each expert's tokens laid out contiguously so its rows form one GEMM
// problem; [MoE-Fusion] ("Boosting MoE Training Throughput with Advanced
// Fusion Kernels") "Eliminating host-device synchronisation": the per-group
// token counts are produced and kept in device memory.
//
// Route = four launches, no host synchronisation:
//   k_route_count   per chunk of assignments, a histogram per local expert
//   k_route_scan    one CTA: exclusive scan over chunks (stable bases), the
//                   counts, the padded offsets, capacity check
//   k_route_scatter per chunk, stable rank of every assignment inside its
//                   expert (ascending flat index t*k+j) -> row_of, tok_of,
//                   prob_perm
//   k_permute_gather one warp per permuted row: 16-byte copies of x rows,
//                   zero fill of pad rows
//   k_unpermute_combine(_vec)  weighted sum of each token's rows (the combine),
//                   or the plain sum (permute backward); vector index loads
//                   for k = 4, 8
//   k_combine_warp  the same sum for the other k <= 32, one warp per token
//   k_combine_bwd   one warp per permuted row: dY_perm and dprob
//   k_permute_gather_qcol / k_combine_bwd_qcol  the gather / the combine
//                   backward by 32-row blocks, each block's rows also cast
//                   column-wise to MXFP8 (the weight-gradient operands)
#include <mutex>

#include "common.cuh"
#include "host_common.h"

namespace moeglu {

constexpr int ROUTE_THREADS = 256;
constexpr int ROUTE_WARPS = ROUTE_THREADS / 32;
constexpr int ROUTE_PER_THREAD = 8;
constexpr int ROUTE_CHUNK = ROUTE_THREADS * ROUTE_PER_THREAD;  // assignments per CTA
constexpr int ROUTE_WARP_SPAN = ROUTE_CHUNK / ROUTE_WARPS;     // contiguous assignments per warp
constexpr int ROUTE_E_MAX = 1024;
constexpr int ALIGN = 32;

// workspace: chunk_counts [n_chunks][E] int32, then one int32 overflow flag
static inline int route_chunks(int T, int k) { return (T * k + ROUTE_CHUNK - 1) / ROUTE_CHUNK; }

__global__ void __launch_bounds__(ROUTE_THREADS) k_route_count(const int32_t* __restrict__ idx, int n_assign,
                                                               int expert_begin, int E,
                                                               int32_t* __restrict__ chunk_counts) {
  __shared__ int32_t hist[ROUTE_E_MAX];
  for (int e = threadIdx.x; e < E; e += ROUTE_THREADS) hist[e] = 0;
  __syncthreads();
  const int base = blockIdx.x * ROUTE_CHUNK;
#pragma unroll
  for (int i = 0; i < ROUTE_PER_THREAD; ++i) {
    const int a = base + i * ROUTE_THREADS + threadIdx.x;
    if (a < n_assign) {
      const int e = __ldg(idx + a) - expert_begin;
      if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += ROUTE_THREADS) chunk_counts[(size_t)blockIdx.x * E + e] = hist[e];
}

// One CTA of 1024 threads.  Thread e turns column e of chunk_counts into its
// exclusive prefix over chunks (the stable base of each chunk inside the
// expert) and produces counts[e]; then a block scan gives the padded offsets.
__global__ void __launch_bounds__(1024) k_route_scan(int32_t* __restrict__ chunk_counts, int n_chunks, int E,
                                                     int R_cap, int32_t* __restrict__ counts,
                                                     int32_t* __restrict__ offsets, int32_t* __restrict__ overflow,
                                                     int32_t* status) {
  __shared__ int32_t warp_sums[32];
  const int e = threadIdx.x;
  int32_t total = 0;
  if (e < E) {
    // eight chunk counts loaded before they are rewritten (one memory round
    // trip per eight chunks instead of one per chunk)
    int c = 0;
    for (; c + 8 <= n_chunks; c += 8) {
      int32_t v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = chunk_counts[(size_t)(c + u) * E + e];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        chunk_counts[(size_t)(c + u) * E + e] = total;
        total += v[u];
      }
    }
    for (; c < n_chunks; ++c) {
      int32_t* p = chunk_counts + (size_t)c * E + e;
      const int32_t v = *p;
      *p = total;
      total += v;
    }
    counts[e] = total;
  }
  // inclusive scan of padded counts across the block
  const int32_t padded = e < E ? (total + ALIGN - 1) / ALIGN * ALIGN : 0;
  int32_t x = padded;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int32_t w = warp_sums[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t y = __shfl_up_sync(0xFFFFFFFFu, w, d);
      if (lane >= d) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int32_t incl = x + (warp > 0 ? warp_sums[warp - 1] : 0);
  if (e < E) offsets[e] = incl - padded;
  if (e == E - 1) {
    offsets[E] = incl;
    const int32_t over = incl > R_cap ? 1 : 0;
    *overflow = over;
    if (over) set_status(status, MOE_ERR_CAPACITY);
  }
}

__global__ void __launch_bounds__(ROUTE_THREADS) k_route_scatter(
    const int32_t* __restrict__ idx, const float* __restrict__ prob, int n_assign, int k, int expert_begin, int E,
    const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ overflow, int32_t* __restrict__ row_of, int32_t* __restrict__ tok_of,
    float* __restrict__ prob_perm) {
  // per warp, per expert: running rank base inside this CTA's chunk
  extern __shared__ int32_t wbase[];  // [ROUTE_WARPS][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk0 = blockIdx.x * ROUTE_CHUNK;
  const int w0 = chunk0 + warp * ROUTE_WARP_SPAN;
  const bool over = *overflow != 0;
  for (int e = threadIdx.x; e < ROUTE_WARPS * E; e += ROUTE_THREADS) wbase[e] = 0;
  // the lane's expert ids and weights of the span, loaded once up front
  constexpr int NI = ROUTE_WARP_SPAN / 32;
  int eid[NI];
  float pv[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int a = w0 + 32 * i + lane;
    eid[i] = -1;
    pv[i] = 0.0f;
    if (a < n_assign) {
      const int e = __ldg(idx + a) - expert_begin;
      if (e >= 0 && e < E) {
        eid[i] = e;
        pv[i] = __ldg(prob + a);
      }
    }
  }
  __syncthreads();
  // pass 1: per-warp histogram of its contiguous span
#pragma unroll
  for (int i = 0; i < NI; ++i)
    if (eid[i] >= 0) atomicAdd(&wbase[warp * E + eid[i]], 1);
  __syncthreads();
  // exclusive prefix over warps, plus the chunk's base within the expert
  for (int e = threadIdx.x; e < E; e += ROUTE_THREADS) {
    int32_t run = chunk_base[(size_t)blockIdx.x * E + e] + offsets[e];
    for (int w = 0; w < ROUTE_WARPS; ++w) {
      const int32_t v = wbase[w * E + e];
      wbase[w * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
  // pass 2: stable rank, 32 consecutive assignments at a time
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int a = w0 + 32 * i + lane;
    const int e = eid[i];
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    if (a < n_assign) {
      if (e >= 0 && !over) {
        const int32_t row = wbase[warp * E + e] + __popc(peers & lt_mask);
        row_of[a] = row;
        tok_of[row] = a / k;
        prob_perm[row] = pv[i];
      } else {
        row_of[a] = -1;
      }
    }
    __syncwarp();
    if (e >= 0 && (peers & lt_mask) == 0) wbase[warp * E + e] += __popc(peers);
    __syncwarp();
  }
}

// One warp per permuted row r < offsets[E]: a real row copies x[tok_of[r]],
// a pad row is zero-filled and gets tok_of = -1, prob_perm = 0.
__global__ void __launch_bounds__(256, 1) k_permute_gather(const uint4* __restrict__ x, int H8, int E,
                                                        const int32_t* __restrict__ counts,
                                                        const int32_t* __restrict__ offsets,
                                                        const int32_t* __restrict__ overflow,
                                                        int32_t* __restrict__ tok_of, float* __restrict__ prob_perm,
                                                        uint4* __restrict__ x_perm) {
  __shared__ int32_t s_off[ROUTE_E_MAX + 1];
  __shared__ int32_t s_cnt[ROUTE_E_MAX];
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    s_off[e] = offsets[e];
    if (e < E) s_cnt[e] = counts[e];
  }
  __syncthreads();
  if (*overflow) return;
  const int R = s_off[E];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int r = blockIdx.x * wpb + warp; r < R; r += gridDim.x * wpb) {
    // expert of row r: last e with s_off[e] <= r
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_off[mid] <= r) lo = mid; else hi = mid - 1;
    }
    const bool real = r < s_off[lo] + s_cnt[lo];
    uint4* dst = x_perm + (size_t)r * H8;
    if (real) {
      const int t = tok_of[r];
      const uint4* src = x + (size_t)t * H8;
      // four 16-byte loads in flight per lane before the stores
      for (int v = lane; v < H8; v += 128) {
        uint4 c[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) c[u] = v + 32 * u < H8 ? __ldg(src + v + 32 * u) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (v + 32 * u < H8) dst[v + 32 * u] = c[u];
      }
    } else {
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int v = lane; v < H8; v += 32) dst[v] = z;
      if (lane == 0) {
        tok_of[r] = -1;
        prob_perm[r] = 0.0f;
      }
    }
  }
}

// Column-wise MXFP8 of the permuted rows, fused into the kernels that write
// them (the weight gradient's operands x_perm and dY_perm; [MoE-Fusion]
// "Fusing MXFP8 and NVFP4 quantisation": MXFP8 = row-wise output plus a
// transposed copy).  A CTA of QF_THREADS owns one 32-row block (one MX block
// along the rows, inside one expert's padded segment) and walks the columns
// in chunks: warp w produces row w of the chunk (stored as by the plain
// kernel, and staged in shared memory), then two threads per column
// quantise the column's 32 values: codes to q_col [C][R_cap] (32 bytes at
// row r0), the E8M0 scale to s_col [C][R_cap / 32].  The next chunk's loads
// are in flight while a chunk is quantised.
constexpr int QF_THREADS = 1024;  // 32 warps: one per row of the block
// chunk widths: the gather 1024 columns (4 gathered 16-byte loads per lane
// and chunk), the combine backward 512 (two input streams)
template <int COLS>
struct Qf {
  static constexpr int V = COLS / 8 / 32;    // 16-byte vectors per lane and row of a chunk
  static constexpr int ROW = COLS * 2 + 16;  // staged bytes per row (padded)
  static constexpr int SMEM = 32 * ROW;
};

// Thread pair (c, h) of each group of 512 columns: rows 16h .. 16h + 15 of
// column c of the staged chunk; the pair's two 16-byte code stores fill one
// 32-byte sector, so a warp instruction writes 16 whole sectors.
template <int COLS>
__device__ __forceinline__ void qf_cast_chunk(const uint8_t* tile, int ncols, int c0, int R_cap, int r0,
                                              uint8_t* __restrict__ q_col, uint8_t* __restrict__ s_col) {
  using Q = Qf<COLS>;
  const int h = threadIdx.x & 1;
#pragma unroll 1
  for (int cg = 0; cg < COLS; cg += QF_THREADS / 2) {
    const int c = cg + (threadIdx.x >> 1);
    uint32_t v[8];  // rows 16h + 2i (low half) and 16h + 2i + 1 (high half)
    uint32_t m = 0;
    if (c < ncols) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t lo = *reinterpret_cast<const uint16_t*>(tile + (16 * h + 2 * i) * Q::ROW + 2 * c);
        const uint32_t hi = *reinterpret_cast<const uint16_t*>(tile + (16 * h + 2 * i + 1) * Q::ROW + 2 * c);
        v[i] = lo | (hi << 16);
        m = max(m, max(lo & 0x7FFFu, hi & 0x7FFFu));
      }
    }
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));  // amax of the column's 32 rows
    if (c < ncols) {
      const uint32_t sb = e8m0_from_amax_bits(m << 16);
      uint32_t codes[4];
      if (sb == 0xFFu) {
#pragma unroll
        for (int w = 0; w < 4; ++w) codes[w] = 0x7F7F7F7Fu;
      } else {
        const float inv = mx_inv_scale(sb);
#pragma unroll
        for (int w = 0; w < 4; ++w)
          codes[w] = e4m3x2(bf16_lo(v[2 * w]) * inv, bf16_hi(v[2 * w]) * inv) |
                     (e4m3x2(bf16_lo(v[2 * w + 1]) * inv, bf16_hi(v[2 * w + 1]) * inv) << 16);
      }
      *reinterpret_cast<uint4*>(q_col + (size_t)(c0 + c) * R_cap + r0 + 16 * h) =
          make_uint4(codes[0], codes[1], codes[2], codes[3]);
      if (h == 0) s_col[(size_t)(c0 + c) * (R_cap / 32) + r0 / 32] = (uint8_t)sb;
    }
  }
}

// Real rows (0..32) of the 32-row block at r0 < offsets[E]: found by one
// binary search over the offsets (each block lies inside one expert).
__device__ __forceinline__ int block_real_rows_g(const int32_t* __restrict__ counts,
                                                 const int32_t* __restrict__ offsets, int E, int r0) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(offsets + mid) <= r0) lo = mid; else hi = mid - 1;
  }
  return max(0, min(32, __ldg(offsets + lo) + __ldg(counts + lo) - r0));
}

// k_permute_gather with the column-wise MXFP8 of x_perm: one CTA per 32-row
// block below offsets[E] (the same rows, zero fill, tok_of / prob_perm of
// pad rows as k_permute_gather).
__global__ void __launch_bounds__(QF_THREADS) k_permute_gather_qcol(
    const uint4* __restrict__ x, int H, int E, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ overflow, int R_cap,
    int32_t* __restrict__ tok_of, float* __restrict__ prob_perm, uint4* __restrict__ x_perm,
    uint8_t* __restrict__ q_col, uint8_t* __restrict__ s_col) {
  using Q = Qf<1024>;
  extern __shared__ __align__(16) uint8_t qf_tile[];  // [32][Q::ROW]
  __shared__ int s_real;
  if (*overflow) return;
  const int r0 = blockIdx.x * 32;
  if (r0 >= __ldg(offsets + E)) return;
  if (threadIdx.x == 0) s_real = block_real_rows_g(counts, offsets, E, r0);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = r0 + warp;
  const bool real = warp < s_real;
  const int H8 = H / 8;
  const uint4* src = x + (real ? (size_t)__ldg(tok_of + r) * H8 : 0);
  uint4* dst = x_perm + (size_t)r * H8;
  if (!real && lane == 0) {
    tok_of[r] = -1;
    prob_perm[r] = 0.0f;
  }
  const uint4 z = make_uint4(0, 0, 0, 0);
  uint4 a[Q::V];
#pragma unroll
  for (int u = 0; u < Q::V; ++u) {
    const int v = lane + 32 * u;
    a[u] = (real && v < H8) ? __ldg(src + v) : z;
  }
  for (int c0 = 0; c0 < H; c0 += 1024) {
    const int ncols = min(1024, H - c0);
#pragma unroll
    for (int u = 0; u < Q::V; ++u) {
      const int v = lane + 32 * u;
      if (8 * v < ncols) {
        dst[c0 / 8 + v] = a[u];
        *reinterpret_cast<uint4*>(qf_tile + warp * Q::ROW + 16 * v) = a[u];
      }
    }
    __syncthreads();
    const int n0 = c0 + 1024;  // next chunk's loads, in flight during the cast
#pragma unroll
    for (int u = 0; u < Q::V; ++u) {
      const int v = n0 / 8 + lane + 32 * u;
      a[u] = (real && v < H8) ? __ldg(src + v) : z;
    }
    qf_cast_chunk<1024>(qf_tile, ncols, c0, R_cap, r0, q_col, s_col);
    __syncthreads();
  }
}

// k_combine_bwd with the column-wise MXFP8 of dY_perm: one CTA per 32-row
// block below offsets[E], warp w on row r0 + w.  The same dY_perm rows, and
// the same dprob: each lane takes the 16-byte chunks lane, lane + 32, ... of
// the row in order (as k_combine_bwd), then the warp's butterfly.
__global__ void __launch_bounds__(QF_THREADS) k_combine_bwd_qcol(
    const uint4* __restrict__ dout, const uint4* __restrict__ y_perm, const int32_t* __restrict__ row_of,
    const int32_t* __restrict__ tok_of, const float* __restrict__ prob_perm, const int32_t* __restrict__ offsets,
    int E, int T, int k, int H, int R_cap, uint4* __restrict__ dY, float* __restrict__ dprob,
    uint8_t* __restrict__ q_col, uint8_t* __restrict__ s_col, int32_t* status) {
  using Q = Qf<512>;
  extern __shared__ __align__(16) uint8_t qf_tile[];  // [32][Q::ROW]
  const size_t nthreads = (size_t)gridDim.x * blockDim.x;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (size_t i = tid; i < (size_t)T * k; i += nthreads)
    if (__ldg(row_of + i) < 0) dprob[i] = 0.0f;
  const int R = __ldg(offsets + E);
  if (R > R_cap) {
    if (tid == 0) set_status(status, MOE_ERR_CAPACITY);
    return;
  }
  const int r0 = blockIdx.x * 32;
  if (r0 >= R) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = r0 + warp;
  const int t = __ldg(tok_of + r);
  const bool real = t >= 0;
  const float p = real ? __ldg(prob_perm + r) : 0.0f;
  const int H8 = H / 8;
  const uint4* g = dout + (real ? (size_t)t * H8 : 0);
  const uint4* y = y_perm + (size_t)r * H8;
  uint4* dst = dY + (size_t)r * H8;
  const uint4 z = make_uint4(0, 0, 0, 0);
  uint4 ga[Q::V], yb[Q::V];
#pragma unroll
  for (int u = 0; u < Q::V; ++u) {
    const int v = lane + 32 * u;
    ga[u] = (real && v < H8) ? __ldg(g + v) : z;
    yb[u] = (real && v < H8) ? __ldg(y + v) : z;
  }
  float dot = 0.0f;
  for (int c0 = 0; c0 < H; c0 += 512) {
    const int ncols = min(512, H - c0);
#pragma unroll
    for (int u = 0; u < Q::V; ++u) {
      const int v = lane + 32 * u;
      if (8 * v < ncols) {
        const uint4 a = ga[u], b = yb[u];
        const float gv[8] = {bf16_lo(a.x), bf16_hi(a.x), bf16_lo(a.y), bf16_hi(a.y),
                             bf16_lo(a.z), bf16_hi(a.z), bf16_lo(a.w), bf16_hi(a.w)};
        const float yv[8] = {bf16_lo(b.x), bf16_hi(b.x), bf16_lo(b.y), bf16_hi(b.y),
                             bf16_lo(b.z), bf16_hi(b.z), bf16_lo(b.w), bf16_hi(b.w)};
#pragma unroll
        for (int i = 0; i < 8; ++i) dot = fmaf(gv[i], yv[i], dot);
        const uint4 o = real ? make_uint4(pack_bf16x2(p * gv[0], p * gv[1]), pack_bf16x2(p * gv[2], p * gv[3]),
                                          pack_bf16x2(p * gv[4], p * gv[5]), pack_bf16x2(p * gv[6], p * gv[7]))
                             : z;
        dst[c0 / 8 + v] = o;
        *reinterpret_cast<uint4*>(qf_tile + warp * Q::ROW + 16 * v) = o;
      }
    }
    __syncthreads();
    const int n0 = c0 + 512;
#pragma unroll
    for (int u = 0; u < Q::V; ++u) {
      const int v = n0 / 8 + lane + 32 * u;
      ga[u] = (real && v < H8) ? __ldg(g + v) : z;
      yb[u] = (real && v < H8) ? __ldg(y + v) : z;
    }
    qf_cast_chunk<512>(qf_tile, ncols, c0, R_cap, r0, q_col, s_col);
    __syncthreads();
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, d);
  if (real && lane < k && __ldg(row_of + (size_t)t * k + lane) == (int32_t)r) dprob[(size_t)t * k + lane] = dot;
}

// out[t] = bf16(sum_j p[t][j] * y_perm[row_of[t*k+j]]) in fp32, j ascending.
// Work items are (token, 8-element vector) pairs, consecutive threads on
// consecutive vectors of one row.
__global__ void __launch_bounds__(256, 1) k_unpermute_combine(const uint4* __restrict__ y, const int32_t* __restrict__ row_of,
                                                           const float* __restrict__ prob, int T, int H8, int k,
                                                           uint4* __restrict__ out) {
  const size_t total = (size_t)T * H8;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / H8);
    const int v = (int)(i - (size_t)t * H8);
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int j = 0; j < k; ++j) {
      const int32_t r = __ldg(row_of + (size_t)t * k + j);
      if (r < 0) continue;
      const float p = prob ? __ldg(prob + (size_t)t * k + j) : 1.0f;  // no weights: permute backward
      const uint4 w = __ldg(y + (size_t)r * H8 + v);
      acc[0] = fmaf(p, bf16_lo(w.x), acc[0]);
      acc[1] = fmaf(p, bf16_hi(w.x), acc[1]);
      acc[2] = fmaf(p, bf16_lo(w.y), acc[2]);
      acc[3] = fmaf(p, bf16_hi(w.y), acc[3]);
      acc[4] = fmaf(p, bf16_lo(w.z), acc[4]);
      acc[5] = fmaf(p, bf16_hi(w.z), acc[5]);
      acc[6] = fmaf(p, bf16_lo(w.w), acc[6]);
      acc[7] = fmaf(p, bf16_hi(w.w), acc[7]);
    }
    out[i] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                        pack_bf16x2(acc[6], acc[7]));
  }
}

// The same sum for k = 4 or 8: one thread per (token, NV 16-byte chunks
// spaced H8 / NV apart, so consecutive threads still touch consecutive
// chunks).  The token's row indices and weights arrive as 16-byte vector
// loads, and each slot's NV row loads are issued together: NV x 16 bytes in
// flight per thread at a modest register count.  Same arithmetic and order
// as above.  WP: with weights (combine); without (permute backward, every
// weight 1) is its own instantiation, since a run-time test of prob in the
// loop cost 20% (the row loads were scheduled less eagerly).  The bound of
// one CTA per SM leaves ptxas free to schedule the loads for latency.
template <int KV, int NV, bool WP>
__global__ void __launch_bounds__(256, 1) k_unpermute_combine_vec(const uint4* __restrict__ y,
                                                               const int32_t* __restrict__ row_of,
                                                               const float* __restrict__ prob, int T, int H8,
                                                               uint4* __restrict__ out) {
  const int Q = (H8 + NV - 1) / NV;
  const size_t total = (size_t)T * Q;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / Q);
    const int v0 = (int)(i - (size_t)t * Q);
    int rj[KV];
    float pj[KV];
#pragma unroll
    for (int q = 0; q < KV / 4; ++q) {
      const int4 r4 = __ldg(reinterpret_cast<const int4*>(row_of + (size_t)t * KV) + q);
      rj[4 * q] = r4.x, rj[4 * q + 1] = r4.y, rj[4 * q + 2] = r4.z, rj[4 * q + 3] = r4.w;
      if constexpr (WP) {
        const float4 p4 = __ldg(reinterpret_cast<const float4*>(prob + (size_t)t * KV) + q);
        pj[4 * q] = p4.x, pj[4 * q + 1] = p4.y, pj[4 * q + 2] = p4.z, pj[4 * q + 3] = p4.w;
      } else {
        pj[4 * q] = pj[4 * q + 1] = pj[4 * q + 2] = pj[4 * q + 3] = 1.0f;  // permute backward
      }
    }
    float acc[NV][8];
#pragma unroll
    for (int n = 0; n < NV; ++n)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[n][e] = 0.0f;
#pragma unroll
    for (int j = 0; j < KV; ++j) {
      if (rj[j] < 0) continue;
      const uint4* src = y + (size_t)rj[j] * H8;
      uint4 w[NV];
#pragma unroll
      for (int n = 0; n < NV; ++n) {
        const int v = v0 + n * Q;
        w[n] = v < H8 ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
      }
      const float p = pj[j];
#pragma unroll
      for (int n = 0; n < NV; ++n) {
        acc[n][0] = fmaf(p, bf16_lo(w[n].x), acc[n][0]);
        acc[n][1] = fmaf(p, bf16_hi(w[n].x), acc[n][1]);
        acc[n][2] = fmaf(p, bf16_lo(w[n].y), acc[n][2]);
        acc[n][3] = fmaf(p, bf16_hi(w[n].y), acc[n][3]);
        acc[n][4] = fmaf(p, bf16_lo(w[n].z), acc[n][4]);
        acc[n][5] = fmaf(p, bf16_hi(w[n].z), acc[n][5]);
        acc[n][6] = fmaf(p, bf16_lo(w[n].w), acc[n][6]);
        acc[n][7] = fmaf(p, bf16_hi(w[n].w), acc[n][7]);
      }
    }
#pragma unroll
    for (int n = 0; n < NV; ++n) {
      const int v = v0 + n * Q;
      if (v < H8)
        out[(size_t)t * H8 + v] = make_uint4(pack_bf16x2(acc[n][0], acc[n][1]), pack_bf16x2(acc[n][2], acc[n][3]),
                                             pack_bf16x2(acc[n][4], acc[n][5]), pack_bf16x2(acc[n][6], acc[n][7]));
    }
  }
}

// The same sum for the other k <= 32, one warp per token.  For k = 4, 8 the
// per-thread form above keeps a whole row's loads in flight at once and is
// faster; for other k the generic kernel issues one 16-byte load per slot and
// thread, and this one U per slot and lane.  Lanes j < k load the token's row
// index and weight once; the warp then streams the rows of the live slots:
// each lane sums U 16-byte chunks (32 apart, so a warp load is 512
// contiguous bytes of a row) over the slots in ascending j, with the same
// fmaf sequence as the kernels above.
template <int U>
__global__ void __launch_bounds__(256, 1) k_combine_warp(const uint4* __restrict__ y, const int32_t* __restrict__ row_of,
                                                      const float* __restrict__ prob, int T, int H8, int k,
                                                      uint4* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    int r = -1;
    float p = 0.0f;
    if (lane < k) {
      r = __ldg(row_of + (size_t)t * k + lane);
      p = prob ? __ldg(prob + (size_t)t * k + lane) : 1.0f;  // no weights: permute backward
    }
    const uint32_t live = __ballot_sync(0xFFFFFFFFu, r >= 0);
    for (int v0 = lane; v0 < H8; v0 += 32 * U) {
      float acc[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[u][e] = 0.0f;
      for (uint32_t m = live; m != 0; m &= m - 1) {
        const int j = __ffs(m) - 1;
        const int rj = __shfl_sync(0xFFFFFFFFu, r, j);
        const float pj = __shfl_sync(0xFFFFFFFFu, p, j);
        const uint4* src = y + (size_t)rj * H8;
        uint4 w[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + 32 * u;
          w[u] = v < H8 ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          acc[u][0] = fmaf(pj, bf16_lo(w[u].x), acc[u][0]);
          acc[u][1] = fmaf(pj, bf16_hi(w[u].x), acc[u][1]);
          acc[u][2] = fmaf(pj, bf16_lo(w[u].y), acc[u][2]);
          acc[u][3] = fmaf(pj, bf16_hi(w[u].y), acc[u][3]);
          acc[u][4] = fmaf(pj, bf16_lo(w[u].z), acc[u][4]);
          acc[u][5] = fmaf(pj, bf16_hi(w[u].z), acc[u][5]);
          acc[u][6] = fmaf(pj, bf16_lo(w[u].w), acc[u][6]);
          acc[u][7] = fmaf(pj, bf16_hi(w[u].w), acc[u][7]);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u;
        if (v < H8)
          out[(size_t)t * H8 + v] = make_uint4(pack_bf16x2(acc[u][0], acc[u][1]), pack_bf16x2(acc[u][2], acc[u][3]),
                                               pack_bf16x2(acc[u][4], acc[u][5]), pack_bf16x2(acc[u][6], acc[u][7]));
      }
    }
  }
}

// Combine backward (the chain rule on the combine above): one warp per
// permuted row r < offsets[E].  Real row (t = tok_of[r] >= 0):
//   dY_perm[r] = bf16(prob_perm[r] * dOut[t])
//   dprob[t*k + j] = <dOut[t], y_perm[r]> for the slot j with row_of = r
//                    (fp32: each lane adds its 16-byte chunks in order, then
//                    a butterfly over the warp, so the order is fixed)
// Pad rows get a zero dY_perm row; slots with row_of < 0 get dprob = 0.
__global__ void __launch_bounds__(256, 1) k_combine_bwd(const uint4* __restrict__ dout, const uint4* __restrict__ y_perm,
                                                     const int32_t* __restrict__ row_of,
                                                     const int32_t* __restrict__ tok_of,
                                                     const float* __restrict__ prob_perm,
                                                     const int32_t* __restrict__ offsets, int E, int T, int k,
                                                     int H8, int R_cap, uint4* __restrict__ dY,
                                                     float* __restrict__ dprob, int32_t* status) {
  const size_t nthreads = (size_t)gridDim.x * blockDim.x;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (size_t i = tid; i < (size_t)T * k; i += nthreads)
    if (__ldg(row_of + i) < 0) dprob[i] = 0.0f;
  int R = __ldg(offsets + E);
  if (R > R_cap) {
    if (tid == 0) set_status(status, MOE_ERR_CAPACITY);
    return;
  }
  const int lane = threadIdx.x & 31;
  const size_t nwarps = nthreads >> 5;
  for (size_t r = tid >> 5; r < (size_t)R; r += nwarps) {
    const int t = __ldg(tok_of + r);
    uint4* dst = dY + r * H8;
    if (t < 0) {
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int v = lane; v < H8; v += 32) dst[v] = z;
      continue;
    }
    const float p = __ldg(prob_perm + r);
    const uint4* g = dout + (size_t)t * H8;
    const uint4* y = y_perm + r * H8;
    float dot = 0.0f;
    for (int v = lane; v < H8; v += 32) {
      const uint4 a = __ldg(g + v), b = __ldg(y + v);
      const float ga[8] = {bf16_lo(a.x), bf16_hi(a.x), bf16_lo(a.y), bf16_hi(a.y),
                           bf16_lo(a.z), bf16_hi(a.z), bf16_lo(a.w), bf16_hi(a.w)};
      const float yb[8] = {bf16_lo(b.x), bf16_hi(b.x), bf16_lo(b.y), bf16_hi(b.y),
                           bf16_lo(b.z), bf16_hi(b.z), bf16_lo(b.w), bf16_hi(b.w)};
#pragma unroll
      for (int i = 0; i < 8; ++i) dot = fmaf(ga[i], yb[i], dot);
      dst[v] = make_uint4(pack_bf16x2(p * ga[0], p * ga[1]), pack_bf16x2(p * ga[2], p * ga[3]),
                          pack_bf16x2(p * ga[4], p * ga[5]), pack_bf16x2(p * ga[6], p * ga[7]));
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, d);
    if (lane < k && __ldg(row_of + (size_t)t * k + lane) == (int32_t)r) dprob[(size_t)t * k + lane] = dot;
  }
}

// Repack (or its inverse) of FC1 rows: one CTA per (expert, packed row).
__global__ void __launch_bounds__(128) k_repack_fc1(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
                                                    int F, int H, int inverse) {
  const int e = blockIdx.y;
  const int p = blockIdx.x;  // packed row
  const int b = p >> 6, o = p & 63;
  const int logical = o < 32 ? b * 32 + o : F + b * 32 + (o - 32);
  const size_t N1 = 2 * (size_t)F;
  const size_t from = (size_t)e * N1 + (inverse ? p : logical);
  const size_t to = (size_t)e * N1 + (inverse ? logical : p);
  if ((H & 7) == 0) {
    const uint4* s = reinterpret_cast<const uint4*>(src + from * H);
    uint4* d = reinterpret_cast<uint4*>(dst + to * H);
    for (int v = threadIdx.x; v < H / 8; v += blockDim.x) d[v] = __ldg(s + v);
  } else {
    for (int h = threadIdx.x; h < H; h += blockDim.x) dst[to * H + h] = src[from * H + h];
  }
}

}  // namespace moeglu

using namespace moeglu;

extern "C" size_t moe_route_workspace_size(int T, int k, int E) {
  if (T <= 0 || k <= 0 || E <= 0) return 256;
  return ((size_t)route_chunks(T, k) * E + 64) * sizeof(int32_t);
}

extern "C" moe_status_t moe_route_permute(const moe_bf16* x, const int32_t* topk_idx, const float* topk_prob, int T,
                                          int H, int k, int expert_begin, int E, int R_cap, moe_bf16* x_perm,
                                          int32_t* row_of, int32_t* tok_of, float* prob_perm, int32_t* counts,
                                          int32_t* offsets, uint8_t* xq_col, uint8_t* xs_col, void* ws,
                                          size_t ws_bytes, int32_t* status, moe_stream_t stream) {
  if (!x || !topk_idx || !topk_prob || !x_perm || !row_of || !tok_of || !prob_perm || !counts || !offsets || !ws)
    return MOE_ERR_ARG;
  if ((xq_col == nullptr) != (xs_col == nullptr) || (xq_col && !aligned16(xq_col))) return MOE_ERR_ARG;
  if (T <= 0 || H <= 0 || (H & 7) || k <= 0 || k > 64 || E <= 0 || E > ROUTE_E_MAX || R_cap <= 0 || (R_cap & 31))
    return MOE_ERR_ARG;
  if ((int64_t)T * k > (int64_t)INT32_MAX / 2) return MOE_ERR_ARG;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_ARG;
  if (ws_bytes < moe_route_workspace_size(T, k, E)) return MOE_ERR_ARG;
  cudaStream_t s = as_stream(stream);
  const int n_assign = T * k;
  const int n_chunks = route_chunks(T, k);
  int32_t* chunk_counts = static_cast<int32_t*>(ws);
  int32_t* overflow = chunk_counts + (size_t)n_chunks * E;
  k_route_count<<<n_chunks, ROUTE_THREADS, 0, s>>>(topk_idx, n_assign, expert_begin, E, chunk_counts);
  k_route_scan<<<1, 1024, 0, s>>>(chunk_counts, n_chunks, E, R_cap, counts, offsets, overflow, status);
  const int scatter_smem = ROUTE_WARPS * E * (int)sizeof(int32_t);
  if (scatter_smem > 48 * 1024 && !set_smem_limit((const void*)k_route_scatter, scatter_smem)) return MOE_ERR_CUDA;
  k_route_scatter<<<n_chunks, ROUTE_THREADS, scatter_smem, s>>>(topk_idx, topk_prob, n_assign, k, expert_begin, E,
                                                                 chunk_counts, offsets, overflow, row_of, tok_of,
                                                                 prob_perm);
  if (xq_col) {
    if (!set_smem_limit((const void*)k_permute_gather_qcol, Qf<1024>::SMEM)) return MOE_ERR_CUDA;
    k_permute_gather_qcol<<<R_cap / 32, QF_THREADS, Qf<1024>::SMEM, s>>>(
        reinterpret_cast<const uint4*>(x), H, E, counts, offsets, overflow, R_cap, tok_of, prob_perm,
        reinterpret_cast<uint4*>(x_perm), xq_col, xs_col);
  } else {
    const int sms = sm_count();
    const int rows_bound = R_cap;
    int grid = (rows_bound + 7) / 8;
    if (grid > sms * 8) grid = sms * 8;
    if (grid < 1) grid = 1;
    k_permute_gather<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(x), H / 8, E, counts, offsets, overflow,
                                          tok_of, prob_perm, reinterpret_cast<uint4*>(x_perm));
  }
  count_launch(4);
  return launch_status();
}

static void launch_combine(const uint4* y, const int32_t* row_of, const float* prob, int T, int H8, int k, uint4* out,
                           cudaStream_t st) {
  constexpr int NV = 4;
  const size_t cap = (size_t)sm_count() * 8;
  // the vector loads of row_of / prob need 16-byte alignment (k = 4 or 8)
  const bool vec_ok = (reinterpret_cast<uintptr_t>(row_of) & 15) == 0 &&
                      (prob == nullptr || (reinterpret_cast<uintptr_t>(prob) & 15) == 0);
  if ((k == 8 || k == 4) && vec_ok) {
    const size_t items = (size_t)T * ((H8 + NV - 1) / NV);
    size_t grid = (items + 255) / 256;
    if (grid > cap) grid = cap;
    if (k == 8 && prob)
      k_unpermute_combine_vec<8, NV, true><<<(int)grid, 256, 0, st>>>(y, row_of, prob, T, H8, out);
    else if (k == 8)
      k_unpermute_combine_vec<8, NV, false><<<(int)grid, 256, 0, st>>>(y, row_of, nullptr, T, H8, out);
    else if (prob)
      k_unpermute_combine_vec<4, NV, true><<<(int)grid, 256, 0, st>>>(y, row_of, prob, T, H8, out);
    else
      k_unpermute_combine_vec<4, NV, false><<<(int)grid, 256, 0, st>>>(y, row_of, nullptr, T, H8, out);
  } else if (k <= 32) {
    size_t grid = ((size_t)T + 7) / 8;  // 8 tokens (warps) per CTA
    if (grid > cap) grid = cap;
    k_combine_warp<4><<<(int)grid, 256, 0, st>>>(y, row_of, prob, T, H8, k, out);
  } else {
    const size_t items = (size_t)T * H8;
    size_t grid = (items + 255) / 256;
    if (grid > cap) grid = cap;
    k_unpermute_combine<<<(int)grid, 256, 0, st>>>(y, row_of, prob, T, H8, k, out);
  }
}

extern "C" moe_status_t moe_unpermute_combine(const moe_bf16* y_perm, const int32_t* row_of, const float* topk_prob,
                                              int T, int H, int k, moe_bf16* out, int32_t* status,
                                              moe_stream_t stream) {
  (void)status;
  if (!y_perm || !row_of || !topk_prob || !out) return MOE_ERR_ARG;
  if (T <= 0 || H <= 0 || (H & 7) || k <= 0) return MOE_ERR_ARG;
  if (!aligned16(y_perm) || !aligned16(out)) return MOE_ERR_ARG;
  launch_combine(reinterpret_cast<const uint4*>(y_perm), row_of, topk_prob, T, H / 8, k,
                 reinterpret_cast<uint4*>(out), as_stream(stream));
  count_launch();
  return launch_status();
}

extern "C" moe_status_t moe_combine_bwd(const moe_bf16* dout, const moe_bf16* y_perm, const int32_t* row_of,
                                        const int32_t* tok_of, const float* prob_perm, const int32_t* offsets,
                                        int T, int H, int k, int E, int R_cap, moe_bf16* dY_perm, float* dprob,
                                        uint8_t* dyq_col, uint8_t* dys_col, int32_t* status, moe_stream_t stream) {
  if (!dout || !y_perm || !row_of || !tok_of || !prob_perm || !offsets || !dY_perm || !dprob) return MOE_ERR_ARG;
  if (T <= 0 || H <= 0 || (H & 7) || k <= 0 || k > 32 || E <= 0 || E > ROUTE_E_MAX || R_cap <= 0) return MOE_ERR_ARG;
  if (!aligned16(dout) || !aligned16(y_perm) || !aligned16(dY_perm)) return MOE_ERR_ARG;
  if ((dyq_col == nullptr) != (dys_col == nullptr)) return MOE_ERR_ARG;
  if (dyq_col) {
    if ((R_cap & 31) || !aligned16(dyq_col)) return MOE_ERR_ARG;
    k_combine_bwd_qcol<<<R_cap / 32, QF_THREADS, Qf<512>::SMEM, as_stream(stream)>>>(
        reinterpret_cast<const uint4*>(dout), reinterpret_cast<const uint4*>(y_perm), row_of, tok_of, prob_perm,
        offsets, E, T, k, H, R_cap, reinterpret_cast<uint4*>(dY_perm), dprob, dyq_col, dys_col, status);
    count_launch();
    return launch_status();
  }
  int grid = sm_count() * 8;
  if (grid < 1) grid = 1;
  k_combine_bwd<<<grid, 256, 0, as_stream(stream)>>>(reinterpret_cast<const uint4*>(dout),
                                                     reinterpret_cast<const uint4*>(y_perm), row_of, tok_of,
                                                     prob_perm, offsets, E, T, k, H / 8, R_cap,
                                                     reinterpret_cast<uint4*>(dY_perm), dprob, status);
  count_launch();
  return launch_status();
}

extern "C" moe_status_t moe_permute_bwd(const moe_bf16* dx_perm, const int32_t* row_of, int T, int H, int k,
                                        moe_bf16* dx, int32_t* status, moe_stream_t stream) {
  (void)status;
  if (!dx_perm || !row_of || !dx) return MOE_ERR_ARG;
  if (T <= 0 || H <= 0 || (H & 7) || k <= 0) return MOE_ERR_ARG;
  if (!aligned16(dx_perm) || !aligned16(dx)) return MOE_ERR_ARG;
  launch_combine(reinterpret_cast<const uint4*>(dx_perm), row_of, nullptr, T, H / 8, k, reinterpret_cast<uint4*>(dx),
                 as_stream(stream));
  count_launch();
  return launch_status();
}

extern "C" moe_status_t moe_repack_fc1(const moe_bf16* W1, moe_bf16* W1p, int E, int F, int H, int inverse,
                                       moe_stream_t stream) {
  if (!W1 || !W1p || W1 == W1p || E <= 0 || F <= 0 || (F & 31) || H <= 0) return MOE_ERR_ARG;
  if ((H & 7) == 0 && (!aligned16(W1) || !aligned16(W1p))) return MOE_ERR_ARG;
  if (E > 65535) return MOE_ERR_ARG;
  dim3 grid(2 * F, E);
  k_repack_fc1<<<grid, 128, 0, as_stream(stream)>>>(W1, W1p, F, H, inverse);
  count_launch();
  return launch_status();
}

// ---------------------------------------------------------------------------
// Routing without any device allocation.
//
// Some callers cannot allocate device memory at the point where they route
// tokens: an inference or training runtime that reserves all GPU memory up
// front in its own pool, or code running inside a driver-level callback
// where cudaMalloc is not allowed.  For them, moe_route_permute_noalloc
// keeps its per-chunk scratch (the stable rank bases and the overflow flag)
// in the file-scope array below instead of a caller-provided workspace.
// The array is part of the library image: every GPU that loads the library
// holds ROUTE_STATIC_SCRATCH_BYTES of it until the process exits.
// ---------------------------------------------------------------------------
namespace moeglu {

constexpr size_t ROUTE_STATIC_SCRATCH_BYTES = 1u << 20;  // 1 MiB
static __device__ __align__(256) int32_t g_route_scratch[ROUTE_STATIC_SCRATCH_BYTES / sizeof(int32_t)];

// Device address of g_route_scratch, looked up once per device.  On the
// host the name g_route_scratch is only a stand-in for the device symbol,
// never a usable address, so the address must come from the runtime.  The
// cached address belongs to the device's primary context as it was at the
// look-up: after cudaDeviceReset the library's module is loaded afresh and
// the cached address is stale (the caller must not use this entry point on a
// device after resetting it).
static int32_t* route_scratch_ptr() {
  static std::mutex mu;
  static int32_t* ptrs[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int32_t*>(p);
  }
  return ptrs[dev];
}

}  // namespace moeglu

extern "C" size_t moe_route_noalloc_max_scratch_bytes(void) { return moeglu::ROUTE_STATIC_SCRATCH_BYTES; }

extern "C" moe_status_t moe_route_permute_noalloc(const moe_bf16* x, const int32_t* topk_idx, const float* topk_prob,
                                                  int T, int H, int k, int expert_begin, int E, int R_cap,
                                                  moe_bf16* x_perm, int32_t* row_of, int32_t* tok_of,
                                                  float* prob_perm, int32_t* counts, int32_t* offsets,
                                                  uint8_t* xq_col, uint8_t* xs_col, int32_t* status,
                                                  moe_stream_t stream) {
  using namespace moeglu;
  if (!x || !topk_idx || !topk_prob || !x_perm || !row_of || !tok_of || !prob_perm || !counts || !offsets)
    return MOE_ERR_ARG;
  if (T <= 0 || H <= 0 || (H & 7) || k <= 0 || k > 64 || E <= 0 || E > ROUTE_E_MAX || R_cap <= 0 || (R_cap & 31))
    return MOE_ERR_ARG;
  if ((int64_t)T * k > (int64_t)INT32_MAX / 2) return MOE_ERR_ARG;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_ARG;
  // the scratch this routing needs must fit the fixed array
  if (moe_route_workspace_size(T, k, E) > ROUTE_STATIC_SCRATCH_BYTES) return MOE_ERR_ARG;
  int32_t* scratch = route_scratch_ptr();
  if (!scratch) return MOE_ERR_CUDA;
  // the same launch sequence as the workspace entry point, on the fixed
  // array (every entry of it that a kernel reads is written first by an
  // earlier kernel of the same call, so nothing needs clearing)
  return moe_route_permute(x, topk_idx, topk_prob, T, H, k, expert_begin, E, R_cap, x_perm, row_of, tok_of, prob_perm,
                           counts, offsets, xq_col, xs_col, scratch, ROUTE_STATIC_SCRATCH_BYTES, status, stream);
}

namespace moeglu {

// Self-test of the bounded pipeline wait that every persistent GEMM uses:
// one thread waits, through the same guard, for phase 0 of an mbarrier.  With
// arrive != 0 the thread arrives first and the wait succeeds at once; with
// arrive == 0 nothing ever arrives, so the wait must give up after the limit,
// record MOE_ERR_TIMEOUT and return (no trap, the context stays usable).
__global__ void k_wait_selftest(int arrive, uint64_t limit_ns, int32_t* status, uint64_t* waited_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (arrive) mbar_arrive(&bar);
    WaitGuard g{&abort_flag, status, limit_ns};
    const uint64_t t0 = globaltimer_ns();
    mbar_wait(&bar, 0u, g);
    *waited_ns = globaltimer_ns() - t0;
  }
}

}  // namespace moeglu

extern "C" moe_status_t moe_wait_selftest(int arrive, int32_t* status, uint64_t* waited_ns, moe_stream_t stream) {
  if (!status || !waited_ns) return MOE_ERR_ARG;
  k_wait_selftest<<<1, 32, 0, as_stream(stream)>>>(arrive, g_wait_limit_ns.load(), status, waited_ns);
  count_launch();
  return launch_status();
}
