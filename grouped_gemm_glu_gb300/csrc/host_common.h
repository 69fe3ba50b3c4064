// Host-side helpers of libmoeglu: TMA descriptor encoding (through the
// driver entry point, so the library does not link libcuda), device
// properties, launch accounting and argument checks.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <atomic>

#include "moeglu.h"

namespace moeglu {

extern std::atomic<uint64_t> g_launches;  // kernels launched by this library
extern std::atomic<uint64_t> g_wait_limit_ns;
extern std::atomic<int> g_cta_pairs;  // bf16 GEMMs on CTA pairs (cta_group::2)
extern std::atomic<int> g_tail_swap_rows;  // pair GEMMs: swapped tail tiles of at most this many rows

inline void count_launch(int n = 1) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

inline cudaStream_t as_stream(moe_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Number of SMs of the current device (cached per device).
int sm_count();

// Clusters of 2 CTAs of `kernel` that fit on the device at once (cached per
// kernel and device); 0 on failure.
int max_active_pairs(const void* kernel, int threads, int smem_bytes);

// CTAs of `kernel` resident per SM at `threads` threads and `smem_bytes` of
// dynamic shared memory (cached; 0 on failure).
int max_active_blocks(const void* kernel, int threads, int smem_bytes);

// Opts a kernel into `bytes` of dynamic shared memory (once per kernel and
// device; returns false on failure).
bool set_smem_limit(const void* kernel, int bytes);

// Encodes a tiled TMA descriptor for a row-major tensor with dims[0] the
// contiguous dimension.  rank 2 or 3; strides_bytes has rank-1 entries.
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Which short activation form a parameter set takes (GluParams::lean):
// 1 SwiGLU without clamps, 2 clamped SwiGLU, 3 GeGLU (exact erf) without
// clamps, 0 the general forms.
inline int glu_lean_kind(const moe_glu_params_t* p) {
  const bool unclamped = __builtin_isinf(p->gate_lo) && __builtin_isinf(p->gate_hi) && __builtin_isinf(p->up_lo) &&
                         __builtin_isinf(p->up_hi);
  if (p->act == MOE_ACT_SWIGLU) return unclamped ? 1 : 2;
  if (p->act == MOE_ACT_GEGLU && unclamped) return 3;
  return 0;
}

// Plain grouped GEMM with bf16 operands through the fused output stage
// (gemm_bf16.cu; the bf16 case of moe_grouped_fc2_fwd).
moe_status_t grouped_gemm_bf16_out(const void* A, const void* W, const int32_t* counts, const int32_t* offsets, int E,
                                   int K, int N, int R_cap, int out_mode, const moe_act_out_t* out, void* ws,
                                   size_t ws_bytes, int sm_margin, int32_t* status, cudaStream_t stream);

inline moe_status_t launch_status() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moeglu
