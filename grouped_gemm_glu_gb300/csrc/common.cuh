// Device-side building blocks shared by the kernels of libmoeglu: status
// plumbing, bounded mbarrier waits, TMA loads, tcgen05 (MMA, tensor-memory
// allocation, loads, copies) and the MX/NVFP4 number-format helpers.
// Everything targets sm_103a and is written as inline PTX.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moeglu.h"

namespace moeglu {

// ---------------------------------------------------------------------------
// Status and time
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_status(int32_t* st, int32_t code) {
  if (st) atomicOr(st, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ uint32_t mbar_test(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok;
}

// try_wait with acquire semantics at cluster scope: for barriers that
// another CTA of the cluster arrives on after writing data the waiter reads.
__device__ __forceinline__ uint32_t mbar_test_cluster(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok;
}

// A wait that gives up.  Every pipeline wait in the persistent kernels goes
// through this: after `limit_ns` (or once another role of the CTA has given
// up) it records MOE_ERR_TIMEOUT in the status word, raises the CTA's abort
// flag and returns false so that the caller can leave its loop.
struct WaitGuard {
  volatile int* abort;
  int32_t* status;
  uint64_t limit_ns;
};

__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, const WaitGuard& g) {
  if (mbar_test(b, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test(b, parity)) return true;
    if ((it & 63u) == 0) {
      if (*g.abort) return false;
      if (globaltimer_ns() - t0 > g.limit_ns) {
        *g.abort = 1;
        set_status(g.status, MOE_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// The bounded wait with cluster-scope acquire (see mbar_test_cluster).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* b, uint32_t parity, const WaitGuard& g) {
  if (mbar_test_cluster(b, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test_cluster(b, parity)) return true;
    if ((it & 63u) == 0) {
      if (*g.abort) return false;
      if (globaltimer_ns() - t0 > g.limit_ns) {
        *g.abort = 1;
        set_status(g.status, MOE_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// 32-bit store into the shared memory of a CTA of the cluster (cluster address).
__device__ __forceinline__ void st_shared_cluster(uint32_t cluster_addr, int32_t v) {
  asm volatile("st.shared::cluster.b32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// TMA (bulk tensor copies global -> shared, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t c0,
                                            int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t c0,
                                            int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// TMA store shared -> global of a 3-D box, tracked per thread in bulk groups.
// The source must have been made visible to the async proxy
// (fence_async_shared by the writing threads) before the store is issued.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* src, int32_t c0, int32_t c1,
                                             int32_t c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the sources of every committed group have been read.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Waits until every committed group has completed (writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 1-D bulk copy global -> shared (async proxy), completion on an mbarrier.
// Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, commit, loads, copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrives once on `bar` when every tcgen05 operation this thread issued
// before it has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulator.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Block-scaled E4M3 x E4M3 MMA with E8M0 scales per 32 elements of K read
// from tensor memory.
__device__ __forceinline__ void umma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Block-scaled E2M1 x E2M1 MMA (NVFP4: packed 4-bit elements, K = 64 per
// instruction) with one E4M3 scale per 16 elements of K: each row's four
// scales of the instruction are the four bytes of its 32-bit scale column.
__device__ __forceinline__ void umma_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Copies 32 rows x 16 bytes of shared memory into 4 tensor-memory columns of
// each of the four 32-lane sub-partitions (the same data in each).
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Shared-memory matrix descriptor: K-major operand tile stored as rows of
// 128 bytes with the 128-byte swizzle (8-row atoms of 1024 bytes).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(1024u >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// Descriptor without swizzle (scale-factor copies): 8-row x 16-byte atoms,
// `sbo` bytes between atoms.
__device__ __forceinline__ uint64_t sdesc_noswizzle(uint32_t saddr, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(sbo >> 4) << 32) | (1ull << 46);
}

// Instruction descriptors (kind::f16 with bf16 operands and fp32 accumulate;
// kind::mxf8f6f4 with E4M3 operands and E8M0 scales).  Both operands K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_mxf8_e8m0(int M, int N) {
  return ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24);
}
// kind::mxf4nvf4: E2M1 operands (format code 1 of that kind), E4M3 scales
// (scale-format bit 23 clear), fp32 accumulate, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_nvf4_e4m3(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ uint32_t idesc_with_sf_ids(uint32_t idesc, uint32_t a_id, uint32_t b_id) {
  return idesc | (b_id << 4) | (a_id << 29);
}

// 32 lanes x 32 consecutive 32-bit columns per thread (thread i <- lane
// base+i), followed by the wait, so the registers are valid on return.
#define MOEGLU_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : MOEGLU_R8(0), MOEGLU_R8(8), MOEGLU_R8(16), MOEGLU_R8(24)
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 128 consecutive columns of the thread's lane (four x32 loads, one wait).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float* v) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
      "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%129];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,"
      "%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%130];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,"
      "%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%131];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : MOEGLU_R8(0), MOEGLU_R8(8), MOEGLU_R8(16), MOEGLU_R8(24), MOEGLU_R8(32), MOEGLU_R8(40), MOEGLU_R8(48),
        MOEGLU_R8(56), MOEGLU_R8(64), MOEGLU_R8(72), MOEGLU_R8(80), MOEGLU_R8(88), MOEGLU_R8(96), MOEGLU_R8(104),
        MOEGLU_R8(112), MOEGLU_R8(120)
      : "r"(taddr), "r"(taddr + 32), "r"(taddr + 64), "r"(taddr + 96)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}
#undef MOEGLU_R8

// ---------------------------------------------------------------------------
// CTA pairs (clusters of 2, tcgen05 cta_group::2)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t cta_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(cta_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on an mbarrier of another CTA of the cluster (cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMA loads into this CTA's shared memory whose completion is reported to
// the mbarrier of the pair's leader CTA (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int32_t c0,
                                                 int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int32_t c0,
                                                 int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, "
      "%5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D (+)= A * B^T over the CTA pair: M = 256 (128 rows of A in each CTA's
// shared memory, 128 accumulator rows in each CTA's tensor memory), B split
// by N between the two CTAs.  Issued by one thread of the even CTA.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on the mbarrier at this shared-memory offset in every CTA of
// `cta_mask` when the pair's prior tcgen05 operations have completed.
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------
// |x| as ordered unsigned bits (NaN sorts above +Inf).
__device__ __forceinline__ uint32_t abs_bits(float x) { return __float_as_uint(x) & 0x7FFFFFFFu; }

// E8M0 block scale from the block's amax bits: OCP MX shared exponent
// floor(log2 amax) - 8 (E4M3 emax), clamped to the E8M0 range; 0xFF (NaN)
// for a non-finite amax.  floor(log2) of a normal float is its exponent
// field - 127; subnormal amax clamps to the floor.
__device__ __forceinline__ uint32_t e8m0_from_amax_bits(uint32_t amax_bits) {
  const uint32_t ex = amax_bits >> 23;
  return ex == 0xFFu ? 0xFFu : (ex > 8u ? ex - 8u : 0u);
}
// 2^(127 - byte) as a float (the exact multiplier that brings the block
// into E4M3 range); valid for byte <= 253.
__device__ __forceinline__ float mx_inv_scale(uint32_t sbyte) { return __uint_as_float((254u - sbyte) << 23); }

// Two floats -> two E4M3 bytes (round to nearest even, saturating), a in
// the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // a -> low half
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Quantises 32 floats of one MX block: returns the scale byte and writes
// the 32 codes (8 words, element 0 in the low byte of word 0).
__device__ __forceinline__ uint32_t mx_quant_block32(const float* v, uint32_t* codes) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) m = max(m, abs_bits(v[i]));
  const uint32_t sb = e8m0_from_amax_bits(m);
  if (sb == 0xFFu) {
#pragma unroll
    for (int w = 0; w < 8; ++w) codes[w] = 0x7F7F7F7Fu;
    return sb;
  }
  const float inv = mx_inv_scale(sb);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t lo = e4m3x2(v[4 * w] * inv, v[4 * w + 1] * inv);
    const uint32_t hi = e4m3x2(v[4 * w + 2] * inv, v[4 * w + 3] * inv);
    codes[w] = lo | (hi << 16);
  }
  return sb;
}

// ---------------------------------------------------------------------------
// Activations (fp32).  Textbook GLU family; see moe_act_t.
// ---------------------------------------------------------------------------
struct GluParams {
  int act;
  float alpha, up_offset, gate_lo, gate_hi, up_lo, up_hi;
  int lean;  // short forms below: SwiGLU 1 (no clamp bound finite) / 2 (clamped), GeGLU 3 (no clamp)
  float nk;  // -alpha * log2(e), for the short forms
};

// logistic function with the approximate divide (about 2 ulp): it feeds
// bf16 / MXFP8 outputs, and an IEEE divide here is a large share of the
// epilogue's instructions
__device__ __forceinline__ float sigmoidf_(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }
// Normal CDF as erfc(-z / sqrt 2) / 2: the erfc form keeps its relative
// precision in the negative tail, where 1 + erf(z / sqrt 2) cancels to 0 for
// z below about -5.9 in single precision.
__device__ __forceinline__ float phi_cdf(float z) { return 0.5f * erfcf(-z * 0.70710678118654752f); }
__device__ __forceinline__ float phi_pdf(float z) { return 0.39894228040143268f * __expf(-0.5f * z * z); }

// Short SwiGLU forms for GluParams::lean (no clamps).  sigma(alpha g) =
// 1 / (1 + 2^(nk g)) with nk = -alpha log2(e) folded on the host (exp(x) =
// 2^(x log2 e)); 2^x is the hardware approximation (ex2.approx), the divide
// the approximate one.  Backward uses d/dg [g sigma(alpha g)] =
// sigma + alpha (g sigma)(1 - sigma).
__device__ __forceinline__ float ex2_hw(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float swiglu_fwd_lean(const GluParams& p, float u, float g) {
  const float s = __fdividef(1.0f, 1.0f + ex2_hw(p.nk * g));
  return (u + p.up_offset) * (g * s);
}
__device__ __forceinline__ void swiglu_bwd_lean(const GluParams& p, float u, float g, float dy, float& du,
                                                float& dg) {
  const float s = __fdividef(1.0f, 1.0f + ex2_hw(p.nk * g));
  const float gs = g * s;
  du = dy * gs;
  dg = dy * (u + p.up_offset) * fmaf(p.alpha * gs, 1.0f - s, s);
}
// GeGLU (exact erf) without clamps: y = (u + c) g Phi(g),
// d/dg [g Phi(g)] = Phi(g) + g phi(g).
__device__ __forceinline__ float phi_cdf(float z);
__device__ __forceinline__ float phi_pdf(float z);
__device__ __forceinline__ float geglu_fwd_lean(const GluParams& p, float u, float g) {
  return (u + p.up_offset) * (g * phi_cdf(g));
}
__device__ __forceinline__ void geglu_bwd_lean(const GluParams& p, float u, float g, float dy, float& du, float& dg) {
  const float c = phi_cdf(g);
  du = dy * (g * c);
  dg = dy * (u + p.up_offset) * fmaf(g, phi_pdf(g), c);
}
// SwiGLU with the clamps (GPT-OSS: gate clamped to [gate_lo, gate_hi]);
// the derivative of a clamp is 1 on the closed interval and 0 outside.
__device__ __forceinline__ float swiglu_fwd_lean_clamped(const GluParams& p, float u, float g) {
  const float gc = fminf(fmaxf(g, p.gate_lo), p.gate_hi);
  const float uc = fminf(fmaxf(u, p.up_lo), p.up_hi) + p.up_offset;
  const float s = __fdividef(1.0f, 1.0f + ex2_hw(p.nk * gc));
  return uc * (gc * s);
}
__device__ __forceinline__ void swiglu_bwd_lean_clamped(const GluParams& p, float u, float g, float dy, float& du,
                                                        float& dg) {
  const float gc = fminf(fmaxf(g, p.gate_lo), p.gate_hi);
  const float uc = fminf(fmaxf(u, p.up_lo), p.up_hi) + p.up_offset;
  const bool in_g = g >= p.gate_lo && g <= p.gate_hi, in_u = u >= p.up_lo && u <= p.up_hi;
  const float s = __fdividef(1.0f, 1.0f + ex2_hw(p.nk * gc));
  const float gs = gc * s;
  du = in_u ? dy * gs : 0.0f;
  dg = in_g ? dy * uc * fmaf(p.alpha * gs, 1.0f - s, s) : 0.0f;
}

// forward: y = act(u, g); sReLU uses u only
__device__ __forceinline__ float act_fwd(const GluParams& p, float u, float g) {
  if (p.act == MOE_ACT_SRELU) {
    const float r = fmaxf(u, 0.0f);
    return r * r;
  }
  const float gc = fminf(fmaxf(g, p.gate_lo), p.gate_hi);
  const float uc = fminf(fmaxf(u, p.up_lo), p.up_hi) + p.up_offset;
  float f;
  if (p.act == MOE_ACT_SWIGLU) {
    f = gc * sigmoidf_(p.alpha * gc);
  } else if (p.act == MOE_ACT_GEGLU) {
    f = gc * phi_cdf(gc);
  } else if (p.act == MOE_ACT_GEGLU_TANH) {
    const float k = 0.79788456080286536f;
    f = 0.5f * gc * (1.0f + tanhf(k * (gc + 0.044715f * gc * gc * gc)));
  } else {  // sReGLU
    const float r = fmaxf(gc, 0.0f);
    f = r * r;
  }
  return uc * f;
}

// backward: (du, dg) for incoming dy
__device__ __forceinline__ void act_bwd(const GluParams& p, float u, float g, float dy, float& du, float& dg) {
  if (p.act == MOE_ACT_SRELU) {
    du = dy * 2.0f * fmaxf(u, 0.0f);
    dg = 0.0f;
    return;
  }
  const float gc = fminf(fmaxf(g, p.gate_lo), p.gate_hi);
  const float uc = fminf(fmaxf(u, p.up_lo), p.up_hi) + p.up_offset;
  const float mg = (g >= p.gate_lo && g <= p.gate_hi) ? 1.0f : 0.0f;
  const float mu = (u >= p.up_lo && u <= p.up_hi) ? 1.0f : 0.0f;
  float f, df;
  if (p.act == MOE_ACT_SWIGLU) {
    const float s = sigmoidf_(p.alpha * gc);
    f = gc * s;
    df = s * (1.0f + p.alpha * gc * (1.0f - s));
  } else if (p.act == MOE_ACT_GEGLU) {
    const float c = phi_cdf(gc);
    f = gc * c;
    df = c + gc * phi_pdf(gc);
  } else if (p.act == MOE_ACT_GEGLU_TANH) {
    const float k = 0.79788456080286536f;
    const float t = tanhf(k * (gc + 0.044715f * gc * gc * gc));
    f = 0.5f * gc * (1.0f + t);
    df = 0.5f * (1.0f + t) + 0.5f * gc * (1.0f - t * t) * k * (1.0f + 3.0f * 0.044715f * gc * gc);
  } else {
    const float r = fmaxf(gc, 0.0f);
    f = r * r;
    df = 2.0f * r;
  }
  du = dy * f * mu;
  dg = dy * uc * df * mg;
}

}  // namespace moeglu
