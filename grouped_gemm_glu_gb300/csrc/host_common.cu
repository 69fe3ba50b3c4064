// Host helpers of libmoeglu (see host_common.h) and the small entry points
// that launch nothing: status read-back, wait limit, launch counter.
#include <map>
#include <mutex>
#include <set>
#include <tuple>

#include "host_common.h"

namespace moeglu {

std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_cta_pairs{1};
std::atomic<int> g_tail_swap_rows{32};

int max_active_pairs(const void* kernel, int threads, int smem_bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_pair(kernel, dev);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 256, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) return 0;
  cache[key] = n;
  return n;
}

int max_active_blocks(const void* kernel, int threads, int smem_bytes) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(kernel, dev, threads, smem_bytes);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem_bytes) != cudaSuccess) return 0;
  cache[key] = n;
  return n;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

bool set_smem_limit(const void* kernel, int bytes) {
  // applied once per (kernel, device, size): later calls, including calls
  // made while a stream is being captured, only look it up
  static std::mutex mu;
  static std::set<std::tuple<const void*, int, int>> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const auto key = std::make_tuple(kernel, dev, bytes);
  std::lock_guard<std::mutex> lock(mu);
  if (done.count(key)) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  done.insert(key);
  return true;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[3];
  cuuint64_t s[2];
  cuuint32_t b[3];
  cuuint32_t es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
  const CUresult r =
      fn(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace moeglu

using namespace moeglu;

extern "C" moe_status_t moe_get_status(const int32_t* status, int32_t* host_out, moe_stream_t stream) {
  if (!status || !host_out) return MOE_ERR_ARG;
  if (cudaMemcpyAsync(host_out, status, sizeof(int32_t), cudaMemcpyDeviceToHost, as_stream(stream)) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

extern "C" void moe_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns ? ns : 1); }

extern "C" uint64_t moe_launch_count(void) { return g_launches.load(); }

extern "C" void moe_set_cta_pairs(int enable) { g_cta_pairs.store(enable ? 1 : 0); }

extern "C" moe_status_t moe_set_tail_swap(int max_rows) {
  if (max_rows < 0 || max_rows > 128 || (max_rows % 32)) return MOE_ERR_ARG;
  g_tail_swap_rows.store(max_rows);
  return MOE_OK;
}
