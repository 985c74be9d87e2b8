// Host helper: TMA tensor maps through the driver's cuTensorMapEncodeTiled,
// reached via the runtime's driver entry point (no link-time libcuda).
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace sage {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

}  // namespace

bool make_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
               const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (fn == nullptr || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides_bytes[i];
  return fn(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, st, b, e,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t set_smem_limit_once(const void* func, int bytes) {
  struct Entry {
    const void* func;
    int dev, bytes;
  };
  static std::mutex mu;
  static Entry seen[128];
  static int n_seen = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_seen; ++i)
    if (seen[i].func == func && seen[i].dev == dev && seen[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  // the largest shared-memory share of the unified L1: the kernels stage
  // their data in shared memory, and kernels that fit two CTAs per SM need
  // the whole carve-out for it
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && n_seen < 128) seen[n_seen++] = Entry{func, dev, bytes};
  return e;
}

cudaError_t bind_device_context(int dev) {
  // The driver calls the library makes before its first launch (tensor-map
  // encoding) need the device's context current in the calling thread. A
  // thread that has only run runtime calls that bind nothing (a framework's
  // cached allocations, device queries) may not have it yet; cudaSetDevice
  // initializes the device's primary context and makes it current (it is no
  // stream operation, so it is also allowed while a stream is being
  // captured). Once per thread and device.
  thread_local uint64_t bound = 0;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const uint64_t bit = uint64_t(1) << dev;
  if (bound & bit) return cudaSuccess;
  cudaError_t e = cudaSetDevice(dev);
  if (e == cudaSuccess) bound |= bit;
  return e;
}

int sm_count_current() {
  static int counts[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (counts[dev] == 0) cudaDeviceGetAttribute(&counts[dev], cudaDevAttrMultiProcessorCount, dev);
  return counts[dev];
}

size_t l2_bytes_current() {
  static int sizes[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (sizes[dev] == 0) cudaDeviceGetAttribute(&sizes[dev], cudaDevAttrL2CacheSize, dev);
  return static_cast<size_t>(sizes[dev]);
}

}  // namespace sage
