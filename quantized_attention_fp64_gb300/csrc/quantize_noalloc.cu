// sage_quantize_noalloc: the quantization prologue with its scratch in a
// buffer that lives inside the library, for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc or any allocating routine: code that
// runs under a fixed memory budget reserved up front, plug-ins handed only
// the tensors they read and write, or hosts whose allocator must not be
// entered from the calling thread. For them this entry point takes inputs
// and outputs only; the prologue's partial key sums and partial V maxima go
// to g_noalloc_scratch below, a file-scope device array of kNoAllocScratch
// bytes that every GPU loading this library holds until the process exits.
//
// In host code the name g_noalloc_scratch is only a host-side stand-in for
// the symbol, not a device address. The first call on each device therefore
// looks up the array's device address with cudaGetSymbolAddress (with that
// device current), checks the result, caches it, and passes it to the
// kernels. That first call per device should be made before any stream
// capture begins.
//
// All calls share the one array, and it keeps whatever the last call left.
// The prologue clears the part that must start at zero (its work counter and
// per-head flags) at the start of every call; every other slot it reads is
// written earlier in the same call. Calls whose
// work overlaps on the GPU (on different streams, or from different host
// threads without ordering) race on the array; order them on one stream.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/sage.h"
#include "common.cuh"

// Size of the built-in scratch buffer: 32 MiB.
constexpr size_t kNoAllocScratch = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratch];

namespace sage {
namespace {

constexpr int kMaxDev = 64;

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDev] = {};

// Device address of g_noalloc_scratch on the current device (looked up once
// per device), or nullptr with *rc set.
void* noalloc_scratch_ptr(int* rc) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev || bind_device_context(dev) != cudaSuccess) {
    *rc = SAGE_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      *rc = SAGE_ERR_CUDA;
      return nullptr;
    }
    if (major != 10 || minor != 3) {
      *rc = SAGE_ERR_ARCH;
      return nullptr;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      *rc = SAGE_ERR_CUDA;
      return nullptr;
    }
    g_noalloc_ptr[dev] = p;
  }
  *rc = SAGE_OK;
  return g_noalloc_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_in(const sage_bf16_tensor* t) {
  if (t == nullptr || t->ptr_dev == nullptr) return SAGE_ERR_NULLPTR;
  if (!aligned16(t->ptr_dev) || t->stride_b % 8 || t->stride_s % 8 || t->stride_h % 8) return SAGE_ERR_ALIGN;
  return SAGE_OK;
}

}  // namespace
}  // namespace sage

using namespace sage;

extern "C" int sage_quantize_noalloc(const sage_bf16_tensor* q, const sage_bf16_tensor* k,
                                     const sage_bf16_tensor* v, int64_t B, int64_t S, int64_t H, int64_t D,
                                     int smooth_k, const sage_quantized* out, void* cuda_stream) {
  int rc;
  if ((rc = check_problem_sizes(B, S, H, D)) != SAGE_OK) return rc;
  if ((rc = check_in(q)) != SAGE_OK || (rc = check_in(k)) != SAGE_OK || (rc = check_in(v)) != SAGE_OK) return rc;
  if (out == nullptr) return SAGE_ERR_NULLPTR;
  const void* ptrs[9] = {out->q_codes_dev, out->k_codes_dev, out->vt_codes_dev, out->q_scale_dev, out->k_scale_dev,
                         out->v_scale_dev, out->k_mean_dev,  out->q16_dev,      out->k16_dev};
  for (const void* p : ptrs) {
    if (p == nullptr) return SAGE_ERR_NULLPTR;
    if (!aligned16(p)) return SAGE_ERR_ALIGN;
  }
  // the built-in buffer bounds the problem size where the prologue uses
  // scratch at all (the cluster kernel of short sequences at D = 128 does
  // not): its scratch must fit in kNoAllocScratch bytes
  if (prologue_uses_scratch(S, D) && prologue_scratch_bytes(B, S, H, D) > kNoAllocScratch)
    return SAGE_ERR_WORKSPACE;
  void* scratch = noalloc_scratch_ptr(&rc);
  if (scratch == nullptr) return rc;
  if (B == 0 || H == 0 || S == 0) return SAGE_OK;
  const Bf16In qi{static_cast<const uint16_t*>(q->ptr_dev), q->stride_b, q->stride_s, q->stride_h};
  const Bf16In ki{static_cast<const uint16_t*>(k->ptr_dev), k->stride_b, k->stride_s, k->stride_h};
  const Bf16In vi{static_cast<const uint16_t*>(v->ptr_dev), v->stride_b, v->stride_s, v->stride_h};
  const Bundle bo{out->q_codes_dev, out->k_codes_dev, out->vt_codes_dev, out->q_scale_dev, out->k_scale_dev,
                  out->v_scale_dev, out->k_mean_dev,  out->q16_dev,      out->k16_dev};
  int* dev_err = device_error_ptr();
  if (dev_err == nullptr) return SAGE_ERR_CUDA;
  const cudaError_t e = launch_prologue(qi, ki, vi, B, S, H, D, smooth_k != 0, bo, scratch, true, dev_err,
                                        static_cast<cudaStream_t>(cuda_stream));
  return e == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA;
}
