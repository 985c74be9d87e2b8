// Shared definitions for the CUDA side of the library (kernels and C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace sage {

constexpr int kHeadDim = 128;     // the head dimension of the pages' workload (64 is also supported)
constexpr int kQKBlock = 32;      // tokens per Q/K scale block ("per 32-row block")
constexpr int kKeyTile = 128;     // keys per online-softmax step; S is padded to this
constexpr float kInt8Max = 127.0f;
constexpr float kE4M3Max = 448.0f;  // largest finite e4m3fn magnitude
constexpr float kPScale = 448.0f;   // p in [0,1] is stored as e4m3(448 p)

__host__ __device__ inline int64_t padded_len(int64_t s) { return (s + kKeyTile - 1) / kKeyTile * kKeyTile; }
__host__ __device__ inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Device error word values: a kernel gave up a bounded wait, or found its
// dynamic shared memory not 1024-byte aligned (it returns before any work).
constexpr int kDevErrTimeout = 1;
constexpr int kDevErrSmemAlign = 2;

// One BF16 input: element (b, s, h, d) at p[b*sb + s*ss + h*sh + d].
struct Bf16In {
  const uint16_t* p;
  int64_t sb, ss, sh;
};

// The quantized bundle (device pointers), mirroring sage_quantized.
struct Bundle {
  int8_t* q_codes;
  int8_t* k_codes;
  uint8_t* vt_codes;
  float* q_scale;
  float* k_scale;
  float* v_scale;
  float* k_mean;
  uint16_t* q16;  // fp16 copies of the codes, [B][H][S_pad][128]
  uint16_t* k16;
};

// BF16 output: element (b, s, h, d) at p[b*sb + s*ss + h*sh + d].
struct Out {
  uint16_t* p;
  int64_t sb, ss, sh;
};

// TMA tensor map over `rank` dimensions (dims[0] contiguous); strides_bytes
// holds rank-1 byte strides of dims 1..rank-1. Returns false on failure.
bool make_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
               const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle);
int sm_count_current();        // SMs of the current device (cached)
// cudaFuncSetAttribute(func, MaxDynamicSharedMemorySize, bytes) and the
// largest shared-memory carve-out on the current device, skipped when it was
// already done there for at least that many bytes (the calls cost
// microseconds, which short calls notice).
cudaError_t set_smem_limit_once(const void* func, int bytes);
size_t l2_bytes_current();     // L2 bytes of the current device (cached)
// Makes the context of device `dev` (the current device) current in the
// calling thread, once per thread and device.
cudaError_t bind_device_context(int dev);

// Launchers implemented by the kernel translation units. Each enqueues on
// `stream` and returns the launch status (cudaGetLastError).
// write_int8: also store the int8 Q/K codes (the fp16 copies, V codes and
// all scales are always written). dev_err: the device error word.
// D: the head dimension (128 or 64; 64 runs the same kernels on head pairs).
cudaError_t launch_prologue(const Bf16In& q, const Bf16In& k, const Bf16In& v, int64_t B, int64_t S,
                            int64_t H, int64_t D, bool smooth_k, const Bundle& out, void* scratch, bool write_int8,
                            int* dev_err, cudaStream_t stream);
// Device address of the current device's error word (set up on first use),
// or nullptr if the runtime call fails.
int* device_error_ptr();
size_t prologue_scratch_bytes(int64_t B, int64_t S, int64_t H, int64_t D);
// Whether launch_prologue touches its scratch for this shape (the cluster
// kernel of short sequences does not).
bool prologue_uses_scratch(int64_t S, int64_t D);
// The size limits every entry point applies: SAGE_OK or a negative SAGE_ERR_*
// code (SHAPE, HEAD_DIM, TOO_LARGE).
int check_problem_sizes(int64_t B, int64_t S, int64_t H, int64_t D);

cudaError_t launch_attention_simt(const Bundle& in, int64_t B, int64_t S, int64_t H, float sm_scale,
                                  const Out& out, bool causal, float* lse, cudaStream_t stream);

// causal: query i sees keys j <= i only. lse: null, or [B][H][S] fp32 that
// receives each row's natural-log log-sum-exp of its logits (of the keys the
// bundle holds, i.e. of k - mean when it was quantized with smooth_k).
cudaError_t launch_attention_tc(const Bundle& in, int64_t B, int64_t S, int64_t H, int64_t D, float sm_scale,
                                const Out& out, bool causal, float* lse, int* dev_err, cudaStream_t stream);

// Test of the bounded wait: one warp waits, with the attention kernel's
// bounded wait, on an mbarrier that nothing completes; when the wait runs out
// the kernel sets *dev_err and returns.
cudaError_t launch_wait_timeout_selftest(int* dev_err, cudaStream_t stream);

// Adds sm_scale * q_i . k_mean to lse[b][h][i] (the smooth_k term that turns
// the log-sum-exp of the mean-reduced keys into that of the original keys).
cudaError_t launch_lse_smooth_k_term(const Bf16In& q, const float* k_mean, int64_t B, int64_t S, int64_t H,
                                     int64_t D, float sm_scale, float* lse, cudaStream_t stream);

}  // namespace sage
