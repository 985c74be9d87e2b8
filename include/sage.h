/*
 * sage.h - C ABI of a GB300 (sm_103a) implementation of SageAttention-style
 * quantized, non-causal attention on BF16 [B, S, H, 128] inputs.
 *
 * The operation (sources are web pages, cited by title and section):
 *
 *  - "aiter-sage-attention: SageAttention for AMD RDNA4 (gfx1201) #1222",
 *    section "The kernel": QK^T is computed in INT8 and PV in FP8, both with
 *    FP32 accumulation; Q and K are quantized per 32-row block and V per
 *    channel. Section "What I have so far": the entry
 *    sageattn(q, k, v, tensor_layout, is_causal, sm_scale, return_lse) raises
 *    on causal, LSE, non-BF16, head dim other than 128 and unequal Q/K/V
 *    shapes instead of falling back silently.
 *  - "Hand-written prologue: faster short calls, no compiler, RX 9060 XT
 *    opt-in (v0.4.0)", section "What changed": the quantization prologue
 *    uses 64-bit offsets (no sequence-length ceiling) and, with smooth_k on,
 *    sums the key mean in fp64.
 *  - "gfx1201 (RDNA4) SageAttention attention backend: aiter package or Hub
 *    kernel?", section "原因分析" (cause analysis): BF16 [B, S, H, 128],
 *    Q/K/V of one shape, no mask, not causal.
 *
 * Arithmetic fixed by this library where the pages are silent (the same
 * readings the test oracle follows):
 *  - Q and K: one fp32 scale per 32 consecutive tokens of one (batch, head)
 *    over all 128 channels, s = amax / 127; code = rint_even(x / s) with x / s
 *    correctly rounded in fp32, in [-127, 127]. K is first reduced by its
 *    per-channel mean when smooth_k is on: k' = fl32(k - mean).
 *  - Key mean: per 32-token chunk a left-to-right fp64 sum from +0.0, chunk
 *    sums combined by a pairwise tree; mean = fl32(total / S) in fp64.
 *  - V: one fp32 scale per (batch, head, channel) over all tokens,
 *    s_v = amax / 448; code = e4m3fn(v / s_v), round to nearest even,
 *    saturating to +-448.
 *  - Attention: logits = S_int * (s_q * s_k) * sm_scale, online softmax in
 *    fp32 over 128-key tiles in ascending order with the exact running
 *    maximum; P stored as e4m3(448 * p); the row sum uses the unquantized p;
 *    O = acc / l * s_v / 448, rounded to bf16 in the input layout.
 *
 * Conventions for every entry point:
 *  - Pointers named *_dev are CUDA device pointers; the caller owns every
 *    buffer. The library allocates no memory and keeps no state between
 *    calls except one device-side error word per GPU (see sage_device_error).
 *  - Work is enqueued on the caller's stream (a cudaStream_t passed as
 *    void*; NULL is the legacy default stream) and runs asynchronously; the
 *    call returns once the work is enqueued.
 *  - Sizes are int64_t. Every offset inside the kernels is 64-bit.
 *  - Return value: SAGE_OK (0) or a negative SAGE_ERR_* code. Arguments are
 *    validated before anything is enqueued; on error nothing is launched.
 *    There is no fallback path of any kind.
 *  - S_pad = ceil(S / 128) * 128 (one key tile). Padded code rows/columns
 *    and padded scale blocks are written as zero.
 *  - S = 0 (or B = 0 or H = 0) is an empty problem: validated, nothing
 *    launched, SAGE_OK.
 *  - Device entries work on the current device (cudaGetDevice) in its
 *    runtime primary context: a thread's first such call on a device makes
 *    that context current in the thread (cudaSetDevice), which the
 *    tensor-map encoding before the first launch needs. A driver-API
 *    context the thread had made current is replaced by it. Calls from
 *    several threads are safe as long as they do not share a scratch or
 *    workspace buffer (see sage_sageattn).
 */
#ifndef SAGE_H
#define SAGE_H

#include <stddef.h>
#include <stdint.h>

/* Symbols of the shared library are hidden except these entry points. */
#if defined(__GNUC__)
#define SAGE_API __attribute__((visibility("default")))
#else
#define SAGE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- errors -- */
enum {
  SAGE_OK = 0,
  SAGE_ERR_CAUSAL = -1,         /* is_causal != 0 (no mask support) */
  SAGE_ERR_LSE = -2,            /* return_lse != 0 */
  SAGE_ERR_DTYPE = -3,          /* an input or output is not BF16 */
  SAGE_ERR_HEAD_DIM = -4,       /* D != 128 (D = 64 is also taken by the bundle entries and sage_sageattn_ex) */
  SAGE_ERR_SHAPE = -5,          /* Q, K, V shapes differ, or a size is negative */
  SAGE_ERR_LAYOUT = -6,         /* tensor_layout is neither "NHD" nor "HND", or channel stride != 1 */
  SAGE_ERR_ALIGN = -7,          /* a base pointer is not 16-byte aligned, or a stride is not a multiple of 8 elements */
  SAGE_ERR_NULLPTR = -8,        /* a required pointer is NULL */
  SAGE_ERR_WORKSPACE = -9,      /* workspace or scratch smaller than required */
  SAGE_ERR_ARCH = -10,          /* current device is not compute capability 10.3 */
  SAGE_ERR_CUDA = -11,          /* a CUDA runtime call or kernel launch failed */
  SAGE_ERR_DEVICE_TIMEOUT = -12,/* a kernel gave up waiting on an internal barrier (see sage_device_error) */
  SAGE_ERR_ARG = -13,           /* another invalid argument (e.g. non-finite or non-positive sm_scale) */
  SAGE_ERR_TOO_LARGE = -14,     /* sizes exceed the library's index limits */
  SAGE_ERR_DEVICE_SMEM = -15    /* a kernel's dynamic shared memory was not 1024-byte aligned; it did no work */
};

/* dtype codes for sage_sageattn */
enum { SAGE_DTYPE_BF16 = 0, SAGE_DTYPE_F16 = 1, SAGE_DTYPE_F32 = 2, SAGE_DTYPE_OTHER = 3 };

/* ------------------------------------------------------------ data types -- */

/* One BF16 input tensor: element (b, s, h, d) lives at
 *   ptr_dev + b*stride_b + s*stride_s + h*stride_h + d      (in elements).
 * The channel stride is 1. "NHD" ([B,S,H,D], contiguous) has
 * stride_b = S*H*D, stride_s = H*D, stride_h = D; "HND" ([B,H,S,D]) has
 * stride_b = H*S*D, stride_h = S*D, stride_s = D. */
typedef struct sage_bf16_tensor {
  const void* ptr_dev;
  int64_t stride_b, stride_s, stride_h;
} sage_bf16_tensor;

/* The quantized bundle written by sage_quantize and read by sage_attention.
 * All pointers are device pointers, 16-byte aligned. D = 128 (or 64).
 *   q_codes, k_codes : int8   [B][H][S_pad][D]     (rows S..S_pad-1 are 0)
 *   vt_codes         : e4m3fn [B][H][D][S_pad]     (V transposed; cols S..S_pad-1 are 0)
 *   q_scale, k_scale : float  [B][H][S_pad/32]     (blocks past ceil(S/32) are 0)
 *   v_scale          : float  [B][H][D]
 *   k_mean           : float  [B][H][D]            (0 when smooth_k is off)
 *   q16, k16         : fp16   [B][H][S_pad][D]     the same Q and K codes as fp16
 *                      values (exact: |code| <= 127). sm_103a has no integer
 *                      tensor-core MMA, so the attention kernel multiplies the
 *                      codes on the fp16 tensor cores; writing them once here
 *                      saves every CTA of the attention kernel from re-widening
 *                      each key tile. */
typedef struct sage_quantized {
  int8_t* q_codes_dev;
  int8_t* k_codes_dev;
  uint8_t* vt_codes_dev;
  float* q_scale_dev;
  float* k_scale_dev;
  float* v_scale_dev;
  float* k_mean_dev;
  uint16_t* q16_dev;
  uint16_t* k16_dev;
} sage_quantized;

/* ----------------------------------------------------------- size queries -- */

/* Bytes of one quantized bundle for (B, S, H, D), each array starting on a
 * 256-byte boundary, in the order of sage_quantized's fields. If base_dev is
 * not NULL, *bundle receives pointers carved from base_dev (which must be
 * 256-byte aligned and at least *bytes long). Errors: SHAPE, HEAD_DIM,
 * TOO_LARGE, NULLPTR (bytes NULL, or bundle NULL with base_dev set),
 * ALIGN (base_dev misaligned). */
SAGE_API int sage_bundle_size(int64_t B, int64_t S, int64_t H, int64_t D, size_t* bytes,
                     void* base_dev, sage_quantized* bundle);

/* Scratch bytes sage_quantize needs (a work counter and per-head flags,
 * per-128-token partial key sums in fp64 and partial V maxima, and each
 * head's reciprocals of its V scales).
 * Errors: as sage_bundle_size. */
SAGE_API int sage_quantize_scratch_size(int64_t B, int64_t S, int64_t H, int64_t D, size_t* bytes);

/* Workspace bytes sage_sageattn needs: one bundle plus the quantize scratch. */
SAGE_API int sage_workspace_size(int64_t B, int64_t S, int64_t H, int64_t D, size_t* bytes);

/* Device workspace bytes sage_sageattn_host needs for n_groups head groups
 * (0: the library's choice): device copies of q, k, v and out, and one
 * bundle plus quantize scratch for each of two groups in flight.
 * Errors: as sage_bundle_size; ARG for n_groups < 0. */
SAGE_API int sage_host_workspace_size(int64_t B, int64_t S, int64_t H, int64_t D, int n_groups, size_t* bytes);

/* ------------------------------------------------------------- operations -- */

/* The quantization prologue ("prepare"): optional smooth_k key mean (fp64
 * sum), INT8 Q/K per 32-token block, e4m3 V per channel, V stored transposed.
 * Defined by "aiter-sage-attention ... #1222", section "The kernel" (the
 * per-block and per-channel quantization), and "Hand-written prologue ...
 * (v0.4.0)", section "What changed" (the fp64 key mean, 64-bit offsets).
 * q, k, v: BF16 tensors of shape (B, S, H, D), D = 128 or 64, with the given
 * strides.
 * scratch_dev: at least sage_quantize_scratch_size bytes, 256-byte aligned;
 * its contents on entry do not matter and are clobbered.
 * Enqueued: for S > 1024, a clear of the scratch header (work counter,
 * per-head flags) and one persistent kernel that computes the statistics and
 * Q codes, finishes each head (key mean, V scales), then writes the K and V
 * codes; for S <= 1024, one kernel launched in clusters of ceil(S / 128) CTAs
 * per head that exchange the head statistics through distributed shared
 * memory and does not touch the scratch (which must still be passed, with the
 * same size). Both give identical results. At D = 64 the same kernels run on
 * head pairs (heads 2j and 2j + 1 as one 128-channel head; each keeps its own
 * block scales and outputs).
 * Errors: NULLPTR, SHAPE, HEAD_DIM, ALIGN, WORKSPACE, TOO_LARGE, ARCH, CUDA. */
SAGE_API int sage_quantize(const sage_bf16_tensor* q, const sage_bf16_tensor* k, const sage_bf16_tensor* v,
                  int64_t B, int64_t S, int64_t H, int64_t D, int smooth_k,
                  const sage_quantized* out, void* scratch_dev, size_t scratch_bytes,
                  void* cuda_stream);

/* sage_quantize for callers that cannot allocate device memory. Some callers
 * cannot call cudaMalloc or any allocating routine (code running under a
 * memory budget fixed up front, plug-ins handed only the tensors they read and
 * write, hosts whose allocator must not be entered from the calling thread),
 * so they cannot provide sage_quantize's scratch buffer. This entry point
 * takes the same inputs and outputs and no scratch: the prologue's partial
 * sums go to a 32 MiB device array built into the library, which every GPU
 * that loads the library holds until the process exits. The web pages this
 * library follows have no counterpart to this entry point.
 * Limit: where the prologue uses scratch, it must need at most 32 MiB of it:
 * sage_quantize_scratch_size(B, S, H, D) <= 32 MiB. That is about
 * B * H * (S_pad * 12 + 512) bytes at D = 128 (about 21 800 (head,
 * 128-token group) pairs) and B * ceil(H / 2) * (S_pad * 12 + 1536) bytes at
 * D = 64 (about 43 600 pairs), with S_pad = ceil(S / 128) * 128; larger
 * problems are rejected with SAGE_ERR_WORKSPACE and nothing is launched.
 * With S <= 1024 the prologue runs as one cluster kernel that uses no
 * scratch, so there the limit does not apply (only the library's general
 * size limits, SAGE_ERR_TOO_LARGE, as for sage_quantize).
 * The first call on each device looks up the array's device address with
 * cudaGetSymbolAddress; make that first call before any stream capture.
 * All calls share the array and it keeps the last call's contents; each call
 * clears the part that must start at zero (a work counter and per-head flags)
 * before its kernel runs. Calls whose work overlaps on the GPU race on the
 * array, so order them on one stream. Allocates nothing; results are identical to
 * sage_quantize's.
 * Errors: NULLPTR, SHAPE, HEAD_DIM, ALIGN, WORKSPACE, TOO_LARGE, ARCH, CUDA. */
SAGE_API int sage_quantize_noalloc(const sage_bf16_tensor* q, const sage_bf16_tensor* k,
                                   const sage_bf16_tensor* v, int64_t B, int64_t S, int64_t H, int64_t D,
                                   int smooth_k, const sage_quantized* out, void* cuda_stream);

/* The attention kernel on a quantized bundle ("aiter-sage-attention ...
 * #1222", section "The kernel"): INT8 QK^T with exact integer
 * accumulation (run on the tcgen05 tensor cores as fp16 x fp16 -> fp32,
 * which is exact for |code| <= 127 and 128 channels), dequantization by
 * s_q * s_k * sm_scale, online fp32 softmax, P -> e4m3, FP8 PV on tcgen05
 * with fp32 accumulation in tensor memory, V scales in the epilogue.
 * Without the causal mask, at D = 128 and from 16 key tiles (S > 1920) the
 * kernel runs with a fourth warpgroup that rescales the output accumulator
 * (512 threads per CTA, else 384); results are the same either way.
 * out: BF16 (B, S, H, D) at out_dev with element strides (ob, os, oh),
 * channel stride 1. sm_scale must be finite and > 0.
 * The kernel is launched as a programmatic dependent of the previous kernel
 * on the stream: it may start while that kernel (normally the prologue)
 * still runs, and waits for it to complete before reading or writing
 * global memory, so stream order holds as for a plain launch.
 * Errors: NULLPTR, SHAPE, HEAD_DIM, ALIGN, ARG, TOO_LARGE, ARCH, CUDA. */
SAGE_API int sage_attention(const sage_quantized* in, int64_t B, int64_t S, int64_t H, int64_t D,
                   float sm_scale, void* out_dev, int64_t ob, int64_t os, int64_t oh,
                   void* cuda_stream);

/* sage_attention with the two flags the sageattn entry of the pages names
 * but rejects ("aiter-sage-attention ... #1222", section "What I have so
 * far": is_causal, return_lse); the page gives their names, not their
 * meaning, so this library reads them as follows.
 *  - is_causal != 0: query i attends to keys j <= i only (Q and K have the
 *    same length, so the mask is the lower triangle). Key tiles a query tile
 *    cannot see are skipped, which gives the same result as masking them.
 *  - lse_dev != NULL: fp32 [B][H][S] (contiguous, 4-byte aligned, caller
 *    owned) receives each query row's natural-log log-sum-exp of its scaled
 *    logits, ln sum_j exp(sm_scale * q_i . k_j) over the keys it sees, from
 *    the same online softmax: lse = m + ln(l). The logits are those of the
 *    bundle's K codes, i.e. of k - mean when the bundle was quantized with
 *    smooth_k; sage_lse_smooth_k_term adds the term that restores the keys'
 *    own log-sum-exp (sage_sageattn_ex does so itself).
 * Errors: as sage_attention, and ALIGN for a misaligned lse_dev. */
SAGE_API int sage_attention_ex(const sage_quantized* in, int64_t B, int64_t S, int64_t H, int64_t D,
                               float sm_scale, int is_causal, void* out_dev, int64_t ob, int64_t os, int64_t oh,
                               float* lse_dev, void* cuda_stream);

/* Adds the smooth_k term to a log-sum-exp: lse[b][h][i] += sm_scale *
 * sum_d q[b, i, h, d] * k_mean[b][h][d], with the BF16 query q (strides as
 * for sage_quantize) and the bundle's key mean k_mean_dev (fp32 [B][H][128],
 * 16-byte aligned). A per-channel key shift moves every logit of row i by the
 * same amount, so this turns the log-sum-exp of the mean-reduced keys into
 * that of the original keys. Enqueued on cuda_stream (one kernel).
 * Errors: NULLPTR, SHAPE, HEAD_DIM, ALIGN, ARG, TOO_LARGE, ARCH, CUDA. */
SAGE_API int sage_lse_smooth_k_term(const sage_bf16_tensor* q, const float* k_mean_dev, int64_t B, int64_t S,
                                    int64_t H, int64_t D, float sm_scale, float* lse_dev, void* cuda_stream);

/* Same contract and result tolerance as sage_attention_ex, computed by a
 * plain SIMT kernel (integer dot products, one thread per query row). It
 * exists to cross-check the tensor-core kernel in tests; it is never used as
 * a fallback. */
SAGE_API int sage_attention_simt(const sage_quantized* in, int64_t B, int64_t S, int64_t H, int64_t D,
                        float sm_scale, int is_causal, void* out_dev, int64_t ob, int64_t os, int64_t oh,
                        float* lse_dev, void* cuda_stream);

/* The sageattn-shaped entry ("aiter-sage-attention ... #1222", section "What
 * I have so far"): quantize q, k, v into the workspace, then run attention
 * into out. Shapes and strides are given in the order of
 * tensor_layout: "NHD" = [B, S, H, D], "HND" = [B, H, S, D]; strides are in
 * elements. out has q's shape with out_strides.
 * workspace_dev: at least sage_workspace_size bytes, 256-byte aligned. The
 * call enqueues two kernels that pass the quantized bundle through it, so
 * calls that share a workspace must not be enqueued concurrently from
 * different threads (their kernels could interleave on the stream); reusing
 * it from one thread in stream order is safe.
 * sm_scale: NaN selects 1/sqrt(D); otherwise it must be finite and > 0.
 * Rejected with an error and nothing launched: is_causal != 0 (CAUSAL),
 * return_lse != 0 (LSE), any dtype other than BF16 (DTYPE), D != 128
 * (HEAD_DIM), Q/K/V shapes not identical (SHAPE), an unknown layout
 * (LAYOUT), a channel stride != 1 (LAYOUT), a device other than
 * compute capability 10.3 (ARCH).
 * Errors also: NULLPTR, ALIGN, WORKSPACE, ARG, TOO_LARGE, CUDA. */
SAGE_API int sage_sageattn(const void* q_dev, const void* k_dev, const void* v_dev,
                  const int64_t q_shape[4], const int64_t k_shape[4], const int64_t v_shape[4],
                  const int64_t q_strides[4], const int64_t k_strides[4], const int64_t v_strides[4],
                  int q_dtype, int k_dtype, int v_dtype, const char* tensor_layout,
                  int is_causal, float sm_scale, int return_lse, int smooth_k,
                  void* out_dev, const int64_t out_strides[4], int out_dtype,
                  void* workspace_dev, size_t workspace_bytes, void* cuda_stream);

/* sage_sageattn with is_causal and return_lse honoured instead of rejected
 * (their reading: see sage_attention_ex). When lse_dev is not NULL it
 * receives the log-sum-exp of the original keys: with smooth_k on, the
 * key-mean term is added (sage_lse_smooth_k_term). All other arguments,
 * checks and errors are those of sage_sageattn (except CAUSAL and LSE), and
 * ALIGN for a misaligned lse_dev. */
SAGE_API int sage_sageattn_ex(const void* q_dev, const void* k_dev, const void* v_dev,
                              const int64_t q_shape[4], const int64_t k_shape[4], const int64_t v_shape[4],
                              const int64_t q_strides[4], const int64_t k_strides[4], const int64_t v_strides[4],
                              int q_dtype, int k_dtype, int v_dtype, const char* tensor_layout, int is_causal,
                              float sm_scale, int smooth_k, void* out_dev, const int64_t out_strides[4],
                              int out_dtype, float* lse_dev, void* workspace_dev, size_t workspace_bytes,
                              void* cuda_stream);

/* Every argument of sage_sageattn_ex in one struct, with the same meaning,
 * checks and errors (tensor_layout: "NHD" or "HND" with its terminating NUL;
 * anything else is LAYOUT). lse_dev may be NULL. For callers whose
 * per-argument marshalling costs more than the call itself (an interpreted
 * binding): they keep one filled struct per signature (shapes, strides,
 * dtypes, layout, flags) and change only the pointers, sm_scale and the
 * stream between calls. The struct is read before the call returns and not
 * kept. */
typedef struct sage_sageattn_args {
  const void* q_dev;
  const void* k_dev;
  const void* v_dev;
  int64_t q_shape[4];
  int64_t k_shape[4];
  int64_t v_shape[4];
  int64_t q_strides[4];
  int64_t k_strides[4];
  int64_t v_strides[4];
  int64_t out_strides[4];
  int32_t q_dtype;
  int32_t k_dtype;
  int32_t v_dtype;
  int32_t out_dtype;
  int32_t is_causal;
  int32_t smooth_k;
  float sm_scale;
  char tensor_layout[4];
  void* out_dev;
  float* lse_dev;
  void* workspace_dev;
  size_t workspace_bytes;
  void* cuda_stream;
} sage_sageattn_args;

/* sage_sageattn_ex on the arguments in *args. Errors: NULLPTR for a NULL
 * args, otherwise those of sage_sageattn_ex. */
SAGE_API int sage_sageattn_args_call(const sage_sageattn_args* args);

/* sageattn on HOST buffers, end to end: q, k, v and out live in host memory
 * (page-locked memory lets the copies run asynchronously; pageable memory
 * works, with staged copies), each contiguous in tensor_layout ("NHD":
 * (B, S, H, D); "HND": (B, H, S, D)) with the given shape (the four tensors
 * have one shape; dtype SAGE_DTYPE_BF16 for all four; D = 128 or 64).
 * The heads are cut into n_groups groups (0: the library's choice, at most
 * 16, at least about 32 MB of inputs per group). On internal streams, the
 * inputs of each group are copied to the device (2-D copies), the prologue
 * and the attention kernel of group g run on one of two compute streams in
 * turn, and group g's output is copied back as soon as it is done; so copies
 * overlap the kernels of the neighbouring groups. Work starts after what
 * cuda_stream already holds and cuda_stream waits for the last copy back:
 * the call is asynchronous like the device entries; synchronize cuda_stream
 * before reading out_host. Results equal sage_sageattn_ex's (no LSE) on
 * the same tensors in device memory.
 * workspace_dev: sage_host_workspace_size(B, S, H, D, n_groups) bytes of
 * device memory, 256-byte aligned, not used by another call at the same time.
 * Errors: DTYPE, NULLPTR, LAYOUT, HEAD_DIM, SHAPE, TOO_LARGE, ARG (sm_scale,
 * n_groups < 0), ALIGN, WORKSPACE, ARCH, CUDA. */
SAGE_API int sage_sageattn_host(const void* q_host, const void* k_host, const void* v_host,
                                const int64_t shape[4], int dtype, const char* tensor_layout, int is_causal,
                                float sm_scale, int smooth_k, void* out_host, int n_groups, void* workspace_dev,
                                size_t workspace_bytes, void* cuda_stream);

/* ---------------------------------------------------------- diagnostics -- */

/* Synchronizes cuda_stream, then reads and clears the current device's error
 * word. Kernels set it (and return early) when a bounded wait on an internal
 * barrier runs out, or, before any work, when their dynamic shared memory is
 * not 1024-byte aligned (the attention kernel uses all of it for aligned
 * operand tiles); they never trap. *code receives SAGE_OK,
 * SAGE_ERR_DEVICE_TIMEOUT or SAGE_ERR_DEVICE_SMEM. Returns SAGE_OK, NULLPTR
 * or CUDA. */
SAGE_API int sage_device_error(void* cuda_stream, int* code);

/* Test support for the bounded waits: enqueues on cuda_stream one kernel
 * whose only warp waits, with the bounded wait every kernel of the library
 * uses, on an internal barrier that nothing ever completes. When the wait's
 * limit (2 s) runs out the kernel sets the device error word and returns;
 * sage_device_error then reports SAGE_ERR_DEVICE_TIMEOUT, and the context
 * remains usable. Nothing else is touched. Returns SAGE_OK, ARCH or CUDA. */
SAGE_API int sage_selftest_wait_timeout(void* cuda_stream);

/* Static description of an error code; never NULL. */
SAGE_API const char* sage_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* SAGE_H */
