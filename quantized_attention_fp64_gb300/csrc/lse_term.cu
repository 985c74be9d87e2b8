// The smooth_k term of the log-sum-exp: lse[b][h][i] += sm_scale * q_i . mean.
//
// With smooth_k on, the K codes are of k - mean, so the attention kernel's
// logits are those of the mean-reduced keys; a per-channel key shift changes
// every logit of row i by the same sm_scale * q_i . mean, which leaves the
// output unchanged but moves the row's log-sum-exp by exactly that much. This
// kernel adds the term back with the bf16 query values (the query codes would
// add their quantization error to it). Source of the flag: "aiter-sage-
// attention: SageAttention for AMD RDNA4 (gfx1201) #1222", section "What I
// have so far" (return_lse); "Hand-written prologue ... (v0.4.0)", section
// "What changed" (the smooth_k key mean).
//
// Bandwidth-bound: it reads Q once (2 bytes per element). One warp per row,
// 4 channels per lane (8-byte loads, one 256-byte row per warp instruction),
// 8 rows per warp, the row loads issued before the reductions.
#include "common.cuh"

namespace sage {
namespace {

constexpr int kRowsPerWarp = 8;
constexpr int kWarpsPerBlock = 8;

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    lse_term_kernel(Bf16In q, const float* __restrict__ k_mean, int64_t S, int64_t H, float sm_scale,
                    float* __restrict__ lse) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t b = blockIdx.z, h = blockIdx.y, bh = b * H + h;
  const int64_t s0 = (static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + warp) * kRowsPerWarp;
  const float4 mu = __ldg(reinterpret_cast<const float4*>(k_mean + bh * kHeadDim + 4 * lane));
  const uint16_t* base = q.p + b * q.sb + h * q.sh + 4 * lane;
  uint2 w[kRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
    w[r] = s0 + r < S ? __ldcs(reinterpret_cast<const uint2*>(base + (s0 + r) * q.ss)) : make_uint2(0u, 0u);
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    float d = __uint_as_float(w[r].x << 16) * mu.x;
    d = fmaf(__uint_as_float(w[r].x & 0xFFFF0000u), mu.y, d);
    d = fmaf(__uint_as_float(w[r].y << 16), mu.z, d);
    d = fmaf(__uint_as_float(w[r].y & 0xFFFF0000u), mu.w, d);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (lane == 0 && s0 + r < S) lse[bh * S + s0 + r] += sm_scale * d;
  }
}

}  // namespace

cudaError_t launch_lse_smooth_k_term(const Bf16In& q, const float* k_mean, int64_t B, int64_t S, int64_t H,
                                     float sm_scale, float* lse, cudaStream_t stream) {
  const int64_t rows_per_block = static_cast<int64_t>(kRowsPerWarp) * kWarpsPerBlock;
  const dim3 grid(static_cast<unsigned>(div_up(S, rows_per_block)), static_cast<unsigned>(H),
                  static_cast<unsigned>(B));
  lse_term_kernel<<<grid, kWarpsPerBlock * 32, 0, stream>>>(q, k_mean, S, H, sm_scale, lse);
  return cudaGetLastError();
}

}  // namespace sage
