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
// D / 32 channels per lane (one whole row per warp instruction), 8 rows per
// warp, the row loads issued before the reductions.
#include "common.cuh"

namespace sage {
namespace {

constexpr int kRowsPerWarp = 8;
constexpr int kWarpsPerBlock = 8;

template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    lse_term_kernel(Bf16In q, const float* __restrict__ k_mean, int64_t S, int64_t H, float sm_scale,
                    float* __restrict__ lse) {
  constexpr int kW = D / 64;  // bf16x2 words per lane
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t b = blockIdx.z, h = blockIdx.y, bh = b * H + h;
  const int64_t s0 = (static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + warp) * kRowsPerWarp;
  float mu[2 * kW];
#pragma unroll
  for (int c = 0; c < 2 * kW; ++c) mu[c] = __ldg(k_mean + bh * D + 2 * kW * lane + c);
  const uint16_t* base = q.p + b * q.sb + h * q.sh + 2 * kW * lane;
  uint32_t w[kRowsPerWarp][kW];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
    for (int x = 0; x < kW; ++x)
      w[r][x] = s0 + r < S ? __ldcs(reinterpret_cast<const unsigned int*>(base + (s0 + r) * q.ss) + x) : 0u;
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    float d = 0.0f;
#pragma unroll
    for (int x = 0; x < kW; ++x) {
      d = fmaf(__uint_as_float(w[r][x] << 16), mu[2 * x], d);
      d = fmaf(__uint_as_float(w[r][x] & 0xFFFF0000u), mu[2 * x + 1], d);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (lane == 0 && s0 + r < S) lse[bh * S + s0 + r] += sm_scale * d;
  }
}

}  // namespace

cudaError_t launch_lse_smooth_k_term(const Bf16In& q, const float* k_mean, int64_t B, int64_t S, int64_t H,
                                     int64_t D, float sm_scale, float* lse, cudaStream_t stream) {
  const int64_t rows_per_block = static_cast<int64_t>(kRowsPerWarp) * kWarpsPerBlock;
  const dim3 grid(static_cast<unsigned>(div_up(S, rows_per_block)), static_cast<unsigned>(H),
                  static_cast<unsigned>(B));
  if (D == 128)
    lse_term_kernel<128><<<grid, kWarpsPerBlock * 32, 0, stream>>>(q, k_mean, S, H, sm_scale, lse);
  else if (D == 64)
    lse_term_kernel<64><<<grid, kWarpsPerBlock * 32, 0, stream>>>(q, k_mean, S, H, sm_scale, lse);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace sage
