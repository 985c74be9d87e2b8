// Quantization prologue: fp64 key mean (smooth_k), INT8 Q/K codes per
// 32-token block, e4m3 V codes per channel written transposed.
//
// Sources: "aiter-sage-attention: SageAttention for AMD RDNA4 (gfx1201)
// #1222", section "The kernel" (Q/K per 32-row block INT8, V per channel
// FP8); "Hand-written prologue: faster short calls, no compiler, RX 9060 XT
// opt-in (v0.4.0)", section "What changed" (64-bit offsets; key mean summed
// in fp64).
//
// Three kernels, all bandwidth-bound, every offset 64-bit:
//  1. stats: one CTA per (256-token group, head, batch); each warp owns 32
//     tokens and each lane 4 channels (one 8-byte load per token, so a warp
//     instruction reads one whole 256-byte row). It writes the Q codes and
//     scales, the fp64 key sum of its group (exact chunk sums, then a 3-level
//     pairwise tree over its 8 chunks) and the group's max |v| per channel.
//  2. finalize: one CTA per head; the pairwise tree over the group sums in
//     fp64 gives the key mean; the max over groups gives the V scales.
//  3. quant: same tiling as 1, heads visited in reverse so the K and V rows
//     stats read last are still in L2; writes K codes/scales and the V codes,
//     transposed to [channel][token] through a 4x4 byte transpose in
//     registers.
//
// Exactness of the key sum. fp64 adds run at under 2 per clock per SM on
// this GPU, far below what the HBM stream needs, so each 32-token chunk is
// summed as an unevaluated pair of floats (TwoSum: hi + lo is the exact
// running sum while lo's own additions are exact). All values are multiples
// of 2^L, the last-bit weight of the smallest nonzero input; with A the sum
// of |x|, every rounding error is below 2^(e(A)-24) and lo stays exact while
// e(A) - L <= 42. In that case every prefix sum also fits in 53 bits, so the
// left-to-right fp64 sum equals the exact sum and hi + lo (added in fp64) is
// bit-identical to it. Otherwise the chunk is re-summed left to right in fp64
// from the values still held in registers.
//
// Exactness of the codes. A code is rint(x / s) with x / s correctly
// rounded. The fast path uses q = x * fl(1/s); |q - x/s| < 2^-16 and
// |fl(x/s) - x/s| <= 2^-18 for |x/s| <= 127.5, so whenever q is farther than
// 2^-15 from a half-integer both round to the same integer; otherwise the
// exact division decides. For e4m3, rounding is monotone, so when q scaled by
// (1 - 2^-21) and by (1 + 2^-21) round to the same code, fl(v/s) (within
// 2^-22 relative of q) does too; otherwise the exact division decides.
#include <cuda_fp16.h>

#include <cfloat>

#include "common.cuh"

namespace sage {
namespace {

constexpr int kWarps = kGroup / 32;            // 8
constexpr float kMagic = 12582912.0f;          // 1.5 * 2^23: q + kMagic = rint_even(q) + kMagic for |q| < 2^22
constexpr float kHalfGuard = 0.5f - 0x1p-15f;  // fast-path guard for rint
constexpr float kDn = 1.0f - 0x1p-21f;
constexpr float kUp = 1.0f + 0x1p-21f;

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Channel c (0..3) of a lane's 4-channel group.
__device__ __forceinline__ float chan(const uint2& w, int c) {
  return c == 0 ? lo_bf16(w.x) : c == 1 ? hi_bf16(w.x) : c == 2 ? lo_bf16(w.y) : hi_bf16(w.y);
}

// Number of tokens s0 .. s0+31 that are below S.
__device__ __forceinline__ int valid_in_chunk(int64_t S, int64_t s0) {
  const int64_t d = S - s0;
  return d <= 0 ? 0 : (d >= 32 ? 32 : static_cast<int>(d));
}

// Loads channels [4*lane, 4*lane+4) of tokens s0 .. s0+31 (zeros past nvalid).
__device__ __forceinline__ void load_chunk(uint2 (&w)[32], const Bf16In& in, int64_t b, int64_t h,
                                           int64_t s0, int nvalid, int lane) {
  const uint16_t* base = in.p + b * in.sb + h * in.sh + 4 * lane;
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    w[t] = make_uint2(0u, 0u);
    if (t < nvalid) w[t] = __ldg(reinterpret_cast<const uint2*>(base + (s0 + t) * in.ss));
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Bits of fl(q + kMagic) where q = fl(x / s); the low byte is the int8 code.
__device__ __forceinline__ uint32_t int8_code_bits(float x, float s, float r, bool fast) {
  if (fast) {
    const float q = __fmul_rn(x, r);
    const float t = __fadd_rn(q, kMagic);
    const float f = __fsub_rn(q, __fsub_rn(t, kMagic));
    if (fabsf(f) < kHalfGuard) return __float_as_uint(t);
  }
  return __float_as_uint(__fadd_rn(__fdiv_rn(x, s), kMagic));
}

__device__ __forceinline__ uint32_t pack_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// Four int8 codes (one word) as four fp16 values, exactly: the fp16 bit
// pattern 0x6400 | (c ^ 0x80) is 1024 + c + 128, and subtracting 1152 leaves c.
__device__ __forceinline__ uint2 codes_to_f16x4(uint32_t w) {
  const uint32_t x = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(x, 0x64646464u, 0x5140);
  const uint32_t b = __byte_perm(x, 0x64646464u, 0x7362);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  return make_uint2(*reinterpret_cast<uint32_t*>(&ha), *reinterpret_cast<uint32_t*>(&hb));
}

// INT8 codes and scale of one 32-token block held by a warp (4 channels per
// lane). Writes rows s0..s0+31 of codes_bh ([S_pad][128]) and the same codes
// as fp16 values to f16_bh ([S_pad][128]); returns the scale.
template <bool kSub>
__device__ __forceinline__ float quantize_int8_block(const uint2 (&w)[32], const float (&mu)[4], int nvalid,
                                                     int8_t* codes_bh, uint16_t* f16_bh, int64_t s0, int lane) {
  float a = 0.0f;
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    if (t < nvalid) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float x = kSub ? __fsub_rn(chan(w[t], c), mu[c]) : chan(w[t], c);
        a = fmaxf(a, fabsf(x));
      }
    }
  }
  a = warp_max(a);
  const float s = __fdiv_rn(a, kInt8Max);
  const bool fast = s >= FLT_MIN;
  const float r = fast ? __frcp_rn(s) : 0.0f;
  uint32_t* out = reinterpret_cast<uint32_t*>(codes_bh + s0 * kHeadDim) + lane;
  uint2* out16 = reinterpret_cast<uint2*>(f16_bh + s0 * kHeadDim) + lane;
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    uint32_t word = 0u;
    if (t < nvalid && a > 0.0f) {
      uint32_t bits[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float x = kSub ? __fsub_rn(chan(w[t], c), mu[c]) : chan(w[t], c);
        bits[c] = int8_code_bits(x, s, r, fast);
      }
      word = pack_low_bytes(bits[0], bits[1], bits[2], bits[3]);
    }
    out[t * (kHeadDim / 4)] = word;
    out16[t * (kHeadDim / 4)] = codes_to_f16x4(word);
  }
  return s;
}

// Exact fp64 chunk sums of the lane's 4 channels over the warp's tokens (see
// the file comment for why the float-pair path is bit-identical).
__device__ __forceinline__ void chunk_sums(const uint2 (&w)[32], int nvalid, double (&out)[4]) {
  float hi[4] = {0.f, 0.f, 0.f, 0.f}, lo[4] = {0.f, 0.f, 0.f, 0.f}, am[4] = {0.f, 0.f, 0.f, 0.f};
  uint32_t umin = 0xFFFFFFFFu;  // (|bits| - 1) of the smallest nonzero magnitude; zeros wrap to all-ones
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    if (t < nvalid) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float x = chan(w[t], c);
        const float s = __fadd_rn(hi[c], x);
        const float bb = __fsub_rn(s, hi[c]);
        const float err = __fadd_rn(__fsub_rn(hi[c], __fsub_rn(s, bb)), __fsub_rn(x, bb));
        hi[c] = s;
        lo[c] = __fadd_rn(lo[c], err);
        am[c] = __fadd_rn(am[c], fabsf(x));
      }
      umin = min(umin, (w[t].x & 0x7FFFu) - 1u);
      umin = min(umin, ((w[t].x >> 16) & 0x7FFFu) - 1u);
      umin = min(umin, (w[t].y & 0x7FFFu) - 1u);
      umin = min(umin, ((w[t].y >> 16) & 0x7FFFu) - 1u);
    }
  }
  int ef = static_cast<int>(((umin + 1u) >> 7) & 0xFFu);
  if (ef == 0) ef = 1;                 // subnormal bf16: last-bit weight 2^-133
  const int lsb = ef - 127 - 7;         // L: exponent of the smallest last-bit weight
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int ea = static_cast<int>((__float_as_uint(am[c]) >> 23) & 0xFFu) - 127;
    if (ea - lsb <= 41) {
      out[c] = __dadd_rn(static_cast<double>(hi[c]), static_cast<double>(lo[c]));
    } else {
      double p = 0.0;
#pragma unroll
      for (int t = 0; t < 32; ++t)
        if (t < nvalid) p = __dadd_rn(p, static_cast<double>(chan(w[t], c)));
      out[c] = p;
    }
  }
}

// Two e4m3 codes: high byte = code(a), low byte = code(b).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(a), "f"(b));
  return r;
}

// Codes of channels (x0, x1) as a 16-bit pair, low byte = x0.
__device__ __forceinline__ uint32_t v_code_pair(float x0, float x1, float s0, float s1, float r0, float r1,
                                                bool fast) {
  if (fast) {
    const float q0 = __fmul_rn(x0, r0), q1 = __fmul_rn(x1, r1);
    const uint32_t dn = e4m3x2(__fmul_rn(q1, kDn), __fmul_rn(q0, kDn));
    const uint32_t up = e4m3x2(__fmul_rn(q1, kUp), __fmul_rn(q0, kUp));
    if (dn == up) return dn;
  }
  return e4m3x2(__fdiv_rn(x1, s1), __fdiv_rn(x0, s0));
}

__global__ void __launch_bounds__(kGroup) prologue_stats_kernel(Bf16In q, Bf16In k, Bf16In v, int64_t S,
                                                                int64_t S_pad, int64_t H, int64_t G,
                                                                int smooth_k, Bundle out,
                                                                double* __restrict__ ksum_part,
                                                                float* __restrict__ vmax_part) {
  __shared__ double ks[kWarps][kHeadDim];
  __shared__ uint32_t vm[kWarps][kHeadDim / 2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t bh = b * H + h;
  const int64_t s0 = g * kGroup + warp * 32;
  const int nvalid = valid_in_chunk(S, s0);

  uint2 w[32];
  // Q codes and scale of this warp's 32-token block.
  if (s0 < S_pad) {
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};
    load_chunk(w, q, b, h, s0, nvalid, lane);
    const float s = quantize_int8_block<false>(w, zero, nvalid, out.q_codes + bh * S_pad * kHeadDim,
                                               out.q16 + bh * S_pad * kHeadDim, s0, lane);
    if (lane == 0) out.q_scale[bh * (S_pad / kQKBlock) + s0 / kQKBlock] = s;
  }
  // Exact fp64 key sums of the chunk.
  if (smooth_k) {
    double sums[4];
    load_chunk(w, k, b, h, s0, nvalid, lane);
    chunk_sums(w, nvalid, sums);
#pragma unroll
    for (int c = 0; c < 4; ++c) ks[warp][4 * lane + c] = sums[c];
  }
  // Max |v| per channel over the chunk (bf16 magnitudes compare as integers).
  load_chunk(w, v, b, h, s0, nvalid, lane);
  uint32_t m01 = 0u, m23 = 0u;
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    m01 = __vmaxu2(m01, w[t].x & 0x7FFF7FFFu);
    m23 = __vmaxu2(m23, w[t].y & 0x7FFF7FFFu);
  }
  vm[warp][2 * lane] = m01;
  vm[warp][2 * lane + 1] = m23;
  __syncthreads();

  if (threadIdx.x < kHeadDim) {
    const int c = threadIdx.x;
    const int64_t slot = (bh * G + g) * kHeadDim + c;
    if (smooth_k) {
      // levels 1..3 of the pairwise tree over the group's 8 chunks
      const double l0 = __dadd_rn(ks[0][c], ks[1][c]);
      const double l1 = __dadd_rn(ks[2][c], ks[3][c]);
      const double l2 = __dadd_rn(ks[4][c], ks[5][c]);
      const double l3 = __dadd_rn(ks[6][c], ks[7][c]);
      ksum_part[slot] = __dadd_rn(__dadd_rn(l0, l1), __dadd_rn(l2, l3));
    }
    uint32_t mb = 0u;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) {
      const uint32_t pair = vm[i][c >> 1];
      mb = max(mb, (c & 1) ? (pair >> 16) : (pair & 0xFFFFu));
    }
    vmax_part[slot] = __uint_as_float(mb << 16);
  }
}

__global__ void __launch_bounds__(kHeadDim) prologue_finalize_kernel(int64_t S, int64_t G, int smooth_k,
                                                                     const double* __restrict__ ksum_part,
                                                                     const float* __restrict__ vmax_part,
                                                                     Bundle out) {
  const int c = threadIdx.x;
  const int64_t bh = blockIdx.x;
  float mu = 0.0f;
  if (smooth_k) {
    // Pairwise tree over the G group sums, padded with +0.0 to a power of
    // two, evaluated streaming: stack[l] holds a finished subtree of 2^l
    // groups. The sums are never -0.0, so adding padding changes nothing.
    double stack[64];
    for (int64_t gi = 0; gi < G; ++gi) {
      double val = ksum_part[(bh * G + gi) * kHeadDim + c];
      int lvl = 0;
      for (int64_t i = gi; i & 1; i >>= 1, ++lvl) val = __dadd_rn(stack[lvl], val);
      stack[lvl] = val;
    }
    double carry = 0.0;
    bool have = false;
    for (int lvl = 0; lvl < 63 && (G >> lvl) != 0; ++lvl) {
      if ((G >> lvl) & 1) {
        carry = have ? __dadd_rn(stack[lvl], carry) : stack[lvl];
        have = true;
      }
    }
    mu = __double2float_rn(__ddiv_rn(carry, static_cast<double>(S)));
  }
  float vmax = 0.0f;
  for (int64_t gi = 0; gi < G; ++gi) vmax = fmaxf(vmax, vmax_part[(bh * G + gi) * kHeadDim + c]);
  out.k_mean[bh * kHeadDim + c] = mu;
  out.v_scale[bh * kHeadDim + c] = __fdiv_rn(vmax, kE4M3Max);
}

__global__ void __launch_bounds__(kGroup) prologue_quant_kernel(Bf16In k, Bf16In v, int64_t S, int64_t S_pad,
                                                                int64_t B, int64_t H, int64_t G, int smooth_k,
                                                                Bundle out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // reverse order: the heads the stats kernel read last come first
  const int64_t g = G - 1 - blockIdx.x, h = H - 1 - blockIdx.y, b = B - 1 - blockIdx.z;
  const int64_t bh = b * H + h;
  const int64_t s0 = g * kGroup + warp * 32;
  if (s0 >= S_pad) return;
  const int nvalid = valid_in_chunk(S, s0);

  uint2 w[32];
  // K codes (of k - mean when smooth_k is on).
  float mu[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) mu[c] = smooth_k ? out.k_mean[bh * kHeadDim + 4 * lane + c] : 0.0f;
  load_chunk(w, k, b, h, s0, nvalid, lane);
  int8_t* kc = out.k_codes + bh * S_pad * kHeadDim;
  uint16_t* k16 = out.k16 + bh * S_pad * kHeadDim;
  const float sk = smooth_k ? quantize_int8_block<true>(w, mu, nvalid, kc, k16, s0, lane)
                            : quantize_int8_block<false>(w, mu, nvalid, kc, k16, s0, lane);
  if (lane == 0) out.k_scale[bh * (S_pad / kQKBlock) + s0 / kQKBlock] = sk;

  // V codes, transposed to [channel][token].
  float sv[4], rv[4];
  bool live[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    sv[c] = out.v_scale[bh * kHeadDim + 4 * lane + c];
    live[c] = sv[c] > 0.0f;
    rv[c] = sv[c] >= FLT_MIN ? __frcp_rn(sv[c]) : 0.0f;
  }
  const bool fast01 = sv[0] >= FLT_MIN && sv[1] >= FLT_MIN;
  const bool fast23 = sv[2] >= FLT_MIN && sv[3] >= FLT_MIN;
  const uint32_t keep = (live[0] ? 0x000000FFu : 0u) | (live[1] ? 0x0000FF00u : 0u) |
                        (live[2] ? 0x00FF0000u : 0u) | (live[3] ? 0xFF000000u : 0u);
  load_chunk(w, v, b, h, s0, nvalid, lane);
  uint32_t cw[4][8];  // cw[c][j]: tokens 4j..4j+3 of channel 4*lane+c
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 4 * j + i;
      uint32_t word = 0u;
      if (t < nvalid) {
        const uint32_t p01 = v_code_pair(lo_bf16(w[t].x), hi_bf16(w[t].x), sv[0], sv[1], rv[0], rv[1], fast01);
        const uint32_t p23 = v_code_pair(lo_bf16(w[t].y), hi_bf16(w[t].y), sv[2], sv[3], rv[2], rv[3], fast23);
        word = (p01 | (p23 << 16)) & keep;
      }
      a[i] = word;
    }
    // 4x4 byte transpose: a[i] = token i's channels -> cw[c][j] = channel c's tokens
    const uint32_t t01l = __byte_perm(a[0], a[1], 0x5140), t01h = __byte_perm(a[0], a[1], 0x7362);
    const uint32_t t23l = __byte_perm(a[2], a[3], 0x5140), t23h = __byte_perm(a[2], a[3], 0x7362);
    cw[0][j] = __byte_perm(t01l, t23l, 0x5410);
    cw[1][j] = __byte_perm(t01l, t23l, 0x7632);
    cw[2][j] = __byte_perm(t01h, t23h, 0x5410);
    cw[3][j] = __byte_perm(t01h, t23h, 0x7632);
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4* dst = reinterpret_cast<uint4*>(out.vt_codes + (bh * kHeadDim + 4 * lane + c) * S_pad + s0);
    dst[0] = make_uint4(cw[c][0], cw[c][1], cw[c][2], cw[c][3]);
    dst[1] = make_uint4(cw[c][4], cw[c][5], cw[c][6], cw[c][7]);
  }
}

struct ScratchLayout {
  size_t ksum_off, vmax_off, total;
};

ScratchLayout scratch_layout(int64_t B, int64_t S, int64_t H) {
  const int64_t G = div_up(S, kGroup);
  const size_t n = static_cast<size_t>(B * H * G * kHeadDim);
  ScratchLayout l;
  l.ksum_off = 0;
  l.vmax_off = (n * sizeof(double) + 255) / 256 * 256;
  l.total = l.vmax_off + (n * sizeof(float) + 255) / 256 * 256;
  return l;
}

}  // namespace

size_t prologue_scratch_bytes(int64_t B, int64_t S, int64_t H) { return scratch_layout(B, S, H).total; }

cudaError_t launch_prologue(const Bf16In& q, const Bf16In& k, const Bf16In& v, int64_t B, int64_t S, int64_t H,
                            bool smooth_k, const Bundle& out, void* scratch, cudaStream_t stream) {
  const int64_t S_pad = padded_len(S);
  const int64_t G = div_up(S, kGroup);
  const ScratchLayout l = scratch_layout(B, S, H);
  double* ksum = reinterpret_cast<double*>(static_cast<char*>(scratch) + l.ksum_off);
  float* vmax = reinterpret_cast<float*>(static_cast<char*>(scratch) + l.vmax_off);
  const dim3 grid(static_cast<unsigned>(G), static_cast<unsigned>(H), static_cast<unsigned>(B));
  prologue_stats_kernel<<<grid, kGroup, 0, stream>>>(q, k, v, S, S_pad, H, G, smooth_k ? 1 : 0, out, ksum, vmax);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prologue_finalize_kernel<<<static_cast<unsigned>(B * H), kHeadDim, 0, stream>>>(S, G, smooth_k ? 1 : 0, ksum,
                                                                                  vmax, out);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prologue_quant_kernel<<<grid, kGroup, 0, stream>>>(k, v, S, S_pad, B, H, G, smooth_k ? 1 : 0, out);
  return cudaGetLastError();
}

}  // namespace sage
