// Quantization prologue for head dimension 64: the same arithmetic as the
// head-dimension-128 prologue, written plainly (three kernels, no ring).
//
// Sources: "aiter-sage-attention: SageAttention for AMD RDNA4 (gfx1201)
// #1222", section "The kernel" (Q/K per 32-row block INT8, V per channel
// FP8); "Hand-written prologue: faster short calls, no compiler, RX 9060 XT
// opt-in (v0.4.0)", sections "What changed" (64-bit offsets; key mean summed
// in fp64) and "Worth knowing" (head dimension 64 is the other workload).
//
//   p64_stats:    one warp per 32-token chunk: Q codes and scale; the
//                 chunk's key sums, left to right in fp64 (the reference order
//                 itself); the chunk's max |v| per channel.
//   p64_finalize: one thread per (head, channel): the pairwise fp64 tree over
//                 the chunk sums (padded with +0.0 to a power of two),
//                 mean = fl32(T / S); V scale = max |v| / 448.
//   p64_codes:    one warp per chunk: K codes of fl(k - mean) and V codes,
//                 V written transposed ([channel][token]).
// Lane l handles channels 2l and 2l+1 (one 128-byte token row per warp
// instruction). Every code is the correctly rounded quotient rounded to the
// code format (rint_even for INT8, e4m3 round-to-nearest-even with
// saturation), so no fast path needs a proof here.
#include <cfloat>

#include <cuda_fp16.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace sage {
namespace {

constexpr int kD = 64;
constexpr int kWarps = 8;                 // chunks per CTA
constexpr int kChunkRows = kQKBlock;      // 32 tokens per chunk
constexpr uint32_t kAbs2 = 0x7FFF7FFFu;

struct P64 {
  Bf16In q, k, v;
  int64_t S, S_pad, H, NC;  // NC: chunks per head (S_pad / 32)
  int smooth_k, write_int8;
  Bundle out;
  double* ksum;  // [B*H][NC][64]
  float* vmax;   // [B*H][NC][64]
};

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t row_word(const Bf16In& t, int64_t b, int64_t s, int64_t h, int lane) {
  return *reinterpret_cast<const uint32_t*>(t.p + b * t.sb + s * t.ss + h * t.sh + 2 * lane);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// INT8 code of x at scale s (s > 0): rint_even of the correctly rounded x / s.
__device__ __forceinline__ int int8_code(float x, float s) { return __float2int_rn(__fdiv_rn(x, s)); }

// Codes of one 32-token block (rows s0 .. s0+31, nvalid of them below S) of
// x - mu for this lane's two channels: writes the fp16 copies (and the int8
// codes when codes_bh is not null) and returns the block scale.
__device__ __forceinline__ float block_codes(const float (&x0)[kChunkRows], const float (&x1)[kChunkRows],
                                             int nvalid, int8_t* codes_bh, uint16_t* f16_bh, int64_t s0, int lane) {
  float a = 0.0f;
  for (int t = 0; t < nvalid; ++t) a = fmaxf(a, fmaxf(fabsf(x0[t]), fabsf(x1[t])));
  a = warp_max(a);
  const float s = __fdiv_rn(a, kInt8Max);
#pragma unroll 4
  for (int t = 0; t < kChunkRows; ++t) {
    int c0 = 0, c1 = 0;
    if (t < nvalid && a > 0.0f) {
      c0 = int8_code(x0[t], s);
      c1 = int8_code(x1[t], s);
    }
    const int64_t off = (s0 + t) * kD + 2 * lane;
    if (codes_bh) *reinterpret_cast<uint16_t*>(codes_bh + off) = static_cast<uint16_t>((c0 & 0xFF) | ((c1 & 0xFF) << 8));
    const __half2 h = __floats2half2_rn(static_cast<float>(c0), static_cast<float>(c1));
    *reinterpret_cast<__half2*>(f16_bh + off) = h;
  }
  return s;
}

__global__ void __launch_bounds__(kWarps * 32) p64_stats(const P64 p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t b = blockIdx.z, h = blockIdx.y, bh = b * p.H + h;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * kWarps + warp;  // chunk
  if (c >= p.NC) return;
  const int64_t s0 = c * kChunkRows;
  const int64_t d = p.S - s0;
  const int nvalid = d <= 0 ? 0 : (d >= kChunkRows ? kChunkRows : static_cast<int>(d));
  float x0[kChunkRows], x1[kChunkRows];
  // Q codes
  for (int t = 0; t < kChunkRows; ++t) {
    const uint32_t w = t < nvalid ? row_word(p.q, b, s0 + t, h, lane) : 0u;
    x0[t] = lo_bf16(w);
    x1[t] = hi_bf16(w);
  }
  const float sq = block_codes(x0, x1, nvalid, p.write_int8 ? p.out.q_codes + bh * p.S_pad * kD : nullptr,
                               p.out.q16 + bh * p.S_pad * kD, s0, lane);
  if (lane == 0) p.out.q_scale[bh * p.NC + c] = sq;
  // key sums of the chunk, left to right in fp64 from +0.0
  if (p.smooth_k) {
    double k0 = 0.0, k1 = 0.0;
    for (int t = 0; t < nvalid; ++t) {
      const uint32_t w = row_word(p.k, b, s0 + t, h, lane);
      k0 = __dadd_rn(k0, static_cast<double>(lo_bf16(w)));
      k1 = __dadd_rn(k1, static_cast<double>(hi_bf16(w)));
    }
    p.ksum[(bh * p.NC + c) * kD + 2 * lane] = k0;
    p.ksum[(bh * p.NC + c) * kD + 2 * lane + 1] = k1;
  }
  // max |v| of the chunk (bf16 magnitudes order as integers)
  uint32_t m = 0u;
  for (int t = 0; t < nvalid; ++t) m = __vmaxu2(m, row_word(p.v, b, s0 + t, h, lane) & kAbs2);
  p.vmax[(bh * p.NC + c) * kD + 2 * lane] = __uint_as_float(m << 16);
  p.vmax[(bh * p.NC + c) * kD + 2 * lane + 1] = __uint_as_float(m & 0xFFFF0000u);
}

__global__ void __launch_bounds__(kD) p64_finalize(const P64 p, int64_t n_chunks) {
  const int ch = threadIdx.x;
  const int64_t bh = blockIdx.x;
  const double* ks = p.ksum + bh * p.NC * kD + ch;
  float vm = 0.0f;
  for (int64_t c = 0; c < n_chunks; ++c) vm = fmaxf(vm, p.vmax[(bh * p.NC + c) * kD + ch]);
  float mu = 0.0f;
  if (p.smooth_k) {
    // pairwise tree over the chunk sums, streaming: stack[l] holds a finished
    // subtree of 2^l leaves; the trailing combination is the padded tree
    double stack[40];
    for (int64_t c = 0; c < n_chunks; ++c) {
      double val = ks[c * kD];
      int lvl = 0;
      for (int64_t k = c; k & 1; k >>= 1, ++lvl) val = __dadd_rn(stack[lvl], val);
      stack[lvl] = val;
    }
    double total = 0.0;
    bool have = false;
    for (int lvl = 0; lvl < 40 && (n_chunks >> lvl) != 0; ++lvl) {
      if ((n_chunks >> lvl) & 1) {
        total = have ? __dadd_rn(stack[lvl], total) : stack[lvl];
        have = true;
      }
    }
    mu = __double2float_rn(__ddiv_rn(total, static_cast<double>(p.S)));
  }
  p.out.k_mean[bh * kD + ch] = mu;
  p.out.v_scale[bh * kD + ch] = __fdiv_rn(vm, kE4M3Max);
}

__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {  // high byte = code(a), low byte = code(b)
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(a), "f"(b));
  return r;
}

__global__ void __launch_bounds__(kWarps * 32) p64_codes(const P64 p) {
  // the attention kernel after it is a programmatic dependent: it may be
  // scheduled now and waits for this grid to end before it reads anything
  tc::griddep_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t b = blockIdx.z, h = blockIdx.y, bh = b * p.H + h;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  if (c >= p.NC) return;
  const int64_t s0 = c * kChunkRows;
  const int64_t d = p.S - s0;
  const int nvalid = d <= 0 ? 0 : (d >= kChunkRows ? kChunkRows : static_cast<int>(d));
  // K codes of fl(k - mean)
  const float mu0 = p.out.k_mean[bh * kD + 2 * lane], mu1 = p.out.k_mean[bh * kD + 2 * lane + 1];
  float x0[kChunkRows], x1[kChunkRows];
  for (int t = 0; t < kChunkRows; ++t) {
    const uint32_t w = t < nvalid ? row_word(p.k, b, s0 + t, h, lane) : 0u;
    x0[t] = __fsub_rn(lo_bf16(w), mu0);
    x1[t] = __fsub_rn(hi_bf16(w), mu1);
  }
  const float sk = block_codes(x0, x1, nvalid, p.write_int8 ? p.out.k_codes + bh * p.S_pad * kD : nullptr,
                               p.out.k16 + bh * p.S_pad * kD, s0, lane);
  if (lane == 0) p.out.k_scale[bh * p.NC + c] = sk;
  // V codes e4m3(fl(v / s_v)), transposed: 32 tokens of each of the lane's channels
  const float sv0 = p.out.v_scale[bh * kD + 2 * lane], sv1 = p.out.v_scale[bh * kD + 2 * lane + 1];
  uint32_t w0[8], w1[8];  // channel 2l / 2l+1: tokens 4j .. 4j+3
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t a0 = 0u, a1 = 0u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int t = 4 * j + q;
      uint32_t pair = 0u;  // low byte channel 2l, high byte channel 2l+1
      if (t < nvalid) {
        const uint32_t w = row_word(p.v, b, s0 + t, h, lane);
        const float y0 = sv0 > 0.0f ? __fdiv_rn(lo_bf16(w), sv0) : 0.0f;
        const float y1 = sv1 > 0.0f ? __fdiv_rn(hi_bf16(w), sv1) : 0.0f;
        pair = e4m3x2(y1, y0);
        if (!(sv0 > 0.0f)) pair &= 0xFF00u;  // a zero channel has code 0
        if (!(sv1 > 0.0f)) pair &= 0x00FFu;
      }
      a0 |= (pair & 0xFFu) << (8 * q);
      a1 |= ((pair >> 8) & 0xFFu) << (8 * q);
    }
    w0[j] = a0;
    w1[j] = a1;
  }
  uint4* d0 = reinterpret_cast<uint4*>(p.out.vt_codes + (bh * kD + 2 * lane) * p.S_pad + s0);
  uint4* d1 = reinterpret_cast<uint4*>(p.out.vt_codes + (bh * kD + 2 * lane + 1) * p.S_pad + s0);
  d0[0] = make_uint4(w0[0], w0[1], w0[2], w0[3]);
  d0[1] = make_uint4(w0[4], w0[5], w0[6], w0[7]);
  d1[0] = make_uint4(w1[0], w1[1], w1[2], w1[3]);
  d1[1] = make_uint4(w1[4], w1[5], w1[6], w1[7]);
}

struct Layout64 {
  size_t ksum_off, vmax_off, total;
};

Layout64 layout64(int64_t B, int64_t S, int64_t H) {
  const size_t n = static_cast<size_t>(B * H) * static_cast<size_t>(padded_len(S) / kQKBlock) * kD;
  Layout64 l;
  l.ksum_off = 0;
  l.vmax_off = (n * sizeof(double) + 255) / 256 * 256;
  l.total = l.vmax_off + (n * sizeof(float) + 255) / 256 * 256;
  return l;
}

}  // namespace

size_t prologue64_scratch_bytes(int64_t B, int64_t S, int64_t H) { return layout64(B, S, H).total; }

cudaError_t launch_prologue64(const Bf16In& q, const Bf16In& k, const Bf16In& v, int64_t B, int64_t S, int64_t H,
                              bool smooth_k, const Bundle& out, void* scratch, bool write_int8, cudaStream_t stream) {
  const Layout64 l = layout64(B, S, H);
  P64 p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.S = S;
  p.S_pad = padded_len(S);
  p.H = H;
  p.NC = p.S_pad / kQKBlock;
  p.smooth_k = smooth_k ? 1 : 0;
  p.write_int8 = write_int8 ? 1 : 0;
  p.out = out;
  p.ksum = reinterpret_cast<double*>(static_cast<char*>(scratch) + l.ksum_off);
  p.vmax = reinterpret_cast<float*>(static_cast<char*>(scratch) + l.vmax_off);
  const dim3 grid(static_cast<unsigned>(div_up(p.NC, kWarps)), static_cast<unsigned>(H), static_cast<unsigned>(B));
  p64_stats<<<grid, kWarps * 32, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  p64_finalize<<<static_cast<unsigned>(B * H), kD, 0, stream>>>(p, div_up(S, kQKBlock));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  p64_codes<<<grid, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace sage
