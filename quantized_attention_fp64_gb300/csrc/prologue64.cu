// Quantization prologue for head dimension 64: the same arithmetic as the
// head-dimension-128 prologue, in three plain kernels.
//
// Sources: "aiter-sage-attention: SageAttention for AMD RDNA4 (gfx1201)
// #1222", section "The kernel" (Q/K per 32-row block INT8, V per channel
// FP8); "Hand-written prologue: faster short calls, no compiler, RX 9060 XT
// opt-in (v0.4.0)", sections "What changed" (64-bit offsets; key mean summed
// in fp64) and "Worth knowing" (head dimension 64 is the other workload).
//
//   p64_stats:  one warp per 32-token chunk: Q codes and scale; the chunk's
//               exact key sums; the chunk's max |v| per channel.
//   p64_finish: one CTA per head, four threads per channel: the pairwise
//               fp64 tree over the chunk sums (padded with +0.0 to a power of
//               two; each thread takes a quarter of the leaves, 16 loads in
//               flight), mean = fl32(T / S); V scale = max |v| / 448.
//   p64_codes:  one warp per chunk: K codes of fl(k - mean) and V codes,
//               V written transposed ([channel][token]).
// Lane l handles channels 2l and 2l+1 (one 128-byte token row per warp
// instruction), the two channels as one packed fp32 pair.
//
// Exactness. A code is the correctly rounded quotient x / s rounded to the
// code format. INT8: t = fl(x*r + 1.5*2^23) with r = fl(1/s) holds
// rint_even(x*r) in its low byte; x*r and fl(x/s) are both within 2^-17 of
// x/s (|x/s| <= 127.5), so when |fl(c - x*r)| < 1/2 - 2^-15 the code c is
// rint_even(fl(x/s)); otherwise the division decides. e4m3: rounding is
// monotone and fl(v/s) lies within 2^-22 relative of q = fl(v*r), r within
// one ulp of 1/s, so when q*(1 - 2^-21) and q*(1 + 2^-21) round to the same
// code, that is the code of fl(v/s); otherwise q decides if q*s == v
// exactly (v/s sits on a code boundary), else the division. Key sums: a TwoSum chain
// of float pairs over the chunk's 32 tokens is exact while the largest and
// the smallest nonzero magnitude of a channel in the chunk are at most 2^36
// apart (inputs are multiples of 2^L, partial sums stay below 2^(E+6), each
// of the 31 TwoSum errors is a multiple of 2^L below 2^(E-19), so their
// fp32 sum is exact while E - 14 <= L + 24); that exact sum is also what the
// left-to-right fp64 sum gives (every prefix fits in 53 bits). Otherwise the
// channel is summed left to right in fp64.
#include <cfloat>

#include <cuda_fp16.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace sage {
namespace {

constexpr int kD = 64;
constexpr int kWarps = 8;                 // chunks per CTA
constexpr int kChunkRows = kQKBlock;      // 32 tokens per chunk
constexpr int kParts = 4;                 // threads per channel in p64_finish
constexpr uint32_t kAbs2 = 0x7FFF7FFFu;
constexpr float kMagic = 12582912.0f;     // 1.5 * 2^23
constexpr float kHalfGuard = 0.5f - 0x1p-15f;
constexpr float kDn = 1.0f - 0x1p-21f;
constexpr float kUp = 1.0f + 0x1p-21f;

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
__device__ __forceinline__ float2 bf2(uint32_t w) { return make_float2(lo_bf16(w), hi_bf16(w)); }

__device__ __forceinline__ uint32_t row_word(const Bf16In& t, int64_t b, int64_t s, int64_t h, int lane) {
  return *reinterpret_cast<const uint32_t*>(t.p + b * t.sb + s * t.ss + h * t.sh + 2 * lane);
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Two fp32 values (both exactly representable) as an fp16x2 word, lo in the low half.
__device__ __forceinline__ uint32_t f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {  // high byte = code(a), low byte = code(b)
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(a), "f"(b));
  return r;
}

// TwoSum of pairs: s = fl(a + b) and the exact error e = (a + b) - s.
__device__ __forceinline__ void two_sum2(float2 a, float2 b, float2& s, float2& e) {
  const float2 neg1 = make_float2(-1.0f, -1.0f);
  s = __fadd2_rn(a, b);
  const float2 bb = __ffma2_rn(a, neg1, s);                       // s - a
  const float2 ea = __ffma2_rn(__ffma2_rn(bb, neg1, s), neg1, a);  // a - (s - bb)
  const float2 eb = __ffma2_rn(bb, neg1, b);                       // b - bb
  e = __fadd2_rn(ea, eb);
}

// Exact path of an INT8 code: bits of fl(fl(x / s) + 1.5*2^23), whose low byte
// is rint_even(fl(x / s)) as an int8. Out of line: it is rare.
__device__ __noinline__ uint32_t exact_code_bits(float x, float s) {
  return __float_as_uint(__fadd_rn(__fdiv_rn(x, s), kMagic));
}

// 1/x to within one ulp (x normal): enough for the V codes' brackets.
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The correctly rounded quotient v / s for the exact path of a V code: q =
// fl(v*r) itself when q*s == v exactly, else the division (r = 0 marks a
// scale the fast path does not take; |v| >= 2^-90 keeps a nonzero residual
// v - q*s above the fp32 underflow threshold).
__device__ __forceinline__ float v_quotient(float v, float s, float r) {
  const float q = __fmul_rn(v, r);
  if (r != 0.0f && fabsf(v) >= 0x1p-90f && __fmaf_rn(-q, s, v) == 0.0f) return q;
  return __fdiv_rn(v, s);
}

// Exact path of a pair of e4m3 codes (low byte channel 2l): rare.
__device__ __noinline__ uint32_t exact_v_pair(uint32_t w, float2 s, float2 r) {
  return e4m3x2(v_quotient(hi_bf16(w), s.y, r.y), v_quotient(lo_bf16(w), s.x, r.x));
}

// INT8 codes of one 32-token block of this lane's two channels: x0 / x1 hold
// the block's values, 0 for rows at or past S, and reload(t) gives row t's
// pair again (the rare exact path indexes rows at run time, which register
// arrays cannot). Writes the fp16 copies of the codes (and the int8 codes
// when codes_bh is not null) of rows s0 .. s0+31 and returns the block
// scale. An all-zero block has scale 0 and codes 0.
template <typename Reload>
__device__ __forceinline__ float block_codes(const float (&x0)[kChunkRows], const float (&x1)[kChunkRows],
                                             Reload reload, int8_t* codes_bh, uint16_t* f16_bh, int64_t s0,
                                             int lane) {
  float a = 0.0f;
#pragma unroll
  for (int t = 0; t < kChunkRows; ++t) a = max3(a, fabsf(x0[t]), fabsf(x1[t]));
  a = warp_max(a);
  const float s = __fdiv_rn(a, kInt8Max);
  const bool any = a > 0.0f;
  const bool fast = s >= FLT_MIN;
  const float r = fast ? __frcp_rn(s) : 0.0f;
  const float2 r2 = make_float2(r, r), nr2 = make_float2(-r, -r);
  const float2 m2 = make_float2(kMagic, kMagic), nm2 = make_float2(-kMagic, -kMagic);
  uint16_t* c8 = codes_bh ? reinterpret_cast<uint16_t*>(codes_bh + s0 * kD) + lane : nullptr;
  uint32_t* c16 = reinterpret_cast<uint32_t*>(f16_bh + s0 * kD) + lane;
  uint32_t redo = 0u;  // bit t: row t needs the exact division
#pragma unroll
  for (int t = 0; t < kChunkRows; ++t) {
    const float2 x = make_float2(x0[t], x1[t]);
    const float2 tt = __ffma2_rn(x, r2, m2);
    const float2 cc = __fadd2_rn(tt, nm2);
    const float2 g = __ffma2_rn(x, nr2, cc);
    if (any && !(fast && fmaxf(fabsf(g.x), fabsf(g.y)) < kHalfGuard)) redo |= 1u << t;
    if (c8)
      __stcs(c8 + t * (kD / 2),
             static_cast<uint16_t>((__float_as_uint(tt.x) & 0xFFu) | ((__float_as_uint(tt.y) & 0xFFu) << 8)));
    __stcs(c16 + t * (kD / 2), any ? f16x2(cc.x, cc.y) : 0u);
  }
  if (redo != 0u) {
    // rare: rows where a fast code could be off by one are recomputed by the
    // division and stored again (same thread, same address: the later store wins)
#pragma unroll 1
    for (int t = 0; t < kChunkRows; ++t) {
      if (!((redo >> t) & 1u)) continue;
      const float2 x = reload(t);
      const uint32_t b0 = exact_code_bits(x.x, s), b1 = exact_code_bits(x.y, s);
      if (c8) __stcs(c8 + t * (kD / 2), static_cast<uint16_t>((b0 & 0xFFu) | ((b1 & 0xFFu) << 8)));
      __stcs(c16 + t * (kD / 2),
             f16x2(__fsub_rn(__uint_as_float(b0), kMagic), __fsub_rn(__uint_as_float(b1), kMagic)));
    }
  }
  return s;
}

// Whether the float-pair key sum of one channel is exact, from the largest
// magnitude bits and the smallest nonzero magnitude bits (0x10000 when the
// channel is all zero) of its bf16 values.
__device__ __forceinline__ bool pair_sum_exact(uint32_t mxb, uint32_t mnb) {
  if (mnb > 0x7FFFu) return true;
  int ef_min = static_cast<int>(mnb >> 7);
  if (ef_min == 0) ef_min = 1;  // subnormal bf16: last-bit weight 2^-133
  int ef_max = static_cast<int>(mxb >> 7);
  if (ef_max == 0) ef_max = 1;
  return ef_max - ef_min <= 36 - 7;  // E - L = (ef_max - 127) - (ef_min - 134)
}

__global__ void __launch_bounds__(kWarps * 32) p64_stats(const P64 p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t b = blockIdx.z, h = blockIdx.y, bh = b * p.H + h;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * kWarps + warp;  // chunk
  if (c >= p.NC) return;
  const int64_t s0 = c * kChunkRows;
  const int64_t d = p.S - s0;
  const int nvalid = d <= 0 ? 0 : (d >= kChunkRows ? kChunkRows : static_cast<int>(d));
  // Q codes
  {
    float x0[kChunkRows], x1[kChunkRows];
#pragma unroll
    for (int t = 0; t < kChunkRows; ++t) {
      const uint32_t w = t < nvalid ? row_word(p.q, b, s0 + t, h, lane) : 0u;
      x0[t] = lo_bf16(w);
      x1[t] = hi_bf16(w);
    }
    auto reload = [&](int t) { return bf2(row_word(p.q, b, s0 + t, h, lane)); };
    const float sq = block_codes(x0, x1, reload, p.write_int8 ? p.out.q_codes + bh * p.S_pad * kD : nullptr,
                                 p.out.q16 + bh * p.S_pad * kD, s0, lane);
    if (lane == 0) p.out.q_scale[bh * p.NC + c] = sq;
  }
  // the chunk's key sums: float pairs, or left to right in fp64 for a
  // channel whose pair sum may be inexact
  if (p.smooth_k) {
    float2 hi = make_float2(0.f, 0.f), lo = make_float2(0.f, 0.f);
    uint32_t mx = 0u, mn = 0xFFFFFFFFu;  // zeros wrap to 0xFFFF and never win the minimum
#pragma unroll
    for (int t = 0; t < kChunkRows; ++t) {
      const uint32_t w = t < nvalid ? row_word(p.k, b, s0 + t, h, lane) : 0u;
      const uint32_t a = w & kAbs2;
      mx = __vmaxu2(mx, a);
      mn = __vminu2(mn, __vsub2(a, 0x00010001u));
      float2 s, e;
      two_sum2(hi, bf2(w), s, e);
      hi = s;
      lo = __fadd2_rn(lo, e);
    }
    double k0 = __dadd_rn(static_cast<double>(hi.x), static_cast<double>(lo.x));
    double k1 = __dadd_rn(static_cast<double>(hi.y), static_cast<double>(lo.y));
    const bool ok0 = pair_sum_exact(mx & 0xFFFFu, (mn & 0xFFFFu) + 1u);
    const bool ok1 = pair_sum_exact(mx >> 16, (mn >> 16) + 1u);
    if (!(ok0 && ok1)) {
      double f0 = 0.0, f1 = 0.0;
      for (int t = 0; t < nvalid; ++t) {
        const uint32_t w = row_word(p.k, b, s0 + t, h, lane);
        f0 = __dadd_rn(f0, static_cast<double>(lo_bf16(w)));
        f1 = __dadd_rn(f1, static_cast<double>(hi_bf16(w)));
      }
      if (!ok0) k0 = f0;
      if (!ok1) k1 = f1;
    }
    *reinterpret_cast<double2*>(p.ksum + (bh * p.NC + c) * kD + 2 * lane) = make_double2(k0, k1);
  }
  // max |v| of the chunk (bf16 magnitudes order as integers)
  uint32_t m = 0u;
#pragma unroll
  for (int t = 0; t < kChunkRows; ++t)
    if (t < nvalid) m = __vmaxu2(m, row_word(p.v, b, s0 + t, h, lane) & kAbs2);
  *reinterpret_cast<float2*>(p.vmax + (bh * p.NC + c) * kD + 2 * lane) =
      make_float2(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}

// Pairwise tree over `n` leaves starting at p (stride kD doubles), padded
// with +0.0 to a power of two, evaluated streaming: stack[l] holds a finished
// subtree of 2^l leaves; aligned blocks of 16 leaves are loaded together and
// reduced as one 16-leaf subtree (what pushing them one by one would build).
// The sums are never -0.0, so padding with +0.0 changes nothing.
__device__ __forceinline__ double tree_sum64(const double* p, int64_t n) {
  double stack[40];
  int64_t gi = 0;
  for (; gi + 16 <= n; gi += 16) {
    double v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = __ldcg(p + (gi + k) * kD);
#pragma unroll
    for (int w = 1; w < 16; w *= 2)
#pragma unroll
      for (int k = 0; k < 16; k += 2 * w) v[k] = __dadd_rn(v[k], v[k + w]);
    double val = v[0];
    int lvl = 4;
    for (int64_t k = gi >> 4; k & 1; k >>= 1, ++lvl) val = __dadd_rn(stack[lvl], val);
    stack[lvl] = val;
  }
  for (; gi < n; ++gi) {
    double val = __ldcg(p + gi * kD);
    int lvl = 0;
    for (int64_t k = gi; k & 1; k >>= 1, ++lvl) val = __dadd_rn(stack[lvl], val);
    stack[lvl] = val;
  }
  double carry = 0.0;
  bool have = false;
  for (int lvl = 0; lvl < 40 && (n >> lvl) != 0; ++lvl) {
    if ((n >> lvl) & 1) {
      carry = have ? __dadd_rn(stack[lvl], carry) : stack[lvl];
      have = true;
    }
  }
  return carry;
}

// Max of `n` chunk maxima starting at p (stride kD floats), 16 loads in flight.
__device__ __forceinline__ float chunk_max64(const float* p, int64_t n) {
  float m = 0.0f;
  int64_t gi = 0;
  for (; gi + 16 <= n; gi += 16) {
    float v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = __ldcg(p + (gi + k) * kD);
#pragma unroll
    for (int k = 0; k < 16; ++k) m = fmaxf(m, v[k]);
  }
  for (; gi < n; ++gi) m = fmaxf(m, __ldcg(p + gi * kD));
  return m;
}

// Thread (part, channel) takes the leaves [part * Q, (part + 1) * Q) of the
// padded tree over P = 2^ceil(log2 n) leaves, Q = P / 4 (when P < 4 part 0
// takes every leaf); the tree's top two levels join the four subtree roots.
__global__ void __launch_bounds__(kParts * kD) p64_finish(const P64 p, int64_t n_chunks) {
  __shared__ double roots[kParts][kD];
  __shared__ float maxima[kParts][kD];
  const int ch = threadIdx.x % kD, part = threadIdx.x / kD;
  const int64_t bh = blockIdx.x;
  int64_t P = 1;
  while (P < n_chunks) P *= 2;
  const int64_t Q = P >= kParts ? P / kParts : P;
  const int64_t first = part * Q;
  const int64_t cnt = first >= n_chunks ? 0 : (n_chunks - first < Q ? n_chunks - first : Q);
  const int64_t base = (bh * p.NC + first) * kD + ch;
  roots[part][ch] = (p.smooth_k && cnt > 0) ? tree_sum64(p.ksum + base, cnt) : 0.0;
  maxima[part][ch] = cnt > 0 ? chunk_max64(p.vmax + base, cnt) : 0.0f;
  __syncthreads();
  if (part == 0) {
    float mu = 0.0f;
    if (p.smooth_k) {
      const double total = P >= kParts ? __dadd_rn(__dadd_rn(roots[0][ch], roots[1][ch]),
                                                   __dadd_rn(roots[2][ch], roots[3][ch]))
                                       : roots[0][ch];
      mu = __double2float_rn(__ddiv_rn(total, static_cast<double>(p.S)));
    }
    const float vm = fmaxf(fmaxf(maxima[0][ch], maxima[1][ch]), fmaxf(maxima[2][ch], maxima[3][ch]));
    p.out.k_mean[bh * kD + ch] = mu;
    p.out.v_scale[bh * kD + ch] = __fdiv_rn(vm, kE4M3Max);
  }
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
  // K codes of fl(k - mean); rows at or past S are 0
  {
    const float2 mu = *reinterpret_cast<const float2*>(p.out.k_mean + bh * kD + 2 * lane);
    const float2 nmu = make_float2(-mu.x, -mu.y);
    float x0[kChunkRows], x1[kChunkRows];
#pragma unroll
    for (int t = 0; t < kChunkRows; ++t) {
      float2 x = make_float2(0.f, 0.f);
      if (t < nvalid) x = __fadd2_rn(bf2(row_word(p.k, b, s0 + t, h, lane)), nmu);
      x0[t] = x.x;
      x1[t] = x.y;
    }
    auto reload = [&](int t) { return __fadd2_rn(bf2(row_word(p.k, b, s0 + t, h, lane)), nmu); };
    const float sk = block_codes(x0, x1, reload, p.write_int8 ? p.out.k_codes + bh * p.S_pad * kD : nullptr,
                                 p.out.k16 + bh * p.S_pad * kD, s0, lane);
    if (lane == 0) p.out.k_scale[bh * p.NC + c] = sk;
  }
  // V codes e4m3(fl(v / s_v)), transposed: 32 tokens of each of the lane's channels
  const float2 sv = *reinterpret_cast<const float2*>(p.out.v_scale + bh * kD + 2 * lane);
  const bool fast = (sv.x >= FLT_MIN || sv.x == 0.0f) && (sv.y >= FLT_MIN || sv.y == 0.0f);
  const float2 rv = make_float2(sv.x >= FLT_MIN ? rcp_approx(sv.x) : 0.0f, sv.y >= FLT_MIN ? rcp_approx(sv.y) : 0.0f);
  const uint32_t keep = (sv.x > 0.0f ? 0x00FFu : 0u) | (sv.y > 0.0f ? 0xFF00u : 0u);  // a zero channel has code 0
  const float2 dn = make_float2(kDn, kDn), up = make_float2(kUp, kUp);
  uint32_t pr[kChunkRows];  // low byte channel 2l, high byte channel 2l+1
  uint32_t wv[kChunkRows];
  uint32_t redo = 0u;
#pragma unroll
  for (int t = 0; t < kChunkRows; ++t) {
    wv[t] = t < nvalid ? row_word(p.v, b, s0 + t, h, lane) : 0u;
    const float2 q = __fmul2_rn(bf2(wv[t]), rv);
    const float2 qd = __fmul2_rn(q, dn), qu = __fmul2_rn(q, up);
    const uint32_t cd = e4m3x2(qd.y, qd.x), cu = e4m3x2(qu.y, qu.x);
    if (!(fast && cd == cu)) redo |= 1u << t;
    pr[t] = cd & keep;
  }
  if (redo != 0u) {
    // rare: tokens whose fast codes are not certain
#pragma unroll
    for (int t = 0; t < kChunkRows; ++t)
      if ((redo >> t) & 1u) pr[t] = exact_v_pair(wv[t], sv, rv) & keep;
  }
  uint32_t w0[8], w1[8];  // channel 2l / 2l+1: tokens 4j .. 4j+3
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    w0[j] = __byte_perm(__byte_perm(pr[4 * j], pr[4 * j + 1], 0x0040),
                        __byte_perm(pr[4 * j + 2], pr[4 * j + 3], 0x0040), 0x5410);
    w1[j] = __byte_perm(__byte_perm(pr[4 * j], pr[4 * j + 1], 0x0051),
                        __byte_perm(pr[4 * j + 2], pr[4 * j + 3], 0x0051), 0x5410);
  }
  uint4* d0 = reinterpret_cast<uint4*>(p.out.vt_codes + (bh * kD + 2 * lane) * p.S_pad + s0);
  uint4* d1 = reinterpret_cast<uint4*>(p.out.vt_codes + (bh * kD + 2 * lane + 1) * p.S_pad + s0);
  __stcs(d0, make_uint4(w0[0], w0[1], w0[2], w0[3]));
  __stcs(d0 + 1, make_uint4(w0[4], w0[5], w0[6], w0[7]));
  __stcs(d1, make_uint4(w1[0], w1[1], w1[2], w1[3]));
  __stcs(d1 + 1, make_uint4(w1[4], w1[5], w1[6], w1[7]));
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
  p64_finish<<<static_cast<unsigned>(B * H), kParts * kD, 0, stream>>>(p, div_up(S, kQKBlock));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  p64_codes<<<grid, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace sage
