// Quantization prologue: fp64 key mean (smooth_k), INT8 Q/K codes per
// 32-token block (plus their exact fp16 copies for the tensor cores), e4m3 V
// codes per channel written transposed.
//
// Sources: "aiter-sage-attention: SageAttention for AMD RDNA4 (gfx1201)
// #1222", section "The kernel" (Q/K per 32-row block INT8, V per channel
// FP8); "Hand-written prologue: faster short calls, no compiler, RX 9060 XT
// opt-in (v0.4.0)", section "What changed" (64-bit offsets; key mean summed
// in fp64).
//
// One persistent kernel, one CTA per SM: two teams of 8 compute warps and 1
// TMA producer warp. The work is a list of items claimed in order from a
// global counter:
//   stats item (head, 256-token group): Q codes and scales; exact fp64 key
//     sums of the group (8 chunks of 32 tokens, then a 3-level pairwise tree);
//     the group's max |v| per channel. The last stats item of a head (counted
//     with an atomic) finishes that head: the pairwise tree over its group sums
//     gives the key mean, the max over groups the V scales; then it publishes
//     the head as ready.
//   codes item (head, 256-token group): K codes of k - mean, V codes
//     (transposed); the producer loads its tiles once the head is ready.
// The codes items of head h come after the stats items of head h + L, so K
// and V are read the second time while still in L2 (L is sized from the L2
// capacity). The producer loads each tensor's 256-token x 128-channel bf16
// tile with one 4-D TMA copy into a 3-stage ring (64 KB per stage), so the
// compute warps always have the next tiles in flight. Items are claimed in a
// global order and every CTA processes its items in claim order, so the
// stats items a codes item waits for were all claimed earlier and always
// progress: the waits end. They are bounded anyway.
//
// Exactness of the key sum. fp64 adds run at under 2 per clock per SM on
// this GPU, far below what the HBM stream needs, so each 32-token chunk is
// summed as unevaluated pairs of floats (TwoSum chains, two-element packed
// arithmetic), which give the exact chunk sum whenever the spread of
// exponents in the chunk is bounded (see chunk_sums); that exact sum is what
// the left-to-right fp64 sum produces too, so the result is bit-identical.
// Otherwise the chunk is summed left to right in fp64.
//
// Exactness of the codes. A code is rint(x / s) with x / s correctly
// rounded in fp32. The fast path multiplies by fl(1/s) and falls back to the
// exact division whenever the product is within 2^-15 of a half-integer
// (quantize_block). For e4m3, rounding is monotone, so when q = fl(v*fl(1/s))
// scaled by (1 - 2^-21) and by (1 + 2^-21) round to the same code, fl(v/s)
// (within 2^-22 relative of q) does too; otherwise the exact division
// decides (v_code_quad). Q and V maxima are taken on the bf16 bit patterns,
// whose magnitudes order as integers.
#include <cuda_fp16.h>

#include <cfloat>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace sage {
namespace {

constexpr int kWarps = kGroup / 32;            // 8 compute warps
constexpr int kTeams = 2;                      // compute teams of kWarps warps
constexpr int kThreads = kTeams * kGroup + 32; // + the producer warp
constexpr int kStages = 3;
constexpr uint32_t kTileBytes = kGroup * kHeadDim * 2;  // one bf16 tile: 256 tokens x 128 channels
constexpr float kMagic = 12582912.0f;          // 1.5 * 2^23: q + kMagic = rint_even(q) + kMagic for |q| < 2^22
constexpr float kHalfGuard = 0.5f - 0x1p-15f;  // fast-path guard for rint
constexpr float kDn = 1.0f - 0x1p-21f;
constexpr float kUp = 1.0f + 0x1p-21f;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait

enum : int { kTensorQ = 0, kTensorK = 1, kTensorV = 2, kEnd = 3 };

// shared memory: kStages tiles, then the barriers and per-stage item tags
constexpr uint32_t kOffBar = kStages * kTileBytes;
constexpr uint32_t kOffMeta = kOffBar + 2 * kStages * 8;
constexpr uint32_t kOffFlags = kOffMeta + kStages * 16;
constexpr uint32_t kSmemBytes = kOffFlags + 16 + 1024;  // + alignment slack

struct Params {
  int64_t S, S_pad, H, NH, G, lag, total;
  int smooth_k, write_int8;
  Bundle out;
  unsigned* next_item;
  unsigned* done;   // [NH]: stats items finished per head
  unsigned* ready;  // [NH]: 1 once the head's key mean and V scales are written
  double* ksum;     // [NH][G][128]
  float* vmax;      // [NH][G][128]
  int* dev_err;
};

struct Item {
  int phase;  // 0 stats, 1 codes
  int64_t bh, g;
};

// Item order: stats(h) for h < lag; then per h: stats(h), codes(h - lag);
// then the codes items of the last lag heads.
__device__ __forceinline__ Item decode_item(int64_t i, int64_t NH, int64_t G, int64_t L) {
  Item it;
  if (i < L * G) {
    it.phase = 0;
    it.bh = i / G;
    it.g = i % G;
    return it;
  }
  i -= L * G;
  if (i < (NH - L) * 2 * G) {
    const int64_t t = L + i / (2 * G), r = i % (2 * G);
    it.phase = r < G ? 0 : 1;
    it.bh = r < G ? t : t - L;
    it.g = r < G ? r : r - G;
    return it;
  }
  i -= (NH - L) * 2 * G;
  it.phase = 1;
  it.bh = NH - L + i / G;
  it.g = i % G;
  return it;
}

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// Both channels of a bf16x2 word as fp32 (exact): .x the low half, .y the high half.
__device__ __forceinline__ float2 bf2(uint32_t w) { return make_float2(lo_bf16(w), hi_bf16(w)); }

constexpr uint32_t kAbs2 = 0x7FFF7FFFu;  // clears the sign bits of a bf16x2 word

// Number of tokens s0 .. s0+31 that are below S.
__device__ __forceinline__ int valid_in_chunk(int64_t S, int64_t s0) {
  const int64_t d = S - s0;
  return d <= 0 ? 0 : (d >= 32 ? 32 : static_cast<int>(d));
}

// Shared-memory tiles hold 256-byte token rows (128 bf16 channels). Two lane
// mappings read them without bank conflicts:
//  - 8-channel lanes: lane l reads channels 8*(l & 15) .. +8 of token
//    2*i + (l >> 4), so one warp instruction covers two whole rows;
//  - 4-channel lanes: lane l reads channels 4*l .. +4 of one token, one row
//    per warp instruction (used where each lane needs all 32 tokens).
__device__ __forceinline__ uint4 tok8(const uint8_t* rows, int t, int lane) {
  return *reinterpret_cast<const uint4*>(rows + t * 256 + (lane & 15) * 16);
}
__device__ __forceinline__ uint2 tok4(const uint8_t* rows, int t, int lane) {
  return *reinterpret_cast<const uint2*>(rows + t * 256 + lane * 8);
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

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ uint32_t pack_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// Two fp32 values (both exactly representable) as an fp16x2 word, lo in the low half.
__device__ __forceinline__ uint32_t f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Exact path of a code: bits of fl(fl(x / s) + kMagic), whose low byte is
// rint_even(fl(x / s)) as an int8. Out of line: the fast path below decides
// all but a few codes in 10^4.
__device__ __noinline__ uint32_t exact_code_bits(float x, float s) {
  return __float_as_uint(__fadd_rn(__fdiv_rn(x, s), kMagic));
}

// INT8 codes and scale of one 32-token block: x (kMu false) or fl(x - mu)
// (kMu true; nmu holds -mu for the lane's 8 channels as pairs). Reads the
// warp's 32 rows of a shared tile with 8-channel lanes; writes rows
// s0..s0+31 of f16_bh ([S_pad][128], the codes as fp16 values) and, when
// codes_bh is not null, of codes_bh ([S_pad][128] int8), with streaming
// stores; rows at or past nvalid are written as zero codes. kFull: nvalid is
// 32. Returns the scale.
//
// Fast path for the codes (two-element packed arithmetic): t = fl(x*r + M)
// with r = fl(1/s) and M = 1.5*2^23 is M + rint_even(x*r) (the spacing of
// floats near M is 1); c = t - M exactly; g = fl(c - x*r). x*r is within
// 2^-17 of x/s, and so is fl(x/s) (|x/s| <= 127.5), so when |g| < 1/2 - 2^-15
// the code c is rint_even(fl(x/s)); otherwise the exact division decides.
template <bool kMu, bool kFull>
__device__ __forceinline__ float quantize_block(const uint8_t* rows, const float2 (&nmu)[4], int nvalid,
                                                int8_t* codes_bh, uint16_t* f16_bh, int64_t s0, int lane) {
  const int half = lane >> 4;
  float a;
  if (!kMu) {
    // block amax on the bf16 bit patterns (magnitudes order as integers)
    uint32_t m0 = 0u, m1 = 0u;
#pragma unroll 8
    for (int i = 0; i < 16; ++i) {
      const int t = 2 * i + half;
      if (kFull || t < nvalid) {
        const uint4 w = tok8(rows, t, lane);
        m0 = __vimax3_u16x2(m0, w.x & kAbs2, w.y & kAbs2);
        m1 = __vimax3_u16x2(m1, w.z & kAbs2, w.w & kAbs2);
      }
    }
    const uint32_t m = __vmaxu2(m0, m1);
    a = __uint_as_float(warp_max_u32(max(m & 0xFFFFu, m >> 16)) << 16);
  } else {
    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll 8
    for (int i = 0; i < 16; ++i) {
      const int t = 2 * i + half;
      if (kFull || t < nvalid) {
        const uint4 w = tok8(rows, t, lane);
        const float2 k0 = __fadd2_rn(bf2(w.x), nmu[0]), k1 = __fadd2_rn(bf2(w.y), nmu[1]);
        const float2 k2 = __fadd2_rn(bf2(w.z), nmu[2]), k3 = __fadd2_rn(bf2(w.w), nmu[3]);
        a0 = max3(a0, fabsf(k0.x), fabsf(k0.y));
        a1 = max3(a1, fabsf(k1.x), fabsf(k1.y));
        a0 = max3(a0, fabsf(k2.x), fabsf(k2.y));
        a1 = max3(a1, fabsf(k3.x), fabsf(k3.y));
      }
    }
    a = warp_max(fmaxf(a0, a1));
  }
  const float s = __fdiv_rn(a, kInt8Max);
  const bool fast = s >= FLT_MIN;
  const float r = fast ? __frcp_rn(s) : 0.0f;
  const float2 r2 = make_float2(r, r), nr2 = make_float2(-r, -r);
  const float2 m2 = make_float2(kMagic, kMagic), nm2 = make_float2(-kMagic, -kMagic);
  uint2* out8 = codes_bh ? reinterpret_cast<uint2*>(codes_bh + s0 * kHeadDim) + (lane & 15) : nullptr;
  uint4* out16 = reinterpret_cast<uint4*>(f16_bh + s0 * kHeadDim) + (lane & 15);
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int t = 2 * i + half;
    uint2 c8 = make_uint2(0u, 0u);
    uint4 c16 = make_uint4(0u, 0u, 0u, 0u);
    if ((kFull || t < nvalid) && a > 0.0f) {
      const uint4 w = tok8(rows, t, lane);
      float2 x[4] = {bf2(w.x), bf2(w.y), bf2(w.z), bf2(w.w)};
      if (kMu) {
#pragma unroll
        for (int k = 0; k < 4; ++k) x[k] = __fadd2_rn(x[k], nmu[k]);
      }
      float2 tt[4], cc[4];
      float g = 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tt[k] = __ffma2_rn(x[k], r2, m2);
        cc[k] = __fadd2_rn(tt[k], nm2);
        const float2 gk = __ffma2_rn(x[k], nr2, cc[k]);
        g = max3(g, fabsf(gk.x), fabsf(gk.y));
      }
      if (!(fast && g < kHalfGuard)) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          tt[k].x = __uint_as_float(exact_code_bits(x[k].x, s));
          tt[k].y = __uint_as_float(exact_code_bits(x[k].y, s));
          cc[k] = __fadd2_rn(tt[k], nm2);
        }
      }
      c8.x = pack_low_bytes(__float_as_uint(tt[0].x), __float_as_uint(tt[0].y), __float_as_uint(tt[1].x),
                            __float_as_uint(tt[1].y));
      c8.y = pack_low_bytes(__float_as_uint(tt[2].x), __float_as_uint(tt[2].y), __float_as_uint(tt[3].x),
                            __float_as_uint(tt[3].y));
      c16 = make_uint4(f16x2(cc[0].x, cc[0].y), f16x2(cc[1].x, cc[1].y), f16x2(cc[2].x, cc[2].y),
                       f16x2(cc[3].x, cc[3].y));
    }
    if (out8) __stcs(out8 + t * (kHeadDim / 8), c8);
    __stcs(out16 + t * (kHeadDim / 8), c16);
  }
  return s;
}

// Left-to-right fp64 sum of one channel (byte offset `cb` in a row) over the
// first nvalid rows: the reference order, used when the float-pair path
// cannot guarantee it.
__device__ __noinline__ double fp64_chunk_sum(const uint8_t* rows, int nvalid, int cb) {
  double p = 0.0;
  for (int t = 0; t < nvalid; ++t)
    p = __dadd_rn(p, static_cast<double>(
                         __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(rows + t * 256 + cb))
                                         << 16)));
  return p;
}

// Exact fp64 sums of one 32-token chunk for the lane's 8 channels (8-channel
// lanes; results valid in every lane, for channels 8*(lane & 15) .. +8).
//
// Each half-warp runs one float-pair chain per channel over its 16 tokens
// (TwoSum: hi + lo stays the exact running sum while lo's own additions are
// exact); the two chains are joined across the half-warps with one more
// TwoSum. Exactness: every input is a multiple of 2^L, L the last-bit weight
// of the smallest nonzero magnitude in the lane's channels; with E the
// exponent of the largest magnitude, every partial sum is below 32 * 2^(E+1)
// = 2^(E+6) in magnitude, so every TwoSum error is a multiple of 2^L below
// 2^(E-19), and lo, which adds 33 of them, stays below 2^(E-13). lo's sums
// are therefore exact in fp32 while E - 13 <= L + 24; the code takes the fast
// result when E - L <= 36. The exact total T = hi + lo is then a multiple of
// 2^L below 2^(E+6) and fits in 53 bits, as does every prefix of the
// left-to-right fp64 sum, which is therefore exact too and equals T;
// fl64(hi + lo) = T. Otherwise the chunk is summed left to right in fp64.
template <bool kFull>
__device__ __forceinline__ void chunk_sums(const uint8_t* rows, int nvalid, int lane, double (&out)[8]) {
  const int half = lane >> 4;
  const float2 neg1 = make_float2(-1.0f, -1.0f);
  float2 hi[4], lo[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) hi[k] = lo[k] = make_float2(0.0f, 0.0f);
  uint32_t mx0 = 0u, mx1 = 0u;                 // largest magnitude bits, per 16-bit half
  uint32_t mn0 = 0xFFFFFFFFu, mn1 = 0xFFFFFFFFu;  // (magnitude bits - 1); zeros wrap to 0xFFFF
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int t = 2 * i + half;
    if (kFull || t < nvalid) {
      const uint4 w = tok8(rows, t, lane);
      const uint32_t a0 = w.x & kAbs2, a1 = w.y & kAbs2, a2 = w.z & kAbs2, a3 = w.w & kAbs2;
      mx0 = __vimax3_u16x2(mx0, a0, a1);
      mx1 = __vimax3_u16x2(mx1, a2, a3);
      mn0 = __vimin3_u16x2(mn0, __vsub2(a0, 0x00010001u), __vsub2(a1, 0x00010001u));
      mn1 = __vimin3_u16x2(mn1, __vsub2(a2, 0x00010001u), __vsub2(a3, 0x00010001u));
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 x = bf2(ws[k]);
        const float2 sum = __fadd2_rn(hi[k], x);
        const float2 bb = __ffma2_rn(hi[k], neg1, sum);                       // sum - hi
        const float2 t2 = __ffma2_rn(__ffma2_rn(bb, neg1, sum), neg1, hi[k]);  // hi - (sum - bb)
        const float2 t3 = __ffma2_rn(bb, neg1, x);                             // x - bb
        hi[k] = sum;
        lo[k] = __fadd2_rn(lo[k], __fadd2_rn(t2, t3));
      }
    }
  }
  // join the two half-warps' chains (both halves compute the same result)
  uint32_t mx = __vmaxu2(mx0, mx1), mn = __vminu2(mn0, mn1);
  mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
  mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, 16));
  const uint32_t mxb = max(mx & 0xFFFFu, mx >> 16);
  const uint32_t mnb = min(mn & 0xFFFFu, mn >> 16) + 1u;  // 0x10000 when every value is zero
  int ef_min = static_cast<int>((mnb >> 7) & 0xFFu);
  if (ef_min == 0) ef_min = 1;  // subnormal bf16: last-bit weight 2^-133
  int ef_max = static_cast<int>(mxb >> 7);
  if (ef_max == 0) ef_max = 1;
  const bool exact = mnb > 0x7FFFu || ef_max - ef_min <= 36 - 7;  // E - L = (ef_max - ef_min) + 7
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 ohi = make_float2(__shfl_xor_sync(0xffffffffu, hi[k].x, 16), __shfl_xor_sync(0xffffffffu, hi[k].y, 16));
    const float2 olo = make_float2(__shfl_xor_sync(0xffffffffu, lo[k].x, 16), __shfl_xor_sync(0xffffffffu, lo[k].y, 16));
    const float2 sum = __fadd2_rn(hi[k], ohi);
    const float2 bb = __ffma2_rn(hi[k], neg1, sum);
    const float2 t2 = __ffma2_rn(__ffma2_rn(bb, neg1, sum), neg1, hi[k]);
    const float2 t3 = __ffma2_rn(bb, neg1, ohi);
    const float2 l = __fadd2_rn(__fadd2_rn(lo[k], olo), __fadd2_rn(t2, t3));
    out[2 * k] = __dadd_rn(static_cast<double>(sum.x), static_cast<double>(l.x));
    out[2 * k + 1] = __dadd_rn(static_cast<double>(sum.y), static_cast<double>(l.y));
  }
  if (!exact) {
#pragma unroll 1
    for (int c = 0; c < 8; ++c) out[c] = fp64_chunk_sum(rows, nvalid, (lane & 15) * 16 + 2 * c);
  }
}

// Two e4m3 codes: high byte = code(a), low byte = code(b).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(a), "f"(b));
  return r;
}

// Exact path of four V codes (out of line: rare); low byte = channel 0.
__device__ __noinline__ uint32_t exact_v_quad(uint2 w, float4 s) {
  const uint32_t p01 = e4m3x2(__fdiv_rn(hi_bf16(w.x), s.y), __fdiv_rn(lo_bf16(w.x), s.x));
  const uint32_t p23 = e4m3x2(__fdiv_rn(hi_bf16(w.y), s.w), __fdiv_rn(lo_bf16(w.y), s.z));
  return p01 | (p23 << 16);
}

// V codes of one token's 4 channels (4-channel lanes), low byte = channel 0.
// Rounding to e4m3 is monotone, and fl(v / s) lies within 2^-22 relative of
// q = fl(v * fl(1/s)); so when q * (1 - 2^-21) and q * (1 + 2^-21) round to
// the same code, that is the code of fl(v / s); otherwise the exact division
// decides.
__device__ __forceinline__ uint32_t v_code_quad(uint2 w, float2 r01, float2 r23, float4 s, bool fast) {
  const float2 q01 = __fmul2_rn(bf2(w.x), r01), q23 = __fmul2_rn(bf2(w.y), r23);
  const float2 dn = make_float2(kDn, kDn), up = make_float2(kUp, kUp);
  const float2 d01 = __fmul2_rn(q01, dn), u01 = __fmul2_rn(q01, up);
  const float2 d23 = __fmul2_rn(q23, dn), u23 = __fmul2_rn(q23, up);
  const uint32_t cd = e4m3x2(d01.y, d01.x) | (e4m3x2(d23.y, d23.x) << 16);
  const uint32_t cu = e4m3x2(u01.y, u01.x) | (e4m3x2(u23.y, u23.x) << 16);
  if (fast && cd == cu) return cd;
  return exact_v_quad(w, s);
}

// Pairwise tree (padded with +0.0 to a power of two) over `n` group sums
// starting at p, stride 128 doubles, evaluated streaming: stack[l] holds a
// finished subtree of 2^l leaves. The sums are never -0.0, so padding with
// +0.0 changes nothing.
__device__ __forceinline__ double tree_sum(const double* p, int64_t n) {
  double stack[40];
  for (int64_t gi = 0; gi < n; ++gi) {
    double val = __ldcg(p + gi * kHeadDim);
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

// Barrier of one compute team (named barrier 1 + team, 256 threads).
__device__ __forceinline__ void team_bar(int team) { asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "n"(kGroup) : "memory"); }

struct Ctx {
  uint32_t bar0;
  volatile int* abort_flag;
  int* dev_err;
  __device__ uint32_t full(int s) const { return bar0 + 8u * static_cast<uint32_t>(s); }
  __device__ uint32_t empty(int s) const { return bar0 + 8u * static_cast<uint32_t>(kStages + s); }
};

// Bounded wait on an mbarrier phase; on expiry sets the error word and the
// CTA's abort flag.
__device__ __forceinline__ bool wait_bar(const Ctx& cx, uint32_t bar, uint32_t parity) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((it & 127u) == 0) {
      if (*cx.abort_flag) return false;
      const uint64_t now = tc::global_timer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kTimeoutNs) {
        *cx.abort_flag = 1;
        atomicExch(cx.dev_err, kDevErrTimeout);
        return false;
      }
    }
  }
}

// Bounded wait until ready[bh] is set by the CTA that finished the head.
__device__ __forceinline__ bool wait_ready(const Ctx& cx, const unsigned* flag) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v != 0u) return true;
    __nanosleep(64);
    if ((it & 63u) == 63u) {
      if (*cx.abort_flag) return false;
      const uint64_t now = tc::global_timer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kTimeoutNs) {
        *cx.abort_flag = 1;
        atomicExch(cx.dev_err, kDevErrTimeout);
        return false;
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    prologue_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const Params prm, int3 s_axis) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ double ks[kWarps][kHeadDim];
  __shared__ uint32_t vm[kWarps][kHeadDim / 2];
  __shared__ float fin_vmax[kHeadDim];
  __shared__ double fin_right[kHeadDim];
  __shared__ int last_flag;  // stats items: this CTA finished the head
  const uint32_t sbase = tc::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int64_t* meta_item = reinterpret_cast<int64_t*>(smem + kOffMeta);             // [kStages]
  int* meta_tensor = reinterpret_cast<int*>(smem + kOffMeta + kStages * 8);     // [kStages]
  Ctx cx;
  cx.bar0 = sbase + kOffBar;
  cx.abort_flag = reinterpret_cast<volatile int*>(smem + kOffFlags);
  cx.dev_err = prm.dev_err;
  if (threadIdx.x == 0) {
    *cx.abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(cx.full(s), 1);
      tc::mbar_init(cx.empty(s), kTeams * kGroup);  // both teams release every stage
    }
    tc::fence_mbar_init();
  }
  __syncthreads();

  if (warp == kTeams * kWarps) {
    // -------------------------------------------------------------- producer --
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_k);
      tc::prefetch_tmap(&tm_v);
      uint32_t cnt = 0;
      int pending[kStages] = {-1, -1, -1};
      bool ok = true;
      while (ok) {
        const int64_t item = static_cast<int64_t>(atomicAdd(prm.next_item, 1u));
        const bool end = item >= prm.total;
        int tensors[3], nt = 0;
        Item it{0, 0, 0};
        if (end) {
          tensors[nt++] = kEnd;
        } else {
          it = decode_item(item, prm.NH, prm.G, prm.lag);
          if (it.phase == 0) {
            tensors[nt++] = kTensorQ;
            if (prm.smooth_k) tensors[nt++] = kTensorK;
            tensors[nt++] = kTensorV;
          } else {
            // a codes item needs the head's key mean and V scales: its tiles
            // enter the ring only once they are published
            if (!(ok = wait_ready(cx, prm.ready + it.bh))) break;
            tensors[nt++] = kTensorK;
            tensors[nt++] = kTensorV;
          }
        }
        for (int n = 0; n < nt && ok; ++n) {
          const uint32_t st = cnt % kStages, ph = (cnt / kStages) & 1u;
          if (!(ok = wait_bar(cx, cx.empty(st), ph ^ 1u))) break;
          meta_item[st] = end ? -1 : item;
          meta_tensor[st] = tensors[n];
          if (tensors[n] == kEnd) {
            tc::mbar_arrive(cx.full(st));
          } else {
            tc::mbar_arrive_expect_tx(cx.full(st), kTileBytes);
            const CUtensorMap* tm = tensors[n] == kTensorQ ? &tm_q : (tensors[n] == kTensorK ? &tm_k : &tm_v);
            const int32_t h = static_cast<int32_t>(it.bh % prm.H), b = static_cast<int32_t>(it.bh / prm.H);
            const int32_t s0 = static_cast<int32_t>(it.g * kGroup);
            // map dims: (channel, s, h, b) or (channel, h, s, b) by stride order
            const int ax = tensors[n] == kTensorQ ? s_axis.x : (tensors[n] == kTensorK ? s_axis.y : s_axis.z);
            if (ax == 1)
              tc::tma_load_4d(sbase + st * kTileBytes, tm, 0, s0, h, b, cx.full(st));
            else
              tc::tma_load_4d(sbase + st * kTileBytes, tm, 0, h, s0, b, cx.full(st));
            pending[st] = static_cast<int>(ph);
          }
          ++cnt;
        }
        if (end) break;
      }
      if (!ok) {
        Ctx drain = cx;
        volatile int no_abort = 0;
        drain.abort_flag = &no_abort;
        for (int s = 0; s < kStages; ++s)
          if (pending[s] >= 0) wait_bar(drain, cx.full(s), static_cast<uint32_t>(pending[s]));
      }
    }
    return;
  }

  // --------------------------------------------------------------- compute --
  // Two teams of 8 warps work on different tiles of the same item: team 0 on
  // the first tile (Q of a stats item, K of a codes item), team 1 on the rest
  // (K sums and V maxima of a stats item, V codes of a codes item). Both
  // teams wait on every stage in ring order, so a parity wait never meets a
  // barrier two phases behind; a team releases the stages it does not use as
  // soon as they are full, and a stage is refilled once both have released it.
  // The tiles of a codes item enter the ring only after the producer has seen
  // the head's statistics published, so the compute warps never wait for them.
  const int team = warp / kWarps, tw = warp % kWarps, tt = threadIdx.x % kGroup;
  const int64_t S = prm.S, S_pad = prm.S_pad, G = prm.G;
  uint32_t cnt = 0;
  // wait for ring position c to be full, then release it unused
  auto pass = [&](uint32_t c) -> bool {
    if (!wait_bar(cx, cx.full(c % kStages), (c / kStages) & 1u)) return false;
    tc::mbar_arrive(cx.empty(c % kStages));
    return true;
  };
  while (true) {
    const uint32_t st = cnt % kStages;
    if (!wait_bar(cx, cx.full(st), (cnt / kStages) & 1u)) break;
    const int64_t item = meta_item[st];
    if (meta_tensor[st] == kEnd) break;
    const Item it = decode_item(item, prm.NH, G, prm.lag);
    const uint32_t n_stages = it.phase == 0 ? (prm.smooth_k ? 3u : 2u) : 2u;
    const int64_t bh = it.bh;
    const int64_t s0 = it.g * kGroup + tw * 32;
    const int nvalid = valid_in_chunk(S, s0);
    const bool in_pad = s0 < S_pad;  // rows past S_pad do not exist in the outputs
    if (team == 1) tc::mbar_arrive(cx.empty(st));  // the first tile is team 0's
    const uint32_t mine = cnt + static_cast<uint32_t>(team);  // this team's first ring position
    const uint8_t* rows = smem + (mine % kStages) * kTileBytes + tw * 32 * 256;
    bool ok = true;

    if (team == 0 && it.phase == 0) {
      // Q codes and scale
      if (in_pad) {
        const float2 nz[4] = {};
        int8_t* qc = prm.write_int8 ? prm.out.q_codes + bh * S_pad * kHeadDim : nullptr;
        uint16_t* q16 = prm.out.q16 + bh * S_pad * kHeadDim;
        const float s = nvalid == 32 ? quantize_block<false, true>(rows, nz, 32, qc, q16, s0, lane)
                                     : quantize_block<false, false>(rows, nz, nvalid, qc, q16, s0, lane);
        if (lane == 0) prm.out.q_scale[bh * (S_pad / kQKBlock) + s0 / kQKBlock] = s;
      }
      tc::mbar_arrive(cx.empty(st));
      for (uint32_t c = 1; c < n_stages && ok; ++c) ok = pass(cnt + c);
      if (!ok) break;
    } else if (team == 1 && it.phase == 0) {
      // K tile: exact fp64 chunk sums
      uint32_t c2 = mine;
      if (!wait_bar(cx, cx.full(c2 % kStages), (c2 / kStages) & 1u)) break;
      if (prm.smooth_k) {
        double sums[8];
        if (nvalid == 32)
          chunk_sums<true>(rows, 32, lane, sums);
        else
          chunk_sums<false>(rows, nvalid, lane, sums);
        tc::mbar_arrive(cx.empty(c2 % kStages));
        ++c2;
        if (lane < 16) {
#pragma unroll
          for (int c = 0; c < 8; ++c) ks[tw][8 * lane + c] = sums[c];
        }
      }
      // V tile: max |v| per channel (bf16 magnitudes compare as integers)
      const uint32_t sv = c2 % kStages;
      if (c2 != mine && !wait_bar(cx, cx.full(sv), (c2 / kStages) & 1u)) break;
      const uint8_t* vr = smem + sv * kTileBytes + tw * 32 * 256;
      const int half = lane >> 4;
      uint32_t m4[4] = {0u, 0u, 0u, 0u};  // channel pairs (8l, 8l+1) .. (8l+6, 8l+7)
      if (nvalid == 32) {
#pragma unroll 4
        for (int i = 0; i < 8; ++i) {
          const uint4 wa = tok8(vr, 4 * i + half, lane), wb = tok8(vr, 4 * i + 2 + half, lane);
          m4[0] = __vimax3_u16x2(m4[0], wa.x & kAbs2, wb.x & kAbs2);
          m4[1] = __vimax3_u16x2(m4[1], wa.y & kAbs2, wb.y & kAbs2);
          m4[2] = __vimax3_u16x2(m4[2], wa.z & kAbs2, wb.z & kAbs2);
          m4[3] = __vimax3_u16x2(m4[3], wa.w & kAbs2, wb.w & kAbs2);
        }
      } else {
        for (int i = 0; i < 16; ++i) {
          const int t = 2 * i + half;
          if (t < nvalid) {
            const uint4 w = tok8(vr, t, lane);
            m4[0] = __vmaxu2(m4[0], w.x & kAbs2);
            m4[1] = __vmaxu2(m4[1], w.y & kAbs2);
            m4[2] = __vmaxu2(m4[2], w.z & kAbs2);
            m4[3] = __vmaxu2(m4[3], w.w & kAbs2);
          }
        }
      }
      tc::mbar_arrive(cx.empty(sv));
#pragma unroll
      for (int k = 0; k < 4; ++k) m4[k] = __vmaxu2(m4[k], __shfl_xor_sync(0xffffffffu, m4[k], 16));
      if (lane < 16) {
#pragma unroll
        for (int k = 0; k < 4; ++k) vm[tw][4 * lane + k] = m4[k];
      }
      team_bar(1);
      if (tt < kHeadDim) {
        const int c = tt;
        const int64_t slot = (bh * G + it.g) * kHeadDim + c;
        if (prm.smooth_k) {
          // levels 1..3 of the pairwise tree over the group's 8 chunks
          const double l0 = __dadd_rn(ks[0][c], ks[1][c]);
          const double l1 = __dadd_rn(ks[2][c], ks[3][c]);
          const double l2 = __dadd_rn(ks[4][c], ks[5][c]);
          const double l3 = __dadd_rn(ks[6][c], ks[7][c]);
          prm.ksum[slot] = __dadd_rn(__dadd_rn(l0, l1), __dadd_rn(l2, l3));
        }
        uint32_t mb = 0u;
#pragma unroll
        for (int i = 0; i < kWarps; ++i) {
          const uint32_t pair = vm[i][c >> 1];
          mb = max(mb, (c & 1) ? (pair >> 16) : (pair & 0xFFFFu));
        }
        prm.vmax[slot] = __uint_as_float(mb << 16);
        __threadfence();
      }
      team_bar(1);
      if (tt == 0) last_flag = atomicAdd(prm.done + bh, 1u) == static_cast<unsigned>(G - 1);
      team_bar(1);
      if (last_flag) {
        // finish the head: the group sums are complete (each writer fenced
        // before counting itself done)
        __threadfence();
        const int c = tt & (kHeadDim - 1), half = tt >> 7;
        int64_t P = 1;
        while (P < G) P *= 2;
        const int64_t lo = half == 0 ? 0 : (P == 1 ? 1 : P / 2);
        const int64_t hi_end = half == 0 ? (P == 1 ? 1 : P / 2) : P;
        const int64_t n = max(int64_t(0), min(G, hi_end) - lo);
        double t = 0.0;
        if (prm.smooth_k && n > 0) t = tree_sum(prm.ksum + (bh * G + lo) * kHeadDim + c, n);
        float vmx = 0.0f;
        for (int64_t gi = lo; gi < lo + n; ++gi) vmx = fmaxf(vmx, __ldcg(prm.vmax + (bh * G + gi) * kHeadDim + c));
        if (half == 1) {
          fin_right[c] = t;
          fin_vmax[c] = vmx;
        }
        team_bar(1);
        if (half == 0) {
          float mu = 0.0f;
          if (prm.smooth_k) {
            const double total = P > 1 ? __dadd_rn(t, fin_right[c]) : t;
            mu = __double2float_rn(__ddiv_rn(total, static_cast<double>(S)));
          }
          prm.out.k_mean[bh * kHeadDim + c] = mu;
          prm.out.v_scale[bh * kHeadDim + c] = __fdiv_rn(fmaxf(vmx, fin_vmax[c]), kE4M3Max);
          __threadfence();
        }
        team_bar(1);
        if (tt == 0) {
          asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(prm.ready + bh), "r"(1u) : "memory");
        }
      }
    } else {
      // codes item (the head's key mean and V scales are published)
      if (team == 1 && !wait_bar(cx, cx.full(mine % kStages), (mine / kStages) & 1u)) break;
      if (team == 0) {
        // K codes of k - mean
        if (in_pad) {
          int8_t* kc = prm.write_int8 ? prm.out.k_codes + bh * S_pad * kHeadDim : nullptr;
          uint16_t* k16 = prm.out.k16 + bh * S_pad * kHeadDim;
          float skv;
          if (prm.smooth_k) {
            const float4* mp = reinterpret_cast<const float4*>(prm.out.k_mean + bh * kHeadDim + 8 * (lane & 15));
            const float4 ma = __ldcg(mp), mb = __ldcg(mp + 1);
            const float2 nmu[4] = {make_float2(-ma.x, -ma.y), make_float2(-ma.z, -ma.w), make_float2(-mb.x, -mb.y),
                                   make_float2(-mb.z, -mb.w)};
            skv = nvalid == 32 ? quantize_block<true, true>(rows, nmu, 32, kc, k16, s0, lane)
                               : quantize_block<true, false>(rows, nmu, nvalid, kc, k16, s0, lane);
          } else {
            const float2 nz[4] = {};
            skv = nvalid == 32 ? quantize_block<false, true>(rows, nz, 32, kc, k16, s0, lane)
                               : quantize_block<false, false>(rows, nz, nvalid, kc, k16, s0, lane);
          }
          if (lane == 0) prm.out.k_scale[bh * (S_pad / kQKBlock) + s0 / kQKBlock] = skv;
        }
        tc::mbar_arrive(cx.empty(st));
        if (!pass(cnt + 1)) break;
      } else {
        // V codes, transposed to [channel][token] (4-channel lanes)
        if (in_pad) {
          const float4 svs = __ldcg(reinterpret_cast<const float4*>(prm.out.v_scale + bh * kHeadDim + 4 * lane));
          const float sc[4] = {svs.x, svs.y, svs.z, svs.w};
          float rv[4];
          uint32_t keep = 0u;
          bool fast = true;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            rv[c] = sc[c] >= FLT_MIN ? __frcp_rn(sc[c]) : 0.0f;
            if (sc[c] > 0.0f) keep |= 0xFFu << (8 * c);
            fast = fast && (sc[c] >= FLT_MIN || sc[c] == 0.0f);  // zero channels are masked to code 0
          }
          const float2 r01 = make_float2(rv[0], rv[1]), r23 = make_float2(rv[2], rv[3]);
          uint32_t cw[4][8];  // cw[c][j]: tokens 4j..4j+3 of channel 4*lane+c
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint32_t a[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int t = 4 * j + q;
              a[q] = (nvalid == 32 || t < nvalid) ? v_code_quad(tok4(rows, t, lane), r01, r23, svs, fast) & keep : 0u;
            }
            // 4x4 byte transpose: a[q] = token q's channels -> cw[c][j] = channel c's tokens
            const uint32_t t01l = __byte_perm(a[0], a[1], 0x5140), t01h = __byte_perm(a[0], a[1], 0x7362);
            const uint32_t t23l = __byte_perm(a[2], a[3], 0x5140), t23h = __byte_perm(a[2], a[3], 0x7362);
            cw[0][j] = __byte_perm(t01l, t23l, 0x5410);
            cw[1][j] = __byte_perm(t01l, t23l, 0x7632);
            cw[2][j] = __byte_perm(t01h, t23h, 0x5410);
            cw[3][j] = __byte_perm(t01h, t23h, 0x7632);
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint4* dst = reinterpret_cast<uint4*>(prm.out.vt_codes + (bh * kHeadDim + 4 * lane + c) * S_pad + s0);
            __stcs(dst, make_uint4(cw[c][0], cw[c][1], cw[c][2], cw[c][3]));
            __stcs(dst + 1, make_uint4(cw[c][4], cw[c][5], cw[c][6], cw[c][7]));
          }
        }
        tc::mbar_arrive(cx.empty(mine % kStages));
      }
    }
    cnt += n_stages;
  }
}

struct ScratchLayout {
  size_t done_off, ready_off, ksum_off, vmax_off, header, total;
};

ScratchLayout scratch_layout(int64_t B, int64_t S, int64_t H) {
  const int64_t G = div_up(S, kGroup);
  const size_t NH = static_cast<size_t>(B * H);
  const size_t n = NH * static_cast<size_t>(G) * kHeadDim;
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  ScratchLayout l;
  l.done_off = 256;
  l.ready_off = l.done_off + r256(NH * 4);
  l.header = l.ready_off + r256(NH * 4);
  l.ksum_off = l.header;
  l.vmax_off = l.ksum_off + r256(n * sizeof(double));
  l.total = l.vmax_off + r256(n * sizeof(float));
  return l;
}

// 4-D bf16 map over one input: dims (channel, a1, a2, b) where (a1, a2) are
// (s, h) or (h, s) in increasing stride order; boxes of 128 channels x 256
// tokens. Returns the position of the token axis (1 or 2), or 0 on failure.
int make_input_map(CUtensorMap* m, const Bf16In& t, int64_t B, int64_t S, int64_t H) {
  const bool s_first = t.ss <= t.sh;
  const uint64_t dims[4] = {static_cast<uint64_t>(kHeadDim), static_cast<uint64_t>(s_first ? S : H),
                            static_cast<uint64_t>(s_first ? H : S), static_cast<uint64_t>(B)};
  const uint64_t strides[3] = {static_cast<uint64_t>((s_first ? t.ss : t.sh) * 2),
                               static_cast<uint64_t>((s_first ? t.sh : t.ss) * 2), static_cast<uint64_t>(t.sb * 2)};
  const uint32_t box[4] = {kHeadDim, s_first ? static_cast<uint32_t>(kGroup) : 1u,
                           s_first ? 1u : static_cast<uint32_t>(kGroup), 1u};
  if (!make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, t.p, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
    return 0;
  return s_first ? 1 : 2;
}

}  // namespace

size_t prologue_scratch_bytes(int64_t B, int64_t S, int64_t H) { return scratch_layout(B, S, H).total; }

cudaError_t launch_prologue(const Bf16In& q, const Bf16In& k, const Bf16In& v, int64_t B, int64_t S, int64_t H,
                            bool smooth_k, const Bundle& out, void* scratch, bool write_int8, int* dev_err,
                            cudaStream_t stream) {
  const ScratchLayout l = scratch_layout(B, S, H);
  char* sc = static_cast<char*>(scratch);
  Params p;
  p.S = S;
  p.S_pad = padded_len(S);
  p.H = H;
  p.NH = B * H;
  p.G = div_up(S, kGroup);
  p.total = 2 * p.NH * p.G;
  // codes of head h follow the stats of head h + lag: the bytes that pass
  // through L2 in between (about lag heads of inputs and outputs) must leave
  // head h's K and V in L2, while lag must exceed the heads in flight
  const double head_bytes = static_cast<double>(S) * kHeadDim * (3 * 2 + 2 * 1 + 2 * 2 + 1);
  int64_t lag = static_cast<int64_t>(0.7 * static_cast<double>(l2_bytes_current()) / head_bytes);
  if (lag < 2) lag = 2;
  if (lag > p.NH) lag = p.NH;
  p.lag = lag;
  p.smooth_k = smooth_k ? 1 : 0;
  p.write_int8 = write_int8 ? 1 : 0;
  p.out = out;
  p.next_item = reinterpret_cast<unsigned*>(sc);
  p.done = reinterpret_cast<unsigned*>(sc + l.done_off);
  p.ready = reinterpret_cast<unsigned*>(sc + l.ready_off);
  p.ksum = reinterpret_cast<double*>(sc + l.ksum_off);
  p.vmax = reinterpret_cast<float*>(sc + l.vmax_off);
  p.dev_err = dev_err;
  CUtensorMap tq, tk, tv;
  const int aq = make_input_map(&tq, q, B, S, H), ak = make_input_map(&tk, k, B, S, H),
            av = make_input_map(&tv, v, B, S, H);
  if (aq == 0 || ak == 0 || av == 0) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(scratch, 0, l.header, stream);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(prologue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int sms = sm_count_current();
  const int grid = static_cast<int>(p.total < sms ? p.total : sms);
  prologue_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p, make_int3(aq, ak, av));
  return cudaGetLastError();
}

}  // namespace sage
