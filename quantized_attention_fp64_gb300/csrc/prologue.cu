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
// One persistent kernel, one CTA per SM: two teams of 8 compute warps (they
// swap roles from one item to the next), a TMA producer warp and a counter
// warp. The work is a list of items claimed in order from a global counter:
//   stats item (head, 128-token group): Q codes and scales; exact fp64 key
//     sums of the group (4 chunks of 32 tokens, then a 2-level pairwise tree);
//     the group's max |v| per channel. The counter warp counts each finished
//     group with an atomic per head; the CTA that counts a head's last group
//     finishes that head (team 1, on a finish marker the producer puts in the
//     ring): the pairwise tree over its group sums gives the key mean, the max
//     over groups the V scales; then it publishes the head as ready.
//   codes item (head, 128-token group): K codes of k - mean, V codes
//     (transposed); the producer loads its tiles once the head is ready.
// All stats items come before all codes items (the general order, codes of
// head h after the stats of head h + L, is kept with L = every head; see the
// launcher for why). The producer loads each tensor's 128-token x 128-channel bf16
// tile with one 4-D TMA copy into a 6-stage ring (32 KB per stage); an item
// takes 2 or 3 stages, so the next items' tiles load while one is computed.
// Two warps share each 32-token block (16 tokens each) and exchange partial
// maxima and sums through shared memory. Items are claimed in a global order
// and every CTA processes its items in claim order, so the stats items a
// codes item waits for were all claimed earlier and always progress: the
// waits end. They are bounded anyway.
//
// Exactness of the key sum. fp64 adds run at under 2 per clock per SM on
// this GPU, far below what the HBM stream needs, so each 32-token chunk is
// summed as unevaluated pairs of floats (TwoSum chains, two-element packed
// arithmetic), which give the exact chunk sum whenever the spread of
// exponents in the chunk is bounded (see key_sum_partial); that exact sum is
// what the left-to-right fp64 sum produces too, so the result is
// bit-identical. Otherwise the chunk is summed left to right in fp64.
//
// Exactness of the codes. A code is rint(x / s) with x / s correctly
// rounded in fp32. The fast path multiplies by fl(1/s) and falls back to the
// exact division whenever the product is within 2^-15 of a half-integer
// (quantize_half_block). For e4m3, rounding is monotone, so when
// q = fl(v*fl(1/s)) scaled by (1 - 2^-21) and by (1 + 2^-21) round to the same
// code, fl(v/s) (within 2^-22 relative of q) does too; otherwise the exact
// division decides, element by element (v_code_brackets, v_codes_exact). Q and V maxima are taken
// on the bf16 bit patterns, whose magnitudes order as integers.
#include <cuda_fp16.h>

#include <cfloat>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace sage {
namespace {

constexpr int kItemTokens = 128;                // tokens of one item (one group)
constexpr int kChunks = kItemTokens / kQKBlock; // 32-token chunks per item
constexpr int kWarps = 8;                       // compute warps per team
constexpr int kHalfRows = 16;                   // tokens per warp (two warps per chunk)
constexpr int kTeamThreads = kWarps * 32;
constexpr int kTeams = 2;
constexpr int kThreads = kTeams * kTeamThreads + 64;  // + the producer and the counter warp
constexpr int kStages = 6;
constexpr uint32_t kTileBytes = kItemTokens * kHeadDim * 2;  // one bf16 tile: 128 tokens x 128 channels
constexpr float kMagic = 12582912.0f;          // 1.5 * 2^23: q + kMagic = rint_even(q) + kMagic for |q| < 2^22
constexpr float kHalfGuard = 0.5f - 0x1p-15f;  // fast-path guard for rint
constexpr float kDn = 1.0f - 0x1p-21f;
constexpr float kUp = 1.0f + 0x1p-21f;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait
static_assert(kChunks * 2 == kWarps, "two warps per 32-token chunk");

// ring entries: a tile of one tensor, a marker to finish a head, the end
enum : int { kTensorQ = 0, kTensorK = 1, kTensorV = 2, kFinish = 3, kEnd = 4 };
constexpr int kEvents = 8;   // ring of "group done" events from the teams to the counter warp
static_assert(kEvents % 2 == 0, "a report slot is always written by the same team");
constexpr int kFinCap = 32;  // heads waiting for their finish marker (see the producer)

// shared memory: kStages tiles; per stage the head statistics a codes item
// needs (key mean and V scales, 1 KB); the barriers; per-stage item tags;
// the event ring and the finish queue
constexpr uint32_t kOffHstat = kStages * kTileBytes;
constexpr uint32_t kHstatBytes = 3 * kHeadDim * 4;  // key mean, V scales, their reciprocals
constexpr uint32_t kOffBar = kOffHstat + kStages * kHstatBytes;
constexpr int kNumBars = 2 * kStages + 2 * kEvents;  // full, empty, event full, event empty
constexpr uint32_t kOffMeta = kOffBar + kNumBars * 8;
constexpr uint32_t kOffEvt = kOffMeta + kStages * 24;  // per stage: item (or head), head, group | phase << 32
constexpr uint32_t kOffFinQ = kOffEvt + kEvents * 8;
constexpr uint32_t kOffFlags = kOffFinQ + kFinCap * 8;  // abort flag, finish-queue tail, groups counted
constexpr uint32_t kSmemBytes = kOffFlags + 16 + 1024;  // + alignment slack

struct Params {
  int64_t S, S_pad, H, NH, G, lag, total;  // H, NH: (virtual) heads per batch and in all
  int64_t Hr;  // head-pair mode: the real head count per batch
  int smooth_k, write_int8;
  Bundle out;
  unsigned* next_item;
  unsigned* done;   // [NH]: stats items finished per head
  unsigned* ready;  // [NH]: 1 once the head's key mean and V scales are written
  double* ksum;     // [NH][G][128]
  float* vmax;      // [NH][G][128]
  float* vrcp;      // [NH][128]: fl(1/s_v) of each finished head (0 for s_v < FLT_MIN)
  float* hstat_v;   // head-pair mode: [NH][256] key mean and V scales of each finished virtual head
  int* dev_err;
};

// Head-pair mode (head dimension 64): virtual head bh = b * H + hp holds the
// real heads 2hp and 2hp + 1 of batch b side by side, as channels 0-63 and
// 64-127 of a 128-channel row, so the kernels below run unchanged on them;
// only the per-block INT8 scales are per real head, and the outputs go to
// the real heads' places in a head-dimension-64 bundle. out_head returns the
// bundle head index (b * Hr + h) of half hf of bh, or -1 for the missing
// second head of an odd head count (its input rows read as zeros).
template <bool kPair>
__device__ __forceinline__ int64_t out_head(const Params& prm, int64_t bh, int hf) {
  if (!kPair) return bh;
  const int64_t b = bh / prm.H, h = 2 * (bh % prm.H) + hf;
  return h < prm.Hr ? b * prm.Hr + h : -1;
}
template <bool kPair>
constexpr int kOutDim = kPair ? kHeadDim / 2 : kHeadDim;

// The lane's output positions for quantize_half_block (8-channel lanes) at
// token s0 of virtual head bh: c16 in the fp16 code copies and c8 in the
// int8 codes (null unless `codes`); both null for a missing head. Returns
// the lane's bundle head index.
template <bool kPair>
__device__ __forceinline__ int64_t lane_codes(const Params& prm, int8_t* codes, uint16_t* f16, int64_t bh,
                                              int64_t s0, int lane, int8_t*& c8, uint16_t*& c16) {
  const int64_t head = out_head<kPair>(prm, bh, kPair ? (lane >> 3) & 1 : 0);
  if (head < 0) {
    c8 = nullptr;
    c16 = nullptr;
    return head;
  }
  const int64_t off = (head * prm.S_pad + s0) * kOutDim<kPair> + 8 * (lane & (kPair ? 7 : 15));
  c8 = codes ? codes + off : nullptr;
  c16 = f16 + off;
  return head;
}

// The scale of a 32-token block: lane 0 (and lane 8 with kPair) of the
// block's first warp stores it for its head.
template <bool kPair>
__device__ __forceinline__ void store_block_scale(float* scales, int64_t head, int64_t nblk, int64_t blk, float s,
                                                  int lane, int sub) {
  if (sub == 0 && (kPair ? (lane & 23) == 0 : lane == 0) && head >= 0) scales[head * nblk + blk] = s;
}

// The lane's V-code position (4-channel lanes: channels 4*lane .. +3,
// transposed rows S_pad apart) at token s0 of virtual head bh, or null for
// a missing head.
template <bool kPair>
__device__ __forceinline__ uint8_t* lane_vt(const Params& prm, int64_t bh, int64_t s0, int lane) {
  const int64_t head = out_head<kPair>(prm, bh, kPair ? lane >> 4 : 0);
  if (head < 0) return nullptr;
  return prm.out.vt_codes + (head * kOutDim<kPair> + ((4 * lane) & (kOutDim<kPair> - 1))) * prm.S_pad + s0;
}

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

// Number of tokens s0 .. s0+n-1 that are below S.
__device__ __forceinline__ int valid_rows(int64_t S, int64_t s0, int n) {
  const int64_t d = S - s0;
  return d <= 0 ? 0 : (d >= n ? n : static_cast<int>(d));
}

// Shared-memory tiles hold 256-byte token rows (128 bf16 channels). Two lane
// mappings read them without bank conflicts:
//  - 8-channel lanes: lane l reads channels 8*(l & 15) .. +8 of token
//    2*i + (l >> 4), so one warp instruction covers two whole rows;
//  - 4-channel lanes: lane l reads channels 4*l .. +4 of one token, one row
//    per warp instruction (used where each lane needs every token).
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

// Maxima over the warp; with kPair over the 16 lanes that share bit 3 of the
// lane index (with 8-channel lanes: the 64 channels of one head of a pair).
template <bool kPair = false>
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    if (!(kPair && o == 8)) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <bool kPair = false>
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    if (!(kPair && o == 8)) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
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

// Barrier of the two warps that share a 32-token block: named barriers 3..10
// (0 is __syncthreads, 1 and 2 the team barriers).
__device__ __forceinline__ void pair_bar(int pair) {
  asm volatile("bar.sync %0, 64;" ::"r"(3 + pair) : "memory");
}

// Exact path of a code: bits of fl(fl(x / s) + kMagic), whose low byte is
// rint_even(fl(x / s)) as an int8. Out of line: the fast path below decides
// all but a few codes in 10^4.
__device__ __noinline__ uint32_t exact_code_bits(float x, float s) {
  return __float_as_uint(__fadd_rn(__fdiv_rn(x, s), kMagic));
}

// One warp's half (16 tokens) of a 32-token INT8 block: codes and scale of x
// (kMu false) or of fl(x - mu) (kMu true; nmu holds -mu for the lane's 8
// channels as pairs). rows: the warp's 16 rows of a shared tile, read with
// 8-channel lanes; nvalid: how many of them are below S (kFull: all 16). The
// block's amax is the max of both halves: each warp posts its own in
// x_mine and reads the other's from x_other after the pair barrier. With
// kPair the 128 channels are two heads of 64 (lanes with bit 3 clear and
// set), each with its own amax, posted in x_mine[0] and x_mine[1]. c16 (and
// c8, when not null) point at the lane's 8 channels of the warp's first row
// in the fp16 code copies (and the int8 codes), rows `row_elems` apart; the
// codes of rows s0 .. s0+15 go there with streaming stores, zero for rows at
// or past nvalid; a null c16 (the missing head of an odd pair) stores
// nothing. Returns the scale of the lane's head.
//
// Fast path for the codes (two-element packed arithmetic): t = fl(x*r + M)
// with r = fl(1/s) and M = 1.5*2^23 is M + rint_even(x*r) (the spacing of
// floats near M is 1); c = t - M exactly; g = fl(c - x*r). x*r is within
// 2^-17 of x/s, and so is fl(x/s) (|x/s| <= 127.5), so when |g| < 1/2 - 2^-15
// the code c is rint_even(fl(x/s)); otherwise the exact division decides.
template <bool kMu, bool kFull, bool kPair = false>
__device__ __forceinline__ float quantize_half_block(const uint8_t* rows, const float2 (&nmu)[4], int nvalid,
                                                     int8_t* c8, uint16_t* c16, int row_elems, int lane,
                                                     volatile float* x_mine, volatile float* x_other, int pair) {
  const int half = lane >> 4;
  float a;
  if (!kMu) {
    // amax on the bf16 bit patterns (magnitudes order as integers)
    uint32_t m0 = 0u, m1 = 0u;
#pragma unroll
    for (int i = 0; i < kHalfRows / 2; ++i) {
      const int t = 2 * i + half;
      if (kFull || t < nvalid) {
        const uint4 w = tok8(rows, t, lane);
        m0 = __vimax3_u16x2(m0, w.x & kAbs2, w.y & kAbs2);
        m1 = __vimax3_u16x2(m1, w.z & kAbs2, w.w & kAbs2);
      }
    }
    const uint32_t m = __vmaxu2(m0, m1);
    a = __uint_as_float(warp_max_u32<kPair>(max(m & 0xFFFFu, m >> 16)) << 16);
  } else {
    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
    for (int i = 0; i < kHalfRows / 2; ++i) {
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
    a = warp_max<kPair>(fmaxf(a0, a1));
  }
  const int hf = kPair ? (lane >> 3) & 1 : 0;
  if (kPair ? (lane & 23) == 0 : lane == 0) x_mine[hf] = a;  // lanes 0 and 8 with kPair
  pair_bar(pair);
  a = fmaxf(a, x_other[hf]);
  const float s = __fdiv_rn(a, kInt8Max);
  const bool fast = s >= FLT_MIN;
  const float r = fast ? __frcp_rn(s) : 0.0f;
  const float2 r2 = make_float2(r, r), nr2 = make_float2(-r, -r);
  const float2 m2 = make_float2(kMagic, kMagic), nm2 = make_float2(-kMagic, -kMagic);
  uint2* out8 = c16 != nullptr ? reinterpret_cast<uint2*>(c8) : nullptr;
  uint4* out16 = reinterpret_cast<uint4*>(c16);
  const int rs = row_elems / 8;  // row stride in 8-element units
  uint32_t redo = 0u;  // bit i: row 2i + half needs the exact division
#pragma unroll
  for (int i = 0; i < kHalfRows / 2; ++i) {
    const int t = 2 * i + half;
    uint2 c8v = make_uint2(0u, 0u);
    uint4 c16v = make_uint4(0u, 0u, 0u, 0u);
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
      if (!(fast && g < kHalfGuard)) redo |= 1u << i;
      c8v = make_uint2(pack_low_bytes(__float_as_uint(tt[0].x), __float_as_uint(tt[0].y), __float_as_uint(tt[1].x),
                                      __float_as_uint(tt[1].y)),
                       pack_low_bytes(__float_as_uint(tt[2].x), __float_as_uint(tt[2].y), __float_as_uint(tt[3].x),
                                      __float_as_uint(tt[3].y)));
      c16v = make_uint4(f16x2(cc[0].x, cc[0].y), f16x2(cc[1].x, cc[1].y), f16x2(cc[2].x, cc[2].y),
                        f16x2(cc[3].x, cc[3].y));
    }
    if (out8) __stcs(out8 + t * rs, c8v);
    if (out16) __stcs(out16 + t * rs, c16v);
  }
  if (redo != 0u && out16) {
    // rare: rows where a fast code could be off by one are recomputed by the
    // exact division and stored again (same thread, same address: the later
    // store wins)
#pragma unroll 1
    for (int i = 0; i < kHalfRows / 2; ++i) {
      if (!((redo >> i) & 1u)) continue;
      const int t = 2 * i + half;
      const uint4 w = tok8(rows, t, lane);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
      uint32_t b[8];
      float cf[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float2 x = bf2(ws[k]);
        if (kMu) x = __fadd2_rn(x, nmu[k]);
        b[2 * k] = exact_code_bits(x.x, s);
        b[2 * k + 1] = exact_code_bits(x.y, s);
        cf[2 * k] = __fsub_rn(__uint_as_float(b[2 * k]), kMagic);
        cf[2 * k + 1] = __fsub_rn(__uint_as_float(b[2 * k + 1]), kMagic);
      }
      if (out8)
        __stcs(out8 + t * rs, make_uint2(pack_low_bytes(b[0], b[1], b[2], b[3]), pack_low_bytes(b[4], b[5], b[6], b[7])));
      __stcs(out16 + t * rs,
             make_uint4(f16x2(cf[0], cf[1]), f16x2(cf[2], cf[3]), f16x2(cf[4], cf[5]), f16x2(cf[6], cf[7])));
    }
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

// TwoSum of pairs: s = fl(a + b) and the exact error e = (a + b) - s.
__device__ __forceinline__ void two_sum2(float2 a, float2 b, float2& s, float2& e) {
  const float2 neg1 = make_float2(-1.0f, -1.0f);
  s = __fadd2_rn(a, b);
  const float2 bb = __ffma2_rn(a, neg1, s);                       // s - a
  const float2 ea = __ffma2_rn(__ffma2_rn(bb, neg1, s), neg1, a);  // a - (s - bb)
  const float2 eb = __ffma2_rn(bb, neg1, b);                       // b - bb
  e = __fadd2_rn(ea, eb);
}

// One warp's part of the exact fp64 sums of a 32-token key chunk: its 16
// rows (8-channel lanes), summed by one float-pair chain per channel in each
// half-warp and joined across the half-warps. On return every lane holds, for
// channels 8*(lane & 15) .. +8 as pairs, hi + lo = the exact sum of its rows
// (while lo's additions are exact, see below), and mx / mn the largest
// magnitude bits and (smallest nonzero magnitude bits - 1) of its rows, per
// 16-bit half.
//
// Exactness (the two warps of a chunk are joined the same way by the
// caller): every input is a multiple of 2^L, L the last-bit weight of the
// smallest nonzero magnitude among the chunk's values in these channels; with
// E the exponent of the largest magnitude, every partial sum is below
// 32 * 2^(E+1) = 2^(E+6), so every TwoSum error is a multiple of 2^L below
// 2^(E-19), and lo, which adds 35 of them (four chains of 8 tokens and three
// joins), stays below 2^(E-13). lo's sums are therefore exact in fp32 while
// E - 13 <= L + 24; the fast result is used when E - L <= 36. The exact total
// T = hi + lo is then a multiple of 2^L below 2^(E+6) and fits in 53 bits, as
// does every prefix of the left-to-right fp64 sum, which is therefore exact
// too and equals T; fl64(hi + lo) = T. Otherwise the chunk is summed left to
// right in fp64.
template <bool kFull>
__device__ __forceinline__ void key_sum_partial(const uint8_t* rows, int nvalid, int lane, float2 (&hi)[4],
                                                float2 (&lo)[4], uint32_t& mx, uint32_t& mn) {
  const int half = lane >> 4;
#pragma unroll
  for (int k = 0; k < 4; ++k) hi[k] = lo[k] = make_float2(0.0f, 0.0f);
  uint32_t mx0 = 0u, mx1 = 0u;
  uint32_t mn0 = 0xFFFFFFFFu, mn1 = 0xFFFFFFFFu;  // zeros wrap to 0xFFFF and never win
#pragma unroll 4
  for (int i = 0; i < kHalfRows / 2; ++i) {
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
        float2 s, e;
        two_sum2(hi[k], bf2(ws[k]), s, e);
        hi[k] = s;
        lo[k] = __fadd2_rn(lo[k], e);
      }
    }
  }
  mx = __vmaxu2(mx0, mx1);
  mn = __vminu2(mn0, mn1);
  mx = __vmaxu2(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
  mn = __vminu2(mn, __shfl_xor_sync(0xffffffffu, mn, 16));
  // join the half-warps' chains (both halves compute the same result)
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 ohi = make_float2(__shfl_xor_sync(0xffffffffu, hi[k].x, 16), __shfl_xor_sync(0xffffffffu, hi[k].y, 16));
    const float2 olo = make_float2(__shfl_xor_sync(0xffffffffu, lo[k].x, 16), __shfl_xor_sync(0xffffffffu, lo[k].y, 16));
    float2 s, e;
    two_sum2(hi[k], ohi, s, e);
    hi[k] = s;
    lo[k] = __fadd2_rn(__fadd2_rn(lo[k], olo), e);
  }
}

// True when the float-pair chunk sums are exact (see key_sum_partial), from
// the chunk's largest magnitude bits and (smallest nonzero magnitude bits - 1)
// per 16-bit half.
__device__ __forceinline__ bool key_sum_exact(uint32_t mx, uint32_t mn) {
  const uint32_t mxb = max(mx & 0xFFFFu, mx >> 16);
  const uint32_t mnb = min(mn & 0xFFFFu, mn >> 16) + 1u;  // 0x10000 when every value is zero
  if (mnb > 0x7FFFu) return true;
  int ef_min = static_cast<int>(mnb >> 7);
  if (ef_min == 0) ef_min = 1;  // subnormal bf16: last-bit weight 2^-133
  int ef_max = static_cast<int>(mxb >> 7);
  if (ef_max == 0) ef_max = 1;
  return ef_max - ef_min <= 36 - 7;  // E - L = (ef_max - 127) - (ef_min - 134)
}

// Two e4m3 codes: high byte = code(a), low byte = code(b).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(a), "f"(b));
  return r;
}

// Fast V codes of one token's 4 channels (4-channel lanes), low byte =
// channel 0: the codes of q * (1 - 2^-21) in cd and of q * (1 + 2^-21) in
// cu, q = fl(v * fl(1/s)). Rounding to e4m3 is monotone, and fl(v / s) lies
// within 2^-22 relative of q; so where the two agree, that is the code of
// fl(v / s), and where they differ the exact division must decide.
__device__ __forceinline__ void v_code_brackets(uint2 w, float2 r01, float2 r23, uint32_t& cd, uint32_t& cu) {
  const float2 q01 = __fmul2_rn(bf2(w.x), r01), q23 = __fmul2_rn(bf2(w.y), r23);
  const float2 dn = make_float2(kDn, kDn), up = make_float2(kUp, kUp);
  const float2 d01 = __fmul2_rn(q01, dn), u01 = __fmul2_rn(q01, up);
  const float2 d23 = __fmul2_rn(q23, dn), u23 = __fmul2_rn(q23, up);
  cd = e4m3x2(d01.y, d01.x) | (e4m3x2(d23.y, d23.x) << 16);
  cu = e4m3x2(u01.y, u01.x) | (e4m3x2(u23.y, u23.x) << 16);
}

// One byte to global memory with the streaming hint.
__device__ __forceinline__ void st_cs_u8(uint8_t* p, uint32_t v) {
  asm volatile("st.global.cs.u8 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Exact path of the V codes (out of line: rare per element, but with bf16
// inputs v / s_v = 448 v / vmax falls exactly on an e4m3 rounding midpoint
// for some channels, e.g. when s_v has few significant bits, so most warps
// meet it somewhere). `redo` flags the tokens of this lane whose fast
// brackets left a channel open (all: every kept channel is open, for scales
// below FLT_MIN). For each, the brackets are recomputed and only the open
// channels are divided exactly, each code stored again as one byte at
// vt_lane[c * S_pad + t] over the fast one this thread stored before (same
// thread, same address: the later store wins).
__device__ __noinline__ void v_codes_exact(const uint8_t* rows, int lane, uint32_t redo, bool all, float2 r01,
                                           float2 r23, float4 svs, uint32_t keep, uint8_t* vt_lane, int64_t S_pad) {
  const float sc[4] = {svs.x, svs.y, svs.z, svs.w};
  while (redo != 0u) {
    const int t = __ffs(redo) - 1;
    redo &= redo - 1u;
    const uint2 w = tok4(rows, t, lane);
    uint32_t cd, cu;
    v_code_brackets(w, r01, r23, cd, cu);
    const uint32_t open = (all ? 0xFFFFFFFFu : (cd ^ cu)) & keep;
    const float v[4] = {lo_bf16(w.x), hi_bf16(w.x), lo_bf16(w.y), hi_bf16(w.y)};
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if ((open >> (8 * c)) & 0xFFu) st_cs_u8(vt_lane + c * S_pad + t, e4m3x2(0.0f, __fdiv_rn(v[c], sc[c])) & 0xFFu);
  }
}

// Exact fp64 sums of one 32-token key chunk, by the two warps of a pair
// (sub 0 and 1, 16 rows each; rows: this warp's rows, read with 8-channel
// lanes; nv: its rows below S; nvc: the chunk's rows below S). The second
// half posts its float pairs and, per lane, the magnitude bounds of the
// lane's 8 channels in xk_*; the first half joins them, replaces the result
// by the left-to-right fp64 sums when the pair sums of a lane's channels may
// be inexact (judged on both halves' bounds for those channels), and writes
// the chunk's 128 sums to ks_chunk.
// `release` runs once the warp has stopped reading its rows.
template <typename Release>
__device__ __forceinline__ void key_chunk_sums(const uint8_t* rows, int nv, int nvc, int sub, int lane, int pair,
                                               float* xk_hi, float* xk_lo, uint32_t* xk_bits, double* ks_chunk,
                                               Release release) {
  float2 hi[4], lo[4];
  uint32_t mx, mn;
  if (nv == kHalfRows)
    key_sum_partial<true>(rows, kHalfRows, lane, hi, lo, mx, mn);
  else
    key_sum_partial<false>(rows, nv, lane, hi, lo, mx, mn);
  if (sub == 1) {
    if (lane < 16) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        xk_hi[8 * lane + 2 * k] = hi[k].x;
        xk_hi[8 * lane + 2 * k + 1] = hi[k].y;
        xk_lo[8 * lane + 2 * k] = lo[k].x;
        xk_lo[8 * lane + 2 * k + 1] = lo[k].y;
      }
    }
    if (lane < 16) {
      // the bounds of this lane's 8 channels (lanes l and l + 16 hold the same)
      xk_bits[lane] = mx;
      xk_bits[16 + lane] = mn;
    }
    pair_bar(pair);
    release();
    return;
  }
  pair_bar(pair);
  const int cb = 8 * (lane & 15);
  double sums[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float2 s, e;
    two_sum2(hi[k], make_float2(xk_hi[cb + 2 * k], xk_hi[cb + 2 * k + 1]), s, e);
    const float2 l = __fadd2_rn(__fadd2_rn(lo[k], make_float2(xk_lo[cb + 2 * k], xk_lo[cb + 2 * k + 1])), e);
    sums[2 * k] = __dadd_rn(static_cast<double>(s.x), static_cast<double>(l.x));
    sums[2 * k + 1] = __dadd_rn(static_cast<double>(s.y), static_cast<double>(l.y));
  }
  if (!key_sum_exact(__vmaxu2(mx, xk_bits[lane & 15]), __vminu2(mn, xk_bits[16 + (lane & 15)]))) {
    // this warp's rows are followed by the second half's in the tile
#pragma unroll 1
    for (int c = 0; c < 8; ++c) sums[c] = fp64_chunk_sum(rows, nvc, (lane & 15) * 16 + 2 * c);
  }
  release();
  if (lane < 16) {
#pragma unroll
    for (int c = 0; c < 8; ++c) ks_chunk[cb + c] = sums[c];
  }
}

// Max |v| of one warp's 16 V rows per channel, as bf16 magnitude bits (they
// order as integers): on return m4[k] holds channels (8l+2k, 8l+2k+1), l =
// lane & 15, in its low and high halves, over the rows of this half-warp
// (tokens of parity lane >> 4); the caller joins the two half-warps.
__device__ __forceinline__ void v_max_rows(const uint8_t* vr, int nv, int lane, uint32_t (&m4)[4]) {
  const int half = lane >> 4;
#pragma unroll
  for (int k = 0; k < 4; ++k) m4[k] = 0u;
  if (nv == kHalfRows) {
#pragma unroll
    for (int i = 0; i < kHalfRows / 4; ++i) {
      const uint4 wa = tok8(vr, 4 * i + half, lane), wb = tok8(vr, 4 * i + 2 + half, lane);
      m4[0] = __vimax3_u16x2(m4[0], wa.x & kAbs2, wb.x & kAbs2);
      m4[1] = __vimax3_u16x2(m4[1], wa.y & kAbs2, wb.y & kAbs2);
      m4[2] = __vimax3_u16x2(m4[2], wa.z & kAbs2, wb.z & kAbs2);
      m4[3] = __vimax3_u16x2(m4[3], wa.w & kAbs2, wb.w & kAbs2);
    }
  } else {
    for (int i = 0; i < kHalfRows / 2; ++i) {
      const int t = 2 * i + half;
      if (t < nv) {
        const uint4 w = tok8(vr, t, lane);
        m4[0] = __vmaxu2(m4[0], w.x & kAbs2);
        m4[1] = __vmaxu2(m4[1], w.y & kAbs2);
        m4[2] = __vmaxu2(m4[2], w.z & kAbs2);
        m4[3] = __vmaxu2(m4[3], w.w & kAbs2);
      }
    }
  }
}

// e4m3 codes of one warp's 16 V rows (4-channel lanes: channels 4*lane ..
// +4, scales svs), written transposed: the 16 tokens of the lane's channel c
// at vt_lane[c * S_pad] (nothing when vt_lane is null). Rows at or past nv
// get code 0. `release` runs once the warp has stopped reading its rows.
template <typename Release>
__device__ __forceinline__ void v_codes_rows(const uint8_t* rows, int nv, int lane, float4 svs, float4 rvs,
                                             uint8_t* vt_lane, int64_t S_pad, Release release) {
  const float sc[4] = {svs.x, svs.y, svs.z, svs.w};
  const float rv[4] = {rvs.x, rvs.y, rvs.z, rvs.w};  // fl(1/s) for s >= FLT_MIN, else 0
  uint32_t keep = 0u;
  bool fast = true;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (sc[c] > 0.0f) keep |= 0xFFu << (8 * c);
    fast = fast && (sc[c] >= FLT_MIN || sc[c] == 0.0f);  // zero channels are masked to code 0
  }
  const float2 r01 = make_float2(rv[0], rv[1]), r23 = make_float2(rv[2], rv[3]);
  uint32_t a[kHalfRows];  // a[t]: the 4 channels' codes of token t
  uint32_t redo = 0u;     // bit t: a channel of token t needs the exact division
#pragma unroll
  for (int t = 0; t < kHalfRows; ++t) {
    a[t] = 0u;
    if (nv == kHalfRows || t < nv) {
      uint32_t cd, cu;
      v_code_brackets(tok4(rows, t, lane), r01, r23, cd, cu);
      if (!(cd == cu && fast)) redo |= 1u << t;
      a[t] = cd & keep;
    }
  }
  if (redo == 0u) release();
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    // 4x4 byte transposes: tokens 4j..4j+3 of channel 4*lane+c
    uint32_t cw[4];
#pragma unroll
    for (int j = 0; j < kHalfRows / 4; ++j) {
      const uint32_t lo01 = __byte_perm(a[4 * j], a[4 * j + 1], (c & 2) ? 0x7362 : 0x5140);
      const uint32_t lo23 = __byte_perm(a[4 * j + 2], a[4 * j + 3], (c & 2) ? 0x7362 : 0x5140);
      cw[j] = __byte_perm(lo01, lo23, (c & 1) ? 0x7632 : 0x5410);
    }
    if (vt_lane) __stcs(reinterpret_cast<uint4*>(vt_lane + c * S_pad), make_uint4(cw[0], cw[1], cw[2], cw[3]));
  }
  if (redo != 0u) {
    if (vt_lane) v_codes_exact(rows, lane, redo, !fast, r01, r23, svs, keep, vt_lane, S_pad);
    release();
  }
}

// Pairwise tree (padded with +0.0 to a power of two) over `n` group sums
// starting at p, stride 128 doubles, evaluated streaming: stack[l] holds a
// finished subtree of 2^l leaves. Aligned blocks of 16 leaves are loaded
// together (16 loads in flight) and reduced as one 16-leaf subtree, which is
// what pushing the 16 leaves one by one would build. The sums are never
// -0.0, so padding with +0.0 changes nothing.
__device__ __forceinline__ double tree_sum(const double* p, int64_t n) {
  double stack[40];
  int64_t gi = 0;
  for (; gi + 16 <= n; gi += 16) {
    double v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = __ldcg(p + (gi + k) * kHeadDim);
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

// Max of `n` group maxima starting at p, stride 128 floats, 16 loads in flight.
__device__ __forceinline__ float group_max(const float* p, int64_t n) {
  float m = 0.0f;
  int64_t gi = 0;
  for (; gi + 16 <= n; gi += 16) {
    float v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = __ldcg(p + (gi + k) * kHeadDim);
#pragma unroll
    for (int k = 0; k < 16; ++k) m = fmaxf(m, v[k]);
  }
  for (; gi < n; ++gi) m = fmaxf(m, __ldcg(p + gi * kHeadDim));
  return m;
}

// Barrier of one compute team (named barrier 1 + team, 256 threads).
__device__ __forceinline__ void team_bar(int team) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "n"(kTeamThreads) : "memory");
}

struct Ctx {
  uint32_t bar0;
  volatile int* abort_flag;
  int* dev_err;
  __device__ uint32_t full(int s) const { return bar0 + 8u * static_cast<uint32_t>(s); }
  __device__ uint32_t empty(int s) const { return bar0 + 8u * static_cast<uint32_t>(kStages + s); }
  __device__ uint32_t evt_full(int e) const { return bar0 + 8u * static_cast<uint32_t>(2 * kStages + e); }
  __device__ uint32_t evt_empty(int e) const { return bar0 + 8u * static_cast<uint32_t>(2 * kStages + kEvents + e); }
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


// Finish head bh with the 256 threads of team 1: the pairwise tree over its
// group key sums gives the key mean, the max over its group maxima the V
// scales (and their correctly rounded reciprocals, which the codes items'
// V codes multiply by, computed once here instead of once per item and warp);
// then the head is published as ready. Every group of the head has
// been counted (by the producer of this CTA, which saw the count complete).
// With kPair the mean and scales go to the two real heads' places and, for
// the codes items, to the virtual head's row of hstat_v.
template <bool kPair>
__device__ __forceinline__ void finish_head(const Params& prm, int64_t bh, int tt, double* fin_right,
                                            float* fin_vmax) {
  const int64_t G = prm.G;
  const int c = tt & (kHeadDim - 1), hf = tt >> 7;
  int64_t P = 1;
  while (P < G) P *= 2;
  const int64_t lo = hf == 0 ? 0 : (P == 1 ? 1 : P / 2);
  const int64_t hi_end = hf == 0 ? (P == 1 ? 1 : P / 2) : P;
  const int64_t n = max(int64_t(0), min(G, hi_end) - lo);
  double t = 0.0;
  if (prm.smooth_k && n > 0) t = tree_sum(prm.ksum + (bh * G + lo) * kHeadDim + c, n);
  const float vmx = n > 0 ? group_max(prm.vmax + (bh * G + lo) * kHeadDim + c, n) : 0.0f;
  if (hf == 1) {
    fin_right[c] = t;
    fin_vmax[c] = vmx;
  }
  team_bar(1);
  if (hf == 0) {
    float mu = 0.0f;
    if (prm.smooth_k) {
      const double total = P > 1 ? __dadd_rn(t, fin_right[c]) : t;
      mu = __double2float_rn(__ddiv_rn(total, static_cast<double>(prm.S)));
    }
    const float vs = __fdiv_rn(fmaxf(vmx, fin_vmax[c]), kE4M3Max);
    const int64_t head = out_head<kPair>(prm, bh, c / kOutDim<kPair>);
    if (head >= 0) {
      prm.out.k_mean[head * kOutDim<kPair> + (c & (kOutDim<kPair> - 1))] = mu;
      prm.out.v_scale[head * kOutDim<kPair> + (c & (kOutDim<kPair> - 1))] = vs;
    }
    if (kPair) {
      prm.hstat_v[bh * 2 * kHeadDim + c] = mu;
      prm.hstat_v[bh * 2 * kHeadDim + kHeadDim + c] = vs;
    }
    prm.vrcp[bh * kHeadDim + c] = vs >= FLT_MIN ? __frcp_rn(vs) : 0.0f;
  }
  team_bar(1);
  if (tt == 0) {
    // release: the mean and scales written by the team (ordered by the
    // barrier) are visible to whoever acquires the flag
    __threadfence();
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(prm.ready + bh), "r"(1u) : "memory");
  }
}

template <bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    prologue_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const Params prm, int3 s_axis) {
  extern __shared__ uint8_t smem_raw[];
  // aligned by pointer arithmetic on the shared array (an integer round trip
  // would hide the address space and turn every tile read into a generic load)
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  // the statistics of the group a team is working on (either team can be)
  __shared__ double ks[kTeams][kChunks][kHeadDim];            // exact chunk sums
  __shared__ uint32_t vm[kTeams][kWarps][kHeadDim / 2];       // per-warp max |v| bits, channel pairs
  __shared__ float xk_hi[kTeams][kChunks][kHeadDim], xk_lo[kTeams][kChunks][kHeadDim];  // second-half key sums
  __shared__ uint32_t xk_bits[kTeams][kChunks][32];           // second-half magnitude bounds per lane
  __shared__ float xa[2][kTeams * kWarps / 2][2][2];  // amax of each half block (per head of a pair), two parities
  __shared__ float fin_vmax[kHeadDim];
  __shared__ double fin_right[kHeadDim];
  // the next kernel of the stream (the attention kernel, launched as a
  // programmatic dependent) may be scheduled once every CTA of this grid has
  // started; it waits for this grid to end before it reads anything
  tc::griddep_launch_dependents();
  const uint32_t sbase = tc::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int64_t* meta_item = reinterpret_cast<int64_t*>(smem + kOffMeta);             // [kStages]
  int64_t* meta_bh = reinterpret_cast<int64_t*>(smem + kOffMeta + kStages * 8); // [kStages]
  // [kStages]: the tensor in the low 32 bits, the item's phase in bit 32, its
  // group above (the producer decodes each item once: 64-bit division by the
  // group count in every consumer thread cost several percent of the kernel)
  int64_t* meta_tg = reinterpret_cast<int64_t*>(smem + kOffMeta + kStages * 16);
  volatile int64_t* evt_bh = reinterpret_cast<volatile int64_t*>(smem + kOffEvt);  // [kEvents]
  int64_t* fin_q = reinterpret_cast<int64_t*>(smem + kOffFinQ);                 // [kFinCap]
  const float* hstat = reinterpret_cast<const float*>(smem + kOffHstat);        // [kStages][256]
  Ctx cx;
  cx.bar0 = sbase + kOffBar;
  cx.abort_flag = reinterpret_cast<volatile int*>(smem + kOffFlags);
  cx.dev_err = prm.dev_err;
  if (threadIdx.x == 0) {
    *cx.abort_flag = 0;
    *reinterpret_cast<volatile uint32_t*>(smem + kOffFlags + 4) = 0u;  // finish-queue tail
    *reinterpret_cast<volatile uint32_t*>(smem + kOffFlags + 8) = 0u;  // groups counted
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(cx.full(s), 1);
      tc::mbar_init(cx.empty(s), kTeams * kTeamThreads);  // both teams release every stage
    }
    for (int e = 0; e < kEvents; ++e) {
      tc::mbar_init(cx.evt_full(e), 1);
      tc::mbar_init(cx.evt_empty(e), 1);
    }
    tc::fence_mbar_init();
  }
  __syncthreads();

  volatile uint32_t* fin_tail_p = reinterpret_cast<volatile uint32_t*>(smem + kOffFlags + 4);  // finish queue tail
  volatile uint32_t* counted_p = reinterpret_cast<volatile uint32_t*>(smem + kOffFlags + 8);   // groups counted

  if (warp == kTeams * kWarps + 1) {
    // --------------------------------------------------------------- counter --
    // Counts the groups the teams report done. The fence and atomic of the count
    // stay off the compute warps and off the producer (a fence there would
    // also wait for its tile loads). When a head's last group is counted the
    // head goes into the finish queue; the producer turns it into a finish
    // marker for team 1. A report with head -1 ends the loop.
    if (lane == 0) {
      uint32_t ev = 0, tail = 0;
      while (true) {
        const uint32_t e = ev % kEvents;
        if (!wait_bar(cx, cx.evt_full(e), (ev / kEvents) & 1u)) break;
        const int64_t h = evt_bh[e];
        tc::mbar_arrive(cx.evt_empty(e));
        ++ev;
        if (h < 0) break;
        // the reporting team's slot writes are ordered before the report (barrier, then
        // release on the mbarrier); the fence makes them visible to the GPU
        // before the count
        __threadfence();
        if (atomicAdd(prm.done + h, 1u) == static_cast<unsigned>(prm.G - 1)) {
          __threadfence();  // acquire the other CTAs' group results
          // the queue never holds more than the groups in flight in this CTA
          // (tiles in the ring plus reports), far below its capacity
          fin_q[tail % kFinCap] = h;
          __threadfence_block();
          *fin_tail_p = ++tail;
        }
        __threadfence_block();
        *counted_p = ev;
      }
    }
    return;
  }

  if (warp == kTeams * kWarps) {
    // -------------------------------------------------------------- producer --
    // Claims items in order and loads their tiles into the ring. Heads the
    // counter warp has finished counting become finish markers, pushed at
    // item boundaries (between the tiles of an item the consumers expect no
    // marker); the codes items of a head enter the ring only after team 1
    // has finished and published it.
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_k);
      tc::prefetch_tmap(&tm_v);
      // Q is read once; K and V are read by the stats item and again by the
      // codes item, so they are marked to stay in L2 where it has room
      const uint64_t pol_first = tc::policy_evict_first(), pol_last = tc::policy_evict_last();
      uint32_t cnt = 0, stats_pushed = 0, fin_head = 0;
      int pending[kStages];
      for (int s = 0; s < kStages; ++s) pending[s] = -1;
      bool ok = true;
      auto fins_waiting = [&]() { return *fin_tail_p != fin_head; };
      // push one finish marker into stage st (the stage is free)
      auto push_finish = [&](uint32_t st) {
        __threadfence_block();  // the queue entry after its tail
        meta_item[st] = fin_q[fin_head++ % kFinCap];
        meta_tg[st] = kFinish;
        tc::mbar_arrive(cx.full(st));
        ++cnt;
      };
      // queued finish markers go into free stages without waiting
      auto push_finish_markers = [&]() {
        while (fins_waiting() && tc::mbar_try_wait(cx.empty(cnt % kStages), ((cnt / kStages) & 1u) ^ 1u))
          push_finish(cnt % kStages);
      };
      // the next ring position, once both teams have released it
      auto next_stage = [&](uint32_t& st, uint32_t& ph) -> bool {
        st = cnt % kStages;
        ph = (cnt / kStages) & 1u;
        return wait_bar(cx, cx.empty(st), ph ^ 1u);
      };
      // bounded wait for a condition
      auto wait_until = [&](auto cond) -> bool {
        uint64_t t0 = 0;
        for (uint32_t it = 0;; ++it) {
          if (cond()) return true;
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
            __nanosleep(32);
          }
        }
      };
      // the next claim is issued one item ahead so its latency overlaps the
      // waits for free stages (items are still processed in claim order)
      unsigned next = atomicAdd(prm.next_item, 1u);
      bool claimed_end = false;
      while (ok) {
        uint32_t st, ph;
        if (fins_waiting()) {
          if (!(ok = next_stage(st, ph))) break;
          push_finish(st);
          continue;
        }
        if (claimed_end) {
          // every stats item pushed is counted, and its head finished if it
          // was the last group, before the end marker
          if (*counted_p == stats_pushed) {
            if (fins_waiting()) continue;
            if (!(ok = next_stage(st, ph))) break;
            meta_item[st] = -1;
            meta_tg[st] = kEnd;
            tc::mbar_arrive(cx.full(st));
            break;
          }
          ok = wait_until([&] { return *counted_p == stats_pushed || fins_waiting(); });
          continue;
        }
        const int64_t item = static_cast<int64_t>(next);
        if (item >= prm.total) {
          claimed_end = true;
          continue;
        }
        next = atomicAdd(prm.next_item, 1u);
        const Item it = decode_item(item, prm.NH, prm.G, prm.lag);
        int tensors[3], nt = 0;
        if (it.phase == 0) {
          tensors[nt++] = kTensorQ;
          if (prm.smooth_k) tensors[nt++] = kTensorK;
          tensors[nt++] = kTensorV;
        } else {
          // a codes item needs the head's key mean and V scales: its tiles
          // enter the ring only once they are published. Meanwhile queued
          // finish markers must still reach team 1 (the head waited for may
          // be one of them)
          const unsigned* flag = prm.ready + it.bh;
          if (!(ok = wait_until([&] {
                  push_finish_markers();
                  unsigned v;
                  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
                  return v != 0u;
                })))
            break;
          tc::fence_proxy_async_global();  // the bulk copies below read what the flag published
          tensors[nt++] = kTensorK;
          tensors[nt++] = kTensorV;
        }
        // the head coordinate: of the real head pair 2hp, 2hp + 1 in head-pair mode
        const int32_t h = static_cast<int32_t>((kPair ? 2 : 1) * (it.bh % prm.H)), b = static_cast<int32_t>(it.bh / prm.H);
        const int32_t s0 = static_cast<int32_t>(it.g * kItemTokens);
        for (int n = 0; n < nt && ok; ++n) {
          if (!(ok = next_stage(st, ph))) break;
          meta_item[st] = item;
          meta_bh[st] = it.bh;
          meta_tg[st] = static_cast<int64_t>(tensors[n]) | (static_cast<int64_t>(it.phase) << 32) | (it.g << 33);
          const bool with_stats = it.phase == 1 && n == 0;  // the codes item's head statistics
          tc::mbar_arrive_expect_tx(cx.full(st), kTileBytes + (with_stats ? kHstatBytes : 0u));
          const CUtensorMap* tm = tensors[n] == kTensorQ ? &tm_q : (tensors[n] == kTensorK ? &tm_k : &tm_v);
          // map dims: (channel, s, h, b) or (channel, h, s, b) by stride order
          const int ax = tensors[n] == kTensorQ ? s_axis.x : (tensors[n] == kTensorK ? s_axis.y : s_axis.z);
          const uint64_t pol = (it.phase == 0 && tensors[n] != kTensorQ) ? pol_last : pol_first;
          if (ax == 1)
            tc::tma_load_4d_hint(sbase + st * kTileBytes, tm, 0, s0, h, b, cx.full(st), pol);
          else
            tc::tma_load_4d_hint(sbase + st * kTileBytes, tm, 0, h, s0, b, cx.full(st), pol);
          if (with_stats) {
            const uint32_t hs = sbase + kOffHstat + st * kHstatBytes;
            const float* km = kPair ? prm.hstat_v + it.bh * 2 * kHeadDim : prm.out.k_mean + it.bh * kHeadDim;
            const float* vsc = kPair ? prm.hstat_v + it.bh * 2 * kHeadDim + kHeadDim : prm.out.v_scale + it.bh * kHeadDim;
            tc::bulk_load(hs, km, kHeadDim * 4, cx.full(st));
            tc::bulk_load(hs + kHeadDim * 4, vsc, kHeadDim * 4, cx.full(st));
            tc::bulk_load(hs + 2 * kHeadDim * 4, prm.vrcp + it.bh * kHeadDim, kHeadDim * 4, cx.full(st));
          }
          pending[st] = static_cast<int>(ph);
          ++cnt;
        }
        if (ok && it.phase == 0) ++stats_pushed;
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
  // Two teams of 8 warps work on different tiles of the same item. Stats
  // item: role 0 the Q tile; role 1 the K sums, the V maxima and the group's
  // results. Codes item: role 1 the K tile, role 0 the V tile. The teams swap
  // roles from one item of a kind to the next (the two roles' work differs by
  // about a quarter, and a team can run ahead of the other only as far as the
  // ring allows; measured 4% faster than fixed roles at B1 H28 S16384).
  // Finish markers always go to team 1. Warps 2c and 2c+1 of a team take the
  // two halves (16 tokens each) of chunk c. Both
  // teams wait on every stage in ring order, so a parity wait never meets a
  // barrier two phases behind; a team releases the stages it does not use as
  // soon as they are full, and a stage is refilled once both have released it.
  const int team = warp / kWarps, tw = warp % kWarps, tt = threadIdx.x % kTeamThreads;
  const int chunk = tw >> 1, sub = tw & 1, pair = warp >> 1;
  const int64_t S = prm.S, S_pad = prm.S_pad, G = prm.G;
  const int64_t nblk = S_pad / kQKBlock;
  const uint32_t row_off = static_cast<uint32_t>(tw * kHalfRows * 256);
  uint32_t cnt = 0, n_stats = 0, n_codes = 0;  // ring position; items of each kind seen
  int xpar = 0;  // slot parity of the amax exchange (both warps of a pair flip together)
  // wait for ring position c to be full, then release it unused
  auto pass = [&](uint32_t c) -> bool {
    if (!wait_bar(cx, cx.full(c % kStages), (c / kStages) & 1u)) return false;
    tc::mbar_arrive(cx.empty(c % kStages));
    return true;
  };
  auto stage_rows = [&](uint32_t c) { return smem + (c % kStages) * kTileBytes + row_off; };
  while (true) {
    const uint32_t st = cnt % kStages;
    if (!wait_bar(cx, cx.full(st), (cnt / kStages) & 1u)) break;
    const int64_t item = meta_item[st];
    const int64_t tg = meta_tg[st];
    const int tensor = static_cast<int>(tg & 0xFFFFFFFF);
    if (tensor == kEnd) {
      if (team == 1 && tt == 0) {
        // tell the counter warp that no report follows
        const uint32_t e = n_stats % kEvents;
        if (wait_bar(cx, cx.evt_empty(e), ((n_stats / kEvents) & 1u) ^ 1u)) {
          evt_bh[e] = -1;
          tc::mbar_arrive(cx.evt_full(e));
        }
      }
      break;
    }
    if (tensor == kFinish) {
      tc::mbar_arrive(cx.empty(st));  // the marker carries no data
      if (team == 1) finish_head<kPair>(prm, item, tt, fin_right, fin_vmax);
      cnt += 1;
      continue;
    }
    Item it;
    it.phase = static_cast<int>((tg >> 32) & 1);
    it.bh = meta_bh[st];
    it.g = tg >> 33;
    const uint32_t n_stages = it.phase == 0 ? (prm.smooth_k ? 3u : 2u) : 2u;
    // the two teams swap roles from one item of a kind to the next, so that
    // neither waits for the other's heavier tile (role 0: the Q tile of a
    // stats item, the V tile of a codes item; role 1: the K and V tiles of a
    // stats item, the K tile of a codes item)
    const uint32_t kind_idx = it.phase == 0 ? n_stats++ : n_codes++;
    const int role = team ^ static_cast<int>(kind_idx & 1u);
    const int64_t bh = it.bh;
    const int64_t s0c = it.g * kItemTokens + chunk * kQKBlock;  // first token of the chunk
    const int64_t s0 = s0c + sub * kHalfRows;                    // first token of this warp
    const int nv = valid_rows(S, s0, kHalfRows);  // this warp's rows below S (every row is below S_pad)
    volatile float* xm = &xa[xpar][pair][sub][0];
    volatile float* xo = &xa[xpar][pair][sub ^ 1][0];
    bool ok = true;

    if (it.phase == 0 && role == 0) {
      // Q codes and scale
      const float2 nz[4] = {};
      int8_t* qc;
      uint16_t* q16;
      const int64_t qh = lane_codes<kPair>(prm, prm.write_int8 ? prm.out.q_codes : nullptr, prm.out.q16, bh, s0, lane,
                                           qc, q16);
      const uint8_t* rows = stage_rows(cnt);
      const float s = nv == kHalfRows ? quantize_half_block<false, true, kPair>(rows, nz, kHalfRows, qc, q16,
                                                                                  kOutDim<kPair>, lane, xm, xo, pair)
                                      : quantize_half_block<false, false, kPair>(rows, nz, nv, qc, q16,
                                                                                   kOutDim<kPair>, lane, xm, xo, pair);
      xpar ^= 1;
      store_block_scale<kPair>(prm.out.q_scale, qh, nblk, s0c / kQKBlock, s, lane, sub);
      tc::mbar_arrive(cx.empty(st));
      for (uint32_t c = 1; c < n_stages && ok; ++c) ok = pass(cnt + c);
      if (!ok) break;
    } else if (it.phase == 0) {
      tc::mbar_arrive(cx.empty(st));  // the Q tile is team 0's
      uint32_t c2 = cnt + 1;
      if (!wait_bar(cx, cx.full(c2 % kStages), (c2 / kStages) & 1u)) break;
      if (prm.smooth_k) {
        // K tile: exact fp64 chunk sums, the second half's partial sums
        // joined into the first half's
        const uint32_t ks_stage = c2 % kStages;
        key_chunk_sums(stage_rows(c2), nv, valid_rows(S, s0c, kQKBlock), sub, lane, pair, xk_hi[team][chunk],
                       xk_lo[team][chunk], xk_bits[team][chunk], ks[team][chunk],
                       [&]() { tc::mbar_arrive(cx.empty(ks_stage)); });
        ++c2;
        if (!wait_bar(cx, cx.full(c2 % kStages), (c2 / kStages) & 1u)) break;
      }
      // V tile: max |v| per channel (bf16 magnitudes compare as integers)
      uint32_t m4[4];  // channel pairs (8l, 8l+1) .. (8l+6, 8l+7)
      v_max_rows(stage_rows(c2), nv, lane, m4);
      tc::mbar_arrive(cx.empty(c2 % kStages));
#pragma unroll
      for (int k = 0; k < 4; ++k) m4[k] = __vmaxu2(m4[k], __shfl_xor_sync(0xffffffffu, m4[k], 16));
      if (lane < 16) {
#pragma unroll
        for (int k = 0; k < 4; ++k) vm[team][tw][4 * lane + k] = m4[k];
      }
      team_bar(team);
      if (tt < kHeadDim) {
        // the group's results: levels 1 and 2 of the pairwise tree over its 4
        // chunk sums, and its max |v| per channel
        const int c = tt;
        const int64_t slot = (bh * G + it.g) * kHeadDim + c;
        if (prm.smooth_k)
          prm.ksum[slot] =
              __dadd_rn(__dadd_rn(ks[team][0][c], ks[team][1][c]), __dadd_rn(ks[team][2][c], ks[team][3][c]));
        uint32_t mb = 0u;
#pragma unroll
        for (int i = 0; i < kWarps; ++i) {
          const uint32_t pr = vm[team][i][c >> 1];
          mb = max(mb, (c & 1) ? (pr >> 16) : (pr & 0xFFFFu));
        }
        prm.vmax[slot] = __uint_as_float(mb << 16);
      }
      team_bar(team);
      if (tt == 0) {
        // report the group to the counter warp; the report of the k-th
        // stats item goes into slot k % kEvents, so each slot has one writer
        // (kEvents is even and the roles alternate) and the counter warp
        // reads the reports in ring order
        const uint32_t e = kind_idx % kEvents;
        if (wait_bar(cx, cx.evt_empty(e), ((kind_idx / kEvents) & 1u) ^ 1u)) {
          evt_bh[e] = bh;
          tc::mbar_arrive(cx.evt_full(e));
        }
      }
    } else if (role == 0) {
      // codes item, team 0: V codes of this warp's 16 tokens, transposed to
      // [channel][token] (4-channel lanes); the V scales come with the K tile
      const float4 svs = *reinterpret_cast<const float4*>(hstat + st * (kHstatBytes / 4) + kHeadDim + 4 * lane);
      const float4 rvs =
          *reinterpret_cast<const float4*>(hstat + st * (kHstatBytes / 4) + 2 * kHeadDim + 4 * lane);
      tc::mbar_arrive(cx.empty(st));  // the K tile is team 1's
      const uint32_t c2 = cnt + 1;
      if (!wait_bar(cx, cx.full(c2 % kStages), (c2 / kStages) & 1u)) break;
      const uint32_t v_stage = c2 % kStages;
      v_codes_rows(stage_rows(c2), nv, lane, svs, rvs, lane_vt<kPair>(prm, bh, s0, lane), S_pad,
                   [&]() { tc::mbar_arrive(cx.empty(v_stage)); });
    } else {
      // codes item, team 1: K codes of k - mean; the key mean comes with the
      // K tile
      int8_t* kc;
      uint16_t* k16;
      const int64_t kh = lane_codes<kPair>(prm, prm.write_int8 ? prm.out.k_codes : nullptr, prm.out.k16, bh, s0, lane,
                                           kc, k16);
      const uint8_t* rows = stage_rows(cnt);
      constexpr int od = kOutDim<kPair>;
      float skv;
      if (prm.smooth_k) {
        const float4* mp = reinterpret_cast<const float4*>(hstat + st * (kHstatBytes / 4) + 8 * (lane & 15));
        const float4 ma = mp[0], mb = mp[1];
        const float2 nmu[4] = {make_float2(-ma.x, -ma.y), make_float2(-ma.z, -ma.w), make_float2(-mb.x, -mb.y),
                               make_float2(-mb.z, -mb.w)};
        skv = nv == kHalfRows
                  ? quantize_half_block<true, true, kPair>(rows, nmu, kHalfRows, kc, k16, od, lane, xm, xo, pair)
                  : quantize_half_block<true, false, kPair>(rows, nmu, nv, kc, k16, od, lane, xm, xo, pair);
      } else {
        const float2 nz[4] = {};
        skv = nv == kHalfRows
                  ? quantize_half_block<false, true, kPair>(rows, nz, kHalfRows, kc, k16, od, lane, xm, xo, pair)
                  : quantize_half_block<false, false, kPair>(rows, nz, nv, kc, k16, od, lane, xm, xo, pair);
      }
      xpar ^= 1;
      store_block_scale<kPair>(prm.out.k_scale, kh, nblk, s0c / kQKBlock, skv, lane, sub);
      tc::mbar_arrive(cx.empty(st));
      if (!pass(cnt + 1)) break;
    }
    cnt += n_stages;
  }
}

// ---------------------------------------------------------------------------
// Short sequences: one cluster of G = ceil(S / 128) <= kShortMaxGroups CTAs
// per (batch, head). CTA g holds group g (tokens 128g .. 128g+127) of the
// head's Q, K and V in shared memory, one TMA copy each, and writes every
// output of that group. Two teams of 8 warps split the work so that the
// chain each warp runs stays short (short calls wait for it): team 0 takes
// the V maxima, codes Q while the group results are exchanged, then codes V;
// team 1 sums K, exchanges the results, finishes the head's statistics and
// codes K. Each CTA keeps its group's key sums and V maxima in its own
// shared memory; after a cluster barrier every CTA reads all G of them over
// distributed shared memory, and a last cluster barrier, waited on at exit,
// keeps each CTA resident until the others have read it. So the prologue is
// a single launch with no global counters and no scratch, and each input byte
// is read once. The shared memory (about 110 KB) and the 64 registers a
// thread leave room for two CTAs per SM, which lets every cluster of 8 CTAs
// of a 16-head problem run at once (with one CTA per SM the GPU holds 15 of
// them, and the 16th ran in a second wave). The arithmetic is the
// persistent kernel's (the same per-warp helpers; the same pairwise tree
// over the group sums, padded with +0.0 to a power of two, where padding
// changes nothing), so the outputs are identical.
constexpr int kShortMaxGroups = 8;                 // the portable cluster size
constexpr int kShortThreads = kTeams * kTeamThreads;
constexpr uint32_t kShortSmemBytes = 3 * kTileBytes + 128;  // Q, K, V tiles + alignment slack

template <bool kPair>
__global__ void __launch_bounds__(kShortThreads, 2)
    prologue_short_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const Params prm, int3 s_axis) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((128u - (tc::smem_u32(smem_raw) & 127u)) & 127u);
  __shared__ double ks[kChunks][kHeadDim];       // exact chunk sums of this group
  __shared__ uint32_t vm[kWarps][kHeadDim / 2];  // per-warp max |v| bits, channel pairs
  __shared__ float xk_hi[kChunks][kHeadDim], xk_lo[kChunks][kHeadDim];  // second-half key sums
  __shared__ uint32_t xk_bits[kChunks][32];      // second-half magnitude bounds per lane
  __shared__ float xa[kTeams * kWarps / 2][2][2];  // block amax exchange of each warp pair (per head of a pair)
  __shared__ double g_sum[kHeadDim];    // this group's key sums (read by the whole cluster)
  __shared__ uint32_t g_max[kHeadDim];  // this group's max |v| bits
  __shared__ __align__(16) float h_mean[kHeadDim];
  __shared__ __align__(16) float h_vscale[kHeadDim];
  __shared__ __align__(16) float h_vrcp[kHeadDim];
  __shared__ __align__(8) uint64_t bars[3];      // Q, K, V tile full
  __shared__ int abort_flag;

  // the next kernel of the stream (the attention kernel, launched as a
  // programmatic dependent) may be scheduled now; it waits for this grid
  tc::griddep_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tt = threadIdx.x;
  const int64_t G = prm.G, S = prm.S, S_pad = prm.S_pad, nblk = S_pad / kQKBlock;
  const int g = static_cast<int>(tc::cluster_ctarank());
  const int64_t bh = static_cast<int64_t>(blockIdx.x) / G;
  const int64_t b = bh / prm.H, h = bh % prm.H;
  const uint32_t sbase = tc::smem_u32(smem);
  Ctx cx;
  cx.bar0 = tc::smem_u32(bars);
  cx.abort_flag = &abort_flag;
  cx.dev_err = prm.dev_err;
  if (tt == 0) {
    abort_flag = 0;
    for (int n = 0; n < 3; ++n) tc::mbar_init(cx.full(n), 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  // first half of the barrier that makes sure every CTA of the cluster runs
  // before any of them stores into another's shared memory
  tc::cluster_arrive_relaxed();
  const int64_t s_group = static_cast<int64_t>(g) * kItemTokens;
  if (tt == 0) {
    const uint64_t pol = tc::policy_evict_first();  // every tile is read once
    const CUtensorMap* maps[3] = {&tm_q, &tm_k, &tm_v};
    const int axes[3] = {s_axis.x, s_axis.y, s_axis.z};
    const int32_t sc = static_cast<int32_t>(s_group), hc = static_cast<int32_t>((kPair ? 2 : 1) * h),
                  bc = static_cast<int32_t>(b);
#pragma unroll
    for (int n = 0; n < 3; ++n) {
      tc::mbar_arrive_expect_tx(cx.full(n), kTileBytes);
      if (axes[n] == 1)
        tc::tma_load_4d_hint(sbase + n * kTileBytes, maps[n], 0, sc, hc, bc, cx.full(n), pol);
      else
        tc::tma_load_4d_hint(sbase + n * kTileBytes, maps[n], 0, hc, sc, bc, cx.full(n), pol);
    }
  }

  // In each team warps 2c and 2c+1 take the two halves (16 tokens each) of
  // chunk c. A failed wait is recorded (error word) but changes no control
  // flow: every thread reaches every barrier below, the cluster's included.
  // Named barriers: 1, team 0's V maxima to team 1 (team 0 arrives, team 1
  // waits); 2, the head's scales from team 1 to team 0; 11, within team 1;
  // 3..10, the warp pairs.
  const int team = warp / kWarps, tw = warp % kWarps, chunk = tw >> 1, sub = tw & 1, pair = warp >> 1;
  const int64_t s0c = s_group + chunk * kQKBlock, s0 = s0c + sub * kHalfRows;
  const int nv = valid_rows(S, s0, kHalfRows);
  const uint32_t row_off = static_cast<uint32_t>(tw * kHalfRows * 256);
  const uint8_t* q_rows = smem + row_off;
  const uint8_t* k_rows = smem + kTileBytes + row_off;
  const uint8_t* v_rows = smem + 2 * kTileBytes + row_off;
  bool ok = true;
  if (team == 0) {
    // the group's max |v| per channel, handed to team 1
    ok = wait_bar(cx, cx.full(2), 0);
    uint32_t m4[4];
    v_max_rows(v_rows, nv, lane, m4);
#pragma unroll
    for (int k = 0; k < 4; ++k) m4[k] = __vmaxu2(m4[k], __shfl_xor_sync(0xffffffffu, m4[k], 16));
    if (lane < 16) {
#pragma unroll
      for (int k = 0; k < 4; ++k) vm[tw][4 * lane + k] = m4[k];
    }
    asm volatile("bar.arrive 1, %0;" ::"n"(kShortThreads) : "memory");
    // team 0 stores nothing into other CTAs: it passes the cluster's
    // barriers at once and codes Q while the group results are exchanged
    tc::cluster_wait_acquire();
    tc::cluster_arrive_relaxed();
    ok = wait_bar(cx, cx.full(0), 0) && ok;
    const float2 nz[4] = {};
    int8_t* qc;
    uint16_t* q16;
    const int64_t qh =
        lane_codes<kPair>(prm, prm.write_int8 ? prm.out.q_codes : nullptr, prm.out.q16, bh, s0, lane, qc, q16);
    constexpr int od = kOutDim<kPair>;
    const float s = nv == kHalfRows
                        ? quantize_half_block<false, true, kPair>(q_rows, nz, kHalfRows, qc, q16, od, lane,
                                                                  &xa[pair][sub][0], &xa[pair][sub ^ 1][0], pair)
                        : quantize_half_block<false, false, kPair>(q_rows, nz, nv, qc, q16, od, lane,
                                                                   &xa[pair][sub][0], &xa[pair][sub ^ 1][0], pair);
    store_block_scale<kPair>(prm.out.q_scale, qh, nblk, s0c / kQKBlock, s, lane, sub);
    tc::cluster_wait_acquire();
    tc::cluster_arrive_relaxed();  // team 0 reads no other CTA's shared memory
    asm volatile("bar.sync 2, %0;" ::"n"(kShortThreads) : "memory");  // the V scales are in h_vscale
    // V codes, transposed (4-channel lanes)
    v_codes_rows(v_rows, nv, lane, *reinterpret_cast<const float4*>(h_vscale + 4 * lane),
                 *reinterpret_cast<const float4*>(h_vrcp + 4 * lane), lane_vt<kPair>(prm, bh, s0, lane), S_pad,
                 [] {});
  } else {
    // the group's exact key sums
    ok = wait_bar(cx, cx.full(1), 0);
    if (prm.smooth_k)
      key_chunk_sums(k_rows, nv, valid_rows(S, s0c, kQKBlock), sub, lane, pair, xk_hi[chunk], xk_lo[chunk],
                     xk_bits[chunk], ks[chunk], [] {});
    asm volatile("bar.sync 1, %0;" ::"n"(kShortThreads) : "memory");  // team 0's V maxima are in vm
    tc::cluster_wait_acquire();  // every CTA of the cluster has started
    const int c = tt - kTeamThreads;
    if (c < kHeadDim) {
      // the group's results: levels 1 and 2 of the pairwise tree over its 4
      // chunk sums, and its max |v| per channel, kept here for the cluster
      const double gs =
          prm.smooth_k ? __dadd_rn(__dadd_rn(ks[0][c], ks[1][c]), __dadd_rn(ks[2][c], ks[3][c])) : 0.0;
      uint32_t mb = 0u;
#pragma unroll
      for (int i = 0; i < kWarps; ++i) {
        const uint32_t pr = vm[i][c >> 1];
        mb = max(mb, (c & 1) ? (pr >> 16) : (pr & 0xFFFFu));
      }
      g_sum[c] = gs;
      g_max[c] = mb;
    }
    // after this barrier every CTA's group results are visible to the cluster
    tc::cluster_arrive_release();
    tc::cluster_wait_acquire();
    double lv[kShortMaxGroups];
    float vmx = 0.0f;
    if (c < kHeadDim) {
      const uint32_t a_sum = tc::smem_u32(&g_sum[c]), a_max = tc::smem_u32(&g_max[c]);
#pragma unroll
      for (int r = 0; r < kShortMaxGroups; ++r) {
        lv[r] = r < G ? tc::ld_cluster_f64(tc::mapa_shared(a_sum, static_cast<uint32_t>(r))) : 0.0;
        if (r < G)
          vmx = fmaxf(vmx, __uint_as_float(tc::ld_cluster_u32(tc::mapa_shared(a_max, static_cast<uint32_t>(r)))
                                           << 16));
      }
    }
    // this thread reads no other CTA's shared memory from here on (release:
    // the loads above are complete before a CTA they read may exit)
    tc::cluster_arrive_release();
    if (c < kHeadDim) {
      // the head's key mean and V scale of channel c (the same in every CTA):
      // the pairwise tree over the P = 2^ceil(log2 G) group sums
#pragma unroll
      for (int w = 1; w < kShortMaxGroups; w *= 2) {
        if (w >= G) break;  // lv[0] already holds the tree of the first P leaves
#pragma unroll
        for (int k = 0; k < kShortMaxGroups; k += 2 * w) lv[k] = __dadd_rn(lv[k], lv[k + w]);
      }
      const float mu = prm.smooth_k ? __double2float_rn(__ddiv_rn(lv[0], static_cast<double>(S))) : 0.0f;
      const float vs = __fdiv_rn(vmx, kE4M3Max);
      h_mean[c] = mu;
      h_vscale[c] = vs;
      h_vrcp[c] = vs >= FLT_MIN ? __frcp_rn(vs) : 0.0f;
      if (g == 0) {
        const int64_t head = out_head<kPair>(prm, bh, c / kOutDim<kPair>);
        if (head >= 0) {
          prm.out.k_mean[head * kOutDim<kPair> + (c & (kOutDim<kPair> - 1))] = mu;
          prm.out.v_scale[head * kOutDim<kPair> + (c & (kOutDim<kPair> - 1))] = vs;
        }
      }
    }
    asm volatile("bar.arrive 2, %0;" ::"n"(kShortThreads) : "memory");  // h_vscale to team 0
    asm volatile("bar.sync 11, %0;" ::"n"(kTeamThreads) : "memory");    // h_mean within team 1
    // K codes of k - mean
    int8_t* kc;
    uint16_t* k16;
    const int64_t kh =
        lane_codes<kPair>(prm, prm.write_int8 ? prm.out.k_codes : nullptr, prm.out.k16, bh, s0, lane, kc, k16);
    constexpr int od = kOutDim<kPair>;
    volatile float* xm = &xa[pair][sub][0];
    volatile float* xo = &xa[pair][sub ^ 1][0];
    float skv;
    if (prm.smooth_k) {
      const float4* mp = reinterpret_cast<const float4*>(h_mean + 8 * (lane & 15));
      const float4 ma = mp[0], mb = mp[1];
      const float2 nmu[4] = {make_float2(-ma.x, -ma.y), make_float2(-ma.z, -ma.w), make_float2(-mb.x, -mb.y),
                             make_float2(-mb.z, -mb.w)};
      skv = nv == kHalfRows
                ? quantize_half_block<true, true, kPair>(k_rows, nmu, kHalfRows, kc, k16, od, lane, xm, xo, pair)
                : quantize_half_block<true, false, kPair>(k_rows, nmu, nv, kc, k16, od, lane, xm, xo, pair);
    } else {
      const float2 nz[4] = {};
      skv = nv == kHalfRows
                ? quantize_half_block<false, true, kPair>(k_rows, nz, kHalfRows, kc, k16, od, lane, xm, xo, pair)
                : quantize_half_block<false, false, kPair>(k_rows, nz, nv, kc, k16, od, lane, xm, xo, pair);
    }
    store_block_scale<kPair>(prm.out.k_scale, kh, nblk, s0c / kQKBlock, skv, lane, sub);
  }
  if (!ok) {
    // let every copy land before the CTA exits
    Ctx drain = cx;
    volatile int no_abort = 0;
    drain.abort_flag = &no_abort;
    for (int n = 0; n < 3; ++n) wait_bar(drain, cx.full(n), 0);
  }
  // the other CTAs of the cluster have read this one's group results
  tc::cluster_wait_acquire();
}

struct ScratchLayout {
  size_t done_off, ready_off, ksum_off, vmax_off, vrcp_off, hstat_off, header, total;
};

// H: the (virtual) heads per batch; pair: head-pair mode, which adds each
// virtual head's key mean and V scales for the codes items.
ScratchLayout scratch_layout(int64_t B, int64_t S, int64_t H, bool pair) {
  const int64_t G = div_up(S, kItemTokens);
  const size_t NH = static_cast<size_t>(B * H);
  const size_t n = NH * static_cast<size_t>(G) * kHeadDim;
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  ScratchLayout l;
  l.done_off = 256;
  l.ready_off = l.done_off + r256(NH * 4);
  l.header = l.ready_off + r256(NH * 4);
  l.ksum_off = l.header;
  l.vmax_off = l.ksum_off + r256(n * sizeof(double));
  l.vrcp_off = l.vmax_off + r256(n * sizeof(float));
  l.hstat_off = l.vrcp_off + r256(NH * kHeadDim * sizeof(float));
  l.total = l.hstat_off + (pair ? r256(NH * 2 * kHeadDim * sizeof(float)) : 0);
  return l;
}

// 4-D bf16 map over one input: dims (channel, a1, a2, b) where (a1, a2) are
// (s, h) or (h, s) in increasing stride order; boxes of 128 channels x 128
// tokens. Returns the position of the token axis (1 or 2), or 0 on failure.
int make_input_map(CUtensorMap* m, const Bf16In& t, int64_t B, int64_t S, int64_t H) {
  const bool s_first = t.ss <= t.sh;
  const uint64_t dims[4] = {static_cast<uint64_t>(kHeadDim), static_cast<uint64_t>(s_first ? S : H),
                            static_cast<uint64_t>(s_first ? H : S), static_cast<uint64_t>(B)};
  const uint64_t strides[3] = {static_cast<uint64_t>((s_first ? t.ss : t.sh) * 2),
                               static_cast<uint64_t>((s_first ? t.sh : t.ss) * 2), static_cast<uint64_t>(t.sb * 2)};
  const uint32_t box[4] = {kHeadDim, s_first ? static_cast<uint32_t>(kItemTokens) : 1u,
                           s_first ? 1u : static_cast<uint32_t>(kItemTokens), 1u};
  if (!make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, t.p, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
    return 0;
  return s_first ? 1 : 2;
}

// 4-D bf16 map over one head-dimension-64 input for head-pair mode: dims
// (channel, h, s, b) with the input's own strides, in whatever order they
// come, and boxes of 64 channels x 2 heads x 128 tokens, which land in shared
// memory as 128 rows of (head 2hp, head 2hp + 1): the 128-channel tile of
// virtual head hp. A missing second head (odd H) reads as zeros.
bool make_pair_map(CUtensorMap* m, const Bf16In& t, int64_t B, int64_t S, int64_t H) {
  const uint64_t dims[4] = {static_cast<uint64_t>(kHeadDim / 2), static_cast<uint64_t>(H), static_cast<uint64_t>(S),
                            static_cast<uint64_t>(B)};
  const uint64_t strides[3] = {static_cast<uint64_t>(t.sh * 2), static_cast<uint64_t>(t.ss * 2),
                               static_cast<uint64_t>(t.sb * 2)};
  const uint32_t box[4] = {kHeadDim / 2, 2u, static_cast<uint32_t>(kItemTokens), 1u};
  return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, t.p, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace

bool prologue_uses_scratch(int64_t S, int64_t D) {
  (void)D;  // both head dimensions use the cluster kernel for short sequences
  return div_up(S, kItemTokens) > kShortMaxGroups;
}

size_t prologue_scratch_bytes(int64_t B, int64_t S, int64_t H, int64_t D) {
  return D == kHeadDim ? scratch_layout(B, S, H, false).total : scratch_layout(B, S, div_up(H, 2), true).total;
}

namespace {

template <bool kPair>
cudaError_t launch_prologue_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const Params& p,
                              int3 axes, void* scratch, size_t header, cudaStream_t stream) {
  cudaError_t e;
  if (p.G <= kShortMaxGroups) {
    // short sequences: one cluster per head, no scratch
    if ((e = set_smem_limit_once(reinterpret_cast<const void*>(prologue_short_kernel<kPair>),
                                 static_cast<int>(kShortSmemBytes))) != cudaSuccess)
      return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.G * p.NH));
    cfg.blockDim = dim3(kShortThreads);
    cfg.dynamicSmemBytes = kShortSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.G);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prologue_short_kernel<kPair>, tq, tk, tv, p, axes);
  }
  if ((e = cudaMemsetAsync(scratch, 0, header, stream)) != cudaSuccess) return e;
  if ((e = set_smem_limit_once(reinterpret_cast<const void*>(prologue_kernel<kPair>), static_cast<int>(kSmemBytes))) !=
      cudaSuccess)
    return e;
  const int sms = sm_count_current();
  const int grid = static_cast<int>(p.total < sms ? p.total : sms);
  prologue_kernel<kPair><<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p, axes);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prologue(const Bf16In& q, const Bf16In& k, const Bf16In& v, int64_t B, int64_t S, int64_t H,
                            int64_t D, bool smooth_k, const Bundle& out, void* scratch, bool write_int8,
                            int* dev_err, cudaStream_t stream) {
  if (D != kHeadDim && D != kHeadDim / 2) return cudaErrorInvalidValue;
  // head dimension 64 runs as head pairs: ceil(H / 2) virtual heads of 128 channels
  const bool pair = D != kHeadDim;
  const int64_t Hv = pair ? div_up(H, 2) : H;
  const ScratchLayout l = scratch_layout(B, S, Hv, pair);
  char* sc = static_cast<char*>(scratch);
  Params p;
  p.S = S;
  p.S_pad = padded_len(S);
  p.H = Hv;
  p.Hr = H;
  p.NH = B * Hv;
  p.G = div_up(S, kItemTokens);
  p.total = 2 * p.NH * p.G;
  // every stats item comes before every codes item (lag = all heads).
  // Interleaving them (codes of head h right after the stats of head h + L,
  // to read K and V the second time from L2) was measured slower at every L:
  // the codes items then wait for heads still being finished, and those
  // waits cost more than the DRAM reads they save
  const int64_t lag = p.NH;
  p.lag = lag;
  p.smooth_k = smooth_k ? 1 : 0;
  p.write_int8 = write_int8 ? 1 : 0;
  p.out = out;
  p.next_item = reinterpret_cast<unsigned*>(sc);
  p.done = reinterpret_cast<unsigned*>(sc + l.done_off);
  p.ready = reinterpret_cast<unsigned*>(sc + l.ready_off);
  p.ksum = reinterpret_cast<double*>(sc + l.ksum_off);
  p.vmax = reinterpret_cast<float*>(sc + l.vmax_off);
  p.vrcp = reinterpret_cast<float*>(sc + l.vrcp_off);
  p.hstat_v = pair ? reinterpret_cast<float*>(sc + l.hstat_off) : nullptr;
  p.dev_err = dev_err;
  CUtensorMap tq, tk, tv;
  if (pair) {
    if (!make_pair_map(&tq, q, B, S, H) || !make_pair_map(&tk, k, B, S, H) || !make_pair_map(&tv, v, B, S, H))
      return cudaErrorInvalidValue;
    return launch_prologue_t<true>(tq, tk, tv, p, make_int3(2, 2, 2), scratch, l.header, stream);
  }
  const int aq = make_input_map(&tq, q, B, S, H), ak = make_input_map(&tk, k, B, S, H),
            av = make_input_map(&tv, v, B, S, H);
  if (aq == 0 || ak == 0 || av == 0) return cudaErrorInvalidValue;
  return launch_prologue_t<false>(tq, tk, tv, p, make_int3(aq, ak, av), scratch, l.header, stream);
}

}  // namespace sage
