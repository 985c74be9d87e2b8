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
//     (transposed), after waiting until the head is ready.
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
// summed as an unevaluated pair of floats (TwoSum: hi + lo is the exact
// running sum while lo's own additions are exact). All values are multiples
// of 2^L, the last-bit weight of the smallest nonzero input; with A the sum
// of |x|, every rounding error is below 2^(e(A)-24), and lo, which gathers
// 33 of them (two chains of 16 tokens and the join), stays exact while
// e(A) - L <= 42 (the float sum of |x| may sit one binade low, so the test
// is e(fl(A)) - L <= 41). In that case every prefix sum also fits in 53 bits, so the
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

// Channel c (0..3) of a lane's 4-channel group.
__device__ __forceinline__ float chan(const uint2& w, int c) {
  return c == 0 ? lo_bf16(w.x) : c == 1 ? hi_bf16(w.x) : c == 2 ? lo_bf16(w.y) : hi_bf16(w.y);
}

// Number of tokens s0 .. s0+31 that are below S.
__device__ __forceinline__ int valid_in_chunk(int64_t S, int64_t s0) {
  const int64_t d = S - s0;
  return d <= 0 ? 0 : (d >= 32 ? 32 : static_cast<int>(d));
}

// Channels [4*lane, 4*lane+4) of token t of the warp's 32 tokens, from a
// shared-memory tile of 256-byte token rows (a warp instruction reads one row).
__device__ __forceinline__ uint2 tok(const uint8_t* rows, int t, int lane) {
  return *reinterpret_cast<const uint2*>(rows + t * 256 + lane * 8);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Exact path of a code: bits of fl(fl(x / s) + kMagic). Kept out of line:
// it runs only when the fast path cannot decide.
__device__ __noinline__ uint32_t exact_code_bits(float x, float s) {
  return __float_as_uint(__fadd_rn(__fdiv_rn(x, s), kMagic));
}

// Bits of fl(q + kMagic) where q = fl(x / s); the low byte is the int8 code.
__device__ __forceinline__ uint32_t int8_code_bits(float x, float s, float r, bool fast) {
  if (fast) {
    const float q = __fmul_rn(x, r);
    const float t = __fadd_rn(q, kMagic);
    const float f = __fsub_rn(q, __fsub_rn(t, kMagic));
    if (fabsf(f) < kHalfGuard) return __float_as_uint(t);
  }
  return exact_code_bits(x, s);
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

// INT8 codes and scale of one 32-token block (the warp's rows of a shared
// tile, 4 channels per lane), of x - mu. Writes rows s0..s0+31 of f16_bh
// ([S_pad][128], the codes as fp16) and, when codes_bh is not null, of
// codes_bh ([S_pad][128] int8); both with streaming stores. Returns the scale.
__device__ __forceinline__ float quantize_int8_block(const uint8_t* rows, const float (&mu)[4], int nvalid,
                                                     int8_t* codes_bh, uint16_t* f16_bh, int64_t s0, int lane) {
  float a = 0.0f;
#pragma unroll 8
  for (int t = 0; t < 32; ++t) {
    if (t < nvalid) {
      const uint2 w = tok(rows, t, lane);
#pragma unroll
      for (int c = 0; c < 4; ++c) a = fmaxf(a, fabsf(__fsub_rn(chan(w, c), mu[c])));
    }
  }
  a = warp_max(a);
  const float s = __fdiv_rn(a, kInt8Max);
  const bool fast = s >= FLT_MIN;
  const float r = fast ? __frcp_rn(s) : 0.0f;
  uint32_t* out = codes_bh ? reinterpret_cast<uint32_t*>(codes_bh + s0 * kHeadDim) + lane : nullptr;
  uint2* out16 = reinterpret_cast<uint2*>(f16_bh + s0 * kHeadDim) + lane;
#pragma unroll 4
  for (int t = 0; t < 32; ++t) {
    uint32_t word = 0u;
    if (t < nvalid && a > 0.0f) {
      const uint2 w = tok(rows, t, lane);
      uint32_t bits[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) bits[c] = int8_code_bits(__fsub_rn(chan(w, c), mu[c]), s, r, fast);
      word = pack_low_bytes(bits[0], bits[1], bits[2], bits[3]);
    }
    if (out) __stcs(out + t * (kHeadDim / 4), word);
    __stcs(out16 + t * (kHeadDim / 4), codes_to_f16x4(word));
  }
  return s;
}

// Left-to-right fp64 sum of channel c over the first nvalid rows (the exact
// reference order, used when the float-pair path cannot guarantee it).
__device__ __noinline__ double fp64_chunk_sum(const uint8_t* rows, int nvalid, int lane, int c) {
  double p = 0.0;
  for (int t = 0; t < nvalid; ++t) p = __dadd_rn(p, static_cast<double>(chan(tok(rows, t, lane), c)));
  return p;
}

// Exact fp64 chunk sums of the lane's 4 channels over the warp's rows (see
// the file comment for why the float-pair path is bit-identical). Even and
// odd tokens run in two float-pair chains for instruction-level parallelism;
// joining them adds one more error term to lo, inside the same bound.
__device__ __forceinline__ void chunk_sums(const uint8_t* rows, int nvalid, int lane, double (&out)[4]) {
  float hi[2][4], lo[2][4], am[2][4];
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int c = 0; c < 4; ++c) hi[k][c] = lo[k][c] = am[k][c] = 0.0f;
  uint32_t umin = 0xFFFFFFFFu;  // (|bits| - 1) of the smallest nonzero magnitude; zeros wrap to all-ones
#pragma unroll 4
  for (int t = 0; t < 32; t += 2) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (t + k < nvalid) {
        const uint2 w = tok(rows, t + k, lane);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float x = chan(w, c);
          const float s = __fadd_rn(hi[k][c], x);
          const float bb = __fsub_rn(s, hi[k][c]);
          const float err = __fadd_rn(__fsub_rn(hi[k][c], __fsub_rn(s, bb)), __fsub_rn(x, bb));
          hi[k][c] = s;
          lo[k][c] = __fadd_rn(lo[k][c], err);
          am[k][c] = __fadd_rn(am[k][c], fabsf(x));
        }
        umin = min(umin, (w.x & 0x7FFFu) - 1u);
        umin = min(umin, ((w.x >> 16) & 0x7FFFu) - 1u);
        umin = min(umin, (w.y & 0x7FFFu) - 1u);
        umin = min(umin, ((w.y >> 16) & 0x7FFFu) - 1u);
      }
    }
  }
  int ef = static_cast<int>(((umin + 1u) >> 7) & 0xFFu);
  if (ef == 0) ef = 1;                 // subnormal bf16: last-bit weight 2^-133
  const int lsb = ef - 127 - 7;         // L: exponent of the smallest last-bit weight
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    // join the chains: TwoSum of the high parts, the error joins lo
    const float s = __fadd_rn(hi[0][c], hi[1][c]);
    const float bb = __fsub_rn(s, hi[0][c]);
    const float err = __fadd_rn(__fsub_rn(hi[0][c], __fsub_rn(s, bb)), __fsub_rn(hi[1][c], bb));
    const float l = __fadd_rn(__fadd_rn(lo[0][c], lo[1][c]), err);
    const float a = __fadd_rn(am[0][c], am[1][c]);
    const int ea = static_cast<int>((__float_as_uint(a) >> 23) & 0xFFu) - 127;
    out[c] = ea - lsb <= 41 ? __dadd_rn(static_cast<double>(s), static_cast<double>(l))
                            : fp64_chunk_sum(rows, nvalid, lane, c);
  }
}

// Two e4m3 codes: high byte = code(a), low byte = code(b).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(a), "f"(b));
  return r;
}

// Exact path of two V codes (out of line: rare).
__device__ __noinline__ uint32_t exact_v_pair(float x0, float x1, float s0, float s1) {
  return e4m3x2(__fdiv_rn(x1, s1), __fdiv_rn(x0, s0));
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
  return exact_v_pair(x0, x1, s0, s1);
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
  __shared__ int ready_ok[kTeams];  // codes items: the head's statistics are published
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
        const float zero[4] = {0.f, 0.f, 0.f, 0.f};
        const float s = quantize_int8_block(rows, zero, nvalid,
                                            prm.write_int8 ? prm.out.q_codes + bh * S_pad * kHeadDim : nullptr,
                                            prm.out.q16 + bh * S_pad * kHeadDim, s0, lane);
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
        double sums[4];
        chunk_sums(rows, nvalid, lane, sums);
        tc::mbar_arrive(cx.empty(c2 % kStages));
        ++c2;
#pragma unroll
        for (int c = 0; c < 4; ++c) ks[tw][4 * lane + c] = sums[c];
      }
      // V tile: max |v| per channel (bf16 magnitudes compare as integers)
      const uint32_t sv = c2 % kStages;
      if (c2 != mine && !wait_bar(cx, cx.full(sv), (c2 / kStages) & 1u)) break;
      const uint8_t* vr = smem + sv * kTileBytes + tw * 32 * 256;
      uint32_t m01 = 0u, m23 = 0u;
#pragma unroll 8
      for (int t = 0; t < 32; ++t) {
        if (t < nvalid) {
          const uint2 w = tok(vr, t, lane);
          m01 = __vmaxu2(m01, w.x & 0x7FFF7FFFu);
          m23 = __vmaxu2(m23, w.y & 0x7FFF7FFFu);
        }
      }
      tc::mbar_arrive(cx.empty(sv));
      vm[tw][2 * lane] = m01;
      vm[tw][2 * lane + 1] = m23;
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
      // codes item: both tiles need the head's statistics
      if (tt == 0) ready_ok[team] = wait_ready(cx, prm.ready + bh) ? 1 : 0;
      team_bar(team);
      const bool head_ready = ready_ok[team] != 0;
      team_bar(team);  // everyone has read ready_ok before thread 0 may write it again
      if (!head_ready) break;
      if (team == 1 && !wait_bar(cx, cx.full(mine % kStages), (mine / kStages) & 1u)) break;
      if (team == 0) {
        // K codes of k - mean
        float mu[4];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          mu[c] = prm.smooth_k ? __ldcg(prm.out.k_mean + bh * kHeadDim + 4 * lane + c) : 0.f;
        if (in_pad) {
          int8_t* kc = prm.write_int8 ? prm.out.k_codes + bh * S_pad * kHeadDim : nullptr;
          uint16_t* k16 = prm.out.k16 + bh * S_pad * kHeadDim;
          const float skv = quantize_int8_block(rows, mu, nvalid, kc, k16, s0, lane);
          if (lane == 0) prm.out.k_scale[bh * (S_pad / kQKBlock) + s0 / kQKBlock] = skv;
        }
        tc::mbar_arrive(cx.empty(st));
        if (!pass(cnt + 1)) break;
      } else {
        // V codes, transposed to [channel][token]
        if (in_pad) {
          float svs[4], rv[4];
          bool live[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            svs[c] = __ldcg(prm.out.v_scale + bh * kHeadDim + 4 * lane + c);
            live[c] = svs[c] > 0.0f;
            rv[c] = svs[c] >= FLT_MIN ? __frcp_rn(svs[c]) : 0.0f;
          }
          const bool fast01 = svs[0] >= FLT_MIN && svs[1] >= FLT_MIN;
          const bool fast23 = svs[2] >= FLT_MIN && svs[3] >= FLT_MIN;
          const uint32_t keep = (live[0] ? 0x000000FFu : 0u) | (live[1] ? 0x0000FF00u : 0u) |
                                (live[2] ? 0x00FF0000u : 0u) | (live[3] ? 0xFF000000u : 0u);
          uint32_t cw[4][8];  // cw[c][j]: tokens 4j..4j+3 of channel 4*lane+c
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint32_t a[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int t = 4 * j + q;
              uint32_t word = 0u;
              if (t < nvalid) {
                const uint2 w = tok(rows, t, lane);
                const uint32_t p01 = v_code_pair(lo_bf16(w.x), hi_bf16(w.x), svs[0], svs[1], rv[0], rv[1], fast01);
                const uint32_t p23 = v_code_pair(lo_bf16(w.y), hi_bf16(w.y), svs[2], svs[3], rv[2], rv[3], fast23);
                word = (p01 | (p23 << 16)) & keep;
              }
              a[q] = word;
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
