// Quantized flash attention on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// Method: "aiter-sage-attention: SageAttention for AMD RDNA4 (gfx1201)
// #1222", section "The kernel": QK^T in INT8 and PV in FP8, both with FP32
// accumulation; Q/K scales per 32-token block, V scales per channel.
//
// INT8 QK^T. sm_103a has no integer tcgen05 MMA, so the int8 codes (kept as
// exact fp16 copies by the prologue: every integer in [-127, 127] is an fp16
// value) are multiplied with kind::f16 into an fp32 accumulator in TMEM. Each
// product is an integer of magnitude <= 127^2 and every partial sum of the 128
// products stays below 2^21, so the fp32 accumulation is exact: S_ij equals the
// INT32 dot product of the codes bit for bit.
//
// FP8 PV. The softmax writes P as e4m3(448 p) into a shared-memory tile (the
// 128-byte-swizzled K-major layout the MMA reads); a kind::f8f6f4 MMA
// multiplies it with the transposed e4m3 V tile; O accumulates in fp32 in TMEM.
//
// Schedule (one persistent CTA per SM; 384 threads, or 512 with the
// correction warpgroup):
//   warp 0      TMA producer: fp16 Q tiles, a 2-stage ring of fp16 K tiles
//               (two 64-channel boxes per tile) and a 4-stage ring of e4m3
//               V^T tiles, all in 128-byte-swizzled boxes. A V tile is held
//               until its PV completes, long after its K tile's QK, so the V
//               ring is the deeper one: the producer, which loads K_j and
//               V_j in turn, then rarely waits for a V stage.
//   warp 1, 2   TMEM allocation (warp 1) and one MMA-issuing thread per query
//               tile: each waits only on its own tile's events.
//   warp 3      idle.
//   warps 4-7   softmax for query tile 0 (TMEM lanes 0..127 = its 128 rows).
//   warps 8-11  softmax for query tile 1.
//   warps 12-15 (kCorr) correction: rescale O_i by alpha before PV_j, for
//               both tiles (a warp reaches the TMEM lanes of its index mod 4
//               only, so a full warpgroup serves the 128 rows).
// A work unit is one (batch, head) and a pair of 128-row query tiles. TMEM
// holds S0, S1, O0, O1 (4 x 128 columns of fp32). Per tile and 128-key step j
// the softmax reads S_j into registers and releases S at once, so the MMA
// thread issues QK_{j+1} while the softmax still works on step j; when P_j is
// in shared memory and O rescaled it issues PV_j. The softmax is online over
// 128-key tiles in ascending order with the exact running maximum; O is
// multiplied by alpha = 2^(m_old - m_new) only in warps where some row's
// maximum grew (alpha = 1 exactly otherwise). Without the correction
// warpgroup the softmax thread does it after storing P_j; with it, the
// softmax thread posts alpha once PV_{j-1} is done and the correction warp of
// its row rescales O while P_j is stored.
// Logits are kept in base 2: x = S * (s_q * sm_scale * log2 e) * s_k, and
// p448 = 2^(x - m + log2 448) is both the e4m3 input and the row-sum term, so
// the epilogue computes O = acc * s_v / l.
//
// Every wait on an mbarrier is bounded; when one runs out the kernel sets the
// device error word, tells the other roles to stop, lets its own copies and
// MMAs drain, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <memory>
#include <mutex>
#include <type_traits>
#include <utility>
#include <vector>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace sage {
namespace {

// threads of a CTA: 12 warps, plus a correction warpgroup when it takes the
// O rescale off the softmax warps (kCorr)
template <bool kCorr>
constexpr int threads_of() { return kCorr ? 512 : 384; }
constexpr int kKStages = 2;
constexpr int kVStages = 4;
constexpr uint32_t kTile8 = 128 * 128;       // bytes of one e4m3 P tile (128 rows x 128 keys)
constexpr uint32_t kSub16 = 128 * 128;       // bytes of one 64-channel fp16 subtile (128 rows)

// Shared memory layout for head dimension D (offsets from a 1024-aligned base).
template <int D>
struct Smem {
  static constexpr uint32_t kTile16 = 128 * D * 2;                     // fp16 Q or K tile: D / 64 subtiles
  static constexpr uint32_t kTileV = D * 128;                          // e4m3 V^T tile: D rows of 128 keys
  static constexpr uint32_t kOffQ16 = 0;                               // 2 query tiles
  static constexpr uint32_t kOffK16 = kOffQ16 + 2 * kTile16;           // K ring
  static constexpr uint32_t kOffV = kOffK16 + kKStages * kTile16;      // V ring
  static constexpr uint32_t kOffP = kOffV + kVStages * kTileV;         // 2 P tiles
  static constexpr uint32_t kOffBar = kOffP + 2 * kTile8;
};
// barriers (8 bytes each)
constexpr int kBarQFull = 0, kBarQEmpty = 1;
constexpr int kBarKFull = 2, kBarKEmpty = kBarKFull + kKStages;
constexpr int kBarVFull = kBarKEmpty + kKStages, kBarVEmpty = kBarVFull + kVStages;
constexpr int kBarSFull = kBarVEmpty + kVStages, kBarSFree = kBarSFull + 2;
constexpr int kBarPFull = kBarSFree + 2, kBarPVDone = kBarPFull + 2;
constexpr int kBarOEmpty = kBarPVDone + 2, kBarDrain = kBarOEmpty + 2;
constexpr int kBarVs = kBarDrain + 2;  // a softmax warpgroup's V scales are parked
constexpr int kBarORdy = kBarVs + 2;   // O of a tile is rescaled for the next PV
constexpr int kBarAlpha = kBarORdy + 2;  // a tile's rescale factors are posted
constexpr int kNumBars = kBarAlpha + 2;
template <int D>
struct SmemTail {
  static constexpr uint32_t kOffTmemSlot = Smem<D>::kOffBar + kNumBars * 8;
  static constexpr uint32_t kOffAbort = kOffTmemSlot + 8;
  static constexpr uint32_t kOffVs = (kOffAbort + 8 + 15) / 16 * 16;  // [warpgroup][D] fp32
  static constexpr uint32_t kOffAlpha = kOffVs + 2 * D * 4;            // [tile][row] fp32
  static constexpr uint32_t kBytes = kOffAlpha + 2 * 128 * 4;
};
static_assert(SmemTail<128>::kBytes <= 232448u, "shared memory of one CTA: at most 227 KB");

// TMEM columns: S of query tile i at 128*i, O of query tile i (D columns) at 256 + D*i
__host__ __device__ constexpr uint32_t col_s(int i) { return 128u * static_cast<uint32_t>(i); }
template <int D>
__host__ __device__ constexpr uint32_t col_o(int i) { return 256u + static_cast<uint32_t>(D) * static_cast<uint32_t>(i); }
// At D = 64 the 128 columns past O hold P of each query tile, two buffers of
// 32 columns (128 e4m3 keys of a row, four per column) at 384 + 64*i + 32*b:
// PV reads P from tensor memory, and the softmax writes P of step j while PV
// of step j-1 still reads the other buffer.
__host__ __device__ constexpr uint32_t col_p(int i, int b) {
  return 384u + 64u * static_cast<uint32_t>(i) + 32u * static_cast<uint32_t>(b);
}
constexpr uint32_t kTmemCols = 512;

constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr int64_t kCorrMinKeyTiles = 16;         // key tiles from which the correction warpgroup is used
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLog2P = 8.807354922057604f;    // log2(448)
constexpr float kLn2 = 0.6931471805599453f;

struct Params {
  int64_t S, S_pad, n_kv, pairs_per_head, n_units;  // pairs_per_head: units per head
  int tiles;   // query tiles per unit: 2 (one per softmax warpgroup), or 1 when few units would leave SMs idle
  float* lse;  // [B][H][S] natural-log log-sum-exp of each row's logits, or null
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  Out out;
  int64_t H;
  float sm_log2;  // sm_scale * log2(e)
  int* dev_err;
};

// Work-unit schedule of the causal kernel. With the mask, the unit of query
// tiles (2p, 2p+1) of a head reads 2p + 2 key tiles, so round-robin units
// leave CTAs unevenly loaded (82.6% of the busiest CTA's work on average at
// B1 H28 S16384). The host assigns units heaviest first, within windows of a
// few heads (their K and V stay in L2 together), each to the CTA with the
// least work so far; CTA b takes units unit[start[b] .. start[b+1]) in that
// order. n = 0: round robin (too many units or CTAs for the table).
constexpr int kSchedMaxUnits = 7168;
constexpr int kSchedMaxCtas = 160;
struct Sched {
  int32_t n;
  uint16_t start[kSchedMaxCtas + 1];
  uint16_t unit[kSchedMaxUnits];
};
struct NoSched {};
template <bool kCausal>
using SchedOf = typename std::conditional<kCausal, Sched, NoSched>::type;

// Key tiles query tile `qt` reads: all of them, or with the causal mask the
// tiles up to its diagonal (Q and K have the same length).
template <bool kCausal>
__device__ __forceinline__ int64_t key_tiles(const Params& prm, int64_t qt) {
  return kCausal ? min(prm.n_kv, qt + 1) : prm.n_kv;
}

// This CTA's units. Without a schedule: u = blockIdx.x, + grid, + 2 grid, ...
// while u < n_units. With one: the table's entries, then -1.
template <bool kCausal>
__device__ __forceinline__ int64_t first_unit(const SchedOf<kCausal>& sc) {
  if constexpr (kCausal) {
    if (sc.n > 0) return sc.start[blockIdx.x] < sc.start[blockIdx.x + 1] ? sc.unit[sc.start[blockIdx.x]] : -1;
  }
  return blockIdx.x;
}
template <bool kCausal>
__device__ __forceinline__ bool unit_valid(const Params& prm, const SchedOf<kCausal>& sc, int64_t u) {
  if constexpr (kCausal) {
    if (sc.n > 0) return u >= 0;
  }
  return u < prm.n_units;
}
// the unit after u, which is this CTA's k-th (k >= 1)
template <bool kCausal>
__device__ __forceinline__ int64_t next_unit(const SchedOf<kCausal>& sc, int64_t u, int64_t k) {
  if constexpr (kCausal) {
    if (sc.n > 0) {
      const int64_t i = static_cast<int64_t>(sc.start[blockIdx.x]) + k;
      return i < sc.start[blockIdx.x + 1] ? static_cast<int64_t>(sc.unit[i]) : -1;
    }
  }
  return u + gridDim.x;
}

struct Ctx {
  uint32_t bar0;
  volatile int* abort_flag;
  int* dev_err;
  __device__ uint32_t bar(int i) const { return bar0 + 8u * static_cast<uint32_t>(i); }
};

// Bounded wait for the phase of `parity` on barrier `bar` to complete.
// (Inlined everywhere: setmaxnreg gives the roles different register
// budgets, and one out-of-line copy cannot be allocated for both.)
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

// Warp-uniform bounded wait: every lane waits; the warp continues only if all did.
__device__ __forceinline__ bool wait_bar_warp(const Ctx& cx, uint32_t bar, uint32_t parity) {
  const bool ok = wait_bar(cx, bar, parity);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {  // high byte = code(a), low byte = code(b)
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Register rebalancing between warpgroups (setmaxnreg is warpgroup-wide: all
// four warps of a warpgroup execute the same instruction). With 12 warps the
// block is launched with 168 registers per thread (384 x 168 = 64512); the
// control warpgroup drops to ctl and the softmax warpgroups rise to softmax
// (128 x 88 + 256 x 208 = 64512). With the correction warpgroup (16 warps, 128
// per thread at launch) the split is 128 x 80 + 256 x 184 + 128 x 64 = 65536.
// At the end every warpgroup moves to ctl, so the shared teardown runs with
// one budget in every warp. The changes sit inside the branches so the
// compiler allocates each branch with its own budget.
template <bool kCorr>
struct Regs {
  static constexpr uint32_t ctl = kCorr ? 80 : 88, softmax = kCorr ? 184 : 208, corr = 64;
  static_assert(128 * ctl + 256 * softmax + (kCorr ? 128 * corr : 0) <= 65536, "register file of one SM");
};
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Shared-memory descriptors of the operand buffers are computed once; the
// start-address field holds (address >> 4) in its low 14 bits and every buffer
// lies below 256 KB, so the descriptor of buffer + offset is descriptor +
// (offset >> 4) with no carry out of the field.
__device__ __forceinline__ uint64_t desc_at(uint64_t base, uint32_t offset) { return base + (offset >> 4); }

// S_i = Q_i K^T for one 128-key tile: D / 16 MMAs of K = 16 over the
// 64-channel subtiles of the fp16 Q and K tiles (dq, dk: descriptors of the
// two tiles' first subtiles).
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t dq, uint64_t dk) {
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t off = static_cast<uint32_t>(ks >> 2) * kSub16 + static_cast<uint32_t>(ks & 3) * 32u;
    tc::mma_f16_ss(d_tmem, desc_at(dq, off), desc_at(dk, off), tc::kIdescM128N128, ks > 0 ? 1u : 0u);
  }
}

// O_i (+)= P_i V for one 128-key tile: 4 MMAs of M = 128, N = D, K = 32;
// V^T in shared memory, 128-byte swizzled; P_i (e4m3, written by the softmax
// warps) in shared memory in the same layout at D = 128 (dp), in tensor
// memory at D = 64 (tp: its first column; 32 keys are 8 columns).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint64_t dp, uint32_t tp, uint64_t dv, bool acc) {
  constexpr uint32_t idesc = D == 128 ? tc::kIdescM128N128 : tc::kIdescM128N64;
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    if constexpr (D == 64)
      tc::mma_f8_ts(d_tmem, tp + 8u * ks, desc_at(dv, 32u * ks), idesc, (acc || ks > 0) ? 1u : 0u);
    else
      tc::mma_f8_ss(d_tmem, desc_at(dp, 32u * ks), desc_at(dv, 32u * ks), idesc, (acc || ks > 0) ? 1u : 0u);
  }
}

// One lane of the warp, chosen by the hardware (elect.sync).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// One 128-key tile of the online softmax for the calling thread's query row
// (TMEM lane `row`): reads S, releases it for the next QK, updates the
// running maximum m and row sum l, waits until the previous PV has finished
// with P and O, writes e4m3(p448) into the shared-memory P tile and rescales O
// when the maximum grew. kTail masks keys at or past nvalid (the last tile of a
// ragged S). At D = 64, P goes to this step's tensor-memory buffer tP instead
// (the previous PV reads the other one), before the wait for that PV, which
// only the O rescale needs. Returns false if a bounded wait ran out.
template <int D, bool kTail, bool kCorr>
__device__ __forceinline__ bool softmax_tile(const Ctx& cx, int i, uint32_t tS, uint32_t tO, uint32_t tP,
                                             float* alpha_row, uint8_t* p_row, int row, const float (&cb)[4],
                                             int nvalid, bool first, uint32_t& pv_cnt, float& m, float& l) {
  uint32_t sr[4][32];
#pragma unroll
  for (int b = 0; b < 4; ++b) tc::tmem_ld32(tS + 32u * b, sr[b]);
  tc::tmem_wait_ld();
  tc::tc_fence_before();
  tc::mbar_arrive(cx.bar(kBarSFree + i));  // S may now be overwritten by the next QK
  if (kTail) {
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (32 * b + k >= nvalid) sr[b][k] = 0xFF800000u;  // -inf
  }
  float mt = -INFINITY;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    float mb = __uint_as_float(sr[b][0]);
#pragma unroll
    for (int k = 1; k < 31; k += 2) mb = max3(mb, __uint_as_float(sr[b][k]), __uint_as_float(sr[b][k + 1]));
    mb = fmaxf(mb, __uint_as_float(sr[b][31]));
    // the scale is >= 0, so the block maximum of S * c is c times that of S
    const float xb = mb * cb[b];
    mt = fmaxf(mt, (kTail && mb == -INFINITY) ? -INFINITY : xb);
  }
  const float m_new = fmaxf(m, mt);
  const bool grew = m_new > m;
  const float alpha = ex2(m - m_new);  // 0 on the first tile
  const float neg = kLog2P - m_new;
  const float2 n2 = make_float2(neg, neg);
  float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
  uint32_t pw[32];  // e4m3 P of the row: word k holds keys 4k..4k+3
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const float2 c2 = make_float2(cb[b], cb[b]);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float2 x01 = __ffma2_rn(make_float2(__uint_as_float(sr[b][4 * k]), __uint_as_float(sr[b][4 * k + 1])),
                                    c2, n2);
      const float2 x23 = __ffma2_rn(
          make_float2(__uint_as_float(sr[b][4 * k + 2]), __uint_as_float(sr[b][4 * k + 3])), c2, n2);
      float2 p01 = make_float2(ex2(x01.x), ex2(x01.y));
      float2 p23 = make_float2(ex2(x23.x), ex2(x23.y));
      if (kTail) {
        const int c0 = 32 * b + 4 * k;
        if (c0 >= nvalid) p01.x = 0.f;
        if (c0 + 1 >= nvalid) p01.y = 0.f;
        if (c0 + 2 >= nvalid) p23.x = 0.f;
        if (c0 + 3 >= nvalid) p23.y = 0.f;
      }
      sa = __fadd2_rn(sa, p01);
      sb = __fadd2_rn(sb, p23);
      pw[8 * b + k] = e4m3x2(p01.y, p01.x) | (e4m3x2(p23.y, p23.x) << 16);
    }
  }
  l = l * alpha + ((sa.x + sa.y) + (sb.x + sb.y));
  m = m_new;
  if constexpr (D == 64) {
    // P of this step into its buffer: the PV that last read it (two steps
    // back) completed before the previous step's wait below returned, and the
    // unit's last PV before the unit's epilogue
    tc::tmem_st32(tP, pw);
    if (!first) {
      // the previous PV must be done with O before the rescale
      if (!wait_bar_warp(cx, cx.bar(kBarPVDone + i), pv_cnt & 1u)) return false;
      ++pv_cnt;
      tc::tc_fence_after();
      if (__any_sync(0xffffffffu, grew)) {
        uint32_t o[D / 32][32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tc::tmem_ld32(tO + 32u * c, o[c]);
        tc::tmem_wait_ld();
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float2 r = __fmul2_rn(make_float2(__uint_as_float(o[c][k]), __uint_as_float(o[c][k + 1])), a2);
            o[c][k] = __float_as_uint(r.x);
            o[c][k + 1] = __float_as_uint(r.y);
          }
          tc::tmem_st32(tO + 32u * c, o[c]);
        }
      }
    }
    tc::tmem_wait_st();  // P (and O) written before the caller signals the MMA issuer
    return true;
  }
  // the previous PV of this tile must be done with P (shared memory) and O
  if (!first) {
    if (!wait_bar_warp(cx, cx.bar(kBarPVDone + i), pv_cnt & 1u)) return false;
    ++pv_cnt;
    tc::tc_fence_after();
    if constexpr (kCorr) {
      // the correction warp of this row rescales O by alpha while P is stored
      alpha_row[0] = alpha;
      tc::mbar_arrive(cx.bar(kBarAlpha + i));
    }
  }
  // P row: 128 bytes, 16-byte chunk c at (c ^ (row & 7)) (128-byte swizzle)
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4*>(p_row + ((c ^ (row & 7)) << 4)) =
        make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
  tc::fence_proxy_async_smem();
  if constexpr (!kCorr) {
    // O rescaled here, when some row of the warp's 32 grew (alpha = 1 exactly otherwise)
    if (!first && __any_sync(0xffffffffu, grew)) {
      uint32_t o[D / 32][32];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tc::tmem_ld32(tO + 32u * c, o[c]);
      tc::tmem_wait_ld();
      const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const float2 r = __fmul2_rn(make_float2(__uint_as_float(o[c][k]), __uint_as_float(o[c][k + 1])), a2);
          o[c][k] = __float_as_uint(r.x);
          o[c][k + 1] = __float_as_uint(r.y);
        }
        tc::tmem_st32(tO + 32u * c, o[c]);
      }
      tc::tmem_wait_st();
    }
  }
  return true;
}

// D: the head dimension (128 or 64). kCausal: the causal mask (a separate
// instantiation, so the unmasked kernel carries none of its branches).
template <int D, bool kCausal, bool kCorr>
__global__ void __launch_bounds__(threads_of<kCorr>(), 1)
    attention_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const Params prm,
                        const __grid_constant__ SchedOf<kCausal> sched) {
  using L = Smem<D>;
  using T = SmemTail<D>;
  // the 128-byte-swizzled operand tiles need 1024-byte alignment, which the
  // declaration asks for (there is no room left for realignment slack)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((tc::smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicExch(prm.dev_err, kDevErrSmemAlign);
    return;
  }
  uint8_t* smem = smem_raw;
  const uint32_t sbase = tc::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctx cx;
  cx.bar0 = sbase + L::kOffBar;
  cx.abort_flag = reinterpret_cast<volatile int*>(smem + T::kOffAbort);
  cx.dev_err = prm.dev_err;

  if (threadIdx.x == 0) {
    *cx.abort_flag = 0;
    tc::mbar_init(cx.bar(kBarQFull), 1);
    // the MMA issuers of the unit's query tiles release Q, K and V stages
    const uint32_t issuers = static_cast<uint32_t>(prm.tiles);
    tc::mbar_init(cx.bar(kBarQEmpty), issuers);
    for (int s = 0; s < kKStages; ++s) {
      tc::mbar_init(cx.bar(kBarKFull + s), 1);
      tc::mbar_init(cx.bar(kBarKEmpty + s), issuers);
    }
    for (int s = 0; s < kVStages; ++s) {
      tc::mbar_init(cx.bar(kBarVFull + s), 1);
      tc::mbar_init(cx.bar(kBarVEmpty + s), issuers);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(cx.bar(kBarSFull + s), 1);
      tc::mbar_init(cx.bar(kBarSFree + s), 128);
      tc::mbar_init(cx.bar(kBarPFull + s), 128);
      tc::mbar_init(cx.bar(kBarPVDone + s), 1);
      tc::mbar_init(cx.bar(kBarOEmpty + s), 128);
      tc::mbar_init(cx.bar(kBarDrain + s), 1);
      tc::mbar_init(cx.bar(kBarVs + s), 128);
      tc::mbar_init(cx.bar(kBarORdy + s), 128);
      tc::mbar_init(cx.bar(kBarAlpha + s), 128);
    }
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(sbase + T::kOffTmemSlot, kTmemCols);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tm_q);
    tc::prefetch_tmap(&tm_k);
    tc::prefetch_tmap(&tm_v);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + T::kOffTmemSlot);
  // launched as a programmatic dependent: the previous kernel of the stream
  // (which writes the bundle, or reads the output buffer) must be complete
  // before any global memory is touched
  tc::griddep_wait();

  if (warp < 4) {
    // control warpgroup: one register decrease for all four warps
    regs_dec<Regs<kCorr>::ctl>();
    if (warp == 0) {
      // ---------------------------------------------------------- producer --
      if (lane == 0) {
        uint32_t k_cnt = 0, v_cnt = 0, u_cnt = 0;
        int k_pending[kKStages], v_pending[kVStages], q_pending = -1;
        for (int s = 0; s < kKStages; ++s) k_pending[s] = -1;
        for (int s = 0; s < kVStages; ++s) v_pending[s] = -1;
        bool ok = true;
        for (int64_t uk = 1, u = first_unit<kCausal>(sched); ok && unit_valid<kCausal>(prm, sched, u);
         u = next_unit<kCausal>(sched, u, uk++)) {
          const int32_t bh = static_cast<int32_t>(u / prm.pairs_per_head);
          const int64_t qt0 = (u % prm.pairs_per_head) * prm.tiles;  // the unit's first query tile
          const int32_t q_row0 = static_cast<int32_t>(qt0 * 128);
          // the unit's query tiles (two 64-channel boxes each)
          if (!(ok = wait_bar(cx, cx.bar(kBarQEmpty), (u_cnt & 1u) ^ 1u))) break;
          tc::mbar_arrive_expect_tx(cx.bar(kBarQFull), static_cast<uint32_t>(prm.tiles) * L::kTile16);
          for (int t = 0; t < prm.tiles; ++t)
#pragma unroll
            for (int x = 0; x < D / 64; ++x)
              tc::tma_load_3d(sbase + L::kOffQ16 + t * L::kTile16 + x * kSub16, &tm_q, 64 * x, q_row0 + 128 * t, bh,
                              cx.bar(kBarQFull));
          q_pending = static_cast<int>(u_cnt & 1u);
          ++u_cnt;
          // the unit's key tiles: those of its last query tile, which sees the most
          const int64_t n_kv_u = key_tiles<kCausal>(prm, qt0 + prm.tiles - 1);
          for (int64_t j = 0; ok && j < n_kv_u; ++j) {
            const uint32_t ks = k_cnt % kKStages, kph = (k_cnt / kKStages) & 1u;
            if (!(ok = wait_bar(cx, cx.bar(kBarKEmpty + ks), kph ^ 1u))) break;
            tc::mbar_arrive_expect_tx(cx.bar(kBarKFull + ks), L::kTile16);
#pragma unroll
            for (int x = 0; x < D / 64; ++x)
              tc::tma_load_3d(sbase + L::kOffK16 + ks * L::kTile16 + x * kSub16, &tm_k, 64 * x,
                              static_cast<int32_t>(j) * 128, bh, cx.bar(kBarKFull + ks));
            k_pending[ks] = static_cast<int>(kph);
            ++k_cnt;
            const uint32_t vs = v_cnt % kVStages, vph = (v_cnt / kVStages) & 1u;
            if (!(ok = wait_bar(cx, cx.bar(kBarVEmpty + vs), vph ^ 1u))) break;
            tc::mbar_arrive_expect_tx(cx.bar(kBarVFull + vs), L::kTileV);
            tc::tma_load_3d(sbase + L::kOffV + vs * L::kTileV, &tm_v, static_cast<int32_t>(j) * 128, 0, bh,
                            cx.bar(kBarVFull + vs));
            v_pending[vs] = static_cast<int>(vph);
            ++v_cnt;
          }
        }
        if (!ok) {
          // let every copy this thread issued land before the CTA exits
          Ctx drain = cx;
          volatile int no_abort = 0;
          drain.abort_flag = &no_abort;
          if (q_pending >= 0) wait_bar(drain, cx.bar(kBarQFull), static_cast<uint32_t>(q_pending));
          for (int s = 0; s < kKStages; ++s)
            if (k_pending[s] >= 0) wait_bar(drain, cx.bar(kBarKFull + s), static_cast<uint32_t>(k_pending[s]));
          for (int s = 0; s < kVStages; ++s)
            if (v_pending[s] >= 0) wait_bar(drain, cx.bar(kBarVFull + s), static_cast<uint32_t>(v_pending[s]));
        }
      }
    } else if (warp <= 2) {
      // ---------------------------------------------- MMA issuer of tile i --
      // The whole warp runs the loop (warp-uniform control flow keeps the
      // descriptors and counters in uniform registers); one elected lane
      // issues the MMAs and commits.
      const int i = warp - 1;
      const bool leader = elect_one();
      const uint32_t d_s = tmem + col_s(i), d_o = tmem + col_o<D>(i);
      const uint64_t dq = tc::sw128_desc(sbase + L::kOffQ16 + static_cast<uint32_t>(i) * L::kTile16);
      const uint64_t dk0 = tc::sw128_desc(sbase + L::kOffK16);
      const uint64_t dv0 = tc::sw128_desc(sbase + L::kOffV);
      const uint64_t dp = tc::sw128_desc(sbase + L::kOffP + static_cast<uint32_t>(i) * kTile8);
      uint32_t k_cnt = 0, v_cnt = 0, u_cnt = 0, sf_cnt = 0, p_cnt = 0, o_cnt = 0;
      bool ok = i < prm.tiles;  // with one query tile per unit the second issuer has no work
      for (int64_t uk = 1, u = first_unit<kCausal>(sched); ok && unit_valid<kCausal>(prm, sched, u);
         u = next_unit<kCausal>(sched, u, uk++)) {
        if (!(ok = wait_bar_warp(cx, cx.bar(kBarQFull), u_cnt & 1u))) break;
        // this tile's key tiles, and the unit's (the ring carries the larger
        // count; a tile releases the stages it does not use without an MMA)
        const int64_t qt0 = (u % prm.pairs_per_head) * prm.tiles, qt = qt0 + i;
        const int64_t n_kv_i = key_tiles<kCausal>(prm, qt), n_kv_u = key_tiles<kCausal>(prm, qt0 + prm.tiles - 1);
        for (int64_t j = 0; ok && j <= n_kv_u; ++j) {
          if (j < n_kv_u) {
            // QK_j once K_j is loaded and the softmax has read S_{j-1}
            const uint32_t ks = k_cnt % kKStages;
            if (!(ok = wait_bar_warp(cx, cx.bar(kBarKFull + ks), (k_cnt / kKStages) & 1u))) break;
            if (j < n_kv_i) {
              if (u_cnt > 0 || j > 0) {
                if (!(ok = wait_bar_warp(cx, cx.bar(kBarSFree + i), sf_cnt & 1u))) break;
                ++sf_cnt;
              }
              tc::tc_fence_after();
              if (leader) {
                issue_qk<D>(d_s, dq, desc_at(dk0, ks * L::kTile16));
                tc::mma_commit(cx.bar(kBarSFull + i));
                tc::mma_commit(cx.bar(kBarKEmpty + ks));
                if (j == n_kv_i - 1) tc::mma_commit(cx.bar(kBarQEmpty));
              }
            } else if (leader) {
              tc::mbar_arrive(cx.bar(kBarKEmpty + ks));  // masked for this tile
            }
            __syncwarp();
            ++k_cnt;
          }
          if (j >= 1) {
            // PV_{j-1} once P_{j-1} is in shared memory (and O rescaled)
            const int64_t jj = j - 1;
            const uint32_t vs = v_cnt % kVStages;
            if (!(ok = wait_bar_warp(cx, cx.bar(kBarVFull + vs), (v_cnt / kVStages) & 1u))) break;
            if (jj < n_kv_i) {
              if (!(ok = wait_bar_warp(cx, cx.bar(kBarPFull + i), p_cnt & 1u))) break;
              ++p_cnt;
              if (jj == 0 && !(ok = wait_bar_warp(cx, cx.bar(kBarOEmpty + i), (u_cnt & 1u) ^ 1u))) break;
              if (kCorr && jj > 0) {
                if (!(ok = wait_bar_warp(cx, cx.bar(kBarORdy + i), o_cnt & 1u))) break;
                ++o_cnt;
              }
              tc::tc_fence_after();
              if (leader) {
                issue_pv<D>(d_o, dp, tmem + col_p(i, static_cast<int>(jj & 1)), desc_at(dv0, vs * L::kTileV), jj > 0);
                tc::mma_commit(cx.bar(kBarPVDone + i));
                tc::mma_commit(cx.bar(kBarVEmpty + vs));
              }
            } else if (leader) {
              tc::mbar_arrive(cx.bar(kBarVEmpty + vs));  // masked for this tile
            }
            __syncwarp();
            ++v_cnt;
          }
        }
        ++u_cnt;
      }
      // drain: all MMAs issued by this warp complete before TMEM is freed
      if (leader) tc::mma_commit(cx.bar(kBarDrain + i));
      __syncwarp();
      Ctx drain = cx;
      volatile int no_abort = 0;
      drain.abort_flag = &no_abort;
      wait_bar(drain, cx.bar(kBarDrain + i), 0);
    }
    __syncwarp();
  } else if (kCorr && warp >= 12) {
    // ----------------------------------------------------------- correction --
    // O_i *= alpha before PV_j of tile i (j >= 1), rows whose maximum grew;
    // the softmax thread of the row posts alpha once PV_{j-1} is done
    regs_dec<Regs<kCorr>::corr>();
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    const float* alpha_buf = reinterpret_cast<const float*>(smem + T::kOffAlpha);
    uint32_t a_cnt[2] = {0u, 0u}, pv_cnt[2] = {0u, 0u};
    bool ok = true;
    for (int64_t uk = 1, u = first_unit<kCausal>(sched); ok && unit_valid<kCausal>(prm, sched, u);
         u = next_unit<kCausal>(sched, u, uk++)) {
      const int64_t qt0 = (u % prm.pairs_per_head) * prm.tiles;
      int64_t n_kv[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) n_kv[i] = i < prm.tiles ? key_tiles<kCausal>(prm, qt0 + i) : 0;
      const int64_t n_max = key_tiles<kCausal>(prm, qt0 + prm.tiles - 1);
      for (int64_t j = 1; ok && j < n_max; ++j) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (i >= prm.tiles || j >= n_kv[i]) continue;
          if (!(ok = wait_bar_warp(cx, cx.bar(kBarAlpha + i), a_cnt[i] & 1u))) break;
          ++a_cnt[i];
          // PV_{j-1} is complete (the softmax thread saw it before posting)
          if (!(ok = wait_bar_warp(cx, cx.bar(kBarPVDone + i), pv_cnt[i] & 1u))) break;
          ++pv_cnt[i];
          tc::tc_fence_after();
          const float alpha = alpha_buf[i * 128 + row];
          if (__any_sync(0xffffffffu, alpha != 1.0f)) {
            const uint32_t tO = tmem + lane_addr + col_o<D>(i);
            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tc::tmem_ld32(tO + 32u * c, o);
              tc::tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 32; k += 2) {
                const float2 r = __fmul2_rn(make_float2(__uint_as_float(o[k]), __uint_as_float(o[k + 1])), a2);
                o[k] = __float_as_uint(r.x);
                o[k + 1] = __float_as_uint(r.y);
              }
              tc::tmem_st32(tO + 32u * c, o);
            }
            tc::tmem_wait_st();
          }
          tc::tc_fence_before();
          tc::mbar_arrive(cx.bar(kBarORdy + i));
        }
      }
      // the unit's last PV of each tile completes a phase this warp does not wait for
#pragma unroll
      for (int i = 0; i < 2; ++i) pv_cnt[i] += i < prm.tiles ? 1u : 0u;
    }
    regs_inc<Regs<kCorr>::ctl>();  // the teardown runs with the control budget in every warp
  } else {
    // -------------------------------------------------------------- softmax --
    regs_inc<Regs<kCorr>::softmax>();
    const int i = (warp - 4) >> 2;        // query tile of this warpgroup
    const int wq = warp & 3;              // TMEM lane quarter
    const int row = wq * 32 + lane;       // row within the query tile
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_addr + col_s(i);
    const uint32_t tO = tmem + lane_addr + col_o<D>(i);
    const uint32_t tP0 = tmem + lane_addr + col_p(i, 0);  // D = 64: this row's P buffers
    uint8_t* p_row = smem + L::kOffP + static_cast<uint32_t>(i) * kTile8 + row * 128;
    float* alpha_row = reinterpret_cast<float*>(smem + T::kOffAlpha) + i * 128 + row;
    const int64_t nblk = prm.S_pad / kQKBlock;
    uint32_t s_cnt = 0, pv_cnt = 0, vs_cnt = 0;
    bool ok = i < prm.tiles;  // with one query tile per unit the second warpgroup has no work
    for (int64_t uk = 1, u = first_unit<kCausal>(sched); ok && unit_valid<kCausal>(prm, sched, u);
         u = next_unit<kCausal>(sched, u, uk++)) {
      const int64_t bh = u / prm.pairs_per_head;
      const int64_t qt = (u % prm.pairs_per_head) * prm.tiles + i;  // this query tile
      const int64_t qrow = qt * 128 + row;                             // query index in the head
      const bool row_valid = qrow < prm.S;
      const float cq = row_valid ? prm.q_scale[bh * nblk + qrow / kQKBlock] * prm.sm_log2 : 0.0f;
      const float* ks = prm.k_scale + bh * nblk;
      // the V scale of channel `row` (the first D threads) is copied into
      // shared memory now, asynchronously, for the epilogue; the previous
      // unit's epilogue has finished reading the buffer in every thread of
      // the warpgroup once the O-empty barrier of that unit completes (all
      // 128 threads arrive on it after their last read)
      float* vs_buf = reinterpret_cast<float*>(smem + T::kOffVs) + i * D;
      if (vs_cnt > 0 && !(ok = wait_bar_warp(cx, cx.bar(kBarOEmpty + i), (vs_cnt - 1) & 1u))) break;
      if (row < D) tc::cp_async4(tc::smem_u32(vs_buf + row), prm.v_scale + bh * D + row);
      float m = -INFINITY, l = 0.0f;
      float cb[4];
      // K scales of a 128-key tile: 4 consecutive floats, 16-byte aligned
      // (S_pad / 32 is a multiple of 4)
      float4 ks_next = __ldg(reinterpret_cast<const float4*>(ks));
      const int64_t n_kv_i = key_tiles<kCausal>(prm, qt);
      for (int64_t j = 0; j < n_kv_i; ++j) {
        cb[0] = cq * ks_next.x;
        cb[1] = cq * ks_next.y;
        cb[2] = cq * ks_next.z;
        cb[3] = cq * ks_next.w;
        // the next tile's scales load while this tile is processed
        if (j + 1 < n_kv_i) ks_next = __ldg(reinterpret_cast<const float4*>(ks + (j + 1) * 4));
        if (!(ok = wait_bar_warp(cx, cx.bar(kBarSFull + i), s_cnt & 1u))) break;
        ++s_cnt;
        tc::tc_fence_after();
        // keys of this tile the row may see: those below S and, on the
        // diagonal tile of the causal mask, those at or before the row. The
        // choice of path must be the same in every lane (the tile code is
        // warp-collective), so a tile with any limit takes the masked path
        // in all lanes, each with its own limit.
        const int64_t below_s = prm.S - j * kKeyTile;
        const bool diagonal = kCausal && j == qt;
        int64_t lim = below_s < kKeyTile ? below_s : kKeyTile;
        if (diagonal && lim > row + 1) lim = row + 1;
        ok = !(diagonal || below_s < kKeyTile)
                 ? softmax_tile<D, false, kCorr>(cx, i, tS, tO, tP0 + 32u * static_cast<uint32_t>(j & 1), alpha_row,
                                                 p_row, row, cb, kKeyTile, j == 0, pv_cnt, m, l)
                 : softmax_tile<D, true, kCorr>(cx, i, tS, tO, tP0 + 32u * static_cast<uint32_t>(j & 1), alpha_row,
                                                p_row, row, cb, static_cast<int>(lim), j == 0, pv_cnt, m, l);
        if (!ok) break;
        tc::tc_fence_before();
        tc::mbar_arrive(cx.bar(kBarPFull + i));
      }
      if (!ok) break;
      // epilogue: the last PV of the unit completes O; O = acc * s_v / l (l
      // counts p448), bf16 in the output layout
      tc::cp_async_wait_all();
      tc::mbar_arrive(cx.bar(kBarVs + i));
      if (!(ok = wait_bar_warp(cx, cx.bar(kBarPVDone + i), pv_cnt & 1u))) break;
      ++pv_cnt;
      if (!(ok = wait_bar_warp(cx, cx.bar(kBarVs + i), vs_cnt & 1u))) break;
      ++vs_cnt;
      tc::tc_fence_after();
      const float inv_l = 1.0f / l;
      if (prm.lse != nullptr && row_valid) {
        // ln(sum_j e^logit) = (m + log2(l) - log2(448)) * ln 2, m and the
        // logits in base 2, l counting 448 * 2^(x - m)
        prm.lse[bh * prm.S + qrow] = (m + log2f(l) - kLog2P) * kLn2;
      }
      // Each warp writes its 32 rows through its 4 KB of this warpgroup's P
      // tile (free once the last PV is done): a lane parks its row's 64
      // bytes of a 32-channel slice, then each store instruction covers 8
      // rows x 64 contiguous bytes instead of 32 rows x 16 bytes. The 16-byte
      // chunk q of staged row r sits at slot (q + r / 2) & 3, so that both
      // the parking and the reading are free of bank conflicts.
      const int64_t b_idx = bh / prm.H, h_idx = bh % prm.H;
      const int64_t row0 = qrow - lane;  // this warp's first row
      uint8_t* stage = smem + L::kOffP + static_cast<uint32_t>(i) * kTile8 + static_cast<uint32_t>(wq) * 4096u;
      const int rr = lane >> 2, qq = lane & 3;  // the row (of 8) and chunk this lane stores
      uint16_t* dst[4];
      bool dst_ok[4];
#pragma unroll
      for (int mm = 0; mm < 4; ++mm) {
        const int64_t r = row0 + 8 * mm + rr;
        dst_ok[mm] = r < prm.S;
        dst[mm] = prm.out.p + b_idx * prm.out.sb + r * prm.out.ss + h_idx * prm.out.sh + 8 * qq;
      }
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tc::tmem_ld32(tO + 32u * c, o);
        tc::tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 s2 = *reinterpret_cast<const float2*>(vs_buf + 32 * c + 2 * k);
          const float a0 = __uint_as_float(o[2 * k]) * inv_l * s2.x;
          const float a1 = __uint_as_float(o[2 * k + 1]) * inv_l * s2.y;
          const __nv_bfloat162 v2 = __floats2bfloat162_rn(a0, a1);
          pk[k] = *reinterpret_cast<const uint32_t*>(&v2);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(stage + lane * 64 + ((q + (lane >> 1)) & 3) * 16) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        __syncwarp();
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
          const int r = 8 * mm + rr;
          const uint4 val = *reinterpret_cast<const uint4*>(stage + r * 64 + ((qq + (r >> 1)) & 3) * 16);
          if (dst_ok[mm]) *reinterpret_cast<uint4*>(dst[mm] + 32 * c) = val;
        }
        __syncwarp();
      }
      tc::tc_fence_before();
      tc::mbar_arrive(cx.bar(kBarOEmpty + i));
    }
    regs_dec<Regs<kCorr>::ctl>();  // the teardown runs with the control budget in every warp
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// The bounded wait put to the test: the only warp waits on a barrier that
// nothing arrives on (phase 0 of a fresh mbarrier never completes); after the
// wait's limit it flags the device error word and the kernel ends, with the
// context still usable.
__global__ void __launch_bounds__(32, 1) wait_timeout_selftest_kernel(int* dev_err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  Ctx cx;
  cx.bar0 = tc::smem_u32(&bar);
  cx.abort_flag = reinterpret_cast<volatile int*>(&abort_flag);
  cx.dev_err = dev_err;
  if (threadIdx.x == 0) {
    *cx.abort_flag = 0;
    tc::mbar_init(cx.bar(0), 1);
    tc::fence_mbar_init();
  }
  __syncwarp();
  wait_bar_warp(cx, cx.bar(0), 0);
}

// 3-D tensor [d2][d1][d0] of `esize`-byte elements; boxes of box0 x box1 x 1
// elements with the 128-byte swizzle (box0 * esize must be 128).
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, uint32_t esize, const void* base, uint64_t d0, uint64_t d1,
              uint64_t d2, uint32_t box0, uint32_t box1) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint64_t strides[2] = {d0 * esize, d0 * d1 * esize};
  const uint32_t box[3] = {box0, box1, 1};
  return make_tmap(m, dt, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// The causal schedule for (units, pairs per head, key tiles, grid), built once
// and kept (a handful of shapes). Null when the table cannot hold it.
const Sched* causal_schedule(int64_t n_units, int64_t pairs, int64_t n_kv, int grid) {
  if (n_units > kSchedMaxUnits || grid > kSchedMaxCtas || grid <= 0) return nullptr;
  struct Entry {
    int64_t n_units, pairs, n_kv;
    int grid;
    std::unique_ptr<Sched> sched;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : cache)
    if (e.n_units == n_units && e.pairs == pairs && e.n_kv == n_kv && e.grid == grid) return e.sched.get();
  constexpr int64_t kWindowHeads = 4;  // heads whose units are ordered together
  constexpr int64_t kUnitOverhead = 2; // fixed cost of a unit, in key tiles
  const int64_t heads = n_units / pairs;
  std::vector<int64_t> order;
  order.reserve(static_cast<size_t>(n_units));
  for (int64_t h0 = 0; h0 < heads; h0 += kWindowHeads)
    for (int64_t pp = pairs - 1; pp >= 0; --pp)
      for (int64_t h = h0; h < std::min(heads, h0 + kWindowHeads); ++h) order.push_back(h * pairs + pp);
  // longest processing time first: each unit to the least loaded CTA
  std::vector<std::pair<int64_t, int>> heap;  // (-load, -cta): std heaps are max-heaps
  for (int c = 0; c < grid; ++c) heap.emplace_back(0, -c);
  std::make_heap(heap.begin(), heap.end());
  std::vector<std::vector<uint16_t>> per(static_cast<size_t>(grid));
  for (int64_t u : order) {
    std::pop_heap(heap.begin(), heap.end());
    auto top = heap.back();
    heap.pop_back();
    const int c = -top.second;
    per[static_cast<size_t>(c)].push_back(static_cast<uint16_t>(u));
    const int64_t tiles = std::min(n_kv, 2 * (u % pairs) + 2);
    heap.emplace_back(top.first - (tiles + kUnitOverhead), top.second);
    std::push_heap(heap.begin(), heap.end());
  }
  std::unique_ptr<Sched> sc(new Sched());
  sc->n = static_cast<int32_t>(n_units);
  int64_t pos = 0;
  for (int c = 0; c < grid; ++c) {
    sc->start[c] = static_cast<uint16_t>(pos);
    for (uint16_t u : per[static_cast<size_t>(c)]) sc->unit[pos++] = u;
  }
  sc->start[grid] = static_cast<uint16_t>(pos);
  if (cache.size() >= 16) cache.erase(cache.begin());
  cache.push_back(Entry{n_units, pairs, n_kv, grid, std::move(sc)});
  return cache.back().sched.get();
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int* dev_err, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(dev_err);
  return cudaGetLastError();
}

cudaError_t launch_attention_tc(const Bundle& in, int64_t B, int64_t S, int64_t H, int64_t D, float sm_scale,
                                const Out& out, bool causal, float* lse, int* dev_err, cudaStream_t stream) {
  if (D != 128 && D != 64) return cudaErrorInvalidValue;
  const int64_t S_pad = padded_len(S);
  const int64_t BH = B * H;
  CUtensorMap tq, tk, tv;
  const uint64_t d = static_cast<uint64_t>(D);
  if (!make_map(&tq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, in.q16, d, static_cast<uint64_t>(S_pad),
                static_cast<uint64_t>(BH), 64, 128) ||
      !make_map(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, in.k16, d, static_cast<uint64_t>(S_pad),
                static_cast<uint64_t>(BH), 64, 128) ||
      !make_map(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, in.vt_codes, static_cast<uint64_t>(S_pad), d,
                static_cast<uint64_t>(BH), 128, static_cast<uint32_t>(D)))
    return cudaErrorInvalidValue;
  Params p;
  p.S = S;
  p.S_pad = S_pad;
  p.n_kv = S_pad / kKeyTile;
  const int sms = sm_count_current();
  // one query tile per unit when that still fits the GPU in one wave (short
  // sequences: twice the CTAs, each with half the chain); pairs otherwise,
  // and always with the causal mask (its schedule is built on pairs)
  p.tiles = (!causal && BH * (S_pad / 128) <= sms) ? 1 : 2;
  p.pairs_per_head = div_up(S_pad / 128, p.tiles);
  p.n_units = BH * p.pairs_per_head;
  p.q_scale = in.q_scale;
  p.k_scale = in.k_scale;
  p.v_scale = in.v_scale;
  p.out = out;
  p.H = H;
  p.sm_log2 = sm_scale * kLog2e;
  p.lse = lse;
  p.dev_err = dev_err;
  const uint32_t smem_bytes = D == 128 ? SmemTail<128>::kBytes : SmemTail<64>::kBytes;
  const int grid = static_cast<int>(p.n_units < sms ? p.n_units : sms);
  // programmatic dependent launch: the CTAs may start (barriers, TMEM,
  // tensor maps) while the previous kernel of the stream, normally the
  // prologue, still runs; they wait for it before reading anything
  // the correction warpgroup pays off for unmasked rows of 2048 keys or more
  // at D = 128 (measured: -1.4% to -2.9% from S = 2048 to 32768, even at
  // S = 1024); with the causal mask (+11%) and at D = 64 (+3%) the rescale in
  // the softmax warps ran faster
  const bool corr = !causal && D == 128 && p.n_kv >= kCorrMinKeyTiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(corr ? threads_of<true>() : threads_of<false>()));
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (!causal) {
    auto kernel = corr ? attention_tc_kernel<128, false, true>
                       : (D == 128 ? attention_tc_kernel<128, false, false> : attention_tc_kernel<64, false, false>);
    if ((e = set_smem_limit_once(reinterpret_cast<const void*>(kernel), static_cast<int>(smem_bytes))) !=
        cudaSuccess)
      return e;
    return cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, p, NoSched{});
  }
  auto kernel = D == 128 ? attention_tc_kernel<128, true, false> : attention_tc_kernel<64, true, false>;
  if ((e = set_smem_limit_once(reinterpret_cast<const void*>(kernel), static_cast<int>(smem_bytes))) != cudaSuccess)
    return e;
  const Sched* sc = causal_schedule(p.n_units, p.pairs_per_head, p.n_kv, grid);
  static const Sched round_robin = [] {
    Sched r{};
    r.n = 0;
    return r;
  }();
  return cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, p, sc != nullptr ? *sc : round_robin);
}

}  // namespace sage
