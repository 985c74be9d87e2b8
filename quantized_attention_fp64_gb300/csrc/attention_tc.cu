// Quantized flash attention on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// Method: "aiter-sage-attention: SageAttention for AMD RDNA4 (gfx1201)
// #1222", section "The kernel": QK^T in INT8 and PV in FP8, both with FP32
// accumulation; Q/K scales per 32-token block, V scales per channel.
//
// INT8 QK^T. sm_103a has no integer tcgen05 MMA, so the int8 codes are widened
// exactly to fp16 (every integer in [-127, 127] is an fp16 value) and
// multiplied with kind::f16 into an fp32 accumulator in TMEM. Each product is
// an integer of magnitude <= 127^2 and every partial sum of the 128 products
// stays below 2^21, so the fp32 accumulation is exact: S_ij equals the INT32
// dot product of the codes bit for bit.
//
// FP8 PV. P is quantized to e4m3 as e4m3(448 p) and written into TMEM over
// the first 32 columns of its own S tile; it is the A operand of a
// kind::f8f6f4 MMA whose B operand is the transposed e4m3 V tile in shared
// memory. O accumulates in fp32 in TMEM.
//
// Schedule (one persistent CTA per SM, 384 threads):
//   warp 0      TMA producer: int8 Q and K tiles into a 2-stage ring, e4m3
//               V^T tiles into a 3-stage ring (128-byte swizzled boxes).
//   warp 1      TMEM allocator and the single MMA-issuing thread.
//   warps 2-3   convert int8 Q/K tiles to fp16 in the 128-byte swizzled
//               K-major layout the MMA reads.
//   warps 4-7   softmax for query tile 0 (TMEM lanes 0..127 = its 128 rows).
//   warps 8-11  softmax for query tile 1.
// A work unit is one (batch, head) and a pair of 128-row query tiles; the two
// softmax warpgroups alternate with the tensor core (while one computes P for
// its tile the MMAs of the other run). TMEM holds S0, S1, O0, O1 (4 x 128
// columns of fp32). The softmax is online over 128-key tiles in ascending
// order with the exact running maximum; a row's O is rescaled only when its
// maximum grows (the factor is exactly 1 otherwise). Logits are kept in base
// 2: x = S * (s_q * sm_scale * log2 e) * s_k, and p448 = 2^(x - m + log2 448)
// is both the e4m3 input and the row-sum term, so the epilogue computes
// O = acc * s_v / l.
//
// Every wait on an mbarrier is bounded; when one runs out the kernel sets the
// device error word, tells the other roles to stop, lets its own copies and
// MMAs drain, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace sage {
namespace {

constexpr int kThreads = 384;
constexpr int kK8Stages = 2;
constexpr int kVStages = 3;
constexpr uint32_t kTile8 = 128 * 128;       // bytes of one int8 / e4m3 tile
constexpr uint32_t kTile16 = 128 * 128 * 2;  // bytes of one fp16 tile (two 64-channel subtiles)
constexpr uint32_t kSub16 = 128 * 128;       // bytes of one 64-channel fp16 subtile

// shared memory layout (offsets from a 1024-aligned base)
constexpr uint32_t kOffQ16 = 0;                                  // 2 tiles
constexpr uint32_t kOffK16 = kOffQ16 + 2 * kTile16;              // 2 buffers
constexpr uint32_t kOffK8 = kOffK16 + 2 * kTile16;               // ring
constexpr uint32_t kOffV = kOffK8 + kK8Stages * kTile8;          // ring
constexpr uint32_t kOffBar = kOffV + kVStages * kTile8;
// barriers (8 bytes each)
constexpr int kBarK8Full = 0, kBarK8Empty = kBarK8Full + kK8Stages;
constexpr int kBarVFull = kBarK8Empty + kK8Stages, kBarVEmpty = kBarVFull + kVStages;
constexpr int kBarK16Full = kBarVEmpty + kVStages, kBarK16Empty = kBarK16Full + 2;
constexpr int kBarQ16Full = kBarK16Empty + 2, kBarQ16Empty = kBarQ16Full + 1;
constexpr int kBarSFull = kBarQ16Empty + 1, kBarPFull = kBarSFull + 2;
constexpr int kBarOFull = kBarPFull + 2, kBarOEmpty = kBarOFull + 2;
constexpr int kBarDrain = kBarOEmpty + 2;
constexpr int kNumBars = kBarDrain + 1;
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemSlot + 8;
constexpr uint32_t kSmemBytes = kOffAbort + 8 + 1024;  // + alignment slack

// TMEM columns: S of query tile i at 128*i, O of query tile i at 256 + 128*i
__host__ __device__ constexpr uint32_t col_s(int i) { return 128u * static_cast<uint32_t>(i); }
__host__ __device__ constexpr uint32_t col_o(int i) { return 256u + 128u * static_cast<uint32_t>(i); }
constexpr uint32_t kTmemCols = 512;

constexpr int kConvThreads = 64;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLog2P = 8.807354922057604f;    // log2(448)

struct Params {
  int64_t S, S_pad, n_kv, pairs_per_head, n_units;
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  Out out;
  int64_t H;
  float sm_log2;  // sm_scale * log2(e)
  int* dev_err;
};

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

// int8 x4 (one word) -> two fp16x2 words, exactly: fp16 bits 0x6400 | (c ^ 0x80)
// is 1024 + c + 128, and subtracting 1152 leaves c.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(x, 0x64646464u, 0x5140);
  const uint32_t b = __byte_perm(x, 0x64646464u, 0x7362);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

// One int8 tile (TMA box of 128 rows x 128 bytes, 128-byte swizzled) to fp16
// in two K-major 128-byte-swizzled subtiles (channels 0-63 and 64-127).
// `ct` in [0, 64) indexes the converting threads.
__device__ __forceinline__ void convert_tile(const uint8_t* src, uint8_t* dst, int ct) {
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int id = i * kConvThreads + ct;
    const int r = id >> 3, c = id & 7;  // row, 16-byte chunk (channels 16c..16c+15)
    const uint4 u = *reinterpret_cast<const uint4*>(src + r * 128 + ((c ^ (r & 7)) << 4));
    uint4 lo, hi;
    i8x4_to_f16x4(u.x, lo.x, lo.y);
    i8x4_to_f16x4(u.y, lo.z, lo.w);
    i8x4_to_f16x4(u.z, hi.x, hi.y);
    i8x4_to_f16x4(u.w, hi.z, hi.w);
    uint8_t* sub = dst + (c >> 2) * kSub16 + r * 128;
    const int cc = (c & 3) * 2;
    *reinterpret_cast<uint4*>(sub + ((cc ^ (r & 7)) << 4)) = lo;
    *reinterpret_cast<uint4*>(sub + (((cc + 1) ^ (r & 7)) << 4)) = hi;
  }
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

// Register rebalancing between warpgroups (setmaxnreg is warpgroup-wide: all
// four warps of a warpgroup execute the same instruction). The block is
// launched with 168 registers per thread (384 x 168 = 64512); the control
// warpgroup drops to kRegsCtl before its role switch and the softmax
// warpgroups rise to kRegsSoftmax (128 x 88 + 256 x 208 = 64512). At the end
// the softmax warpgroups drop to kRegsCtl too, so the shared teardown runs
// with one budget in every warp. The changes sit inside the branches so the
// compiler allocates each branch with its own budget.
constexpr uint32_t kRegsCtl = 88, kRegsSoftmax = 208;
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}


// S_i = Q_i K^T for one 128-key tile: 8 MMAs of K = 16 over the two
// 64-channel subtiles of the fp16 Q and K tiles. The empty asm keeps the
// compiler from hoisting the (loop-invariant) descriptors of every buffer into
// registers; they are recomputed from the base addresses, a few integer ops.
__device__ __forceinline__ void issue_qk(uint32_t tmem, uint32_t sbase, int i, uint32_t buf) {
  uint32_t qa = sbase + kOffQ16 + static_cast<uint32_t>(i) * kTile16, ka = sbase + kOffK16 + buf * kTile16;
  asm volatile("" : "+r"(qa), "+r"(ka));
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t off = static_cast<uint32_t>(ks >> 2) * kSub16 + static_cast<uint32_t>(ks & 3) * 32u;
    tc::mma_f16_ss(tmem + col_s(i), tc::sw128_desc(qa + off), tc::sw128_desc(ka + off), tc::kIdescM128N128,
                   ks > 0 ? 1u : 0u);
  }
}

// O_i (+)= P_i V for one 128-key tile: 4 MMAs of K = 32, P from TMEM (the
// first 32 columns of S_i), V^T from shared memory.
__device__ __forceinline__ void issue_pv(uint32_t tmem, uint32_t sbase, int i, uint32_t vst, bool acc) {
  uint32_t va = sbase + kOffV + vst * kTile8;
  asm volatile("" : "+r"(va));
#pragma unroll
  for (int ks = 0; ks < 4; ++ks)
    tc::mma_f8_ts(tmem + col_o(i), tmem + col_s(i) + 8u * ks, tc::sw128_desc(va + 32u * ks), tc::kIdescM128N128,
                  (acc || ks > 0) ? 1u : 0u);
}

// One 128-key tile of the online softmax for the calling thread's query row
// (TMEM lane): reads S, updates the running maximum m and row sum l, writes
// e4m3(p448) into the first 32 columns of S, and rescales O when the maximum
// grew. kTail masks keys at or past nvalid (the last tile of a ragged S).
template <bool kTail>
__device__ __forceinline__ void softmax_tile(uint32_t tS, uint32_t tO, const float (&cb)[4], int nvalid, bool first,
                                             float& m, float& l) {
  uint32_t sr[4][32];
#pragma unroll
  for (int b = 0; b < 4; ++b) tc::tmem_ld32(tS + 32u * b, sr[b]);
  tc::tmem_wait_ld();
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
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const float2 c2 = make_float2(cb[b], cb[b]);
    uint32_t pw[8];
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
      pw[k] = e4m3x2(p01.y, p01.x) | (e4m3x2(p23.y, p23.x) << 16);
    }
    tc::tmem_st8(tS + 8u * b, pw);
  }
  l = l * alpha + ((sa.x + sa.y) + (sb.x + sb.y));
  m = m_new;
  // O rescale (S is no longer needed, so its registers hold O): PV of the
  // previous tile has completed, because S of this tile was committed after it.
  if (!first && __any_sync(0xffffffffu, grew)) {
    uint32_t o[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) tc::tmem_ld32(tO + 32u * c, o[c]);
    tc::tmem_wait_ld();
    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        const float2 r = __fmul2_rn(make_float2(__uint_as_float(o[c][k]), __uint_as_float(o[c][k + 1])), a2);
        o[c][k] = __float_as_uint(r.x);
        o[c][k + 1] = __float_as_uint(r.y);
      }
      tc::tmem_st32(tO + 32u * c, o[c]);
    }
  }
  tc::tmem_wait_st();
}

__global__ void __launch_bounds__(kThreads, 1)
    attention_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const Params prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = tc::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ctx cx;
  cx.bar0 = sbase + kOffBar;
  cx.abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  cx.dev_err = prm.dev_err;

  if (threadIdx.x == 0) {
    *cx.abort_flag = 0;
    for (int s = 0; s < kK8Stages; ++s) {
      tc::mbar_init(cx.bar(kBarK8Full + s), 1);
      tc::mbar_init(cx.bar(kBarK8Empty + s), kConvThreads);
    }
    for (int s = 0; s < kVStages; ++s) {
      tc::mbar_init(cx.bar(kBarVFull + s), 1);
      tc::mbar_init(cx.bar(kBarVEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(cx.bar(kBarK16Full + s), kConvThreads);
      tc::mbar_init(cx.bar(kBarK16Empty + s), 1);
      tc::mbar_init(cx.bar(kBarSFull + s), 1);
      tc::mbar_init(cx.bar(kBarPFull + s), 128);
      tc::mbar_init(cx.bar(kBarOFull + s), 1);
      tc::mbar_init(cx.bar(kBarOEmpty + s), 128);
    }
    tc::mbar_init(cx.bar(kBarQ16Full), kConvThreads);
    tc::mbar_init(cx.bar(kBarQ16Empty), 1);
    tc::mbar_init(cx.bar(kBarDrain), 1);
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(sbase + kOffTmemSlot, kTmemCols);
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
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemSlot);
  const int64_t n_kv = prm.n_kv;
  if (warp < 4) {
  // control warpgroup: one register decrease for all four warps
  regs_dec<kRegsCtl>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      uint32_t k8_cnt = 0, v_cnt = 0;
      int k8_pending[kK8Stages], v_pending[kVStages];
      for (int s = 0; s < kK8Stages; ++s) k8_pending[s] = -1;
      for (int s = 0; s < kVStages; ++s) v_pending[s] = -1;
      bool ok = true;
      for (int64_t u = blockIdx.x; ok && u < prm.n_units; u += gridDim.x) {
        const int32_t bh = static_cast<int32_t>(u / prm.pairs_per_head);
        const int32_t q_row0 = static_cast<int32_t>((u % prm.pairs_per_head) * 256);
        // items of the int8 ring: Q tile 0, Q tile 1, then K tiles; V^T tiles interleaved
        for (int64_t item = -2; ok && item < n_kv; ++item) {
          {
            const uint32_t st = k8_cnt % kK8Stages, ph = (k8_cnt / kK8Stages) & 1u;
            if (!(ok = wait_bar(cx, cx.bar(kBarK8Empty + st), ph ^ 1u))) break;
            const uint32_t full = cx.bar(kBarK8Full + st);
            tc::mbar_arrive_expect_tx(full, kTile8);
            const uint32_t dst = sbase + kOffK8 + st * kTile8;
            if (item < 0)
              tc::tma_load_3d(dst, &tm_q, 0, q_row0 + static_cast<int32_t>(item + 2) * 128, bh, full);
            else
              tc::tma_load_3d(dst, &tm_k, 0, static_cast<int32_t>(item) * 128, bh, full);
            k8_pending[st] = static_cast<int>(ph);
            ++k8_cnt;
          }
          if (item >= 0) {
            const uint32_t st = v_cnt % kVStages, ph = (v_cnt / kVStages) & 1u;
            if (!(ok = wait_bar(cx, cx.bar(kBarVEmpty + st), ph ^ 1u))) break;
            const uint32_t full = cx.bar(kBarVFull + st);
            tc::mbar_arrive_expect_tx(full, kTile8);
            tc::tma_load_3d(sbase + kOffV + st * kTile8, &tm_v, static_cast<int32_t>(item) * 128, 0, bh, full);
            v_pending[st] = static_cast<int>(ph);
            ++v_cnt;
          }
        }
      }
      if (!ok) {
        // let every copy this thread issued land before the CTA exits
        Ctx drain = cx;
        volatile int no_abort = 0;
        drain.abort_flag = &no_abort;
        for (int s = 0; s < kK8Stages; ++s)
          if (k8_pending[s] >= 0) wait_bar(drain, cx.bar(kBarK8Full + s), static_cast<uint32_t>(k8_pending[s]));
        for (int s = 0; s < kVStages; ++s)
          if (v_pending[s] >= 0) wait_bar(drain, cx.bar(kBarVFull + s), static_cast<uint32_t>(v_pending[s]));
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA --
    if (lane == 0) {
      uint32_t k16_cnt = 0, v_cnt = 0, unit_cnt = 0, p_cnt[2] = {0, 0};
      bool ok = true;
      for (int64_t u = blockIdx.x; ok && u < prm.n_units; u += gridDim.x) {
        if (!(ok = wait_bar(cx, cx.bar(kBarQ16Full), unit_cnt & 1u))) break;
        tc::tc_fence_after();
        // step 0: both QK MMAs
        uint32_t buf = k16_cnt & 1u;
        if (!(ok = wait_bar(cx, cx.bar(kBarK16Full + buf), (k16_cnt >> 1) & 1u))) break;
        tc::tc_fence_after();
        issue_qk(tmem, sbase, 0, buf);
        tc::mma_commit(cx.bar(kBarSFull + 0));
        issue_qk(tmem, sbase, 1, buf);
        tc::mma_commit(cx.bar(kBarSFull + 1));
        tc::mma_commit(cx.bar(kBarK16Empty + buf));
        ++k16_cnt;
        for (int64_t j = 1; ok && j <= n_kv; ++j) {
          const bool last = (j == n_kv);
          const uint32_t vst = v_cnt % kVStages;
          if (!last) {
            buf = k16_cnt & 1u;
            if (!(ok = wait_bar(cx, cx.bar(kBarK16Full + buf), (k16_cnt >> 1) & 1u))) break;
          }
          if (!(ok = wait_bar(cx, cx.bar(kBarVFull + vst), (v_cnt / kVStages) & 1u))) break;
          for (int i = 0; i < 2; ++i) {
            if (!(ok = wait_bar(cx, cx.bar(kBarPFull + i), p_cnt[i] & 1u))) break;
            ++p_cnt[i];
            if (j == 1 && !(ok = wait_bar(cx, cx.bar(kBarOEmpty + i), (unit_cnt & 1u) ^ 1u))) break;
            tc::tc_fence_after();
            issue_pv(tmem, sbase, i, vst, j > 1);  // PV of step j-1
            if (last) {
              tc::mma_commit(cx.bar(kBarOFull + i));
            } else {
              issue_qk(tmem, sbase, i, buf);  // QK of step j
              tc::mma_commit(cx.bar(kBarSFull + i));
            }
          }
          if (!ok) break;
          tc::mma_commit(cx.bar(kBarVEmpty + vst));
          ++v_cnt;
          if (!last) {
            tc::mma_commit(cx.bar(kBarK16Empty + buf));
            ++k16_cnt;
            if (j == n_kv - 1) tc::mma_commit(cx.bar(kBarQ16Empty));
          }
        }
        if (ok && n_kv == 1) tc::mma_commit(cx.bar(kBarQ16Empty));
        ++unit_cnt;
      }
      // drain: all MMAs issued by this thread complete before TMEM is freed
      tc::mma_commit(cx.bar(kBarDrain));
      Ctx drain = cx;
      volatile int no_abort = 0;
      drain.abort_flag = &no_abort;
      wait_bar(drain, cx.bar(kBarDrain), 0);
    }
  } else {
    // ----------------------------------------------------------- converters --
    const int ct = threadIdx.x - 64;
    uint32_t k8_cnt = 0, k16_cnt = 0, unit_cnt = 0;
    bool ok = true;
    for (int64_t u = blockIdx.x; ok && u < prm.n_units; u += gridDim.x) {
      if (!(ok = wait_bar_warp(cx, cx.bar(kBarQ16Empty), (unit_cnt & 1u) ^ 1u))) break;
      for (int64_t item = -2; item < n_kv; ++item) {
        const uint32_t st = k8_cnt % kK8Stages;
        if (!(ok = wait_bar_warp(cx, cx.bar(kBarK8Full + st), (k8_cnt / kK8Stages) & 1u))) break;
        uint8_t* dst;
        uint32_t buf = 0;
        if (item < 0) {
          dst = smem + kOffQ16 + static_cast<uint32_t>(item + 2) * kTile16;
        } else {
          buf = k16_cnt & 1u;
          if (!(ok = wait_bar_warp(cx, cx.bar(kBarK16Empty + buf), ((k16_cnt >> 1) & 1u) ^ 1u))) break;
          dst = smem + kOffK16 + buf * kTile16;
        }
        convert_tile(smem + kOffK8 + st * kTile8, dst, ct);
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(cx.bar(kBarK8Empty + st));
        ++k8_cnt;
        if (item == -1) tc::mbar_arrive(cx.bar(kBarQ16Full));
        if (item >= 0) {
          tc::mbar_arrive(cx.bar(kBarK16Full + buf));
          ++k16_cnt;
        }
      }
      ++unit_cnt;
    }
  }
  __syncwarp();
  } else {
    // -------------------------------------------------------------- softmax --
    regs_inc<kRegsSoftmax>();
    const int i = (warp - 4) >> 2;        // query tile of this warpgroup
    const int wq = warp & 3;              // TMEM lane quarter
    const int row = wq * 32 + lane;       // row within the query tile
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_addr + col_s(i);
    const uint32_t tO = tmem + lane_addr + col_o(i);
    const int64_t nblk = prm.S_pad / kQKBlock;
    uint32_t s_cnt = 0, unit_cnt = 0;
    bool ok = true;
    for (int64_t u = blockIdx.x; ok && u < prm.n_units; u += gridDim.x) {
      const int64_t bh = u / prm.pairs_per_head;
      const int64_t qrow = (u % prm.pairs_per_head) * 256 + i * 128 + row;  // query index in the head
      const bool row_valid = qrow < prm.S;
      const float cq = row_valid ? prm.q_scale[bh * nblk + qrow / kQKBlock] * prm.sm_log2 : 0.0f;
      const float* ks = prm.k_scale + bh * nblk;
      float m = -INFINITY, l = 0.0f;
      float cb[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) cb[b] = cq * __ldg(ks + b);
      for (int64_t j = 0; j < n_kv; ++j) {
        if (!(ok = wait_bar_warp(cx, cx.bar(kBarSFull + i), s_cnt & 1u))) break;
        ++s_cnt;
        tc::tc_fence_after();
        const int64_t nvalid = prm.S - j * kKeyTile;  // keys of this tile below S
        if (nvalid >= kKeyTile)
          softmax_tile<false>(tS, tO, cb, kKeyTile, j == 0, m, l);
        else
          softmax_tile<true>(tS, tO, cb, static_cast<int>(nvalid), j == 0, m, l);
        tc::tc_fence_before();
        tc::mbar_arrive(cx.bar(kBarPFull + i));
        if (j + 1 < n_kv) {
#pragma unroll
          for (int b = 0; b < 4; ++b) cb[b] = cq * __ldg(ks + (j + 1) * 4 + b);
        }
      }
      if (!ok) break;
      // epilogue: O = acc * s_v / l (l counts p448), bf16 in the output layout
      if (!(ok = wait_bar_warp(cx, cx.bar(kBarOFull + i), unit_cnt & 1u))) break;
      tc::tc_fence_after();
      const float inv_l = 1.0f / l;
      const float* sv = prm.v_scale + bh * kHeadDim;
      const int64_t b_idx = bh / prm.H, h_idx = bh % prm.H;
      uint16_t* dst = prm.out.p + b_idx * prm.out.sb + qrow * prm.out.ss + h_idx * prm.out.sh;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tc::tmem_ld32(tO + 32u * c, o);
        tc::tmem_wait_ld();
        if (row_valid) {
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 s2 = __ldg(reinterpret_cast<const float2*>(sv + 32 * c + 2 * k));
            const float a0 = __uint_as_float(o[2 * k]) * inv_l * s2.x;
            const float a1 = __uint_as_float(o[2 * k + 1]) * inv_l * s2.y;
            const __nv_bfloat162 v2 = __floats2bfloat162_rn(a0, a1);
            pk[k] = *reinterpret_cast<const uint32_t*>(&v2);
          }
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int k = 0; k < 4; ++k) d4[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(cx.bar(kBarOEmpty + i));
      ++unit_cnt;
    }
    regs_dec<kRegsCtl>();  // the teardown runs with the control budget in every warp
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// 3-D byte tensor [d2][d1][d0] with 128 x 128 boxes, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint64_t strides[2] = {d0, d0 * d1};
  const uint32_t box[3] = {128, 128, 1};
  return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

cudaError_t launch_attention_tc(const Bundle& in, int64_t B, int64_t S, int64_t H, float sm_scale, const Out& out,
                                int* dev_err, cudaStream_t stream) {
  const int64_t S_pad = padded_len(S);
  const int64_t BH = B * H;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, in.q_codes, kHeadDim, static_cast<uint64_t>(S_pad), static_cast<uint64_t>(BH)) ||
      !make_map(&tk, in.k_codes, kHeadDim, static_cast<uint64_t>(S_pad), static_cast<uint64_t>(BH)) ||
      !make_map(&tv, in.vt_codes, static_cast<uint64_t>(S_pad), kHeadDim, static_cast<uint64_t>(BH)))
    return cudaErrorInvalidValue;
  Params p;
  p.S = S;
  p.S_pad = S_pad;
  p.n_kv = S_pad / kKeyTile;
  p.pairs_per_head = div_up(S_pad / 128, 2);
  p.n_units = BH * p.pairs_per_head;
  p.q_scale = in.q_scale;
  p.k_scale = in.k_scale;
  p.v_scale = in.v_scale;
  p.out = out;
  p.H = H;
  p.sm_log2 = sm_scale * kLog2e;
  p.dev_err = dev_err;
  cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int sms = sm_count_current();
  const int grid = static_cast<int>(p.n_units < sms ? p.n_units : sms);
  attention_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace sage
