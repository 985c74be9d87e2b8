// Plain SIMT quantized attention: one thread per query row, integer dot
// products (dp4a) for QK^T, the online softmax over 128-key tiles, P rounded
// to e4m3(448 p), and PV accumulated in fp32 registers.
//
// Method: "aiter-sage-attention: SageAttention for AMD RDNA4 (gfx1201)
// #1222", section "The kernel" (INT8 QK^T, FP8 PV, FP32 accumulation).
// This kernel exists so tests can cross-check the tensor-core kernel with an
// independent GPU implementation of the same steps (including the causal mask
// and the log-sum-exp); the library never uses it in place of the tensor-core
// kernel.
#include <cuda_bf16.h>

#include "common.cuh"

namespace sage {
namespace {

constexpr int kRows = 128;  // query rows per CTA (one per thread)

__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(a), "f"(b));
  return r;
}

// Values of two e4m3 codes (low byte -> .x, high byte -> .y).
__device__ __forceinline__ float2 e4m3x2_decode(uint32_t pair) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(pair)));
  __half2 hv = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(hv);
}

__global__ void __launch_bounds__(kRows, 1) attention_simt_kernel(Bundle in, int64_t S, int64_t S_pad, int64_t H,
                                                                  float sm_scale, Out out, int causal,
                                                                  float* lse) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* ks = reinterpret_cast<uint32_t*>(smem);                      // [128 keys][32 words]
  float* vs = reinterpret_cast<float*>(smem + kKeyTile * kHeadDim);      // [128 keys][128 dims]

  const int tid = threadIdx.x;
  const int64_t h = blockIdx.y, b = blockIdx.z;
  const int64_t bh = b * H + h;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRows + tid;  // < S_pad
  const int64_t nblk = S_pad / kQKBlock;

  uint32_t qw[32];
  {
    const uint4* src = reinterpret_cast<const uint4*>(in.q_codes + (bh * S_pad + row) * kHeadDim);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 u = src[i];
      qw[4 * i] = u.x; qw[4 * i + 1] = u.y; qw[4 * i + 2] = u.z; qw[4 * i + 3] = u.w;
    }
  }
  const float sq = in.q_scale[bh * nblk + row / kQKBlock];
  float acc[kHeadDim];
#pragma unroll
  for (int d = 0; d < kHeadDim; ++d) acc[d] = 0.0f;
  float m = -INFINITY, l = 0.0f;

  // with the causal mask, the CTA's rows see the key tiles up to its own
  const int64_t key_end = causal ? min(S, (static_cast<int64_t>(blockIdx.x) + 1) * kRows) : S;
  for (int64_t j0 = 0; j0 < key_end; j0 += kKeyTile) {
    __syncthreads();
    {
      const uint4* src = reinterpret_cast<const uint4*>(in.k_codes + (bh * S_pad + j0) * kHeadDim);
      uint4* dst = reinterpret_cast<uint4*>(ks);
      for (int i = tid; i < kKeyTile * kHeadDim / 16; i += kRows) dst[i] = src[i];
      // thread tid decodes channel tid of the 128 keys of the tile
      const uint4* vsrc = reinterpret_cast<const uint4*>(in.vt_codes + (bh * kHeadDim + tid) * S_pad + j0);
      for (int i = 0; i < 8; ++i) {
        const uint4 u = vsrc[i];
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
        for (int wi = 0; wi < 4; ++wi) {
          const float2 lo = e4m3x2_decode(wv[wi] & 0xFFFFu);
          const float2 hi = e4m3x2_decode(wv[wi] >> 16);
          const int j = 16 * i + 4 * wi;
          vs[(j + 0) * kHeadDim + tid] = lo.x;
          vs[(j + 1) * kHeadDim + tid] = lo.y;
          vs[(j + 2) * kHeadDim + tid] = hi.x;
          vs[(j + 3) * kHeadDim + tid] = hi.y;
        }
      }
    }
    __syncthreads();
    int nk = static_cast<int>(S - j0 < kKeyTile ? S - j0 : kKeyTile);
    if (causal && row - j0 + 1 < nk) nk = static_cast<int>(row - j0 + 1);  // keys j <= row (at least one)
    // pass 1: tile maximum of the logits
    float tmax = -INFINITY;
    for (int j = 0; j < nk; ++j) {
      int s = 0;
#pragma unroll
      for (int w = 0; w < 32; ++w) s = __dp4a(static_cast<int>(qw[w]), static_cast<int>(ks[j * 32 + w]), s);
      const float c = __fmul_rn(__fmul_rn(sq, in.k_scale[bh * nblk + (j0 + j) / kQKBlock]), sm_scale);
      tmax = fmaxf(tmax, __fmul_rn(static_cast<float>(s), c));
    }
    const float m_new = fmaxf(m, tmax);
    const float alpha = expf(m - m_new);
    l = l * alpha;
#pragma unroll
    for (int d = 0; d < kHeadDim; ++d) acc[d] *= alpha;
    // pass 2: probabilities, row sum, e4m3(448 p) times V
    for (int j = 0; j < nk; ++j) {
      int s = 0;
#pragma unroll
      for (int w = 0; w < 32; ++w) s = __dp4a(static_cast<int>(qw[w]), static_cast<int>(ks[j * 32 + w]), s);
      const float c = __fmul_rn(__fmul_rn(sq, in.k_scale[bh * nblk + (j0 + j) / kQKBlock]), sm_scale);
      const float p = expf(__fsub_rn(__fmul_rn(static_cast<float>(s), c), m_new));
      l += p;
      const float pq = e4m3x2_decode(e4m3x2(0.0f, __fmul_rn(kPScale, p))).x;
      const float* vrow = vs + j * kHeadDim;
#pragma unroll
      for (int d = 0; d < kHeadDim; ++d) acc[d] = fmaf(pq, vrow[d], acc[d]);
    }
    m = m_new;
  }
  if (row >= S) return;
  if (lse != nullptr) lse[bh * S + row] = m + logf(l);
  const float* sv = in.v_scale + bh * kHeadDim;
  uint16_t* dst = out.p + b * out.sb + row * out.ss + h * out.sh;
#pragma unroll
  for (int d = 0; d < kHeadDim; d += 2) {
    const float o0 = __fdiv_rn(__fmul_rn(__fdiv_rn(acc[d], l), sv[d]), kPScale);
    const float o1 = __fdiv_rn(__fmul_rn(__fdiv_rn(acc[d + 1], l), sv[d + 1]), kPScale);
    const __nv_bfloat162 pr = __floats2bfloat162_rn(o0, o1);
    *reinterpret_cast<__nv_bfloat162*>(dst + d) = pr;
  }
}

}  // namespace

cudaError_t launch_attention_simt(const Bundle& in, int64_t B, int64_t S, int64_t H, float sm_scale,
                                  const Out& out, bool causal, float* lse, cudaStream_t stream) {
  const int64_t S_pad = padded_len(S);
  const size_t smem = static_cast<size_t>(kKeyTile) * kHeadDim + static_cast<size_t>(kKeyTile) * kHeadDim * 4;
  cudaError_t e = cudaFuncSetAttribute(attention_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(S_pad / kRows), static_cast<unsigned>(H), static_cast<unsigned>(B));
  attention_simt_kernel<<<grid, kRows, smem, stream>>>(in, S, S_pad, H, sm_scale, out, causal ? 1 : 0, lse);
  return cudaGetLastError();
}

}  // namespace sage
