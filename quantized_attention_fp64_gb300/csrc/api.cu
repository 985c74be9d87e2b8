// C ABI of the library: argument validation, buffer layout, dispatch.
//
// Entry-point contract: "aiter-sage-attention: SageAttention for AMD RDNA4
// (gfx1201) #1222", section "What I have so far" -- sageattn(q, k, v,
// tensor_layout, is_causal, sm_scale, return_lse) rejects causal, LSE,
// non-BF16, head dim other than 128 and unequal Q/K/V shapes with an error
// and never falls back. Everything is validated on the host before any work
// is enqueued.
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/sage.h"
#include "common.cuh"

namespace sage {
// The size limits every entry point applies (offsets stay within 64-bit
// arithmetic, work-item counters within 32 bits).
int check_problem_sizes(int64_t B, int64_t S, int64_t H, int64_t D) {
  constexpr int64_t kMaxBH = 65535;
  constexpr int64_t kMaxS = int64_t(1) << 31;
  constexpr int64_t kMaxElems = int64_t(1) << 44;
  if (B < 0 || S < 0 || H < 0 || D < 0) return SAGE_ERR_SHAPE;
  if (D != kHeadDim && D != 64) return SAGE_ERR_HEAD_DIM;
  if (B > kMaxBH || H > kMaxBH || S > kMaxS) return SAGE_ERR_TOO_LARGE;
  if (B * H > kMaxBH * 16) return SAGE_ERR_TOO_LARGE;
  if (B * H * padded_len(S) > kMaxElems / D) return SAGE_ERR_TOO_LARGE;
  return SAGE_OK;
}

namespace {

// Set by kernels that give up a bounded wait; read and cleared by
// sage_device_error. Host code reaches it through cudaGetSymbolAddress.
__device__ int g_device_error = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_err_ptr[kMaxDevices] = {};
int g_arch_ok[kMaxDevices] = {};  // 0 unknown, 1 ok, -1 wrong architecture

// Largest accepted sizes: every index stays far inside int64, the grids stay
// inside CUDA's limits (H and B are grid dimensions of the prologue) and the
// 2-D and 3-D tensor maps of the attention kernel keep 32-bit coordinates.
constexpr int64_t kMaxBH = 65535;
constexpr int64_t kMaxS = int64_t(1) << 31;
constexpr int64_t kMaxElems = int64_t(1) << 44;

int check_device(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SAGE_ERR_CUDA;
  if (bind_device_context(dev) != cudaSuccess) return SAGE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_arch_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return SAGE_ERR_CUDA;
    g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (g_arch_ok[dev] < 0) return SAGE_ERR_ARCH;
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return SAGE_ERR_CUDA;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  *dev_out = dev;
  return SAGE_OK;
}

int check_sizes(int64_t B, int64_t S, int64_t H, int64_t D) { return check_problem_sizes(B, S, H, D); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool stride_ok(int64_t s) { return s % 8 == 0; }

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

constexpr int kBundleArrays = 9;

struct BundleLayout {
  size_t off[kBundleArrays];
  size_t total;
};

BundleLayout bundle_layout(int64_t B, int64_t S, int64_t H, int64_t D) {
  const size_t bh = static_cast<size_t>(B * H);
  const size_t sp = static_cast<size_t>(padded_len(S));
  const size_t d = static_cast<size_t>(D);
  const size_t sizes[kBundleArrays] = {bh * sp * d,                bh * sp * d,                bh * sp * d,
                                       bh * (sp / kQKBlock) * 4,   bh * (sp / kQKBlock) * 4,   bh * d * 4,
                                       bh * d * 4,                 bh * sp * d * 2,            bh * sp * d * 2};
  BundleLayout l;
  size_t o = 0;
  for (int i = 0; i < kBundleArrays; ++i) {
    l.off[i] = o;
    o += round256(sizes[i]);
  }
  l.total = o;
  return l;
}

Bundle carve(void* base, const BundleLayout& l) {
  char* c = static_cast<char*>(base);
  Bundle b;
  b.q_codes = reinterpret_cast<int8_t*>(c + l.off[0]);
  b.k_codes = reinterpret_cast<int8_t*>(c + l.off[1]);
  b.vt_codes = reinterpret_cast<uint8_t*>(c + l.off[2]);
  b.q_scale = reinterpret_cast<float*>(c + l.off[3]);
  b.k_scale = reinterpret_cast<float*>(c + l.off[4]);
  b.v_scale = reinterpret_cast<float*>(c + l.off[5]);
  b.k_mean = reinterpret_cast<float*>(c + l.off[6]);
  b.q16 = reinterpret_cast<uint16_t*>(c + l.off[7]);
  b.k16 = reinterpret_cast<uint16_t*>(c + l.off[8]);
  return b;
}

int check_bundle(const sage_quantized* in, bool need_mean) {
  if (in == nullptr) return SAGE_ERR_NULLPTR;
  const void* ptrs[kBundleArrays] = {in->q_codes_dev, in->k_codes_dev, in->vt_codes_dev,
                                     in->q_scale_dev, in->k_scale_dev,  in->v_scale_dev,
                                     in->k_mean_dev,  in->q16_dev,      in->k16_dev};
  for (int i = 0; i < kBundleArrays; ++i) {
    if (i == 6 && !need_mean) continue;
    if (ptrs[i] == nullptr) return SAGE_ERR_NULLPTR;
    if (!aligned16(ptrs[i])) return SAGE_ERR_ALIGN;
  }
  return SAGE_OK;
}

Bundle to_bundle(const sage_quantized* in) {
  Bundle b;
  b.q_codes = in->q_codes_dev;
  b.k_codes = in->k_codes_dev;
  b.vt_codes = in->vt_codes_dev;
  b.q_scale = in->q_scale_dev;
  b.k_scale = in->k_scale_dev;
  b.v_scale = in->v_scale_dev;
  b.k_mean = in->k_mean_dev;
  b.q16 = in->q16_dev;
  b.k16 = in->k16_dev;
  return b;
}

int check_bf16_in(const sage_bf16_tensor* t) {
  if (t == nullptr || t->ptr_dev == nullptr) return SAGE_ERR_NULLPTR;
  if (!aligned16(t->ptr_dev)) return SAGE_ERR_ALIGN;
  if (!stride_ok(t->stride_b) || !stride_ok(t->stride_s) || !stride_ok(t->stride_h)) return SAGE_ERR_ALIGN;
  return SAGE_OK;
}

int check_out(const void* out, int64_t ob, int64_t os, int64_t oh) {
  if (out == nullptr) return SAGE_ERR_NULLPTR;
  if (!aligned16(out) || !stride_ok(ob) || !stride_ok(os) || !stride_ok(oh)) return SAGE_ERR_ALIGN;
  return SAGE_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA; }

typedef cudaError_t (*AttnLaunch)(const Bundle&, int64_t, int64_t, int64_t, int64_t, float, const Out&, bool,
                                  float*, int*, cudaStream_t);

cudaError_t simt_adapter(const Bundle& in, int64_t B, int64_t S, int64_t H, int64_t, float sm, const Out& o,
                         bool causal, float* lse, int*, cudaStream_t st) {
  return launch_attention_simt(in, B, S, H, sm, o, causal, lse, st);
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int attention_common(const sage_quantized* in, int64_t B, int64_t S, int64_t H, int64_t D, float sm_scale,
                     bool causal, void* out_dev, int64_t ob, int64_t os, int64_t oh, float* lse_dev, void* stream,
                     AttnLaunch launch) {
  int rc = check_sizes(B, S, H, D);
  if (rc != SAGE_OK) return rc;
  if ((rc = check_bundle(in, false)) != SAGE_OK) return rc;
  if ((rc = check_out(out_dev, ob, os, oh)) != SAGE_OK) return rc;
  if (lse_dev != nullptr && !aligned4(lse_dev)) return SAGE_ERR_ALIGN;
  if (!std::isfinite(sm_scale) || !(sm_scale > 0.0f)) return SAGE_ERR_ARG;
  int dev = 0;
  if ((rc = check_device(&dev)) != SAGE_OK) return rc;
  if (B == 0 || H == 0 || S == 0) return SAGE_OK;
  Out o{static_cast<uint16_t*>(out_dev), ob, os, oh};
  return cuda_status(launch(to_bundle(in), B, S, H, D, sm_scale, o, causal, lse_dev, g_err_ptr[dev],
                            static_cast<cudaStream_t>(stream)));
}

}  // namespace

int* device_error_ptr() {
  int dev = 0;
  if (check_device(&dev) != SAGE_OK) return nullptr;
  return g_err_ptr[dev];
}

}  // namespace sage

namespace sage {
namespace {

// The sageattn path after the checks that differ between the two entries:
// prologue into the workspace, attention (causal, lse as given), and with
// lse and smooth_k the key-mean term of the log-sum-exp.
int sageattn_impl(const void* q_dev, const void* k_dev, const void* v_dev, const int64_t q_shape[4],
                  const int64_t k_shape[4], const int64_t v_shape[4], const int64_t q_strides[4],
                  const int64_t k_strides[4], const int64_t v_strides[4], int q_dtype, int k_dtype, int v_dtype,
                  const char* tensor_layout, bool causal, float sm_scale, float* lse_dev, int smooth_k,
                  void* out_dev, const int64_t out_strides[4], int out_dtype, void* workspace_dev,
                  size_t workspace_bytes, void* cuda_stream) {
  if (q_dtype != SAGE_DTYPE_BF16 || k_dtype != SAGE_DTYPE_BF16 || v_dtype != SAGE_DTYPE_BF16 ||
      out_dtype != SAGE_DTYPE_BF16)
    return SAGE_ERR_DTYPE;
  if (q_shape == nullptr || k_shape == nullptr || v_shape == nullptr || q_strides == nullptr ||
      k_strides == nullptr || v_strides == nullptr || out_strides == nullptr || tensor_layout == nullptr)
    return SAGE_ERR_NULLPTR;
  int is_nhd;
  if (std::strcmp(tensor_layout, "NHD") == 0) is_nhd = 1;
  else if (std::strcmp(tensor_layout, "HND") == 0) is_nhd = 0;
  else return SAGE_ERR_LAYOUT;
  // axis positions of (b, s, h, d) in the given layout
  const int ax_s = is_nhd ? 1 : 2, ax_h = is_nhd ? 2 : 1;
  const int64_t B = q_shape[0], S = q_shape[ax_s], H = q_shape[ax_h], D = q_shape[3];
  if (D != kHeadDim && D != 64 && D >= 0) return SAGE_ERR_HEAD_DIM;
  for (int i = 0; i < 4; ++i)
    if (k_shape[i] != q_shape[i] || v_shape[i] != q_shape[i]) return SAGE_ERR_SHAPE;
  int rc = check_sizes(B, S, H, D);
  if (rc != SAGE_OK) return rc;
  const int64_t* st[4] = {q_strides, k_strides, v_strides, out_strides};
  for (int i = 0; i < 4; ++i)
    if (st[i][3] != 1) return SAGE_ERR_LAYOUT;
  if (!(std::isnan(sm_scale) || (std::isfinite(sm_scale) && sm_scale > 0.0f))) return SAGE_ERR_ARG;
  const float scale = std::isnan(sm_scale) ? static_cast<float>(1.0 / std::sqrt(static_cast<double>(D))) : sm_scale;
  const sage_bf16_tensor qt{q_dev, q_strides[0], q_strides[ax_s], q_strides[ax_h]};
  const sage_bf16_tensor kt{k_dev, k_strides[0], k_strides[ax_s], k_strides[ax_h]};
  const sage_bf16_tensor vt{v_dev, v_strides[0], v_strides[ax_s], v_strides[ax_h]};
  if ((rc = check_bf16_in(&qt)) != SAGE_OK || (rc = check_bf16_in(&kt)) != SAGE_OK ||
      (rc = check_bf16_in(&vt)) != SAGE_OK)
    return rc;
  if ((rc = check_out(out_dev, out_strides[0], out_strides[ax_s], out_strides[ax_h])) != SAGE_OK) return rc;
  if (lse_dev != nullptr && !aligned4(lse_dev)) return SAGE_ERR_ALIGN;
  if (workspace_dev == nullptr) return SAGE_ERR_NULLPTR;
  if ((reinterpret_cast<uintptr_t>(workspace_dev) & 255u) != 0) return SAGE_ERR_ALIGN;
  const BundleLayout bl = bundle_layout(B, S, H, D);
  const size_t scratch = prologue_scratch_bytes(B, S, H, D);
  if (workspace_bytes < bl.total + scratch) return SAGE_ERR_WORKSPACE;
  int dev = 0;
  if ((rc = check_device(&dev)) != SAGE_OK) return rc;
  if (B == 0 || H == 0 || S == 0) return SAGE_OK;
  const Bundle bundle = carve(workspace_dev, bl);
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  const Bf16In qi{static_cast<const uint16_t*>(q_dev), qt.stride_b, qt.stride_s, qt.stride_h};
  const Bf16In ki{static_cast<const uint16_t*>(k_dev), kt.stride_b, kt.stride_s, kt.stride_h};
  const Bf16In vi{static_cast<const uint16_t*>(v_dev), vt.stride_b, vt.stride_s, vt.stride_h};
  // the int8 Q/K codes are not read by the attention kernel, so this path
  // keeps only their fp16 copies
  if ((rc = cuda_status(launch_prologue(qi, ki, vi, B, S, H, D, smooth_k != 0, bundle,
                                        static_cast<char*>(workspace_dev) + bl.total, false, g_err_ptr[dev],
                                        stream))) != SAGE_OK)
    return rc;
  const Out o{static_cast<uint16_t*>(out_dev), out_strides[0], out_strides[ax_s], out_strides[ax_h]};
  if ((rc = cuda_status(launch_attention_tc(bundle, B, S, H, D, scale, o, causal, lse_dev, g_err_ptr[dev], stream))) !=
      SAGE_OK)
    return rc;
  if (lse_dev != nullptr && smooth_k != 0)
    return cuda_status(launch_lse_smooth_k_term(qi, bundle.k_mean, B, S, H, D, scale, lse_dev, stream));
  return SAGE_OK;
}

// ------------------------------------------------------------ host buffers --
// sage_sageattn_host: host-resident q, k, v and out. The heads are cut into
// G groups; one internal stream copies the groups' inputs in (2-D copies: a
// group is a column block of every token row in NHD, a block of heads of
// every batch in HND), two compute streams take the groups in turn (the
// prologue and attention of group g), one stream copies the outputs back. So
// the copies of one group overlap the kernels of its neighbours, and one
// group's attention tail overlaps the next group's kernels.

constexpr int kHostMaxGroups = 16;
constexpr size_t kHostGroupBytes = size_t(32) << 20;  // aim: at least 32 MB of inputs per group

struct HostPlan {
  int64_t hg = 0, G = 0;  // heads per group, groups
  size_t grp_in = 0;      // bytes of one bf16 tensor of a group
  size_t off_q = 0, off_k = 0, off_v = 0, off_o = 0, off_bundle[2] = {0, 0}, off_scratch[2] = {0, 0}, total = 0;
};

HostPlan host_plan(int64_t B, int64_t S, int64_t H, int64_t D, int n_groups) {
  HostPlan p;
  const size_t in_bytes = static_cast<size_t>(B * S * H * D) * 2;
  int64_t G = n_groups;
  if (G <= 0) {
    // at most 10 groups unless asked: at the video size (28 heads) 10 groups
    // of 3 heads measured 2.79 ms, 7 of 4 2.87, 14 of 2 3.08 per call
    G = static_cast<int64_t>(3 * in_bytes / kHostGroupBytes);
    G = G < 1 ? 1 : (G > 10 ? 10 : G);
  }
  if (G > kHostMaxGroups) G = kHostMaxGroups;
  if (G > H) G = H > 0 ? H : 1;
  p.hg = H > 0 ? div_up(H, G) : 1;
  p.G = H > 0 ? div_up(H, p.hg) : 1;
  p.grp_in = static_cast<size_t>(B * S * p.hg * D) * 2;
  const size_t region = round256(p.grp_in * static_cast<size_t>(p.G));
  const size_t bundle = bundle_layout(B, S, p.hg, D).total;
  const size_t scratch = round256(prologue_scratch_bytes(B, S, p.hg, D));
  size_t o = 0;
  p.off_q = o;
  o += region;
  p.off_k = o;
  o += region;
  p.off_v = o;
  o += region;
  p.off_o = o;
  o += region;
  for (int i = 0; i < 2; ++i) {
    p.off_bundle[i] = o;
    o += bundle;
    p.off_scratch[i] = o;
    o += scratch;
  }
  p.total = o;
  return p;
}

// Internal streams and events, created once per device; the enqueue of one
// call holds the device's lock (the events are reused call after call).
struct HostStreams {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr, comp[2] = {nullptr, nullptr};
  cudaEvent_t ev[2 + 2 * kHostMaxGroups] = {};
};
HostStreams g_host[kMaxDevices];
std::mutex g_host_mu[kMaxDevices];

cudaError_t host_streams(int dev, HostStreams** out) {
  HostStreams& h = g_host[dev];
  if (!h.ready) {
    cudaError_t e;
    cudaStream_t* ss[4] = {&h.h2d, &h.d2h, &h.comp[0], &h.comp[1]};
    for (cudaStream_t* st : ss)
      if (*st == nullptr && (e = cudaStreamCreateWithFlags(st, cudaStreamNonBlocking)) != cudaSuccess) return e;
    for (cudaEvent_t& ev : h.ev)
      if (ev == nullptr && (e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    h.ready = true;
  }
  *out = &h;
  return cudaSuccess;
}

// The 2-D copy of heads [h0, h0 + n) of one bf16 tensor between its full
// host layout and the group's packed device layout (either direction).
cudaError_t copy_heads(void* dst, const void* src, bool to_device, bool nhd, int64_t B, int64_t S, int64_t H,
                       int64_t D, int64_t h0, int64_t n, cudaStream_t st) {
  const size_t e = 2;
  const size_t row_full = static_cast<size_t>(nhd ? H * D : H * S * D) * e;  // pitch of the full tensor
  const size_t row_grp = static_cast<size_t>(nhd ? n * D : n * S * D) * e;   // pitch of the group
  const size_t col0 = static_cast<size_t>(nhd ? h0 * D : h0 * S * D) * e;    // first byte of the group in a row
  const size_t rows = static_cast<size_t>(nhd ? B * S : B);
  if (to_device)
    return cudaMemcpy2DAsync(dst, row_grp, static_cast<const char*>(src) + col0, row_full, row_grp, rows,
                             cudaMemcpyDefault, st);
  return cudaMemcpy2DAsync(static_cast<char*>(dst) + col0, row_full, src, row_grp, row_grp, rows, cudaMemcpyDefault,
                           st);
}

int sageattn_host_impl(const void* q_host, const void* k_host, const void* v_host, const int64_t shape[4],
                       int dtype, const char* tensor_layout, bool causal, float sm_scale, int smooth_k,
                       void* out_host, int n_groups, void* workspace_dev, size_t workspace_bytes,
                       void* cuda_stream) {
  if (dtype != SAGE_DTYPE_BF16) return SAGE_ERR_DTYPE;
  if (shape == nullptr || tensor_layout == nullptr) return SAGE_ERR_NULLPTR;
  bool nhd;
  if (std::strcmp(tensor_layout, "NHD") == 0) nhd = true;
  else if (std::strcmp(tensor_layout, "HND") == 0) nhd = false;
  else return SAGE_ERR_LAYOUT;
  const int64_t B = shape[0], S = nhd ? shape[1] : shape[2], H = nhd ? shape[2] : shape[1], D = shape[3];
  int rc = check_sizes(B, S, H, D);
  if (rc != SAGE_OK) return rc;
  if (!(std::isnan(sm_scale) || (std::isfinite(sm_scale) && sm_scale > 0.0f))) return SAGE_ERR_ARG;
  if (n_groups < 0) return SAGE_ERR_ARG;
  const float scale = std::isnan(sm_scale) ? static_cast<float>(1.0 / std::sqrt(static_cast<double>(D))) : sm_scale;
  if (B == 0 || H == 0 || S == 0) return SAGE_OK;
  if (q_host == nullptr || k_host == nullptr || v_host == nullptr || out_host == nullptr || workspace_dev == nullptr)
    return SAGE_ERR_NULLPTR;
  if ((reinterpret_cast<uintptr_t>(workspace_dev) & 255u) != 0) return SAGE_ERR_ALIGN;
  const HostPlan pl = host_plan(B, S, H, D, n_groups);
  if (workspace_bytes < pl.total) return SAGE_ERR_WORKSPACE;
  int dev = 0;
  if ((rc = check_device(&dev)) != SAGE_OK) return rc;
  std::lock_guard<std::mutex> lock(g_host_mu[dev]);
  HostStreams* hs = nullptr;
  if (host_streams(dev, &hs) != cudaSuccess) return SAGE_ERR_CUDA;
  char* ws = static_cast<char*>(workspace_dev);
  cudaStream_t user = static_cast<cudaStream_t>(cuda_stream);
  cudaEvent_t ev_start = hs->ev[0], ev_end = hs->ev[1];
  cudaEvent_t* ev_in = hs->ev + 2;
  cudaEvent_t* ev_done = hs->ev + 2 + kHostMaxGroups;
  cudaError_t e = cudaEventRecord(ev_start, user);
  // every internal stream starts after the work already on the caller's stream
  cudaStream_t all[4] = {hs->h2d, hs->d2h, hs->comp[0], hs->comp[1]};
  for (int i = 0; i < 4 && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(all[i], ev_start, 0);
  const void* src[3] = {q_host, k_host, v_host};
  const size_t off_in[3] = {pl.off_q, pl.off_k, pl.off_v};
  for (int64_t g = 0; g < pl.G && e == cudaSuccess; ++g) {
    const int64_t h0 = g * pl.hg, n = (H - h0 < pl.hg) ? H - h0 : pl.hg;
    for (int t = 0; t < 3 && e == cudaSuccess; ++t)
      e = copy_heads(ws + off_in[t] + g * pl.grp_in, src[t], true, nhd, B, S, H, D, h0, n, hs->h2d);
    if (e == cudaSuccess) e = cudaEventRecord(ev_in[g], hs->h2d);
  }
  for (int64_t g = 0; g < pl.G && e == cudaSuccess; ++g) {
    const int64_t h0 = g * pl.hg, n = (H - h0 < pl.hg) ? H - h0 : pl.hg;
    cudaStream_t c = hs->comp[g & 1];
    if ((e = cudaStreamWaitEvent(c, ev_in[g], 0)) != cudaSuccess) break;
    // the group's packed tensors: [B][S][n][D] (NHD) or [B][n][S][D] (HND)
    const int64_t sb = S * n * D, ss = nhd ? n * D : D, sh = nhd ? D : S * D;
    const Bf16In qi{reinterpret_cast<const uint16_t*>(ws + pl.off_q + g * pl.grp_in), sb, ss, sh};
    const Bf16In ki{reinterpret_cast<const uint16_t*>(ws + pl.off_k + g * pl.grp_in), sb, ss, sh};
    const Bf16In vi{reinterpret_cast<const uint16_t*>(ws + pl.off_v + g * pl.grp_in), sb, ss, sh};
    const Out o{reinterpret_cast<uint16_t*>(ws + pl.off_o + g * pl.grp_in), sb, ss, sh};
    const Bundle bundle = carve(ws + pl.off_bundle[g & 1], bundle_layout(B, S, n, D));
    if ((e = launch_prologue(qi, ki, vi, B, S, n, D, smooth_k != 0, bundle, ws + pl.off_scratch[g & 1], false,
                             g_err_ptr[dev], c)) != cudaSuccess)
      break;
    if ((e = launch_attention_tc(bundle, B, S, n, D, scale, o, causal, nullptr, g_err_ptr[dev], c)) != cudaSuccess)
      break;
    e = cudaEventRecord(ev_done[g], c);
  }
  for (int64_t g = 0; g < pl.G && e == cudaSuccess; ++g) {
    const int64_t h0 = g * pl.hg, n = (H - h0 < pl.hg) ? H - h0 : pl.hg;
    if ((e = cudaStreamWaitEvent(hs->d2h, ev_done[g], 0)) != cudaSuccess) break;
    e = copy_heads(out_host, ws + pl.off_o + g * pl.grp_in, false, nhd, B, S, H, D, h0, n, hs->d2h);
  }
  // the caller's stream resumes once every output group is back (the last
  // copy-out follows every kernel: each copy waited for its group)
  if (e == cudaSuccess) e = cudaEventRecord(ev_end, hs->d2h);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(user, ev_end, 0);
  return cuda_status(e);
}

}  // namespace
}  // namespace sage

using namespace sage;

extern "C" {

int sage_bundle_size(int64_t B, int64_t S, int64_t H, int64_t D, size_t* bytes, void* base_dev,
                     sage_quantized* bundle) {
  if (bytes == nullptr) return SAGE_ERR_NULLPTR;
  const int rc = check_sizes(B, S, H, D);
  if (rc != SAGE_OK) return rc;
  const BundleLayout l = bundle_layout(B, S, H, D);
  *bytes = l.total;
  if (base_dev != nullptr) {
    if (bundle == nullptr) return SAGE_ERR_NULLPTR;
    if ((reinterpret_cast<uintptr_t>(base_dev) & 255u) != 0) return SAGE_ERR_ALIGN;
    const Bundle b = carve(base_dev, l);
    bundle->q_codes_dev = b.q_codes;
    bundle->k_codes_dev = b.k_codes;
    bundle->vt_codes_dev = b.vt_codes;
    bundle->q_scale_dev = b.q_scale;
    bundle->k_scale_dev = b.k_scale;
    bundle->v_scale_dev = b.v_scale;
    bundle->k_mean_dev = b.k_mean;
    bundle->q16_dev = b.q16;
    bundle->k16_dev = b.k16;
  }
  return SAGE_OK;
}

int sage_quantize_scratch_size(int64_t B, int64_t S, int64_t H, int64_t D, size_t* bytes) {
  if (bytes == nullptr) return SAGE_ERR_NULLPTR;
  const int rc = check_sizes(B, S, H, D);
  if (rc != SAGE_OK) return rc;
  *bytes = prologue_scratch_bytes(B, S, H, D);
  return SAGE_OK;
}

int sage_workspace_size(int64_t B, int64_t S, int64_t H, int64_t D, size_t* bytes) {
  if (bytes == nullptr) return SAGE_ERR_NULLPTR;
  const int rc = check_sizes(B, S, H, D);
  if (rc != SAGE_OK) return rc;
  *bytes = bundle_layout(B, S, H, D).total + prologue_scratch_bytes(B, S, H, D);
  return SAGE_OK;
}

int sage_host_workspace_size(int64_t B, int64_t S, int64_t H, int64_t D, int n_groups, size_t* bytes) {
  if (bytes == nullptr) return SAGE_ERR_NULLPTR;
  const int rc = check_sizes(B, S, H, D);
  if (rc != SAGE_OK) return rc;
  if (n_groups < 0) return SAGE_ERR_ARG;
  *bytes = host_plan(B, S, H, D, n_groups).total;
  return SAGE_OK;
}

int sage_sageattn_host(const void* q_host, const void* k_host, const void* v_host, const int64_t shape[4],
                       int dtype, const char* tensor_layout, int is_causal, float sm_scale, int smooth_k,
                       void* out_host, int n_groups, void* workspace_dev, size_t workspace_bytes, void* cuda_stream) {
  return sageattn_host_impl(q_host, k_host, v_host, shape, dtype, tensor_layout, is_causal != 0, sm_scale, smooth_k,
                            out_host, n_groups, workspace_dev, workspace_bytes, cuda_stream);
}

int sage_quantize(const sage_bf16_tensor* q, const sage_bf16_tensor* k, const sage_bf16_tensor* v, int64_t B,
                  int64_t S, int64_t H, int64_t D, int smooth_k, const sage_quantized* out, void* scratch_dev,
                  size_t scratch_bytes, void* cuda_stream) {
  int rc = check_sizes(B, S, H, D);
  if (rc != SAGE_OK) return rc;
  if ((rc = check_bf16_in(q)) != SAGE_OK || (rc = check_bf16_in(k)) != SAGE_OK || (rc = check_bf16_in(v)) != SAGE_OK)
    return rc;
  if ((rc = check_bundle(out, true)) != SAGE_OK) return rc;
  if (scratch_dev == nullptr) return SAGE_ERR_NULLPTR;
  if ((reinterpret_cast<uintptr_t>(scratch_dev) & 255u) != 0) return SAGE_ERR_ALIGN;
  if (scratch_bytes < prologue_scratch_bytes(B, S, H, D)) return SAGE_ERR_WORKSPACE;
  int dev = 0;
  if ((rc = check_device(&dev)) != SAGE_OK) return rc;
  if (B == 0 || H == 0 || S == 0) return SAGE_OK;
  const Bf16In qi{static_cast<const uint16_t*>(q->ptr_dev), q->stride_b, q->stride_s, q->stride_h};
  const Bf16In ki{static_cast<const uint16_t*>(k->ptr_dev), k->stride_b, k->stride_s, k->stride_h};
  const Bf16In vi{static_cast<const uint16_t*>(v->ptr_dev), v->stride_b, v->stride_s, v->stride_h};
  return cuda_status(launch_prologue(qi, ki, vi, B, S, H, D, smooth_k != 0, to_bundle(out), scratch_dev, true,
                                     g_err_ptr[dev], static_cast<cudaStream_t>(cuda_stream)));
}

int sage_attention(const sage_quantized* in, int64_t B, int64_t S, int64_t H, int64_t D, float sm_scale,
                   void* out_dev, int64_t ob, int64_t os, int64_t oh, void* cuda_stream) {
  return attention_common(in, B, S, H, D, sm_scale, false, out_dev, ob, os, oh, nullptr, cuda_stream,
                          launch_attention_tc);
}

int sage_attention_ex(const sage_quantized* in, int64_t B, int64_t S, int64_t H, int64_t D, float sm_scale,
                      int is_causal, void* out_dev, int64_t ob, int64_t os, int64_t oh, float* lse_dev,
                      void* cuda_stream) {
  return attention_common(in, B, S, H, D, sm_scale, is_causal != 0, out_dev, ob, os, oh, lse_dev, cuda_stream,
                          launch_attention_tc);
}

int sage_attention_simt(const sage_quantized* in, int64_t B, int64_t S, int64_t H, int64_t D, float sm_scale,
                        int is_causal, void* out_dev, int64_t ob, int64_t os, int64_t oh, float* lse_dev,
                        void* cuda_stream) {
  if (D != kHeadDim) return SAGE_ERR_HEAD_DIM;  // the cross-check kernel is written for 128 channels
  return attention_common(in, B, S, H, D, sm_scale, is_causal != 0, out_dev, ob, os, oh, lse_dev, cuda_stream,
                          simt_adapter);
}

int sage_lse_smooth_k_term(const sage_bf16_tensor* q, const float* k_mean_dev, int64_t B, int64_t S, int64_t H,
                           int64_t D, float sm_scale, float* lse_dev, void* cuda_stream) {
  int rc = check_sizes(B, S, H, D);
  if (rc != SAGE_OK) return rc;
  if ((rc = check_bf16_in(q)) != SAGE_OK) return rc;
  if (k_mean_dev == nullptr || lse_dev == nullptr) return SAGE_ERR_NULLPTR;
  if (!aligned16(k_mean_dev) || !aligned4(lse_dev)) return SAGE_ERR_ALIGN;
  if (!std::isfinite(sm_scale) || !(sm_scale > 0.0f)) return SAGE_ERR_ARG;
  int dev = 0;
  if ((rc = check_device(&dev)) != SAGE_OK) return rc;
  if (B == 0 || H == 0 || S == 0) return SAGE_OK;
  const Bf16In qi{static_cast<const uint16_t*>(q->ptr_dev), q->stride_b, q->stride_s, q->stride_h};
  return cuda_status(launch_lse_smooth_k_term(qi, k_mean_dev, B, S, H, D, sm_scale, lse_dev,
                                              static_cast<cudaStream_t>(cuda_stream)));
}

int sage_sageattn(const void* q_dev, const void* k_dev, const void* v_dev, const int64_t q_shape[4],
                  const int64_t k_shape[4], const int64_t v_shape[4], const int64_t q_strides[4],
                  const int64_t k_strides[4], const int64_t v_strides[4], int q_dtype, int k_dtype, int v_dtype,
                  const char* tensor_layout, int is_causal, float sm_scale, int return_lse, int smooth_k,
                  void* out_dev, const int64_t out_strides[4], int out_dtype, void* workspace_dev,
                  size_t workspace_bytes, void* cuda_stream) {
  // The contract's rejections come first, in the order the pages list them.
  if (is_causal) return SAGE_ERR_CAUSAL;
  if (return_lse) return SAGE_ERR_LSE;
  if (q_dtype == SAGE_DTYPE_BF16 && k_dtype == SAGE_DTYPE_BF16 && v_dtype == SAGE_DTYPE_BF16 &&
      out_dtype == SAGE_DTYPE_BF16 && q_shape != nullptr && q_shape[3] != kHeadDim && q_shape[3] >= 0)
    return SAGE_ERR_HEAD_DIM;
  return sageattn_impl(q_dev, k_dev, v_dev, q_shape, k_shape, v_shape, q_strides, k_strides, v_strides, q_dtype,
                       k_dtype, v_dtype, tensor_layout, false, sm_scale, nullptr, smooth_k, out_dev, out_strides,
                       out_dtype, workspace_dev, workspace_bytes, cuda_stream);
}

int sage_sageattn_ex(const void* q_dev, const void* k_dev, const void* v_dev, const int64_t q_shape[4],
                     const int64_t k_shape[4], const int64_t v_shape[4], const int64_t q_strides[4],
                     const int64_t k_strides[4], const int64_t v_strides[4], int q_dtype, int k_dtype, int v_dtype,
                     const char* tensor_layout, int is_causal, float sm_scale, int smooth_k, void* out_dev,
                     const int64_t out_strides[4], int out_dtype, float* lse_dev, void* workspace_dev,
                     size_t workspace_bytes, void* cuda_stream) {
  return sageattn_impl(q_dev, k_dev, v_dev, q_shape, k_shape, v_shape, q_strides, k_strides, v_strides, q_dtype,
                       k_dtype, v_dtype, tensor_layout, is_causal != 0, sm_scale, lse_dev, smooth_k, out_dev,
                       out_strides, out_dtype, workspace_dev, workspace_bytes, cuda_stream);
}

int sage_sageattn_args_call(const sage_sageattn_args* a) {
  if (a == nullptr) return SAGE_ERR_NULLPTR;
  char layout[5] = {a->tensor_layout[0], a->tensor_layout[1], a->tensor_layout[2], a->tensor_layout[3], 0};
  if (layout[3] != 0) return SAGE_ERR_LAYOUT;
  return sageattn_impl(a->q_dev, a->k_dev, a->v_dev, a->q_shape, a->k_shape, a->v_shape, a->q_strides,
                       a->k_strides, a->v_strides, a->q_dtype, a->k_dtype, a->v_dtype, layout, a->is_causal != 0,
                       a->sm_scale, a->lse_dev, a->smooth_k, a->out_dev, a->out_strides, a->out_dtype,
                       a->workspace_dev, a->workspace_bytes, a->cuda_stream);
}

int sage_device_error(void* cuda_stream, int* code) {
  if (code == nullptr) return SAGE_ERR_NULLPTR;
  int dev = 0;
  int rc = check_device(&dev);
  if (rc != SAGE_OK) return rc;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SAGE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, g_err_ptr[dev], sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SAGE_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(g_err_ptr[dev], &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return SAGE_ERR_CUDA;
  *code = v == 0 ? SAGE_OK : (v == kDevErrSmemAlign ? SAGE_ERR_DEVICE_SMEM : SAGE_ERR_DEVICE_TIMEOUT);
  return SAGE_OK;
}

int sage_selftest_wait_timeout(void* cuda_stream) {
  int dev = 0;
  const int rc = check_device(&dev);
  if (rc != SAGE_OK) return rc;
  return cuda_status(launch_wait_timeout_selftest(g_err_ptr[dev], static_cast<cudaStream_t>(cuda_stream)));
}

const char* sage_strerror(int code) {
  switch (code) {
    case SAGE_OK: return "success";
    case SAGE_ERR_CAUSAL: return "is_causal is not supported (non-causal attention only)";
    case SAGE_ERR_LSE: return "return_lse is not supported";
    case SAGE_ERR_DTYPE: return "inputs and output must be bfloat16";
    case SAGE_ERR_HEAD_DIM: return "head dimension must be 128 (or 64 on the entries that take it)";
    case SAGE_ERR_SHAPE: return "q, k and v must have identical, non-negative shapes";
    case SAGE_ERR_LAYOUT: return "tensor_layout must be \"NHD\" or \"HND\" with a unit channel stride";
    case SAGE_ERR_ALIGN: return "pointers must be 16-byte aligned and strides multiples of 8 elements";
    case SAGE_ERR_NULLPTR: return "a required pointer is NULL";
    case SAGE_ERR_WORKSPACE: return "workspace or scratch buffer is too small";
    case SAGE_ERR_ARCH: return "the current device is not compute capability 10.3 (sm_103)";
    case SAGE_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case SAGE_ERR_DEVICE_TIMEOUT: return "a kernel gave up waiting on an internal barrier";
    case SAGE_ERR_ARG: return "invalid argument (sm_scale must be finite and positive)";
    case SAGE_ERR_TOO_LARGE: return "sizes exceed the library's limits";
    case SAGE_ERR_DEVICE_SMEM: return "a kernel found its shared memory window misaligned and did no work";
    default: return "unknown error code";
  }
}

}  // extern "C"
