// internal.h -- launchers shared between the translation units of libsa.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/sa.h"

namespace sa {

// Sizes of one problem: Q [B, H, Lq, d], K and V [B, Hkv, Lkv, d].
struct Dims {
  int B, H, Hkv, Lq, Lkv, d;
};

// The sequence length padded to whole 128-token tiles: the row count of every
// quantised layout (rows past L hold zero codes and zero scales).
inline int padded_len(int L) { return (L + 127) & ~127; }

// Element strides of a bf16 (or float32 output) tensor of `heads` heads with d
// contiguous: element (b, h, t, c) sits at b*b_ + h*h_ + t*t_ + c.  BHLD
// ([B, heads, L, d]) and BLHD ([B, L, heads, d], flag SA_LAYOUT_BLHD).
struct Strides {
  long long b, h, t;
};
inline Strides layout_strides(bool blhd, int heads, int L, int d) {
  return blhd ? Strides{(long long)L * heads * d, d, (long long)heads * d}
              : Strides{(long long)heads * L * d, (long long)L * d, d};
}

// Per-device once-only set-up (kernel attributes such as the dynamic
// shared-memory size are properties of a function on one device): run(), a
// callable returning cudaError_t, on the first call for the current device;
// later calls on that device return cudaSuccess.  Concurrent first calls may
// both run it (the set-up is idempotent).
constexpr int kMaxDevices = 64;
template <typename F>
inline cudaError_t once_per_device(std::atomic<bool> (&done)[kMaxDevices], F run) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = run();
  if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
  return e;
}

// Number of SMs of the current device (cached per device; 0 if unknown).
inline int device_sm_count() {
  static std::atomic<int> cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < kMaxDevices && cache[dev].load(std::memory_order_relaxed) > 0) return cache[dev].load();
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Launch configuration of a programmatic dependent launch: the kernel may
// start while the kernel before it in the stream finishes (once that one's
// CTAs have all signalled griddepcontrol.launch_dependents or exited) and
// must execute griddepcontrol.wait before it reads anything that kernel
// writes.  `attr` is the caller's storage for the one launch attribute.
inline cudaLaunchConfig_t pdl_launch_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                            cudaLaunchAttribute* attr) {
  attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr->val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c = {};
  c.gridDim = grid;
  c.blockDim = block;
  c.dynamicSmemBytes = smem;
  c.stream = s;
  c.attrs = attr;
  c.numAttrs = 1;
  return c;
}

// The softmax scale in base-2 units, c = log2(e) / sqrt(d), rounded once to
// float32 (d = 64: log2(e) / 8; d = 128: log2(e) * 2^-3.5).
template <int D>
__host__ __device__ constexpr float softmax_scale_log2() {
  static_assert(D == 64 || D == 128, "head dimension");
  return static_cast<float>(1.4426950408889634074 * (D == 64 ? 0.125 : 0.088388347648318440550));
}

// Barrier-wait limit used by the attention kernels (nanoseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// quant.cu
// The smooth-K mean is summed in chunks of kMeanChunk tokens (one float32
// partial sum per chunk and channel, then the chunk sums in order); a problem
// needs kmean_partial_floats(dm) floats of partial sums.
constexpr int kMeanChunk = 128;
inline size_t kmean_partial_floats(const Dims& dm) {
  return (size_t)dm.B * dm.Hkv * (size_t)(padded_len(dm.Lkv) / kMeanChunk) * (size_t)dm.d;
}
// tq / tk / tv: the bf16 Q, K and V heads (make_bf16_head_map: boxes of 64
// channels x 128 tokens, 128B swizzle, zeros past L).  with_q false: K and V
// only (out.q_codes / out.q_sf untouched, tq unused), for the attention
// kernel that quantises Q itself.
cudaError_t launch_quantize(const Dims& dm, const sa_fp4_qkv& out, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, cudaStream_t s, bool with_q = true);
// Same kernels, K-mean partial sums in the library's fixed per-device array.
constexpr size_t kStaticScratchFloats = SA_STATIC_SCRATCH_FLOATS;
cudaError_t launch_quantize_static_scratch(const Dims& dm, const sa_fp4_qkv& out, const CUtensorMap& tq,
                                           const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s);

// Split-KV partial results (device, caller's workspace): for split s and
// padded row R = (b*H + h)*Lp + t, the unnormalised O row at o + (s*rows + R)*d
// and (m, l) at ml + 2*(s*rows + R), rows = B*H*Lp.  Unused with nsplit 1.
struct SplitOut {
  float* o;
  float* ml;
};
inline size_t splitkv_workspace_bytes(const Dims& dm, int nsplit) {
  const size_t rows = (size_t)dm.B * dm.H * padded_len(dm.Lq);
  return nsplit > 1 ? (size_t)nsplit * rows * ((size_t)dm.d + 2) * sizeof(float) : 0;
}
inline SplitOut splitkv_layout(void* ws, const Dims& dm, int nsplit) {
  const size_t rows = (size_t)dm.B * dm.H * padded_len(dm.Lq);
  float* f = static_cast<float*>(ws);
  return SplitOut{f, f + (size_t)nsplit * rows * dm.d};
}

// attn_bf16.cu
cudaError_t launch_attn_bf16(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, void* o,
                             const Strides& so, const Dims& dm, int causal, bool out_f32, int nsplit,
                             const SplitOut& part, cudaStream_t s);
// attn_nvfp4.cu.  ds: the smooth-Q score corrections ([B*H][Lqp/128][Lkvp]
// float32, added to every score of its query tile and key before the
// softmax), or nullptr for the plain SA3 path.
// fuse_q: Q arrives in bf16 (tq a make_bf16_head_map of it) and the kernel
// quantises it itself, with sa_quantize's arithmetic (qkv.q_codes / q_sf
// unused).
cudaError_t launch_attn_nvfp4(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const sa_fp4_qkv& qkv, void* o, const Strides& so, const Dims& dm, int causal,
                              bool out_f32, int nsplit, const SplitOut& part, cudaStream_t s,
                              const float* ds = nullptr, bool fuse_q = false);
// smooth_q.cu: after sa_quantize, Q re-quantised as Q' = Q - its 128-token
// block mean (x.q_codes / x.q_sf overwritten, the means to qmean
// [B*H][Lqp/128][d]) and the score corrections ds [B*H][Lqp/128][Lkvp] from
// the means and x.k_codes / x.k_sf.  q: bf16 with element strides sq.
cudaError_t launch_smooth_q(const void* q, const Strides& sq, const Dims& dm, const sa_fp4_qkv& x, float* qmean,
                            float* ds, cudaStream_t s);
// Test support: the FP32 score tile of the NVFP4 attention kernel's S step for
// query tile qt of head (b, h) and key tile kt of its kv head, [128][128] to
// `out` (device); tq / tk as for launch_attn_nvfp4.
cudaError_t launch_nvfp4_score_tile(const CUtensorMap& tq, const CUtensorMap& tk, const sa_fp4_qkv& x,
                                    const Dims& dm, int b, int h, int qt, int kt, float* out, cudaStream_t s);
// Test support: ex2_out[i] = the softmax's exp2 of x[i], lg2_out[i] = its
// log2 of y[i] (device buffers of n floats).
cudaError_t launch_exp_path_selftest(const float* x, const float* y, int n, float* ex2_out, float* lg2_out,
                                     cudaStream_t s);
// attn_decode.cu: NVFP4 attention for problems with at most 16 query rows per
// kv head ((H / Hkv) * Lq <= 16: decode steps), the rows of a kv head's query
// heads taken together; tk / tv as for launch_attn_nvfp4.  nsplit key shares
// per (batch, kv head) (partial results and splitkv.cu's combine when > 1).
// nsplit kStreamK: equal ranges of the (pair, key tile) items over
// decode_range_ctas CTAs, partial results of cut pairs in a workspace of
// decode_range_workspace_bytes (two slots of 16 rows per CTA).
bool decode_eligible(const Dims& dm);
int decode_nsplit(const Dims& dm, int sms);
int decode_range_ctas(const Dims& dm, int sms);
size_t decode_range_workspace_bytes(const Dims& dm, int sms);
SplitOut decode_range_layout(void* ws, const Dims& dm, int sms);
cudaError_t launch_attn_decode(const CUtensorMap& tk, const CUtensorMap& tv, const sa_fp4_qkv& x, void* o,
                               const Strides& so, const Dims& dm, int causal, bool out_f32, int nsplit,
                               const SplitOut& part, cudaStream_t s);
// splitkv.cu: O from the nsplit partial results of every row t < L.
cudaError_t launch_splitkv_combine(const SplitOut& part, int nsplit, const Dims& dm, void* o, const Strides& so,
                                   bool out_f32, cudaStream_t s);

// Stream-K (nsplit == kStreamK): persistent CTAs, one per SM, over equal
// ranges of (pair, key tile) items.  A pair cut by a range boundary leaves
// partial results in two slots per CTA (slot 2c: the CTA's first unit, 2c + 1:
// its last), 2 * BM rows of d + 2 floats each.
constexpr int kStreamK = -1;
inline size_t streamk_workspace_bytes(const Dims& dm, int ctas) {
  return (size_t)2 * ctas * 256 * ((size_t)dm.d + 2) * sizeof(float);
}
struct AttnWork;
cudaError_t launch_streamk_combine(const AttnWork& w, int ctas, const SplitOut& part, const Dims& dm, void* o,
                                   const Strides& so, bool out_f32, cudaStream_t s);
inline SplitOut streamk_layout(void* ws, const Dims& dm, int ctas) {
  float* f = static_cast<float*>(ws);
  return SplitOut{f, f + (size_t)2 * ctas * 256 * dm.d};
}

// Per-unit readers of the device error word (each clears its word).
cudaError_t attn_bf16_read_error(int* out);
cudaError_t attn_nvfp4_read_error(int* out);
cudaError_t quant_read_error(int* out);

}  // namespace sa
