// splitkv.cu -- the combine pass of split-KV attention.
//
// With split-KV each CTA of an attention kernel covers a contiguous share of
// a query tile's key tiles (online softmax, "FlashAttention kernels",
// sections 0-1) and leaves, per row, its unnormalised accumulator a_s, its row
// sum l_s -- both in units of 2^m_s for the split's own reference maximum m_s
// (log2 units; -inf when no key of the share was visible) -- instead of O.
// Merging the shares is the online-softmax rescaling step applied once more:
//   M = max_s m_s,  O = sum_s 2^(m_s - M) a_s / sum_s 2^(m_s - M) l_s.
// In the NVFP4 path every share has the same extra factor 1/2688 in both a_s
// and l_s (the first P level), so it cancels here as it does in O = A / lam.
// The P quantisation is per key tile, and shares are whole key tiles, so the
// split changes only the float32 summation order.
//
// One warp per row; lane i holds columns i, i + 32, ... (coalesced 128-byte
// rows).  Memory-bound and small: it reads nsplit * d + 2 floats per row.

#include <cuda_bf16.h>

#include "internal.h"
#include "work.cuh"

namespace sa {
namespace {

constexpr int kRowsPerCta = 8;

template <int D, bool OUT32>
__global__ void __launch_bounds__(32 * kRowsPerCta) splitkv_combine_kernel(const SplitOut part, int nsplit,
                                                                         long long nrows, int L, int Lp,
                                                                         long long split_rows, int H,
                                                                         const Strides so, void* out) {
  const long long row = (long long)blockIdx.x * kRowsPerCta + threadIdx.x / 32;
  if (row >= nrows) return;
  const int lane = threadIdx.x % 32;
  const long long bh = row / L;
  const long long prow = bh * Lp + row % L;          // row in the padded partial layout
  float mmax = -INFINITY;
  for (int s = 0; s < nsplit; ++s) {
    const float2 ml = *reinterpret_cast<const float2*>(part.ml + 2 * (s * split_rows + prow));
    if (ml.y > 0.f) mmax = fmaxf(mmax, ml.x);
  }
  float acc[D / 32];
#pragma unroll
  for (int i = 0; i < D / 32; ++i) acc[i] = 0.f;
  float lsum = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float2 ml = *reinterpret_cast<const float2*>(part.ml + 2 * (s * split_rows + prow));
    if (!(ml.y > 0.f)) continue;                     // an empty share (its a_s is never read)
    const float w = exp2f(ml.x - mmax);
    lsum = fmaf(w, ml.y, lsum);
    const float* a = part.o + (s * split_rows + prow) * D;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] = fmaf(w, a[lane + 32 * i], acc[i]);
  }
  const float inv = 1.f / lsum;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    const long long idx = (bh / H) * so.b + (bh % H) * so.h + (row % L) * so.t + lane + 32 * i;
    if constexpr (OUT32)
      static_cast<float*>(out)[idx] = acc[i] * inv;
    else
      static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(acc[i] * inv);
  }
}

template <int D, bool OUT32>
cudaError_t launch(const SplitOut& part, int nsplit, const Dims& dm, void* o, const Strides& so, cudaStream_t s) {
  const long long nrows = (long long)dm.B * dm.H * dm.Lq;
  const int Lp = padded_len(dm.Lq);
  const long long split_rows = (long long)dm.B * dm.H * Lp;
  const long long ctas = (nrows + kRowsPerCta - 1) / kRowsPerCta;
  splitkv_combine_kernel<D, OUT32><<<(unsigned)ctas, 32 * kRowsPerCta, 0, s>>>(part, nsplit, nrows, dm.Lq, Lp,
                                                                              split_rows, dm.H, so, o);
  return cudaGetLastError();
}

// Stream-K: CTAs (k, y) for cut pair k and y in 0..31, eight rows each (one
// per warp), so the latency-bound row merges run spread over the GPU.  A cut
// pair's segments -- one per CTA whose range meets it -- are merged into O;
// pairs no boundary cuts were written whole by the attention kernel.
template <int D, bool OUT32>
__global__ void __launch_bounds__(32 * kRowsPerCta) streamk_combine_kernel(const __grid_constant__ StreamKCuts cuts,
                                                                         const SplitOut part, int L, int H,
                                                                         const Strides so, void* out) {
  const int* e = cuts.e[blockIdx.x];
  const int bh = e[0], qt0 = e[1], nq = e[2], cta0 = e[3], nseg = e[4] - e[3] + 1, first_last = e[5];
  const int rr = blockIdx.y * kRowsPerCta + threadIdx.x / 32;   // row of the pair (query tile rr / 128)
  const int t = qt0 * 128 + rr;                                  // its token
  if (rr >= nq * 128 || t >= L) return;
  const int lane = threadIdx.x % 32;
  float mmax = -INFINITY;
  for (int k = 0; k < nseg; ++k) {
    const long long prow = (long long)(2 * (cta0 + k) + (k == 0 ? first_last : 0)) * 256 + rr;
    const float2 ml = *reinterpret_cast<const float2*>(part.ml + 2 * prow);
    if (ml.y > 0.f) mmax = fmaxf(mmax, ml.x);
  }
  float acc[D / 32];
#pragma unroll
  for (int i = 0; i < D / 32; ++i) acc[i] = 0.f;
  float lsum = 0.f;
  for (int k = 0; k < nseg; ++k) {
    const long long prow = (long long)(2 * (cta0 + k) + (k == 0 ? first_last : 0)) * 256 + rr;
    const float2 ml = *reinterpret_cast<const float2*>(part.ml + 2 * prow);
    if (!(ml.y > 0.f)) continue;                     // a segment without keys for this row
    const float wgt = exp2f(ml.x - mmax);
    lsum = fmaf(wgt, ml.y, lsum);
    const float* a = part.o + prow * D;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] = fmaf(wgt, a[lane + 32 * i], acc[i]);
  }
  const float inv = 1.f / lsum;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    const long long idx = (long long)(bh / H) * so.b + (long long)(bh % H) * so.h + (long long)t * so.t + lane + 32 * i;
    if constexpr (OUT32)
      static_cast<float*>(out)[idx] = acc[i] * inv;
    else
      static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(acc[i] * inv);
  }
}

template <int D, bool OUT32>
cudaError_t launch_sk(const AttnWork& w, int ctas, const SplitOut& part, const Dims& dm, void* o, const Strides& so,
                      cudaStream_t s) {
  StreamKCuts cuts;
  make_streamk_cuts(w, ctas, &cuts);
  if (cuts.n == 0) return cudaSuccess;               // no pair was cut
  streamk_combine_kernel<D, OUT32><<<dim3(cuts.n, 256 / kRowsPerCta), 32 * kRowsPerCta, 0, s>>>(cuts, part, dm.Lq,
                                                                                                dm.H, so, o);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_streamk_combine(const AttnWork& w, int ctas, const SplitOut& part, const Dims& dm, void* o,
                                   const Strides& so, bool out_f32, cudaStream_t s) {
  if (dm.d == 64)
    return out_f32 ? launch_sk<64, true>(w, ctas, part, dm, o, so, s) : launch_sk<64, false>(w, ctas, part, dm, o, so, s);
  return out_f32 ? launch_sk<128, true>(w, ctas, part, dm, o, so, s) : launch_sk<128, false>(w, ctas, part, dm, o, so, s);
}

cudaError_t launch_splitkv_combine(const SplitOut& part, int nsplit, const Dims& dm, void* o, const Strides& so,
                                   bool out_f32, cudaStream_t s) {
  if (dm.d == 64)
    return out_f32 ? launch<64, true>(part, nsplit, dm, o, so, s) : launch<64, false>(part, nsplit, dm, o, so, s);
  return out_f32 ? launch<128, true>(part, nsplit, dm, o, so, s) : launch<128, false>(part, nsplit, dm, o, so, s);
}

}  // namespace sa
