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
// Eight lanes per row, four rows per warp; lane i of a row holds columns
// 32j + 4i .. 32j + 4i + 3 (j < d/32), so that the eight lanes of a row read
// 128 contiguous bytes of a partial row per load and write contiguous output
// per store.  Small: it reads nsplit * d + 2 floats per row, from
// L2 as a rule, so its cost is load latency and the per-row scalar work (the
// weights 2^(m_s - M) and 1 / l); the loads of up to four partial rows are
// issued together and the scalar work is shared by eight lanes instead of 32.

#include <cuda_bf16.h>

#include <type_traits>

#include "internal.h"
#include "sm100.cuh"
#include "work.cuh"

namespace sa {
namespace {

constexpr int kLanesPerRow = 8;                       // lanes sharing one output row
constexpr int kRowsPerCta = 256 / kLanesPerRow;          // 256 threads, 32 rows
constexpr int kSegBatch = 4;                             // partial rows whose loads are issued together

// Merges the nseg partial rows seg(0), seg(1), ... of one output row; called
// by the kLanesPerRow lanes of the row, lane i of them holding the columns
// 32j + 4i + c (out[4j + c], j < D/32, c < 4).  The loads of kSegBatch segments
// (their (m, l) and their O rows) are issued before any is used, so a row
// costs one memory round trip with up to four segments; the
// arithmetic is the same in every case: M first, then the weighted sums in
// segment order.
template <int D, typename SegRow>
__device__ __forceinline__ void merge_partials(const SplitOut& part, int nseg, SegRow seg,
                                               float (&out)[D / kLanesPerRow]) {
  constexpr int V = D / kLanesPerRow, V4 = V / 4;
  const int sub = threadIdx.x % kLanesPerRow;
  float mmax = -INFINITY, lsum = 0.f;
  float acc[V];
#pragma unroll
  for (int c = 0; c < V; ++c) acc[c] = 0.f;
  auto load = [&](int k, float2& ml, float4 (&a)[V4]) {
    const long long r = seg(k);
    ml = *reinterpret_cast<const float2*>(part.ml + 2 * r);
    const float4* src = reinterpret_cast<const float4*>(part.o + r * D);
#pragma unroll
    for (int j = 0; j < V4; ++j) a[j] = src[j * kLanesPerRow + sub];
  };
  auto accumulate = [&](const float2& ml, const float4 (&a)[V4]) {
    if (!(ml.y > 0.f)) return;                          // an empty segment (its O row is not read)
    const float w = exp2f(ml.x - mmax);
    lsum = fmaf(w, ml.y, lsum);
#pragma unroll
    for (int j = 0; j < V4; ++j) {
      acc[4 * j + 0] = fmaf(w, a[j].x, acc[4 * j + 0]);
      acc[4 * j + 1] = fmaf(w, a[j].y, acc[4 * j + 1]);
      acc[4 * j + 2] = fmaf(w, a[j].z, acc[4 * j + 2]);
      acc[4 * j + 3] = fmaf(w, a[j].w, acc[4 * j + 3]);
    }
  };
  if (nseg <= kSegBatch) {
    float2 ml[kSegBatch];
    float4 a[kSegBatch][V4];
#pragma unroll
    for (int i = 0; i < kSegBatch; ++i) {
      if (i < nseg)
        load(i, ml[i], a[i]);
      else
        ml[i] = make_float2(-INFINITY, 0.f);
    }
#pragma unroll
    for (int i = 0; i < kSegBatch; ++i)
      if (ml[i].y > 0.f) mmax = fmaxf(mmax, ml[i].x);
#pragma unroll
    for (int i = 0; i < kSegBatch; ++i) accumulate(ml[i], a[i]);
  } else {
    for (int k0 = 0; k0 < nseg; k0 += kSegBatch) {
      float2 ml[kSegBatch];
#pragma unroll
      for (int i = 0; i < kSegBatch; ++i)
        ml[i] = k0 + i < nseg ? *reinterpret_cast<const float2*>(part.ml + 2 * seg(k0 + i))
                              : make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int i = 0; i < kSegBatch; ++i)
        if (ml[i].y > 0.f) mmax = fmaxf(mmax, ml[i].x);
    }
    for (int k0 = 0; k0 < nseg; k0 += kSegBatch) {
      float2 ml[kSegBatch];
      float4 a[kSegBatch][V4];
#pragma unroll
      for (int i = 0; i < kSegBatch; ++i) {
        if (k0 + i < nseg)
          load(k0 + i, ml[i], a[i]);
        else
          ml[i] = make_float2(-INFINITY, 0.f);
      }
#pragma unroll
      for (int i = 0; i < kSegBatch; ++i) accumulate(ml[i], a[i]);
    }
  }
  const float inv = 1.f / lsum;
#pragma unroll
  for (int c = 0; c < V; ++c) out[c] = acc[c] * inv;
}

// Stores a lane's columns 32j + 4i + c of the output row starting at element
// idx (rows are 16-byte aligned; i = the lane's index within its row).
template <int D, bool OUT32>
__device__ __forceinline__ void store_row_part(void* out, long long idx, const float (&v)[D / kLanesPerRow]) {
  constexpr int V4 = D / kLanesPerRow / 4;
  const int sub = threadIdx.x % kLanesPerRow;
  if constexpr (OUT32) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + idx);
#pragma unroll
    for (int j = 0; j < V4; ++j)
      o[j * kLanesPerRow + sub] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  } else {
    uint2* o = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + idx);
#pragma unroll
    for (int j = 0; j < V4; ++j) {
      const __nv_bfloat162 h0 = __floats2bfloat162_rn(v[4 * j], v[4 * j + 1]);
      const __nv_bfloat162 h1 = __floats2bfloat162_rn(v[4 * j + 2], v[4 * j + 3]);
      o[j * kLanesPerRow + sub] =
          make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
    }
  }
}

template <int D, bool OUT32>
__global__ void __launch_bounds__(kRowsPerCta * kLanesPerRow) splitkv_combine_kernel(const SplitOut part, int nsplit,
                                                                         long long nrows, int L, int Lp,
                                                                         long long split_rows, int H,
                                                                         const Strides so, void* out) {
  pdl_wait();                                        // the partial results are written
  const long long row = (long long)blockIdx.x * kRowsPerCta + threadIdx.x / kLanesPerRow;
  if (row >= nrows) return;
  const long long bh = row / L;
  const long long prow = bh * Lp + row % L;          // row in the padded partial layout
  float v[D / kLanesPerRow];
  merge_partials<D>(part, nsplit, [&](int s) { return s * split_rows + prow; }, v);
  store_row_part<D, OUT32>(out, (bh / H) * so.b + (bh % H) * so.h + (row % L) * so.t, v);
}

template <int D, bool OUT32>
cudaError_t launch(const SplitOut& part, int nsplit, const Dims& dm, void* o, const Strides& so, cudaStream_t s) {
  const long long nrows = (long long)dm.B * dm.H * dm.Lq;
  const int Lp = padded_len(dm.Lq);
  const long long split_rows = (long long)dm.B * dm.H * Lp;
  const long long ctas = (nrows + kRowsPerCta - 1) / kRowsPerCta;
  // a programmatic dependent launch behind the attention kernel: its launch
  // is processed while the attention CTAs finish
  cudaLaunchAttribute attr;
  const cudaLaunchConfig_t cfg = pdl_launch_config(dim3((unsigned)ctas), dim3(kRowsPerCta * kLanesPerRow), 0, s, &attr);
  return cudaLaunchKernelEx(&cfg, splitkv_combine_kernel<D, OUT32>, part, nsplit, nrows, dm.Lq, Lp, split_rows, dm.H,
                            so, o);
}

// Stream-K: CTAs (k, y) for cut pair k and y in 0..7, 32 rows each, so the
// latency-bound row merges run spread over the GPU.  A cut
// pair's segments -- one per CTA whose range meets it -- are merged into O;
// pairs no boundary cuts were written whole by the attention kernel.
template <int D, bool OUT32>
__global__ void __launch_bounds__(kRowsPerCta * kLanesPerRow) streamk_combine_kernel(const __grid_constant__ StreamKCuts cuts,
                                                                         const SplitOut part, int L, int H,
                                                                         const Strides so, void* out) {
  pdl_wait();                                        // the partial results are written
  const int* e = cuts.e[blockIdx.x];
  const int bh = e[0], qt0 = e[1], nq = e[2], cta0 = e[3], nseg = e[4] - e[3] + 1, first_last = e[5];
  const int rr = blockIdx.y * kRowsPerCta + threadIdx.x / kLanesPerRow;   // row of the pair (query tile rr / 128)
  const int t = qt0 * 128 + rr;                                  // its token
  if (rr >= nq * 128 || t >= L) return;
  float v[D / kLanesPerRow];
  merge_partials<D>(
      part, nseg, [&](int k) { return (long long)(2 * (cta0 + k) + (k == 0 ? first_last : 0)) * 256 + rr; }, v);
  store_row_part<D, OUT32>(out, (long long)(bh / H) * so.b + (long long)(bh % H) * so.h + (long long)t * so.t, v);
}

template <int D, bool OUT32>
cudaError_t launch_sk(const AttnWork& w, int ctas, const SplitOut& part, const Dims& dm, void* o, const Strides& so,
                      cudaStream_t s) {
  StreamKCuts cuts;
  make_streamk_cuts(w, ctas, &cuts);
  if (cuts.n == 0) return cudaSuccess;               // no pair was cut
  cudaLaunchAttribute attr;
  const cudaLaunchConfig_t cfg =
      pdl_launch_config(dim3(cuts.n, 256 / kRowsPerCta), dim3(kRowsPerCta * kLanesPerRow), 0, s, &attr);
  return cudaLaunchKernelEx(&cfg, streamk_combine_kernel<D, OUT32>, cuts, part, dm.Lq, dm.H, so, o);
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
