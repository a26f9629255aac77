// smooth_q.cu -- the smooth-Q variant's quantiser and score correction.
//
// Source: page "kernel overview", SageAttention evolution chain ("Smooth-K ->
// Smooth-Q+K"): besides subtracting the token mean of K, Q is smoothed by
// subtracting its mean over a block of tokens before quantisation, and the
// block mean's share of the scores is added back.  The block is the
// attention kernel's 128-row query tile of one head.  For tile i of a head:
//   qbar_i = (sum of the tile's valid rows, float32, row by row from 0) / n_i
//   Q'_t   = RN(q_t - qbar_i), quantised as Q (1x16 groups along d, e4m3
//            scales, e2m1 codes; IEEE float32 quotients, so the codes are
//            bit-exact functions of the inputs)
//   dS[i, j] = qbar_i . K^'_j      (K^' the dequantised smoothed key row j)
// so that the attention kernel's scores Q^'_t K^'^T + dS[i] equal
// (Q^'_t + qbar_i) K^'^T: only Q's representation changes.
//
// Two launches after sa_quantize (which leaves K^', V^ and the plain Q codes):
// sq_quant_kernel overwrites the Q codes and scales with those of Q' and
// writes qbar; sq_ds_kernel forms dS from qbar and the K codes and scales.
// dS: per 1x16 group g of key row j, t_g = sum over the group's channels of
// qbar_c * e2m1_c (FMA chain in channel order from 0), then
// dS = sum over groups of t_g * s_g (FMA chain in group order from 0); its
// error is below (D/16 + 17) * 2^-24 * sum_c |qbar_c K^'_jc|.

#include <cuda_bf16.h>

#include "internal.h"
#include "sm100.cuh"

namespace sa {
namespace {

constexpr int kSqRows = 128;                         // rows of a Q block (the attention kernel's query tile)

// e2m1 nibble -> float, exactly: magnitude 0, 0.5 for exponent field 0,
// else 2^(e - 1) * (1 + m / 2); sign from bit 3.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  const uint32_t mag = e ? (((126u + e) << 23) | (m << 22)) : (m ? 0x3F000000u : 0u);
  return __uint_as_float(mag | ((c & 8u) << 28));
}

// One CTA per (batch * head, query tile); thread r owns row r of the tile.
template <int D>
__global__ void __launch_bounds__(kSqRows)
    sq_quant_kernel(const __nv_bfloat16* __restrict__ q, const Strides sq, int H, int Lq, int Lqp,
                    uint8_t* __restrict__ qc, uint8_t* __restrict__ qsf, float* __restrict__ qmean) {
  // rows padded by 16 bytes: a quarter-warp's 16-byte reads of 8 rows at
  // the same column hit distinct banks
  constexpr int kStride = D + 8;
  __shared__ __align__(16) __nv_bfloat16 tile[kSqRows * kStride];
  __shared__ float mean[D];
  const int nqt = Lqp / kSqRows;
  const int bh = blockIdx.x / nqt, qt = blockIdx.x % nqt;
  const int b = bh / H, h = bh % H;
  const int t0 = qt * kSqRows;
  const int n = min(kSqRows, Lq - t0);                 // valid rows (>= 1: the tile holds a row < Lq)
  // the tile, 16-byte chunks; rows past Lq as zeros
  for (int i = threadIdx.x; i < kSqRows * D / 8; i += kSqRows) {
    const int r = i / (D / 8), c8 = (i % (D / 8)) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < n)
      v = *reinterpret_cast<const uint4*>(q + (long long)b * sq.b + (long long)h * sq.h + (long long)(t0 + r) * sq.t +
                                          c8);
    *reinterpret_cast<uint4*>(tile + r * kStride + c8) = v;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < D; c += kSqRows) {
    float s = 0.f;
    for (int r = 0; r < n; ++r) s = __fadd_rn(s, __bfloat162float(tile[r * kStride + c]));
    const float m = __fdiv_rn(s, static_cast<float>(n));
    mean[c] = m;
    qmean[((size_t)bh * nqt + qt) * D + c] = m;
  }
  __syncthreads();
  const int r = threadIdx.x;
  uint32_t codes[D / 8];
  uint32_t sfw[D / 64];
#pragma unroll
  for (int k = 0; k < D / 64; ++k) sfw[k] = 0u;
#pragma unroll
  for (int g = 0; g < D / 16; ++g) {
    float x[16];
    float amax = 0.f;
    const uint4* src = reinterpret_cast<const uint4*>(tile + r * kStride + 16 * g);
    const uint4 w0 = src[0], w1 = src[1];
    const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      // rows past Lq stay zero (zero codes and scales, as in every layout)
      const float qv = __uint_as_float(i & 1 ? (w[i / 2] & 0xFFFF0000u) : (w[i / 2] << 16));
      x[i] = r < n ? __fsub_rn(qv, mean[16 * g + i]) : 0.f;
      amax = fmaxf(amax, fabsf(x[i]));
    }
    const uint32_t s8 = cvt_e4m3x2(__fdiv_rn(amax, 6.0f), 0.f) & 0xFFu;
    const float s = e4m3_to_f32(s8);
    float y[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = s8 ? __fdiv_rn(x[i], s) : 0.f;
    codes[2 * g] = s8 ? cvt_e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]) : 0u;
    codes[2 * g + 1] = s8 ? cvt_e2m1x8(y[8], y[9], y[10], y[11], y[12], y[13], y[14], y[15]) : 0u;
    sfw[g / 4] |= s8 << (8 * (g % 4));
  }
  uint4* cdst = reinterpret_cast<uint4*>(qc + ((size_t)bh * Lqp + t0 + r) * (D / 2));
#pragma unroll
  for (int i = 0; i < D / 32; ++i)
    cdst[i] = make_uint4(codes[4 * i], codes[4 * i + 1], codes[4 * i + 2], codes[4 * i + 3]);
  // scale word of row r in 64-channel block k: byte (r % 32) * 16 + (r / 32) * 4 of the block
#pragma unroll
  for (int k = 0; k < D / 64; ++k)
    *reinterpret_cast<uint32_t*>(qsf + (((size_t)bh * nqt + qt) * (D / 64) + k) * 512 + (r & 31) * 16 +
                                 (r >> 5) * 4) = sfw[k];
}

constexpr int kDsStage = 16;                         // query tiles whose means are staged at once

// One CTA per (batch * head, key tile); thread j owns key row j of the tile
// (its kv head's smoothed key, dequantised once into registers) and writes
// dS of that key for every query tile of the head.
template <int D>
__global__ void __launch_bounds__(kSqRows)
    sq_ds_kernel(const uint8_t* __restrict__ kc, const uint8_t* __restrict__ ksf, const float* __restrict__ qmean,
                 int H, int Hkv, int Lqp, int Lkvp, float* __restrict__ ds) {
  __shared__ __align__(16) float qb[kDsStage * D];
  const int bh = blockIdx.x, kt = blockIdx.y;
  const int nqt = Lqp / kSqRows;
  const int G = H / Hkv;
  const long long bhk = (long long)(bh / H) * Hkv + (bh % H) / G;
  const int j = threadIdx.x, key = kt * kSqRows + j;
  float kv[D];
  float sg[D / 16];
  const uint4* crow = reinterpret_cast<const uint4*>(kc + ((size_t)bhk * Lkvp + key) * (D / 2));
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    const uint4 w = crow[i];
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int e = 0; e < 8; ++e) kv[32 * i + 8 * k + e] = e2m1_value((ww[k] >> (4 * e)) & 0xFu);
  }
#pragma unroll
  for (int k = 0; k < D / 64; ++k) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(ksf + (((size_t)bhk * (Lkvp / kSqRows) + kt) * (D / 64) + k) *
                                                                    512 + (j & 31) * 16 + (j >> 5) * 4);
#pragma unroll
    for (int g = 0; g < 4; ++g) sg[4 * k + g] = e4m3_to_f32((w >> (8 * g)) & 0xFFu);
  }
  for (int i0 = 0; i0 < nqt; i0 += kDsStage) {
    const int ni = min(kDsStage, nqt - i0);
    __syncthreads();                                     // the previous stage is consumed
    for (int e = threadIdx.x; e < ni * D; e += kSqRows) qb[e] = qmean[((size_t)bh * nqt + i0) * D + e];
    __syncthreads();
    for (int i = 0; i < ni; ++i) {
      const float4* m4 = reinterpret_cast<const float4*>(qb + i * D);
      float acc = 0.f;
#pragma unroll
      for (int g = 0; g < D / 16; ++g) {
        float t = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 mq = m4[4 * g + c];
          t = fmaf(mq.x, kv[16 * g + 4 * c], t);
          t = fmaf(mq.y, kv[16 * g + 4 * c + 1], t);
          t = fmaf(mq.z, kv[16 * g + 4 * c + 2], t);
          t = fmaf(mq.w, kv[16 * g + 4 * c + 3], t);
        }
        acc = fmaf(t, sg[g], acc);
      }
      ds[((size_t)bh * nqt + i0 + i) * Lkvp + key] = acc;
    }
  }
}

template <int D>
cudaError_t launch_sq(const void* q, const Strides& sq, const Dims& dm, const sa_fp4_qkv& x, float* qmean, float* ds,
                      cudaStream_t s) {
  const int Lqp = padded_len(dm.Lq), Lkvp = padded_len(dm.Lkv);
  const long long ctas = (long long)dm.B * dm.H * (Lqp / kSqRows);
  sq_quant_kernel<D><<<(unsigned)ctas, kSqRows, 0, s>>>(static_cast<const __nv_bfloat16*>(q), sq, dm.H, dm.Lq, Lqp,
                                                        static_cast<uint8_t*>(x.q_codes),
                                                        static_cast<uint8_t*>(x.q_sf), qmean);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sq_ds_kernel<D><<<dim3((unsigned)(dm.B * dm.H), (unsigned)(Lkvp / kSqRows)), kSqRows, 0, s>>>(
      static_cast<const uint8_t*>(x.k_codes), static_cast<const uint8_t*>(x.k_sf), qmean, dm.H, dm.Hkv, Lqp, Lkvp,
      ds);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_smooth_q(const void* q, const Strides& sq, const Dims& dm, const sa_fp4_qkv& x, float* qmean,
                            float* ds, cudaStream_t s) {
  return dm.d == 64 ? launch_sq<64>(q, sq, dm, x, qmean, ds, s) : launch_sq<128>(q, sq, dm, x, qmean, ds, s);
}

}  // namespace sa
