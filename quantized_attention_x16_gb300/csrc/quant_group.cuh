// quant_group.cuh -- the 1x16 NVFP4 group arithmetic of the quantiser, shared
// by sa_quantize (quant.cu) and the attention kernel's in-kernel quantisation
// of Q (attn_nvfp4.cu), so that both produce the same bytes.
//
// Source: page "GPU kernel porting with AI agents", section "Sage Attention
// 3" (1x16 NVFP4 groups with FP8 e4m3 scales).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "sm100.cuh"

namespace sa {
namespace qg {

// ---------------------------------------------------------------------------
// Group arithmetic.
//
// Every 1x16 group: s8 = e4m3_rne_sat(RN(max|x| / 6)), code_i =
// e2m1_rne_sat(RN(x_i / s)) with s = decode(s8), all codes +0 when s8 == 0.
// Neither quotient uses a divide instruction:
//  * RN(max|x| / 6): Markstein's correction step.  With y = RN(1/6), q0 =
//    RN(a*y) and the exact remainder r = a - q0*6 from one FMA, RN(q0 + r*y)
//    = RN(a/6).
//  * code_i from q = RN(x*yh + RN(x*yl)) (one product and one FMA), where
//    yh = RD(1/s) and yl = RN((1 - s*yh) * yh): the residual 1 - s*yh is
//    exact and >= 0, and yh + yl is 1/s to 2^-46, so q is x/s plus at most
//    2^-45 |x/s| before its one rounding.  The code of q can differ from the
//    code of RN(x/s) only where that rounding is decided differently next to
//    an e2m1 boundary T, i.e. for x/s within 2^-45 of T or of a float32
//    midpoint T +- ulp/2 beside it.  x/s = T exactly gives q = T.  A midpoint
//    T +- ulp/2 has a 25-bit odd significand, so s (4 significant bits) times
//    it is no float32 and x/s stays at least 2^-30 (relative) away from it.
//    So the codes are those of the correctly rounded quotient, for bf16 x (Q,
//    V) and float32 x (K' = K - mean) alike; this is checked on the host for
//    every bf16 x and every e4m3 scale, and for every float32 significand
//    near each boundary.  yl >= 0 keeps the sign of a zero x (+0 * yh + +0 =
//    +0, -0 * yh + -0 = -0).  (yh, yl) is looked up by the scale byte in a
//    128-entry shared-memory table.

// max(|a|, |b|) per bf16 half (the result's sign bits are not used).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Per-half maxima of |x| over n words -> (max of the low halves, max of the high halves) as floats.
template <int N>
__device__ __forceinline__ void absmax_halves(const uint32_t* w, float& lo, float& hi) {
  uint32_t m[N];
#pragma unroll
  for (int i = 0; i < N; ++i) m[i] = w[i];
#pragma unroll
  for (int s = 1; s < N; s *= 2)
#pragma unroll
    for (int i = 0; i + s < N; i += 2 * s) m[i] = absmax_bf16x2(m[i], m[i + s]);
  lo = __uint_as_float((m[0] & 0x7FFFu) << 16);
  hi = __uint_as_float(m[0] & 0x7FFF0000u);
}

// RN(a / 6) for a >= 0 (Markstein step, exact).
__device__ __forceinline__ float div6_rn(float a) {
  const float y6 = __uint_as_float(0x3E2AAAABu);        // RN(1/6)
  const float q6 = a * y6;
  return fmaf(fmaf(-q6, 6.0f, a), y6, q6);
}

// The e4m3 scale bytes of two groups from their max |x| (low byte: a0).
__device__ __forceinline__ uint32_t scale_pair(float a0, float a1) {
  return cvt_e4m3x2(div6_rn(a0), div6_rn(a1));
}

// Codes of 16 values x[0..15] for scale byte s8: two words.  Tab: the
// reciprocal table, indexed by the scale byte (a pointer, or SharedRtab).
template <class Tab>
__device__ __forceinline__ void codes_group(const float* x, uint32_t s8, const Tab& rtab, uint32_t* codes) {
  const float2 r = rtab[s8];
  float q[16];
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    float t0, t1;
    mul2(t0, t1, x[i], x[i + 1], r.y, r.y);
    fma2(q[i], q[i + 1], x[i], x[i + 1], r.x, r.x, t0, t1);
  }
  const bool z = s8 == 0u;
  codes[0] = z ? 0u : cvt_e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
  codes[1] = z ? 0u : cvt_e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]);
}

// bf16 pair word -> two floats (channel/token 2i in the low half).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The two-term reciprocal (yh, yl) of e4m3 scale byte s8 for codes_group
// (0 and the NaN code: unused).
__device__ __forceinline__ float2 rtab_entry(uint32_t s8) {
  float2 r = make_float2(0.f, 0.f);
  if (s8 != 0u && s8 != 0x7Fu) {
    const float sf = e4m3_to_f32(s8);
    const float yh = __frcp_rd(sf);
    r = make_float2(yh, __fmul_rn(fmaf(-sf, yh, 1.0f), yh));
  }
  return r;
}

// The reciprocal table at a shared-memory address: lookups are shared-window
// loads even where the compiler cannot see which window a pointer is in.
struct SharedRtab {
  uint32_t base;
  __device__ __forceinline__ float2 operator[](uint32_t s8) const {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(base + 8u * s8));
    return v;
  }
};

// Row rr (0..127) of a 64-channel x 128-token bf16 box as TMA leaves it with
// the 128B swizzle (16-byte chunk i of row rr at chunk i ^ (rr & 7)): 32
// words, channel pair i in word i (channel 2i in the low half).
__device__ __forceinline__ void load_box_row(const uint8_t* box, int rr, uint32_t (&w)[32]) {
  const uint8_t* src = box + rr * 128;
  const uint32_t x7 = (uint32_t)(rr & 7) << 4;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + (((uint32_t)i << 4) ^ x7));
    w[4 * i] = v.x;
    w[4 * i + 1] = v.y;
    w[4 * i + 2] = v.z;
    w[4 * i + 3] = v.w;
  }
}

// One quad of Q (64 channels of one token, four 1x16 groups): the codes (8
// words, channel 8j + e in nibble e of word j) and the scale word (group g in
// byte g).
template <class Tab>
__device__ __forceinline__ void quant_q_quad(const uint32_t (&w)[32], const Tab& rtab, uint32_t (&codes)[8],
                                             uint32_t& sfw) {
  float am[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float lo, hi;
    absmax_halves<8>(w + 8 * g, lo, hi);
    am[g] = fmaxf(lo, hi);
  }
  sfw = scale_pair(am[0], am[1]) | (scale_pair(am[2], am[3]) << 16);
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float x[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = bf16_lo(w[8 * g + i]);
      x[2 * i + 1] = bf16_hi(w[8 * g + i]);
    }
    codes_group(x, (sfw >> (8 * g)) & 0xFFu, rtab, codes + 2 * g);
  }
}

}  // namespace qg
}  // namespace sa
