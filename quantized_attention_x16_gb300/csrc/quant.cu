// quant.cu -- smooth-K mean and NVFP4 (e2m1, 1x16 groups, e4m3 scales)
// quantisation of Q, K' = K - mean_tokens(K) and V.
//
// Source: page "GPU kernel porting with AI agents", section "Sage Attention
// 3" (1x16 NVFP4 groups with FP8 e4m3 scales); page "kernel overview",
// SageAttention technique chain (smooth-K first).  Every floating-point step
// that decides a code is IEEE float32 (no fast-math in this unit): scale =
// e4m3_rne_sat(absmax / 6), code = e2m1_rne_sat(x / scale), so the outputs
// are bit-exact functions of the inputs.
//
// The launches are HBM-bandwidth bound (algorithmic bytes: read Q, V once and
// K twice -- the second K read is served by L2 -- and write codes and scales).

#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "sm100.cuh"

namespace sa {

namespace {

constexpr int kMeanChunk = 128;   // tokens per sequential partial sum

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Quantises one 1x16 group: returns the e4m3 scale byte, writes 2 words of codes.
__device__ __forceinline__ uint32_t quant_group16(const float* x, uint32_t* codes) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const float s = __fdiv_rn(amax, 6.0f);
  const uint32_t s8 = cvt_e4m3x2(s, 0.f) & 0xFFu;
  if (s8 == 0u) {
    codes[0] = 0u;
    codes[1] = 0u;
    return 0u;
  }
  const float sf = e4m3_to_f32(s8);
  // x / sf, correctly rounded, without a per-element division: with
  // y = RN(1/sf), q0 = RN(x*y) and the exact remainder r = x - q0*sf (one
  // FMA), q = RN(q0 + r*y) equals RN(x/sf) for every float32 x and every e4m3
  // scale (Markstein's correction step; checked exhaustively over all 2^23
  // significands against each of the eight e4m3 significands -- a scale's
  // exponent only shifts the result; zero inputs are handled by the sign copy).
  const float y = __frcp_rn(sf);
  float q[16];
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    float q0a, q0b, ra, rb;
    mul2(q0a, q0b, x[i], x[i + 1], y, y);
    fma2(ra, rb, -q0a, -q0b, sf, sf, x[i], x[i + 1]);
    fma2(q[i], q[i + 1], ra, rb, y, y, q0a, q0b);
    // the quotient carries the sign of x; the correction step would turn an
    // input of exactly -0.0 into +0 (+0 + -0 = +0), which would lose code 0x8
    q[i] = copysignf(q[i], x[i]);
    q[i + 1] = copysignf(q[i + 1], x[i + 1]);
  }
  codes[0] = cvt_e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
  codes[1] = cvt_e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]);
  return s8;
}

// ---------------------------------------------------------------------------
// Three launches, 256 threads per CTA:
//   1. kpart_kernel : smooth-K partial sums, one thread per channel pair of one
//                     128-token chunk, summed token by token (the documented
//                     order); reads K once.
//   2. kfinal_kernel: mean[c] = (partials summed in chunk order) / L.
//   3. quant_kernel : three kinds of CTA --
//        K CTAs first (K was just read by launch 1 and is still in L2):
//                one thread per 1x16 group of K - mean along d;
//        Q CTAs: one thread per 1x16 group along d (coalesced 32-byte reads,
//                8-byte code writes; the four scales of a 64-element chunk
//                are gathered with shuffles into one 32-bit store in the MMA
//                scale layout);
//        V CTAs: two 64-token chunks of one (b, kv head) staged in SMEM, one
//                thread per (chunk, channel) quantising four 16-token groups.

constexpr int kThreadsQ = 256;
constexpr int kVChunks = 2;                             // 64-token chunks per V CTA (L % 128 == 0)

struct QuantArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  uint8_t *qc, *qsf, *kc, *ksf, *vc, *vsf;
  float* part;      // [B*Hkv][L/128][D]
  float* kmean;     // [B*Hkv][D]
  int L, nbh_q, nbh_kv;
  long long nq_groups, nk_groups;
  int nblk_k, nblk_q, nblk_v;
};

// Writes the group's codes and gathers the four scale bytes of its 64-element
// chunk (four consecutive lanes) into one word in the MMA scale layout.
template <int D>
__device__ __forceinline__ void store_row_group(uint8_t* codes_base, uint8_t* sf_base, long long row, int gi,
                                                int L, uint32_t s8, const uint32_t* codes, bool valid) {
  uint32_t w = valid ? (s8 << (8 * (gi & 3))) : 0u;
  w |= __shfl_xor_sync(0xffffffffu, w, 1);
  w |= __shfl_xor_sync(0xffffffffu, w, 2);
  if (!valid) return;
  *reinterpret_cast<uint2*>(codes_base + row * (D / 2) + gi * 8) = make_uint2(codes[0], codes[1]);
  if ((gi & 3) == 0) {
    const long long bh = row / L;
    const int t = (int)(row % L), rb = t / 128, r = t % 128;
    const long long blk = (bh * (L / 128) + rb) * (D / 64) + gi / 4;
    *reinterpret_cast<uint32_t*>(sf_base + blk * 512 + (r % 32) * 16 + (r / 32) * 4) = w;
  }
}

// One group of Q (mean == nullptr) or of K - mean along d.
template <int D>
__device__ __forceinline__ void quant_rows_cta(const __nv_bfloat16* src_base, const float* mean, uint8_t* codes_base,
                                               uint8_t* sf_base, long long ngroups, int L, int blk) {
  const long long g = (long long)blk * kThreadsQ + threadIdx.x;
  const bool valid = g < ngroups;
  const long long row = valid ? g / (D / 16) : 0;
  const int gi = (int)(g % (D / 16));
  uint32_t codes[2] = {0u, 0u};
  uint32_t s8 = 0;
  if (valid) {
    float x[16];
    const uint4* src = reinterpret_cast<const uint4*>(src_base + row * D + gi * 16);
    bf16x8_to_f32(__ldg(src), x);
    bf16x8_to_f32(__ldg(src + 1), x + 8);
    if (mean != nullptr) {
      const float4* m4 = reinterpret_cast<const float4*>(mean + (row / L) * D + gi * 16);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 m = __ldg(m4 + i);
        x[4 * i + 0] = __fsub_rn(x[4 * i + 0], m.x);
        x[4 * i + 1] = __fsub_rn(x[4 * i + 1], m.y);
        x[4 * i + 2] = __fsub_rn(x[4 * i + 2], m.z);
        x[4 * i + 3] = __fsub_rn(x[4 * i + 3], m.w);
      }
    }
    s8 = quant_group16(x, codes);
  }
  store_row_group<D>(codes_base, sf_base, row, gi, L, s8, codes, valid);
}

template <int D>
__device__ __forceinline__ void quant_v_cta(const QuantArgs& a, int blk, __nv_bfloat16* tile) {
  constexpr int kChunks = kVChunks;
  const int cpb = a.L / 64;                             // chunks per head (even)
  const int first = blk * kChunks;                      // global chunk index
  const int bh = first / cpb, tc0 = first % cpb;
  const __nv_bfloat16* src = a.v + ((size_t)bh * a.L + (size_t)tc0 * 64) * D;
  constexpr int kVec = kChunks * 64 * D / 8;
#pragma unroll
  for (int i = threadIdx.x; i < kVec; i += kThreadsQ)
    reinterpret_cast<uint4*>(tile)[i] = __ldg(reinterpret_cast<const uint4*>(src) + i);
  __syncthreads();
  if (threadIdx.x >= kChunks * D) return;               // d = 64: half the CTA only loads
  const int ch = threadIdx.x / D, c = threadIdx.x % D;
  const int tc = tc0 + ch;
  uint32_t codes[8];
  uint32_t sfw = 0;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = __bfloat162float(tile[(ch * 64 + 16 * g + i) * D + c]);
    sfw |= quant_group16(x, codes + 2 * g) << (8 * g);
  }
  uint8_t* cdst = a.vc + ((size_t)bh * D + c) * (a.L / 2) + (size_t)tc * 32;
  reinterpret_cast<uint4*>(cdst)[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
  reinterpret_cast<uint4*>(cdst)[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
  uint8_t* sblk = a.vsf + ((size_t)bh * cpb + tc) * 512;
  *reinterpret_cast<uint32_t*>(sblk + (c % 32) * 16 + (c / 32) * 4) = sfw;
  if (D == 64) *reinterpret_cast<uint32_t*>(sblk + (c % 32) * 16 + (c / 32 + 2) * 4) = 0u;   // padding rows
}

// part[bh][chunk][c] = sum over the chunk's 128 tokens, token by token from 0.
template <int D>
__global__ void __launch_bounds__(kThreadsQ) kpart_kernel(const QuantArgs a) {
  constexpr int kPairs = D / 2;
  constexpr int kChunksPerCta = kThreadsQ / kPairs;
  const int nchunk = a.L / kMeanChunk;
  const int gchunk = blockIdx.x * kChunksPerCta + threadIdx.x / kPairs;     // over B*Hkv*nchunk
  if (gchunk >= a.nbh_kv * nchunk) return;
  const int bh = gchunk / nchunk, chunk = gchunk % nchunk;
  const int c = 2 * (threadIdx.x % kPairs);
  const uint32_t* src =
      reinterpret_cast<const uint32_t*>(a.k + ((size_t)bh * a.L + (size_t)chunk * kMeanChunk) * D + c);
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 1
  for (int t0 = 0; t0 < kMeanChunk; t0 += 32) {
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = __ldg(src + (size_t)(t0 + i) * (D / 2));
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      acc0 = __fadd_rn(acc0, __uint_as_float(w[i] << 16));
      acc1 = __fadd_rn(acc1, __uint_as_float(w[i] & 0xFFFF0000u));
    }
  }
  *reinterpret_cast<float2*>(a.part + ((size_t)bh * nchunk + chunk) * D + c) = make_float2(acc0, acc1);
}

// mean[bh][c] = (partials summed in chunk order) / L; one thread per (bh, c).
template <int D>
__global__ void __launch_bounds__(kThreadsQ) kfinal_kernel(const QuantArgs a) {
  const int i = blockIdx.x * kThreadsQ + threadIdx.x;
  if (i >= a.nbh_kv * D) return;
  const int bh = i / D, c = i % D;
  const int nchunk = a.L / kMeanChunk;
  const float* p = a.part + (size_t)bh * nchunk * D + c;
  float tot = 0.f;
#pragma unroll 1
  for (int c0 = 0; c0 < nchunk; c0 += 8) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = (c0 + j < nchunk) ? p[(size_t)(c0 + j) * D] : 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (c0 + j < nchunk) tot = __fadd_rn(tot, v[j]);
  }
  a.kmean[i] = __fdiv_rn(tot, (float)a.L);
}

template <int D>
__global__ void __launch_bounds__(kThreadsQ) quant_kernel(const QuantArgs a) {
  __shared__ __align__(16) __nv_bfloat16 tile[kVChunks * 64 * D];
  const int blk = blockIdx.x;
  if (blk < a.nblk_k) {
    quant_rows_cta<D>(a.k, a.kmean, a.kc, a.ksf, a.nk_groups, a.L, blk);
  } else if (blk < a.nblk_k + a.nblk_q) {
    quant_rows_cta<D>(a.q, nullptr, a.qc, a.qsf, a.nq_groups, a.L, blk - a.nblk_k);
  } else {
    quant_v_cta<D>(a, blk - a.nblk_k - a.nblk_q, tile);
  }
}

template <int D>
cudaError_t launch_quantize_impl(const void* q, const void* k, const void* v, const Dims& dm,
                                 const sa_fp4_qkv& out, float* partials, cudaStream_t s) {
  QuantArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.qc = static_cast<uint8_t*>(out.q_codes);
  a.qsf = static_cast<uint8_t*>(out.q_sf);
  a.kc = static_cast<uint8_t*>(out.k_codes);
  a.ksf = static_cast<uint8_t*>(out.k_sf);
  a.vc = static_cast<uint8_t*>(out.v_codes);
  a.vsf = static_cast<uint8_t*>(out.v_sf);
  a.part = partials;
  a.kmean = out.k_mean;
  a.L = dm.L;
  a.nbh_q = dm.B * dm.H;
  a.nbh_kv = dm.B * dm.Hkv;
  a.nq_groups = (long long)a.nbh_q * dm.L * (D / 16);
  a.nk_groups = (long long)a.nbh_kv * dm.L * (D / 16);
  a.nblk_q = (int)((a.nq_groups + kThreadsQ - 1) / kThreadsQ);
  a.nblk_k = (int)((a.nk_groups + kThreadsQ - 1) / kThreadsQ);
  a.nblk_v = a.nbh_kv * (dm.L / 64) / kVChunks;
  const int kchunks = a.nbh_kv * (dm.L / kMeanChunk);
  const int kcpb = kThreadsQ / (D / 2);
  kpart_kernel<D><<<(kchunks + kcpb - 1) / kcpb, kThreadsQ, 0, s>>>(a);
  kfinal_kernel<D><<<(a.nbh_kv * D + kThreadsQ - 1) / kThreadsQ, kThreadsQ, 0, s>>>(a);
  quant_kernel<D><<<a.nblk_k + a.nblk_q + a.nblk_v, kThreadsQ, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const void* q, const void* k, const void* v, const Dims& dm, const sa_fp4_qkv& out,
                            cudaStream_t s) {
  float* part = static_cast<float*>(out.workspace);
  return dm.d == 64 ? launch_quantize_impl<64>(q, k, v, dm, out, part, s)
                    : launch_quantize_impl<128>(q, k, v, dm, out, part, s);
}

// ---------------------------------------------------------------------------
// Allocation-free variant (sa_quantize_static_scratch).  The K-mean partial
// sums go to a fixed array compiled into this library instead of the
// caller's workspace.  Each device that loads the library holds the array
// (kStaticScratchFloats floats, 4 MiB) until the process exits.  Its device
// address is looked up once per device, on the first call made with that
// device current; host code never passes the array's own name to a kernel.
namespace {

static __device__ __align__(256) float g_quant_scratch[kStaticScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
float* g_scratch_addr[kMaxDevices] = {};

cudaError_t static_scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_quant_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_quantize_static_scratch(const void* q, const void* k, const void* v, const Dims& dm,
                                           const sa_fp4_qkv& out, cudaStream_t s) {
  const size_t need = (size_t)dm.B * dm.Hkv * (dm.L / kMeanChunk) * dm.d;
  if (need > kStaticScratchFloats) return cudaErrorInvalidValue;
  float* part = nullptr;
  cudaError_t e = static_scratch_address(&part);
  if (e != cudaSuccess) return e;
  // Every partial sum read is written first by the same call (the K CTAs of
  // the first launch), so earlier contents of the array never reach the
  // outputs and nothing needs clearing.
  return dm.d == 64 ? launch_quantize_impl<64>(q, k, v, dm, out, part, s)
                    : launch_quantize_impl<128>(q, k, v, dm, out, part, s);
}

}  // namespace sa
