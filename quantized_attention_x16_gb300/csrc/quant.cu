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
// All kernels are HBM-bandwidth bound: 16-byte vector loads, one thread per
// 64-element unit (four groups) for Q/K, an SMEM-staged transpose for V.

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
  float q[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) q[i] = __fdiv_rn(x[i], sf);
  codes[0] = cvt_e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
  codes[1] = cvt_e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]);
  return s8;
}

// part[bh][chunk][c] = sum over the chunk's 128 tokens, in token order.
// One thread owns 8 channels of one chunk.
__global__ void __launch_bounds__(128) kmean_partial_kernel(const __nv_bfloat16* __restrict__ k,
                                                            float* __restrict__ part, int L, int d, int nchunk) {
  const int tpc = d / 8;
  const int cpb = blockDim.x / tpc;
  const int bh = blockIdx.y;
  const int chunk = blockIdx.x * cpb + threadIdx.x / tpc;
  const int c0 = (threadIdx.x % tpc) * 8;
  if (chunk >= nchunk) return;
  const __nv_bfloat16* src = k + ((size_t)bh * L + (size_t)chunk * kMeanChunk) * d + c0;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll 8
  for (int t = 0; t < kMeanChunk; ++t) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(src + (size_t)t * d));
    float f[8];
    bf16x8_to_f32(u, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], f[i]);
  }
  float4* dst = reinterpret_cast<float4*>(part + ((size_t)bh * nchunk + chunk) * d + c0);
  dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// mu[bh][c] = (sum of the chunk partials in chunk order) / L.
__global__ void __launch_bounds__(128) kmean_final_kernel(const float* __restrict__ part, float* __restrict__ mu,
                                                          int nbh, int nchunk, int d, int L) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nbh * d) return;
  const int bh = i / d, c = i % d;
  const float* p = part + (size_t)bh * nchunk * d + c;
  float tot = 0.f;
  for (int ch = 0; ch < nchunk; ++ch) tot = __fadd_rn(tot, p[(size_t)ch * d]);
  mu[i] = __fdiv_rn(tot, (float)L);
}

// One thread = one 64-element unit (4 groups along d) of one Q or K row.
__global__ void __launch_bounds__(256) quant_qk_kernel(const __nv_bfloat16* __restrict__ q,
                                                       const __nv_bfloat16* __restrict__ k,
                                                       const float* __restrict__ mu, uint8_t* __restrict__ qc,
                                                       uint8_t* __restrict__ qsf, uint8_t* __restrict__ kc,
                                                       uint8_t* __restrict__ ksf, int L, int d, long long nq,
                                                       long long nk) {
  const int nkc = d / 64;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < nq + nk; u += stride) {
    const bool is_k = u >= nq;
    const long long unit = is_k ? u - nq : u;
    const long long row = unit / nkc;            // (b*heads + h) * L + t
    const int kcol = (int)(unit % nkc);
    const __nv_bfloat16* src = (is_k ? k : q) + row * d + kcol * 64;
    const long long bh = row / L;
    const int t = (int)(row % L);
    float x[64];
#pragma unroll
    for (int i = 0; i < 8; ++i) bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(src) + i), x + 8 * i);
    if (is_k) {
      const float4* m4 = reinterpret_cast<const float4*>(mu + bh * d + kcol * 64);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 m = __ldg(m4 + i);
        x[4 * i + 0] = __fsub_rn(x[4 * i + 0], m.x);
        x[4 * i + 1] = __fsub_rn(x[4 * i + 1], m.y);
        x[4 * i + 2] = __fsub_rn(x[4 * i + 2], m.z);
        x[4 * i + 3] = __fsub_rn(x[4 * i + 3], m.w);
      }
    }
    uint32_t codes[8];
    uint32_t sfw = 0;
#pragma unroll
    for (int g = 0; g < 4; ++g) sfw |= quant_group16(x + 16 * g, codes + 2 * g) << (8 * g);
    uint8_t* cdst = (is_k ? kc : qc) + row * (d / 2) + kcol * 32;
    reinterpret_cast<uint4*>(cdst)[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
    reinterpret_cast<uint4*>(cdst)[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
    const int rb = t / 128, r = t % 128;
    const long long blk = (bh * (L / 128) + rb) * nkc + kcol;
    uint8_t* sdst = (is_k ? ksf : qsf) + blk * 512 + (r % 32) * 16 + (r / 32) * 4;
    *reinterpret_cast<uint32_t*>(sdst) = sfw;
  }
}

// One CTA = one (b, kv head) x 64-token chunk; one thread per channel.  The
// 64 x d bf16 tile is staged in SMEM, then each thread quantises its channel's
// four 16-token groups and writes the transposed codes.
__global__ void __launch_bounds__(128) quant_v_kernel(const __nv_bfloat16* __restrict__ v, uint8_t* __restrict__ vc,
                                                      uint8_t* __restrict__ vsf, int L, int d) {
  __shared__ __align__(16) __nv_bfloat16 tile[64 * 128];
  const int bh = blockIdx.y, tc = blockIdx.x;
  const __nv_bfloat16* src = v + ((size_t)bh * L + (size_t)tc * 64) * d;
  const int nvec = 64 * d / 8;
  for (int i = threadIdx.x; i < nvec; i += blockDim.x)
    reinterpret_cast<uint4*>(tile)[i] = __ldg(reinterpret_cast<const uint4*>(src) + i);
  __syncthreads();
  const int c = threadIdx.x;
  uint32_t codes[8];
  uint32_t sfw = 0;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = __bfloat162float(tile[(16 * g + i) * d + c]);
    sfw |= quant_group16(x, codes + 2 * g) << (8 * g);
  }
  uint8_t* cdst = vc + ((size_t)bh * d + c) * (L / 2) + (size_t)tc * 32;
  reinterpret_cast<uint4*>(cdst)[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
  reinterpret_cast<uint4*>(cdst)[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
  uint8_t* sblk = vsf + ((size_t)bh * (L / 64) + tc) * 512;
  *reinterpret_cast<uint32_t*>(sblk + (c % 32) * 16 + (c / 32) * 4) = sfw;
  if (d == 64) *reinterpret_cast<uint32_t*>(sblk + (c % 32) * 16 + (c / 32 + 2) * 4) = 0u;   // padding rows
}

}  // namespace

cudaError_t launch_quantize(const void* q, const void* k, const void* v, const Dims& dm, const sa_fp4_qkv& out,
                            cudaStream_t s) {
  const int nchunk = dm.L / kMeanChunk;
  const int nbh = dm.B * dm.Hkv;
  const int cpb = 128 / (dm.d / 8);
  float* part = static_cast<float*>(out.workspace);
  kmean_partial_kernel<<<dim3((nchunk + cpb - 1) / cpb, nbh), 128, 0, s>>>(
      static_cast<const __nv_bfloat16*>(k), part, dm.L, dm.d, nchunk);
  kmean_final_kernel<<<(nbh * dm.d + 127) / 128, 128, 0, s>>>(part, out.k_mean, nbh, nchunk, dm.d, dm.L);
  const long long nq = (long long)dm.B * dm.H * dm.L * (dm.d / 64);
  const long long nk = (long long)nbh * dm.L * (dm.d / 64);
  const long long blocks = (nq + nk + 255) / 256;
  quant_qk_kernel<<<(unsigned)(blocks < 65535 * 16 ? blocks : 65535 * 16), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), out.k_mean,
      static_cast<uint8_t*>(out.q_codes), static_cast<uint8_t*>(out.q_sf), static_cast<uint8_t*>(out.k_codes),
      static_cast<uint8_t*>(out.k_sf), dm.L, dm.d, nq, nk);
  quant_v_kernel<<<dim3(dm.L / 64, nbh), dm.d, 0, s>>>(static_cast<const __nv_bfloat16*>(v),
                                                       static_cast<uint8_t*>(out.v_codes),
                                                       static_cast<uint8_t*>(out.v_sf), dm.L, dm.d);
  return cudaGetLastError();
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
  // Every partial sum read below is written first by kmean_partial_kernel in
  // the same call, so earlier contents of the array never reach the outputs
  // and nothing needs clearing.
  const int nchunk = dm.L / kMeanChunk;
  const int nbh = dm.B * dm.Hkv;
  const int cpb = 128 / (dm.d / 8);
  kmean_partial_kernel<<<dim3((nchunk + cpb - 1) / cpb, nbh), 128, 0, s>>>(
      static_cast<const __nv_bfloat16*>(k), part, dm.L, dm.d, nchunk);
  kmean_final_kernel<<<(nbh * dm.d + 127) / 128, 128, 0, s>>>(part, out.k_mean, nbh, nchunk, dm.d, dm.L);
  const long long nq = (long long)dm.B * dm.H * dm.L * (dm.d / 64);
  const long long nk = (long long)nbh * dm.L * (dm.d / 64);
  const long long blocks = (nq + nk + 255) / 256;
  quant_qk_kernel<<<(unsigned)(blocks < 65535 * 16 ? blocks : 65535 * 16), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), out.k_mean,
      static_cast<uint8_t*>(out.q_codes), static_cast<uint8_t*>(out.q_sf), static_cast<uint8_t*>(out.k_codes),
      static_cast<uint8_t*>(out.k_sf), dm.L, dm.d, nq, nk);
  quant_v_kernel<<<dim3(dm.L / 64, nbh), dm.d, 0, s>>>(static_cast<const __nv_bfloat16*>(v),
                                                       static_cast<uint8_t*>(out.v_codes),
                                                       static_cast<uint8_t*>(out.v_sf), dm.L, dm.d);
  return cudaGetLastError();
}

}  // namespace sa
