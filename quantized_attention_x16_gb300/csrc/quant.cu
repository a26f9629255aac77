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
//
// Both divisions are done as correctly rounded quotients without a divide
// instruction (Markstein's correction step: with y = RN(1/b), q0 = RN(x*y)
// and the exact remainder r = x - q0*b from one FMA, RN(q0 + r*y) = RN(x/b)).
// This was checked exhaustively over all 2^23 significands against each
// divisor significand 9/8 .. 15/8, which covers b = 6 (= 12/8 * 4) and every
// e4m3 scale; exponents only shift the result.
//  * scale: s = RN(max|x| / 6) with y = RN(1/6);
//  * codes: the quotient is formed for the divisor -s, i.e. qn = RN(x / -s) =
//    -RN(x / s) (rounding is symmetric), and the code sign bits are flipped
//    afterwards (e2m1 is sign-magnitude).  This keeps the sign of a zero
//    input: x = -0.0 gives qn = +0 and code 0x8, x = +0.0 gives code 0x0.
__device__ __forceinline__ uint32_t quant_group16(const float* x, uint32_t* codes) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const float y6 = __uint_as_float(0x3E2AAAABu);        // RN(1/6)
  const float q6 = amax * y6;
  const float s = fmaf(fmaf(-q6, 6.0f, amax), y6, q6);
  const uint32_t s8 = cvt_e4m3x2(s, 0.f) & 0xFFu;
  if (s8 == 0u) {
    codes[0] = 0u;
    codes[1] = 0u;
    return 0u;
  }
  float sf, unused;
  e4m3x2_to_f32(s8, sf, unused);
  const float ny = -__frcp_rn(sf);                      // RN(1 / -sf)
  float q[16];
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    float n0, n1, t0, t1;
    mul2(n0, n1, x[i], x[i + 1], ny, ny);               // q0' = RN(x * y')
    fma2(t0, t1, n0, n1, sf, sf, x[i], x[i + 1]);       // r' = x - q0' * (-sf), exact
    fma2(q[i], q[i + 1], t0, t1, ny, ny, n0, n1);       // RN(q0' + r' * y')
  }
  codes[0] = cvt_e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]) ^ 0x88888888u;
  codes[1] = cvt_e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]) ^ 0x88888888u;
  return s8;
}

// ---------------------------------------------------------------------------
// Two launches, 256 threads per CTA.
//   1. quant_vk_kernel -- two kinds of CTA:
//        V CTAs:     one thread per (channel pair, 32 tokens): 32 4-byte loads
//                    (each warp load is one 128-byte row segment), two
//                    16-token groups per channel, codes stored transposed;
//        Kpart CTAs: smooth-K partial sums, one thread per channel pair of one
//                    128-token chunk, summed token by token from 0 (the
//                    documented order).  They run last, so K is still in L2
//                    for launch 2.
//   2. quant_kq_kernel -- two kinds of CTA:
//        K CTAs:     one per (b, kv head, 512-token block).  The head's
//                    partial sums are staged in shared memory (coalesced, all
//                    loads in flight) and summed in chunk order, then / L: the
//                    same float operations in the same order in every CTA, so
//                    mu is bit-exact and identical everywhere; the head's first
//                    CTA also writes mu.  K - mu is then quantised quad by
//                    quad, reading K from L2.
//        Q CTAs:     each thread quantises kQuadsPerThread "quads" (64
//                    consecutive channels of one row = four 1x16 groups = one
//                    32-bit word of scale bytes), the next quad's eight
//                    16-byte loads in flight while the current one is
//                    computed.  Q streams from HBM while the K CTAs wait on L2.

constexpr int kThreadsQ = 256;
constexpr int kQuadsPerThread = 1;                      // Q quads per thread
constexpr int kKTokens = 512;                           // tokens per K CTA
constexpr int kMeanSlice = 32;                          // 128-token chunks staged per pass

struct QuantArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  uint8_t *qc, *qsf, *kc, *ksf, *vc, *vsf;
  float* part;      // [B*Hkv][L/128][D]
  float* kmean;     // [B*Hkv][D]
  int L, nbh_q, nbh_kv;
  long long nq_quads;
  int nblk_q, nblk_v, nblk_kpart, nblk_k_per_head, nblk_k;
};

// Loads the 64 bf16 values of one quad (eight 16-byte loads, all in flight).
__device__ __forceinline__ void load_quad(const __nv_bfloat16* src, uint4 (&w)[8]) {
  const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = __ldg(p + i);
}

// Quantises one quad (minus the 64 means at `mean`, when given) and stores its
// 32 bytes of codes and its scale word.  `row` is the global row (b*H + h)*L + t,
// `quad` the 64-channel block within the row.
template <int D>
__device__ __forceinline__ void quant_quad(const uint4 (&w)[8], const float* mean, uint8_t* codes_base,
                                           uint8_t* sf_base, long long row, int quad, int L) {
  uint32_t codes[8];
  uint32_t sfw = 0;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float x[16];
    bf16x8_to_f32(w[2 * g], x);
    bf16x8_to_f32(w[2 * g + 1], x + 8);
    if (mean != nullptr) {
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = __fsub_rn(x[i], mean[16 * g + i]);
    }
    sfw |= quant_group16(x, codes + 2 * g) << (8 * g);
  }
  uint4* cdst = reinterpret_cast<uint4*>(codes_base + row * (D / 2) + quad * 32);
  cdst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
  cdst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
  const long long bh = row / L;
  const int t = (int)(row % L), rb = t / 128, r = t % 128;
  const long long blk = (bh * (L / 128) + rb) * (D / 64) + quad;
  *reinterpret_cast<uint32_t*>(sf_base + blk * 512 + (r % 32) * 16 + (r / 32) * 4) = sfw;
}

template <int D>
__device__ __forceinline__ void quant_q_cta(const QuantArgs& a, int blk) {
  // quads blk*256*kQuadsPerThread + i*256 + tid, i = 0 .. kQuadsPerThread-1
  long long gq = (long long)blk * kThreadsQ * kQuadsPerThread + threadIdx.x;
  uint4 w[8];
  if (gq < a.nq_quads) load_quad(a.q + (gq / (D / 64)) * D + (gq % (D / 64)) * 64, w);
#pragma unroll 1
  for (int i = 0; i < kQuadsPerThread && gq < a.nq_quads; ++i, gq += kThreadsQ) {
    const long long row = gq / (D / 64);
    const int quad = (int)(gq % (D / 64));
    uint4 cur[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) cur[k] = w[k];
    const long long nx = gq + kThreadsQ;
    if (i + 1 < kQuadsPerThread && nx < a.nq_quads) load_quad(a.q + (nx / (D / 64)) * D + (nx % (D / 64)) * 64, w);
    quant_quad<D>(cur, nullptr, a.qc, a.qsf, row, quad, a.L);
  }
}

// One thread per (channel pair, 32 tokens = two 16-token groups).  Items are
// ordered channel pair fastest, so a warp covers 64 consecutive channels of
// the same 32 tokens and each of its 32 loads reads one 128-byte segment of a
// V row.  A channel's two scale bytes are one half of its 64-token scale word.
template <int D>
__device__ __forceinline__ void quant_v_cta(const QuantArgs& a, int blk) {
  constexpr int kPairs = D / 2;
  const long long item = (long long)blk * kThreadsQ + threadIdx.x;
  const int npb = a.L / 32;                             // 32-token pieces per head
  if (item >= (long long)a.nbh_kv * npb * kPairs) return;
  const int c = 2 * (int)(item % kPairs);
  const long long piece = item / kPairs;                // over B*Hkv*npb
  const long long bh = piece / npb;
  const int tp = (int)(piece % npb);
  const uint32_t* src = reinterpret_cast<const uint32_t*>(a.v + ((size_t)bh * a.L + (size_t)tp * 32) * D + c);
  uint32_t w[32];
#pragma unroll
  for (int t = 0; t < 32; ++t) w[t] = __ldg(src + (size_t)t * (D / 2));
  uint8_t* sblk = a.vsf + ((size_t)bh * (a.L / 64) + tp / 2) * 512 + (tp % 2) * 2;
#pragma unroll
  for (int h = 0; h < 2; ++h) {                         // channel c + h
    uint32_t codes[4];
    uint32_t sfw = 0;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        x[i] = __uint_as_float(h ? (w[16 * g + i] & 0xFFFF0000u) : (w[16 * g + i] << 16));
      sfw |= quant_group16(x, codes + 2 * g) << (8 * g);
    }
    const int ch = c + h;
    *reinterpret_cast<uint4*>(a.vc + ((size_t)bh * D + ch) * (a.L / 2) + (size_t)tp * 16) =
        make_uint4(codes[0], codes[1], codes[2], codes[3]);
    *reinterpret_cast<uint16_t*>(sblk + (ch % 32) * 16 + (ch / 32) * 4) = (uint16_t)sfw;
    if (D == 64) *reinterpret_cast<uint16_t*>(sblk + (ch % 32) * 16 + (ch / 32 + 2) * 4) = 0;   // padding rows
  }
}

// part[bh][chunk][c] = sum over the chunk's 128 tokens, token by token from 0.
template <int D>
__device__ __forceinline__ void kpart_cta(const QuantArgs& a, int blk) {
  constexpr int kPairs = D / 2;
  constexpr int kChunksPerCta = kThreadsQ / kPairs;
  const int nchunk = a.L / kMeanChunk;
  const int gchunk = blk * kChunksPerCta + threadIdx.x / kPairs;     // over B*Hkv*nchunk
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

template <int D>
__global__ void __launch_bounds__(kThreadsQ, 3) quant_vk_kernel(const QuantArgs a) {
  const int blk = blockIdx.x;
  if (blk < a.nblk_q)
    quant_q_cta<D>(a, blk);
  else if (blk < a.nblk_q + a.nblk_v)
    quant_v_cta<D>(a, blk - a.nblk_q);
  else
    kpart_cta<D>(a, blk - a.nblk_q - a.nblk_v);
}

// mean[c] = (partials summed in chunk order) / L for one (b, kv head), into
// shared memory; written to k_mean as well when `publish`.
template <int D>
__device__ __forceinline__ void head_mean(const QuantArgs& a, int bh, float* mean, float* stage, bool publish) {
  const int nchunk = a.L / kMeanChunk;
  const float* part = a.part + (size_t)bh * nchunk * D;
  float tot = 0.f;
  for (int c0 = 0; c0 < nchunk; c0 += kMeanSlice) {
    const int nc = min(kMeanSlice, nchunk - c0);
    __syncthreads();                                    // previous slice consumed
    // all of this thread's loads are issued before the first store
    constexpr int kPer = kMeanSlice * D / kThreadsQ;
    float v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = threadIdx.x + k * kThreadsQ;
      v[k] = i < nc * D ? __ldcg(part + (size_t)c0 * D + i) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) stage[threadIdx.x + k * kThreadsQ] = v[k];
    __syncthreads();
    if (threadIdx.x < D)
      for (int j = 0; j < nc; ++j) tot = __fadd_rn(tot, stage[j * D + threadIdx.x]);
  }
  if (threadIdx.x < D) {
    const float mu = __fdiv_rn(tot, (float)a.L);
    mean[threadIdx.x] = mu;
    if (publish) a.kmean[(size_t)bh * D + threadIdx.x] = mu;
  }
  __syncthreads();
}

template <int D>
__device__ __forceinline__ void quant_k_cta(const QuantArgs& a, int blk, float* mean, float* stage) {
  constexpr int kQuadsPerRow = D / 64;
  const int bh = blk / a.nblk_k_per_head;
  const int t0 = (blk % a.nblk_k_per_head) * kKTokens;
  const int nquads = min(kKTokens, a.L - t0) * kQuadsPerRow;
  const __nv_bfloat16* kbase = a.k + ((size_t)bh * a.L + t0) * D;
  // the first quad's loads are in flight while the mean is formed
  int qi = threadIdx.x;
  uint4 w[8];
  if (qi < nquads) load_quad(kbase + (size_t)(qi / kQuadsPerRow) * D + (qi % kQuadsPerRow) * 64, w);
  head_mean<D>(a, bh, mean, stage, t0 == 0);
  for (; qi < nquads; qi += kThreadsQ) {
    const int quad = qi % kQuadsPerRow;
    const long long row = (long long)bh * a.L + t0 + qi / kQuadsPerRow;
    uint4 cur[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) cur[k] = w[k];
    const int nx = qi + kThreadsQ;
    if (nx < nquads) load_quad(kbase + (size_t)(nx / kQuadsPerRow) * D + (nx % kQuadsPerRow) * 64, w);
    quant_quad<D>(cur, mean + quad * 64, a.kc, a.ksf, row, quad, a.L);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreadsQ) quant_kq_kernel(const QuantArgs a) {
  __shared__ __align__(16) float mean[D];
  __shared__ __align__(16) float stage[kMeanSlice * D];
  quant_k_cta<D>(a, (int)blockIdx.x, mean, stage);
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
  a.nq_quads = (long long)a.nbh_q * dm.L * (D / 64);
  a.nblk_q = (int)((a.nq_quads + kThreadsQ * kQuadsPerThread - 1) / (kThreadsQ * kQuadsPerThread));
  a.nblk_v = (int)(((long long)a.nbh_kv * (dm.L / 32) * (D / 2) + kThreadsQ - 1) / kThreadsQ);
  const int kchunks = a.nbh_kv * (dm.L / kMeanChunk);
  const int kcpb = kThreadsQ / (D / 2);
  a.nblk_kpart = (kchunks + kcpb - 1) / kcpb;
  a.nblk_k_per_head = (dm.L + kKTokens - 1) / kKTokens;
  a.nblk_k = a.nbh_kv * a.nblk_k_per_head;
  quant_vk_kernel<D><<<a.nblk_q + a.nblk_v + a.nblk_kpart, kThreadsQ, 0, s>>>(a);
  quant_kq_kernel<D><<<a.nblk_k, kThreadsQ, 0, s>>>(a);
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
  // Every partial sum read is written first by the same call (the partial-sum
  // CTAs of its first launch), so earlier contents of the array never reach
  // the outputs and nothing needs clearing.
  return dm.d == 64 ? launch_quantize_impl<64>(q, k, v, dm, out, part, s)
                    : launch_quantize_impl<128>(q, k, v, dm, out, part, s);
}

}  // namespace sa
