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
//   1. quant_v_mean_kernel -- clusters of kMeanCluster CTAs, of two kinds:
//        mean clusters (first in the grid, so that the latency-bound sums
//                    start at once and run beside the bandwidth-bound V CTAs):
//                    one per (b, kv head).  CTA r sums its share of the
//                    head's 128-token chunks, one thread per channel pair and
//                    chunk, token by token from 0 (the documented order), into
//                    the scratch buffer.  After a cluster barrier
//                    (release/acquire at cluster scope) CTA 0 adds the chunk
//                    sums in chunk order and divides by L (bit-exact mu), and
//                    writes mu;
//        V clusters: eight independent CTAs, one thread per channel pair and
//                    32 tokens: 32 4-byte loads (each warp load is one 128-byte
//                    row segment), two 16-token groups per channel, codes
//                    stored transposed.
//   2. quant_qk_kernel -- persistent CTAs over tiles of 256 "quads" (a quad =
//        64 consecutive channels of one row = four 1x16 groups = one 32-bit
//        word of scale bytes) of one head: one round of Q tiles (one per CTA),
//        then the K tiles, then the other Q tiles.  It is a programmatic
//        dependent launch: its CTAs start while launch 1 drains and quantise
//        Q, which launch 1 does not touch; before its first K tile each CTA
//        waits for launch 1 to complete (mu), and K then comes from L2, where
//        launch 1 has just read it.  Tiles arrive by TMA in
//        128B-swizzled shared memory (boxes of 64 channels x 128 tokens of one
//        head; tokens past L arrive as zeros) through a two-stage ring; each
//        thread reads its quad with conflict-free 16-byte loads, subtracts mu
//        for K (64 means through L1), and stores 32 bytes of codes and the
//        scale word in the MMA scale layout.
// Every layout holds Lp = L rounded up to 128 tokens per head; the tokens
// past L are written as zero codes with zero scales (Q and K rows, V token
// groups), and a V group that straddles L is quantised with zeros for its
// missing tokens.

constexpr int kThreadsQ = 256;
constexpr int kMeanCluster = 8;                          // CTAs per head in the mean clusters

template <int D>
struct TileQK {
  static constexpr int kRows = kThreadsQ / (D / 64);     // rows per tile: 128 (d = 128), 256 (d = 64)
  static constexpr int kBoxes = 2;                       // 128-row x 64-channel boxes per tile
  static constexpr int kBoxBytes = 128 * 64 * 2;
  static constexpr int kSmemBytes = kBoxes * kBoxBytes;
};

struct QuantArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  uint8_t *qc, *qsf, *kc, *ksf, *vc, *vsf;
  float* part;      // scratch: chunk sums [B*Hkv][Lp/128][D]
  float* kmean;     // [B*Hkv][D]
  int Lq, Lqp, Lkv, Lkvp, nbh_q, nbh_kv, chunks_per_cta;   // Q and K/V tokens (and padded to 128)
  int H, Hkv;                       // heads of Q and of K / V (bh = b * heads + h)
  Strides sq, skv;                  // element strides of the bf16 Q and K / V (BHLD or BLHD)
  int tph_q, tph_k;                 // Q / K tiles of kRows tokens per head
  int ntile_q, ntile_k, nblk_v;
  int nq_first;                     // launch 2: Q tiles taken before the K tiles (the rest after)
  int nclu_mean, nclu_v;            // launch 1: mean clusters, V clusters
  uint64_t wait_ns;
};

// Quantises one quad (minus the 64 means at `mean`, when given) and stores its
// 32 bytes of codes and its scale word: token t of head bh (rows of Lp tokens
// per head), `quad` the 64-channel block within the row.
template <int D>
__device__ __forceinline__ void quant_quad(const uint4 (&w)[8], const float* mean, uint8_t* codes_base,
                                           uint8_t* sf_base, long long bh, int t, int quad, int Lp) {
  uint32_t codes[8];
  uint32_t sfw = 0;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float x[16];
    bf16x8_to_f32(w[2 * g], x);
    bf16x8_to_f32(w[2 * g + 1], x + 8);
    if (mean != nullptr) {
      const float4* m4 = reinterpret_cast<const float4*>(mean + 16 * g);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 m = __ldg(m4 + i);
        x[4 * i + 0] = __fsub_rn(x[4 * i + 0], m.x);
        x[4 * i + 1] = __fsub_rn(x[4 * i + 1], m.y);
        x[4 * i + 2] = __fsub_rn(x[4 * i + 2], m.z);
        x[4 * i + 3] = __fsub_rn(x[4 * i + 3], m.w);
      }
    }
    sfw |= quant_group16(x, codes + 2 * g) << (8 * g);
  }
  uint4* cdst = reinterpret_cast<uint4*>(codes_base + (bh * Lp + t) * (D / 2) + quad * 32);
  cdst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
  cdst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
  const int rb = t / 128, r = t % 128;
  const long long blk = (bh * (Lp / 128) + rb) * (D / 64) + quad;
  *reinterpret_cast<uint32_t*>(sf_base + blk * 512 + (r % 32) * 16 + (r / 32) * 4) = sfw;
}

// Whether tile `tile` of launch 2 is a K tile: tiles [0, nq_first) are Q
// tiles, then come the K tiles, then the other Q tiles.
__device__ __forceinline__ bool tile_is_k(const QuantArgs& a, int tile) {
  return tile >= a.nq_first && tile < a.nq_first + a.ntile_k;
}
// Head and first token of Q/K tile `tile`.
__device__ __forceinline__ void tile_head(const QuantArgs& a, int tile, int rows, bool& is_k, int& bh, int& t0) {
  is_k = tile_is_k(a, tile);
  const int u = is_k ? tile - a.nq_first : (tile < a.nq_first ? tile : tile - a.ntile_k);
  const int tph = is_k ? a.tph_k : a.tph_q;
  bh = u / tph;
  t0 = (u % tph) * rows;
}

// Issues the TMA copies of Q/K tile `tile` into `dst`: tokens [t0, t0 + kRows)
// of one head, boxes of 64 channels x 128 tokens (d = 128: the two channel
// halves; d = 64: two token blocks).  Tokens past L (and a second box wholly
// past Lp) arrive as zeros.
template <int D>
__device__ __forceinline__ void issue_tile_qk(const QuantArgs& a, const CUtensorMap* tq, const CUtensorMap* tk,
                                              int tile, uint8_t* dst, uint64_t* bar) {
  using T = TileQK<D>;
  bool is_k;
  int bh, t0;
  tile_head(a, tile, T::kRows, is_k, bh, t0);
  const CUtensorMap* map = is_k ? tk : tq;
  const int heads = is_k ? a.Hkv : a.H;
  mbar_arrive_expect_tx(bar, T::kBoxes * T::kBoxBytes);
#pragma unroll
  for (int b = 0; b < T::kBoxes; ++b) {
    const int x = D == 128 ? 64 * b : 0;
    const int y = D == 128 ? t0 : t0 + 128 * b;
    tma_load_4d(dst + b * T::kBoxBytes, map, bar, x, y, bh % heads, bh / heads);
  }
}

// Quantises the tile in `src` (128B swizzle: 16-byte chunk i of box row rr
// sits at chunk i ^ (rr & 7)); one quad per thread.
template <int D>
__device__ __forceinline__ void quant_tile_smem(const QuantArgs& a, int tile, const uint8_t* src) {
  using T = TileQK<D>;
  bool is_k;
  int bh, t0;
  tile_head(a, tile, T::kRows, is_k, bh, t0);
  const int r = threadIdx.x / (D / 64), quad = threadIdx.x % (D / 64);
  const int t = t0 + r;
  if (t >= (is_k ? a.Lkvp : a.Lqp)) return;
  const int box = D == 128 ? quad : r / 128, rr = D == 128 ? r : r % 128;
  const uint8_t* base = src + box * T::kBoxBytes + rr * 128;
  uint4 w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = *reinterpret_cast<const uint4*>(base + ((i ^ (rr & 7)) * 16));
  // a token past L arrived as zeros; K' there is kept zero (no mean subtracted)
  if (is_k)
    quant_quad<D>(w, t < a.Lkv ? a.kmean + (size_t)bh * D + quad * 64 : nullptr, a.kc, a.ksf, bh, t, quad, a.Lkvp);
  else
    quant_quad<D>(w, nullptr, a.qc, a.qsf, bh, t, quad, a.Lqp);
}

// One thread per (channel pair, 32 tokens = two 16-token groups).  Items are
// ordered channel pair fastest, so a warp covers 64 consecutive channels of
// the same 32 tokens and each of its 32 loads reads one 128-byte segment of a
// V row.  A channel's two scale bytes are one half of its 64-token scale word.
template <int D>
__device__ __forceinline__ void quant_v_cta(const QuantArgs& a, int blk) {
  constexpr int kPairs = D / 2;
  const long long item = (long long)blk * kThreadsQ + threadIdx.x;
  const int npb = a.Lkvp / 32;                          // 32-token pieces per head (padded length)
  if (item >= (long long)a.nbh_kv * npb * kPairs) return;
  const int c = 2 * (int)(item % kPairs);
  const long long piece = item / kPairs;                // over B*Hkv*npb
  const long long bh = piece / npb;
  const int tp = (int)(piece % npb);
  const int nvalid = a.Lkv - tp * 32;                   // tokens of this piece below Lkv (may be <= 0)
  const long long vb = bh / a.Hkv, vh = bh % a.Hkv;
  const uint32_t* src =
      reinterpret_cast<const uint32_t*>(a.v + vb * a.skv.b + vh * a.skv.h + (long long)tp * 32 * a.skv.t + c);
  const size_t tstep = (size_t)(a.skv.t / 2);           // token stride in bf16 pairs
  uint32_t w[32];
  if (nvalid >= 32) {
#pragma unroll
    for (int t = 0; t < 32; ++t) w[t] = __ldg(src + t * tstep);
  } else {
    // the ragged end of the head: tokens past L count as zeros
#pragma unroll
    for (int t = 0; t < 32; ++t) w[t] = t < nvalid ? __ldg(src + t * tstep) : 0u;
  }
  uint8_t* sblk = a.vsf + ((size_t)bh * (a.Lkvp / 64) + tp / 2) * 512 + (tp % 2) * 2;
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
    *reinterpret_cast<uint4*>(a.vc + ((size_t)bh * D + ch) * (a.Lkvp / 2) + (size_t)tp * 16) =
        make_uint4(codes[0], codes[1], codes[2], codes[3]);
    *reinterpret_cast<uint16_t*>(sblk + (ch % 32) * 16 + (ch / 32) * 4) = (uint16_t)sfw;
    if (D == 64) *reinterpret_cast<uint16_t*>(sblk + (ch % 32) * 16 + (ch / 32 + 2) * 4) = 0;   // padding rows
  }
}

// mu[bh][c] = (chunk sums in chunk order) / L, chunk sum = the chunk's tokens
// (128, fewer in a ragged last chunk) added token by token from 0.  Called by
// all CTAs of one cluster.
template <int D>
__device__ __forceinline__ void mean_cluster(const QuantArgs& a, int bh) {
  constexpr int kPairs = D / 2;
  constexpr int kChunksAtOnce = kThreadsQ / kPairs;
  const uint32_t rank = cluster_ctarank();
  const int nchunk = a.Lkvp / kMeanChunk, cpc = a.chunks_per_cta;
  const int first = (int)rank * cpc, last = min(nchunk, first + cpc);
  const int c = 2 * (threadIdx.x % kPairs);
  for (int ch = first + (int)threadIdx.x / kPairs; ch < last; ch += kChunksAtOnce) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(a.k + (long long)(bh / a.Hkv) * a.skv.b +
                                                            (long long)(bh % a.Hkv) * a.skv.h +
                                                            (long long)ch * kMeanChunk * a.skv.t + c);
    const size_t tstep = (size_t)(a.skv.t / 2);         // token stride in bf16 pairs
    float acc0 = 0.f, acc1 = 0.f;
    const int nvalid = a.Lkv - ch * kMeanChunk;         // tokens of this chunk below Lkv
#pragma unroll 1
    for (int t0 = 0; t0 < kMeanChunk; t0 += 32) {
      // a token past L adds +0, which leaves a float32 sum unchanged (the
      // sum starts at +0 and never becomes -0)
      uint32_t w[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = t0 + i < nvalid ? __ldg(src + (t0 + i) * tstep) : 0u;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        acc0 = __fadd_rn(acc0, __uint_as_float(w[i] << 16));
        acc1 = __fadd_rn(acc1, __uint_as_float(w[i] & 0xFFFF0000u));
      }
    }
    *reinterpret_cast<float2*>(a.part + ((size_t)bh * nchunk + ch) * D + c) = make_float2(acc0, acc1);
  }
  cluster_sync();                                       // every chunk sum of the head is written
  if (rank == 0 && threadIdx.x < D) {
    const int col = threadIdx.x;
    float tot = 0.f;
#pragma unroll 1
    for (int c0 = 0; c0 < nchunk; c0 += 8) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int ch = c0 + j;
        v[j] = ch < nchunk ? __ldcg(a.part + ((size_t)bh * nchunk + ch) * D + col) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (c0 + j < nchunk) tot = __fadd_rn(tot, v[j]);
    }
    a.kmean[(size_t)bh * D + col] = __fdiv_rn(tot, (float)a.Lkv);
  }
}

// Clusters [0, nclu_mean) compute the means, the rest quantise V.  Every CTA
// lets the dependent quant_qk_kernel launch at once (it waits for this
// launch's completion before it reads mu).
template <int D>
__global__ void __cluster_dims__(kMeanCluster, 1, 1) __launch_bounds__(kThreadsQ)
    quant_v_mean_kernel(const QuantArgs a) {
  pdl_launch_dependents();
  const int clu = blockIdx.x / kMeanCluster;
  if (clu < a.nclu_mean) {
    mean_cluster<D>(a, clu);
    return;
  }
  const int blk = (clu - a.nclu_mean) * kMeanCluster + (int)(blockIdx.x % kMeanCluster);
  if (blk < a.nblk_v) quant_v_cta<D>(a, blk);
}

// Persistent: CTA c takes tiles c, c + G, c + 2G, ... (G = grid size) through
// a two-stage TMA ring, the next tile's copy in flight while the current one
// is quantised.
template <int D>
__global__ void __launch_bounds__(kThreadsQ, 3) quant_qk_kernel(const __grid_constant__ CUtensorMap tmap_q,
                                                             const __grid_constant__ CUtensorMap tmap_k,
                                                             const QuantArgs a) {
  using T = TileQK<D>;
  // the attention launch behind this one may start (it waits for this
  // launch's completion before it reads the codes)
  pdl_launch_dependents();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[2];
  __shared__ int abort_flag;
  const int ntiles = a.ntile_k + a.ntile_q, G = gridDim.x;
  if (threadIdx.x == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const bool leader = threadIdx.x == 0;
  int tile = blockIdx.x;
  int issued[2] = {0, 0};                               // loads issued per stage (leader's count)
  if (leader) {
    if (tile < ntiles) {
      issue_tile_qk<D>(a, &tmap_q, &tmap_k, tile, smem, &full[0]);
      issued[0] = 1;
    }
    if (tile + G < ntiles) {
      issue_tile_qk<D>(a, &tmap_q, &tmap_k, tile + G, smem + T::kSmemBytes, &full[1]);
      issued[1] = 1;
    }
  }
  bool ok = true, waited = false;
  int i = 0;
  for (; tile < ntiles; ++i, tile += G) {
    const int st = i & 1;
    if (!mbar_wait(&full[st], (i >> 1) & 1, &abort_flag, a.wait_ns)) {
      ok = false;
      break;
    }
    if (!waited && tile_is_k(a, tile)) {
      pdl_wait();                                       // mu is written by launch 1
      waited = true;
    }
    quant_tile_smem<D>(a, tile, smem + st * T::kSmemBytes);
    __syncthreads();                                    // stage st has been read by every thread
    if (leader && tile + 2 * G < ntiles) {
      issue_tile_qk<D>(a, &tmap_q, &tmap_k, tile + 2 * G, smem + st * T::kSmemBytes, &full[st]);
      ++issued[st];
    }
  }
  if (!ok && leader) {
    // never leave with a copy in flight: wait (bounded) for each stage's last
    // issued load, the use-th load of a stage completing phase use - 1
    for (int st = 0; st < 2; ++st) {
      const int consumed = (i + 1 - st) / 2;            // loads of stage st waited for so far
      if (issued[st] > consumed) mbar_wait_drain(&full[st], (issued[st] - 1) & 1, a.wait_ns);
    }
  }
  // this launch completes only after launch 1 has: what follows in the stream
  // may then read every output of sa_quantize
  if (!waited) pdl_wait();
}

template <int D>
cudaError_t launch_quantize_impl(const void* q, const void* k, const void* v, const Dims& dm, bool blhd,
                                 const sa_fp4_qkv& out, float* partials, const CUtensorMap& tq,
                                 const CUtensorMap& tk, cudaStream_t s) {
  using T = TileQK<D>;
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
  a.Lq = dm.Lq;
  a.Lqp = padded_len(dm.Lq);
  a.Lkv = dm.Lkv;
  a.Lkvp = padded_len(dm.Lkv);
  a.H = dm.H;
  a.Hkv = dm.Hkv;
  a.sq = layout_strides(blhd, dm.H, dm.Lq, dm.d);
  a.skv = layout_strides(blhd, dm.Hkv, dm.Lkv, dm.d);
  a.nbh_q = dm.B * dm.H;
  a.nbh_kv = dm.B * dm.Hkv;
  const int nchunk = a.Lkvp / kMeanChunk;
  a.chunks_per_cta = (nchunk + kMeanCluster - 1) / kMeanCluster;
  a.tph_q = (a.Lqp + T::kRows - 1) / T::kRows;
  a.tph_k = (a.Lkvp + T::kRows - 1) / T::kRows;
  a.ntile_q = a.nbh_q * a.tph_q;
  a.ntile_k = a.nbh_kv * a.tph_k;
  a.nblk_v = (int)(((long long)a.nbh_kv * (a.Lkvp / 32) * (D / 2) + kThreadsQ - 1) / kThreadsQ);
  a.nclu_mean = a.nbh_kv;
  a.nclu_v = (a.nblk_v + kMeanCluster - 1) / kMeanCluster;
  a.wait_ns = kWaitLimitNs;
  constexpr int kSmem = 2 * T::kSmemBytes + 1024;        // two stages + alignment slack
  static std::atomic<bool> attr_done[kMaxDevices];   // kernel attributes are per device
  cudaError_t ea = once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(quant_qk_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (ea != cudaSuccess) return ea;
  const int ntiles = a.ntile_k + a.ntile_q;
  const int sms = device_sm_count() > 0 ? device_sm_count() : 148;
  const int grid = ntiles < 3 * sms ? ntiles : 3 * sms;    // three resident CTAs per SM
  // one round of Q tiles runs beside launch 1; K follows while it is in L2
  a.nq_first = a.ntile_q < grid ? a.ntile_q : grid;
  quant_v_mean_kernel<D><<<(a.nclu_mean + a.nclu_v) * kMeanCluster, kThreadsQ, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // launch 2 may start while launch 1 drains (programmatic dependent launch)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreadsQ);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quant_qk_kernel<D>, tq, tk, a);
}

}  // namespace

cudaError_t quant_read_error(int* out) { return read_and_clear_device_error(out); }

cudaError_t launch_quantize(const void* q, const void* k, const void* v, const Dims& dm, bool blhd,
                            const sa_fp4_qkv& out, const CUtensorMap& tq, const CUtensorMap& tk, cudaStream_t s) {
  float* part = static_cast<float*>(out.workspace);
  return dm.d == 64 ? launch_quantize_impl<64>(q, k, v, dm, blhd, out, part, tq, tk, s)
                    : launch_quantize_impl<128>(q, k, v, dm, blhd, out, part, tq, tk, s);
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
                                           const sa_fp4_qkv& out, const CUtensorMap& tq, const CUtensorMap& tk,
                                           cudaStream_t s) {
  // (sa_quantize_static_scratch has checked kmean_partial_floats(dm) <=
  // kStaticScratchFloats before calling)
  float* part = nullptr;
  cudaError_t e = static_scratch_address(&part);
  if (e != cudaSuccess) return e;
  // Every chunk sum read is written first by the same call (its first
  // launch), so earlier contents of the array never reach the outputs and
  // nothing needs clearing.
  return dm.d == 64 ? launch_quantize_impl<64>(q, k, v, dm, false, out, part, tq, tk, s)
                    : launch_quantize_impl<128>(q, k, v, dm, false, out, part, tq, tk, s);
}

}  // namespace sa
