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
#include "quant_group.cuh"
#include "sm100.cuh"

namespace sa {

namespace {


using namespace qg;   // the group arithmetic (quant_group.cuh)

// ---------------------------------------------------------------------------
// Two launches of one persistent kernel body, each CTA a TMA producer warp and
// kWorkers worker warps over a ring of kStages tiles.  A tile is 32 KB of one
// bf16 head: two TMA boxes of 64 channels x 128 tokens, 128B-swizzled (16-byte
// chunk c of box row rr at chunk c ^ (rr & 7)); d = 128: 128 tokens, the two
// channel halves; d = 64: 256 tokens.  Tokens past L arrive as zeros.  Every
// worker warp waits for every tile of its CTA in order, takes a fixed share
// of it and releases the ring slot with one arrival; warps are not
// synchronised with each other beyond that, so a warp with more work on one
// tile (the mean sums) catches up on the next ones.
//   pass 1: Q tiles alternating with K-mean tiles (an odd grid, so that each
//     CTA alternates too):
//     Q    one thread per quad (64 channels of one token = four 1x16 groups =
//          one 32-bit scale word): eight conflict-free 16-byte shared loads,
//          32 bytes of codes and the scale word stored in the MMA scale layout;
//     mean two warps per tile (which two rotates from tile to tile), one
//          thread per channel pair: the chunk sum of 128 tokens, token by
//          token from 0, to the scratch buffer.
//   pass 2 (a programmatic dependent launch of pass 1): V tiles and the K'
//     tiles, each CTA over round-robin V tiles and a contiguous range of K'
//     tiles, two V tiles first and then the two kinds alternating.  The V
//     tiles and the K loads need nothing from pass 1; before its first K'
//     tile each CTA waits for pass 1 (griddepcontrol.wait) and forms the
//     means of its range's heads (chunk sums added in chunk order, divided by
//     L).  K is then mostly in L2, where pass 1 has just read it.
//     V    one thread per channel pair and 32 tokens (two 16-token groups per
//          channel): 32 four-byte shared loads (a warp reads 32 words of one
//          box row), 16 bytes of transposed codes per channel;
//     K'   as Q, on K' = RN(k - mean) in float32.
// Every layout holds Lp = L rounded up to 128 tokens per head; the tokens past
// L are written as zero codes with zero scales (Q and K rows, V token groups),
// and a V group that straddles L is quantised with zeros for its missing
// tokens.

constexpr int kWorkers = 8;                              // worker warps per CTA
constexpr int kThreadsQ = (kWorkers + 1) * 32;           // + one TMA producer warp
constexpr int kStages = 3;
constexpr int kCtasPerSm = 2;
constexpr int kBoxBytes = 128 * 64 * 2;                  // 128 tokens x 64 bf16 channels
constexpr int kTileBytes = 2 * kBoxBytes;
constexpr int kMaxMeanHeads = 8;                         // heads per pass-2 CTA range (at most)
constexpr int kSmemQ = kStages * kTileBytes + 1024;      // ring + alignment slack

template <int D>
struct TileGeo {
  static constexpr int kRows = D == 128 ? 128 : 256;    // tokens per tile
};

enum TileKind { kTileQ = 0, kTileV = 1, kTileMean = 2, kTileK = 3 };

struct QuantArgs {
  uint8_t *qc, *qsf, *kc, *ksf, *vc, *vsf;
  float* part;      // chunk sums [B*Hkv][Lkvp/128][D]
  float* kmean;     // [B*Hkv][D]
  int Lkv, Lqp, Lkvp;
  int H, Hkv;
  int tph_q, tph_k;                 // tiles per head of Q and of K / V
  uint32_t dq_m, dq_l, dk_m, dk_l;  // u / tph_q and u / tph_k as (umulhi(u, m) + u) >> l
  int ntile_q, ntile_k;             // Q tiles; K tiles (= V tiles = mean tiles)
  uint64_t wait_ns;
};

struct TileRef {
  int kind, bh, t0;
};

// floor(u / d) for 0 <= u < 2^31 from (m, l) = (floor(2^32 (2^l - d) / d) + 1,
// ceil(log2 d)) (Granlund and Montgomery's multiply-shift division).
__host__ __device__ inline void fastdiv_params(uint32_t d, uint32_t& m, uint32_t& l) {
  l = 0;
  while ((1ull << l) < d) ++l;
  m = (uint32_t)((((1ull << 32) * ((1ull << l) - d)) / d) + 1);
}
__device__ __forceinline__ int fastdiv(int u, uint32_t m, uint32_t l) {
  return (int)((__umulhi((uint32_t)u, m) + (uint32_t)u) >> l);
}

template <int D>
__device__ __forceinline__ TileRef head_tile(int kind, int u, int tph, uint32_t m, uint32_t l) {
  const int bh = fastdiv(u, m, l);
  return TileRef{kind, bh, (u - bh * tph) * TileGeo<D>::kRows};
}

// Element j of two lists merged alternately (x first, then the rest of the
// longer one): sets `second` (an element of y) and returns the index in its
// list.
__device__ __forceinline__ int merge_at(int nx, int ny, int j, bool& second) {
  const int m = min(nx, ny);
  if (j < 2 * m) {
    second = (j & 1) != 0;
    return j >> 1;
  }
  second = ny > nx;
  return j - m;
}

// Pass 1, tile u of ntile_q + ntile_k: Q and mean tiles merged alternately.
template <int D>
__device__ __forceinline__ TileRef pass1_tile(const QuantArgs& a, int u) {
  bool mean;
  const int j = merge_at(a.ntile_q, a.ntile_k, u, mean);
  return mean ? head_tile<D>(kTileMean, j, a.tph_k, a.dk_m, a.dk_l) : head_tile<D>(kTileQ, j, a.tph_q, a.dq_m, a.dq_l);
}

// Pass 2, CTA c of G: its V tiles c, c + G, ... (nv) and the K' tiles of its
// contiguous range [k0, k0 + nk), in the order: the first nv0 = min(nv, 2) V
// tiles (they need nothing from pass 1 and cover its wait), then K' and the
// other V tiles merged alternately.
template <int D>
__device__ __forceinline__ TileRef pass2_tile(const QuantArgs& a, int c, int G, int nv, int k0, int nk, int i) {
  const int nv0 = min(nv, 2);
  if (i < nv0) return head_tile<D>(kTileV, c + i * G, a.tph_k, a.dk_m, a.dk_l);
  bool v;
  const int j = merge_at(nk, nv - nv0, i - nv0, v);
  return v ? head_tile<D>(kTileV, c + (nv0 + j) * G, a.tph_k, a.dk_m, a.dk_l)
           : head_tile<D>(kTileK, k0 + j, a.tph_k, a.dk_m, a.dk_l);
}

// Issues the two box copies of tile t into dst.  K read for its mean (pass
// 1) is kept in L2 for pass 2's K' tiles (evict_last); every other read is
// the data's last (evict_first), which leaves L2 to K and to the outputs the
// attention kernel reads next.
template <int D>
__device__ __forceinline__ void issue_tile(const TileRef& t, const CUtensorMap* tq, const CUtensorMap* tk,
                                           const CUtensorMap* tv, const QuantArgs& a, uint8_t* dst, uint64_t* bar) {
  const CUtensorMap* map = t.kind == kTileQ ? tq : (t.kind == kTileV ? tv : tk);
  const int heads = t.kind == kTileQ ? a.H : a.Hkv;
  const uint64_t pol = t.kind == kTileMean ? l2_policy_evict_last() : l2_policy_evict_first();
  mbar_arrive_expect_tx(bar, kTileBytes);
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const int x = D == 128 ? 64 * b : 0;
    const int y = D == 128 ? t.t0 : t.t0 + 128 * b;
    tma_load_4d_hint(dst + b * kBoxBytes, map, bar, x, y, t.bh % heads, t.bh / heads, pol);
  }
}

// Q (IS_K false) or K' (IS_K true: `nmean` = -mean of the head, in shared
// memory) rows of a tile: one quad per thread.  d = 128: warp w takes box
// w & 1 (the quad) and rows 32 (w >> 1) + lane; d = 64: rows 32 w + lane.  A
// quarter-warp reads 8 consecutive rows of one box: 8 distinct chunks.
template <int D, bool IS_K>
__device__ __forceinline__ void quant_rows(const QuantArgs& a, const TileRef& t, const uint8_t* tile, int warp,
                                           int lane, const float2* rtab, const float* nmean) {
  const int tl = D == 128 ? 32 * (warp >> 1) + lane : 32 * warp + lane;
  const int box = D == 128 ? (warp & 1) : (tl >> 7);
  const int rr = tl & 127, quad = D == 128 ? box : 0;
  const int tok = t.t0 + tl;
  const int Lp = IS_K ? a.Lkvp : a.Lqp;
  if (tok >= Lp) return;                               // (d = 64: warp-uniform)
  uint32_t w[32];
  load_box_row(tile + box * kBoxBytes, rr, w);
  uint32_t codes[8];
  uint32_t sfw;
  if constexpr (!IS_K) {
    quant_q_quad(w, rtab, codes, sfw);
  } else {
    // K' = RN(k - mean); a token past L arrived as zeros and K' there is kept
    // zero (no mean subtracted)
    const bool sub = tok < a.Lkv;
    float x[4][16], am[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const float4* m4 = reinterpret_cast<const float4*>(nmean + quad * 64 + 16 * g);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 m = sub ? m4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        add2(x[g][4 * i], x[g][4 * i + 1], bf16_lo(w[8 * g + 2 * i]), bf16_hi(w[8 * g + 2 * i]), m.x, m.y);
        add2(x[g][4 * i + 2], x[g][4 * i + 3], bf16_lo(w[8 * g + 2 * i + 1]), bf16_hi(w[8 * g + 2 * i + 1]), m.z,
             m.w);
      }
      float mx = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fabsf(x[g][i]));
      am[g] = mx;
    }
    sfw = scale_pair(am[0], am[1]) | (scale_pair(am[2], am[3]) << 16);
#pragma unroll
    for (int g = 0; g < 4; ++g) codes_group(x[g], (sfw >> (8 * g)) & 0xFFu, rtab, codes + 2 * g);
  }
  uint8_t* cbase = IS_K ? a.kc : a.qc;
  uint8_t* sbase = IS_K ? a.ksf : a.qsf;
  uint4* cdst = reinterpret_cast<uint4*>(cbase + ((size_t)t.bh * Lp + tok) * (D / 2) + quad * 32);
  cdst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
  cdst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
  const int r = tok & 127;
  const size_t blk = ((size_t)t.bh * (Lp / 128) + (tok >> 7)) * (D / 64) + quad;
  *reinterpret_cast<uint32_t*>(sbase + blk * 512 + (r & 31) * 16 + (r >> 5) * 4) = sfw;
}

// Row offsets within a box row of the word of channel pair `lane` (0..31) for
// the 8 swizzle phases: chunk (lane >> 2) ^ phase, word lane & 3.
__device__ __forceinline__ void pair_offsets(int lane, uint32_t (&off)[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) off[k] = ((((uint32_t)lane >> 2) ^ (uint32_t)k) << 4) | (((uint32_t)lane & 3u) << 2);
}

// V tile: one thread per channel pair and 32 tokens.  d = 128: warp w takes
// box w & 1 and tokens 32 (w >> 1) ..; d = 64: tokens 32 w .. (box w / 4).
template <int D>
__device__ __forceinline__ void quant_v(const QuantArgs& a, const TileRef& t, const uint8_t* tile, int warp, int lane,
                                        const float2* rtab) {
  const int box = D == 128 ? (warp & 1) : (warp >> 2);
  const int tl0 = D == 128 ? 32 * (warp >> 1) : 32 * warp;
  const int tok0 = t.t0 + tl0;
  if (tok0 >= a.Lkvp) return;                           // (d = 64: warp-uniform)
  const uint8_t* src = tile + box * kBoxBytes + (tl0 & 127) * 128;
  uint32_t off[8];
  pair_offsets(lane, off);
  uint32_t w[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) w[j] = *reinterpret_cast<const uint32_t*>(src + j * 128 + off[j & 7]);
  // per-channel maxima of the two 16-token groups (low halves: channel c)
  float a0, a1, b0, b1;
  absmax_halves<16>(w, a0, a1);
  absmax_halves<16>(w + 16, b0, b1);
  const uint32_t s01 = scale_pair(a0, a1);              // group 0: channel c (low byte), c + 1
  const uint32_t s23 = scale_pair(b0, b1);              // group 1
  const int c = (D == 128 ? 64 * box : 0) + 2 * lane;
  uint8_t* sblk = a.vsf + ((size_t)t.bh * (a.Lkvp / 64) + (tok0 >> 6)) * 512 + ((tok0 & 63) >> 4);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t codes[4];
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = h ? bf16_hi(w[16 * g + i]) : bf16_lo(w[16 * g + i]);
      codes_group(x, ((g ? s23 : s01) >> (8 * h)) & 0xFFu, rtab, codes + 2 * g);
    }
    const int ch = c + h;
    *reinterpret_cast<uint4*>(a.vc + ((size_t)t.bh * D + ch) * (a.Lkvp / 2) + (tok0 >> 1)) =
        make_uint4(codes[0], codes[1], codes[2], codes[3]);
    const uint32_t sc = ((s01 >> (8 * h)) & 0xFFu) | (((s23 >> (8 * h)) & 0xFFu) << 8);
    *reinterpret_cast<uint16_t*>(sblk + (ch & 31) * 16 + (ch >> 5) * 4) = (uint16_t)sc;
    if (D == 64) *reinterpret_cast<uint16_t*>(sblk + (ch & 31) * 16 + ((ch >> 5) + 2) * 4) = 0;   // padding rows
  }
}

// K-mean tile, on the two warps `sel` (0 or 1 = box for d = 128, chunk half
// for d = 64): thread = channel pair, the 128-token chunk sum token by token
// from 0 (a token past L adds +0, which leaves a float32 sum unchanged: the
// sum starts at +0 and never becomes -0).
template <int D>
__device__ __forceinline__ void mean_chunk(const QuantArgs& a, const TileRef& t, const uint8_t* tile, int sel,
                                           int lane) {
  const int tok0 = D == 128 ? t.t0 : t.t0 + 128 * sel;
  if (tok0 >= a.Lkvp) return;
  const uint8_t* src = tile + sel * kBoxBytes;
  uint32_t off[8];
  pair_offsets(lane, off);
  float s0 = 0.f, s1 = 0.f;
#pragma unroll 2
  for (int j0 = 0; j0 < 128; j0 += 8) {
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = *reinterpret_cast<const uint32_t*>(src + (j0 + k) * 128 + off[k]);
#pragma unroll
    for (int k = 0; k < 8; ++k) add2(s0, s1, s0, s1, bf16_lo(w[k]), bf16_hi(w[k]));
  }
  const int c = (D == 128 ? 64 * sel : 0) + 2 * lane;
  const int nchunk = a.Lkvp / kMeanChunk;
  *reinterpret_cast<float2*>(a.part + ((size_t)t.bh * nchunk + (tok0 / kMeanChunk)) * D + c) = make_float2(s0, s1);
}

template <int D, int PASS>
__global__ void __launch_bounds__(kThreadsQ, kCtasPerSm)
    quant_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v, const QuantArgs a) {
  // the launch behind this one (pass 2, or the attention) may be scheduled at
  // once: it waits for this launch's completion before it reads its outputs
  pdl_launch_dependents();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[kStages], empty[kStages], mean_ready;
  __shared__ int abort_flag;
  __shared__ float2 rtab[128];
  __shared__ __align__(16) float nmean[PASS == 2 ? kMaxMeanHeads * D : 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the tiles of this CTA: pass 1 c, c + G, ... of ntile_q + ntile_k; pass 2
  // nv V tiles and the K' tiles [k0, k0 + nk)
  const int G = gridDim.x, c = blockIdx.x;
  const int n1 = a.ntile_q + a.ntile_k;
  const int nv = c < a.ntile_k ? (a.ntile_k - c + G - 1) / G : 0;
  // pass 2: K' tiles cut into G near-equal contiguous ranges (the first
  // ntile_k % G of them one tile longer)
  const int kq = a.ntile_k / G, kr = a.ntile_k % G;
  const int k0 = c * kq + min(c, kr), nk = kq + (c < kr ? 1 : 0);
  const int kh0 = k0 / a.tph_k;                         // first head of the K' range
  const int ntiles = PASS == 1 ? (c < n1 ? (n1 - c + G - 1) / G : 0) : nv + nk;
  auto tile_at = [&](int i) {
    return PASS == 1 ? pass1_tile<D>(a, c + i * G) : pass2_tile<D>(a, c, G, nv, k0, nk, i);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWorkers);
    }
    mbar_init(&mean_ready, D / 32);
    abort_flag = 0;
    fence_barrier_init();
  }
  if (threadIdx.x < 128) rtab[threadIdx.x] = rtab_entry(threadIdx.x);   // (yh, yl) of each scale byte
  __syncthreads();

  if (warp == kWorkers) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int i = 0;
      bool ok = true;
      for (; i < ntiles; ++i) {
        const int st = i % kStages;
        if (i >= kStages && !mbar_wait_backoff(&empty[st], ((i / kStages) - 1) & 1, &abort_flag, a.wait_ns, 64)) {
          ok = false;
          break;
        }
        issue_tile<D>(tile_at(i), &tmap_q, &tmap_k, &tmap_v, a, ring + st * kTileBytes, &full[st]);
      }
      if (!ok) {
        // never leave with a copy in flight: wait (bounded) for each stage's
        // last load (tiles 0 .. i - 1 were issued, tile j to stage j % kStages;
        // the n-th load of a stage completes its phase n - 1)
        for (int st = 0; st < kStages; ++st) {
          const int n = (i - st + kStages - 1) / kStages;
          if (n > 0) mbar_wait_drain(&full[st], (n - 1) & 1, a.wait_ns);
        }
      }
    }
  } else {
    // ----------------------------------------------------------------- workers
    // one tile: wait for its copy, quantise this warp's share, release the
    // slot (every warp sees every phase of every stage in order)
    auto work = [&](int i) -> bool {
      const int st = i % kStages;
      if (!mbar_wait(&full[st], (i / kStages) & 1, &abort_flag, a.wait_ns)) return false;
      const uint8_t* tile = ring + st * kTileBytes;
      const TileRef t = tile_at(i);
      if (t.kind == kTileQ) {
        quant_rows<D, false>(a, t, tile, warp, lane, rtab, nullptr);
      } else if (t.kind == kTileV) {
        quant_v<D>(a, t, tile, warp, lane, rtab);
      } else if (t.kind == kTileMean) {
        const int w0 = 2 * (i & 3);                     // the two warps of this mean tile
        if (warp == w0 || warp == w0 + 1) mean_chunk<D>(a, t, tile, warp - w0, lane);
      } else {
        quant_rows<D, true>(a, t, tile, warp, lane, rtab, nmean + (t.bh - kh0) * D);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      return true;
    };
    // pass 2: the tiles before the first K' tile (all of them without K' tiles)
    const int nfirst = PASS == 1 ? ntiles : (nk > 0 ? min(nv, 2) : ntiles);
    bool ok = true;
    for (int i = 0; ok && i < nfirst; ++i) ok = work(i);
    if (PASS == 2 && ok && nk > 0) {
      // before the first K' tile: the chunk sums are written by pass 1
      pdl_wait();
      // -mean of every head of the range (warps 0 .. D/32 - 1, one channel each)
      if (threadIdx.x < D) {
        const int ch = threadIdx.x;
        const int nchunk = a.Lkvp / kMeanChunk;
        const int h1 = (k0 + nk - 1) / a.tph_k;
        for (int bh = kh0; bh <= h1; ++bh) {
          const float* p = a.part + (size_t)bh * nchunk * D + ch;
          float tot = 0.f;
#pragma unroll 1
          for (int c0 = 0; c0 < nchunk; c0 += 16) {
            float v[16];                                // 16 loads in flight, then the adds in order
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = c0 + j < nchunk ? __ldcg(p + (size_t)(c0 + j) * D) : 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c0 + j < nchunk) tot = __fadd_rn(tot, v[j]);
          }
          const float mu = __fdiv_rn(tot, (float)a.Lkv);
          nmean[(bh - kh0) * D + ch] = -mu;
          if (k0 <= bh * a.tph_k) a.kmean[(size_t)bh * D + ch] = mu;   // the range holding the head's first tile
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&mean_ready);
      }
      ok = mbar_wait(&mean_ready, 0, &abort_flag, a.wait_ns);
      for (int i = nfirst; ok && i < ntiles; ++i) ok = work(i);
    }
  }
  // (pass 2 completes only after pass 1 has: the workers of every CTA with
  // K' tiles waited for it, so what follows in the stream may then read
  // every output of sa_quantize)
}

template <int D>
cudaError_t launch_quantize_impl(const Dims& dm, const sa_fp4_qkv& out, float* partials, const CUtensorMap& tq,
                                 const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s, bool with_q = true) {
  constexpr int R = TileGeo<D>::kRows;
  QuantArgs a;
  a.qc = static_cast<uint8_t*>(out.q_codes);
  a.qsf = static_cast<uint8_t*>(out.q_sf);
  a.kc = static_cast<uint8_t*>(out.k_codes);
  a.ksf = static_cast<uint8_t*>(out.k_sf);
  a.vc = static_cast<uint8_t*>(out.v_codes);
  a.vsf = static_cast<uint8_t*>(out.v_sf);
  a.part = partials;
  a.kmean = out.k_mean;
  a.Lkv = dm.Lkv;
  a.Lqp = padded_len(dm.Lq);
  a.Lkvp = padded_len(dm.Lkv);
  a.H = dm.H;
  a.Hkv = dm.Hkv;
  a.tph_q = (a.Lqp + R - 1) / R;
  a.tph_k = (a.Lkvp + R - 1) / R;
  a.ntile_q = with_q ? dm.B * dm.H * a.tph_q : 0;       // (without Q: pass 1 takes the K-mean tiles only)
  a.ntile_k = dm.B * dm.Hkv * a.tph_k;
  a.wait_ns = kWaitLimitNs;
  fastdiv_params((uint32_t)a.tph_q, a.dq_m, a.dq_l);
  fastdiv_params((uint32_t)a.tph_k, a.dk_m, a.dk_l);
  static std::atomic<bool> attr_done[kMaxDevices];   // kernel attributes are per device
  cudaError_t ea = once_per_device(attr_done, [] {
    cudaError_t e = cudaFuncSetAttribute(quant_kernel<D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemQ);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(quant_kernel<D, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemQ);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  const int sms = device_sm_count() > 0 ? device_sm_count() : 148;
  const int slots = kCtasPerSm * sms;
  const int n1 = a.ntile_q + a.ntile_k;
  // an odd grid, so that CTA c (tiles c, c + G, ...) alternates between Q and
  // mean tiles instead of taking only one kind
  const int odd_slots = (slots & 1) ? slots : slots - 1;
  const int grid1 = n1 < odd_slots ? n1 : odd_slots;
  // pass 2: one CTA per slot (fewer with fewer K tiles), each over a
  // near-equal contiguous range of K' tiles (floor or ceil of ntile_k /
  // grid2: every slot busy, no SM with twice the tiles of another) spanning
  // at most kMaxMeanHeads heads (a range of r tiles spans at most
  // ceil((r - 1) / tph_k) + 1 heads)
  const int max_range = (kMaxMeanHeads - 1) * a.tph_k + 1;
  int grid2 = a.ntile_k < slots ? a.ntile_k : slots;
  if (grid2 < (a.ntile_k + max_range - 1) / max_range) grid2 = (a.ntile_k + max_range - 1) / max_range;
  quant_kernel<D, 1><<<grid1, kThreadsQ, kSmemQ, s>>>(tq, tk, tv, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // pass 2 may start while pass 1 drains (programmatic dependent launch)
  cudaLaunchAttribute attr;
  const cudaLaunchConfig_t cfg = pdl_launch_config(dim3(grid2), dim3(kThreadsQ), kSmemQ, s, &attr);
  return cudaLaunchKernelEx(&cfg, quant_kernel<D, 2>, tq, tk, tv, a);
}

}  // namespace

cudaError_t quant_read_error(int* out) { return read_and_clear_device_error(out); }

cudaError_t launch_quantize(const Dims& dm, const sa_fp4_qkv& out, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, cudaStream_t s, bool with_q) {
  float* part = static_cast<float*>(out.workspace);
  return dm.d == 64 ? launch_quantize_impl<64>(dm, out, part, tq, tk, tv, s, with_q)
                    : launch_quantize_impl<128>(dm, out, part, tq, tk, tv, s, with_q);
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

cudaError_t launch_quantize_static_scratch(const Dims& dm, const sa_fp4_qkv& out, const CUtensorMap& tq,
                                           const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
  // (sa_quantize_static_scratch has checked kmean_partial_floats(dm) <=
  // kStaticScratchFloats before calling)
  float* part = nullptr;
  cudaError_t e = static_scratch_address(&part);
  if (e != cudaSuccess) return e;
  // Every chunk sum read is written first by the same call (its first
  // launch), so earlier contents of the array never reach the outputs and
  // nothing needs clearing.
  return dm.d == 64 ? launch_quantize_impl<64>(dm, out, part, tq, tk, tv, s)
                    : launch_quantize_impl<128>(dm, out, part, tq, tk, tv, s);
}

}  // namespace sa
