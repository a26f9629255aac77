// attn_decode.cu -- NVFP4 attention for a few query rows per key/value head:
// a decode step (one query token; the G query heads of a kv head read the
// same keys and values) or a short chunk of queries.
//
// The same computation as attn_nvfp4.cu -- SageAttention3's two-level P
// quantisation ("GPU kernel porting with AI agents", section "Sage Attention
// 3": a per-row, per-key-tile first level s1 = rowmax / (448 * 6), then 1x16
// groups with e4m3 scales) inside FlashAttention's online softmax ("FlashAttention
// kernels", sections 0-1), with the keys split over CTAs and the partial
// results merged afterwards (Flash-Decoding, section 3 of that page) -- laid
// out for nr <= 16 query rows instead of 128:
//   S^T = K' Q^T     M = 128 keys,     N = 16 query rows, K = d
//   O^T += V^T P^T   M = 128 channels, N = 16 query rows, K = 128 keys
// both block-scaled FP4 tcgen05 MMAs with fp32 accumulators in tensor memory.
// A softmax thread owns one key of the tile (one tensor-memory lane of S^T)
// and all 16 rows (its 16 columns); a row's tile maximum is a maximum over
// the 128 lanes (warp shuffles, then the four warps' partial maxima through
// shared memory), a 1x16 group of P is 16 consecutive lanes (shuffles).  So
// the softmax spends its work on the nr valid rows only, where a 128-row
// tile would run a full pass per key tile for them.  The row sums stay per
// key (per thread) and are added up once, at the end of the unit.
//
// Numerics follow attn_nvfp4.cu step for step per (row, key): base-2 logits
// x = S * log2(e) / sqrt(d); a key tile is skipped for a row when its maximum
// is more than 64 (log2 units) below the running maximum; P2 = 2^(x - m_t) *
// 448 * 6; group scale e4m3(RN(max16(P2) * RN(1/6))); codes e2m1(P2 / s2); O
// kept in units of the latest live tile maximum, rescaled per tile.
//
// Warps: 0 TMA producer (and the Q gather), 1 MMA issuer, 2-5 softmax (warp w
// reads tensor-memory lanes 32 (w % 4) ..).  A CTA works through segments
// (key tiles of one (batch, kv head) pair): one key share of a pair, with the
// partial results of several shares merged by splitkv.cu's combine pass; or,
// balanced over the SMs, an equal range of all (pair, key tile) items, with
// the pairs that ranges cut merged by decode_combine_kernel.

#include <cuda_bf16.h>

#include "internal.h"
#include "sm100.cuh"

namespace sa {
namespace {

constexpr int kNR = 16;                      // query rows per pair (MMA N)
constexpr int kDecThreads = 192;
constexpr int kDecNSK = 3;                   // K stages (released by S^T, read ahead for it)
constexpr int kDecNSV = 2;                   // V stages (released by P.V, a tile later); four CTAs of the
                                             // 4-row kernel fit an SM
constexpr int kKeys = 128;                   // keys per tile
constexpr float kLog2PRangeDec = 11.392317422778761f;   // log2(448 * 6)
constexpr float kSkipBelowDec = 64.0f;                   // log2 units

template <int D>
struct CfgDec {
  static constexpr int NSK = kDecNSK, NSV = kDecNSV;
  static constexpr int kRowBytes = D / 2;                // packed codes per Q / K row
  static constexpr int kQBytes = kNR * kRowBytes;
  static constexpr int kQSfBytes = (D / 64) * 512;
  static constexpr int kKBytes = kKeys * kRowBytes;
  static constexpr int kKSfBytes = (D / 64) * 512;
  static constexpr int kVBytes = 128 * (kKeys / 2);      // V^T as 128 rows x 64 bytes (d = 64: rows >= 64 unused)
  static constexpr int kVLoadBytes = D * (kKeys / 2);
  static constexpr int kVSfBytes = 2 * 512;
  static constexpr int kPBytes = kNR * (kKeys / 2);      // P^T: 16 rows x 64 bytes
  static constexpr int kPSfBytes = 2 * 512;
  static constexpr int kOffQ = 0;                        // [2] by segment parity
  static constexpr int kOffK = 2048;
  static_assert(kQBytes <= 1024, "Q^T region");
  static constexpr int kOffV = kOffK + NSK * kKBytes;
  static constexpr int kOffP = kOffV + NSV * kVBytes;     // [2]
  static constexpr int kOffQSf = kOffP + 2 * kPBytes;     // [2] by segment parity
  static constexpr int kOffKSf = kOffQSf + 2 * kQSfBytes;
  static constexpr int kOffVSf = kOffKSf + NSK * kKSfBytes;
  static constexpr int kOffPSf = kOffVSf + NSV * kVSfBytes;  // [2]
  static constexpr int kOffRed = kOffPSf + 2 * kPSfBytes;    // [2][4 warps][16 rows] row maxima, then [4][16] sums
  static constexpr int kOffBar = kOffRed + 3 * 4 * kNR * 4;
  static constexpr int kNumBars = 2 + 2 + 2 * NSK + 2 * NSV + 2 + 2 + 2 + 2 + 2 + 1 + 2;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
  static constexpr uint32_t kQKSwz = (D == 128) ? kSwizzle64B : kSwizzle32B;
  static constexpr uint32_t kQKSbo = 8 * kRowBytes;
  // tensor-memory columns: S^T and the two O^T accumulators by key-tile
  // parity, and the scale factors (Q scales by segment parity; K, V and P
  // scales by key-tile parity: a tcgen05.cp is not ordered after earlier MMAs
  // that read the columns it overwrites)
  static constexpr uint32_t kColS = 0;                    // + 16 * (g & 1)
  static constexpr uint32_t kColO = 32;                   // + 16 * (g & 1)
  static constexpr uint32_t kColSfQ = 64;                 // + 8 * (k & 1)
  static constexpr uint32_t kColSfK = 80;                 // + 8 * (g & 1)
  static constexpr uint32_t kColSfV = 96;                 // + 8 * (g & 1)
  static constexpr uint32_t kColSfP = 112;                // + 8 * (g & 1)
  static constexpr uint32_t kTmemCols = 128;
  static constexpr uint32_t kIdesc = idesc_nvf4(128, kNR);
  static_assert(kColSfP + 16 <= kTmemCols, "tensor memory");
};

__device__ __forceinline__ uint64_t ddesc(uint32_t saddr, uint32_t sbo, uint32_t swz) {
  return sdesc(saddr, 16, sbo, swz);
}
__device__ __forceinline__ uint64_t ddesc_sf(uint32_t saddr) { return sdesc(saddr, 0, 128, kSwizzleNone); }
__device__ __forceinline__ uint64_t ddadd(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }
__device__ __forceinline__ void dcopy_sf(uint32_t tcol, uint64_t d0, uint32_t off, int nblk) {
  for (int i = 0; i < nblk; ++i) tmem_cp_32x128b_warpx4(tcol + 4 * i, ddadd(d0, off + 512 * i));
}

// One e2m1 code (low nibble) of v, round-to-nearest-even, saturating.
__device__ __forceinline__ uint32_t cvt_e2m1_one(float v) {
  uint16_t r;
  asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\tcvt.u16.u8 %0, b;\n\t}"
      : "=h"(r)
      : "f"(0.0f), "f"(v));
  return r & 0xFu;
}

struct DecArgs {
  const uint8_t* q_codes;
  const uint8_t* q_sf;
  const uint8_t* k_sf;
  const uint8_t* v_sf;
  void* out;
  SplitOut part;
  Strides so;
  long long rows;        // shares: B * H * Lqp, the padded query rows of one share's partial results
  long long items;       // ranges: pairs * key tiles
  int ranges;            // 0: key shares (nsplit per pair), 1: equal ranges of (pair, key tile) items
  int H, Hkv, Lq, Lkv, causal, nsplit, nr, ntk;
  uint64_t wait_ns;
};

// A CTA's work is a list of segments: key tiles [j0, j1) of one (batch, kv
// head) pair, and where the segment's result goes.
//   shares: one segment, share s = c % nsplit of pair c / nsplit; its result
//     is O itself (nsplit 1) or split-KV partial rows (splitkv.cu's layout);
//   ranges: the items [c * I / C, (c + 1) * I / C) of the (pair, key tile)
//     items laid end to end, cut into one segment per pair; a whole pair
//     writes O, a cut one its partial rows to slot 2c (the CTA's first
//     segment) or 2c + 1 (its last), 16 rows of d + 2 floats each, which
//     decode_combine_kernel merges.
struct DecSeg {
  int pair, j0, j1, slot;
  bool direct;
};
__device__ __forceinline__ long long range_start(const DecArgs& a, int c) { return (long long)c * a.items / gridDim.x; }
template <bool RANGES>
__device__ __forceinline__ int dec_nseg(const DecArgs& a, int c) {
  if constexpr (!RANGES) return 1;
  const long long i0 = range_start(a, c), i1 = range_start(a, c + 1);
  return i1 > i0 ? (int)((i1 - 1) / a.ntk - i0 / a.ntk + 1) : 0;
}
template <bool RANGES>
__device__ __forceinline__ DecSeg dec_seg(const DecArgs& a, int c, int k) {
  DecSeg sg;
  if constexpr (!RANGES) {
    const int share = c % a.nsplit;
    sg.pair = c / a.nsplit;
    sg.j0 = (int)((long long)share * a.ntk / a.nsplit);
    sg.j1 = (int)((long long)(share + 1) * a.ntk / a.nsplit);
    sg.slot = share;
    sg.direct = a.nsplit == 1;
    return sg;
  }
  const long long i0 = range_start(a, c), i1 = range_start(a, c + 1);
  const long long p0 = i0 / a.ntk, plast = (i1 - 1) / a.ntk;
  sg.pair = (int)(p0 + k);
  sg.j0 = k == 0 ? (int)(i0 % a.ntk) : 0;
  sg.j1 = sg.pair == plast ? (int)((i1 - 1) % a.ntk) + 1 : a.ntk;
  sg.direct = sg.j0 == 0 && sg.j1 == a.ntk;
  sg.slot = k == 0 ? 2 * c : 2 * c + 1;
  return sg;
}

// CTAs per SM: shared memory and tensor memory (128 columns) hold four; the
// registers of the 8- and 16-row kernels two
template <int NR>
constexpr int dec_ctas_per_sm() {
  return NR <= 4 ? 4 : 2;
}

template <int D, int NR, bool OUT32, bool RANGES>
__global__ void __launch_bounds__(kDecThreads, dec_ctas_per_sm<NR>())
    attn_decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                       const DecArgs a) {
  using C = CfgDec<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;                // [2] by segment parity
  uint64_t* q_empty = bars + 2;           // [2]: the segment's S^T MMAs are complete
  uint64_t* k_full = bars + 4;
  uint64_t* k_empty = k_full + C::NSK;
  uint64_t* v_full = k_empty + C::NSK;
  uint64_t* v_empty = v_full + C::NSV;
  uint64_t* s_full = v_empty + C::NSV;    // [2]
  uint64_t* s_free = s_full + 2;          // [2], 128 arrivals
  uint64_t* p_full = s_free + 2;          // [2], 128 arrivals
  uint64_t* o_done = p_full + 2;          // [2]: one phase per P.V into that accumulator
  uint64_t* red_full = o_done + 2;        // [2], 4 arrivals (the softmax warps' row maxima)
  uint64_t* sum_full = red_full + 2;      // 4 arrivals per segment (their row sums)
  uint64_t* drain = sum_full + 1;         // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(smem + C::kOffRed);   // [2][4][16] maxima, then [4][16] sums

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int Lqp = (a.Lq + 127) & ~127, Lkvp = (a.Lkv + 127) & ~127;
  const int G = a.H / a.Hkv;
  const int cta = blockIdx.x;
  const int nseg = dec_nseg<RANGES>(a, cta);
  const int nr = a.nr;                   // valid rows: r = g * Lq + t, query head kvh * G + g, token t
  // the segments' key tiles laid end to end: global tile g = gbase(k) + j
  // (barrier phases, stages and buffers count g over the whole list)
  int gtotal = 0;
  for (int k = 0; k < nseg; ++k) {
    const DecSeg sg = dec_seg<RANGES>(a, cta, k);
    gtotal += sg.j1 - sg.j0;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i) mbar_init(bars + i, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_free + i, 128);
      mbar_init(p_full + i, 128);
      mbar_init(red_full + i, 4);
    }
    mbar_init(sum_full, 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // scale blocks of Q and P^T: rows the segments do not use must hold finite
  // scales (zero)
  for (int i = threadIdx.x; i < (2 * C::kQSfBytes + 2 * C::kPSfBytes) / 16; i += kDecThreads) {
    uint8_t* p = i < 2 * C::kQSfBytes / 16 ? smem + C::kOffQSf + 16 * i
                                           : smem + C::kOffPSf + 16 * (i - 2 * C::kQSfBytes / 16);
    *reinterpret_cast<uint4*>(p) = make_uint4(0u, 0u, 0u, 0u);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Per segment: its query rows into Q buffer k & 1 (once the S^T MMAs of
    // segment k - 2 are complete), then its K and V tiles: K(g) and V(g - 1)
    // per step, K, which the S^T MMAs release a tile before the P.V MMAs
    // release V, running one tile further ahead.
    const bool leader = elect_one();
    if (leader) {
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
    }
    pdl_wait();                                          // the codes are written (programmatic launch)
    int nk = 0, nv = 0, nq = 0;
    int kseg = 0, jseg = 0;                              // the segment and local tile of K step g
    DecSeg sg = nseg > 0 ? dec_seg<RANGES>(a, cta, 0) : DecSeg{0, 0, 0, 0, true};
    int vseg = 0, vj = 0;                                // the segment and local tile of V step g - 1
    DecSeg vsg = sg;
    for (int g = 0; ok && g <= gtotal; ++g) {
      if (g < gtotal) {
        while (jseg >= sg.j1 - sg.j0) {                  // (segments have at least one tile)
          ++kseg;
          jseg = 0;
          sg = dec_seg<RANGES>(a, cta, kseg);
        }
        if (jseg == 0) {
          // Q^T of segment kseg: rows r < nr gathered from their heads' rows
          // (16-byte chunks, the swizzle of the K-major operand: 64-byte rows
          // chunk c at c ^ ((r >> 1) & 3), 32-byte rows chunk c at
          // c ^ ((r >> 2) & 1)); rows >= nr zero
          const int qb = kseg & 1;
          if (kseg >= 2) ok = mbar_wait_backoff_warp(q_empty + qb, ((kseg >> 1) - 1) & 1, abort_flag, a.wait_ns, 128);
          if (!ok) break;
          const int b = sg.pair / a.Hkv, kvh = sg.pair % a.Hkv;
          constexpr int kCpr = C::kRowBytes / 16;        // chunks per row
          for (int id = lane; id < kNR * kCpr; id += 32) {
            const int r = id / kCpr, c = id % kCpr;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r < nr) {
              const int gq = r / a.Lq, t = r % a.Lq;
              const long long bhq = (long long)b * a.H + (long long)kvh * G + gq;
              v = __ldg(reinterpret_cast<const uint4*>(a.q_codes + (bhq * Lqp + t) * C::kRowBytes) + c);
            }
            const int phase = D == 128 ? ((r >> 1) & 3) : ((r >> 2) & 1);
            *reinterpret_cast<uint4*>(smem + C::kOffQ + qb * 1024 + r * C::kRowBytes + ((c ^ phase) << 4)) = v;
          }
          // Q scales: row r's four group scales of 64-channel block kc at
          // byte r * 16 of block kc (rows < 32 of a 512-byte block)
          for (int id = lane; id < nr * (D / 64); id += 32) {
            const int r = id / (D / 64), kc = id % (D / 64);
            const int gq = r / a.Lq, t = r % a.Lq;
            const long long bhq = (long long)b * a.H + (long long)kvh * G + gq;
            const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(
                a.q_sf + ((bhq * (Lqp / 128) + t / 128) * (D / 64) + kc) * 512 + (t % 32) * 16 + (t / 32) * 4));
            *reinterpret_cast<uint32_t*>(smem + C::kOffQSf + qb * C::kQSfBytes + kc * 512 + r * 16) = w;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (leader) mbar_arrive(q_full + qb);
          ++nq;
        }
        const int s = g % C::NSK, ja = sg.j0 + jseg;
        const long long bhk = sg.pair;
        if (g >= C::NSK) ok = mbar_wait_backoff_warp(k_empty + s, ((g / C::NSK) - 1) & 1, abort_flag, a.wait_ns, 128);
        if (!ok) break;
        if (leader) {
          mbar_arrive_expect_tx(k_full + s, C::kKBytes + C::kKSfBytes);
          tma_load_2d(smem + C::kOffK + s * C::kKBytes, &tmap_k, k_full + s, 0,
                      (int)(bhk * Lkvp + (long long)ja * kKeys));
          bulk_load(smem + C::kOffKSf + s * C::kKSfBytes, a.k_sf + (bhk * (Lkvp / 128) + ja) * C::kKSfBytes,
                    C::kKSfBytes, k_full + s);
        }
        __syncwarp();
        ++nk;
        ++jseg;
      }
      if (g >= 1) {
        const int gv = g - 1, s = gv % C::NSV;
        while (vj >= vsg.j1 - vsg.j0) {
          ++vseg;
          vj = 0;
          vsg = dec_seg<RANGES>(a, cta, vseg);
        }
        const int ja = vsg.j0 + vj;
        const long long bhk = vsg.pair;
        if (gv >= C::NSV) ok = mbar_wait_backoff_warp(v_empty + s, ((gv / C::NSV) - 1) & 1, abort_flag, a.wait_ns, 128);
        if (!ok) break;
        if (leader) {
          mbar_arrive_expect_tx(v_full + s, C::kVLoadBytes + C::kVSfBytes);
          tma_load_2d(smem + C::kOffV + s * C::kVBytes, &tmap_v, v_full + s, ja * (kKeys / 2), (int)(bhk * D));
          bulk_load(smem + C::kOffVSf + s * C::kVSfBytes, a.v_sf + (bhk * (Lkvp / 64) + 2 * ja) * 512, C::kVSfBytes,
                    v_full + s);
        }
        __syncwarp();
        ++nv;
        ++vj;
      }
    }
    if (*abort_flag) {
      // let every copy already issued land before the CTA goes away (the
      // query rows are plain stores, complete already)
      for (int g = (nk > C::NSK ? nk - C::NSK : 0); g < nk; ++g)
        mbar_wait_drain(k_full + g % C::NSK, (g / C::NSK) & 1, a.wait_ns);
      for (int g = (nv > C::NSV ? nv - C::NSV : 0); g < nv; ++g)
        mbar_wait_drain(v_full + g % C::NSV, (g / C::NSV) & 1, a.wait_ns);
    }
    (void)nq;
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // S^T(0), S^T(1), P.V(0), S^T(2), P.V(1), ... over the global tiles:
    // S^T one tile ahead in the other S^T buffer.  S^T(g) reuses buffer g & 1
    // once the softmax has read S^T(g - 2); K scales of tile g go to the
    // columns of its parity, last read by S^T(g - 2) (whose commit is that
    // stage's k_empty phase); V and P^T scales likewise, last read by
    // P.V(g - 2), which the softmax warps have seen complete before they
    // release P^T(g).  A segment's Q scales go to the columns of its parity
    // once the S^T MMAs of segment k - 2 are complete (its q_empty phase);
    // P.V(g) accumulates into O^T buffer g & 1, fresh for the first two tiles
    // of a segment.
    const bool leader = elect_one();
    const uint32_t sb = smem_u32(smem);
    const uint64_t dQ0 = ddesc(sb + C::kOffQ, C::kQKSbo, C::kQKSwz);
    const uint64_t dK0 = ddesc(sb + C::kOffK, C::kQKSbo, C::kQKSwz);
    const uint64_t dV0 = ddesc(sb + C::kOffV, 512, kSwizzle64B);
    const uint64_t dP0 = ddesc(sb + C::kOffP, 512, kSwizzle64B);
    const uint64_t dSf0 = ddesc_sf(sb);
    int kseg = -1, jseg = 0, nseg_tiles = 0;            // S side: segment, local tile, its tile count
    int pseg_j = 0, pseg_n = 0, pk = -1;                 // P.V side
    for (int g = 0; ok && g <= gtotal; ++g) {
      if (g < gtotal) {
        if (jseg >= nseg_tiles) {
          ++kseg;
          jseg = 0;
          const DecSeg sg = dec_seg<RANGES>(a, cta, kseg);
          nseg_tiles = sg.j1 - sg.j0;
          const int qb = kseg & 1;
          ok = mbar_wait_warp(q_full + qb, (kseg >> 1) & 1, abort_flag, a.wait_ns);
          if (ok && kseg >= 2) ok = mbar_wait_warp(q_empty + qb, ((kseg >> 1) - 1) & 1, abort_flag, a.wait_ns);
          if (!ok) break;
          tc_fence_after();
          if (leader) dcopy_sf(tbase + C::kColSfQ + 8 * qb, dSf0, C::kOffQSf + qb * C::kQSfBytes, D / 64);
          __syncwarp();
        }
        const int s = g % C::NSK, qb = kseg & 1;
        ok = mbar_wait_warp(k_full + s, (g / C::NSK) & 1, abort_flag, a.wait_ns);
        if (ok && g >= 2)
          ok = mbar_wait_warp(k_empty + (g - 2) % C::NSK, ((g - 2) / C::NSK) & 1, abort_flag, a.wait_ns) &&
               mbar_wait_warp(s_free + (g & 1), ((g >> 1) - 1) & 1, abort_flag, a.wait_ns);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sfk = tbase + C::kColSfK + 8 * (g & 1);
        if (leader) {
          dcopy_sf(sfk, dSf0, C::kOffKSf + s * C::kKSfBytes, D / 64);
#pragma unroll
          for (int kk = 0; kk < D / 64; ++kk)
            mma_nvf4(tbase + C::kColS + 16 * (g & 1), ddadd(dK0, s * C::kKBytes + kk * 32),
                     ddadd(dQ0, qb * 1024 + kk * 32), C::kIdesc, sfk + 4 * kk, tbase + C::kColSfQ + 8 * qb + 4 * kk,
                     kk > 0 ? 1u : 0u);
          tc_commit(s_full + (g & 1));
          tc_commit(k_empty + s);
          if (jseg + 1 == nseg_tiles) tc_commit(q_empty + qb);   // the segment's last S^T
        }
        __syncwarp();
        ++jseg;
      }
      if (g >= 1) {
        const int gv = g - 1, s = gv % C::NSV;
        if (pseg_j >= pseg_n) {
          ++pk;
          pseg_j = 0;
          const DecSeg sg = dec_seg<RANGES>(a, cta, pk);
          pseg_n = sg.j1 - sg.j0;
        }
        ok = mbar_wait_warp(v_full + s, (gv / C::NSV) & 1, abort_flag, a.wait_ns) &&
             mbar_wait_warp(p_full + (gv & 1), (gv >> 1) & 1, abort_flag, a.wait_ns);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sfv = tbase + C::kColSfV + 8 * (gv & 1), sfp = tbase + C::kColSfP + 8 * (gv & 1);
        if (leader) {
          dcopy_sf(sfv, dSf0, C::kOffVSf + s * C::kVSfBytes, 2);
          dcopy_sf(sfp, dSf0, C::kOffPSf + (gv & 1) * C::kPSfBytes, 2);
#pragma unroll
          for (int kk = 0; kk < kKeys / 64; ++kk)
            mma_nvf4(tbase + C::kColO + 16 * (gv & 1), ddadd(dV0, s * C::kVBytes + kk * 32),
                     ddadd(dP0, (gv & 1) * C::kPBytes + kk * 32), C::kIdesc, sfv + 4 * kk, sfp + 4 * kk,
                     (pseg_j > 1 || kk > 0) ? 1u : 0u);
          tc_commit(o_done + (gv & 1));
          tc_commit(v_empty + s);
        }
        __syncwarp();
        ++pseg_j;
      }
    }
    if (!ok) {
      if (leader) tc_commit(drain);
      __syncwarp();
      mbar_wait_drain(drain, 0, a.wait_ns);
    }
  } else {
    // ------------------------------------------------------------- softmax
    // Two O^T accumulators, tile g into buffer g & 1, each in units of its own
    // reference (the latest live tile maximum accumulated into it; the P.V of
    // tile g - 1 may still run while tile g's P^T is formed), merged at the
    // end of a segment: O = sum_X O_X 2^(m_X - M), l = sum_X l_X 2^(m_X - M),
    // M = max_X m_X.  (The per-accumulator state is picked with selects, not
    // indexed by the tile parity, so that it stays in registers.)
    const int wq = warp % 4;                             // lane quarter of S^T / O^T
    const int k = wq * 32 + lane;                        // key of the tile (S^T lane), channel of O^T
    const uint32_t lane_addr = tbase + ((wq * 32) << 16);
    const float c = softmax_scale_log2<D>();
    // row r may see keys below lim[r]: Lkv, or under the causal mask
    // t + Lkv - Lq + 1 (t = r % Lq); rows >= nr none
    int lim[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) lim[r] = r >= nr ? 0 : (a.causal ? r % a.Lq + a.Lkv - a.Lq + 1 : a.Lkv);
    int g = 0;                                           // global tile
    for (int kseg = 0; ok && kseg < nseg; ++kseg) {
      const DecSeg sg = dec_seg<RANGES>(a, cta, kseg);
      const int nt = sg.j1 - sg.j0;
      float m_run[NR], m_ref0[NR], m_ref1[NR], lam0[NR], lam1[NR];
      uint32_t href0 = 0u, href1 = 0u;                   // bit r: row r has had a live tile in that accumulator
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        m_run[r] = -INFINITY;
        m_ref0[r] = m_ref1[r] = 0.f;
        lam0[r] = lam1[r] = 0.f;
      }
      for (int j = 0; ok && j < nt; ++j, ++g) {
        const int sb = g & 1, ja = sg.j0 + j;
        ok = mbar_wait_warp(s_full + sb, (g >> 1) & 1, abort_flag, a.wait_ns);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[16];
        tmem_ld16(lane_addr + C::kColS + 16 * sb, sr);
        tmem_ld_wait(sr);
        tc_fence_before();
        mbar_arrive(s_free + sb);
        // keys this row may not see: past Lkv and, causal, past t + Lkv - Lq
        const int kpos = ja * kKeys + k;
        float x[NR], gm[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          x[r] = kpos < lim[r] ? __uint_as_float(sr[r]) : -INFINITY;
          gm[r] = x[r];
        }
        // the 1x16 groups of keys are 16 consecutive lanes: their maxima
        // first, then one more step for the warp's, then the four warps'
#pragma unroll
        for (int o = 1; o < 16; o <<= 1)
#pragma unroll
          for (int r = 0; r < NR; ++r) gm[r] = fmaxf(gm[r], __shfl_xor_sync(0xffffffffu, gm[r], o));
        float* rm = red + sb * 64;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const float wm = fmaxf(gm[r], __shfl_xor_sync(0xffffffffu, gm[r], 16));
          if (lane == 0) rm[wq * 16 + r] = wm;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(red_full + sb);
        ok = mbar_wait_warp(red_full + sb, (g >> 1) & 1, abort_flag, a.wait_ns);
        if (!ok) break;
        uint32_t nib[2] = {0u, 0u}, s8v[NR];
        float corr[NR];
        bool any_corr = false;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const float mx = fmaxf(fmaxf(rm[r], rm[16 + r]), fmaxf(rm[32 + r], rm[48 + r]));
          const float m_t = mx * c;
          const float m_new = fmaxf(m_run[r], m_t);
          const bool live = (m_t > -INFINITY) && (m_t >= m_new - kSkipBelowDec);
          m_run[r] = m_new;
          const bool hr = ((sb ? href1 : href0) >> r) & 1u;
          corr[r] = (live && hr) ? ex2_approx((sb ? m_ref1[r] : m_ref0[r]) - m_t) : 1.f;
          any_corr |= corr[r] != 1.f;
          const float bias = live ? kLog2PRangeDec - m_t : -INFINITY;
          const float sa = ex2_approx(fmaf(gm[r], c, bias)) * (1.0f / 6.0f);
          s8v[r] = cvt_e4m3x2(sa, 0.f) & 0xFFu;
          float fg = e4m3_to_f32(s8v[r]);
          fg = fg == 0.f ? 1.f : fg;
          const float bg = bias - lg2_approx(fg);
          const float p = ex2_approx(fmaf(x[r], c, bg));
          nib[r >> 3] |= cvt_e2m1_one(p) << (4 * (r & 7));
          // a live tile: the accumulator's row sum rescaled and extended, its
          // reference moved to this tile (selects, no branches, so that the
          // rows' chains interleave)
          const float lnew = fmaf(hr ? (sb ? lam1[r] : lam0[r]) : 0.f, corr[r], p * fg);
          const bool up0 = live && !sb, up1 = live && sb;
          lam0[r] = up0 ? lnew : lam0[r];
          lam1[r] = up1 ? lnew : lam1[r];
          m_ref0[r] = up0 ? m_t : m_ref0[r];
          m_ref1[r] = up1 ? m_t : m_ref1[r];
          href0 |= (up0 ? 1u : 0u) << r;
          href1 |= (up1 ? 1u : 0u) << r;
        }
        // P^T and its scales go to buffer sb, last read by P.V(g - 2): wait
        // for it (its accumulator is rescaled below as well)
        if (g >= 2) {
          ok = mbar_wait_warp(o_done + sb, ((g >> 1) - 1) & 1, abort_flag, a.wait_ns);
          if (!ok) break;
          tc_fence_after();
        }
        // P^T row r, byte k / 2 (even key in the low nibble), 64B-swizzled:
        // 16-byte chunk c of row r at c ^ ((r >> 1) & 3)
        uint8_t* pt = smem + C::kOffP + sb * C::kPBytes;
        const uint32_t o0 = __shfl_xor_sync(0xffffffffu, nib[0], 1);
        const uint32_t o1 = NR > 8 ? __shfl_xor_sync(0xffffffffu, nib[1], 1) : 0u;
        if ((k & 1) == 0) {
          const int byte = k >> 1;
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            const uint32_t lo = (nib[r >> 3] >> (4 * (r & 7))) & 0xFu;
            const uint32_t hi = (((r >> 3) ? o1 : o0) >> (4 * (r & 7))) & 0xFu;
            pt[r * 64 + ((((byte >> 4) ^ ((r >> 1) & 3)) << 4) | (byte & 15))] = (uint8_t)(lo | (hi << 4));
          }
        }
        if ((k & 15) == 0) {
          uint8_t* psf = smem + C::kOffPSf + sb * C::kPSfBytes + (k / 64) * 512 + ((k / 16) & 3);
#pragma unroll
          for (int r = 0; r < NR; ++r) psf[r * 16] = (uint8_t)s8v[r];
        }
        fence_proxy_async_smem();
        if (j >= 2 && any_corr) {                        // (uniform: every thread has the same rows)
          const uint32_t tO = lane_addr + C::kColO + 16 * sb;
          uint32_t o[16];
          tmem_ld16(tO, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int r = 0; r < NR; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * corr[r]);
          tmem_st16(tO, o);
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(p_full + sb);
      }
      if (!ok) break;
      // the segment's last P.V into each accumulator
      const int gl = g - 1;
      ok = mbar_wait_warp(o_done + (gl & 1), (gl >> 1) & 1, abort_flag, a.wait_ns);
      if (ok && nt > 1) ok = mbar_wait_warp(o_done + ((gl - 1) & 1), ((gl - 1) >> 1) & 1, abort_flag, a.wait_ns);
      if (!ok) break;
      // per row: the merged reference M and the weights of the two accumulators
      float w0[NR], w1[NR], mm[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const bool h0 = (href0 >> r) & 1u, h1 = (href1 >> r) & 1u;
        mm[r] = fmaxf(h0 ? m_ref0[r] : -INFINITY, h1 ? m_ref1[r] : -INFINITY);
        w0[r] = h0 ? ex2_approx(m_ref0[r] - mm[r]) : 0.f;
        w1[r] = h1 ? ex2_approx(m_ref1[r] - mm[r]) : 0.f;
      }
      // the row sums: per key so far, now over the tile's 128 keys
      float* rs = red + 128;
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        float v = fmaf(lam0[r], w0[r], lam1[r] * w1[r]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) rs[wq * 16 + r] = v;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(sum_full);
      ok = mbar_wait_warp(sum_full, kseg & 1, abort_flag, a.wait_ns);
      if (!ok) break;
      tc_fence_after();
      uint32_t oa[16], ob[16];
      tmem_ld16(lane_addr + C::kColO, oa);
      tmem_ld16(lane_addr + C::kColO + 16, ob);
      tmem_ld_wait(oa);
      tmem_launder(ob);
      if (k < D) {
        const int b = sg.pair / a.Hkv, kvh = sg.pair % a.Hkv;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          if (r >= nr) break;
          const float l = (rs[r] + rs[16 + r]) + (rs[32 + r] + rs[48 + r]);
          // an accumulator without a live tile holds no P.V of this segment
          const float ov = fmaf(w0[r] != 0.f ? __uint_as_float(oa[r]) : 0.f, w0[r],
                                (w1[r] != 0.f ? __uint_as_float(ob[r]) : 0.f) * w1[r]);
          const int gq = r / a.Lq, t = r % a.Lq;
          const long long bhq = (long long)b * a.H + (long long)kvh * G + gq;
          if (sg.direct) {
            const float v = ov * (1.f / l);
            const long long off =
                (long long)b * a.so.b + ((long long)kvh * G + gq) * a.so.h + (long long)t * a.so.t + k;
            if constexpr (OUT32)
              static_cast<float*>(a.out)[off] = v;
            else
              static_cast<__nv_bfloat16*>(a.out)[off] = __float2bfloat16_rn(v);
          } else {
            // shares: share `slot` of padded row (b * H + h) * Lqp + t;
            // ranges: row r of slot `slot`
            const long long R = RANGES ? (long long)sg.slot * kNR + r : (long long)sg.slot * a.rows + bhq * Lqp + t;
            a.part.o[R * D + k] = ov;
            if (k == 0) *reinterpret_cast<float2*>(a.part.ml + 2 * R) = make_float2(mm[r], l);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // every output of this CTA is stored: a combine launch queued behind this
  // one (programmatic dependent launch) may be scheduled
  pdl_launch_dependents();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
  }
}

// Ranges: O of every pair that the ranges cut, from its segments' partial
// rows (slot 2c when the pair is CTA c's first segment, else 2c + 1), merged
// in CTA order: M = max m_c, O = sum_c 2^(m_c - M) a_c / sum_c 2^(m_c - M) l_c.
// One CTA per pair, one warp per row (rows w, w + 4, ...), lane i holding
// channels [i V, i V + V); the loads of up to eight segments are issued
// before any is used.
template <int D, bool OUT32>
__global__ void __launch_bounds__(128)
    decode_combine_kernel(const SplitOut part, long long items, int ctas, int ntk, int nr, int H, int Hkv, int Lq,
                          const Strides so, void* __restrict__ out) {
  constexpr int V = D / 32, kBatch = 8;
  pdl_wait();                                            // the partial rows are written
  const int p = blockIdx.x, warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  auto cta_of = [&](long long i) { return (int)(((i + 1) * ctas + items - 1) / items) - 1; };
  const int c_lo = cta_of((long long)p * ntk), c_hi = cta_of((long long)(p + 1) * ntk - 1);
  if (c_lo == c_hi) return;                              // a whole pair: its CTA wrote O
  const int nseg = c_hi - c_lo + 1;
  auto row_of = [&](int i, int r) {
    const int cc = c_lo + i;
    const int slot = ((long long)cc * items / ctas) / ntk == p ? 2 * cc : 2 * cc + 1;
    return (long long)slot * kNR + r;
  };
  const int G = H / Hkv, b = p / Hkv, kvh = p % Hkv;
  for (int r = warp; r < nr; r += 4) {
    float mmax = -INFINITY;
    for (int s0 = 0; s0 < nseg; s0 += kBatch) {
      float2 ml[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        ml[i] = s0 + i < nseg ? *reinterpret_cast<const float2*>(part.ml + 2 * row_of(s0 + i, r))
                              : make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        if (ml[i].y > 0.f) mmax = fmaxf(mmax, ml[i].x);
    }
    float lsum = 0.f, acc[V];
#pragma unroll
    for (int c = 0; c < V; ++c) acc[c] = 0.f;
    for (int s0 = 0; s0 < nseg; s0 += kBatch) {
      float2 ml[kBatch];
      float ov[kBatch][V];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        ml[i] = make_float2(-INFINITY, 0.f);
        if (s0 + i < nseg) {
          const long long R = row_of(s0 + i, r);
          ml[i] = *reinterpret_cast<const float2*>(part.ml + 2 * R);
#pragma unroll
          for (int c = 0; c < V; ++c) ov[i][c] = part.o[R * D + lane * V + c];
        }
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        if (!(ml[i].y > 0.f)) continue;                  // no segment, or no visible key for this row
        const float w = exp2f(ml[i].x - mmax);
        lsum = fmaf(w, ml[i].y, lsum);
#pragma unroll
        for (int c = 0; c < V; ++c) acc[c] = fmaf(w, ov[i][c], acc[c]);
      }
    }
    const float inv = 1.f / lsum;
    const int gq = r / Lq, t = r % Lq;
    const long long off = (long long)b * so.b + ((long long)kvh * G + gq) * so.h + (long long)t * so.t + lane * V;
#pragma unroll
    for (int c = 0; c < V; ++c) {
      if constexpr (OUT32)
        static_cast<float*>(out)[off + c] = acc[c] * inv;
      else
        static_cast<__nv_bfloat16*>(out)[off + c] = __float2bfloat16_rn(acc[c] * inv);
    }
  }
}

template <int D, int NR, bool OUT32>
cudaError_t launch_dec(const CUtensorMap& tk, const CUtensorMap& tv, const sa_fp4_qkv& x, void* o,
                       const Strides& so, const Dims& dm, int causal, int nsplit, const SplitOut& part,
                       cudaStream_t s) {
  using C = CfgDec<D>;
  static std::atomic<bool> attr_done[kMaxDevices];   // kernel attributes are per device
  cudaError_t e = once_per_device(attr_done, [] {
    cudaError_t r = cudaFuncSetAttribute(attn_decode_kernel<D, NR, OUT32, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(attn_decode_kernel<D, NR, OUT32, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  DecArgs a;
  a.q_codes = static_cast<const uint8_t*>(x.q_codes);
  a.q_sf = static_cast<const uint8_t*>(x.q_sf);
  a.k_sf = static_cast<const uint8_t*>(x.k_sf);
  a.v_sf = static_cast<const uint8_t*>(x.v_sf);
  a.out = o;
  a.part = part;
  a.so = so;
  a.H = dm.H;
  a.Hkv = dm.Hkv;
  a.Lq = dm.Lq;
  a.Lkv = dm.Lkv;
  a.causal = causal;
  a.nr = (dm.H / dm.Hkv) * dm.Lq;
  a.ntk = (dm.Lkv + kKeys - 1) / kKeys;
  a.rows = (long long)dm.B * dm.H * padded_len(dm.Lq);
  a.ranges = nsplit == kStreamK;
  a.nsplit = a.ranges ? 1 : nsplit;
  a.items = (long long)dm.B * dm.Hkv * a.ntk;
  a.wait_ns = kWaitLimitNs;
  const int ctas = a.ranges ? decode_range_ctas(dm, device_sm_count()) : dm.B * dm.Hkv * nsplit;
  // a programmatic dependent launch: the CTAs' set-up overlaps the end of
  // the kernel before; the producer waits for it before its first load
  cudaLaunchAttribute attr;
  const cudaLaunchConfig_t cfg = pdl_launch_config(dim3(ctas), dim3(kDecThreads), C::kSmemBytes, s, &attr);
  // (the shares' instantiation has the one-segment list folded in)
  e = a.ranges ? cudaLaunchKernelEx(&cfg, attn_decode_kernel<D, NR, OUT32, true>, tk, tv, a)
               : cudaLaunchKernelEx(&cfg, attn_decode_kernel<D, NR, OUT32, false>, tk, tv, a);
  if (e != cudaSuccess) return e;
  if (a.ranges) {
    cudaLaunchAttribute attr2;
    const cudaLaunchConfig_t cfg2 = pdl_launch_config(dim3(dm.B * dm.Hkv), dim3(128), 0, s, &attr2);
    e = cudaLaunchKernelEx(&cfg2, decode_combine_kernel<D, OUT32>, part, a.items, ctas, a.ntk, a.nr, dm.H, dm.Hkv,
                           dm.Lq, so, o);
  } else if (nsplit > 1) {
    e = launch_splitkv_combine(part, nsplit, dm, o, so, OUT32, s);
  }
  return e;
}

// The kernel for the rows of a kv head: 4, 8 or 16 (the smallest that holds them).
template <int D, bool OUT32>
cudaError_t launch_dec_rows(const CUtensorMap& tk, const CUtensorMap& tv, const sa_fp4_qkv& x, void* o,
                            const Strides& so, const Dims& dm, int causal, int nsplit, const SplitOut& part,
                            cudaStream_t s) {
  const int nr = (dm.H / dm.Hkv) * dm.Lq;
  if (nr <= 4) return launch_dec<D, 4, OUT32>(tk, tv, x, o, so, dm, causal, nsplit, part, s);
  if (nr <= 8) return launch_dec<D, 8, OUT32>(tk, tv, x, o, so, dm, causal, nsplit, part, s);
  return launch_dec<D, 16, OUT32>(tk, tv, x, o, so, dm, causal, nsplit, part, s);
}

}  // namespace

bool decode_eligible(const Dims& dm) { return (long long)(dm.H / dm.Hkv) * dm.Lq <= kNR; }

int decode_range_ctas(const Dims& dm, int sms) {
  const long long items = (long long)dm.B * dm.Hkv * ((dm.Lkv + kKeys - 1) / kKeys);
  const int nr = (dm.H / dm.Hkv) * dm.Lq;
  const long long slots = (long long)(sms > 0 ? sms : 1) * (nr <= 4 ? 3 : dec_ctas_per_sm<16>());
  return (int)(items < slots ? items : slots);
}

size_t decode_range_workspace_bytes(const Dims& dm, int sms) {
  return (size_t)2 * decode_range_ctas(dm, sms) * kNR * ((size_t)dm.d + 2) * sizeof(float);
}

SplitOut decode_range_layout(void* ws, const Dims& dm, int sms) {
  float* f = static_cast<float*>(ws);
  return SplitOut{f, f + (size_t)2 * decode_range_ctas(dm, sms) * kNR * dm.d};
}

int decode_nsplit(const Dims& dm, int sms) {
  // as many key shares as let the (batch, kv head) pairs fill one wave of
  // resident CTAs (no partial second wave), at least one, at most one per
  // key tile
  const int ntk = (dm.Lkv + kKeys - 1) / kKeys;
  const long long pairs = (long long)dm.B * dm.Hkv;
  const int nr = (dm.H / dm.Hkv) * dm.Lq;
  const long long slots = (long long)(sms > 0 ? sms : 1) * (nr <= 4 ? dec_ctas_per_sm<4>() : dec_ctas_per_sm<16>());
  long long n = slots / pairs;
  if (n < 1) n = 1;
  if (n > ntk) n = ntk;
  return (int)n;
}

cudaError_t launch_attn_decode(const CUtensorMap& tk, const CUtensorMap& tv, const sa_fp4_qkv& x, void* o,
                               const Strides& so, const Dims& dm, int causal, bool out_f32, int nsplit,
                               const SplitOut& part, cudaStream_t s) {
  if (dm.d == 64)
    return out_f32 ? launch_dec_rows<64, true>(tk, tv, x, o, so, dm, causal, nsplit, part, s)
                   : launch_dec_rows<64, false>(tk, tv, x, o, so, dm, causal, nsplit, part, s);
  return out_f32 ? launch_dec_rows<128, true>(tk, tv, x, o, so, dm, causal, nsplit, part, s)
                 : launch_dec_rows<128, false>(tk, tv, x, o, so, dm, causal, nsplit, part, s);
}

}  // namespace sa
