// attn_nvfp4.cu -- SageAttention3-style fused attention forward with NVFP4
// operands on tcgen05 block-scaled tensor cores.
//
// Method (page "GPU kernel porting with AI agents", section "Sage Attention
// 3"): Q, K' (smooth-K applied) and V are e2m1 in 1x16 groups with e4m3
// scales (produced by sa_quantize); S = Q^ K^'^T is one block-scaled FP4 MMA
// per 64 of d; P is quantised in two levels inside the kernel -- per row and
// 128-key tile it is rescaled so that its maximum is 448 x 6 = 2688, then
// microscaled to e2m1 in 1x16 groups along the keys with e4m3 scales -- and
// O += P^ V^ is a second block-scaled FP4 MMA.  Online softmax tile by tile
// (page "FlashAttention kernels", sections 0-1).
//
// Per row and tile j with tile maximum m_j (base-2 logits x = S*log2(e)/sqrt(d)):
//   P2   = 2^(x - m_j) * 2688                 (first level; max exactly 2688)
//   P^   = e2m1(P2 / s2) * s2, s2 = e4m3(max16(P2) / 6)   (second level)
//   A_j  = A_{j-1} * 2^(m_{j-1} - m_j) + P^ V^      (tensor memory, FP32)
//   lam_j = lam_{j-1} * 2^(m_{j-1} - m_j) + sum(P2)
// and O = A / lam: the first-level factor s1 = 2^(m_j - m_run)/2688 and the
// running-max factor cancel between A and lam, so the accumulator is kept in
// units of the latest tile's maximum.  A tile whose maximum lies more than
// 2^64 below the running maximum contributes below float32 resolution and is
// skipped for that row (its P^ row is zero).
//
// Arithmetic per element: the group maximum of P2 is 2^(max16(x) - m_j) * 2688
// (2^x is increasing), and the division by the group scale is folded into
// the exponent, P2 / s2 = 2^(x*c + b - log2 s2); so one FMA and one exp2 give
// the value to encode, and sum(P2) = sum over groups of s2 * sum(P2/s2).
//
// CTA layout (384 threads): warps 0-3 / 4-7 own query tiles 0 / 1 (one thread
// per row: softmax, P quantisation, O correction, epilogue); warp 8 issues TMA
// and bulk copies; warp 9 issues the S MMAs and warp 10 the P.V MMAs, each
// with the scale-factor copies they need (the three warps run their loops with
// all lanes and issue from one elected lane); warp 11 idles (fused Q: it
// stages bf16 Q).  Tensor memory: S
// (128 columns, shared by both query tiles), O0, O1 (d columns each), then
// scale factors (4 columns per 64-deep K chunk, copied from SMEM with
// tcgen05.cp, replicated to the four lane quarters).
//
// A CTA works through a list of units (work.cuh): one entry of the work list,
// or, persistent under stream-K, a range of (pair, key tile) items that spans
// several pairs.  Every role walks the same list and counts its barrier
// phases, stages and buffers over the whole list, so the next unit's Q and
// first K/V tiles load, and its first S is computed, while the softmax warps
// finish the current one.  Q and its scales are double-buffered by unit
// parity.
//
// Smooth-Q variant (SQ; page "kernel overview", evolution chain "Smooth-K ->
// Smooth-Q+K"): Q' = Q - (its 128-row tile's mean) was quantised instead of
// Q, and each score gets the tile mean's share back before the softmax:
// S = Q^' K^'^T + dS[query tile][key], dS from smooth_q.cu.  The softmax
// warpgroup of a query tile stages its 512-byte dS row of each key tile in
// shared memory (a bulk copy issued by its thread 0 one tile ahead, three
// buffers) and adds it to the scores; the rest is unchanged.
//
// Fused-Q variant (FQ): the kernel reads bf16 Q and quantises it itself, with
// the arithmetic of sa_quantize (quant_group.cuh), so the result is the same
// bytes and the same O.  Warp 11 copies a unit's bf16 Q tiles by TMA into a
// staging area (64-channel x 128-token boxes, 128B swizzle) once the previous
// unit's were quantised; each softmax thread quantises its own row of its
// query tile into the Q buffer of the unit's parity: the next unit's at the
// start of each unit (the first unit's own as well), so that it is ready as early as
// a loaded Q would be.  Q's full barriers then count the eight softmax warps.

#include <cuda_bf16.h>

#include "internal.h"
#include "quant_group.cuh"
#include "sm100.cuh"
#include "work.cuh"

namespace sa {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kThreads = 384;
constexpr uint32_t kProducerSleepNs = 256;   // poll interval of the TMA producer's waits
constexpr uint32_t kStageSleepNs = 512;      // poll interval of the fused-Q staging warp's waits
constexpr int kSoftmaxRegs = 200;   // 8 softmax warps
constexpr int kOtherRegs = 96;      // producer / MMA warpgroup
constexpr int kLaunchRegs = 168;    // 65536 / 384 rounded down to a multiple of 8
static_assert(8 * 32 * kSoftmaxRegs + 4 * 32 * kOtherRegs <= kThreads * kLaunchRegs, "register split");
// smooth-Q: the softmax warps also stage and add the score corrections
// (measured on llm_prefill: 296 -> 280 us with 8 more registers each)
constexpr int kSoftmaxRegsSq = 208, kOtherRegsSq = 80;
static_assert(8 * 32 * kSoftmaxRegsSq + 4 * 32 * kOtherRegsSq <= kThreads * kLaunchRegs, "register split");
constexpr float kLog2PRange = 11.392317422778761f;   // log2(448 * 6)
constexpr float kSkipBelow = 64.0f;                   // log2 units

template <int D>
struct CfgF4 {
  static constexpr int NS = 4;
  static constexpr int kRowBytes = D / 2;                  // packed codes per Q/K row
  static constexpr int kQBytes = BM * kRowBytes;           // one Q tile of codes
  static constexpr int kQSfBytes = (D / 64) * 512;         // its scale blocks
  static constexpr int kKBytes = BN * kRowBytes;
  static constexpr int kKSfBytes = (D / 64) * 512;
  static constexpr int kVBytes = D * (BN / 2);             // V^T tile: d rows x 64 bytes
  static constexpr int kVSfBytes = 2 * 512;                // two 64-token chunks
  static constexpr int kPBytes = BM * (BN / 2);            // P^ tile: 128 rows x 64 bytes
  static constexpr int kPSfBytes = 2 * 512;
  static constexpr int kOffQ = 0;                          // [unit parity][query tile]
  static constexpr int kOffK = kOffQ + 4 * kQBytes;
  static constexpr int kOffV = kOffK + NS * kKBytes;
  static constexpr int kOffP = kOffV + NS * kVBytes;
  static constexpr int kOffQSf = kOffP + 4 * kPBytes;      // P^ double-buffered per query tile
  static constexpr int kOffKSf = kOffQSf + 4 * kQSfBytes;
  static constexpr int kOffVSf = kOffKSf + NS * kKSfBytes;
  static constexpr int kOffPSf = kOffVSf + NS * kVSfBytes;
  // smooth-Q: the score-correction rows of 128 keys, [query tile][3 buffers]
  static constexpr int kOffDs = kOffPSf + 4 * kPSfBytes;
  static constexpr int kOffBar = kOffDs + 2 * 3 * 512;
  static constexpr int kNumBars = 4 + 4 * NS + 8 + 2 + 6 + 1;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
  // fused Q (the kernel quantises bf16 Q itself): the unit's bf16 Q tiles as
  // TMA boxes of 64 channels x 128 tokens (128B swizzle, 1024-byte aligned)
  // and the reciprocal table of the quantiser's quotients
  static constexpr int kStageBox = 128 * 64 * 2;
  static constexpr int kOffQStage = (kOffBar + kNumBars * 8 + 16 + 1023) & ~1023;
  static constexpr int kOffRtab = kOffQStage + 2 * (D / 64) * kStageBox;
  static constexpr int kSmemBytesFq = kOffRtab + 128 * 8 + 1024;
  // Q/K rows of 64 bytes use the 64B swizzle, rows of 32 bytes the 32B one.
  static constexpr uint32_t kQKSwz = (D == 128) ? kSwizzle64B : kSwizzle32B;
  static constexpr uint32_t kQKSbo = 8 * kRowBytes;
  // tensor-memory columns: one S region, which the two query tiles take in
  // turns (separate regions at d = 64, where they fit, measured slower: the
  // turns keep the two softmax warpgroups out of step)
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColO0 = 128;
  static constexpr uint32_t kColSf = 128 + 2 * D;
  // K and V scale columns are double-buffered by tile parity: a tcgen05.cp
  // is not ordered after earlier MMAs that read the columns it overwrites, so
  // tile j+1's scales must not land where tile j's MMAs may still be reading.
  // Q scales likewise by unit parity: [unit parity][query tile] x 8 columns.
  static constexpr uint32_t kColSfQ = kColSf + 0;      // + 16 * (unit & 1) + 8 * q
  static constexpr uint32_t kColSfK = kColSf + 32;     // + 8 * (j & 1)
  static constexpr uint32_t kColSfV = kColSf + 48;     // + 8 * (j & 1)
  static constexpr uint32_t kColSfP0 = kColSf + 64;
  static constexpr uint32_t kColSfP1 = kColSf + 72;
  static constexpr uint32_t kIdescS = idesc_nvf4(BM, BN);
  static constexpr uint32_t kIdescPV = idesc_nvf4(BM, D);
  static_assert(kColSf + 80 <= 512, "tensor memory overflow");
};

struct BarsF4 {
  uint64_t *q_full, *q_empty, *k_full, *k_empty, *v_full, *v_empty, *s_full, *s_free, *p_full, *o_done, *drain,
      *ds_full, *qs_full;
};

// Shared-memory matrix descriptors: each issuing warp builds a base
// descriptor per operand region once, after its register reallocation, and
// adds a byte offset per use (the start-address field is the address / 16;
// every offset here is a multiple of 16) -- the scheme of the BF16 kernel.
// (An earlier build that issued its MMAs from a divergent single-lane branch
// fed the first MMA of every CTA an all-zero A descriptor with this scheme;
// since the issuing warps run converged and issue from an elected lane, the
// precomputed descriptors give exact results, which the one-key-tile-per-CTA
// parity test checks on every row.)
__device__ __forceinline__ uint64_t desc_qk(uint32_t saddr, uint32_t sbo, uint32_t swz) {
  return sdesc(saddr, 16, sbo, swz);
}
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) { return sdesc(saddr, 0, 128, kSwizzleNone); }
__device__ __forceinline__ uint64_t dadd(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

// Copies `nblk` consecutive 512-byte scale blocks at shared address `saddr` to
// tensor memory columns [col, col + 4*nblk), replicated across the four lane
// quarters.
__device__ __forceinline__ void copy_sf(uint32_t tcol, uint32_t saddr, int nblk) {
  for (int i = 0; i < nblk; ++i) tmem_cp_32x128b_warpx4(tcol + 4 * i, desc_sf(saddr + 512 * i));
}
__device__ __forceinline__ void copy_sf_d(uint32_t tcol, uint64_t d0, uint32_t off, int nblk) {
  for (int i = 0; i < nblk; ++i) tmem_cp_32x128b_warpx4(tcol + 4 * i, dadd(d0, off + 512 * i));
}

// One 512-byte smooth-Q correction row (128 keys) into shared memory,
// completing on `bar`.
__device__ __forceinline__ void ds_copy(uint8_t* dst, const float* src, uint64_t* bar) {
  mbar_arrive_expect_tx(bar, 512);
  bulk_load(dst, src, 512, bar);
}

// Fused Q: row r (0..127) of one query tile, quantised from its staged bf16
// boxes (D/64 boxes of 64 channels x 128 tokens, 128B swizzle: 16-byte chunk
// i of row r at chunk i ^ (r & 7)) into a Q buffer as the Q loads would leave
// sa_quantize's bytes there: codes in K-major rows (64B swizzle for 64-byte
// rows: 16-byte chunk c at c ^ ((r >> 1) & 3); 32B swizzle for 32-byte rows:
// c ^ ((r >> 2) & 1)), the scale word of each 64-channel block at byte
// (r % 32) * 16 + (r / 32) * 4 of its 512-byte block.  Arguments are
// shared-memory addresses.
template <int D>
__device__ __forceinline__ void fq_quant_row(uint32_t stage, uint32_t rtab, uint32_t qtile, uint32_t qsf, int r) {
  using C = CfgF4<D>;
  const qg::SharedRtab tab{rtab};
  const uint32_t x7 = (uint32_t)(r & 7) << 4;
#pragma unroll
  for (int quad = 0; quad < D / 64; ++quad) {
    uint32_t w[32], codes[8], sfw;
    const uint32_t src = stage + quad * C::kStageBox + r * 128;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = lds_f4(src + (((uint32_t)i << 4) ^ x7));
      w[4 * i] = __float_as_uint(v.x);
      w[4 * i + 1] = __float_as_uint(v.y);
      w[4 * i + 2] = __float_as_uint(v.z);
      w[4 * i + 3] = __float_as_uint(v.w);
    }
    qg::quant_q_quad(w, tab, codes, sfw);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int ch = 2 * quad + h;
      const int phys = D == 128 ? (ch ^ ((r >> 1) & 3)) : (ch ^ ((r >> 2) & 1));
      sts_u4(qtile + r * C::kRowBytes + phys * 16, codes[4 * h], codes[4 * h + 1], codes[4 * h + 2], codes[4 * h + 3]);
    }
    sts_u32(qsf + quad * 512 + (r & 31) * 16 + (r >> 5) * 4, sfw);
  }
}

template <int D, bool OUT32, bool SQ, bool FQ>
__global__ void __launch_bounds__(kThreads, 1)
    attn_nvfp4_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const uint8_t* __restrict__ q_sf,
                      const uint8_t* __restrict__ k_sf, const uint8_t* __restrict__ v_sf,
                      void* __restrict__ out_ptr, int H, int Hkv, int Lq, int Lkv, int causal, const AttnWork work,
                      const SplitOut part, const Strides so, const float* __restrict__ ds, uint64_t wait_ns) {
  using C = CfgF4<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_base = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  BarsF4 bars;
  bars.q_full = bar_base;                 // [unit parity]
  bars.q_empty = bar_base + 2;            // [unit parity]: that unit's S MMAs are complete
  bars.k_full = bar_base + 4;
  bars.k_empty = bars.k_full + C::NS;
  bars.v_full = bars.k_empty + C::NS;
  bars.v_empty = bars.v_full + C::NS;
  bars.s_full = bars.v_empty + C::NS;
  bars.s_free = bars.s_full + 2;
  bars.p_full = bars.s_free + 2;
  bars.o_done = bars.p_full + 2;
  bars.drain = bars.o_done + 2;
  bars.ds_full = bars.drain + 2;          // [query tile][3]
  bars.qs_full = bars.ds_full + 6;        // fused Q: the unit's bf16 Q tiles have landed in the staging
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_base + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // the quantised operands hold Lq and Lkv rounded up to whole tiles per head
  const int Lqp = (Lq + 127) & ~127, Lkvp = (Lkv + 127) & ~127;
  const int G = H / Hkv;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i) mbar_init(bar_base + i, 1);
    for (int q = 0; q < 2; ++q) {
      mbar_init(bars.s_free + q, 128);
      mbar_init(bars.p_full + q, 128);
      if constexpr (FQ) mbar_init(bars.q_full + q, 8);   // one arrival per softmax warp
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if constexpr (FQ) {
    if (threadIdx.x < 128)
      reinterpret_cast<float2*>(smem + C::kOffRtab)[threadIdx.x] = qg::rtab_entry(threadIdx.x);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  // (each role below walks the CTA's unit list with its own iterator)
  if (warp >= 8) {
    // Register split: the launch gives every thread kLaunchRegs; this
    // warpgroup (producer, MMA issuer, two idle warps) keeps kOtherRegs and the
    // two softmax warpgroups take kSoftmaxRegs (the SQ pair for the smooth-Q
    // variant; sums checked above).
    reg_dealloc<SQ ? kOtherRegsSq : kOtherRegs>();
    // The producer and MMA warps run their loops with all 32 lanes (waits are
    // warp-wide, addresses and descriptors warp-uniform); one elected lane
    // issues each TMA copy, tcgen05 instruction and commit.
    if (warp == 8) {
      // ---------------------------------------------------------- producer
      const bool leader = elect_one();
      UnitIter it;
      unit_iter_init(work, it);
      AttnUnitRef u;
      if (leader) {
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
      }
      pdl_wait();                                       // the inputs are written (programmatic launch)
      // K and V tiles and Q units issued so far (over the whole list); the
      // counts also tell the abort path which copies may still be in flight
      int nk = 0, nv = 0, ug = 0;
      bool ok = true;
      while (ok && unit_next(work, it, u)) {
        const int qb = ug & 1;
        const long long bhq = u.bh;
        const long long bhk = (long long)(u.bh / H) * Hkv + (u.bh % H) / G;
        if constexpr (!FQ) {
          // Q of this unit into buffer qb, once the S MMAs of unit ug-2 (the
          // last to read that buffer) are complete
          if (ug >= 2 && !mbar_wait_backoff_warp(bars.q_empty + qb, ((ug >> 1) - 1) & 1, abort_flag, wait_ns,
                                                 kProducerSleepNs)) {
            ok = false;
            break;
          }
          if (leader) {
            mbar_arrive_expect_tx(bars.q_full + qb, u.nq * (C::kQBytes + C::kQSfBytes));
            for (int q = 0; q < u.nq; ++q) {
              const int qt = u.qt0 + q;
              tma_load_2d(smem + C::kOffQ + (2 * qb + q) * C::kQBytes, &tmap_q, bars.q_full + qb, 0,
                          (int)(bhq * Lqp + (long long)qt * BM));
              bulk_load(smem + C::kOffQSf + (2 * qb + q) * C::kQSfBytes,
                        q_sf + (bhq * (Lqp / 128) + qt) * C::kQSfBytes, C::kQSfBytes, bars.q_full + qb);
            }
          }
        }
        ++ug;
        const int nt = u.n[0] > u.n[1] ? u.n[0] : u.n[1];
        for (int j = 0; j < nt; ++j) {
          const int s = nk % C::NS;
          const uint32_t par = ((nk / C::NS) - 1) & 1;
          const int ja = u.jb + j;                      // the key tile
          if (nk >= C::NS &&
              !mbar_wait_backoff_warp(bars.k_empty + s, par, abort_flag, wait_ns, kProducerSleepNs)) {
            ok = false;
            break;
          }
          if (leader) {
            mbar_arrive_expect_tx(bars.k_full + s, C::kKBytes + C::kKSfBytes);
            tma_load_2d(smem + C::kOffK + s * C::kKBytes, &tmap_k, bars.k_full + s, 0,
                        (int)(bhk * Lkvp + (long long)ja * BN));
            bulk_load(smem + C::kOffKSf + s * C::kKSfBytes, k_sf + (bhk * (Lkvp / 128) + ja) * C::kKSfBytes,
                      C::kKSfBytes, bars.k_full + s);
          }
          ++nk;
          if (nv >= C::NS &&
              !mbar_wait_backoff_warp(bars.v_empty + s, par, abort_flag, wait_ns, kProducerSleepNs)) {
            ok = false;
            break;
          }
          if (leader) {
            mbar_arrive_expect_tx(bars.v_full + s, C::kVBytes + C::kVSfBytes);
            tma_load_2d(smem + C::kOffV + s * C::kVBytes, &tmap_v, bars.v_full + s, ja * (BN / 2),
                        (int)(bhk * D));
            bulk_load(smem + C::kOffVSf + s * C::kVSfBytes, v_sf + (bhk * (Lkvp / 64) + 2 * ja) * 512,
                      C::kVSfBytes, bars.v_full + s);
          }
          ++nv;
        }
      }
      if (*abort_flag) {
        // let every copy already issued land before the CTA (and its shared
        // memory) goes away: the last issue into each Q buffer and each stage
        if constexpr (!FQ) {
          for (int g = (ug > 2 ? ug - 2 : 0); g < ug; ++g)
            mbar_wait_drain(bars.q_full + (g & 1), (g >> 1) & 1, wait_ns);
        }
        for (int g = (nk > C::NS ? nk - C::NS : 0); g < nk; ++g)
          mbar_wait_drain(bars.k_full + g % C::NS, (g / C::NS) & 1, wait_ns);
        for (int g = (nv > C::NS ? nv - C::NS : 0); g < nv; ++g)
          mbar_wait_drain(bars.v_full + g % C::NS, (g / C::NS) & 1, wait_ns);
      }
    } else if (warp == 9) {
      // ---------------------------------------------------------- S issuer
      // S0(0), S1(0), S0(1), S1(1), ... into the one S region; each waits
      // until the softmax warps have read the previous S (over the whole
      // list).  Scale-factor buffers in tensor memory are rewritten only once
      // the MMAs that read them are complete (a tcgen05.cp is not ordered
      // after them): a tile's K scales go to the buffer of its parity, last
      // read by the S MMAs of tile gk - 2, whose commit is that stage's
      // k_empty phase; a unit's Q scales to the buffer of its parity, last
      // read by unit ug - 2, whose commit is q_empty.
      const bool leader = elect_one();
      const uint32_t sb = smem_u32(smem);
      const uint32_t tS = tbase + C::kColS;
      const uint64_t dQ0 = desc_qk(sb + C::kOffQ, C::kQKSbo, C::kQKSwz);
      const uint64_t dK0 = desc_qk(sb + C::kOffK, C::kQKSbo, C::kQKSwz);
      const uint64_t dSf0 = desc_sf(sb);
      UnitIter it;
      unit_iter_init(work, it);
      AttnUnitRef u;
      int last_q = -1;
      uint32_t last_par = 0;
      int cs[2] = {0, 0};       // S MMAs issued per query tile
      int gk = 0, ug = 0;
      bool ok = true;
      while (ok && unit_next(work, it, u)) {
        const int qb = ug & 1;
        const int nt = u.n[0] > u.n[1] ? u.n[0] : u.n[1];
        ok = mbar_wait_warp(bars.q_full + qb, (ug >> 1) & 1, abort_flag, wait_ns);
        if (!ok) break;
        // Q scales of this unit to the columns of its parity.  (A unit without
        // key tiles issues no MMA, and so no copy whose completion a commit
        // would have to cover.)
        if (ok && nt > 0 && ug >= 2)
          ok = mbar_wait_warp(bars.q_empty + qb, ((ug >> 1) - 1) & 1, abort_flag, wait_ns);
        if (!ok) break;
        if (nt > 0) {
          tc_fence_after();
          if (leader)
            for (int q = 0; q < u.nq; ++q)
              copy_sf_d(tbase + C::kColSfQ + 16 * qb + 8 * q, dSf0, C::kOffQSf + (2 * qb + q) * C::kQSfBytes, D / 64);
          __syncwarp();
        }
        for (int j = 0; ok && j < nt; ++j, ++gk) {
          const int s = gk % C::NS;
          ok = mbar_wait_warp(bars.k_full + s, (gk / C::NS) & 1, abort_flag, wait_ns);
          if (ok && gk >= 2)
            ok = mbar_wait_warp(bars.k_empty + (gk - 2) % C::NS, ((gk - 2) / C::NS) & 1, abort_flag, wait_ns);
          if (!ok) break;
          tc_fence_after();
          const uint32_t sfk = tbase + C::kColSfK + 8 * (gk & 1);
          if (leader) copy_sf_d(sfk, dSf0, C::kOffKSf + s * C::kKSfBytes, D / 64);
          __syncwarp();
          for (int q = 0; ok && q < 2; ++q) {
            if (j >= (q ? u.n[1] : u.n[0])) continue;
            if (last_q >= 0) ok = mbar_wait_warp(bars.s_free + last_q, last_par, abort_flag, wait_ns);
            if (!ok) break;
            tc_fence_after();
            const uint32_t sfq = tbase + C::kColSfQ + 16 * qb + 8 * q;
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < D / 64; ++kk)
                mma_nvf4(tS, dadd(dQ0, (2 * qb + q) * C::kQBytes + kk * 32), dadd(dK0, s * C::kKBytes + kk * 32),
                         C::kIdescS,
                         sfq + 4 * kk, sfk + 4 * kk, kk > 0 ? 1u : 0u);
              tc_commit(bars.s_full + q);
            }
            __syncwarp();
            last_q = q;
            last_par = cs[q] & 1;
            ++cs[q];
          }
          if (ok && leader) tc_commit(bars.k_empty + s);      // K slot free once these S MMAs are done
          __syncwarp();
        }
        if (!ok) break;
        if (leader) tc_commit(bars.q_empty + qb);            // Q buffer free once this unit's S MMAs are done
        __syncwarp();
        ++ug;
      }
      if (!ok) {
        if (leader) tc_commit(bars.drain);
        __syncwarp();
        mbar_wait_drain(bars.drain, 0, wait_ns);
      }
    } else if (warp == 10) {
      // ---------------------------------------------------------- P.V issuer
      // P0.V(j), P1.V(j), ... each once its softmax warps have written P^.
      // V scales of a tile go to the buffer of its parity, last read by the
      // P.V MMAs two tiles earlier, which the softmax warps have seen complete
      // before releasing the previous P^.  The first P.V of a unit starts the
      // accumulator afresh: the softmax warps read the previous unit's O
      // before they release that P^.
      const bool leader = elect_one();
      const uint32_t sb = smem_u32(smem);
      const uint64_t dP0 = desc_qk(sb + C::kOffP, 512, kSwizzle64B);
      const uint64_t dV0 = desc_qk(sb + C::kOffV, 512, kSwizzle64B);
      const uint64_t dSf0 = desc_sf(sb);
      UnitIter it;
      unit_iter_init(work, it);
      AttnUnitRef u;
      int cp[2] = {0, 0};       // P.V MMAs issued per query tile
      int gk = 0;
      bool ok = true;
      while (ok && unit_next(work, it, u)) {
        const int nt = u.n[0] > u.n[1] ? u.n[0] : u.n[1];
        for (int j = 0; ok && j < nt; ++j, ++gk) {
          const int s = gk % C::NS;
          ok = mbar_wait_warp(bars.v_full + s, (gk / C::NS) & 1, abort_flag, wait_ns);
          if (!ok) break;
          tc_fence_after();
          const uint32_t sfv = tbase + C::kColSfV + 8 * (gk & 1);
          if (leader) copy_sf_d(sfv, dSf0, C::kOffVSf + s * C::kVSfBytes, 2);
          __syncwarp();
          for (int q = 0; ok && q < 2; ++q) {
            if (j >= (q ? u.n[1] : u.n[0])) continue;
            ok = mbar_wait_warp(bars.p_full + q, cp[q] & 1, abort_flag, wait_ns);
            if (!ok) break;
            tc_fence_after();
            const uint32_t sfp = tbase + (q ? C::kColSfP1 : C::kColSfP0);
            const uint32_t tO = tbase + C::kColO0 + q * D;
            if (leader) {
              const int pb = 2 * q + (cp[q] & 1);            // P^ buffer of this tile
              copy_sf_d(sfp, dSf0, C::kOffPSf + pb * C::kPSfBytes, 2);
#pragma unroll
              for (int kk = 0; kk < BN / 64; ++kk)
                mma_nvf4(tO, dadd(dP0, pb * C::kPBytes + kk * 32), dadd(dV0, s * C::kVBytes + kk * 32), C::kIdescPV,
                         sfp + 4 * kk, sfv + 4 * kk, (j > 0 || kk > 0) ? 1u : 0u);
              tc_commit(bars.o_done + q);
            }
            __syncwarp();
            ++cp[q];
          }
          if (ok && leader) tc_commit(bars.v_empty + s);      // V slot free once these P.V MMAs are done
          __syncwarp();
        }
      }
      if (!ok) {
        if (leader) tc_commit(bars.drain + 1);
        __syncwarp();
        mbar_wait_drain(bars.drain + 1, 0, wait_ns);
      }
    } else if (FQ && warp == 11) {
      // ------------------------------------------------- fused Q: staging
      // A unit's bf16 Q tiles (tokens past Lq read as zeros) into the staging,
      // once every softmax warp has quantised the previous unit's from it
      // (that unit's Q full barrier).
      const bool leader = elect_one();
      UnitIter it;
      unit_iter_init(work, it);
      AttnUnitRef u;
      pdl_wait();                                       // Q is written (programmatic launch)
      int ug = 0;
      bool ok = true;
      while (ok && unit_next(work, it, u)) {
        // (a wait of about one unit: polled with sleeps, so as not to take
        // issue slots from the softmax warps of this SM sub-partition)
        if (ug >= 1)
          ok = mbar_wait_backoff_warp(bars.q_full + ((ug - 1) & 1), ((ug - 1) >> 1) & 1, abort_flag, wait_ns,
                                      kStageSleepNs);
        if (!ok) break;
        if (leader) {
          // (bf16 Q is read once: its lines go first when L2 needs room)
          const uint64_t pol = l2_policy_evict_first();
          mbar_arrive_expect_tx(bars.qs_full, u.nq * (D / 64) * C::kStageBox);
          for (int q = 0; q < u.nq; ++q)
            for (int b = 0; b < D / 64; ++b)
              tma_load_4d_hint(smem + C::kOffQStage + (q * (D / 64) + b) * C::kStageBox, &tmap_q, bars.qs_full,
                               64 * b, (u.qt0 + q) * BM, (int)(u.bh % H), (int)(u.bh / H), pol);
        }
        __syncwarp();
        ++ug;
      }
      // the last copy has landed before the shared memory goes away (after
      // an abort it may not have been waited for)
      if (ug > 0) mbar_wait_drain(bars.qs_full, (ug - 1) & 1, wait_ns);
    }
  } else {
    reg_alloc<SQ ? kSoftmaxRegsSq : kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax + P quantisation
    // (smooth-Q: these threads copy the score corrections written by the
    // launch before, so they wait for it too)
    if constexpr (SQ) pdl_wait();
    const int q = warp / 4;
    // Smooth-Q: the correction row of each (query tile, key tile) reaches
    // shared memory by a bulk copy issued by thread 0 of the warpgroup one
    // tile ahead, into buffer t % 3 for this slot's tile t (t = cq over the
    // whole list).  Buffer (t + 1) % 3 last held tile t - 2, which every
    // thread of the warpgroup has finished: thread 0 reaches tile t once S(t)
    // is complete, issued after every thread loaded S(t - 1).
    const bool ds_issuer = (threadIdx.x % 128) == 0;
    int ds_hi = 0;                                      // tiles of this slot whose copy is issued (issuer only)
    const int r = (warp % 4) * 32 + lane;
    const uint32_t lane_addr = tbase + (((warp % 4) * 32) << 16);
    const float c = softmax_scale_log2<D>();
    uint8_t* prow0 = smem + C::kOffP + 2 * q * C::kPBytes + r * 64;
    uint8_t* psf0 = smem + C::kOffPSf + 2 * q * C::kPSfBytes + (r % 32) * 16 + (r / 32) * 4;
    const uint32_t ocol = C::kColO0 + q * D;
    UnitIter it;
    unit_iter_init(work, it);
    AttnUnitRef u;
    int cq = 0;               // tiles of this query-tile slot so far (over the whole list)
    bool ok = true;
    // Fused Q: this thread's row of query tile q of unit g (index over the
    // whole list) into Q buffer g & 1, once the unit's bf16 tiles are staged
    // and the S MMAs of unit g - 2 (the buffer's last readers) are complete;
    // every warp arrives on the buffer's full barrier, quantising or not.
    auto fq_unit = [&](const AttnUnitRef& v, int g) -> bool {
      const int qb = g & 1;
      if (!mbar_wait_warp(bars.qs_full, g & 1, abort_flag, wait_ns)) return false;
      if (g >= 2 && !mbar_wait_warp(bars.q_empty + qb, ((g >> 1) - 1) & 1, abort_flag, wait_ns)) return false;
      if (q < v.nq) {
        const uint32_t sb = smem_u32(smem);
        fq_quant_row<D>(sb + C::kOffQStage + q * (D / 64) * C::kStageBox, sb + C::kOffRtab,
                        sb + C::kOffQ + (2 * qb + q) * C::kQBytes, sb + C::kOffQSf + (2 * qb + q) * C::kQSfBytes, r);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.q_full + qb);
      return true;
    };
    int us = -1;              // fused Q: index of the current unit over the whole list
    while (ok && unit_next(work, it, u)) {
      const int nq = q ? u.n[1] : u.n[0];
      ++us;
      if constexpr (FQ) {
        // the next unit's Q (and, for the first unit, its own), so that the S
        // MMAs find it ready when they reach the next unit
        for (int k = us == 0 ? 0 : 1; ok && k < 2; ++k) {
          AttnUnitRef v = u;
          bool has = true;
          if (k == 1) {
            UnitIter t = it;
            has = unit_next(work, t, v);
          }
          if (has) ok = fq_unit(v, us + k);
        }
        if (!ok) break;
      }
      if (q >= u.nq) continue;                         // the unit has no second query tile
      const int qt = u.qt0 + q;
      float m_run = -INFINITY, m_ref = 0.f, lam = 0.f;
      bool have_ref = false;
      for (int j = 0; j < nq; ++j, ++cq) {
        if (!mbar_wait_warp(bars.s_full + q, cq & 1, abort_flag, wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int i = 0; i < 4; ++i) tmem_ld32(lane_addr + C::kColS + 32 * i, sr[i]);
        tmem_ld_wait(sr[0]);
        tmem_launder(sr[1]);
        tmem_launder(sr[2]);
        tmem_launder(sr[3]);
        tc_fence_before();
        mbar_arrive(bars.s_free + q);
        float sv[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) sv[i] = __uint_as_float(sr[i / 32][i % 32]);
        const int ja = u.jb + j;
        if constexpr (SQ) {
          // smooth-Q: S = Q^' K^'^T + dS, dS the query tile's correction of
          // these 128 keys (the same for every row: broadcast reads)
          if (ds_issuer) {
            // this slot's correction rows of the unit are contiguous: the
            // whole range is prefetched into L2 when the unit starts
            const float* row0 = ds + (((long long)u.bh * (Lqp / BM) + qt) * Lkvp + (long long)u.jb * BN);
            if (j == 0) {
              bulk_prefetch_l2(row0, (uint32_t)nq * 512u);
              ds_copy(smem + C::kOffDs + (3 * q + cq % 3) * 512, row0, bars.ds_full + 3 * q + cq % 3);
            }
            if (j + 1 < nq) {
              const int t = (cq + 1) % 3;
              ds_copy(smem + C::kOffDs + (3 * q + t) * 512, row0 + (j + 1) * BN, bars.ds_full + 3 * q + t);
            }
            ds_hi = j + 1 < nq ? cq + 2 : cq + 1;
          }
          if (!mbar_wait_warp(bars.ds_full + 3 * q + cq % 3, (cq / 3) & 1, abort_flag, wait_ns)) {
            ok = false;
            break;
          }
          // (shared-window loads, four in flight before their adds)
          const uint32_t dsa = smem_u32(smem + C::kOffDs + (3 * q + cq % 3) * 512);
#pragma unroll
          for (int i0 = 0; i0 < 32; i0 += 4) {
            float4 t[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) t[i] = lds_f4(dsa + 16 * (i0 + i));
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int e = 4 * (i0 + i);
              add2(sv[e], sv[e + 1], sv[e], sv[e + 1], t[i].x, t[i].y);
              add2(sv[e + 2], sv[e + 3], sv[e + 2], sv[e + 3], t[i].z, t[i].w);
            }
          }
        }
        // keys this row may not see: past Lkv (the zero padding of a ragged
        // last tile) and, causal, past its position qt*128 + r + Lkv - Lq
        int lim = Lkv - ja * BN;
        if (causal) lim = min(lim, qt * BM + r + work.coff - ja * BN + 1);
        lim = min(lim, BN);
        if (lim < BN) {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= lim) sv[i] = -INFINITY;
        }
        float gm[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) gm[g] = max16(sv + 16 * g);
        const float mx = max3(max3(gm[0], gm[1], gm[2]), max3(gm[3], gm[4], gm[5]), fmaxf(gm[6], gm[7]));
        const float m_t = mx * c;
        const float m_new = fmaxf(m_run, m_t);
        const bool live = (m_t > -INFINITY) && (m_t >= m_new - kSkipBelow);
        m_run = m_new;
        uint32_t codes[4];
        uint32_t sfw[2] = {0u, 0u};
        const float corr = (live && have_ref) ? ex2_approx(m_ref - m_t) : 1.f;
        // whether O must be rescaled to the new tile maximum (warp-uniform)
        const bool do_corr = j > 0 && __any_sync(0xffffffffu, corr != 1.f);
        // P^ of this tile goes to buffer cq & 1, last read by the P.V two
        // tiles back, whose completion this thread waited for at the
        // previous tile (or in the previous unit's epilogue)
        uint8_t* prow = prow0 + (cq & 1) * C::kPBytes;
        uint8_t* psf = psf0 + (cq & 1) * C::kPSfBytes;
        {
          // Warp-uniform: a row that skips this tile gets bias = -inf, so its
          // P2, codes, scales and sum are all zero (the O chunks below use
          // warp-collective tensor-memory instructions).
          const float bias = live ? kLog2PRange - m_t : -INFINITY;
          // group scales s2 = e4m3(max16(P2) / 6) from the group maxima of
          // P2 = 2^(x*c + bias), and the exponent offsets b_g = bias - log2 s2 so
          // that P2 / s2 = 2^(x*c + b_g).  A zero scale (the group underflows:
          // every P2 < 6 * 2^-10) keeps b_g = bias; its values are then below
          // 0.25 and encode as code 0, and its sum is P2's own.
          float bg[8], fg[8];
          uint32_t s16[4];
#pragma unroll
          for (int g = 0; g < 8; g += 2) {
            float a0, a1;
            fma2(a0, a1, gm[g], gm[g + 1], c, c, bias, bias);
            a0 = ex2_approx(a0);
            a1 = ex2_approx(a1);
            mul2(a0, a1, a0, a1, 1.0f / 6.0f, 1.0f / 6.0f);
            s16[g / 2] = cvt_e4m3x2(a0, a1);
            e4m3x2_to_f32(s16[g / 2], fg[g], fg[g + 1]);
          }
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            fg[g] = fg[g] == 0.f ? 1.f : fg[g];
            bg[g] = bias - lg2_approx(fg[g]);
          }
          sfw[0] = s16[0] | (s16[1] << 16);
          sfw[1] = s16[2] | (s16[3] << 16);
          float rs = 0.f;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            float uu[2] = {0.f, 0.f};
            float* pp = sv + 16 * g;
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              fma2(pp[i], pp[i + 1], pp[i], pp[i + 1], c, c, bg[g], bg[g]);
              pp[i] = ex2_approx(pp[i]);
              pp[i + 1] = ex2_approx(pp[i + 1]);
              add2(uu[0], uu[1], uu[0], uu[1], pp[i], pp[i + 1]);
            }
            rs = fmaf(uu[0] + uu[1], fg[g], rs);
            codes[2 * (g & 1)] = cvt_e2m1x8(pp[0], pp[1], pp[2], pp[3], pp[4], pp[5], pp[6], pp[7]);
            codes[2 * (g & 1) + 1] = cvt_e2m1x8(pp[8], pp[9], pp[10], pp[11], pp[12], pp[13], pp[14], pp[15]);
            if (g & 1) {
              // P^ row r, 16-byte chunk g/2 (two groups), 64B-swizzled: chunk c at
              // c ^ ((r >> 1) & 3); stored as soon as it is encoded
              const int ch = g >> 1;
              *reinterpret_cast<uint4*>(prow + ((ch ^ ((r >> 1) & 3)) * 16)) =
                  make_uint4(codes[0], codes[1], codes[2], codes[3]);
            }
          }
          if (live) {
            lam = have_ref ? fmaf(lam, corr, rs) : rs;
            m_ref = m_t;
            have_ref = true;
          }
        }
        *reinterpret_cast<uint32_t*>(psf) = sfw[0];
        *reinterpret_cast<uint32_t*>(psf + 512) = sfw[1];
        if (j > 0) {
          // O may be rescaled once P.V of the last tile is done (long since, as
          // a rule: the P work of this tile ran in between)
          if (!mbar_wait_warp(bars.o_done + q, (cq - 1) & 1, abort_flag, wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (do_corr) {
          // the O row to the new tile maximum: all chunks loaded before one
          // wait (the score registers are free again), scaled, stored back
          uint32_t o[D / 32][32];
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(lane_addr + ocol + 32 * cc, o[cc]);
          tmem_ld_wait(o[0]);
#pragma unroll
          for (int cc = 1; cc < D / 32; ++cc) tmem_launder(o[cc]);
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float x0 = __uint_as_float(o[cc][i]), x1 = __uint_as_float(o[cc][i + 1]);
              mul2(x0, x1, x0, x1, corr, corr);
              o[cc][i] = __float_as_uint(x0);
              o[cc][i + 1] = __float_as_uint(x1);
            }
            tmem_st32(lane_addr + ocol + 32 * cc, o[cc]);
          }
          tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bars.p_full + q);
      }
      if (!ok) break;
      // ---- the unit's result for this row: O, or a partial for the combine
      // pass (O unnormalised in units of 2^m_ref / 2688 as is lam, m_ref
      // (-inf if no key tile was live) and lam)
      const bool row_in = qt * BM + r < Lq;             // rows of the padding are not stored
      const bool partial = u.slot >= 0;
      const long long bhq = u.bh;
      long long prow;
      if (work.streamk)
        prow = (long long)u.slot * (2 * BM) + q * BM + r;
      else
        prow = ((long long)u.slot * work.nbh + bhq) * Lqp + (long long)qt * BM + r;
      if (partial && nq == 0 && row_in)
        *reinterpret_cast<float2*>(part.ml + 2 * prow) = make_float2(-INFINITY, 0.f);
      if (nq > 0) {
        if (!mbar_wait_warp(bars.o_done + q, (cq - 1) & 1, abort_flag, wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float inv_l = 1.f / lam;
        const long long obase = (bhq / H) * so.b + (bhq % H) * so.h + ((long long)qt * BM + r) * so.t;
        if (partial && row_in)
          *reinterpret_cast<float2*>(part.ml + 2 * prow) = make_float2(have_ref ? m_ref : -INFINITY, lam);
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(lane_addr + ocol + 32 * cc, o);
          tmem_ld_wait(o);
          if (!row_in) continue;
          if (partial) {
            float4* dst = reinterpret_cast<float4*>(part.o + prow * D + 32 * cc);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                   __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
            continue;
          }
          // (O is not read again here: streaming stores, so that its lines
          // leave L2 before the K and V tiles other CTAs still read)
          if constexpr (OUT32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out_ptr) + obase + 32 * cc);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              __stcs(dst + i, make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                          __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l));
          } else {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out_ptr) + obase + 32 * cc);
#pragma unroll
            for (int i = 0; i < 4; ++i) __stcs(dst + i, make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]));
          }
        }
        // (the tensor-memory loads above are complete: the next unit's first
        // P.V, which overwrites O, is issued only after this thread's next
        // p_full arrival)
      }
    }
    if constexpr (SQ) {
      // after an abort, let the correction copies still in flight land
      // before the shared memory goes away (the last copy into each buffer)
      if (ds_issuer && !ok)
        for (int t = ds_hi > 3 ? ds_hi - 3 : 0; t < ds_hi; ++t)
          mbar_wait_drain(bars.ds_full + 3 * q + t % 3, (t / 3) & 1, wait_ns);
    }
  }

  tc_fence_before();
  __syncthreads();
  // every output of this CTA is stored: a combine launch queued behind this
  // one (programmatic dependent launch) may be scheduled
  pdl_launch_dependents();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, bool OUT32, bool SQ, bool FQ>
cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const sa_fp4_qkv& x,
                     void* o, const Strides& so, const Dims& dm, int causal, int nsplit, const SplitOut& part,
                     const float* ds, cudaStream_t s) {
  using C = CfgF4<D>;
  constexpr int kSmem = FQ ? C::kSmemBytesFq : C::kSmemBytes;
  // kernel attributes are per device: set them on the first launch on each
  static std::atomic<bool> attr_done[kMaxDevices];
  cudaError_t e = once_per_device(attr_done, [] {
    // The warpgroup register split assumes kLaunchRegs registers per thread at
    // launch; with fewer, a setmaxnreg increase could never be satisfied.
    cudaFuncAttributes fa;
    cudaError_t r = cudaFuncGetAttributes(&fa, attn_nvfp4_kernel<D, OUT32, SQ, FQ>);
    if (r != cudaSuccess) return r;
    if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(attn_nvfp4_kernel<D, OUT32, SQ, FQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmem);
  });
  if (e != cudaSuccess) return e;
  int ctas = 0;
  const AttnWork work = nsplit == kStreamK
                            ? make_streamk_work(dm.B, dm.H, dm.Lq, dm.Lkv, causal, device_sm_count(), &ctas)
                            : make_attn_work(dm.B, dm.H, dm.Lq, dm.Lkv, causal, device_sm_count(), &ctas, nsplit);
  // a programmatic dependent launch: the CTAs' set-up overlaps the end of
  // the kernel before (sa_quantize's last launch, as a rule); the producer
  // waits for it before its first load
  cudaLaunchAttribute attr;
  const cudaLaunchConfig_t cfg = pdl_launch_config(dim3(ctas), dim3(kThreads), kSmem, s, &attr);
  e = cudaLaunchKernelEx(&cfg, attn_nvfp4_kernel<D, OUT32, SQ, FQ>, tq, tk, tv,
                                     static_cast<const uint8_t*>(x.q_sf), static_cast<const uint8_t*>(x.k_sf),
                                     static_cast<const uint8_t*>(x.v_sf), o, dm.H, dm.Hkv, dm.Lq, dm.Lkv, causal,
                                     work, part, so, ds, kWaitLimitNs);
  if (e == cudaSuccess && work.streamk) e = launch_streamk_combine(work, ctas, part, dm, o, so, OUT32, s);
  else if (e == cudaSuccess && work.nsplit > 1) e = launch_splitkv_combine(part, work.nsplit, dm, o, so, OUT32, s);
  return e;
}

// Test support: the FP32 score tile S = Q^ K^'^T of one (query tile, key
// tile) from the attention kernel's own S step -- the same tensor maps,
// shared-memory descriptors, scale-factor copies and block-scaled MMAs -- read
// back from tensor memory and written row-major [128][128] to `out`.  One CTA
// of 128 threads (warp w reads lanes 32w..32w+31); every wait bounded.
template <int D>
__global__ void __launch_bounds__(128, 1)
    nvfp4_score_tile_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                            const uint8_t* __restrict__ q_sf, const uint8_t* __restrict__ k_sf, int qrow, int krow,
                            long long qsf_blk, long long ksf_blk, float* __restrict__ out, uint64_t wait_ns) {
  using C = CfgF4<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = smem;
  uint8_t* sk = smem + C::kQBytes;
  uint8_t* sqsf = sk + C::kKBytes;
  uint8_t* sksf = sqsf + C::kQSfBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sksf + C::kKSfBytes);   // [0] loads, [1] MMA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_init(bar + 1, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  constexpr uint32_t kColSfQ = 128, kColSfK = 128 + 4 * (D / 64);
  bool ok = true;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, C::kQBytes + C::kKBytes + C::kQSfBytes + C::kKSfBytes);
    tma_load_2d(sq, &tmap_q, bar, 0, qrow);
    tma_load_2d(sk, &tmap_k, bar, 0, krow);
    bulk_load(sqsf, q_sf + qsf_blk * C::kQSfBytes, C::kQSfBytes, bar);
    bulk_load(sksf, k_sf + ksf_blk * C::kKSfBytes, C::kKSfBytes, bar);
  }
  if (warp == 0) {
    ok = mbar_wait_warp(bar, 0, abort_flag, wait_ns);
    if (ok) {
      tc_fence_after();
      if (elect_one()) {
        const uint32_t sb = smem_u32(smem);
        copy_sf(tbase + kColSfQ, smem_u32(sqsf), D / 64);
        copy_sf(tbase + kColSfK, smem_u32(sksf), D / 64);
#pragma unroll
        for (int kk = 0; kk < D / 64; ++kk)
          mma_nvf4(tbase, desc_qk(sb + kk * 32, C::kQKSbo, C::kQKSwz),
                   desc_qk(sb + C::kQBytes + kk * 32, C::kQKSbo, C::kQKSwz), C::kIdescS, tbase + kColSfQ + 4 * kk,
                   tbase + kColSfK + 4 * kk, kk > 0 ? 1u : 0u);
        tc_commit(bar + 1);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  ok = mbar_wait_warp(bar + 1, 0, abort_flag, wait_ns);
  if (ok) {
    tc_fence_after();
    const uint32_t lane_addr = tbase + ((warp * 32) << 16);
    const int r = warp * 32 + lane;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t s[32];
      tmem_ld32(lane_addr + 32 * cc, s);
      tmem_ld_wait(s);
      float4* dst = reinterpret_cast<float4*>(out + (long long)r * 128 + 32 * cc);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dst[i] = make_float4(__uint_as_float(s[4 * i]), __uint_as_float(s[4 * i + 1]), __uint_as_float(s[4 * i + 2]),
                             __uint_as_float(s[4 * i + 3]));
    }
  } else {
    // the MMA may still be in flight if only the wait gave up: let it land
    // before the tensor memory goes away
    mbar_wait_drain(bar + 1, 0, wait_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 256);
  }
}

// Test support: the exponent path's builtins as the softmax uses them,
// ex2_out[i] = ex2_approx(x[i]), lg2_out[i] = lg2_approx(y[i]).
__global__ void exp_path_selftest_kernel(const float* __restrict__ x, const float* __restrict__ y, int n,
                                         float* __restrict__ ex2_out, float* __restrict__ lg2_out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    ex2_out[i] = ex2_approx(x[i]);
    lg2_out[i] = lg2_approx(y[i]);
  }
}

template <int D>
cudaError_t launch_score_tile(const CUtensorMap& tq, const CUtensorMap& tk, const sa_fp4_qkv& x, const Dims& dm, int b,
                              int h, int qt, int kt, float* out, cudaStream_t s) {
  using C = CfgF4<D>;
  const int smem = C::kQBytes + C::kKBytes + C::kQSfBytes + C::kKSfBytes + 32 + 1024;
  static std::atomic<bool> attr_done[kMaxDevices];
  cudaError_t e = once_per_device(attr_done, [smem] {
    return cudaFuncSetAttribute(nvfp4_score_tile_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (e != cudaSuccess) return e;
  const int Lqp = padded_len(dm.Lq), Lkvp = padded_len(dm.Lkv);
  const long long bhq = (long long)b * dm.H + h;
  const long long bhk = (long long)b * dm.Hkv + h / (dm.H / dm.Hkv);
  nvfp4_score_tile_kernel<D><<<1, 128, smem, s>>>(tq, tk, static_cast<const uint8_t*>(x.q_sf),
                                                  static_cast<const uint8_t*>(x.k_sf), (int)(bhq * Lqp + qt * 128),
                                                  (int)(bhk * Lkvp + kt * 128), bhq * (Lqp / 128) + qt,
                                                  bhk * (Lkvp / 128) + kt, out, kWaitLimitNs);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_nvfp4_score_tile(const CUtensorMap& tq, const CUtensorMap& tk, const sa_fp4_qkv& x,
                                    const Dims& dm, int b, int h, int qt, int kt, float* out, cudaStream_t s) {
  return dm.d == 64 ? launch_score_tile<64>(tq, tk, x, dm, b, h, qt, kt, out, s)
                    : launch_score_tile<128>(tq, tk, x, dm, b, h, qt, kt, out, s);
}

cudaError_t launch_exp_path_selftest(const float* x, const float* y, int n, float* ex2_out, float* lg2_out,
                                     cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  exp_path_selftest_kernel<<<(n + 255) / 256, 256, 0, s>>>(x, y, n, ex2_out, lg2_out);
  return cudaGetLastError();
}

template <int D, bool SQ, bool FQ>
cudaError_t launch_dq(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const sa_fp4_qkv& qkv,
                      void* o, const Strides& so, const Dims& dm, int causal, bool out_f32, int nsplit,
                      const SplitOut& part, const float* ds, cudaStream_t s) {
  return out_f32 ? launch_d<D, true, SQ, FQ>(tq, tk, tv, qkv, o, so, dm, causal, nsplit, part, ds, s)
                 : launch_d<D, false, SQ, FQ>(tq, tk, tv, qkv, o, so, dm, causal, nsplit, part, ds, s);
}

template <int D>
cudaError_t launch_variant(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const sa_fp4_qkv& qkv, void* o, const Strides& so, const Dims& dm, int causal,
                           bool out_f32, int nsplit, const SplitOut& part, cudaStream_t s, const float* ds,
                           bool fuse_q) {
  if (ds) return launch_dq<D, true, false>(tq, tk, tv, qkv, o, so, dm, causal, out_f32, nsplit, part, ds, s);
  if (fuse_q) return launch_dq<D, false, true>(tq, tk, tv, qkv, o, so, dm, causal, out_f32, nsplit, part, ds, s);
  return launch_dq<D, false, false>(tq, tk, tv, qkv, o, so, dm, causal, out_f32, nsplit, part, ds, s);
}

cudaError_t launch_attn_nvfp4(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const sa_fp4_qkv& qkv, void* o, const Strides& so, const Dims& dm, int causal,
                              bool out_f32, int nsplit, const SplitOut& part, cudaStream_t s, const float* ds,
                              bool fuse_q) {
  if (ds && fuse_q) return cudaErrorInvalidValue;          // (the two variants do not combine)
  return dm.d == 64 ? launch_variant<64>(tq, tk, tv, qkv, o, so, dm, causal, out_f32, nsplit, part, s, ds, fuse_q)
                    : launch_variant<128>(tq, tk, tv, qkv, o, so, dm, causal, out_f32, nsplit, part, s, ds, fuse_q);
}

cudaError_t attn_nvfp4_read_error(int* out) { return read_and_clear_device_error(out); }

}  // namespace sa
