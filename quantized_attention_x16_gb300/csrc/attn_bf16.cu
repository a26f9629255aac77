// attn_bf16.cu -- exact BF16 fused attention forward on tcgen05 tensor cores.
//
// Data flow (page "FlashAttention kernels", sections 0-1): tile by tile with
// online softmax; the Lq x Lkv scores never leave the SM.  Work partitioning
// (same page, FA2): one CTA per (batch, head, 256 query rows).  Hardware
// mapping: TMA tile loads into 128B-swizzled SMEM, tcgen05 MMAs with FP32
// accumulators in tensor memory, warp specialisation (load / MMA / softmax
// roles) as in the Blackwell attention pipelines the page "kernel overview"
// describes (AVO: MMA, softmax, correction and load warps).
//
// CTA layout (384 threads):
//   warps 0-3  : softmax + correction + epilogue of query tile 0 (one thread
//                per row)
//   warps 4-7  : the same for query tile 1
//   warp 8     : TMA producer (Q once, then K/V tiles into an NS-stage ring)
//   warp 9     : S MMA issuer, warp 10: P.V MMA issuer (each runs its loop
//                with all lanes and issues from one elected lane; operand
//                descriptors are built once, a use adds its byte offset to
//                the start-address field)
//   warp 11    : idle
// Tensor memory (512 columns): S (one 128-column region shared by the two
// query tiles), O0, O1 (d columns each), P0, P1 (64 columns each, bf16
// pairs).  S = Q K^T is read into registers, P = 2^(x - m) is written back as
// bf16 into tensor memory and consumed by the P.V MMA as its A operand.
// Online softmax keeps a stale maximum until the true one exceeds it by more
// than 2^8 (exact in real arithmetic; the O rescale then runs rarely).

#include <cuda_bf16.h>

#include "internal.h"
#include "sm100.cuh"
#include "work.cuh"

namespace sa {
namespace {

constexpr int BM = 128;         // query rows per tile
constexpr int BN = 128;         // keys per KV tile
constexpr int kThreads = 384;
constexpr uint32_t kProducerSleepNs = 256;   // poll interval of the TMA producer's waits
constexpr int kSoftmaxRegs = 200;   // 8 softmax warps
constexpr int kOtherRegs = 104;      // producer / MMA warpgroup
constexpr int kLaunchRegs = 168;    // 65536 / 384 rounded down to a multiple of 8
static_assert(8 * 32 * kSoftmaxRegs + 4 * 32 * kOtherRegs <= kThreads * kLaunchRegs, "register split");
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int D>
struct CfgBF16 {
  static constexpr int NS = (D == 64) ? 4 : 2;            // K/V ring depth
  static constexpr int kHalfBytes = 128 * 64 * 2;         // one [128 x 64] bf16 box (16 KB)
  static constexpr int kTileBytes = (D / 64) * kHalfBytes;
  static constexpr int kOffQ = 0;                         // Q0, Q1
  static constexpr int kOffK = kOffQ + 2 * kTileBytes;
  static constexpr int kOffV = kOffK + NS * kTileBytes;
  static constexpr int kOffBar = kOffV + NS * kTileBytes;
  static constexpr int kNumBars = 1 + 4 * NS + 8 + 2;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;   // + alignment slack
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColO0 = 128;
  static constexpr uint32_t kColP0 = 128 + 2 * D;
  static constexpr uint32_t kIdescS = idesc_bf16(BM, BN, 0, 0);
  static constexpr uint32_t kIdescPV = idesc_bf16(BM, D, 0, 1);
};

struct BarsBF16 {
  uint64_t* q_full;
  uint64_t* k_full;
  uint64_t* k_empty;
  uint64_t* v_full;
  uint64_t* v_empty;
  uint64_t* s_full;   // [2]
  uint64_t* s_free;   // [2]
  uint64_t* p_full;   // [2]
  uint64_t* o_done;   // [2]
  uint64_t* drain;    // MMA clean-up on abort
};

// A shared-memory descriptor displaced by `bytes` (16-byte units land in the
// 14-bit start-address field; addresses stay below 256 KB, so no carry).
__device__ __forceinline__ uint64_t dadd(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

template <int D, bool OUT32>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bf16_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, void* __restrict__ out_ptr, int H, int Hkv,
                     int Lq, int Lkv, int causal, const AttnWork work, const SplitOut part, const Strides so,
                     uint64_t wait_ns) {
  using C = CfgBF16<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_base = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  BarsBF16 bars;
  bars.q_full = bar_base;
  bars.k_full = bar_base + 1;
  bars.k_empty = bars.k_full + C::NS;
  bars.v_full = bars.k_empty + C::NS;
  bars.v_empty = bars.v_full + C::NS;
  bars.s_full = bars.v_empty + C::NS;
  bars.s_free = bars.s_full + 2;
  bars.p_full = bars.s_free + 2;
  bars.o_done = bars.p_full + 2;
  bars.drain = bars.o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_base + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int bh, qt0, nqu, sp;
  attn_unit(work, (int)blockIdx.x, bh, qt0, nqu, sp);              // this CTA's query tiles and split
  const int h = bh % H, b = bh / H;
  const int hk = h / (H / Hkv);
  const bool q1_valid = nqu == 2;
  int ntq[2];
  // key tiles (a ragged last one is zero-filled past Lkv), up to the causal
  // limit of each query tile
  ntq[0] = q_tile_keys(work, qt0);
  ntq[1] = q1_valid ? q_tile_keys(work, qt0 + 1) : 0;
  // key tiles [jb, jb + ntq[q]) of this CTA; loop indices below count from jb
  const int jb = work.nsplit > 1 ? split_range(sp, work.nsplit, ntq) : 0;
  const int nt = ntq[0] > ntq[1] ? ntq[0] : ntq[1];

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumBars; ++i) mbar_init(bar_base + i, 1);
    for (int q = 0; q < 2; ++q) {
      mbar_init(bars.s_free + q, 128);
      mbar_init(bars.p_full + q, 128);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  const int bhq = b * H + h;                                // head index of the partial results
  const long long obase0 = (long long)b * so.b + (long long)h * so.h;   // this head in O

  if (warp >= 8) {
    // Register split: the launch gives every thread kLaunchRegs; this
    // warpgroup (producer, MMA issuer, two idle warps) keeps kOtherRegs and the
    // two softmax warpgroups take kSoftmaxRegs (sum checked above).
    reg_dealloc<kOtherRegs>();
    // The producer and MMA warps run their loops with all 32 lanes (waits are
    // warp-wide, addresses and descriptors warp-uniform); one elected lane
    // issues each TMA copy, tcgen05 instruction and commit.
    if (warp == 8) {
      // ---------------------------------------------------------- producer
      const bool leader = elect_one();
      const int nq = q1_valid ? 2 : 1;
      if (leader) {
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
      }
      pdl_wait();                                       // the inputs are written (programmatic launch)
      if (leader) {
        mbar_arrive_expect_tx(bars.q_full, nq * C::kTileBytes);
        for (int q = 0; q < nq; ++q)
          for (int hh = 0; hh < D / 64; ++hh)
            tma_load_4d(smem + C::kOffQ + q * C::kTileBytes + hh * C::kHalfBytes, &tmap_q, bars.q_full, hh * 64,
                        (qt0 + q) * BM, h, b);
      }
      int issued = 0;
      for (int j = 0; j < nt; ++j) {
        const int s = j % C::NS;
        const uint32_t par = ((j / C::NS) - 1) & 1;
        const int y = (jb + j) * BN;
        if (j >= C::NS && !mbar_wait_backoff_warp(bars.k_empty + s, par, abort_flag, wait_ns, kProducerSleepNs)) break;
        if (leader) {
          mbar_arrive_expect_tx(bars.k_full + s, C::kTileBytes);
          for (int hh = 0; hh < D / 64; ++hh)
            tma_load_4d(smem + C::kOffK + s * C::kTileBytes + hh * C::kHalfBytes, &tmap_k, bars.k_full + s,
                        hh * 64, y, hk, b);
        }
        if (j >= C::NS && !mbar_wait_backoff_warp(bars.v_empty + s, par, abort_flag, wait_ns, kProducerSleepNs)) {
          issued = 2 * j + 1;
          break;
        }
        if (leader) {
          mbar_arrive_expect_tx(bars.v_full + s, C::kTileBytes);
          for (int hh = 0; hh < D / 64; ++hh)
            tma_load_4d(smem + C::kOffV + s * C::kTileBytes + hh * C::kHalfBytes, &tmap_v, bars.v_full + s,
                        hh * 64, y, hk, b);
        }
        issued = 2 * j + 2;
      }
      if (*abort_flag) {
        // drain: wait (bounded) for every armed load so none lands after exit
        mbar_wait_drain(bars.q_full, 0, wait_ns);
        for (int u = (issued > 2 * C::NS ? issued - 2 * C::NS : 0); u < issued; ++u) {
          const int j = u / 2, s = j % C::NS;
          mbar_wait_drain((u % 2 == 0) ? bars.k_full + s : bars.v_full + s, (j / C::NS) & 1, wait_ns);
        }
      }
    } else if (warp == 9) {
      // ---------------------------------------------------------- S issuer
      // S0(0), S1(0), S0(1), S1(1), ... into the one S region; each waits
      // until the softmax warps have read the previous S.
      const bool leader = elect_one();
      const uint64_t dQ = sdesc(smem_u32(smem + C::kOffQ), 16, 1024, kSwizzle128B);
      const uint64_t dK = sdesc(smem_u32(smem + C::kOffK), 16, 1024, kSwizzle128B);
      const uint32_t tS = tbase + C::kColS;
      int last_q = -1, last_j = 0;
      bool ok = mbar_wait_warp(bars.q_full, 0, abort_flag, wait_ns);
      for (int j = 0; ok && j < nt; ++j) {
        const int s = j % C::NS;
        ok = mbar_wait_warp(bars.k_full + s, (j / C::NS) & 1, abort_flag, wait_ns);
        if (!ok) break;
        for (int q = 0; ok && q < 2; ++q) {
          if (j >= ntq[q]) continue;
          if (last_q >= 0) ok = mbar_wait_warp(bars.s_free + last_q, last_j & 1, abort_flag, wait_ns);
          if (!ok) break;
          tc_fence_after();
          const uint64_t a0 = dadd(dQ, q * C::kTileBytes), b0 = dadd(dK, s * C::kTileBytes);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk / 4) * C::kHalfBytes + (kk % 4) * 32;
              mma_bf16_ss(tS, dadd(a0, off), dadd(b0, off), C::kIdescS, kk > 0 ? 1u : 0u);
            }
            tc_commit(bars.s_full + q);
          }
          __syncwarp();
          last_q = q;
          last_j = j;
        }
        if (ok && leader) tc_commit(bars.k_empty + s);      // K slot free once these S MMAs are done
        __syncwarp();
      }
      if (!ok) {
        // drain the tensor pipe before tensor memory is released
        if (leader) tc_commit(bars.drain);
        __syncwarp();
        mbar_wait_drain(bars.drain, 0, wait_ns);
      }
    } else if (warp == 10) {
      // ---------------------------------------------------------- P.V issuer
      // P0.V(j), P1.V(j), ... each once its softmax warps have stored P.
      const bool leader = elect_one();
      const uint64_t dV = sdesc(smem_u32(smem + C::kOffV), C::kHalfBytes, 1024, kSwizzle128B);
      bool ok = true;
      for (int j = 0; ok && j < nt; ++j) {
        const int s = j % C::NS;
        ok = mbar_wait_warp(bars.v_full + s, (j / C::NS) & 1, abort_flag, wait_ns);
        if (!ok) break;
        for (int q = 0; ok && q < 2; ++q) {
          if (j >= ntq[q]) continue;
          ok = mbar_wait_warp(bars.p_full + q, j & 1, abort_flag, wait_ns);
          if (!ok) break;
          tc_fence_after();
          const uint64_t b0 = dadd(dV, s * C::kTileBytes);
          const uint32_t tO = tbase + C::kColO0 + q * D, tP = tbase + C::kColP0 + q * 64;
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_bf16_ts(tO, tP + kk * 8, dadd(b0, kk * 16 * 128), C::kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
            tc_commit(bars.o_done + q);
          }
          __syncwarp();
        }
        if (ok && leader) tc_commit(bars.v_empty + s);      // V slot free once these P.V MMAs are done
        __syncwarp();
      }
      if (!ok) {
        if (leader) tc_commit(bars.drain + 1);
        __syncwarp();
        mbar_wait_drain(bars.drain + 1, 0, wait_ns);
      }
    }
  } else {
    reg_alloc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax
    const int q = warp / 4;
    const int r = (warp % 4) * 32 + lane;                      // row within the query tile
    const uint32_t lane_addr = tbase + (((warp % 4) * 32) << 16);
    const int qt = qt0 + q;
    const float c = softmax_scale_log2<D>();
    const uint32_t ocol = C::kColO0 + q * D;
    float m_use = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntq[q]; ++j) {
      if (!mbar_wait_warp(bars.s_full + q, j & 1, abort_flag, wait_ns)) {
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
      // keys this row may not see: past Lkv (the zero fill of a ragged last
      // tile) and, causal, past its position qt*128 + r + Lkv - Lq
      int lim = Lkv - (jb + j) * BN;
      if (causal) lim = min(lim, qt * BM + r + work.coff - (jb + j) * BN + 1);
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
      float alpha = 1.f;
      bool resc = false;
      if (m_t > m_use + kRescaleThreshold) {
        alpha = ex2_approx(m_use - m_t);
        m_use = m_t;
        resc = (j > 0);
      }
      const float negm = -m_use;
      float sp[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) sp[i] = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        float p0, p1;
        fma2(p0, p1, sv[2 * i], sv[2 * i + 1], c, c, negm, negm);
        p0 = ex2_approx(p0);
        p1 = ex2_approx(p1);
        const int a = i % 4;
        add2(sp[2 * a], sp[2 * a + 1], sp[2 * a], sp[2 * a + 1], p0, p1);
        pk[i] = pack_bf16x2(p0, p1);
      }
      const float sum = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
      l = l * alpha + sum;
      if (j > 0) {
        if (!mbar_wait_warp(bars.o_done + q, (j - 1) & 1, abort_flag, wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, resc)) {     // rare: one 32-column chunk at a time
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(lane_addr + ocol + 32 * cc, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float a = __uint_as_float(o[i]), bb = __uint_as_float(o[i + 1]);
            mul2(a, bb, a, bb, alpha, alpha);
            o[i] = __float_as_uint(a);
            o[i + 1] = __float_as_uint(bb);
          }
          tmem_st32(lane_addr + ocol + 32 * cc, o);
        }
      }
      uint32_t p_lo[32], p_hi[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        p_lo[i] = pk[i];
        p_hi[i] = pk[32 + i];
      }
      tmem_st32(lane_addr + C::kColP0 + q * 64, p_lo);
      tmem_st32(lane_addr + C::kColP0 + q * 64 + 32, p_hi);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bars.p_full + q);
    }
    // ---- epilogue: O / l
    const bool row_in = qt * BM + r < Lq;               // rows past Lq (a ragged last tile) are not stored
    // split-KV: this CTA's partial result of the row -- O unnormalised (in
    // units of 2^m_use, as is l), m_use (-inf if no key was visible) and l --
    // goes to split sp's slot; a combine pass forms O
    const bool split = work.nsplit > 1;
    const long long prow = ((long long)sp * work.nbh + bhq) * padded_len_dev(Lq) + (long long)qt * BM + r;
    if (split && ok && ntq[q] == 0 && (q == 0 || q1_valid) && row_in)
      *reinterpret_cast<float2*>(part.ml + 2 * prow) = make_float2(-INFINITY, 0.f);
    if (ok && ntq[q] > 0 && mbar_wait_warp(bars.o_done + q, (ntq[q] - 1) & 1, abort_flag, wait_ns)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const long long obase = obase0 + ((long long)qt * BM + r) * so.t;
      if (split && row_in) *reinterpret_cast<float2*>(part.ml + 2 * prow) = make_float2(m_use, l);
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(lane_addr + ocol + 32 * cc, o);
        tmem_ld_wait(o);
        if (!row_in) continue;
        if (split) {
          float4* dst = reinterpret_cast<float4*>(part.o + prow * D + 32 * cc);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                 __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
          continue;
        }
        if constexpr (OUT32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out_ptr) + obase + 32 * cc);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                 __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l);
        } else {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out_ptr) + obase + 32 * cc);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
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

template <int D, bool OUT32>
cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, void* o, const Strides& so,
                     const Dims& dm, int causal, int nsplit, const SplitOut& part, cudaStream_t s) {
  using C = CfgBF16<D>;
  // kernel attributes are per device: set them on the first launch on each
  static std::atomic<bool> attr_done[kMaxDevices];
  cudaError_t e = once_per_device(attr_done, [] {
    // The warpgroup register split assumes kLaunchRegs registers per thread at
    // launch; with fewer, a setmaxnreg increase could never be satisfied.
    cudaFuncAttributes fa;
    cudaError_t r = cudaFuncGetAttributes(&fa, attn_bf16_kernel<D, OUT32>);
    if (r != cudaSuccess) return r;
    if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(attn_bf16_kernel<D, OUT32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  int ctas = 0;
  const AttnWork work = make_attn_work(dm.B, dm.H, dm.Lq, dm.Lkv, causal, device_sm_count(), &ctas, nsplit);
  // a programmatic dependent launch: the CTAs' set-up overlaps the end of
  // the kernel before; the producer waits for it before its first load
  cudaLaunchAttribute attr;
  const cudaLaunchConfig_t cfg = pdl_launch_config(dim3(ctas), dim3(kThreads), C::kSmemBytes, s, &attr);
  e = cudaLaunchKernelEx(&cfg, attn_bf16_kernel<D, OUT32>, tq, tk, tv, o, dm.H, dm.Hkv, dm.Lq, dm.Lkv,
                                     causal, work, part, so, kWaitLimitNs);
  if (e == cudaSuccess && work.nsplit > 1) e = launch_splitkv_combine(part, work.nsplit, dm, o, so, OUT32, s);
  return e;
}

}  // namespace

cudaError_t launch_attn_bf16(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, void* o,
                             const Strides& so, const Dims& dm, int causal, bool out_f32, int nsplit,
                             const SplitOut& part, cudaStream_t s) {
  if (dm.d == 64) return out_f32 ? launch_d<64, true>(tq, tk, tv, o, so, dm, causal, nsplit, part, s)
                                 : launch_d<64, false>(tq, tk, tv, o, so, dm, causal, nsplit, part, s);
  return out_f32 ? launch_d<128, true>(tq, tk, tv, o, so, dm, causal, nsplit, part, s)
                 : launch_d<128, false>(tq, tk, tv, o, so, dm, causal, nsplit, part, s);
}

cudaError_t attn_bf16_read_error(int* out) { return read_and_clear_device_error(out); }

}  // namespace sa
