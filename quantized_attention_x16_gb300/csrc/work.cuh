// work.cuh -- the work list of the fused attention kernels.
//
// One CTA per unit.  A unit is normally a "pair": two consecutive 128-row
// query tiles of one (batch, head), which share every K/V tile the CTA loads.
// Units are numbered in dispatch order:
//  * non-causal: head-major (the CTAs that run together share K/V in L2);
//  * causal: heaviest first across all heads (pair p of a head sees 2p + 2
//    key tiles), so the short units fill the end of the grid.
// When the equal-cost pairs of a non-causal problem leave a last wave that
// would occupy at most half of the SMs, the pairs of that wave are split into
// single-tile units: two singles run side by side on two SMs in well under
// the time of one pair, so the tail shrinks.
// Split-KV (nsplit > 1, for problems with too few pairs to fill the SMs):
// unit u is split u % nsplit of pair u / nsplit; the split covers a contiguous
// share of the pair's key tiles (see split_range) and leaves a partial result
// for a combine pass.
#pragma once

#include <cuda_runtime.h>

namespace sa {

struct AttnWork {
  int nqt;     // 128-row query tiles per head
  int ppr;     // pair slots per head, ceil(nqt / 2)
  int nbh;     // B * H
  int npair;   // units [0, npair) are pairs; then 2 * (ppr * nbh - npair) singles
  int causal;
  int nsplit;  // key-range splits per pair (1: none)
};

// Host: the work list for a problem and the number of CTAs to launch.
inline AttnWork make_attn_work(int B, int H, int L, int causal, int num_sms, int* ctas, int nsplit = 1) {
  AttnWork w;
  w.nqt = (L + 127) / 128;   // a ragged last tile counts as a tile
  w.ppr = (w.nqt + 1) / 2;
  w.nbh = B * H;
  w.causal = causal;
  w.nsplit = nsplit > 1 ? nsplit : 1;
  const long long pairs = (long long)w.ppr * w.nbh;
  if (w.nsplit > 1) {
    w.npair = (int)pairs;
    *ctas = (int)(pairs * w.nsplit);
    return w;
  }
  long long split = 0;
  if (!causal && (w.nqt % 2) == 0 && num_sms > 0) {
    const long long rem = pairs % num_sms;
    if (rem > 0 && 2 * rem <= num_sms) split = rem;
  }
  w.npair = (int)(pairs - split);
  *ctas = (int)(pairs + split);
  return w;
}

// Splits of the key range for split-KV, chosen only while the pairs alone
// leave at least half of the SMs idle, and only as far as every share keeps
// kMinShareTiles key tiles: a CTA costs about 6 us of fixed work (prologue,
// pipeline ramp, epilogue) besides ~1 us per key tile, and the combine pass
// about 6 us more, so shorter shares lose time (measured on the GB300:
// B1 H8 L1024, eight key tiles per query tile, takes 19 us unsplit and 24-25
// us in two or four shares).  Returns 1 (no split) otherwise.
constexpr int kMinShareTiles = 16;
inline int choose_nsplit(int B, int H, int L, int num_sms) {
  const int nkt = (L + 127) / 128;
  const long long pairs = (long long)((nkt + 1) / 2) * B * H;
  if (num_sms <= 0 || pairs <= 0 || 2 * pairs > num_sms) return 1;
  int s = (int)(num_sms / pairs);
  if (s > nkt / kMinShareTiles) s = nkt / kMinShareTiles;
  if (s > 16) s = 16;
  return s > 1 ? s : 1;
}

__device__ __forceinline__ int padded_len_dev(int L) { return (L + 127) & ~127; }

// Device: the key tiles [jb, jb + n[q]) that split `sp` of `nsplit` covers for
// each query tile q, given each query tile's full count n[q] (query tile 1
// never has fewer than query tile 0): the union of the pair's key tiles is
// cut into nsplit near-equal contiguous pieces.
__device__ __forceinline__ int split_range(int sp, int nsplit, int (&n)[2]) {
  const int nun = n[1] > n[0] ? n[1] : n[0];
  const int jb = sp * nun / nsplit, je = (sp + 1) * nun / nsplit;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int e = n[q] < je ? n[q] : je;
    n[q] = e > jb ? e - jb : 0;
  }
  return jb;
}

// Device: (b*H + h, first query tile, number of query tiles, split) of unit u.
__device__ __forceinline__ void attn_unit(const AttnWork& w, int u, int& bh, int& qt0, int& nq, int& sp) {
  sp = u % w.nsplit;
  u /= w.nsplit;
  const int p = u < w.npair ? u : w.npair + (u - w.npair) / 2;   // pair slot in dispatch order
  int pi;
  if (w.causal) {
    pi = w.ppr - 1 - p / w.nbh;
    bh = p % w.nbh;
  } else {
    pi = p % w.ppr;
    bh = p / w.ppr;
  }
  qt0 = 2 * pi;
  if (u < w.npair) {
    nq = (qt0 + 1 < w.nqt) ? 2 : 1;
  } else {
    qt0 += (u - w.npair) & 1;
    nq = 1;
  }
}

}  // namespace sa
