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
#pragma once

#include <cuda_runtime.h>

namespace sa {

struct AttnWork {
  int nqt;     // 128-row query tiles per head
  int ppr;     // pair slots per head, ceil(nqt / 2)
  int nbh;     // B * H
  int npair;   // units [0, npair) are pairs; then 2 * (ppr * nbh - npair) singles
  int causal;
};

// Host: the work list for a problem and the number of CTAs to launch.
inline AttnWork make_attn_work(int B, int H, int L, int causal, int num_sms, int* ctas) {
  AttnWork w;
  w.nqt = (L + 127) / 128;   // a ragged last tile counts as a tile
  w.ppr = (w.nqt + 1) / 2;
  w.nbh = B * H;
  w.causal = causal;
  const long long pairs = (long long)w.ppr * w.nbh;
  long long split = 0;
  if (!causal && (w.nqt % 2) == 0 && num_sms > 0) {
    const long long rem = pairs % num_sms;
    if (rem > 0 && 2 * rem <= num_sms) split = rem;
  }
  w.npair = (int)(pairs - split);
  *ctas = (int)(pairs + split);
  return w;
}

// Device: (b*H + h, first query tile, number of query tiles) of unit u.
__device__ __forceinline__ void attn_unit(const AttnWork& w, int u, int& bh, int& qt0, int& nq) {
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
