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

constexpr int kMaxStreamKCtas = 160;   // persistent grid cap (one CTA per SM)
constexpr int kMaxStreamKGroups = 512;  // causal stream-K: query-tile pairs per head (Lq <= 128k)

struct AttnWork {
  int nqt;     // 128-row query tiles per head (from Lq)
  int nkt;     // 128-key tiles per head (from Lkv)
  int coff;    // causal: key j is visible to query i iff j <= i + coff (coff = Lkv - Lq)
  int ppr;     // pair slots per head, ceil(nqt / 2)
  int nbh;     // B * H
  int npair;   // units [0, npair) are pairs; then 2 * (ppr * nbh - npair) singles
  int causal;
  int nsplit;  // key-range splits per pair (1: none)
  int streamk; // 1: persistent CTAs over equal ranges of (pair, key tile) items
  long long items;   // stream-K: total items (key tiles over all pairs)
  int sk_x0[kMaxStreamKCtas + 1];   // stream-K: first item of CTA c's range (c = 0..C)
  long long sk_grp[kMaxStreamKGroups + 1];   // causal stream-K: items before pair group g
};

// Key tiles query tile qt needs: all of them, or under the causal mask up to
// the tile holding the last key its last row may see.
__host__ __device__ inline int q_tile_keys(const AttnWork& w, int qt) {
  if (!w.causal) return w.nkt;
  const long long n = ((long long)qt * 128 + 127 + w.coff) / 128 + 1;
  return (int)(n < w.nkt ? n : w.nkt);
}

// Host: the work list for a problem and the number of CTAs to launch.
inline AttnWork make_attn_work(int B, int H, int Lq, int Lkv, int causal, int num_sms, int* ctas, int nsplit = 1) {
  AttnWork w;
  w.nqt = (Lq + 127) / 128;   // a ragged last tile counts as a tile
  w.nkt = (Lkv + 127) / 128;
  w.coff = Lkv - Lq;
  w.ppr = (w.nqt + 1) / 2;
  w.nbh = B * H;
  w.causal = causal;
  w.nsplit = nsplit > 1 ? nsplit : 1;
  w.streamk = 0;
  w.items = 0;
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

// ---------------------------------------------------------------- stream-K
// Persistent scheduling: the pairs (in dispatch order, no singles) are laid
// end to end as "items", one per key tile of the pair's union key range, and
// CTA c of C takes items [c*T/C, (c+1)*T/C).  Every SM then gets the same
// number of key-tile steps; a pair cut by a range boundary is computed in
// segments whose partial results a combine pass merges.

// Key tiles of pair slot p (dispatch order): the union of its query tiles'
// ranges (causal: up to the diagonal of its second query tile).
__host__ __device__ inline int sk_pair_tiles(const AttnWork& w, long long p) {
  if (!w.causal) return w.nkt;
  const int pi = w.ppr - 1 - (int)(p / w.nbh);
  const int qt0 = 2 * pi;
  return q_tile_keys(w, qt0 + 1 < w.nqt ? qt0 + 1 : qt0);
}

// Items before pair slot p.  Causal: the pairs of group g (index pi =
// ppr-1-g in every head) all have the same tile count; sk_grp[g] holds the
// items of the groups before g (filled on the host).
__host__ __device__ inline long long sk_prefix(const AttnWork& w, long long p) {
  if (!w.causal) return p * w.nkt;
  const long long g = p / w.nbh;
  return w.sk_grp[g] + (p - g * w.nbh) * sk_pair_tiles(w, p);
}

// The pair holding item x (0 <= x < items).
__host__ __device__ inline long long sk_pair_of(const AttnWork& w, long long x) {
  long long lo = 0, hi = (long long)w.ppr * w.nbh - 1;
  while (lo < hi) {                               // last p with prefix(p) <= x
    const long long mid = (lo + hi + 1) / 2;
    if (sk_prefix(w, mid) <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// First item of CTA c's range, and the CTA whose range holds item x.
__host__ __device__ inline long long sk_start(const AttnWork& w, long long c, long long C) {
  return c * w.items / C;
}
__host__ __device__ inline long long sk_cta_of(const AttnWork& w, long long x, long long C) {
  return ((x + 1) * C - 1) / w.items;
}

// One unit of a CTA's work: query tiles qt0 (and qt0 + 1 if nq == 2) of head
// bh, key tiles [jb, jb + n[q]) for query tile q, and where its result goes:
// slot -1 = O itself; split-KV = share index; stream-K = partial slot
// 2c (the CTA's first unit) or 2c + 1 (its last).
struct AttnUnitRef {
  int bh, qt0, nq, jb, n[2], slot;
};

__host__ __device__ inline void pair_head(const AttnWork& w, long long p, int& bh, int& qt0, int& nq) {
  int pi;
  if (w.causal) {
    pi = w.ppr - 1 - (int)(p / w.nbh);
    bh = (int)(p % w.nbh);
  } else {
    pi = (int)(p % w.ppr);
    bh = (int)(p / w.ppr);
  }
  qt0 = 2 * pi;
  nq = (qt0 + 1 < w.nqt) ? 2 : 1;
}

// Walks the units of one CTA; every warp role of the CTA walks the same list.
struct UnitIter {
  int x, xe, p;     // stream-K: next item, end of range, its pair
  int x0;           // stream-K: first item of the range
  int done;
};

// Host: the stream-K work list (pairs only) and its grid, one CTA per SM (or
// per item when there are fewer items).
// The ranges are fixed on the host (first items in sk_x0, 32-bit: stream-K
// is used only while the item count fits).
inline AttnWork make_streamk_work(int B, int H, int Lq, int Lkv, int causal, int num_sms, int* ctas) {
  AttnWork w = make_attn_work(B, H, Lq, Lkv, causal, num_sms, ctas, 2);   // pairs only
  w.nsplit = 1;
  w.streamk = 1;
  if (causal) {
    w.sk_grp[0] = 0;
    for (int g = 0; g < w.ppr && g < kMaxStreamKGroups; ++g)
      w.sk_grp[g + 1] = w.sk_grp[g] + (long long)w.nbh * sk_pair_tiles(w, (long long)g * w.nbh);
  }
  w.items = causal ? w.sk_grp[w.ppr] : sk_prefix(w, (long long)w.ppr * w.nbh);
  long long c = w.items < num_sms ? w.items : num_sms;
  if (c > kMaxStreamKCtas) c = kMaxStreamKCtas;
  if (c < 1) c = 1;
  for (long long i = 0; i <= c; ++i) w.sk_x0[i] = (int)sk_start(w, i, c);
  *ctas = (int)c;
  return w;
}
inline bool streamk_fits(int B, int H, int Lq, int Lkv, int causal) {
  const long long nqt = (Lq + 127) / 128, nkt = (Lkv + 127) / 128;
  if (causal && (nqt + 1) / 2 > kMaxStreamKGroups) return false;
  return (nqt + 1) / 2 * (long long)B * H * nkt < (1ll << 31);
}

// The pairs that range boundaries cut, for the combine pass: per cut pair its
// head, first query tile and query-tile count, the first and last CTA whose
// range meets it (cta0, cta1), and whether it is cta0's last unit (cta0_last;
// otherwise it begins cta0's range).  Segment k of the pair sits in slot
// 2 (cta0 + k) + (k == 0 && cta0_last).
struct StreamKCuts {
  int n;
  int e[kMaxStreamKCtas][6];   // bh, qt0, nq, cta0, cta1, cta0_last
};
inline void make_streamk_cuts(const AttnWork& w, int C, StreamKCuts* cuts) {
  cuts->n = 0;
  auto cta_of = [&](long long x) {             // last CTA whose range starts at or before x
    int c = 0;
    while (c + 1 < C && w.sk_x0[c + 1] <= x) ++c;
    return c;
  };
  for (int c = 1; c < C; ++c) {
    const long long x = w.sk_x0[c];
    if (x >= w.items) break;
    const long long p = sk_pair_of(w, x), P = sk_prefix(w, p);
    if (x == P || w.sk_x0[c - 1] > P) continue;   // no cut, or an earlier boundary cut this pair
    int* e = cuts->e[cuts->n++];
    const int nt = sk_pair_tiles(w, p);
    int pi;
    if (w.causal) {
      pi = w.ppr - 1 - (int)(p / w.nbh);
      e[0] = (int)(p % w.nbh);
    } else {
      pi = (int)(p % w.ppr);
      e[0] = (int)(p / w.ppr);
    }
    e[1] = 2 * pi;
    e[2] = 2 * pi + 1 < w.nqt ? 2 : 1;
    e[3] = cta_of(P);
    e[4] = cta_of(P + nt - 1);
    e[5] = w.sk_x0[e[3]] < P ? 1 : 0;
  }
}

// Splits of the key range for split-KV, chosen only while the pairs alone
// leave at least half of the SMs idle, and only as far as every share keeps
// kMinShareTiles key tiles: a CTA costs about 6 us of fixed work (prologue,
// pipeline ramp, epilogue) besides ~1 us per key tile, and the combine pass
// about 6 us more, so shorter shares lose time (measured on the GB300:
// B1 H8 L1024, eight key tiles per query tile, takes 19 us unsplit and 24-25
// us in two or four shares).  Returns 1 (no split) otherwise.
constexpr int kMinShareTiles = 16;
inline int choose_nsplit(int B, int H, int Lq, int Lkv, int num_sms) {
  const int nqt = (Lq + 127) / 128, nkt = (Lkv + 127) / 128;
  const long long pairs = (long long)((nqt + 1) / 2) * B * H;
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
__host__ __device__ inline int split_range(int sp, int nsplit, int (&n)[2]) {
  const int nun = n[1] > n[0] ? n[1] : n[0];
  const int jb = sp * nun / nsplit, je = (sp + 1) * nun / nsplit;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int e = n[q] < je ? n[q] : je;
    n[q] = e > jb ? e - jb : 0;
  }
  return jb;
}

// Stream-K range walk of CTA `cta` (host-callable, for tests of the schedule).
__host__ __device__ inline void sk_iter_init(const AttnWork& w, int cta, UnitIter& it) {
  it.done = 0;
  it.x0 = w.sk_x0[cta];
  it.x = it.x0;
  it.xe = w.sk_x0[cta + 1];
  it.p = it.x < it.xe ? (int)sk_pair_of(w, it.x) : 0;
}
__host__ __device__ inline bool sk_next(const AttnWork& w, int cta, UnitIter& it, AttnUnitRef& u) {
  if (it.x >= it.xe) return false;
  const int P = (int)sk_prefix(w, it.p);
  const int nt = sk_pair_tiles(w, it.p);
  const int a = it.x - P;
  const int b = it.xe - P < nt ? it.xe - P : nt;
  pair_head(w, it.p, u.bh, u.qt0, u.nq);
  u.jb = a;
  const int n0 = q_tile_keys(w, u.qt0);
  const int n1 = u.nq == 2 ? q_tile_keys(w, u.qt0 + 1) : 0;
  u.n[0] = (n0 < b ? n0 : b) > a ? (n0 < b ? n0 : b) - a : 0;
  u.n[1] = (n1 < b ? n1 : b) > a ? (n1 < b ? n1 : b) - a : 0;
  u.slot = (a == 0 && b == nt) ? -1 : 2 * cta + (it.x == it.x0 ? 0 : 1);
  it.x = P + b;
  ++it.p;
  return true;
}

__device__ __forceinline__ void unit_iter_init(const AttnWork& w, UnitIter& it) {
  it.done = 0;
  if (w.streamk) sk_iter_init(w, blockIdx.x, it);
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

namespace sa {

// Next unit of this CTA (false when none is left).
__device__ __forceinline__ bool unit_next(const AttnWork& w, UnitIter& it, AttnUnitRef& u) {
  if (it.done) return false;
  if (!w.streamk) {
    // one unit: this CTA's entry of the work list (a share of it under split-KV)
    int sp;
    attn_unit(w, (int)blockIdx.x, u.bh, u.qt0, u.nq, sp);
    u.n[0] = q_tile_keys(w, u.qt0);
    u.n[1] = u.nq == 2 ? q_tile_keys(w, u.qt0 + 1) : 0;
    u.jb = w.nsplit > 1 ? split_range(sp, w.nsplit, u.n) : 0;
    u.slot = w.nsplit > 1 ? sp : -1;
    it.done = 1;
    return true;
  }
  return sk_next(w, (int)blockIdx.x, it, u);
}

}  // namespace sa
