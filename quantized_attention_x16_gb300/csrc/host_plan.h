// host_plan.h -- the chunking of sa_attn_fwd_host (host code only, no CUDA
// calls: the SM count is a parameter, so a CPU program can check the plan).
//
// The problem is cut into chunks of consecutive (batch, kv head) pairs, each
// with all G = H / Hkv of its query heads.  A chunk's attention launch has
// units_per_pair CTAs per pair; the pipeline is bound by the host link, and
// what no copy-in overlaps is the compute and copy-out of the last chunk, so
// the library's chunking of the NVFP4 path lets the last chunks shrink and
// gives a chunk whose CTAs would leave half of the SMs idle split-KV shares.
#pragma once

#include <vector>

namespace sa {

constexpr int kTailMinShareTiles = 8;   // split-KV shares of the shrinking last chunks

// Attention CTAs of one (batch, kv head) pair: its G heads' query-tile pairs.
inline long long units_per_pair(int G, int L) { return (long long)G * (((L + 127) / 128 + 1) / 2); }

// Pairs per chunk: the most whose attention CTAs fit in one wave on the SMs
// (a chunk's kernels then take about one CTA lifetime), and at least two
// chunks when there are two pairs or more.
inline int default_chunk_pairs(int B, int H, int Hkv, int L, int sms) {
  const int G = H / Hkv, pairs = B * Hkv;
  const long long units = units_per_pair(G, L);
  long long n = sms / (units > 0 ? units : 1);
  if (n < 1) n = 1;
  if (pairs >= 2 && n > (pairs + 1) / 2) n = (pairs + 1) / 2;
  return (int)n;
}

// Split-KV shares for a chunk of n pairs in the library's chunking: enough to
// fill the SMs when its CTAs would leave half of them idle, each share keeping
// kTailMinShareTiles key tiles, at most 16.
inline int chunk_nsplit(int n, int G, int L, int sms) {
  const int nkt = (L + 127) / 128;
  const long long units = (long long)n * units_per_pair(G, L);
  if (sms <= 0 || units <= 0 || 2 * units > sms) return 1;
  long long sp = sms / units;
  if (sp > nkt / kTailMinShareTiles) sp = nkt / kTailMinShareTiles;
  if (sp > 16) sp = 16;
  return sp > 1 ? (int)sp : 1;
}

struct Chunk {
  int n, nsplit;
};

// The chunks in order.  A caller's chunk size, or the BF16 path: chunks of
// chunk_pairs (default n; the last one ragged), no split-KV.  The library's
// chunking of the NVFP4 path: chunks of n pairs, the last ones shrinking by
// halves down to min(2, n) pairs (built from the end: 2, 4, 8, ... capped at
// n), split-KV where chunk_nsplit says so.
inline std::vector<Chunk> chunk_plan(int B, int H, int Hkv, int L, int chunk_pairs, bool fp4, int sms) {
  const int pairs = B * Hkv, G = H / Hkv;
  const int n = default_chunk_pairs(B, H, Hkv, L, sms);
  std::vector<Chunk> plan;
  if (chunk_pairs > 0 || !fp4) {
    const int m = chunk_pairs > 0 ? chunk_pairs : n;
    for (int p0 = 0; p0 < pairs; p0 += m) plan.push_back(Chunk{pairs - p0 < m ? pairs - p0 : m, 1});
    return plan;
  }
  int rem = pairs, size = n < 2 ? n : 2;
  while (rem > 0) {
    const int t = size < rem ? size : rem;
    plan.push_back(Chunk{t, chunk_nsplit(t, G, L, sms)});
    rem -= t;
    size = 2 * size < n ? 2 * size : n;
  }
  for (size_t i = 0, j = plan.size() - 1; i < j; ++i, --j) {
    const Chunk c = plan[i];
    plan[i] = plan[j];
    plan[j] = c;
  }
  return plan;
}

}  // namespace sa
