// Host check of the attention work schedules (work.cuh), no GPU needed.
//
// For many shapes, causal or not, and grid sizes:
//  * stream-K: the pair prefix sums equal brute-force sums of the pairs' key
//    tiles; walking every CTA's range covers every (pair, key tile) item once;
//    units are whole pairs exactly when slot == -1, and a partial unit's slot
//    is 2c (it begins CTA c's range) or 2c + 1 (it ends it); the cut table
//    lists every cut pair once, and its segments are exactly the partial
//    units of that pair, in CTA order;
//  * split-KV: the shares of each pair tile its key range;
//  * with a query length different from the key length, each query tile's
//    key-tile count is the number of key tiles holding a key its rows may see
//    (brute force over rows and keys under the bottom-right causal mask).
// Prints "OK" and returns 0, or prints the first failure and returns 1.
#include <cstdio>
#include <vector>

#include "../../quantized_attention_x16_gb300/csrc/work.cuh"

using namespace sa;

static int fail(const char* what, int B, int H, int L, int causal, int C) {
  std::printf("FAIL %s: B=%d H=%d L=%d causal=%d C=%d\n", what, B, H, L, causal, C);
  return 1;
}

static int check_key_counts(int Lq, int Lkv, int causal) {
  int ctas = 0;
  const AttnWork w = make_attn_work(1, 1, Lq, Lkv, causal, 152, &ctas);
  for (int qt = 0; qt < w.nqt; ++qt) {
    int need = 0;                                 // key tiles holding a key some valid row may see
    for (int r = qt * 128; r < qt * 128 + 128 && r < Lq; ++r) {
      const int last = causal ? r + (Lkv - Lq) : Lkv - 1;
      const int tiles = last / 128 + 1;
      if (tiles > need) need = tiles;
    }
    if (q_tile_keys(w, qt) != need) return fail("key tiles of a query tile", Lq, Lkv, qt, causal, 0);
  }
  return 0;
}

static int check_streamk(int B, int H, int L, int Lkv, int causal, int sms) {
  int C = 0;
  AttnWork w = make_streamk_work(B, H, L, Lkv, causal, sms, &C);
  const long long npairs = (long long)w.ppr * w.nbh;
  long long acc = 0;
  for (long long p = 0; p < npairs; ++p) {
    if (sk_prefix(w, p) != acc) return fail("prefix", B, H, L, causal, C);
    acc += sk_pair_tiles(w, p);
  }
  if (acc != w.items) return fail("items", B, H, L, causal, C);
  for (long long x = 0; x < w.items; x += 1 + w.items / 97) {   // pair_of on a sample of items
    const long long p = sk_pair_of(w, x);
    if (sk_prefix(w, p) > x || x >= sk_prefix(w, p) + sk_pair_tiles(w, p)) return fail("pair_of", B, H, L, causal, C);
  }
  std::vector<int> seen(w.items, 0);
  // partial units per pair: (cta, slot)
  std::vector<std::vector<std::pair<int, int>>> parts(npairs);
  for (int c = 0; c < C; ++c) {
    UnitIter it;
    sk_iter_init(w, c, it);
    AttnUnitRef u;
    int k = 0;
    long long prev_end = w.sk_x0[c];
    while (sk_next(w, c, it, u)) {
      // recover the pair from the unit's head and query tile
      long long p = -1;
      for (long long q = 0; q < npairs && p < 0; ++q) {
        int bh, qt0, nq;
        pair_head(w, q, bh, qt0, nq);
        if (bh == u.bh && qt0 == u.qt0) p = q;
      }
      if (p < 0) return fail("unit pair", B, H, L, causal, C);
      const int nt = sk_pair_tiles(w, p);
      const int cnt = u.n[0] > u.n[1] ? u.n[0] : u.n[1];
      if (sk_prefix(w, p) + u.jb != prev_end) return fail("contiguous", B, H, L, causal, C);
      for (int j = 0; j < cnt; ++j) ++seen[sk_prefix(w, p) + u.jb + j];
      prev_end = sk_prefix(w, p) + u.jb + cnt;
      const bool whole = u.jb == 0 && cnt == nt;
      if (whole != (u.slot == -1)) return fail("slot -1", B, H, L, causal, C);
      if (!whole) {
        const int want = 2 * c + (sk_prefix(w, p) + u.jb == w.sk_x0[c] ? 0 : 1);
        if (u.slot != want) return fail("slot", B, H, L, causal, C);
        parts[p].push_back({c, u.slot});
      }
      // per query tile counts: never past the tiles the query tile may see
      if (u.jb + u.n[0] > q_tile_keys(w, u.qt0)) return fail("causal range", B, H, L, causal, C);
      if (u.nq == 2 && u.jb + u.n[1] > q_tile_keys(w, u.qt0 + 1)) return fail("causal range 1", B, H, L, causal, C);
      ++k;
    }
    if (prev_end != w.sk_x0[c + 1]) return fail("range end", B, H, L, causal, C);
  }
  for (long long x = 0; x < w.items; ++x)
    if (seen[x] != 1) return fail("coverage", B, H, L, causal, C);
  StreamKCuts cuts;
  make_streamk_cuts(w, C, &cuts);
  int ncut = 0;
  for (long long p = 0; p < npairs; ++p) ncut += parts[p].empty() ? 0 : 1;
  if (ncut != cuts.n) return fail("cut count", B, H, L, causal, C);
  for (int i = 0; i < cuts.n; ++i) {
    const int* e = cuts.e[i];
    long long p = -1;
    for (long long q = 0; q < npairs && p < 0; ++q) {
      int bh, qt0, nq;
      pair_head(w, q, bh, qt0, nq);
      if (bh == e[0] && qt0 == e[1]) p = q;
    }
    if (p < 0 || parts[p].size() != (size_t)(e[4] - e[3] + 1)) return fail("cut segments", B, H, L, causal, C);
    for (int kk = 0; kk <= e[4] - e[3]; ++kk) {
      const int slot = 2 * (e[3] + kk) + (kk == 0 ? e[5] : 0);
      if (parts[p][kk].first != e[3] + kk || parts[p][kk].second != slot) return fail("cut slot", B, H, L, causal, C);
    }
  }
  return 0;
}

static int check_split(int B, int H, int L, int Lkv, int causal, int nsplit) {
  AttnWork w;
  int ctas = 0;
  w = make_attn_work(B, H, L, Lkv, causal, 152, &ctas, nsplit);
  for (int p = 0; p < w.ppr * w.nbh; ++p) {
    const int pi = causal ? w.ppr - 1 - p / w.nbh : p % w.ppr;
    const int qt0 = 2 * pi;
    int full[2] = {q_tile_keys(w, qt0), qt0 + 1 < w.nqt ? q_tile_keys(w, qt0 + 1) : 0};
    int next[2] = {0, 0};
    for (int s = 0; s < w.nsplit; ++s) {
      int n[2] = {full[0], full[1]};
      const int jb = split_range(s, w.nsplit, n);
      for (int q = 0; q < 2; ++q) {
        if (n[q] > 0 && jb != next[q]) return fail("split contiguous", B, H, L, causal, nsplit);
        next[q] += n[q];
      }
    }
    if (next[0] != full[0] || next[1] != full[1]) return fail("split coverage", B, H, L, causal, nsplit);
  }
  return 0;
}

int main() {
  // B, H, Lq, Lkv (Lkv >= Lq: the causal mask needs it)
  const int shapes[][4] = {{1, 1, 128, 128}, {1, 1, 200, 200}, {1, 2, 640, 640}, {2, 16, 4096, 4096},
                           {1, 32, 8192, 8192}, {1, 3, 1000, 1000}, {3, 5, 1536, 1536}, {1, 8, 16384, 16384},
                           {1, 24, 16384, 16384}, {2, 1, 384, 384}, {4, 8, 1, 4096}, {2, 3, 16, 1000},
                           {1, 2, 200, 8192}, {3, 4, 300, 333}, {1, 1, 128, 32768}, {8, 4, 129, 2048}};
  const int grids[] = {1, 2, 7, 64, 148, 152, 160};
  for (auto& sh : shapes)
    for (int causal = 0; causal < 2; ++causal) {
      if (check_key_counts(sh[2], sh[3], causal)) return 1;
      for (int g : grids)
        if (check_streamk(sh[0], sh[1], sh[2], sh[3], causal, g)) return 1;
      for (int ns : {2, 3, 4, 7, 16})
        if (check_split(sh[0], sh[1], sh[2], sh[3], causal, ns)) return 1;
    }
  std::printf("OK\n");
  return 0;
}
