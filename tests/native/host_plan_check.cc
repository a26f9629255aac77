// Host check of the chunking of sa_attn_fwd_host (host_plan.h), no GPU.
//
// For many problem shapes, SM counts and chunk requests:
//  * the chunks cover the (batch, kv head) pairs once, in order;
//  * a caller's chunk size (or the BF16 path) gives equal chunks, the last
//    one ragged, and no split-KV;
//  * the library's NVFP4 chunking never exceeds the default chunk, never
//    grows toward the end after its first chunk (which takes what is left
//    over when the pairs do not fill the doubling tail and whole default
//    chunks), ends with min(2, n) pairs, and splits a chunk only
//    while its CTAs leave half of the SMs idle, into at most 16 shares of at
//    least kTailMinShareTiles key tiles that together fit the SMs;
//  * the default chunk fits one wave of CTAs (or is one pair) and leaves at
//    least two chunks when there are two pairs or more.
// Prints "OK" and returns 0, or prints the first failure and returns 1.
#include <cstdio>
#include <vector>

#include "../../quantized_attention_x16_gb300/csrc/host_plan.h"

using namespace sa;

static int fail(const char* what, int B, int H, int Hkv, int L, int cp, int fp4, int sms) {
  std::printf("FAIL %s: B=%d H=%d Hkv=%d L=%d chunk_pairs=%d fp4=%d sms=%d\n", what, B, H, Hkv, L, cp, fp4, sms);
  return 1;
}

static int check(int B, int H, int Hkv, int L, int cp, bool fp4, int sms) {
  const int pairs = B * Hkv, G = H / Hkv, nkt = (L + 127) / 128;
  const int n = default_chunk_pairs(B, H, Hkv, L, sms);
  const long long units = units_per_pair(G, L);
  if (n < 1 || (n > 1 && units * n > sms)) return fail("default chunk: one wave", B, H, Hkv, L, cp, fp4, sms);
  if (pairs >= 2 && n > (pairs + 1) / 2) return fail("default chunk: two chunks", B, H, Hkv, L, cp, fp4, sms);
  const std::vector<Chunk> plan = chunk_plan(B, H, Hkv, L, cp, fp4, sms);
  long long sum = 0;
  for (const Chunk& c : plan) {
    if (c.n < 1) return fail("empty chunk", B, H, Hkv, L, cp, fp4, sms);
    sum += c.n;
  }
  if (sum != pairs) return fail("coverage", B, H, Hkv, L, cp, fp4, sms);
  if (cp > 0 || !fp4) {
    const int m = cp > 0 ? cp : n;
    for (size_t i = 0; i < plan.size(); ++i) {
      if (plan[i].nsplit != 1) return fail("split in a caller's chunking", B, H, Hkv, L, cp, fp4, sms);
      if (i + 1 < plan.size() ? plan[i].n != m : plan[i].n > m) return fail("equal chunks", B, H, Hkv, L, cp, fp4, sms);
    }
    return 0;
  }
  const int want_last = (n < 2 ? n : 2) < pairs ? (n < 2 ? n : 2) : pairs;
  if (plan.back().n != want_last) return fail("last chunk", B, H, Hkv, L, cp, fp4, sms);
  for (size_t i = 0; i < plan.size(); ++i) {
    const Chunk& c = plan[i];
    if (c.n > n) return fail("chunk above the default", B, H, Hkv, L, cp, fp4, sms);
    if (i > 0 && i + 1 < plan.size() && plan[i + 1].n > c.n) return fail("chunks grow", B, H, Hkv, L, cp, fp4, sms);
    const long long u = (long long)c.n * units;
    if (c.nsplit > 1) {
      if (2 * u > sms || c.nsplit > 16 || nkt / c.nsplit < kTailMinShareTiles || c.nsplit * u > sms)
        return fail("split", B, H, Hkv, L, cp, fp4, sms);
    } else if (2 * u <= sms && sms / u >= 2 && nkt / kTailMinShareTiles >= 2) {
      return fail("a split chunk left unsplit", B, H, Hkv, L, cp, fp4, sms);
    }
  }
  return 0;
}

int main() {
  const int shapes[][4] = {{2, 16, 16, 4096}, {1, 32, 8, 8192}, {1, 24, 24, 16384}, {1, 2, 2, 256},
                           {1, 8, 8, 1024}, {3, 6, 3, 384}, {2, 4, 2, 1000}, {1, 4, 4, 2048},
                           {1, 8, 4, 2100}, {16, 32, 8, 512}, {5, 1, 1, 33000}, {1, 1, 1, 1}};
  const int sms_list[] = {1, 2, 64, 148, 152, 160};
  const int cps[] = {0, 1, 3, 7};
  for (auto& sh : shapes)
    for (int sms : sms_list)
      for (int cp : cps)
        for (int fp4 = 0; fp4 < 2; ++fp4)
          if (check(sh[0], sh[1], sh[2], sh[3], cp, fp4 != 0, sms)) return 1;
  std::printf("OK\n");
  return 0;
}
