// Host-side checks of the work split and the tiled weight layout, compiled
// with g++ against the library's own header (no GPU needed).
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "kernels.h"

using namespace tld;

static int fails = 0;
#define CHECK(c, ...)                      \
  do {                                     \
    if (!(c)) {                            \
      std::printf("FAIL %s: ", #c);        \
      std::printf(__VA_ARGS__);            \
      std::printf("\n");                   \
      if (++fails > 20) std::exit(1);      \
    }                                      \
  } while (0)

static void check_split(int64_t total, int parts) {
  CHECK(split_begin(total, parts, 0) == 0, "start");
  CHECK(split_begin(total, parts, parts) == total, "end");
  int64_t prev = 0;
  for (int p = 0; p < parts; ++p) {
    const int64_t a = split_begin(total, parts, p), b = split_begin(total, parts, p + 1);
    CHECK(b >= a && b - a <= total / parts + 1 && b - a >= total / parts, "balanced %ld %d", (long)total, parts);
    CHECK(a == prev, "contiguous");
    prev = b;
    for (int64_t u = a; u < b; ++u) CHECK(split_owner(total, parts, u) == p, "owner %ld", (long)u);
    if (total * parts < (1LL << 31)) {
      CHECK(split_begin32((int)total, parts, p) == a, "split_begin32");
      for (int64_t u = a; u < b; ++u)
        CHECK(split_owner32((int)total, parts, (int)u) == p, "owner32 %ld", (long)u);
    }
  }
}

static void check_tiled(int N, int K) {
  const int ktiles = (K + kTileK - 1) / kTileK;
  std::vector<int> seen((size_t)N * K, 0);
  for (int r = 0; r < N; ++r)
    for (int k = 0; k < K; ++k) {
      const int64_t o = tiled_elem_offset(r, k, K);
      CHECK(o >= 0 && o < (int64_t)N * K, "range %d %d", r, k);
      if (o >= 0 && o < (int64_t)N * K) seen[o]++;
    }
  for (size_t i = 0; i < seen.size(); ++i) CHECK(seen[i] == 1, "bijective at %zu (N=%d K=%d)", i, N, K);
  // tile t starts where tiled_elem_offset puts its first element; ranges are 16-byte multiples
  const int64_t ntiles = (int64_t)(N / kTileR) * ktiles;
  for (int64_t t = 0; t <= ntiles; ++t) {
    const int64_t off = tile_byte_offset(t, ktiles, K);
    CHECK(off % 16 == 0, "tile offset alignment");
    if (t < ntiles) {
      const int64_t rb = t / ktiles, kt = t % ktiles;
      CHECK(off == 2 * tiled_elem_offset(rb * kTileR, kt * kTileK, K), "tile start");
    }
  }
  CHECK(tile_byte_offset(ntiles, ktiles, K) == 2LL * N * K, "total bytes");
  for (int64_t a = 0; a + kStageTiles <= ntiles; a += 7) {
    const int64_t bytes = tile_byte_offset(a + kStageTiles, ktiles, K) - tile_byte_offset(a, ktiles, K);
    CHECK(bytes <= kStageBytes && bytes % 16 == 0, "stage bytes %ld", (long)bytes);
  }
}

int main() {
  for (int64_t total : {1, 2, 3, 7, 151, 152, 153, 384, 1000, 49152, 22016 * 43})
    for (int parts : {1, 5, 148, 152, 160}) check_split(total, parts);
  for (int K : {8, 264, 512, 1000, 1408, 2048, 4096}) check_tiled(16, K);
  check_tiled(64, 11008);
  std::printf(fails ? "FAILED %d\n" : "OK\n", fails);
  return fails ? 1 : 0;
}
