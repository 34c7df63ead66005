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
  const TileGeom g = tile_geom(K, false);
  std::vector<int> seen((size_t)N * K, 0);
  for (int r = 0; r < N; ++r)
    for (int k = 0; k < K; ++k) {
      const int64_t o = tiled_elem_offset(r, k, K);
      CHECK(o >= 0 && o < (int64_t)N * K, "range %d %d", r, k);
      if (o >= 0 && o < (int64_t)N * K) seen[o]++;
    }
  for (size_t i = 0; i < seen.size(); ++i) CHECK(seen[i] == 1, "bijective at %zu (N=%d K=%d)", i, N, K);
  // tile t starts where tiled_elem_offset puts its first element; ranges are 16-byte multiples
  const int64_t ntiles = (int64_t)(N / kTileR) * g.ktiles;
  for (int64_t t = 0; t <= ntiles; ++t) {
    const int64_t off = tile_byte_offset(t, g);
    CHECK(off % 16 == 0, "tile offset alignment");
    if (t < ntiles) {
      const int64_t rb = t / g.ktiles, kt = t % g.ktiles;
      CHECK(off == 2 * tiled_elem_offset(rb * kTileR, kt * kTileK, K), "tile start");
    }
  }
  CHECK(tile_byte_offset(ntiles, g) == 2LL * N * K, "total bytes");
  for (int64_t a = 0; a + kStageTiles <= ntiles; a += 7) {
    const int64_t bytes = tile_byte_offset(a + kStageTiles, g) - tile_byte_offset(a, g);
    CHECK(bytes <= kStageBytes && bytes % 16 == 0, "stage bytes %ld", (long)bytes);
  }
}

// q4: every nibble byte and every scale lands on a distinct byte of the
// matrix; each tile is 16-byte aligned and stages fit the q4 stage size.
static void check_tiled_q4(int N, int K) {
  const TileGeom g = tile_geom(K, true);
  const int64_t total = (int64_t)(N / kTileR) * g.rb_bytes;
  CHECK(total == (int64_t)N * (K / 2 + K / 16), "q4 bytes");
  std::vector<int> seen((size_t)total, 0);
  for (int r = 0; r < N; ++r) {
    for (int c2 = 0; c2 < K / 2; ++c2) {
      const int64_t o = q4_nibble_byte(r, c2, K);
      CHECK(o >= 0 && o < total, "q4 nibble range");
      if (o >= 0 && o < total) seen[o]++;
    }
    for (int b = 0; b < K / 32; ++b) {
      const int64_t o = q4_scale_byte(r, b, K);
      CHECK(o >= 0 && o + 1 < total && o % 2 == 0, "q4 scale range");
      if (o >= 0 && o + 1 < total) {
        seen[o]++;
        seen[o + 1]++;
      }
    }
  }
  for (size_t i = 0; i < seen.size(); ++i) CHECK(seen[i] == 1, "q4 bijective at %zu (K=%d)", i, K);
  const int64_t ntiles = (int64_t)(N / kTileR) * g.ktiles;
  for (int64_t t = 0; t <= ntiles; ++t) CHECK(tile_byte_offset(t, g) % 16 == 0, "q4 tile alignment");
  for (int64_t a = 0; a + kStageTiles <= ntiles; a += 3) {
    const int64_t bytes = tile_byte_offset(a + kStageTiles, g) - tile_byte_offset(a, g);
    CHECK(bytes <= kStageBytesQ4 && bytes % 16 == 0, "q4 stage bytes %ld", (long)bytes);
  }
}

int main() {
  for (int64_t total : {1, 2, 3, 7, 151, 152, 153, 384, 1000, 49152, 22016 * 43})
    for (int parts : {1, 5, 148, 152, 160}) check_split(total, parts);
  // the attention cluster's shares: a head's chunks (fewer than the CTAs too)
  // and the merge's 32-element blocks over the cluster sizes in use
  for (int64_t total : {1, 4, 8, 16, 32, 33, 35, 64, 65})
    for (int parts : {2, 3, 4, 8, 12, 16}) check_split(total, parts);
  for (int K : {8, 264, 512, 1000, 1408, 2048, 4096}) check_tiled(16, K);
  check_tiled(64, 11008);
  for (int K : {64, 512, 1408, 2048, 4096, 11008}) check_tiled_q4(8, K);
  std::printf(fails ? "FAILED %d\n" : "OK\n", fails);
  return fails ? 1 : 0;
}
