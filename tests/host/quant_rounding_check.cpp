// The int8 quantizer forms every quotient from the block's reciprocal:
// RN(1/d) = rd, q = RN(z rd), r = z - d q exactly (one fused multiply-add),
// quotient RN(q + r rd) (Markstein's correction); the block scale amax / 127
// the same way from RN(1/127).  This checks, in IEEE fp32 on the host (no
// contraction but the explicit fused multiply-adds), that scale and codes equal
// those of the IEEE division for random inputs and for quotients placed next to
// the rounding boundaries k + 1/2; and that no code of an element |z| <= amax,
// the block's absmax itself included, leaves [-127, 127] before clamping (the
// kernels skip the clamp on that path).
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <initializer_list>

static float div_rn_from_rcp(float a, float b, float rb) {
  const float q = a * rb;
  const float r = std::fmaf(-q, b, a);
  return std::fmaf(r, rb, q);
}

static int code_of(float q) {
  const int v = (int)std::nearbyintf(q);
  return v > 127 ? 127 : (v < -127 ? -127 : v);
}

static uint64_t s = 0x9E3779B97F4A7C15ull;
static double uni() {  // SplitMix64 -> [0, 1)
  uint64_t z = (s += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return (double)((z ^ (z >> 31)) >> 11) * 0x1.0p-53;
}

int main() {
  long bad_d = 0, bad_q = 0, bad_div = 0, n = 0, beyond = 0;
  const float r127 = 1.0f / 127.0f;
  for (int t = 0; t < 2000000; ++t) {
    const float amax = (float)std::exp(std::log(1e-30) + uni() * (std::log(1e6) - std::log(1e-30)));
    const float d = div_rn_from_rcp(amax, 127.0f, r127);
    if (d != amax / 127.0f) ++bad_d;
    const float rd = 1.0f / d;
    // a random element of the block, and one whose quotient sits next to k + 1/2
    const float z = (float)((2.0 * uni() - 1.0) * amax);
    const int k = (int)(uni() * 127.0);
    float zb = (float)((k + 0.5) * (double)d);
    uint32_t bits;
    std::memcpy(&bits, &zb, 4);
    bits += (int)(uni() * 9.0) - 4;
    std::memcpy(&zb, &bits, 4);
    if (uni() < 0.5) zb = -zb;
    for (float x : {z, zb, amax, -amax}) {
      if (std::fabs(x) > amax) continue;
      ++n;
      const float qm = div_rn_from_rcp(x, d, rd), qi = x / d;
      if (qm != qi) ++bad_div;
      if (code_of(qm) != code_of(qi)) ++bad_q;
      if (std::fabs(std::nearbyintf(qm)) > 127.0f) ++beyond;
    }
  }
  std::printf("scales differing %ld; quotients differing %ld, codes differing %ld, "
              "unclamped codes beyond +-127 %ld of %ld\n", bad_d, bad_div, bad_q, beyond, n);
  const bool bad = bad_d || bad_q || bad_div || beyond;
  std::printf(bad ? "FAILED\n" : "OK\n");
  return bad ? 1 : 0;
}
