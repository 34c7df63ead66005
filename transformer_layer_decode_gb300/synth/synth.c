/*
 * Seeded synthetic inputs for the batch-1 decode layer: weights, norm weights,
 * block-quantized weights, the prefilled KV cache and the per-step input hidden
 * vector.  This file draws numbers and stores them in the storage formats the
 * layer reads (bf16, fp16, packed int4); it performs none of the layer's
 * arithmetic.  Both the fp64 oracle and the CUDA path consume its output.
 *
 * Generator (counter based, so any element can be regenerated on its own):
 *   mix(s)        = SplitMix64 output function applied to state s
 *                   (Steele, Lea, Flood, "Fast splittable pseudorandom number
 *                   generators", OOPSLA 2014; the constants of Java 8's
 *                   SplittableRandom / Vigna's splitmix64.c).
 *   key           = mix(mix(mix(seed) ^ (layer+1)) ^ (tensor+1))
 *   normal i      : pair p = i/2, a = mix(key + 2p), b = mix(key + 2p + 1),
 *                   u1 = ((a>>11)+1)·2^-53 in (0,1], u2 = (b>>11)·2^-53 in [0,1),
 *                   r = sqrt(-2 ln u1), z = r·cos(2π u2) for even i,
 *                   r·sin(2π u2) for odd i (Box and Muller, 1958).
 *   uniform int4 i: mix(key + i) >> 60, minus 8   (uniform on [-8, 7]).
 * Storage rounding is round-to-nearest-even, done in double straight to the
 * target format (no double rounding through fp32).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix(uint64_t s) {
  uint64_t z = s + GOLDEN_GAMMA;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_splitmix64(uint64_t s) { return mix(s); }

uint64_t synth_key(uint64_t seed, int64_t layer, int64_t tensor) {
  return mix(mix(mix(seed) ^ (uint64_t)(layer + 1)) ^ (uint64_t)(tensor + 1));
}

static inline double normal_at(uint64_t key, uint64_t i) {
  uint64_t p = i >> 1;
  uint64_t a = mix(key + 2 * p), b = mix(key + 2 * p + 1);
  double u1 = (double)((a >> 11) + 1) * 0x1.0p-53;
  double u2 = (double)(b >> 11) * 0x1.0p-53;
  double r = sqrt(-2.0 * log(u1));
  double t = 6.283185307179586476925286766559 * u2;
  return (i & 1) ? r * sin(t) : r * cos(t);
}

/* double -> nearest bf16 (ties to even), returned as the raw 16 bits. */
static inline uint16_t to_bf16(double d) {
  if (d == 0.0) return signbit(d) ? 0x8000 : 0;
  int e;
  double m = frexp(d, &e);             /* |m| in [0.5, 1) */
  double q = nearbyint(ldexp(m, 8));   /* 8 significant bits, RNE */
  float f = (float)ldexp(q, e - 8);    /* exact: q has at most 9 bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* double -> nearest fp16 (ties to even), subnormals included, raw 16 bits. */
static inline uint16_t to_fp16(double d) {
  uint16_t sign = signbit(d) ? 0x8000 : 0;
  double a = fabs(d);
  if (a == 0.0) return sign;
  double q;
  int e;
  if (a < 0x1.0p-14) {                 /* subnormal grid: k * 2^-24 */
    q = nearbyint(a * 0x1.0p24);
    if (q >= 1024.0) return sign | (uint16_t)(1 << 10); /* rounds up to min normal */
    return sign | (uint16_t)q;
  }
  double m = frexp(a, &e);             /* a = m 2^e, m in [0.5,1) */
  q = nearbyint(ldexp(m, 11));         /* 11 significant bits, RNE */
  if (q >= 2048.0) { q /= 2.0; e += 1; }
  int exp16 = e - 1 + 15;              /* value = (q/1024) * 2^(e-1) */
  if (exp16 >= 31) return sign | 0x7C00; /* overflow to inf (not reached) */
  uint16_t mant = (uint16_t)((int)q - 1024);
  return sign | (uint16_t)(exp16 << 10) | mant;
}

uint16_t synth_round_bf16(double d) { return to_bf16(d); }
uint16_t synth_round_fp16(double d) { return to_fp16(d); }

/* out[j] = bf16(mean + std * N_j) for j in [0, count), N_j = normal at index start+j. */
void synth_normal_bf16(uint64_t seed, int64_t layer, int64_t tensor, uint64_t start,
                       uint64_t count, double mean, double stdev, uint16_t* out) {
  uint64_t key = synth_key(seed, layer, tensor);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < (int64_t)count; ++j)
    out[j] = to_bf16(mean + stdev * normal_at(key, start + (uint64_t)j));
}

/* Same draws, stored as fp32 (the value of the bf16-rounded draw, exactly). */
void synth_normal_bf16_as_f32(uint64_t seed, int64_t layer, int64_t tensor, uint64_t start,
                              uint64_t count, double mean, double stdev, float* out) {
  uint64_t key = synth_key(seed, layer, tensor);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < (int64_t)count; ++j) {
    uint32_t u = (uint32_t)to_bf16(mean + stdev * normal_at(key, start + (uint64_t)j)) << 16;
    memcpy(&out[j], &u, 4);
  }
}

/* out[j] = fp16(|mean + std * N_j|). */
void synth_absnormal_fp16(uint64_t seed, int64_t layer, int64_t tensor, uint64_t start,
                          uint64_t count, double mean, double stdev, uint16_t* out) {
  uint64_t key = synth_key(seed, layer, tensor);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < (int64_t)count; ++j)
    out[j] = to_fp16(fabs(mean + stdev * normal_at(key, start + (uint64_t)j)));
}

/* Uniform int4 quants on [-8, 7] for a [rows][cols] matrix (cols % 32 == 0),
 * packed two per byte: element 2i in the low nibble and 2i+1 in the high nibble
 * of byte i of the row, each stored as q + 8 in [0, 15].  Row-major, cols/2
 * bytes per row. */
void synth_q4_packed(uint64_t seed, int64_t layer, int64_t tensor, uint64_t rows,
                     uint64_t cols, uint8_t* out) {
  uint64_t key = synth_key(seed, layer, tensor);
  uint64_t half = cols / 2;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < (int64_t)rows; ++r) {
    for (uint64_t b = 0; b < half; ++b) {
      uint64_t i0 = (uint64_t)r * cols + 2 * b;
      uint8_t lo = (uint8_t)(mix(key + i0) >> 60);       /* q + 8 */
      uint8_t hi = (uint8_t)(mix(key + i0 + 1) >> 60);
      out[(uint64_t)r * half + b] = (uint8_t)(lo | (hi << 4));
    }
  }
}
