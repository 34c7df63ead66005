/*
 * fp64 CPU oracle of one batch-1 decode step through a Llama-style decoder
 * stack.  TEST INFRASTRUCTURE ONLY: tests/, the smoke check and the benchmark's
 * cpu_baseline / reference leg use it; the CUDA library never does, and the two
 * share no code.
 *
 * What it computes is the plain unfused op chain of one decoder layer, in the
 * order the pages list it ("RDNA4 Decode Kernel Fusion: Pipeline Barriers, Not
 * Launches, Are the Win", section "Decode is where the bubble has nowhere to
 * go"): input RMSNorm, weight multiply, QKV projection, RoPE on q and k,
 * attention against the KV cache, output projection, post-attention RMSNorm
 * and multiply, gate and up projections, SwiGLU, down projection.  The same
 * page (section "Fusion removes the barrier by removing the write", Figure 1
 * caption) states that fusion leaves this arithmetic unchanged, so the fused
 * GPU path must reach this result up to rounding.
 *
 * The pages give no formulas.  Readings taken where they are silent:
 *   RMSNorm      n = x / sqrt(mean(x^2) + eps) * w   (eps inside the root, w direct)
 *   RoPE         rotate-half pairs (i, i + d/2), angle pos * theta^(-2i/d); the
 *                interleaved form rotates pairs (2i, 2i + 1) by the same angle
 *   KV append    rotated k and raw v stored as bf16 (round to nearest even) at
 *                row pos; the new token then attends to rows 0..pos
 *   attention    softmax(q.K^T / sqrt(d)) V, query head h reads KV head
 *                floor(h * n_kv / n_q)
 *   residuals    pre-norm: h1 = x + Wo o, out = h1 + Wd a
 *   SwiGLU       a = silu(gate) * up, silu(z) = z / (1 + e^-z)
 *   int4 path    weight = fp16 scale * (nibble - 8) per 32-block; every GEMV
 *                input is quantized per 32-block to int8 with an fp32 absmax
 *                scale (amax/127, round half to even, clamp to +-127); the
 *                integer block dot is exact, everything after it is fp64
 * Every sum below runs over its index in natural order, in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Planted mistakes for the pin tests (tests/ only): 0 = none. */
static int g_mutation = 0;
void orc_set_mutation(int m) { g_mutation = m; }
int orc_get_mutation(void) { return g_mutation; }
enum {
  MUT_NONE = 0,
  MUT_RMS_NO_EPS = 1,       /* eps dropped */
  MUT_RMS_NO_WEIGHT = 2,    /* weight multiply dropped */
  MUT_ROPE_SIGN = 3,        /* rotation direction flipped */
  MUT_ROPE_FREQ = 4,        /* exponent -i/d instead of -2i/d */
  MUT_ATTN_NO_SCALE = 5,    /* 1/sqrt(d) dropped */
  MUT_ATTN_GQA_MOD = 6,     /* h mod n_kv instead of contiguous groups */
  MUT_SILU_ON_UP = 7,       /* silu applied to the up projection */
  MUT_NO_RESIDUAL2 = 8,     /* second residual dropped */
  MUT_GEMV_TRANSPOSE = 9,   /* weight read as [in][out] */
  MUT_Q4_NO_OFFSET = 10,    /* nibble read without the -8 offset */
  MUT_ATTN_SKIP_LAST = 11,  /* new token does not attend to itself */
  MUT_Q4_STALE_N1 = 12,     /* gate/up input reuses the int8 codes of n1 */
  MUT_Q4_O_TENSOR_SCALE = 13, /* o quantized with one scale over the whole vector */
  MUT_Q4_A_NO_DX = 14,      /* down projection drops the block scales of a */
  MUT_ROPE_PAIR_SWAP = 15,  /* interleaved RoPE rotating (2i+1, 2i) instead of (2i, 2i+1) */
  MUT_ARGMAX_LAST_TIE = 16, /* greedy choice keeps the last of equal logits */
  MUT_LM_NO_NORM = 17,      /* LM head without the final RMSNorm */
  MUT_ATTN_NO_MAX = 18,     /* softmax weights exp(s) without the running max subtracted */
};

/* ---- storage formats ---------------------------------------------------- */

double orc_bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

double orc_fp16_value(uint16_t h) {
  int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(1024 + m), e - 25);
  return s ? -v : v;
}

/* Nearest bf16 (ties to even) of a double, as raw bits. */
uint16_t orc_bf16_round(double d) {
  if (d == 0.0 || !isfinite(d)) {
    float f = (float)d;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
  }
  double a = fabs(d);
  int e = ilogb(a);                         /* 2^e <= a < 2^(e+1) */
  double ulp = ldexp(1.0, e - 7);           /* bf16 keeps 8 significant bits */
  double r = nearbyint(a / ulp) * ulp;      /* exact scaling, RNE */
  float f = (float)(d < 0 ? -r : r);
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* ---- the layer's operations ---------------------------------------------- */

/* RMSNorm and its weight multiply (the RMS_NORM + MUL pair of "RDNA4 Decode
 * Kernel Fusion", section "Fusion removes the barrier by removing the write"). */
void orc_rmsnorm(const double* x, const uint16_t* w, int H, double eps, double* out) {
  double ss = 0.0;
  for (int i = 0; i < H; ++i) ss += x[i] * x[i];
  double ms = ss / H;
  double r = 1.0 / sqrt(ms + (g_mutation == MUT_RMS_NO_EPS ? 0.0 : eps));
  for (int i = 0; i < H; ++i)
    out[i] = x[i] * r * (g_mutation == MUT_RMS_NO_WEIGHT ? 1.0 : orc_bf16_value(w[i]));
}

/* Batch-1 projection: y[j] = sum_k W[j][k] x[k], W bf16 row-major [N][K]. */
void orc_gemv_bf16(const uint16_t* W, int N, int K, const double* x, double* y) {
#pragma omp parallel for schedule(static)
  for (int j = 0; j < N; ++j) {
    double s = 0.0;
    if (g_mutation == MUT_GEMV_TRANSPOSE && N == K) {
      for (int k = 0; k < K; ++k) s += orc_bf16_value(W[(size_t)k * N + j]) * x[k];
    } else {
      const uint16_t* row = W + (size_t)j * K;
      for (int k = 0; k < K; ++k) s += orc_bf16_value(row[k]) * x[k];
    }
    y[j] = s;
  }
}

/* RoPE on n_heads consecutive heads of size d at absolute position pos. */
void orc_rope(double* h, int n_heads, int d, int pos, double theta) {
  int half = d / 2;
  for (int hd = 0; hd < n_heads; ++hd) {
    double* v = h + (size_t)hd * d;
    for (int i = 0; i < half; ++i) {
      double expo = (g_mutation == MUT_ROPE_FREQ) ? -(double)i / d : -2.0 * i / d;
      double phi = pos * pow(theta, expo);
      double c = cos(phi), s = sin(phi);
      if (g_mutation == MUT_ROPE_SIGN) s = -s;
      double a = v[i], b = v[i + half];
      v[i] = a * c - b * s;
      v[i + half] = a * s + b * c;
    }
  }
}

/* One query head against n cached rows of its KV head (K, V bf16, row stride d). */
void orc_attention_head(const double* q, const uint16_t* K, const uint16_t* V, int n, int d,
                        double* o) {
  if (g_mutation == MUT_ATTN_SKIP_LAST && n > 1) n -= 1;
  double scale = (g_mutation == MUT_ATTN_NO_SCALE) ? 1.0 : 1.0 / sqrt((double)d);
  double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double m = -INFINITY;
  for (int t = 0; t < n; ++t) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i) acc += q[i] * orc_bf16_value(K[(size_t)t * d + i]);
    s[t] = acc * scale;
    if (s[t] > m) m = s[t];
  }
  double z = 0.0;
  for (int t = 0; t < n; ++t) {
    s[t] = exp(s[t] - (g_mutation == MUT_ATTN_NO_MAX ? 0.0 : m));
    z += s[t];
  }
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  for (int t = 0; t < n; ++t) {
    double p = s[t] / z;
    for (int i = 0; i < d; ++i) o[i] += p * orc_bf16_value(V[(size_t)t * d + i]);
  }
  free(s);
}

/* RoPE with interleaved pairs: dims (2i, 2i + 1) of each head are rotated by
 * pos * theta^(-2i/d), the pairing of models whose rotary embedding treats
 * adjacent dims as one complex number. */
void orc_rope_interleaved(double* h, int n_heads, int d, int pos, double theta) {
  for (int hd = 0; hd < n_heads; ++hd) {
    double* v = h + (size_t)hd * d;
    for (int i = 0; i < d / 2; ++i) {
      double phi = pos * pow(theta, -2.0 * i / d);
      double c = cos(phi), s = sin(phi);
      int e = 2 * i, o = 2 * i + 1;
      if (g_mutation == MUT_ROPE_PAIR_SWAP) {
        e = 2 * i + 1;
        o = 2 * i;
      }
      double a = v[e], b = v[o];
      v[e] = a * c - b * s;
      v[o] = a * s + b * c;
    }
  }
}

/* Query head -> KV head (contiguous groups). */
int orc_kv_head_of(int h, int n_q, int n_kv) {
  if (g_mutation == MUT_ATTN_GQA_MOD) return h % n_kv;
  return (int)((long)h * n_kv / n_q);
}

double orc_silu(double z) { return z / (1.0 + exp(-z)); }

void orc_swiglu(const double* g, const double* u, int F, double* a) {
  for (int j = 0; j < F; ++j)
    a[j] = (g_mutation == MUT_SILU_ON_UP) ? g[j] * orc_silu(u[j]) : orc_silu(g[j]) * u[j];
}

/* ---- block-quantized int4 weights, int8 activations ---------------------- */

/* Per 32-block absmax quantization of a GEMV input.  amax and the scale are
 * fp32; each element is divided in fp32 and rounded half to even. */
void orc_quantize_act(const double* z, int K, int8_t* qx, float* dx) {
  for (int b = 0; b < K / 32; ++b) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) {
      double a = fabs(z[b * 32 + i]);
      if (a > amax) amax = a;
    }
    float d = (float)amax / 127.0f;
    dx[b] = d;
    for (int i = 0; i < 32; ++i) {
      int q = 0;
      if (d != 0.0f) {
        float r = nearbyintf((float)z[b * 32 + i] / d);
        q = (int)r;
        if (q > 127) q = 127;
        if (q < -127) q = -127;
      }
      qx[b * 32 + i] = (int8_t)q;
    }
  }
}

static inline int nibble_at(const uint8_t* row, int k) {
  uint8_t byte = row[k >> 1];
  int u = (k & 1) ? (byte >> 4) : (byte & 15);
  return (g_mutation == MUT_Q4_NO_OFFSET) ? u : u - 8;
}

/* Exact integer block dots: out[j][b] = sum_{i<32} qw[j][32b+i] * qx[32b+i]. */
void orc_q4_blockdots(const uint8_t* Wq, int N, int K, const int8_t* qx, int64_t* out) {
  int nb = K / 32;
#pragma omp parallel for schedule(static)
  for (int j = 0; j < N; ++j) {
    const uint8_t* row = Wq + (size_t)j * (K / 2);
    for (int b = 0; b < nb; ++b) {
      int64_t acc = 0;
      for (int i = 0; i < 32; ++i) acc += (int64_t)nibble_at(row, 32 * b + i) * qx[32 * b + i];
      out[(size_t)j * nb + b] = acc;
    }
  }
}

/* y[j] = sum_b scale[j][b] * dx[b] * (integer block dot), in double. */
void orc_gemv_q4(const uint8_t* Wq, const uint16_t* Ws, int N, int K, const int8_t* qx,
                 const float* dx, double* y) {
  int nb = K / 32;
#pragma omp parallel for schedule(static)
  for (int j = 0; j < N; ++j) {
    const uint8_t* row = Wq + (size_t)j * (K / 2);
    double s = 0.0;
    for (int b = 0; b < nb; ++b) {
      int64_t acc = 0;
      for (int i = 0; i < 32; ++i) acc += (int64_t)nibble_at(row, 32 * b + i) * qx[32 * b + i];
      s += orc_fp16_value(Ws[(size_t)j * nb + b]) * (double)dx[b] * (double)acc;
    }
    y[j] = s;
  }
}

/* ---- one decoder layer, one token ---------------------------------------- */

typedef struct orc_dims {
  int32_t hidden, n_q_heads, n_kv_heads, head_dim, ffn, max_ctx, q4;
  int32_t rope_interleaved; /* 0: rotate-half pairs, 1: interleaved pairs */
  double rms_eps, rope_theta;
} orc_dims;

/* Weights of one layer.  bf16 matrices are [out][in]; for q4 the packed
 * nibbles are [out][in/2] bytes and the fp16 scales [out][in/32].  The KV
 * cache of the layer is K, V bf16 [n_kv_heads][max_ctx][head_dim]. */
typedef struct orc_layer {
  const uint16_t* attn_norm;
  const uint16_t* ffn_norm;
  const uint16_t* w[7];   /* wq wk wv wo wgate wup wdown (bf16) */
  const uint8_t* q[7];    /* q4 nibbles */
  const uint16_t* s[7];   /* q4 fp16 scales */
  uint16_t* kcache;
  uint16_t* vcache;
} orc_layer;

enum { W_Q = 0, W_K, W_V, W_O, W_GATE, W_UP, W_DOWN };

/* The int8 codes of the four GEMV inputs of a layer (n1, o, n2, a), slot by
 * slot.  Bit s of `given` clear: slot s is quantized here and, if q[s] is set,
 * its codes and scales are copied out.  Bit s set: slot s uses q[s], d[s]
 * instead of quantizing.  z[s], if set, receives the fp64 vector slot s
 * quantizes (or would quantize).  The integer dots are defined on whatever
 * codes the quantizer decided; a decision made on fp32 values elsewhere may
 * differ by one from this fp64 chain's where a value sits on a rounding
 * boundary, and feeding one side's codes to the other separates that from the
 * arithmetic around it. */
typedef struct orc_qtap {
  int8_t* q[4];
  float* d[4];
  double* z[4];
  double* kz;        /* optional: this token's rotated k [n_kv*d], fp64, before storage */
  double* vz;        /* optional: this token's v [n_kv*d], fp64, before storage */
  int32_t given;
  int32_t kv_given;  /* nonzero: the cache row pos already holds this token's k, v */
} orc_qtap;

/* The quantized form of GEMV input `slot` (bf16 weights: nothing to do). */
static void quantize_input(const orc_dims* D, orc_qtap* tap, int slot, const double* z, int K,
                           int8_t* qbuf, float* dbuf) {
  if (!D->q4) return;
  if (tap && tap->z[slot]) memcpy(tap->z[slot], z, sizeof(double) * (size_t)K);
  if (tap && ((tap->given >> slot) & 1) && tap->q[slot]) {
    memcpy(qbuf, tap->q[slot], (size_t)K);
    memcpy(dbuf, tap->d[slot], sizeof(float) * (size_t)(K / 32));
    return;
  }
  if (g_mutation == MUT_Q4_O_TENSOR_SCALE && slot == 1) {
    /* planted mistake: one absmax over all of o instead of one per block */
    double amax = 0.0;
    for (int i = 0; i < K; ++i)
      if (fabs(z[i]) > amax) amax = fabs(z[i]);
    float d = (float)amax / 127.0f;
    for (int i = 0; i < K; ++i) {
      int q = d != 0.0f ? (int)nearbyintf((float)z[i] / d) : 0;
      qbuf[i] = (int8_t)(q > 127 ? 127 : (q < -127 ? -127 : q));
    }
    for (int b = 0; b < K / 32; ++b) dbuf[b] = d;
  } else {
    orc_quantize_act(z, K, qbuf, dbuf);
  }
  if (tap && tap->q[slot]) {
    memcpy(tap->q[slot], qbuf, (size_t)K);
    memcpy(tap->d[slot], dbuf, sizeof(float) * (size_t)(K / 32));
  }
}

/* y = W x: bf16 weights on x itself, q4 weights on x's quantized form. */
static void project(const orc_dims* D, const orc_layer* L, int which, int N, int K,
                    const double* x, double* y, const int8_t* qbuf, const float* dbuf) {
  if (!D->q4) {
    orc_gemv_bf16(L->w[which], N, K, x, y);
  } else if (g_mutation == MUT_Q4_A_NO_DX && which == W_DOWN) {
    /* planted mistake: the block scales of a left out of the down projection */
    float* ones = (float*)malloc(sizeof(float) * (size_t)(K / 32));
    for (int b = 0; b < K / 32; ++b) ones[b] = 1.0f;
    orc_gemv_q4(L->q[which], L->s[which], N, K, qbuf, ones, y);
    free(ones);
  } else {
    orc_gemv_q4(L->q[which], L->s[which], N, K, qbuf, dbuf, y);
  }
}

/* x[H] -> out[H] at position pos; appends this token's k, v to row pos. */
int orc_layer_step(const orc_dims* D, const orc_layer* L, int pos, const double* x, double* out,
                   orc_qtap* tap) {
  const int H = D->hidden, nq = D->n_q_heads, nkv = D->n_kv_heads, d = D->head_dim,
            F = D->ffn;
  if (pos < 0 || pos >= D->max_ctx) return -1;
  const int Kmax = (H > F ? H : F) > nq * d ? (H > F ? H : F) : nq * d;
  double* n1 = (double*)malloc(sizeof(double) * H);
  double* q = (double*)malloc(sizeof(double) * nq * d);
  double* k = (double*)malloc(sizeof(double) * nkv * d);
  double* v = (double*)malloc(sizeof(double) * nkv * d);
  double* o = (double*)malloc(sizeof(double) * nq * d);
  double* h1 = (double*)malloc(sizeof(double) * H);
  double* y = (double*)malloc(sizeof(double) * H);
  double* n2 = (double*)malloc(sizeof(double) * H);
  double* g = (double*)malloc(sizeof(double) * F);
  double* u = (double*)malloc(sizeof(double) * F);
  double* a = (double*)malloc(sizeof(double) * F);
  int8_t* qb = (int8_t*)malloc((size_t)Kmax);
  float* db = (float*)malloc(sizeof(float) * (size_t)(Kmax / 32 + 1));
  int8_t* qb_n1 = (int8_t*)malloc((size_t)H);               /* planted-mistake hook only */
  float* db_n1 = (float*)malloc(sizeof(float) * (size_t)(H / 32 + 1));

  /* input RMSNorm + weight multiply */
  orc_rmsnorm(x, L->attn_norm, H, D->rms_eps, n1);
  /* q, k, v projections */
  quantize_input(D, tap, 0, n1, H, qb, db);
  if (D->q4) {
    memcpy(qb_n1, qb, (size_t)H);
    memcpy(db_n1, db, sizeof(float) * (size_t)(H / 32));
  }
  project(D, L, W_Q, nq * d, H, n1, q, qb, db);
  project(D, L, W_K, nkv * d, H, n1, k, qb, db);
  project(D, L, W_V, nkv * d, H, n1, v, qb, db);
  /* RoPE on q and k */
  if (D->rope_interleaved) {
    orc_rope_interleaved(q, nq, d, pos, D->rope_theta);
    orc_rope_interleaved(k, nkv, d, pos, D->rope_theta);
  } else {
    orc_rope(q, nq, d, pos, D->rope_theta);
    orc_rope(k, nkv, d, pos, D->rope_theta);
  }
  if (tap && tap->kz) memcpy(tap->kz, k, sizeof(double) * (size_t)nkv * d);
  if (tap && tap->vz) memcpy(tap->vz, v, sizeof(double) * (size_t)nkv * d);
  /* KV append at row pos (storage rounding to bf16 is itself a decision made
     on floating point; a test may hand the row in instead, see orc_qtap) */
  if (!(tap && tap->kv_given))
    for (int hh = 0; hh < nkv; ++hh)
      for (int i = 0; i < d; ++i) {
        size_t at = ((size_t)hh * D->max_ctx + pos) * d + i;
        L->kcache[at] = orc_bf16_round(k[hh * d + i]);
        L->vcache[at] = orc_bf16_round(v[hh * d + i]);
      }
  /* attention over rows 0..pos */
#pragma omp parallel for schedule(static)
  for (int hq = 0; hq < nq; ++hq) {
    int gk = orc_kv_head_of(hq, nq, nkv);
    const uint16_t* Kh = L->kcache + (size_t)gk * D->max_ctx * d;
    const uint16_t* Vh = L->vcache + (size_t)gk * D->max_ctx * d;
    orc_attention_head(q + (size_t)hq * d, Kh, Vh, pos + 1, d, o + (size_t)hq * d);
  }
  /* output projection + residual */
  quantize_input(D, tap, 1, o, nq * d, qb, db);
  project(D, L, W_O, H, nq * d, o, y, qb, db);
  for (int i = 0; i < H; ++i) h1[i] = x[i] + y[i];
  /* post-attention RMSNorm + multiply */
  orc_rmsnorm(h1, L->ffn_norm, H, D->rms_eps, n2);
  /* gate, up, SwiGLU */
  quantize_input(D, tap, 2, n2, H, qb, db);
  if (D->q4 && g_mutation == MUT_Q4_STALE_N1) {  /* planted mistake: n1's codes reused */
    memcpy(qb, qb_n1, (size_t)H);
    memcpy(db, db_n1, sizeof(float) * (size_t)(H / 32));
  }
  project(D, L, W_GATE, F, H, n2, g, qb, db);
  project(D, L, W_UP, F, H, n2, u, qb, db);
  orc_swiglu(g, u, F, a);
  /* down projection + residual */
  quantize_input(D, tap, 3, a, F, qb, db);
  project(D, L, W_DOWN, H, F, a, y, qb, db);
  for (int i = 0; i < H; ++i) out[i] = (g_mutation == MUT_NO_RESIDUAL2) ? y[i] : h1[i] + y[i];

  free(n1); free(q); free(k); free(v); free(o); free(h1); free(y); free(n2);
  free(g); free(u); free(a); free(qb); free(db); free(qb_n1); free(db_n1);
  return 0;
}

/* The stack: x_{l+1} = layer_l(x_l).  per_layer_out (n_layers*H) may be NULL. */
int orc_stack_step(const orc_dims* D, const orc_layer* layers, int n_layers, int pos,
                   const double* x_in, double* x_out, double* per_layer_out) {
  const int H = D->hidden;
  double* cur = (double*)malloc(sizeof(double) * H);
  double* nxt = (double*)malloc(sizeof(double) * H);
  memcpy(cur, x_in, sizeof(double) * H);
  for (int l = 0; l < n_layers; ++l) {
    int rc = orc_layer_step(D, &layers[l], pos, cur, nxt, NULL);
    if (rc) { free(cur); free(nxt); return rc; }
    if (per_layer_out) memcpy(per_layer_out + (size_t)l * H, nxt, sizeof(double) * H);
    double* t = cur; cur = nxt; nxt = t;
  }
  memcpy(x_out, cur, sizeof(double) * H);
  free(cur);
  free(nxt);
  return 0;
}

/* ---- after the stack: LM head and greedy choice --------------------------- */

/* The token after the stack's output x[H]: the final RMSNorm and its weight
 * multiply, the vocabulary projection (W bf16 [V][H]) into logits[V], and the
 * greedy choice, the index of the largest logit (the lowest index among equal
 * ones).  "RDNA4 Decode Kernel Fusion", section "What it does to the token",
 * Table 1 ("LM head + sampling"). */
int orc_lm_head(const double* x, int H, const uint16_t* norm_w, const uint16_t* W, int V,
                double eps, double* logits) {
  double* n = (double*)malloc(sizeof(double) * (size_t)H);
  if (g_mutation == MUT_LM_NO_NORM) {
    for (int i = 0; i < H; ++i) n[i] = x[i];
  } else {
    orc_rmsnorm(x, norm_w, H, eps, n);
  }
  orc_gemv_bf16(W, V, H, n, logits);
  int best = 0;
  for (int j = 1; j < V; ++j)
    if (logits[j] > logits[best] || (g_mutation == MUT_ARGMAX_LAST_TIE && logits[j] == logits[best]))
      best = j;
  free(n);
  return best;
}
