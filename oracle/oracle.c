/*
 * Oracle of the routed MoE feed-forward step over Q8_0 weights: plain,
 * single-threaded, fp64. TEST INFRASTRUCTURE ONLY (see oracle.h for what it
 * computes, which passages it follows and who may call it).
 *
 * Compiled with -ffp-contract=off so that every a*b+c below is two roundings,
 * the same on every host.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ formats */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int ex = (h >> 10) & 0x1F;
  int frac = h & 0x3FF;
  double v;
  if (ex == 0)
    v = ldexp((double)frac, -24); /* subnormal: frac * 2^-24 */
  else if (ex == 31)
    v = frac ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + frac), ex - 25); /* (1 + frac/1024) * 2^(ex-15) */
  return sign ? -v : v;
}

/* Nearest integer to a non-negative double, ties to even. Exact: floor and the
 * difference of two doubles within one binade are exact. */
static double round_nearest_even_nonneg(double s) {
  double fl = floor(s);
  double diff = s - fl;
  if (diff > 0.5) return fl + 1.0;
  if (diff < 0.5) return fl;
  return fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;
}

uint16_t oracle_double_to_half(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isnan(x)) return 0x7E00;
  if (a >= 65520.0) return sign | 0x7C00; /* 65520 is the tie between 65504 and 2^16: even side overflows */
  if (a < ldexp(1.0, -14)) {
    /* subnormal (or zero): units of 2^-24; a carry to 1024 is the smallest normal, same bits */
    double m = round_nearest_even_nonneg(ldexp(a, 24));
    return sign | (uint16_t)m;
  }
  int e2;
  frexp(a, &e2);       /* a = f * 2^e2, f in [0.5, 1) */
  int E = e2 - 1;      /* a in [2^E, 2^(E+1)) */
  double m = round_nearest_even_nonneg(ldexp(a, 10 - E)); /* in [1024, 2048] */
  if (m == 2048.0) {
    m = 1024.0;
    E += 1;
  }
  if (E + 15 >= 31) return sign | 0x7C00;
  return sign | (uint16_t)(((E + 15) << 10) | ((int)m - 1024));
}

/* bfloat16 is the upper half of a binary32. */
double oracle_bf16_to_double(uint16_t b) {
  union {
    uint32_t u;
    float f;
  } v;
  v.u = (uint32_t)b << 16;
  return (double)v.f;
}

/* ------------------------------------------------------------------- Q8_0 */

static double round_half_away(double v) {
  double a = fabs(v);
  double fl = floor(a);
  double r = (a - fl >= 0.5) ? fl + 1.0 : fl;
  return v < 0 ? -r : r;
}

int oracle_q8_0_quantize(const float *w, int64_t rows, int64_t K, uint8_t *blocks) {
  if (rows < 0 || K <= 0 || K % ORACLE_Q8_0_BLOCK) return -1;
  int64_t nb = K / ORACLE_Q8_0_BLOCK;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float *x = w + r * K + b * ORACLE_Q8_0_BLOCK;
      uint8_t *blk = blocks + (r * nb + b) * ORACLE_Q8_0_BYTES;
      double amax = 0.0;
      for (int i = 0; i < ORACLE_Q8_0_BLOCK; ++i) {
        double a = fabs((double)x[i]);
        if (a > amax) amax = a;
      }
      double d = amax / 127.0;
      uint16_t dh = oracle_double_to_half(d);
      blk[0] = (uint8_t)(dh & 0xFF);
      blk[1] = (uint8_t)(dh >> 8);
      for (int i = 0; i < ORACLE_Q8_0_BLOCK; ++i) {
        double q = 0.0;
        if (amax > 0.0) {
          q = round_half_away((double)x[i] / d);
          if (q > 127.0) q = 127.0;
          if (q < -127.0) q = -127.0;
        }
        blk[2 + i] = (uint8_t)(int8_t)q;
      }
    }
  }
  return 0;
}

static double block_scale(const uint8_t *blk) {
  return oracle_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
}

int oracle_q8_0_dequantize(const uint8_t *blocks, int64_t rows, int64_t K, double *w) {
  if (rows < 0 || K <= 0 || K % ORACLE_Q8_0_BLOCK) return -1;
  int64_t nb = K / ORACLE_Q8_0_BLOCK;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t *blk = blocks + (r * nb + b) * ORACLE_Q8_0_BYTES;
      double d = block_scale(blk);
      for (int i = 0; i < ORACLE_Q8_0_BLOCK; ++i)
        w[r * K + b * ORACLE_Q8_0_BLOCK + i] = d * (double)(int8_t)blk[2 + i];
    }
  return 0;
}

/* Row `r` of a Q8_0 matrix with K columns, dotted with v[K] in column order. */
static double q8_0_row_dot(const uint8_t *blocks, int64_t r, int64_t K, const double *v) {
  int64_t nb = K / ORACLE_Q8_0_BLOCK;
  double acc = 0.0;
  for (int64_t b = 0; b < nb; ++b) {
    const uint8_t *blk = blocks + (r * nb + b) * ORACLE_Q8_0_BYTES;
    double d = block_scale(blk);
    for (int i = 0; i < ORACLE_Q8_0_BLOCK; ++i) {
      double wv = d * (double)(int8_t)blk[2 + i]; /* exact: 11-bit scale times 8-bit code */
      acc += wv * v[b * ORACLE_Q8_0_BLOCK + i];
    }
  }
  return acc;
}

/* ----------------------------------------------------------------- router */

void oracle_router_logits(const uint16_t *x, int64_t T, int64_t H, const float *Wr, const float *bias,
                          int64_t E, double *z) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int64_t h = 0; h < H; ++h) acc += oracle_bf16_to_double(x[t * H + h]) * (double)Wr[e * H + h];
      if (bias) acc += (double)bias[e];
      z[t * E + e] = acc;
    }
}

void oracle_topk_gates(const double *z, int64_t T, int64_t E, int64_t k, int32_t *ids, double *gates) {
  unsigned char *taken = (unsigned char *)malloc((size_t)E);
  for (int64_t t = 0; t < T; ++t) {
    const double *zt = z + t * E;
    memset(taken, 0, (size_t)E);
    /* descending logit; among equal logits the lower id comes first */
    for (int64_t j = 0; j < k; ++j) {
      int64_t best = -1;
      for (int64_t e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || zt[e] > zt[best]) best = e; /* strict '>' keeps the lower id on ties */
      }
      taken[best] = 1;
      ids[t * k + j] = (int32_t)best;
    }
    /* softmax restricted to the selection: the full denominator cancels */
    double zmax = zt[ids[t * k]];
    double sum = 0.0;
    for (int64_t j = 0; j < k; ++j) sum += exp(zt[ids[t * k + j]] - zmax);
    if (gates)
      for (int64_t j = 0; j < k; ++j) gates[t * k + j] = exp(zt[ids[t * k + j]] - zmax) / sum;
  }
  free(taken);
}

void oracle_gates_full_softmax(const double *z, int64_t T, int64_t E, int64_t k, const int32_t *ids,
                               double *gates) {
  double *p = (double *)malloc(sizeof(double) * (size_t)E);
  for (int64_t t = 0; t < T; ++t) {
    const double *zt = z + t * E;
    double zmax = zt[0];
    for (int64_t e = 1; e < E; ++e)
      if (zt[e] > zmax) zmax = zt[e];
    double den = 0.0;
    for (int64_t e = 0; e < E; ++e) den += exp(zt[e] - zmax);
    for (int64_t e = 0; e < E; ++e) p[e] = exp(zt[e] - zmax) / den;
    double sel = 0.0;
    for (int64_t j = 0; j < k; ++j) sel += p[ids[t * k + j]];
    for (int64_t j = 0; j < k; ++j) gates[t * k + j] = p[ids[t * k + j]] / sel;
  }
  free(p);
}

void oracle_permutation(const int32_t *ids, int64_t T, int64_t k, int64_t E, int32_t *offsets, int32_t *perm,
                        int32_t *inv) {
  for (int64_t e = 0; e <= E; ++e) offsets[e] = 0;
  for (int64_t s = 0; s < T * k; ++s) offsets[ids[s] + 1] += 1; /* counts, shifted by one */
  for (int64_t e = 0; e < E; ++e) offsets[e + 1] += offsets[e]; /* exclusive prefix sum */
  int64_t p = 0;
  for (int64_t e = 0; e < E; ++e)
    for (int64_t t = 0; t < T; ++t)
      for (int64_t j = 0; j < k; ++j)
        if (ids[t * k + j] == e) perm[p++] = (int32_t)(t * k + j);
  if (inv)
    for (int64_t q = 0; q < T * k; ++q) inv[perm[q]] = (int32_t)q;
}

/* ------------------------------------------------------------------ experts */

/* SiLU(g) * u, SiLU(a) = a / (1 + e^-a). */
static double silu_times(double g, double u) { return g / (1.0 + exp(-g)) * u; }

void oracle_expert_ffn(const uint8_t *wg, const uint8_t *wu, const uint8_t *wd, int64_t H, int64_t I,
                       const double *x, double *y) {
  double *a = (double *)malloc(sizeof(double) * (size_t)I);
  for (int64_t i = 0; i < I; ++i) {
    double g = q8_0_row_dot(wg, i, H, x);
    double u = q8_0_row_dot(wu, i, H, x);
    a[i] = silu_times(g, u);
  }
  for (int64_t o = 0; o < H; ++o) y[o] = q8_0_row_dot(wd, o, I, a);
  free(a);
}

static int sizes_ok(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, int64_t S) {
  return T >= 0 && H > 0 && I > 0 && H % ORACLE_Q8_0_BLOCK == 0 && I % ORACLE_Q8_0_BLOCK == 0 && E > 0 &&
         k >= 1 && k <= E && (S == 0 || S == 1);
}

int oracle_moe_experts(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, int64_t S, const uint16_t *x,
                       const int32_t *ids, const double *gates, const uint8_t *const *w_gate,
                       const uint8_t *const *w_up, const uint8_t *const *w_down, double *out) {
  if (!sizes_ok(T, H, I, E, k, S)) return -1;
  double *xt = (double *)malloc(sizeof(double) * (size_t)H);
  double *y = (double *)malloc(sizeof(double) * (size_t)H);
  int rc = 0;
  for (int64_t t = 0; t < T && rc == 0; ++t) {
    for (int64_t h = 0; h < H; ++h) xt[h] = oracle_bf16_to_double(x[t * H + h]);
    double *ot = out + t * H;
    for (int64_t h = 0; h < H; ++h) ot[h] = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      int32_t e = ids[t * k + j];
      if (!w_gate[e] || !w_up[e] || !w_down[e]) {
        rc = -2;
        break;
      }
      oracle_expert_ffn(w_gate[e], w_up[e], w_down[e], H, I, xt, y);
      double g = gates[t * k + j];
      for (int64_t h = 0; h < H; ++h) ot[h] += g * y[h];
    }
    for (int64_t s = 0; s < S && rc == 0; ++s) { /* always-on expert, weight 1 */
      int64_t e = E + s;
      if (!w_gate[e] || !w_up[e] || !w_down[e]) {
        rc = -2;
        break;
      }
      oracle_expert_ffn(w_gate[e], w_up[e], w_down[e], H, I, xt, y);
      for (int64_t h = 0; h < H; ++h) ot[h] += y[h];
    }
  }
  free(xt);
  free(y);
  return rc;
}

int oracle_moe_forward(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, int64_t S, const uint16_t *x,
                       const float *Wr, const float *bias, const uint8_t *const *w_gate,
                       const uint8_t *const *w_up, const uint8_t *const *w_down, int32_t *ids, double *gates,
                       double *out) {
  if (!sizes_ok(T, H, I, E, k, S)) return -1;
  if (T == 0) return 0;
  double *z = (double *)malloc(sizeof(double) * (size_t)(T * E));
  int32_t *id = ids ? ids : (int32_t *)malloc(sizeof(int32_t) * (size_t)(T * k));
  double *g = gates ? gates : (double *)malloc(sizeof(double) * (size_t)(T * k));
  oracle_router_logits(x, T, H, Wr, bias, E, z);
  oracle_topk_gates(z, T, E, k, id, g);
  int rc = oracle_moe_experts(T, H, I, E, k, S, x, id, g, w_gate, w_up, w_down, out);
  free(z);
  if (!ids) free(id);
  if (!gates) free(g);
  return rc;
}

/* ------------------------------------------------------- Q8 activations */

int oracle_q8_activations(const float *v, int64_t n, int64_t blk, double *out, int8_t *q, float *d) {
  if (n < 0 || blk <= 0 || n % blk) return -1;
  for (int64_t b = 0; b < n / blk; ++b) {
    const float *x = v + b * blk;
    float amax = 0.0f;
    for (int64_t i = 0; i < blk; ++i) {
      float a = fabsf(x[i]);
      if (a > amax) amax = a;
    }
    float db = amax / 127.0f; /* fp32 division */
    if (d) d[b] = db;
    for (int64_t i = 0; i < blk; ++i) {
      double qi = 0.0;
      if (amax > 0.0f) {
        float r = x[i] / db; /* fp32 division; its exact value decides the code */
        qi = round_half_away((double)r);
        if (qi > 127.0) qi = 127.0;
        if (qi < -127.0) qi = -127.0;
      }
      if (q) q[b * blk + i] = (int8_t)qi;
      out[b * blk + i] = qi * (double)db;
    }
  }
  return 0;
}

/* One expert on one token, Q8 activations: x8 is the token's already
 * quantised x (fp64 [H]); h goes through the same rule in blocks of 16. */
static void expert_ffn_q8act(const uint8_t *wg, const uint8_t *wu, const uint8_t *wd, int64_t H, int64_t I,
                             const double *x8, double *y) {
  float *a32 = (float *)malloc(sizeof(float) * (size_t)I);
  double *a8 = (double *)malloc(sizeof(double) * (size_t)I);
  for (int64_t i = 0; i < I; ++i) {
    double g = q8_0_row_dot(wg, i, H, x8);
    double u = q8_0_row_dot(wu, i, H, x8);
    a32[i] = (float)silu_times(g, u); /* rounded to fp32 */
  }
  oracle_q8_activations(a32, I, 16, a8, NULL, NULL);
  for (int64_t o = 0; o < H; ++o) y[o] = q8_0_row_dot(wd, o, I, a8);
  free(a32);
  free(a8);
}

int oracle_moe_experts_q8act(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, int64_t S, const uint16_t *x,
                             const int32_t *ids, const double *gates, const uint8_t *const *w_gate,
                             const uint8_t *const *w_up, const uint8_t *const *w_down, double *out) {
  if (!sizes_ok(T, H, I, E, k, S) || I % 16) return -1;
  float *x32 = (float *)malloc(sizeof(float) * (size_t)H);
  double *x8 = (double *)malloc(sizeof(double) * (size_t)H);
  double *y = (double *)malloc(sizeof(double) * (size_t)H);
  int rc = 0;
  for (int64_t t = 0; t < T && rc == 0; ++t) {
    for (int64_t h = 0; h < H; ++h) x32[h] = (float)oracle_bf16_to_double(x[t * H + h]); /* exact */
    oracle_q8_activations(x32, H, ORACLE_Q8_0_BLOCK, x8, NULL, NULL);
    double *ot = out + t * H;
    for (int64_t h = 0; h < H; ++h) ot[h] = 0.0;
    for (int64_t j = 0; j < k + S && rc == 0; ++j) {
      const int64_t e = j < k ? ids[t * k + j] : E + (j - k); /* then the always-on expert, weight 1 */
      if (!w_gate[e] || !w_up[e] || !w_down[e]) {
        rc = -2;
        break;
      }
      expert_ffn_q8act(w_gate[e], w_up[e], w_down[e], H, I, x8, y);
      const double g = j < k ? gates[t * k + j] : 1.0;
      for (int64_t h = 0; h < H; ++h) ot[h] += g * y[h];
    }
  }
  free(x32);
  free(x8);
  free(y);
  return rc;
}
