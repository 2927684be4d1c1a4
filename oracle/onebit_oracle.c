/*
 * onebit_oracle.c -- ORACLE (test infrastructure only; see onebit_oracle.h for the sources, the
 * precision reading and the layout).  Plain loops in the order the method states its steps.
 * Compile with: gcc -O2 -ffp-contract=off -fPIC -shared onebit_oracle.c -lm
 */
#include "onebit_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ element helpers */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
float ora_half_to_float(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int frac = h & 0x3ff;
  float mag;
  if (expo == 0) {
    mag = ldexpf((float)frac, -24);                 /* subnormal: frac * 2^-24 */
  } else if (expo == 31) {
    mag = frac ? NAN : INFINITY;
  } else {
    mag = ldexpf((float)(1024 + frac), expo - 25);  /* (1 + frac/1024) * 2^(expo-15) */
  }
  return sign ? -mag : mag;
}

/* bfloat16 is the upper half of a binary32. */
float ora_bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

float ora_grad_value(const void* g, int32_t dtype, int64_t e) {
  if (dtype == ORA_F32) return ((const float*)g)[e];
  if (dtype == ORA_F16) return ora_half_to_float(((const uint16_t*)g)[e]);
  return ora_bf16_to_float(((const uint16_t*)g)[e]);
}

int64_t ora_words(int64_t len) { return (len + 31) / 32; }

void ora_shard(int64_t len, int32_t n, int32_t j, int64_t* lo, int64_t* hi) {
  int64_t per = 32 * ((len + 32 * (int64_t)n - 1) / (32 * (int64_t)n));
  int64_t a = (int64_t)j * per, b = a + per;
  if (a > len) a = len;
  if (b > len) b = len;
  *lo = a;
  *hi = b;
}

/* ------------------------------------------------------------------ the compressor */

/* ||v||_2 / sqrt(len).  Squares of fp32 values are exact in double; the sum is a Neumaier
 * compensated sum; sqrt(sum / len) in double, rounded once to fp32. */
float ora_rms(const float* v, int64_t len) {
  if (len <= 0) return 0.0f;
  double sum = 0.0, comp = 0.0;
  for (int64_t e = 0; e < len; ++e) {
    double sq = (double)v[e] * (double)v[e];
    double t = sum + sq;
    if (fabs(sum) >= fabs(sq))
      comp += (sum - t) + sq;
    else
      comp += (sq - t) + sum;
    sum = t;
  }
  return (float)sqrt((sum + comp) / (double)len);
}

double ora_norm2(const float* v, int64_t len) {
  double sum = 0.0, comp = 0.0;
  for (int64_t e = 0; e < len; ++e) {
    double sq = (double)v[e] * (double)v[e];
    double t = sum + sq;
    if (fabs(sum) >= fabs(sq))
      comp += (sum - t) + sq;
    else
      comp += (sq - t) + sum;
    sum = t;
  }
  return sqrt(sum + comp);
}

void ora_pack_signs(const float* v, int64_t len, uint32_t* words) {
  int64_t nw = ora_words(len);
  for (int64_t w = 0; w < nw; ++w) words[w] = 0u;
  for (int64_t e = 0; e < len; ++e)
    if (v[e] >= 0.0f) words[e / 32] |= 1u << (e % 32);
}

void ora_unpack_signs(const uint32_t* words, int64_t len, float scale, float* out) {
  for (int64_t e = 0; e < len; ++e) out[e] = ((words[e / 32] >> (e % 32)) & 1u) ? scale : -scale;
}

float ora_compress(const float* c, int64_t len, uint32_t* words, float* err) {
  float s = ora_rms(c, len);
  ora_pack_signs(c, len, words);
  for (int64_t e = 0; e < len; ++e) err[e] = (c[e] >= 0.0f) ? c[e] - s : c[e] + s;
  return s;
}

/* ------------------------------------------------------------------ stages */

static int64_t total_numel(const ora_config* cfg) {
  int64_t d = 0;
  for (int k = 0; k < cfg->n_tensors; ++k) d += cfg->numel[k];
  return d;
}

static int64_t total_words(const ora_config* cfg) {
  int64_t w = 0;
  for (int k = 0; k < cfg->n_tensors; ++k) w += ora_words(cfg->numel[k]);
  return w;
}

static int check_cfg(const ora_config* cfg) {
  if (!cfg || cfg->n_workers < 1 || cfg->n_tensors < 1 || !cfg->numel) return 1;
  for (int k = 0; k < cfg->n_tensors; ++k)
    if (cfg->numel[k] < 0) return 1;
  return 0;
}

/* One Adam update of one element with gradient g ([P2] summary formulas). */
static void adam_element(const ora_config* cfg, float bc1, float bc2, float g, float* m, float* v, float* x) {
  const float b1 = cfg->beta1, omb1 = 1.0f - cfg->beta1;
  const float b2 = cfg->beta2, omb2 = 1.0f - cfg->beta2;
  *m = b1 * *m + omb1 * g;
  *v = b2 * *v + omb2 * (g * g);
  float mh = *m, vh = *v;
  if (cfg->bias_correction) {
    mh = mh / bc1;
    vh = vh / bc2;
  }
  *x = *x - cfg->lr * (mh / (sqrtf(vh) + cfg->eps));
}

int ora_warmup_step(const ora_config* cfg, int64_t t, float* x, float* m, float* v,
                    const void* const* grads) {
  if (check_cfg(cfg) || t < 1) return 1;
  const int n = cfg->n_workers, T = cfg->n_tensors;
  const float bc1 = (float)(1.0 - pow((double)cfg->beta1, (double)t));
  const float bc2 = (float)(1.0 - pow((double)cfg->beta2, (double)t));
  int64_t off = 0;
  for (int k = 0; k < T; ++k) {
    const int64_t L = cfg->numel[k];
    for (int64_t e = 0; e < L; ++e) {
      /* the uncompressed allreduce of the warm-up stage: mean of the n worker gradients,
       * summed in worker order */
      float acc = 0.0f;
      for (int i = 0; i < n; ++i) acc = acc + ora_grad_value(grads[(int64_t)i * T + k], cfg->grad_dtype, e);
      const float g = acc / (float)n;
      const int64_t p = off + e;
      adam_element(cfg, bc1, bc2, g, &m[p], &v[p], &x[p]);
    }
    off += L;
  }
  return 0;
}

int ora_freeze(const ora_config* cfg, int64_t t_freeze, const float* v, float* den) {
  if (check_cfg(cfg) || t_freeze < 1) return 1;
  const int64_t D = total_numel(cfg);
  const float bc2 = (float)(1.0 - pow((double)cfg->beta2, (double)t_freeze));
  for (int64_t p = 0; p < D; ++p) {
    const float vu = cfg->bias_correction ? v[p] / bc2 : v[p];
    den[p] = sqrtf(vu) + cfg->eps;
  }
  return 0;
}

/* Each worker, each tensor: 1-bit compression of c with error feedback ([P1] Sec. 4.3, 11). */
static void workers_compress(const ora_config* cfg, const float* c, float* delta, uint32_t* wbits, float* wscale) {
  const int n = cfg->n_workers, T = cfg->n_tensors;
  const int64_t D = total_numel(cfg), W = total_words(cfg);
  for (int i = 0; i < n; ++i) {
    int64_t off = 0, woff = 0;
    for (int k = 0; k < T; ++k) {
      const int64_t L = cfg->numel[k];
      wscale[(int64_t)i * T + k] =
          ora_compress(c + (int64_t)i * D + off, L, wbits + (int64_t)i * W + woff, delta + (int64_t)i * D + off);
      off += L;
      woff += ora_words(L);
    }
  }
}

/* Server shard j of tensor k: average of the n decompressed messages, plus the server error. */
static void server_average(const ora_config* cfg, const uint32_t* wbits, const float* wscale, const float* eps_srv,
                           float* a) {
  const int n = cfg->n_workers, T = cfg->n_tensors;
  const int64_t W = total_words(cfg);
  int64_t off = 0, woff = 0;
  for (int k = 0; k < T; ++k) {
    const int64_t L = cfg->numel[k];
    for (int64_t e = 0; e < L; ++e) {
      float acc = 0.0f;
      for (int i = 0; i < n; ++i) {
        const uint32_t bit = (wbits[(int64_t)i * W + woff + e / 32] >> (e % 32)) & 1u;
        const float s = wscale[(int64_t)i * T + k];
        acc = acc + (bit ? s : -s);
      }
      a[off + e] = acc / (float)n + eps_srv[off + e];
    }
    off += L;
    woff += ora_words(L);
  }
}

/* Recompress every shard with server error feedback; bcast receives the broadcast S*sign(a). */
static void server_recompress(const ora_config* cfg, const float* a, float* eps_srv, uint32_t* sbits, float* sscale,
                              float* bcast) {
  const int n = cfg->n_workers, T = cfg->n_tensors;
  int64_t off = 0, woff = 0;
  for (int k = 0; k < T; ++k) {
    const int64_t L = cfg->numel[k];
    for (int64_t w = 0; w < ora_words(L); ++w) sbits[woff + w] = 0u;
    for (int j = 0; j < n; ++j) {
      int64_t lo, hi;
      ora_shard(L, n, j, &lo, &hi);
      const float S = ora_rms(a + off + lo, hi - lo);
      sscale[(int64_t)k * n + j] = S;
      for (int64_t e = lo; e < hi; ++e) {
        const int64_t p = off + e;
        const int bit = a[p] >= 0.0f;
        if (bit) sbits[woff + e / 32] |= 1u << (e % 32);
        eps_srv[p] = bit ? a[p] - S : a[p] + S;
        bcast[p] = bit ? S : -S;
      }
    }
    off += L;
    woff += ora_words(L);
  }
}

/* Scratch for one step: c [n][D], a [D], broadcast [D]. */
static float* step_scratch(const ora_config* cfg, float** c, float** a, float** b) {
  const int64_t D = total_numel(cfg);
  const size_t d1 = (size_t)(D > 0 ? D : 1);
  float* buf = (float*)malloc(sizeof(float) * d1 * ((size_t)cfg->n_workers + 2));
  if (!buf) return NULL;
  *c = buf;
  *a = buf + d1 * (size_t)cfg->n_workers;
  *b = *a + d1;
  return buf;
}

int ora_compress_step(const ora_config* cfg, float* x, float* m, const float* den, float* delta,
                      float* eps_srv, const void* const* grads, uint32_t* wbits, float* wscale,
                      uint32_t* sbits, float* sscale) {
  if (check_cfg(cfg)) return 1;
  const int n = cfg->n_workers, T = cfg->n_tensors;
  const int64_t D = total_numel(cfg);
  const float b1 = cfg->beta1, omb1 = 1.0f - cfg->beta1;
  float *c, *a, *bcast;
  float* buf = step_scratch(cfg, &c, &a, &bcast);
  if (!buf) return 2;

  /* 1. each worker: local momentum, then add its error memory */
  for (int i = 0; i < n; ++i) {
    int64_t off = 0;
    for (int k = 0; k < T; ++k) {
      const int64_t L = cfg->numel[k];
      const void* g = grads[(int64_t)i * T + k];
      for (int64_t e = 0; e < L; ++e) {
        const int64_t p = off + e;
        const float mi = b1 * m[p] + omb1 * ora_grad_value(g, cfg->grad_dtype, e);
        c[(int64_t)i * D + p] = mi + delta[(int64_t)i * D + p];
      }
      off += L;
    }
  }
  /* 2-3. worker compression; 4. server average + server error */
  workers_compress(cfg, c, delta, wbits, wscale);
  server_average(cfg, wbits, wscale, eps_srv, a);
  /* 5-7. recompression; the broadcast is the shared m; x -= lr * m / (sqrt(v_frozen) + eps) */
  server_recompress(cfg, a, eps_srv, sbits, sscale, bcast);
  for (int64_t p = 0; p < D; ++p) {
    m[p] = bcast[p];
    x[p] = x[p] - cfg->lr * (m[p] / den[p]);
  }
  free(buf);
  return 0;
}

int ora_ec_adam_step(const ora_config* cfg, int64_t t, float* x, float* m, float* v, float* delta,
                     float* eps_srv, const void* const* grads, uint32_t* wbits, float* wscale, uint32_t* sbits,
                     float* sscale) {
  if (check_cfg(cfg) || t < 1) return 1;
  const int n = cfg->n_workers, T = cfg->n_tensors;
  const int64_t D = total_numel(cfg);
  const float bc1 = (float)(1.0 - pow((double)cfg->beta1, (double)t));
  const float bc2 = (float)(1.0 - pow((double)cfg->beta2, (double)t));
  float *c, *a, *bcast;
  float* buf = step_scratch(cfg, &c, &a, &bcast);
  if (!buf) return 2;

  /* 1. each worker: its gradient plus its error memory */
  for (int i = 0; i < n; ++i) {
    int64_t off = 0;
    for (int k = 0; k < T; ++k) {
      const int64_t L = cfg->numel[k];
      const void* g = grads[(int64_t)i * T + k];
      for (int64_t e = 0; e < L; ++e) {
        const int64_t p = off + e;
        c[(int64_t)i * D + p] = ora_grad_value(g, cfg->grad_dtype, e) + delta[(int64_t)i * D + p];
      }
      off += L;
    }
  }
  /* 2. worker compression; 3. server average + error; 4. recompression and broadcast */
  workers_compress(cfg, c, delta, wbits, wscale);
  server_average(cfg, wbits, wscale, eps_srv, a);
  server_recompress(cfg, a, eps_srv, sbits, sscale, bcast);
  /* 5. every worker runs Adam on the broadcast gradient */
  for (int64_t p = 0; p < D; ++p) adam_element(cfg, bc1, bc2, bcast[p], &m[p], &v[p], &x[p]);
  free(buf);
  return 0;
}
