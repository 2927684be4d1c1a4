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

int ora_warmup_step(const ora_config* cfg, int64_t t, float* x, float* m, float* v,
                    const void* const* grads) {
  if (check_cfg(cfg) || t < 1) return 1;
  const int n = cfg->n_workers, T = cfg->n_tensors;
  const float b1 = cfg->beta1, omb1 = 1.0f - cfg->beta1;
  const float b2 = cfg->beta2, omb2 = 1.0f - cfg->beta2;
  const float lr = cfg->lr, eps = cfg->eps;
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
      m[p] = b1 * m[p] + omb1 * g;
      v[p] = b2 * v[p] + omb2 * (g * g);
      float mh = m[p], vh = v[p];
      if (cfg->bias_correction) {
        mh = mh / bc1;
        vh = vh / bc2;
      }
      x[p] = x[p] - lr * (mh / (sqrtf(vh) + eps));
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

int ora_compress_step(const ora_config* cfg, float* x, float* m, const float* den, float* delta,
                      float* eps_srv, const void* const* grads, uint32_t* wbits, float* wscale,
                      uint32_t* sbits, float* sscale) {
  if (check_cfg(cfg)) return 1;
  const int n = cfg->n_workers, T = cfg->n_tensors;
  const int64_t D = total_numel(cfg), W = total_words(cfg);
  const float b1 = cfg->beta1, omb1 = 1.0f - cfg->beta1;
  const float lr = cfg->lr;

  float* c = (float*)malloc(sizeof(float) * (size_t)(D > 0 ? D : 1) * (size_t)n);
  float* a = (float*)malloc(sizeof(float) * (size_t)(D > 0 ? D : 1));
  if (!c || !a) {
    free(c);
    free(a);
    return 2;
  }

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

  /* 2-3. each worker, each tensor: 1-bit compression with error feedback */
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

  /* 4. server shard j of tensor k: average of the n decompressed messages, plus the server error */
  {
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

  /* 5-7. recompress each shard with server error feedback; the broadcast result is the shared m;
   * preconditioned update x -= lr * m / (sqrt(v_frozen) + eps) */
  {
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
          m[p] = bit ? S : -S;
          x[p] = x[p] - lr * (m[p] / den[p]);
        }
      }
      off += L;
      woff += ora_words(L);
    }
  }

  free(c);
  free(a);
  (void)D;
  return 0;
}
