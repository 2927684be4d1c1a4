/*
 * onebit_oracle.h -- the ORACLE for the 1-bit Adam optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded C restatement of the method
 * ("1-bit Adam: Communication Efficient Large-Scale Training with Adam's Convergence Speed",
 * Tang et al. 2021), written from the method's description and used as the reference that the CUDA
 * path is checked against.  Only the test suite, the package's smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header, table or constant with the CUDA
 * library, and the CUDA library never calls it.
 *
 * Sources (by page title and section):
 *   [P1] "1-bit Adam: Communication Efficient Large-Scale Training with Adam's Convergence Speed"
 *        (paperlayer summary of arXiv 2102.02888v2): Sec. 3.3 (frozen variance = momentum SGD with a
 *        coordinate-wise learning rate), Sec. 4.1 (error compensation), Sec. 4.3 (1-bit sign + scale
 *        that preserves the magnitude), Sec. 6 (all-to-all, server average + recompress, allgather),
 *        Sec. 11 (per-chunk parameter-server form: worker EC compression, server average and
 *        recompression, broadcast of m_{t+1}).
 *   [P2] "1-bit Adam (Two-Stage Preconditioner-Frozen Error-Compensated Adam)" (AIMech curated page):
 *        summary formulas v_t = b2 v + (1-b2) g^2, m_t = b1 m + (1-b1) g, V = diag(sqrt(v_Tw)+eps),
 *        x_t = x_{t-1} - gamma V^{-1} m_hat_t; a "gather-then-broadcast" exchange in which every
 *        worker keeps an error memory delta^(i) and every server shard keeps one, epsilon.
 *   [P4] "1-bit Adam" (codewithpapers method page): scale = |compensated| / |quantized|.
 *
 * Precision.  The pages do not fix a precision.  State (x, m, v/den, worker and server errors) is
 * fp32 as the workload defines it, and every elementwise step is evaluated in fp32 in one fixed
 * operation order, because the sign of an fp32 value decides an output bit: both this oracle and the
 * CUDA path take that decision in fp32.  Norms are taken in double (exact squares, compensated sum),
 * then sqrt(sum/len) in double, rounded once to fp32.  Build with -ffp-contract=off (no fused
 * multiply-add anywhere).
 *
 * Layout (all host memory, caller-owned).  A parameter list has T tensors of numel L_k (L_k >= 0);
 * per-element arrays are the concatenation of the tensors without padding (D = sum L_k, tensor k at
 * offset sum_{k'<k} L_k').  Sign words: tensor k owns ceil(L_k/32) uint32 words, concatenated
 * (W = sum ceil(L_k/32)); bit b of word w of tensor k is element 32w+b; a set bit means the value is
 * >= 0 (so +0 and -0 give 1, NaN gives 0); bits past L_k are 0.  Scales are per tensor: a worker has
 * one scale per tensor, a tensor has n server shards (Sec. 11 of [P1]: parameter server per chunk).
 * Shard rule (the pages are silent): S_k = 32*ceil(L_k/(32 n)), shard j = [j S_k, min((j+1)S_k, L_k)),
 * which may be short or empty; an empty shard has scale 0.
 */
#ifndef ONEBIT_ORACLE_H
#define ONEBIT_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORA_F32 = 0, ORA_F16 = 1, ORA_BF16 = 2 };

typedef struct {
  float beta1;              /* b1 */
  float beta2;              /* b2 */
  float eps;                /* epsilon in V = diag(sqrt(v) + epsilon) */
  float lr;                 /* gamma */
  int32_t n_workers;        /* n >= 1 */
  int32_t n_tensors;        /* T >= 1 */
  const int64_t* numel;     /* [T] */
  int32_t grad_dtype;       /* ORA_F32 / ORA_F16 / ORA_BF16 */
  int32_t bias_correction;  /* 0: the pages' formulas; 1: Kingma-Ba bias correction in warm-up */
} ora_config;

/* ---- element helpers ---- */
float ora_half_to_float(uint16_t h);       /* IEEE binary16 -> binary32, exact */
float ora_bf16_to_float(uint16_t b);       /* bfloat16 -> binary32, exact */
float ora_grad_value(const void* g, int32_t dtype, int64_t e);
int64_t ora_words(int64_t len);            /* ceil(len / 32) */
void ora_shard(int64_t len, int32_t n, int32_t j, int64_t* lo, int64_t* hi);

/* ---- the 1-bit compressor ([P1] Sec. 4.3, [P4]) ---- */
float ora_rms(const float* v, int64_t len);                       /* ||v||_2 / sqrt(len); 0 if len == 0 */
void ora_pack_signs(const float* v, int64_t len, uint32_t* words); /* bit = (v >= 0) */
void ora_unpack_signs(const uint32_t* words, int64_t len, float scale, float* out); /* +-scale */
/* scale = ora_rms(c); words = signs of c; err = c - scale * sign(c).  Returns the scale. */
float ora_compress(const float* c, int64_t len, uint32_t* words, float* err);

/* ||v||_2 in double (exact squares, compensated sum, one sqrt): the norm of the variance whose
 * stabilisation during warm-up motivates freezing the variance ([P1] Sec. 3.3). */
double ora_norm2(const float* v, int64_t len);

/* ---- the optimizer stages ---- */
/* One uncompressed Adam step on the mean of the n workers' gradients ([P2] summary formulas).
 * t is the 1-based index of this step (used only by bias correction).
 * grads: host array of n*T pointers, grads[i*T+k] -> L_k values of grad_dtype. */
int ora_warmup_step(const ora_config* cfg, int64_t t, float* x, float* m, float* v,
                    const void* const* grads);
/* den = sqrt(v) + eps after t_freeze warm-up steps (V of [P2]); with bias correction
 * v is first divided by (1 - b2^t_freeze). */
int ora_freeze(const ora_config* cfg, int64_t t_freeze, const float* v, float* den);
/* One compression-stage step ([P1] Sec. 11, [P2] mechanism 2):
 *   worker i:  m_i = b1 m + (1-b1) g_i;  c_i = m_i + delta_i;  per tensor k:
 *              s_ik = rms(c_i on k);  bits_i = sign(c_i);  delta_i = c_i - s_ik sign(c_i)
 *   server (tensor k, shard j): a = (sum_{i=0..n-1} s_ik sign_i) / n + eps_srv
 *              S_kj = rms(a on the shard);  bitsS = sign(a);  eps_srv = a - S_kj sign(a)
 *   broadcast: m = S_kj sign(a) (the shared momentum);  x = x - lr * (m / den)
 * delta: [n][D]; eps_srv: [D]; wbits: [n][W]; wscale: [n][T]; sbits: [W]; sscale: [T][n]. */
int ora_compress_step(const ora_config* cfg, float* x, float* m, const float* den, float* delta,
                      float* eps_srv, const void* const* grads, uint32_t* wbits, float* wscale,
                      uint32_t* sbits, float* sscale);

/* The baseline the method is contrasted with ([P1] Sec. 3.2 and 4.2): error-compensated 1-bit
 * compression applied to the GRADIENTS, with plain Adam on the result.  t is the 1-based step index
 * (bias correction only).
 *   worker i:  c_i = g_i + delta_i;  per tensor: s_ik = rms(c_i);  bits_i = sign(c_i);
 *              delta_i = c_i - s_ik sign(c_i)
 *   server:    a = (sum_i s_ik sign_i) / n + eps_srv;  per shard: S = rms(a);  eps_srv = a - S sign(a)
 *   every worker:  g_hat = S sign(a);  m = b1 m + (1-b1) g_hat;  v = b2 v + (1-b2) g_hat^2;
 *              x = x - lr * (mh / (sqrt(vh) + eps))   (mh, vh bias-corrected if configured)
 * Same array layouts as ora_compress_step. */
int ora_ec_adam_step(const ora_config* cfg, int64_t t, float* x, float* m, float* v, float* delta,
                     float* eps_srv, const void* const* grads, uint32_t* wbits, float* wscale, uint32_t* sbits,
                     float* sscale);

#ifdef __cplusplus
}
#endif
#endif
