/*
 * oracle.c -- plain, slow, fp64 CPU oracle of the MLA KV prolog.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * library: it reads the same input bits and computes the definition of each
 * step, one scalar loop at a time, in double precision.
 *
 * Sources (web pages; quoted by title and section):
 *   [MIG] "DeepSeek-V2-Lite-Chat MLA KV Prolog 迁移指南：基于 PyPTO 融合算子与
 *         aclgraph 的 NPU 推理优化实践" (dpshk.com/news/4811369)
 *   [R1]  "DeepSeek-R1或Kimi-K2模型在NPU实现高性能推理"
 *         (gitcode.com/cann/cann-recipes-infer, models/deepseek_r1 README)
 *
 * The seven steps of the KV prolog are listed in [MIG] §"背景：为什么要迁移
 * MLA KV Prolog" (kv_a_proj, split, RMSNorm, kv_b_proj, reshape+split, RoPE,
 * assemble); the tensor shapes are in [MIG] §"精度验证：Golden 对比测试"; the
 * Python flow (reshape to [b*s, hidden], matmul with the pre-transposed
 * weight, slice, rms_norm, kv_b matmul, view into k_nope/value, RoPE,
 * assemble, reshape back to [b, H, s, .]) is in [MIG] §"源码级原理：KV Prolog
 * 的混合优化实现".  Readings where the pages are silent:
 *   - RoPE: [MIG] only says "x*cos + x_rot*sin".  The DeepSeek-V2 convention
 *     is used: de-interleave (x'[j] = x[2j], x'[32+j] = x[2j+1]) then
 *     out = x'*cos[p] + rotate_half(x')*sin[p], rotate_half(x') =
 *     [-x'[32:], x'[:32]]; the output stays in de-interleaved order.
 *   - No intermediate rounding: every step is carried in double.
 *   - RMSNorm: mean of squares over the 512 latent entries, eps inside the
 *     square root, gamma after the normalisation, no bias.
 *   - W8A8 (the quant mode named in [R1] §"权重转换"): per-token symmetric
 *     int8 activation quantisation in float32 (amax, 127/amax, one multiply,
 *     round-to-nearest-even, clamp to [-127,127]); int8 weights with one fp32
 *     scale per output channel; integer accumulation; dequantisation
 *     acc * s_x * s_w.
 *
 * Build: gcc -O2 -std=c11 -fno-fast-math -ffp-contract=off [-fopenmp] -shared
 * -fPIC.  -ffp-contract=off matters: the float32 quantisation below must be
 * one rounding per operation on every host (aarch64 gcc would otherwise fuse
 * multiply-adds).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* 16-bit float encodings (IEEE binary16 and bfloat16), written from the
 * format definitions: sign | exponent | fraction, bias 15 / 127.           */
/* ------------------------------------------------------------------ */

double oracle_f16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int frac = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
  } else if (expo == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    v = ldexp(1024.0 + frac, expo - 15 - 10);
  }
  return sign ? -v : v;
}

double oracle_bf16_to_double(uint16_t b) {
  int sign = (b >> 15) & 1;
  int expo = (b >> 7) & 0xff;
  int frac = b & 0x7f;
  double v;
  if (expo == 0) {
    v = ldexp((double)frac, -133); /* frac * 2^-126 * 2^-7 */
  } else if (expo == 255) {
    v = frac ? NAN : INFINITY;
  } else {
    v = ldexp(128.0 + frac, expo - 127 - 7);
  }
  return sign ? -v : v;
}

/* Round a double to a binary floating format with `mant` fraction bits,
 * minimum normal exponent `emin` and maximum exponent `emax`, to nearest,
 * ties to even, and return the encoded bits (1 sign, exponent, mant).      */
static uint16_t encode_rne(double x, int mant, int emin, int emax, int ebits) {
  uint16_t sign = (uint16_t)(signbit(x) ? (1u << (mant + ebits)) : 0u);
  uint16_t expmask = (uint16_t)((1u << ebits) - 1u);
  if (isnan(x)) return (uint16_t)((expmask << mant) | (1u << (mant - 1)));
  double a = fabs(x);
  if (isinf(a)) return (uint16_t)(sign | (expmask << mant));
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);          /* a = m * 2^e2, m in [0.5, 1)  ->  a in [2^(e2-1), 2^e2) */
  int E = e2 - 1;
  if (E < emin) E = emin; /* subnormal range shares the quantum of the smallest binade */
  double quantum = ldexp(1.0, E - mant);
  double q = rint(a / quantum); /* exact scaling by a power of two; rint = RNE */
  double r = q * quantum;
  /* overflow: the largest finite value is (2 - 2^-mant) * 2^emax */
  double maxfin = ldexp(2.0 - ldexp(1.0, -mant), emax);
  if (r > maxfin) return (uint16_t)(sign | (expmask << mant));
  if (r < ldexp(1.0, emin)) {
    /* subnormal (or rounded up exactly to the smallest normal, handled below) */
    uint32_t f = (uint32_t)q; /* q < 2^mant */
    return (uint16_t)(sign | f);
  }
  int er;
  frexp(r, &er);
  int Er = er - 1;
  double frac = ldexp(r, mant - Er) - ldexp(1.0, mant);
  uint32_t bexp = (uint32_t)(Er + (int)expmask / 2);
  return (uint16_t)(sign | (bexp << mant) | (uint32_t)frac);
}

uint16_t oracle_double_to_f16(double x) { return encode_rne(x, 10, -14, 15, 5); }
uint16_t oracle_double_to_bf16(double x) { return encode_rne(x, 7, -126, 127, 8); }

static double load16(const uint16_t* p, int64_t i, int dtype) {
  return dtype == 0 ? oracle_f16_to_double(p[i]) : oracle_bf16_to_double(p[i]);
}

/* ------------------------------------------------------------------ */
/* Step kernels, each the plain definition.                             */
/* ------------------------------------------------------------------ */

/* kv_a_proj / kv_b_proj for one token row: y[n] = sum_k x[k] * W[k][n],
 * W stored [in, out] row-major (the pre-transposed weight of [MIG]
 * §"源码级原理", step 1).                                                  */
void oracle_vec_matmul(const double* x, const double* W, int64_t K, int64_t N, double* y) {
  for (int64_t n = 0; n < N; ++n) {
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) acc += x[k] * W[k * N + n];
    y[n] = acc;
  }
}

/* RMSNorm ([MIG] §"背景" step 3, §"源码级原理" step 3):
 * y = x / sqrt(mean(x^2) + eps) * gamma.                                 */
void oracle_rmsnorm(const double* x, int64_t n, const double* gamma, double eps, double* y) {
  double ss = 0.0;
  for (int64_t i = 0; i < n; ++i) ss += x[i] * x[i];
  double denom = sqrt(ss / (double)n + eps);
  for (int64_t i = 0; i < n; ++i) y[i] = x[i] / denom * gamma[i];
}

/* RoPE on one rope vector of even length d ([MIG] §"背景" step 6; the
 * de-interleave + rotate_half reading, see the file header).  cos_row and
 * sin_row are the caller's fp32 table rows for this token's position.      */
void oracle_rope(const double* x, int d, const float* cos_row, const float* sin_row, double* y) {
  int half = d / 2;
  double xd[256]; /* de-interleaved copy; d <= 256 */
  for (int j = 0; j < half; ++j) {
    xd[j] = x[2 * j];
    xd[half + j] = x[2 * j + 1];
  }
  for (int i = 0; i < d; ++i) {
    double rot = (i < half) ? -xd[i + half] : xd[i - half];
    y[i] = xd[i] * (double)cos_row[i] + rot * (double)sin_row[i];
  }
}

/* ------------------------------------------------------------------ */
/* Whole KV prolog                                                      */
/* ------------------------------------------------------------------ */

typedef struct {
  int64_t hidden, rank, rope, heads, nope, vdim, max_pos;
  double eps;
  int dtype; /* 0 = fp16, 1 = bf16 bits */
} oracle_dims;

/* Promote n 16-bit values (fp16 or bf16 bits) to double, bit-exactly. */
void oracle_promote16(const uint16_t* src, int64_t n, int dtype, double* dst) {
  for (int64_t i = 0; i < n; ++i) dst[i] = load16(src, i, dtype);
}

/* One token row: the seven steps in the pages' order.
 *   x [hidden]: the token's hidden row, promoted to double.
 *   Wa [hidden, rank+rope], g [rank], Wb [rank, heads*(nope+vdim)]: the
 *   weights promoted to double, [in, out] row-major (the pre-transposed
 *   layout of [MIG] §"源码级原理" step 1).
 *   cos_row / sin_row [rope]: fp32 table rows at this token's position.
 *   Outputs for this row: k_nope [heads][nope], value [heads][vdim],
 *   k_pe [rope].                                                          */
void oracle_kv_prolog_token(const oracle_dims* d, const double* x, const double* Wa,
                            const double* g, const double* Wb, const float* cos_row,
                            const float* sin_row, double* k_nope, double* value, double* k_pe) {
  const int64_t h = d->hidden, r = d->rank, dr = d->rope, H = d->heads;
  const int64_t na = r + dr, hd = d->nope + d->vdim, nb = H * hd;
  double* C = (double*)malloc(sizeof(double) * na);
  double* n = (double*)malloc(sizeof(double) * r);
  double* KV = (double*)malloc(sizeof(double) * nb);

  /* step 1: kv_a_proj, C = x * W_kva */
  oracle_vec_matmul(x, Wa, h, na, C);
  /* step 2: split -> compressed_kv = C[0:r], k_pe = C[r:r+dr] */
  const double* ckv = C;
  const double* kpe = C + r;
  /* step 3: RMSNorm of compressed_kv */
  oracle_rmsnorm(ckv, r, g, d->eps, n);
  /* step 4: kv_b_proj, KV = n * W_kvb */
  oracle_vec_matmul(n, Wb, r, nb, KV);
  /* step 5: reshape [H, nope+v] and split into k_nope / value */
  for (int64_t hh = 0; hh < H; ++hh) {
    for (int64_t i = 0; i < d->nope; ++i) k_nope[hh * d->nope + i] = KV[hh * hd + i];
    for (int64_t i = 0; i < d->vdim; ++i) value[hh * d->vdim + i] = KV[hh * hd + d->nope + i];
  }
  /* step 6: RoPE on k_pe */
  oracle_rope(kpe, (int)dr, cos_row, sin_row, k_pe);
  free(C); free(n); free(KV);
}

/* Step 7 (assemble): full outputs in head-major layout
 *   k_nope [b, H, s, nope], value [b, H, s, vdim], k_pe [b, 1, s, rope]
 * with token row t = bi*s + si ([MIG] §"源码级原理" steps 1 and 5).
 * Inputs are the raw 16-bit bits (dtype 0 = fp16, 1 = bf16).  `rows`
 * (length n_rows) selects which token rows to compute; rows not listed are
 * left untouched.  nthreads > 1 splits the rows over OpenMP threads when
 * the library was built with OpenMP.  Returns the number of listed rows
 * whose position was outside [0, max_pos) (those rows are not written).   */
int oracle_kv_prolog(const oracle_dims* d, int64_t b, int64_t s, const uint16_t* hidden,
                     const int32_t* positions, const uint16_t* W_kva, const uint16_t* gamma,
                     const uint16_t* W_kvb, const float* cosb, const float* sinb,
                     const int64_t* rows, int64_t n_rows, int nthreads, double* k_nope,
                     double* value, double* k_pe) {
  const int64_t h = d->hidden, r = d->rank, H = d->heads, dn = d->nope, dv = d->vdim,
                dr = d->rope;
  const int64_t na = r + dr, nb = H * (dn + dv);
  int bad = 0;
  (void)b;
  (void)nthreads;
  /* read the I/O-dtype weights bit-exactly and promote them to double */
  double* Wa = (double*)malloc(sizeof(double) * h * na);
  double* Wb = (double*)malloc(sizeof(double) * r * nb);
  double* g = (double*)malloc(sizeof(double) * r);
  oracle_promote16(W_kva, h * na, d->dtype, Wa);
  oracle_promote16(W_kvb, r * nb, d->dtype, Wb);
  oracle_promote16(gamma, r, d->dtype, g);
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1) reduction(+ : bad)
#endif
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t t = rows[i];
    int64_t bi = t / s, si = t % s;
    int32_t p = positions[t];
    if (p < 0 || p >= d->max_pos) {
      bad += 1;
      continue;
    }
    double* x = (double*)malloc(sizeof(double) * h);
    double* kn = (double*)malloc(sizeof(double) * H * dn);
    double* vv = (double*)malloc(sizeof(double) * H * dv);
    double kp[256];
    oracle_promote16(hidden + t * h, h, d->dtype, x);
    oracle_kv_prolog_token(d, x, Wa, g, Wb, cosb + (int64_t)p * dr, sinb + (int64_t)p * dr, kn,
                           vv, kp);
    for (int64_t hh = 0; hh < H; ++hh) {
      for (int64_t e = 0; e < dn; ++e) k_nope[((bi * H + hh) * s + si) * dn + e] = kn[hh * dn + e];
      for (int64_t e = 0; e < dv; ++e) value[((bi * H + hh) * s + si) * dv + e] = vv[hh * dv + e];
    }
    for (int64_t e = 0; e < dr; ++e) k_pe[(bi * s + si) * dr + e] = kp[e];
    free(x); free(kn); free(vv);
  }
  free(Wa); free(Wb); free(g);
  return bad;
}

/* Latent-cache variant: steps 1, 2, 3 and 6 only -- the normalised
 * compressed_kv row that a weight-absorbed attention caches instead of
 * k_nope / value, and the roped k_pe.  latent [T, rank] (row t = bi*s + si),
 * k_pe [b, 1, s, rope].  Same row selection, threads and return value as
 * oracle_kv_prolog.                                                        */
int oracle_kv_latent(const oracle_dims* d, int64_t b, int64_t s, const uint16_t* hidden,
                     const int32_t* positions, const uint16_t* W_kva, const uint16_t* gamma,
                     const float* cosb, const float* sinb, const int64_t* rows, int64_t n_rows,
                     int nthreads, double* latent, double* k_pe) {
  const int64_t h = d->hidden, r = d->rank, dr = d->rope, na = r + dr;
  int bad = 0;
  (void)b;
  (void)nthreads;
  double* Wa = (double*)malloc(sizeof(double) * h * na);
  double* g = (double*)malloc(sizeof(double) * r);
  oracle_promote16(W_kva, h * na, d->dtype, Wa);
  oracle_promote16(gamma, r, d->dtype, g);
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1) reduction(+ : bad)
#endif
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t t = rows[i];
    int32_t p = positions[t];
    if (p < 0 || p >= d->max_pos) {
      bad += 1;
      continue;
    }
    double* x = (double*)malloc(sizeof(double) * h);
    double* C = (double*)malloc(sizeof(double) * na);
    oracle_promote16(hidden + t * h, h, d->dtype, x);
    oracle_vec_matmul(x, Wa, h, na, C);                 /* step 1 */
    oracle_rmsnorm(C, r, g, d->eps, latent + t * r);    /* steps 2, 3 */
    oracle_rope(C + r, (int)dr, cosb + (int64_t)p * dr, sinb + (int64_t)p * dr,
                k_pe + t * dr);                         /* step 6 */
    free(x); free(C);
  }
  free(Wa); free(g);
  return bad;
}

/* ------------------------------------------------------------------ */
/* W8A8 full MLA prolog (Q side + KV side), int8 weights                */
/* ------------------------------------------------------------------ */

/* Per-token symmetric int8 quantisation in float32.  Every operation is a
 * single IEEE float32 operation: amax = max|x|; inv = 127/amax;
 * q = clamp(rint(x*inv), -127, 127); s = amax/127.  amax == 0 gives q = 0
 * and s = 0.                                                               */
void oracle_quant_row_f32(const float* x, int64_t n, int8_t* q, float* s) {
  float amax = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  if (amax == 0.0f) {
    for (int64_t i = 0; i < n; ++i) q[i] = 0;
    *s = 0.0f;
    return;
  }
  volatile float inv = 127.0f / amax;
  for (int64_t i = 0; i < n; ++i) {
    volatile float y = x[i] * inv;
    float r = rintf(y);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    q[i] = (int8_t)r;
  }
  volatile float sc = amax / 127.0f;
  *s = sc;
}

/* Integer GEMM row: acc[n] = sum_k q[k] * W[k][n], W int8 [K, N] row-major,
 * accumulated in int64 (the brute-force definition).                      */
void oracle_int_gemm_row(const int8_t* q, const int8_t* W, int64_t K, int64_t N, int64_t* acc) {
  for (int64_t n = 0; n < N; ++n) {
    int64_t a = 0;
    for (int64_t k = 0; k < K; ++k) a += (int64_t)q[k] * (int64_t)W[k * N + n];
    acc[n] = a;
  }
}

/* Full int GEMM over M rows (used by the accumulator bit-exactness tests). */
void oracle_int_gemm(const int8_t* A, const int8_t* W, int64_t M, int64_t K, int64_t N,
                     int64_t* acc) {
  for (int64_t m = 0; m < M; ++m) oracle_int_gemm_row(A + m * K, W, K, N, acc + m * N);
}

typedef struct {
  int64_t hidden, q_rank, kv_rank, rope, heads, nope, vdim, max_pos;
  double eps;
} oracle_w8a8_dims;

/* One token of the W8A8 prolog.  hidden: bf16 bits [T, hidden].
 * W_qa [hidden, q_rank], W_qb [q_rank, heads*(nope+rope)],
 * W_kva [hidden, kv_rank+rope], W_kvb [kv_rank, heads*(nope+vdim)]: int8,
 * each with fp32 per-output-channel scales.  gamma_q [q_rank], gamma_kv
 * [kv_rank]: bf16 bits.  Outputs (double): q_nope [heads][nope], q_pe
 * [heads][rope], k_nope [heads][nope], value [heads][vdim], k_pe [rope].
 * Optional debug outputs (may be NULL): the int8 activations and scales fed
 * to q_b and kv_b.                                                         */
int oracle_w8a8_token(const oracle_w8a8_dims* d, int64_t t, const uint16_t* hidden,
                      const int32_t* positions, const int8_t* W_qa, const float* s_qa,
                      const uint16_t* gamma_q, const int8_t* W_qb, const float* s_qb,
                      const int8_t* W_kva, const float* s_kva, const uint16_t* gamma_kv,
                      const int8_t* W_kvb, const float* s_kvb, const float* cosb,
                      const float* sinb, double* q_nope, double* q_pe, double* k_nope,
                      double* value, double* k_pe, int8_t* dbg_q1, float* dbg_s1,
                      int8_t* dbg_c1, float* dbg_s2) {
  const int64_t h = d->hidden, rq = d->q_rank, rk = d->kv_rank, dr = d->rope, H = d->heads;
  const int64_t na = rk + dr, qhd = d->nope + dr, nq = H * qhd, kvhd = d->nope + d->vdim,
                nkv = H * kvhd;
  int32_t p = positions[t];
  if (p < 0 || p >= d->max_pos) return 1;
  const float* crow = cosb + (int64_t)p * dr;
  const float* srow = sinb + (int64_t)p * dr;

  float* xf = (float*)malloc(sizeof(float) * h);
  int8_t* xq = (int8_t*)malloc((size_t)h);
  int64_t nmax = rq;
  if (nq > nmax) nmax = nq;
  if (nkv > nmax) nmax = nkv;
  int64_t* acc_q = (int64_t*)malloc(sizeof(int64_t) * nmax);
  int64_t* acc_a = (int64_t*)malloc(sizeof(int64_t) * na);
  double* yq = (double*)malloc(sizeof(double) * rq);
  double* ya = (double*)malloc(sizeof(double) * na);
  double* gq = (double*)malloc(sizeof(double) * rq);
  double* gk = (double*)malloc(sizeof(double) * rk);
  double* nq_ = (double*)malloc(sizeof(double) * rq);
  double* nk_ = (double*)malloc(sizeof(double) * rk);
  float* nqf = (float*)malloc(sizeof(float) * rq);
  float* nkf = (float*)malloc(sizeof(float) * rk);
  int8_t* q1 = (int8_t*)malloc((size_t)rq);
  int8_t* c1 = (int8_t*)malloc((size_t)rk);
  double* yb = (double*)malloc(sizeof(double) * nmax);
  float s_x, s1, s2;

  /* activation quantisation of the hidden row (shared by q_a and kv_a) */
  for (int64_t k = 0; k < h; ++k) xf[k] = (float)oracle_bf16_to_double(hidden[t * h + k]);
  oracle_quant_row_f32(xf, h, xq, &s_x);

  /* q_a_proj and kv_a_proj: integer GEMMs, then dequantise */
  oracle_int_gemm_row(xq, W_qa, h, rq, acc_q);
  for (int64_t n = 0; n < rq; ++n) yq[n] = (double)acc_q[n] * (double)s_x * (double)s_qa[n];
  oracle_int_gemm_row(xq, W_kva, h, na, acc_a);
  for (int64_t n = 0; n < na; ++n) ya[n] = (double)acc_a[n] * (double)s_x * (double)s_kva[n];

  /* RMSNorms */
  for (int64_t c = 0; c < rq; ++c) gq[c] = oracle_bf16_to_double(gamma_q[c]);
  for (int64_t c = 0; c < rk; ++c) gk[c] = oracle_bf16_to_double(gamma_kv[c]);
  oracle_rmsnorm(yq, rq, gq, d->eps, nq_);
  oracle_rmsnorm(ya, rk, gk, d->eps, nk_);

  /* requantise the normalised vectors (taken to float32, then the float32
   * quantisation above)                                                   */
  for (int64_t c = 0; c < rq; ++c) nqf[c] = (float)nq_[c];
  for (int64_t c = 0; c < rk; ++c) nkf[c] = (float)nk_[c];
  oracle_quant_row_f32(nqf, rq, q1, &s1);
  oracle_quant_row_f32(nkf, rk, c1, &s2);
  if (dbg_q1) memcpy(dbg_q1, q1, (size_t)rq);
  if (dbg_c1) memcpy(dbg_c1, c1, (size_t)rk);
  if (dbg_s1) *dbg_s1 = s1;
  if (dbg_s2) *dbg_s2 = s2;

  /* q_b_proj -> [H, nope+rope] -> q_nope, RoPE(q_pe) */
  oracle_int_gemm_row(q1, W_qb, rq, nq, acc_q);
  for (int64_t j = 0; j < nq; ++j) yb[j] = (double)acc_q[j] * (double)s1 * (double)s_qb[j];
  for (int64_t hh = 0; hh < H; ++hh) {
    for (int64_t i = 0; i < d->nope; ++i) q_nope[hh * d->nope + i] = yb[hh * qhd + i];
    oracle_rope(yb + hh * qhd + d->nope, (int)dr, crow, srow, q_pe + hh * dr);
  }
  /* kv_b_proj -> [H, nope+v] -> k_nope, value */
  oracle_int_gemm_row(c1, W_kvb, rk, nkv, acc_q);
  for (int64_t j = 0; j < nkv; ++j) yb[j] = (double)acc_q[j] * (double)s2 * (double)s_kvb[j];
  for (int64_t hh = 0; hh < H; ++hh) {
    for (int64_t i = 0; i < d->nope; ++i) k_nope[hh * d->nope + i] = yb[hh * kvhd + i];
    for (int64_t i = 0; i < d->vdim; ++i) value[hh * d->vdim + i] = yb[hh * kvhd + d->nope + i];
  }
  /* RoPE(k_pe) */
  oracle_rope(ya + rk, (int)dr, crow, srow, k_pe);

  free(xf); free(xq); free(acc_q); free(acc_a); free(yq); free(ya); free(gq); free(gk);
  free(nq_); free(nk_); free(nqf); free(nkf); free(q1); free(c1); free(yb);
  return 0;
}

/* Head-major assembly of the W8A8 outputs for the listed rows:
 *   q_nope [b, H, s, nope], q_pe [b, H, s, rope], k_nope [b, H, s, nope],
 *   value [b, H, s, vdim], k_pe [b, 1, s, rope].                           */
int oracle_w8a8(const oracle_w8a8_dims* d, int64_t b, int64_t s, const uint16_t* hidden,
                const int32_t* positions, const int8_t* W_qa, const float* s_qa,
                const uint16_t* gamma_q, const int8_t* W_qb, const float* s_qb,
                const int8_t* W_kva, const float* s_kva, const uint16_t* gamma_kv,
                const int8_t* W_kvb, const float* s_kvb, const float* cosb, const float* sinb,
                const int64_t* rows, int64_t n_rows, int nthreads, double* q_nope, double* q_pe,
                double* k_nope, double* value, double* k_pe) {
  const int64_t H = d->heads, dn = d->nope, dv = d->vdim, dr = d->rope;
  int bad = 0;
  (void)b;
  (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1) reduction(+ : bad)
#endif
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t t = rows[i];
    int64_t bi = t / s, si = t % s;
    double* qn = (double*)malloc(sizeof(double) * H * dn);
    double* qp = (double*)malloc(sizeof(double) * H * dr);
    double* kn = (double*)malloc(sizeof(double) * H * dn);
    double* vv = (double*)malloc(sizeof(double) * H * dv);
    double kp[256];
    if (oracle_w8a8_token(d, t, hidden, positions, W_qa, s_qa, gamma_q, W_qb, s_qb, W_kva, s_kva,
                          gamma_kv, W_kvb, s_kvb, cosb, sinb, qn, qp, kn, vv, kp, NULL, NULL,
                          NULL, NULL)) {
      bad += 1;
    } else {
      for (int64_t hh = 0; hh < H; ++hh) {
        int64_t o = (bi * H + hh) * s + si;
        for (int64_t e = 0; e < dn; ++e) q_nope[o * dn + e] = qn[hh * dn + e];
        for (int64_t e = 0; e < dr; ++e) q_pe[o * dr + e] = qp[hh * dr + e];
        for (int64_t e = 0; e < dn; ++e) k_nope[o * dn + e] = kn[hh * dn + e];
        for (int64_t e = 0; e < dv; ++e) value[o * dv + e] = vv[hh * dv + e];
      }
      for (int64_t e = 0; e < dr; ++e) k_pe[(bi * s + si) * dr + e] = kp[e];
    }
    free(qn); free(qp); free(kn); free(vv);
  }
  return bad;
}

/* Debug view of one W8A8 token: the int8 operands and scales the oracle
 * feeds to q_b_proj and kv_b_proj.                                         */
int oracle_w8a8_token_operands(const oracle_w8a8_dims* d, int64_t t, const uint16_t* hidden,
                               const int32_t* positions, const int8_t* W_qa, const float* s_qa,
                               const uint16_t* gamma_q, const int8_t* W_kva, const float* s_kva,
                               const uint16_t* gamma_kv, const float* cosb, const float* sinb,
                               int8_t* q1, float* s1, int8_t* c1, float* s2) {
  /* run the token with tiny dummy q_b / kv_b (heads = 0 makes them empty) */
  oracle_w8a8_dims d0 = *d;
  d0.heads = 0;
  double kp[256];
  return oracle_w8a8_token(&d0, t, hidden, positions, W_qa, s_qa, gamma_q, NULL, NULL, W_kva,
                           s_kva, gamma_kv, NULL, NULL, cosb, sinb, NULL, NULL, NULL, NULL, kp, q1,
                           s1, c1, s2);
}

int oracle_openmp_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Round n doubles to fp16 (dtype 0) or bf16 (dtype 1), nearest-even, and
 * return the rounded values as doubles (used to compare against outputs
 * stored in those formats).                                                */
void oracle_round_array(const double* x, int64_t n, int dtype, double* out) {
  for (int64_t i = 0; i < n; ++i) {
    if (isnan(x[i])) {
      out[i] = x[i];
    } else if (dtype == 0) {
      out[i] = oracle_f16_to_double(oracle_double_to_f16(x[i]));
    } else {
      out[i] = oracle_bf16_to_double(oracle_double_to_bf16(x[i]));
    }
  }
}
