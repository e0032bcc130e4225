/*
 * CPU oracle for the fused MoE finalize + rank sum + residual + RMSNorm (+ FP8 / NVFP4 quant).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the benchmark's CPU
 * baseline load this file.  The CUDA library never links it, includes it or calls it.  It shares
 * no code, header, table or constant with the CUDA sources.
 *
 * It is written to be slow and obviously correct: one token at a time, one hidden index at a time,
 * every floating-point operation spelled out in the order the definition gives.  Build with
 * -O1 -ffp-contract=off and no fast-math, so that no multiply-add is fused unless `fmaf` is
 * written.  Floats are evaluated in float (FLT_EVAL_METHOD 0 on x86-64 and AArch64).
 *
 * Sources (web pages, cited by title and section):
 *  [P1] flashinfer PR #6631 "perf(comm): gather MoE-finalize routes together and accumulate in FP32"
 *       - Description: the routed sum, the routed_scaling_factor, the shared-expert add and the sum
 *         over ranks stay in FP32; each rank's finalized row is rounded once; the rank sum is rounded
 *         once before the residual add and RMSNorm, which work on the rounded sum.
 *       - Test changes / commit message: routes set to -1 contribute nothing; one bound check per
 *         route; zero-initialised FP32 accumulator; the factor is 1.0 when scaling is off.
 *       - Benchmark script (fi_finalize_bench.py) FP64 reference: gather x weights, sum over k,
 *         times the factor, plus shared; sum over ranks; plus residual; RMSNorm in FP64 times weight.
 *       - "mean abs error vs FP64" table: pins which values are rounded (see tests).
 *  [P2] TensorRT-LLM PR #16778 "MoE: fp32 accumulation in deferred MoEAllReduce finalize" - Fix:
 *       top-k sum and shared add in an FP32 array, rounded to the activation type once.
 *  [P4] flashinfer PR #3385 "feat: MNNVL Allreduce quant fusion and performance optimization"
 *       - ranks accumulated in the fixed order 0..world_size-1 (rank-indexed slots);
 *       - FP8 / NVFP4 quantised outputs; scale-factor layouts LINEAR and SWIZZLED_128x4.
 *
 * Readings where the pages leave a step open (each also listed in the design notes):
 *  - the k loop is a chain of fused multiply-adds fmaf(scale_k, row_k, acc), k = 0..K-1, from +0;
 *  - the factor multiplies the routed sum, then the shared row is added (two rounded operations);
 *  - a route is valid iff 0 <= idx < rows; an absent scale array means every scale is 1.0;
 *  - RMSNorm: ms = (sequential FP32 sum of x*x) / H, rstd = 1 / sqrt(ms + eps) (two correctly
 *    rounded operations), y = round((x * rstd) * gamma);
 *  - quantisation reads the rounded norm_out values; FP8 q = e4m3(v * s) with s an encode scale;
 *    NVFP4 per 16-element block: sf = e4m3((amax / 6) * g), es = g / float(sf) (0 if sf is 0),
 *    code = e2m1(v * es), even element in the low nibble;
 *  - the SWIZZLED_128x4 byte offset follows the public cuBLAS description of its 1-D block-scaling
 *    factor layout (128-row x 4-column tiles of 512 bytes, row r of a tile at (r%32)*16+(r/32)*4).
 *
 * Number formats are implemented from their definitions (IEEE 754 binary16, bfloat16 = the top half
 * of binary32, OCP 8-bit FP E4M3, OCP MX E2M1): one routine rounds a real to the nearest value of a
 * binary format with ties to even, and the encoders look the rounded value up.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_BF16 = 0, OR_FP16 = 1, OR_FP32 = 2 };
enum { OR_QUANT_NONE = 0, OR_QUANT_FP8 = 1, OR_QUANT_NVFP4 = 2 };
enum { OR_SF_ROW_MAJOR = 0, OR_SF_SWIZZLED_128x4 = 1 };
enum { OR_MODE_FP32_ACCUM = 0, OR_MODE_STEP_ROUNDED = 1 };

/* ------------------------------------------------------------------------------------------ */
/* Number formats                                                                             */
/* ------------------------------------------------------------------------------------------ */

static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* Nearest value of a binary floating-point format to the finite real `x`, ties to even.
 * The format has `mbits` explicit mantissa bits and minimum normal exponent `emin`; below 2^emin
 * values are spaced like the lowest binade (subnormals).  No overflow handling here.
 * In the binade [2^e, 2^(e+1)) the spacing is 2^(e - mbits); x / spacing is exact in double
 * (a power-of-two scaling of a value with at most 24 significant bits), and rint() in the default
 * rounding mode rounds it to the nearest integer, ties to even. */
static double round_to_format(double x, int mbits, int emin) {
  if (x == 0.0) return x;
  double a = fabs(x);
  int e2;
  frexp(a, &e2);            /* a = f * 2^e2 with f in [0.5, 1) */
  int e = e2 - 1;           /* floor(log2(a)) */
  if (e < emin) e = emin;
  double q = ldexp(1.0, e - mbits);
  double n = rint(a / q);
  return copysign(n * q, x);
}

/* bfloat16: 8 exponent bits (bias 127), 7 mantissa bits; overflow rounds to infinity. */
uint16_t oracle_f32_to_bf16(float x) {
  if (isnan(x)) return (uint16_t)(((bits_from_f32(x) >> 16) & 0x8000u) | 0x7fc0u);
  if (isinf(x)) return (uint16_t)(x < 0 ? 0xff80u : 0x7f80u);
  double r = round_to_format((double)x, 7, -126);
  const double maxf = ldexp(255.0, 120);  /* (2 - 2^-7) * 2^127 */
  if (fabs(r) > maxf) return (uint16_t)(r < 0 ? 0xff80u : 0x7f80u);
  float rf = (float)r;                    /* exact: r has 8 significant bits */
  return (uint16_t)(bits_from_f32(rf) >> 16);
}

float oracle_bf16_to_f32(uint16_t b) { return f32_from_bits((uint32_t)b << 16); }

/* binary16: 5 exponent bits (bias 15), 10 mantissa bits, max 65504; overflow rounds to infinity. */
uint16_t oracle_f32_to_fp16(float x) {
  uint16_t sign = (bits_from_f32(x) >> 16) & 0x8000u;
  if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
  if (isinf(x)) return (uint16_t)(sign | 0x7c00u);
  double r = fabs(round_to_format((double)x, 10, -14));
  if (r > 65504.0) return (uint16_t)(sign | 0x7c00u);
  if (r == 0.0) return sign;
  int e2;
  frexp(r, &e2);
  int e = e2 - 1;
  if (e < -14) {                           /* subnormal: r = m * 2^-24 */
    uint32_t m = (uint32_t)ldexp(r, 24);
    return (uint16_t)(sign | m);
  }
  uint32_t m = (uint32_t)(ldexp(r, 10 - e) - 1024.0);
  return (uint16_t)(sign | ((uint32_t)(e + 15) << 10) | m);
}

float oracle_fp16_to_f32(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 31) v = m ? NAN : INFINITY;
  else if (e == 0) v = ldexp((double)m, -24);
  else v = ldexp((double)(1024 + m), e - 25);
  return (float)(s ? -v : v);
}

/* OCP FP8 E4M3: 4 exponent bits (bias 7), 3 mantissa bits, no infinities, S.1111.111 is NaN,
 * largest finite 448. */
float oracle_e4m3_to_f32(uint8_t c) {
  int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp((double)(8 + m), e - 10);
  return (float)(s ? -v : v);
}

/* Round to E4M3, ties to even, saturating to +-448 ("satfinite"); NaN -> 0x7f. */
uint8_t oracle_f32_to_e4m3(float x) {
  if (isnan(x)) return 0x7f;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = isinf(x) ? 448.0 : fabs(round_to_format((double)x, 3, -6));
  if (a > 448.0) a = 448.0;
  for (uint8_t c = 0; c < 0x7f; ++c)       /* codes 0x00..0x7e are the non-negative finite values */
    if ((double)oracle_e4m3_to_f32(c) == a) return (uint8_t)(sign | c);
  abort();                                 /* unreachable: every rounded value has a code */
}

/* OCP MX FP4 E2M1: 2 exponent bits (bias 1), 1 mantissa bit; values 0, .5, 1, 1.5, 2, 3, 4, 6. */
float oracle_e2m1_to_f32(uint8_t c) {
  int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return (float)(s ? -v : v);
}

/* Round to E2M1, ties to even, saturating to +-6; the sign of zero is kept. */
uint8_t oracle_f32_to_e2m1(float x) {
  uint8_t sign = signbit(x) ? 0x8 : 0x0;
  double a = isinf(x) ? 6.0 : fabs(round_to_format((double)x, 1, 0));
  if (a > 6.0) a = 6.0;
  for (uint8_t c = 0; c < 8; ++c)
    if ((double)oracle_e2m1_to_f32(c) == a) return (uint8_t)(sign | c);
  abort();
}

static float act_load(const void* p, int64_t i, int dt) {
  switch (dt) {
    case OR_BF16: return oracle_bf16_to_f32(((const uint16_t*)p)[i]);
    case OR_FP16: return oracle_fp16_to_f32(((const uint16_t*)p)[i]);
    default: return ((const float*)p)[i];
  }
}

static uint16_t act_round_bits(float x, int dt) {
  return dt == OR_BF16 ? oracle_f32_to_bf16(x) : oracle_f32_to_fp16(x);
}

static float act_round(float x, int dt) {
  uint16_t b = act_round_bits(x, dt);
  return dt == OR_BF16 ? oracle_bf16_to_f32(b) : oracle_fp16_to_f32(b);
}

/* ------------------------------------------------------------------------------------------ */
/* Scale-factor layouts                                                                       */
/* ------------------------------------------------------------------------------------------ */

/* Bytes of the NVFP4 block-scale buffer for T rows of H elements (one byte per 16 elements).
 * Row-major: T * H/16.  SWIZZLED_128x4: rows padded to 128 and the H/16 columns padded to 4. */
int64_t oracle_sf_bytes(int64_t T, int64_t H, int layout) {
  int64_t cols = H / 16;
  if (layout == OR_SF_ROW_MAJOR) return T * cols;
  int64_t row_tiles = (T + 127) / 128, col_tiles = (cols + 3) / 4;
  return row_tiles * 128 * col_tiles * 4;
}

/* Byte offset of the scale of row m, 16-element block k. */
int64_t oracle_sf_offset(int64_t m, int64_t k, int64_t H, int layout) {
  int64_t cols = H / 16;
  if (layout == OR_SF_ROW_MAJOR) return m * cols + k;
  int64_t col_tiles = (cols + 3) / 4;
  int64_t tile = (m / 128) * col_tiles + (k / 4);   /* 128 x 4 tiles, column tiles innermost */
  int64_t r = m % 128;
  return tile * 512 + (r % 32) * 16 + (r / 32) * 4 + (k % 4);
}

/* ------------------------------------------------------------------------------------------ */
/* The fused finalize                                                                         */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
  const void* gemm2;     /* [rows, H] act: permuted GEMM2 output of this partial               */
  int64_t rows;
  const int32_t* perm;   /* [T, K]: expanded route -> permuted row; outside [0, rows) = skip    */
  const void* scale;     /* [T, K] scale dtype, or NULL (every scale 1.0)                      */
  const void* shared;    /* [T, H] act, or NULL (no shared expert)                             */
} oracle_partial;

typedef struct {
  int32_t T, H, K, R;
  int32_t act_dtype, scale_dtype;
  float rsf, eps;
  const oracle_partial* partials;
  const void* residual;  /* [T, H] act */
  const void* gamma;     /* [H] act    */
  int32_t t0, t1;        /* compute tokens t0 <= t < t1 (outputs indexed by absolute t) */
  int32_t mode;          /* OR_MODE_FP32_ACCUM (the method) or OR_MODE_STEP_ROUNDED (old kernel) */
  /* outputs (NULL = not wanted) */
  uint16_t* residual_out;  /* [T, H] act bits */
  uint16_t* norm_out;      /* [T, H] act bits */
  uint16_t* routed_out;    /* [T, H] act bits: the rounded rank sum S, before the residual add */
} oracle_args;

/* Quantise rows t0..t1-1 of an act-typed [T, H] tensor (the rounded norm_out).  [P4] */
void oracle_quantize(const uint16_t* v_bits, int32_t act_dtype, int32_t T, int32_t H,
                     int32_t t0, int32_t t1, int32_t quant, float qscale, int32_t sf_layout,
                     uint8_t* quant_out, uint8_t* sf_out) {
  (void)T;
  for (int32_t t = t0; t < t1; ++t) {
    const uint16_t* row = v_bits + (int64_t)t * H;
    if (quant == OR_QUANT_FP8) {
      for (int32_t h = 0; h < H; ++h) {
        float v = act_load(row, h, act_dtype);
        float p = v * qscale;
        quant_out[(int64_t)t * H + h] = oracle_f32_to_e4m3(p);
      }
    } else if (quant == OR_QUANT_NVFP4) {
      for (int32_t b = 0; b < H / 16; ++b) {
        float v[16];
        float amax = 0.0f;
        for (int i = 0; i < 16; ++i) {
          v[i] = act_load(row, (int64_t)b * 16 + i, act_dtype);
          float a = fabsf(v[i]);
          if (a > amax) amax = a;
        }
        float sf_in = (amax / 6.0f) * qscale;
        uint8_t sf = oracle_f32_to_e4m3(sf_in);
        float sf_val = oracle_e4m3_to_f32(sf);
        float es = (sf_val == 0.0f) ? 0.0f : qscale / sf_val;
        uint8_t* q = quant_out + (int64_t)t * (H / 2) + b * 8;
        for (int j = 0; j < 8; ++j) {
          uint8_t lo = oracle_f32_to_e2m1(v[2 * j] * es);
          uint8_t hi = oracle_f32_to_e2m1(v[2 * j + 1] * es);
          q[j] = (uint8_t)(lo | (hi << 4));
        }
        sf_out[oracle_sf_offset(t, b, H, sf_layout)] = sf;
      }
    }
  }
}

/* The definition, token by token.  [P1] Description and Test changes; [P2] Fix; [P4] rank order. */
void oracle_finalize(const oracle_args* a) {
  const int32_t H = a->H, K = a->K, R = a->R, dt = a->act_dtype;
  float* x = (float*)malloc(sizeof(float) * (size_t)H);
  for (int32_t t = a->t0; t < a->t1; ++t) {
    for (int32_t h = 0; h < H; ++h) {
      float s = 0.0f;
      for (int32_t r = 0; r < R; ++r) {
        const oracle_partial* P = &a->partials[r];
        float acc = 0.0f;
        for (int32_t k = 0; k < K; ++k) {
          int32_t idx = P->perm[(int64_t)t * K + k];
          if (idx < 0 || (int64_t)idx >= P->rows) continue;            /* masked route */
          float sc = P->scale ? act_load(P->scale, (int64_t)t * K + k, a->scale_dtype) : 1.0f;
          float row = act_load(P->gemm2, (int64_t)idx * H + h, dt);
          if (a->mode == OR_MODE_FP32_ACCUM) {
            acc = fmaf(sc, row, acc);
          } else {                     /* old kernel: every product and sum rounded to act */
            float prod = act_round(act_round(sc, dt) * row, dt);
            acc = act_round(acc + prod, dt);
          }
        }
        if (a->mode == OR_MODE_FP32_ACCUM) {
          acc = acc * a->rsf;
          if (P->shared) acc = acc + act_load(P->shared, (int64_t)t * H + h, dt);
          s = s + act_round(acc, dt);                                   /* p_r rounded once  */
        } else {
          acc = act_round(acc * act_round(a->rsf, dt), dt);
          if (P->shared) acc = act_round(acc + act_load(P->shared, (int64_t)t * H + h, dt), dt);
          s = act_round(s + acc, dt);
        }
      }
      float S = act_round(s, dt);                                        /* rank sum rounded once */
      if (a->routed_out) a->routed_out[(int64_t)t * H + h] = act_round_bits(S, dt);
      float res = act_load(a->residual, (int64_t)t * H + h, dt);
      uint16_t ro = act_round_bits(S + res, dt);
      if (a->residual_out) a->residual_out[(int64_t)t * H + h] = ro;
      x[h] = (dt == OR_BF16) ? oracle_bf16_to_f32(ro) : oracle_fp16_to_f32(ro);
    }
    float ss = 0.0f;
    for (int32_t h = 0; h < H; ++h) ss = ss + x[h] * x[h];
    float ms = ss / (float)H;
    float rstd = 1.0f / sqrtf(ms + a->eps);
    if (a->norm_out)
      for (int32_t h = 0; h < H; ++h) {
        float g = act_load(a->gamma, h, dt);
        a->norm_out[(int64_t)t * H + h] = act_round_bits((x[h] * rstd) * g, dt);
      }
  }
  free(x);
}

/* The same formula with no intermediate rounding, in double: the FP64 reference of the benchmark
 * script in [P1].  Masked routes are skipped.  Outputs [T, H] doubles for rows t0..t1-1. */
void oracle_finalize_fp64(const oracle_args* a, double* residual_ref, double* norm_ref) {
  const int32_t H = a->H, K = a->K, R = a->R, dt = a->act_dtype;
  for (int32_t t = a->t0; t < a->t1; ++t) {
    double ss = 0.0;
    double* res = residual_ref + (int64_t)t * H;
    for (int32_t h = 0; h < H; ++h) {
      double sum = 0.0;
      for (int32_t r = 0; r < R; ++r) {
        const oracle_partial* P = &a->partials[r];
        double part = 0.0;
        for (int32_t k = 0; k < K; ++k) {
          int32_t idx = P->perm[(int64_t)t * K + k];
          if (idx < 0 || (int64_t)idx >= P->rows) continue;
          double sc = P->scale ? (double)act_load(P->scale, (int64_t)t * K + k, a->scale_dtype) : 1.0;
          part += sc * (double)act_load(P->gemm2, (int64_t)idx * H + h, dt);
        }
        part *= (double)a->rsf;
        if (P->shared) part += (double)act_load(P->shared, (int64_t)t * H + h, dt);
        sum += part;
      }
      res[h] = sum + (double)act_load(a->residual, (int64_t)t * H + h, dt);
      ss += res[h] * res[h];
    }
    double rstd = 1.0 / sqrt(ss / (double)H + (double)a->eps);
    for (int32_t h = 0; h < H; ++h)
      norm_ref[(int64_t)t * H + h] = res[h] * rstd * (double)act_load(a->gamma, h, dt);
  }
}

/* ------------------------------------------------------------------------------------------ */
/* Array forms of the format conversions (for the tests' sweeps)                              */
/* ------------------------------------------------------------------------------------------ */

void oracle_f32_to_bf16_array(const float* x, uint16_t* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_f32_to_bf16(x[i]);
}
void oracle_f32_to_fp16_array(const float* x, uint16_t* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_f32_to_fp16(x[i]);
}
void oracle_f32_to_e4m3_array(const float* x, uint8_t* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_f32_to_e4m3(x[i]);
}
void oracle_f32_to_e2m1_array(const float* x, uint8_t* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_f32_to_e2m1(x[i]);
}
float oracle_fmaf(float a, float b, float c) { return fmaf(a, b, c); }

/* Offsets of every (row, block) scale of a T x H tensor, row-major order of (m, k). */
void oracle_sf_offsets(int64_t T, int64_t H, int layout, int64_t* out) {
  for (int64_t m = 0; m < T; ++m)
    for (int64_t k = 0; k < H / 16; ++k) out[m * (H / 16) + k] = oracle_sf_offset(m, k, H, layout);
}
