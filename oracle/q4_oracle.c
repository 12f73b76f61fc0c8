/*
 * q4_oracle.c — CPU oracle for the Q4_0 block-quantized matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link
 * or call this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it.  It shares no code, header, table or constant
 * generator with the CUDA library: every conversion below is written out
 * here from its definition.
 *
 * What it computes (plain definitions, no blocking, no reordering):
 *
 *  1. quantize   — per row n and per 32-weight block b along K:
 *                  m   = the element of largest |x| (first in index order on
 *                        equal |x|);
 *                  d32 = m / -8 (fp32, exact: division by a power of two);
 *                  q_k = clamp(round(x_k / d32) + 8, 0, 15), IEEE fp32
 *                        division, round half away from zero; an all-zero
 *                        block has d32 = 0 and q_k = 8;
 *                  d16 = fp16(d32), round to nearest even.
 *                  The pages never define the 4-bit format: the continuous-
 *                  batching investigation ("Why Continuous Batching Slowed
 *                  Down My LLM Inference Engine", intro) says only "4-bit
 *                  quantized Qwen2.5 7B" on Candle's quantized Metal path
 *                  (§"Two Rows of Input, Two Different Kernels").  The block
 *                  rule above is the Q4_0 definition this library adopts.
 *  2. pack       — canonical 18-byte block: d16 little-endian, then 16 bytes
 *                  where byte j holds q_j (low nibble) and q_{j+16} (high).
 *  3. dequantize — w = (q - 8) * float(d16); exact in fp32 (a 4-bit integer
 *                  times an 11-bit significand).
 *  4. matmul     — y[m,n] = sum_k w[n,k] * x[m,k] in fp64, ascending k,
 *                  rounded once to fp32.  Every product is exact in fp64.
 *                  This is the linear layer whose GEMV/GEMM kernel choice the
 *                  investigation traces (§"Two Rows of Input…", §"Same
 *                  Prompt, Different Story"); the fast kernels must reach the
 *                  same value up to rounding order.
 *  5. bound      — B[m,n] = 1e-5 * sum_k |w[n,k] x[m,k]| + 1e-6, the
 *                  per-element tolerance the GPU result is held to.
 *  6. argmax     — greedy pick over a row of fp32 logits: the largest value,
 *                  lowest index on exact ties, NaN never wins (§"Same Prompt,
 *                  Different Story": greedy decoding selects the token with
 *                  the highest score).
 *
 * Status values (the oracle's own; numerically the same as the library's
 * documented codes so that tests can compare them):
 *   0 ok, 2 bad shape (K not a multiple of 32, N or K < 1),
 *   4 non-finite input weight, 5 scale out of fp16 range.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define Q4O_OK 0
#define Q4O_ERR_SHAPE 2
#define Q4O_ERR_NONFINITE 4
#define Q4O_ERR_RANGE 5

#define Q4O_BLOCK 32
#define Q4O_BLOCK_BYTES 18

/* ---- fp16 <-> fp32, written from the IEEE 754 binary16 definition ---- */

static uint32_t f32_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

static float bits_f32(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round-to-nearest-even conversion of an fp32 value to binary16 bits. */
uint16_t q4o_f32_to_f16(float f) {
  uint32_t x = f32_bits(f);
  uint32_t sign = (x >> 16) & 0x8000u;
  uint32_t ax = x & 0x7FFFFFFFu;
  if (ax >= 0x7F800000u) /* inf or NaN */
    return (uint16_t)(sign | 0x7C00u | (ax > 0x7F800000u ? 0x0200u : 0u));
  /* 65520 = 65504 + half an ulp: at or above it the nearest binary16 is inf */
  if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);
  if (ax >= 0x38800000u) { /* >= 2^-14: a normal binary16 */
    uint32_t exp16 = (ax >> 23) - 127u + 15u;
    uint32_t mant = ax & 0x7FFFFFu;
    uint32_t h = (exp16 << 10) | (mant >> 13);
    uint32_t rem = mant & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u; /* carry may bump exponent */
    return (uint16_t)(sign | h);
  }
  /* below 2^-14: binary16 subnormal k * 2^-24 with k = rne(|f| * 2^24) */
  if (ax < 0x00800000u) return (uint16_t)sign; /* fp32 subnormal: far below 2^-25 */
  {
    int32_t e = (int32_t)(ax >> 23) - 127;             /* |f| = sig * 2^(e-23) */
    uint32_t sig = (ax & 0x7FFFFFu) | 0x800000u;       /* 24-bit significand */
    int32_t shift = -(e + 1);                          /* |f|*2^24 = sig >> shift */
    uint32_t k, rem, half;
    if (shift > 24) return (uint16_t)sign;             /* < 2^-25: rounds to zero */
    k = sig >> shift;
    rem = sig & ((1u << shift) - 1u);
    half = 1u << (shift - 1);
    if (rem > half || (rem == half && (k & 1u))) k += 1u;
    return (uint16_t)(sign | k);
  }
}

/* Exact widening of binary16 bits to fp32. */
float q4o_f16_to_f32(uint16_t h) {
  uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
  uint32_t e = ((uint32_t)h >> 10) & 0x1Fu;
  uint32_t m = (uint32_t)h & 0x3FFu;
  if (e == 0) {
    float v = ldexpf((float)m, -24);
    return sign ? -v : v;
  }
  if (e == 31) return bits_f32(sign | 0x7F800000u | (m << 13));
  return bits_f32(sign | ((e - 15u + 127u) << 23) | (m << 13));
}

/* ---- quantize / pack / dequantize ---- */

static int shape_ok(int64_t N, int64_t K) {
  return N >= 1 && K >= Q4O_BLOCK && (K % Q4O_BLOCK) == 0;
}

/* Quantize one 32-weight block into its canonical 18 bytes. */
static int quantize_block(const float* xb, uint8_t* out) {
  int i, imax = 0;
  float amax, m, d;
  uint16_t d16;
  uint8_t q[Q4O_BLOCK];
  for (i = 0; i < Q4O_BLOCK; ++i)
    if (!isfinite(xb[i])) return Q4O_ERR_NONFINITE;
  amax = fabsf(xb[0]);
  for (i = 1; i < Q4O_BLOCK; ++i) {
    if (fabsf(xb[i]) > amax) { /* strict: the first of equal |x| wins */
      amax = fabsf(xb[i]);
      imax = i;
    }
  }
  m = xb[imax];
  d = m / -8.0f;
  d16 = q4o_f32_to_f16(d);
  if ((d16 & 0x7C00u) == 0x7C00u) return Q4O_ERR_RANGE;
  for (i = 0; i < Q4O_BLOCK; ++i) {
    int qi;
    if (d == 0.0f) {
      qi = 8;
    } else {
      float r = roundf(xb[i] / d); /* half away from zero */
      qi = (int)r + 8;
      if (qi < 0) qi = 0;
      if (qi > 15) qi = 15;
    }
    q[i] = (uint8_t)qi;
  }
  out[0] = (uint8_t)(d16 & 0xFFu);
  out[1] = (uint8_t)(d16 >> 8);
  for (i = 0; i < 16; ++i) out[2 + i] = (uint8_t)(q[i] | (q[i + 16] << 4));
  return Q4O_OK;
}

/* w: fp32 [N,K] row-major.  blocks: N*K/32 canonical 18-byte blocks, row n's
 * blocks in ascending K order, rows in ascending n. */
int q4o_quantize(const float* w, int64_t N, int64_t K, uint8_t* blocks) {
  int64_t nb, n, b;
  int status = Q4O_OK;
  if (!shape_ok(N, K)) return Q4O_ERR_SHAPE;
  nb = K / Q4O_BLOCK;
  for (n = 0; n < N; ++n) {
    for (b = 0; b < nb; ++b) {
      int s = quantize_block(w + n * K + b * Q4O_BLOCK, blocks + (n * nb + b) * Q4O_BLOCK_BYTES);
      if (s != Q4O_OK && status == Q4O_OK) status = s;
    }
  }
  return status;
}

static int block_q(const uint8_t* blk, int j) {
  return j < 16 ? (blk[2 + j] & 0x0F) : (blk[2 + j - 16] >> 4);
}

static float block_d(const uint8_t* blk) {
  return q4o_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
}

/* w: fp32 [N,K] = (q - 8) * d16 for every weight. */
int q4o_dequantize(const uint8_t* blocks, int64_t N, int64_t K, float* w) {
  int64_t nb, n, b;
  int j;
  if (!shape_ok(N, K)) return Q4O_ERR_SHAPE;
  nb = K / Q4O_BLOCK;
  for (n = 0; n < N; ++n)
    for (b = 0; b < nb; ++b) {
      const uint8_t* blk = blocks + (n * nb + b) * Q4O_BLOCK_BYTES;
      float d = block_d(blk);
      for (j = 0; j < Q4O_BLOCK; ++j)
        w[n * K + b * Q4O_BLOCK + j] = (float)(block_q(blk, j) - 8) * d;
    }
  return Q4O_OK;
}

/* ---- matmul ---- */

/* One output element: y = sum_k w[n,k] x[m,k], fp64, ascending k. */
static void dot_one(const uint8_t* blocks, int64_t nb, int64_t n, const float* xrow,
                    double* y64, double* absdot) {
  double s = 0.0, a = 0.0;
  int64_t b;
  int j;
  for (b = 0; b < nb; ++b) {
    const uint8_t* blk = blocks + (n * nb + b) * Q4O_BLOCK_BYTES;
    double d = (double)block_d(blk);
    for (j = 0; j < Q4O_BLOCK; ++j) {
      double p = (double)(block_q(blk, j) - 8) * d * (double)xrow[b * Q4O_BLOCK + j];
      s += p;
      a += fabs(p);
    }
  }
  *y64 = s;
  *absdot = a;
}

/* x: fp32 [M,K] row-major.  y: fp32 [M,N] (may be NULL).  y64: the fp64 sums
 * before rounding (may be NULL).  bound: 1e-5*sum|w x| + 1e-6 (may be NULL). */
int q4o_matmul(const uint8_t* blocks, int64_t N, int64_t K, const float* x, int64_t M,
               float* y, double* y64, double* bound) {
  int64_t nb, i;
  if (!shape_ok(N, K) || M < 0) return Q4O_ERR_SHAPE;
  nb = K / Q4O_BLOCK;
#pragma omp parallel for schedule(static)
  for (i = 0; i < M * N; ++i) {
    int64_t m = i / N, n = i % N;
    double s, a;
    dot_one(blocks, nb, n, x + m * K, &s, &a);
    if (y) y[i] = (float)s;
    if (y64) y64[i] = s;
    if (bound) bound[i] = 1e-5 * a + 1e-6;
  }
  return Q4O_OK;
}

/* The same, for P chosen (m, n) pairs: pairs[2p] = m, pairs[2p+1] = n. */
int q4o_matmul_pairs(const uint8_t* blocks, int64_t N, int64_t K, const float* x, int64_t M,
                     const int64_t* pairs, int64_t P, float* y, double* y64, double* bound) {
  int64_t nb, p;
  if (!shape_ok(N, K) || M < 0) return Q4O_ERR_SHAPE;
  for (p = 0; p < P; ++p)
    if (pairs[2 * p] < 0 || pairs[2 * p] >= M || pairs[2 * p + 1] < 0 || pairs[2 * p + 1] >= N)
      return Q4O_ERR_SHAPE;
  nb = K / Q4O_BLOCK;
#pragma omp parallel for schedule(static)
  for (p = 0; p < P; ++p) {
    double s, a;
    dot_one(blocks, nb, pairs[2 * p + 1], x + pairs[2 * p] * K, &s, &a);
    if (y) y[p] = (float)s;
    if (y64) y64[p] = s;
    if (bound) bound[p] = 1e-5 * a + 1e-6;
  }
  return Q4O_OK;
}

/* ---- argmax ---- */

/* Per row of y[M,N] (fp32): the index of the largest value, the lowest index
 * on exact ties; NaN compares below everything. */
int q4o_argmax(const float* y, int64_t M, int64_t N, int32_t* idx) {
  int64_t m, n;
  if (M < 0 || N < 1) return Q4O_ERR_SHAPE;
  for (m = 0; m < M; ++m) {
    const float* r = y + m * N;
    int64_t best = -1;
    for (n = 0; n < N; ++n) {
      if (isnan(r[n])) continue;
      if (best < 0 || r[n] > r[best]) best = n;
    }
    idx[m] = (int32_t)(best < 0 ? 0 : best);
  }
  return Q4O_OK;
}

/* Threads the oracle's loops use from now on (n >= 1); returns the previous
 * count.  Only the benchmark's single-core timing calls it. */
int q4o_set_threads(int n) {
#ifdef _OPENMP
  const int prev = omp_get_max_threads();
  if (n >= 1) omp_set_num_threads(n);
  return prev;
#else
  (void)n;
  return 1;
#endif
}

int q4o_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
