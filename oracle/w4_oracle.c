/*
 * w4_oracle.c — plain CPU oracle for the 4-bit-weight mixed-precision GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load this library.  The
 * product path (libw4) never links, loads or calls it, and shares no code,
 * header, table or constant with it.
 *
 * What it computes (citations are to the source pages, by title and
 * section):
 *
 *  - Machete Readme ("Machete (Mixed Precision Cutlass-Based GEMM)"),
 *    section "Overview": the product is dequant(W) applied to a, with
 *    dequant(W) = w_q * w_s - w_z, the zero-point w_z subtracted AFTER the
 *    scale so that it is one fused multiply-add; w_z is therefore the
 *    pre-scaled zero-point.  The Readme writes the weight on the left of
 *    "@ a"; this oracle returns the conventional [M,N] = a[M,K] x W[K,N]
 *    orientation (the transposed statement of the same product).
 *  - vLLM API page "rdna_hybrid_w4a16", function pack_int4_exllama_shuffle
 *    and the docstring of _triton_w4a16_skinny_fmt_kernel: the ExLlama
 *    shuffle packing of eight K-values into one int32 in the order
 *    [0,2,4,6,1,3,5,7] (value j sits at shift (j/2)*4 + (j%2)*16), the
 *    symmetric bias of 8 (ZP_BIAS), and group scales along K.
 *  - pytorch/ao PR #1113 "support W4A8 Marlin kernel": W4A8 (int4 weights,
 *    int8 activations) with per-channel or per-group (group 128) weight
 *    scales, symmetric weights only, int32 accumulation, fp16 output, and
 *    per-token activation scales (vLLM PR #6547 "Enable Dynamic Per Token
 *    fp8" gives the per-token rationale).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - the two sequential layouts KN_SEQ [K/8][N] and NK_SEQ [N][K/8] put
 *    K-value j of a word at bits 4j;
 *  - int4 nibbles are two's complement (value q - 16 when q >= 8);
 *  - W4A8 per-group: an int8 group scale sg[g][n] multiplies the int4 value
 *    to give the int8 weight v*sg that enters the integer product;
 *  - W4A8 epilogue: out = acc * s_tok[m] * s_ch[n] (exact here, in fp64).
 *  - dynamic per-token activation quantization: s = amax/127 and
 *    q = round-half-even(a/s), in fp32 (or_quant_per_token).
 *  - fp8 activations are OCP E4M3 (bias 7, largest value 448, no
 *    infinity), encoded to nearest-even and saturated at 448, with
 *    per-token scales amax/448; W4A8-fp8 is per-channel.
 *
 * Arithmetic: floating-point results in fp64 with k ascending; integer
 * results in int64; the per-token quantizer in fp32, the precision its codes
 * are decided in.  Every function is pinned by tests under tests/ against
 * values the pages print, closed forms, invariants and library routines.
 */
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <math.h>

#define OR_KN_SEQ 0
#define OR_NK_SEQ 1
#define OR_NK_EXLLAMA 2

#define OR_UINT4B8 0
#define OR_UINT4 1
#define OR_INT4 2

/* Position of K-value j (0..7) inside its 32-bit word.
 * Sequential layouts: bits 4j (reading, not on the pages).
 * ExLlama: value j at (j/2)*4 + (j%2)*16, i.e. the word holds
 * v0 | v2<<4 | v4<<8 | v6<<12 | v1<<16 | v3<<20 | v5<<24 | v7<<28
 * ("rdna_hybrid_w4a16", pack_int4_exllama_shuffle). */
static int or_shift(int layout, int j) {
  if (layout == OR_NK_EXLLAMA) return (j / 2) * 4 + (j % 2) * 16;
  return 4 * j;
}

/* Index of the int32 word holding W[k][n] in the given input layout. */
static int64_t or_word_index(int layout, int64_t K, int64_t N, int64_t k, int64_t n) {
  if (layout == OR_KN_SEQ) return (k / 8) * N + n;
  return n * (K / 8) + k / 8; /* NK_SEQ and NK_EXLLAMA: [N][K/8] */
}

/* Stored nibble q (0..15) of W[k][n]. */
int or_nibble(const int32_t* w, int layout, int64_t K, int64_t N, int64_t k, int64_t n) {
  uint32_t word = (uint32_t)w[or_word_index(layout, K, N, k, n)];
  return (int)((word >> or_shift(layout, (int)(k % 8))) & 0xFu);
}

/* Unpack every nibble: q[k*N + n] in 0..15. */
void or_unpack(const int32_t* w, int layout, int64_t K, int64_t N, uint8_t* q) {
  for (int64_t k = 0; k < K; ++k)
    for (int64_t n = 0; n < N; ++n)
      q[k * N + n] = (uint8_t)or_nibble(w, layout, K, N, k, n);
}

/* Pack logical nibbles q[k*N + n] (0..15) into the given layout. */
void or_pack(const uint8_t* q, int layout, int64_t K, int64_t N, int32_t* w) {
  int64_t words = (K / 8) * N;
  for (int64_t i = 0; i < words; ++i) w[i] = 0;
  for (int64_t k = 0; k < K; ++k)
    for (int64_t n = 0; n < N; ++n) {
      int64_t wi = or_word_index(layout, K, N, k, n);
      uint32_t v = (uint32_t)(q[k * N + n] & 0xF) << or_shift(layout, (int)(k % 8));
      w[wi] = (int32_t)((uint32_t)w[wi] | v);
    }
}

/* Integer value of a stored nibble for a weight type:
 * uint4b8 -> q - 8 (symmetric bias 8, "rdna_hybrid_w4a16" ZP_BIAS);
 * uint4   -> q (asymmetric, used with zero-points);
 * int4    -> two's complement nibble, q - 16 when q >= 8. */
int or_value(int q, int wtype) {
  if (wtype == OR_UINT4B8) return q - 8;
  if (wtype == OR_UINT4) return q;
  return q >= 8 ? q - 16 : q;
}

/* Dequantized weight, Machete Readme "Overview": w_hat = w_q * w_s - w_z,
 * with w_q the integer value of the nibble, w_s the group scale and w_z the
 * pre-scaled zero-point of group g = k / group_size, column n.  fp64: exact
 * for 4-bit values times 16-bit scales. */
static double or_what(const int32_t* w, int layout, int wtype, int64_t K, int64_t N,
                      const double* s, const double* z, int64_t group_size,
                      int64_t k, int64_t n) {
  int64_t g = k / group_size;
  double v = (double)or_value(or_nibble(w, layout, K, N, k, n), wtype);
  double zz = z ? z[g * N + n] : 0.0;
  return v * s[g * N + n] - zz;
}

/* One output element of W4A16: ref = sum_k a[m][k] * w_hat[k][n], k
 * ascending, fp64; absref = sum_k |a[m][k] * w_hat[k][n]| (for the error
 * bound). */
static void or_w4a16_one(int64_t N, int64_t K, const double* a, const int32_t* w,
                         int layout, int wtype, const double* s, const double* z,
                         int64_t group_size, int64_t m, int64_t n, double* ref,
                         double* absref) {
  double acc = 0.0, aacc = 0.0;
  for (int64_t k = 0; k < K; ++k) {
    double t = a[m * K + k] * or_what(w, layout, wtype, K, N, s, z, group_size, k, n);
    acc += t;
    aacc += fabs(t);
  }
  *ref = acc;
  *absref = aacc;
}

/* Full W4A16 product: a [M][K] (fp64 copies of the fp16/bf16 activations),
 * packed weights w in `layout`, scales s [G][N], optional pre-scaled zeros
 * z [G][N] (NULL = no zero-points), group_size dividing K.
 * Writes ref [M][N] and absref [M][N]. */
void or_w4a16(int64_t M, int64_t N, int64_t K, const double* a, const int32_t* w,
              int layout, int wtype, const double* s, const double* z,
              int64_t group_size, double* ref, double* absref) {
  int64_t total = M * N;
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t i = 0; i < total; ++i)
    or_w4a16_one(N, K, a, w, layout, wtype, s, z, group_size, i / N, i % N, &ref[i],
                 &absref[i]);
}

/* W4A16 on a list of sampled output positions (rows[i], cols[i]). */
void or_w4a16_elems(int64_t M, int64_t N, int64_t K, const double* a, const int32_t* w,
                    int layout, int wtype, const double* s, const double* z,
                    int64_t group_size, int64_t count, const int64_t* rows,
                    const int64_t* cols, double* ref, double* absref) {
  (void)M;
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t i = 0; i < count; ++i)
    or_w4a16_one(N, K, a, w, layout, wtype, s, z, group_size, rows[i], cols[i], &ref[i],
                 &absref[i]);
}

/* Integer weight of W4A8, pytorch/ao PR #1113: the int4 value itself
 * (per-channel), or the int4 value times its int8 group scale sg[g][n]
 * (per-group), so the product with int8 activations is an integer. */
static int64_t or_wint(const int32_t* w, int layout, int wtype, int64_t K, int64_t N,
                       const int8_t* sg, int64_t group_size, int64_t k, int64_t n) {
  int64_t v = or_value(or_nibble(w, layout, K, N, k, n), wtype);
  if (sg) v *= (int64_t)sg[(k / group_size) * N + n];
  return v;
}

static int64_t or_w4a8_one(int64_t N, int64_t K, const int8_t* a, const int32_t* w,
                           int layout, int wtype, const int8_t* sg, int64_t group_size,
                           int64_t m, int64_t n) {
  int64_t acc = 0;
  for (int64_t k = 0; k < K; ++k)
    acc += (int64_t)a[m * K + k] * or_wint(w, layout, wtype, K, N, sg, group_size, k, n);
  return acc;
}

/* Full W4A8 integer accumulator acc [M][N] (int64, exact). sg may be NULL
 * (per-channel). */
void or_w4a8(int64_t M, int64_t N, int64_t K, const int8_t* a, const int32_t* w,
             int layout, int wtype, const int8_t* sg, int64_t group_size, int64_t* acc) {
  int64_t total = M * N;
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t i = 0; i < total; ++i)
    acc[i] = or_w4a8_one(N, K, a, w, layout, wtype, sg, group_size, i / N, i % N);
}

void or_w4a8_elems(int64_t M, int64_t N, int64_t K, const int8_t* a, const int32_t* w,
                   int layout, int wtype, const int8_t* sg, int64_t group_size,
                   int64_t count, const int64_t* rows, const int64_t* cols, int64_t* acc) {
  (void)M;
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t i = 0; i < count; ++i)
    acc[i] = or_w4a8_one(N, K, a, w, layout, wtype, sg, group_size, rows[i], cols[i]);
}

/* W4A8 output before its final rounding: acc * s_tok[m] * s_ch[n] in fp64
 * (per-token activation scale times per-channel weight scale). */
void or_w4a8_scale(int64_t count, const int64_t* acc, const int64_t* rows,
                   const int64_t* cols, const double* s_tok, const double* s_ch,
                   double* ref) {
  for (int64_t i = 0; i < count; ++i)
    ref[i] = (double)acc[i] * s_tok[rows[i]] * s_ch[cols[i]];
}

/* Dynamic per-token int8 quantization of the activations that feed W4A8.
 * vLLM PR #6547 "Enable Dynamic Per Token fp8" (summary): one activation
 * scale per token, computed at run time from that token's own values;
 * pytorch/ao PR #1113 "support W4A8 Marlin kernel": the W4A8 activations
 * are symmetric int8.  The pages print no formula; the reading taken is the
 * plain symmetric one, every step in fp32 (the precision the quantized code
 * is decided in):
 *   amax      = max_k |a[m][k]|            (exact: inputs are fp16/bf16)
 *   s_tok[m]  = amax / 127                 (one correctly rounded division)
 *   q[m][k]   = nearest integer to a[m][k] / s_tok[m] (the quotient rounded
 *               once to fp32, then to an integer, ties to even), within
 *               [-127, 127]
 * A row with amax == 0 gets s_tok = 0 and codes 0.  a is fp32 [M][K]
 * (exact copies of the fp16/bf16 inputs), q int8 [M][K], s_tok fp32 [M]. */
void or_quant_per_token(int64_t M, int64_t K, const float* a, int8_t* q, float* s_tok) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    const float* row = a + m * K;
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      const float v = fabsf(row[k]);
      if (v > amax) amax = v;
    }
    const float s = amax / 127.0f;
    s_tok[m] = s;
    for (int64_t k = 0; k < K; ++k) {
      if (amax == 0.0f) {
        q[m * K + k] = 0;
        continue;
      }
      const float x = row[k] / s;
      float r = rintf(x); /* default rounding mode: to nearest, ties to even */
      if (r > 127.0f) r = 127.0f;
      if (r < -127.0f) r = -127.0f;
      q[m * K + k] = (int8_t)r;
    }
  }
}

/* ---- fp8 activations (vLLM PR #9855 "[Kernel] Initial Machete W4A8
 * support + Refactors": QQQ-style W4A8 "including fp8 activations", with an
 * int4 -> fp8 weight converter).  The pages do not define the fp8 format;
 * the reading taken is the E4M3 format of the OCP 8-bit floating point
 * specification: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent field 0 holds the subnormals m/8 * 2^-6; the all-ones pattern
 * S.1111.111 is NaN and there is no infinity, so the largest value is
 * 1.75 * 2^8 = 448.  Every int4 weight value -8..7 is exact in it. */

/* Value of an E4M3 code (NaN for S.1111.111). */
double or_e4m3_decode(int code) {
  const int sign = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m / 8.0, -6);
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* E4M3 code of a finite fp32 value: the nearest representable value, ties
 * to the even mantissa, magnitudes at or above 448 saturated to 448 (the
 * "satfinite" reading: rounding first, then clamping to the largest finite
 * value, which gives 448 for every magnitude >= 448). */
int or_e4m3_encode(float x) {
  const int sign = signbit(x) ? 0x80 : 0;
  const float a = fabsf(x);
  if (a >= 448.0f) return sign | 0x7E;
  if (a < 0x1p-6f) {                       /* subnormal range: steps of 2^-9 */
    const int q = (int)rintf(a * 512.0f);  /* exact scaling; 8 becomes 0x08 */
    return sign | q;
  }
  int e;
  const float f = frexpf(a, &e);           /* a = f * 2^e, f in [0.5, 1) */
  e -= 1;                                  /* a = (2f) * 2^e, 2f in [1, 2) */
  int m = (int)rintf((2.0f * f - 1.0f) * 8.0f); /* exact before the rounding */
  if (m == 8) {
    m = 0;
    e += 1;
  }
  return sign | ((e + 7) << 3) | m;
}

void or_e4m3_decode_n(int64_t n, const uint8_t* codes, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = or_e4m3_decode(codes[i]);
}
void or_e4m3_encode_n(int64_t n, const float* x, uint8_t* codes) {
  for (int64_t i = 0; i < n; ++i) codes[i] = (uint8_t)or_e4m3_encode(x[i]);
}

/* Dynamic per-token fp8 quantization (vLLM PR #6547 "Enable Dynamic Per
 * Token fp8": one scale per token from that token's values).  Reading, in
 * fp32 as for the int8 codes: s_tok = amax / 448, and each code is the E4M3
 * encoding of the quotient a / s_tok rounded once to fp32.  A zero row gets
 * s_tok = 0 and codes 0. */
void or_quant_per_token_fp8(int64_t M, int64_t K, const float* a, uint8_t* q, float* s_tok) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    const float* row = a + m * K;
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      const float v = fabsf(row[k]);
      if (v > amax) amax = v;
    }
    const float s = amax / 448.0f;
    s_tok[m] = s;
    for (int64_t k = 0; k < K; ++k)
      q[m * K + k] = amax == 0.0f ? 0 : (uint8_t)or_e4m3_encode(row[k] / s);
  }
}

/* W4A8 with fp8 activations, per-channel: ref[m][n] = sum_k
 * decode(a[m][k]) * v(q[k][n]) in fp64 with k ascending (every product and
 * partial sum is a multiple of 2^-9 below 2^44, so the sum is exact), and
 * absref the sum of |terms|.  The output is ref * s_tok[m] * s_ch[n]. */
void or_w4a8_fp8(int64_t M, int64_t N, int64_t K, const uint8_t* a, const int32_t* w, int layout,
                 int wtype, double* ref, double* absref) {
  double lut[256];
  for (int c = 0; c < 256; ++c) lut[c] = or_e4m3_decode(c);
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0, aacc = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double t = lut[a[m * K + k]] * (double)or_value(or_nibble(w, layout, K, N, k, n), wtype);
        acc += t;
        aacc += fabs(t);
      }
      ref[m * N + n] = acc;
      absref[m * N + n] = aacc;
    }
}

/* Threads the oracle's parallel loops use (1 when built without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
#endif
int or_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
