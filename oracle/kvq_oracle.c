/*
 * kvq_oracle.c -- plain, slow, single-threaded CPU oracle for attention over a
 * sub-byte quantized KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent reference that the CUDA
 * library is checked against.  It shares no code, header, table or constant
 * generator with the CUDA path, and the product never calls it.  Only the tests,
 * the smoke check and the benchmark's CPU-baseline leg load it.
 *
 * Sources followed (page titles as printed on the pages):
 *  [P1] "qwen27 CUDA: an opt-in 4-bit attention cache (262K on a 24 GB card)",
 *       section "What it is": 144-byte rows of Hadamard-rotated 32-value groups,
 *       4-bit codes plus an fp16 scale; queries rotated once, attention in the
 *       rotated space over 512-key chunks plus the tail with an in-order merge,
 *       output rotated back once; prompt chunks attend over decoded slots.
 *  [P2] "feat(kvcache): add reliable quantized KV cache", PR body and the
 *       test-fix commit: 32 values -> 16 bytes + one fp16 scale; symmetric
 *       4-bit codes; exact-scale blocks (amax 8 -> scale 1, codes equal inputs).
 *  [P3] "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant", KV8 base commit:
 *       MLA latent rows as e4m3 bytes with a per-row f32 scale amax/448, RNE
 *       encoder saturating at +-448, signed zero kept, NaN stored as 0, guard for
 *       a subnormal amax; absorbed attention where the latent is key and value;
 *       split-T commit: (H,P) partials (m, z, cl) merged by log-sum-exp; DSA
 *       gather over selected absolute rows.
 *
 * Readings taken where the pages are silent (each one also listed in the design
 * notes of the repository):
 *  R1  The rotation is the natural-order (Sylvester) 32-point Walsh-Hadamard
 *      matrix scaled by 1/sqrt(32), no random signs.  It is symmetric and its own
 *      inverse.
 *  R2  The store computes the rotation in fp32 by the butterfly with stages
 *      h = 1, 2, 4, 8, 16 in that order, (a, b) -> (a + b, a - b) with a the lower
 *      index, then multiplies every value once by the fp32 constant 1/sqrt(32).
 *  R3  scale = fp16_rne(amax / 8), saturated to 65504; codes are computed with the
 *      stored fp16 scale: code = clamp(rint_even(y / s), -8, 7) + 8; s == 0 gives
 *      code 8 everywhere.
 *  R4  Row layout: the groups' 16-byte code blocks in group order (group G at
 *      bytes 16G .. 16G + 15, the plainest reading of "32 values -> 16 bytes +
 *      one fp16 scale"); inside a block, byte b holds element 2b in its low
 *      nibble and element 2b + 1 in its high nibble.
 *  R5  A decode query at context N attends T keys; the split uses partitions
 *      [512p, 512p + 512) with the last one the tail; the merge takes partitions
 *      in ascending order.
 *  R7  TQ4 rows ([P3] "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant", PR
 *      body, "Why rotated-int4": a randomized-Hadamard rotation, then a fixed
 *      16-level Lloyd-Max codebook for N(0,1) scaled by radius/sqrt(n); the
 *      rotation keeps the radius, so one scale per row).  The pages leave the
 *      details open; read here as: n = head_dim; the random signs are a
 *      caller-given bit mask (bit i set: element i negated before the
 *      transform); y = fp32 butterfly of the signed row (stages h = 1 .. n/2 as
 *      in R2) times fp32(1/sqrt(n)); ss = fp32 sum of the fp32 squares by the
 *      pairwise tree (stage h adds element i + h into i for i a multiple of
 *      2h); scale = fp16_sat(sqrtf(ss * (1/n))), and the codes use the stored
 *      fp16 scale; the codebook is the Lloyd-Max levels rounded to fp16 (8
 *      magnitudes M_0 < .. < M_7, the levels being +-M_m); code = 8 * [v < 0] +
 *      #{k < 7 : |v| > (M_k + M_{k+1}) / 2} for v = y / scale (fp32 division;
 *      a tie goes to the smaller magnitude); scale 0 gives code 0 everywhere.
 *      Value = (code & 8 ? -1 : 1) * M_{code & 7} * scale, in the rotated space;
 *      queries are rotated by the same signed transform, outputs back by its
 *      inverse (signs after the transform).  Codes are stored as in R4.
 *  R6  fp8 rows: separate scales for the latent part and the rope part, each
 *      amax/448; codes = e4m3(x * (448/amax)) with 448/amax computed once in fp32;
 *      amax == 0 or a non-finite 448/amax stores all-zero codes.
 *  R7  In absorbed attention the value is the latent part only.
 *
 * Floating point: the store and the fp8 encoder run in fp32 because their
 * results are integers (codes) decided by fp32 arithmetic in the same precision
 * as the GPU kernels; everything else (rotation of queries, attention, merge)
 * runs in fp64.
 *
 * Parity pins: every function here is pinned by tests that do not reuse this
 * code (library conversions, closed forms, brute force, the pages' exact-scale
 * special case).  Absolute agreement with the pages' own kernels is unpinned:
 * no page prints a worked numeric example of a stored row or of an attention
 * output.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Scalar conversions, written from the IEEE / OCP format definitions.        */
/* ------------------------------------------------------------------------- */

/* Round a non-negative double to the nearest integer, ties to even. */
static double round_half_even(double q) {
  double f = floor(q);
  double d = q - f;
  if (d > 0.5) return f + 1.0;
  if (d < 0.5) return f;
  return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* fp32 -> IEEE binary16, round to nearest even; overflow gives +-inf, NaN gives
 * the canonical quiet NaN 0x7E00 (sign kept). */
uint16_t kvo_f32_to_f16(float xf) {
  double x = (double)xf;
  uint16_t sign = signbit(xf) ? 0x8000u : 0u;
  if (isnan(xf)) return (uint16_t)(sign | 0x7E00u);
  double a = fabs(x);
  if (a == 0.0) return sign;
  if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u); /* rounds past 65504 */
  if (a < ldexp(1.0, -14)) {                            /* subnormal range */
    double m = round_half_even(a * ldexp(1.0, 24));     /* units of 2^-24 */
    return (uint16_t)(sign | (uint16_t)m);              /* m == 1024 is the min normal */
  }
  int e;
  double fr = frexp(a, &e); /* a = fr * 2^e, fr in [0.5, 1) */
  int ex = e - 1;           /* a = (2 fr) * 2^ex, 2 fr in [1, 2) */
  double m = round_half_even((2.0 * fr - 1.0) * 1024.0);
  if (m == 1024.0) { m = 0.0; ex += 1; }
  if (ex > 15) return (uint16_t)(sign | 0x7C00u);
  return (uint16_t)(sign | (uint16_t)((ex + 15) << 10) | (uint16_t)m);
}

/* Same, but a finite input never becomes infinite: saturate to +-65504. */
uint16_t kvo_f32_to_f16_sat(float x) {
  uint16_t h = kvo_f32_to_f16(x);
  if ((h & 0x7FFFu) == 0x7C00u) h = (uint16_t)((h & 0x8000u) | 0x7BFFu);
  return h;
}

double kvo_f16_to_f64(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1F, m = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = (m == 0) ? INFINITY : NAN;
  else v = ldexp(1.0 + m / 1024.0, e - 15);
  return s ? -v : v;
}

/* fp32 -> bfloat16, round to nearest even (the top 16 bits of the fp32 pattern
 * after rounding the dropped 16 bits); NaN stays a quiet NaN. */
uint16_t kvo_f32_to_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  if (isnan(x)) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lower = u & 0xFFFFu, upper = u >> 16;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;
}

float kvo_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float x;
  memcpy(&x, &u, 4);
  return x;
}

/* OCP e4m3 (the "fn" variant): 1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; exponent 0 is subnormal (m * 2^-9); 0x7F and 0xFF are NaN; no infinity;
 * the largest finite value is 448 (0x7E). */
double kvo_e4m3_to_f64(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* [P3] encoder reading: round to nearest even on the exact value, saturate to
 * +-448, keep the sign of zero, store NaN as the inert code 0x00. */
uint8_t kvo_f32_to_e4m3(float xf) {
  if (isnan(xf)) return 0x00;
  uint8_t sign = signbit(xf) ? 0x80 : 0x00;
  double a = fabs((double)xf);
  if (a == 0.0) return sign;
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  uint8_t code;
  if (a < ldexp(1.0, -6)) {                         /* subnormal: steps of 2^-9 */
    double m = round_half_even(a * ldexp(1.0, 9));  /* 0..8; 8 is 2^-6 = code 0x08 */
    code = (uint8_t)m;
  } else {
    int e;
    double fr = frexp(a, &e);
    int ex = e - 1;                                  /* a = (2 fr) 2^ex */
    double m = round_half_even((2.0 * fr - 1.0) * 8.0);
    if (m == 8.0) { m = 0.0; ex += 1; }              /* carry into the next binade */
    int field = ((ex + 7) << 3) | (int)m;
    if (field > 0x7E) field = 0x7E;                  /* would be NaN or above 448 */
    code = (uint8_t)field;
  }
  return (uint8_t)(sign | code);
}

/* ------------------------------------------------------------------------- */
/* Hadamard rotation                                                          */
/* ------------------------------------------------------------------------- */

/* R2: fp32 butterfly used by the store, in place on 32 values. */
void kvo_fwht32_f32(float* x) {
  for (int h = 1; h < 32; h <<= 1) {
    for (int i = 0; i < 32; i++) {
      if (i & h) continue;
      float a = x[i], b = x[i + h];
      x[i] = a + b;
      x[i + h] = a - b;
    }
  }
  const float c = (float)(1.0 / sqrt(32.0));
  for (int i = 0; i < 32; i++) x[i] = x[i] * c;
}

/* R1: y = H x by the matrix definition, H[i][j] = (-1)^popcount(i & j) / sqrt(32),
 * in fp64.  Used for queries and outputs of attention. */
void kvo_hadamard32_f64(const double* x, double* y) {
  const double c = 1.0 / sqrt(32.0);
  for (int i = 0; i < 32; i++) {
    double acc = 0.0;
    for (int j = 0; j < 32; j++) {
      int par = __builtin_popcount((unsigned)(i & j)) & 1;
      acc += par ? -x[j] : x[j];
    }
    y[i] = acc * c;
  }
}

/* ------------------------------------------------------------------------- */
/* 4-bit rotated rows                                                         */
/* ------------------------------------------------------------------------- */

/* Quantise one row of D fp32 values (D a multiple of 32) into its stored code
 * bytes (D/2, layout R4) and NG fp16 scales, following R2 and R3; `rotate` = 0 skips the
 * rotation (the unrotated Q4_0 form of "feat(kvcache): add reliable quantized
 * KV cache", PR body: 32 values -> 16 bytes + one fp16 scale, symmetric). */
static void q4_quantize_row(const float* x, int D, uint8_t* codes_out, uint16_t* scales, int rotate) {
  int NG = D / 32;
  for (int G = 0; G < NG; G++) {
    float y[32];
    for (int i = 0; i < 32; i++) y[i] = x[32 * G + i];
    if (rotate) kvo_fwht32_f32(y);
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) {
      float a = fabsf(y[i]);
      if (a > amax) amax = a;
    }
    float s32 = amax / 8.0f;
    uint16_t s16 = kvo_f32_to_f16_sat(s32);
    scales[G] = s16;
    float s = (float)kvo_f16_to_f64(s16);
    int codes[32];
    for (int i = 0; i < 32; i++) {
      int c;
      if (s == 0.0f) {
        c = 8;
      } else {
        float r = y[i] / s;                  /* IEEE fp32 division */
        double q = (r < 0.0f) ? -round_half_even(-(double)r) : round_half_even((double)r);
        if (q < -8.0) q = -8.0;
        if (q > 7.0) q = 7.0;
        c = (int)q + 8;
      }
      codes[i] = c;
    }
    for (int b = 0; b < 16; b++)
      codes_out[16 * G + b] = (uint8_t)(codes[2 * b] | (codes[2 * b + 1] << 4));
  }
}

void kvo_q4_quantize_row(const float* x, int D, uint8_t* codes, uint16_t* scales) {
  q4_quantize_row(x, D, codes, scales, 1);
}

void kvo_q4_0_quantize_row(const float* x, int D, uint8_t* codes, uint16_t* scales) {
  q4_quantize_row(x, D, codes, scales, 0);
}

/* Tables of every fp16 and e4m3 value, filled once from the definitions above so
 * that long attention loops do not call ldexp per element. */
static double g_f16_table[65536];
static double g_e4m3_table[256];
static int g_tables_ready = 0;
static void ensure_tables(void) {
  if (g_tables_ready) return;
  for (int i = 0; i < 65536; i++) g_f16_table[i] = kvo_f16_to_f64((uint16_t)i);
  for (int i = 0; i < 256; i++) g_e4m3_table[i] = kvo_e4m3_to_f64((uint8_t)i);
  g_tables_ready = 1;
}

/* Value of element e of a stored row: (code - 8) * scale, in fp64. */
static double q4_element(const uint8_t* stored, const uint16_t* scales, int D, int e) {
  int G = e / 32, i = e % 32;
  int o = 16 * G + i / 2; /* R4 */
  int code = (i % 2) ? (stored[o] >> 4) : (stored[o] & 0xF);
  (void)D;
  return (double)(code - 8) * g_f16_table[scales[G]];
}

void kvo_q4_dequant_row(const uint8_t* stored, const uint16_t* scales, int D, double* out) {
  ensure_tables();
  for (int e = 0; e < D; e++) out[e] = q4_element(stored, scales, D, e);
}

/* ------------------------------------------------------------------------- */
/* TQ4 rows (R7)                                                              */
/* ------------------------------------------------------------------------- */

/* The 16-level Lloyd-Max quantizer of N(0,1) (levels +-M_m), each magnitude
 * rounded to the nearest fp16 value (written out exactly). */
static const double kTq4M[8] = {0.12841796875, 0.387939453125, 0.65673828125, 0.9423828125,
                                1.255859375,   1.6181640625,   2.068359375,   2.732421875};

double kvo_tq4_level(int code) { return (code & 8 ? -1.0 : 1.0) * kTq4M[code & 7]; }

static int tq4_sign(const uint32_t* signs, int i) { return (signs[i / 32] >> (i % 32)) & 1; }

/* The store's rotation: y = fp32 butterfly of the signed row, times fp32(1/sqrt(n)). */
void kvo_tq4_rotate_f32(const float* x, int n, const uint32_t* signs, float* y) {
  for (int i = 0; i < n; i++) y[i] = tq4_sign(signs, i) ? -x[i] : x[i];
  for (int h = 1; h < n; h <<= 1)
    for (int i = 0; i < n; i++) {
      if (i & h) continue;
      float a = y[i], b = y[i + h];
      y[i] = a + b;
      y[i + h] = a - b;
    }
  const float c = (float)(1.0 / sqrt((double)n));
  for (int i = 0; i < n; i++) y[i] = y[i] * c;
}

/* The transform by its matrix definition, fp64: forward y = H (s * x) / sqrt(n),
 * inverse y = s * (H x) / sqrt(n), H[i][j] = (-1)^popcount(i & j). */
void kvo_tq4_rotate_f64(const double* x, int n, const uint32_t* signs, int inverse, double* y) {
  const double c = 1.0 / sqrt((double)n);
  for (int i = 0; i < n; i++) {
    double acc = 0.0;
    for (int j = 0; j < n; j++) {
      double xj = (!inverse && tq4_sign(signs, j)) ? -x[j] : x[j];
      acc += (__builtin_popcount((unsigned)(i & j)) & 1) ? -xj : xj;
    }
    y[i] = acc * c;
    if (inverse && tq4_sign(signs, i)) y[i] = -y[i];
  }
}

/* Quantise one row of n fp32 values (R7): n/2 code bytes (R4 order) and one fp16
 * scale (returned). */
uint16_t kvo_tq4_quantize_row(const float* x, int n, const uint32_t* signs, uint8_t* codes_out) {
  float* y = (float*)malloc(sizeof(float) * n);
  float* v = (float*)malloc(sizeof(float) * n);
  kvo_tq4_rotate_f32(x, n, signs, y);
  for (int i = 0; i < n; i++) v[i] = y[i] * y[i];
  for (int h = 1; h < n; h <<= 1)
    for (int i = 0; i < n; i += 2 * h) v[i] = v[i] + v[i + h];
  float ss = v[0];
  uint16_t s16 = kvo_f32_to_f16_sat(sqrtf(ss * (1.0f / (float)n)));
  float s = (float)kvo_f16_to_f64(s16);
  float tau[7];
  for (int k = 0; k < 7; k++) tau[k] = ((float)kTq4M[k] + (float)kTq4M[k + 1]) * 0.5f;
  for (int i = 0; i < n; i += 2) {
    int c[2];
    for (int e = 0; e < 2; e++) {
      c[e] = 0;
      if (s > 0.0f) {
        float r = y[i + e] / s; /* IEEE fp32 division */
        float a = fabsf(r);
        int m = 0;
        for (int k = 0; k < 7; k++) m += a > tau[k];
        c[e] = (r < 0.0f ? 8 : 0) | m;
      }
    }
    codes_out[i / 2] = (uint8_t)(c[0] | (c[1] << 4));
  }
  free(y);
  free(v);
  return s16;
}

/* Rotated-space values of one stored TQ4 row, fp64. */
void kvo_tq4_dequant_row(const uint8_t* codes, uint16_t scale, int n, double* out) {
  double s = kvo_f16_to_f64(scale);
  for (int i = 0; i < n; i++) {
    int c = (i % 2) ? (codes[i / 2] >> 4) : (codes[i / 2] & 0xF);
    out[i] = kvo_tq4_level(c) * s;
  }
}

/* ------------------------------------------------------------------------- */
/* Cache description used by the oracle (its own struct, not the library's).  */
/* ------------------------------------------------------------------------- */

/* KVO_Q4_0: the 4-bit rows without the rotation (same codes, scales and layout). */
enum { KVO_Q4 = 0, KVO_BF16 = 1, KVO_FP8 = 2, KVO_Q4_0 = 3, KVO_TQ4 = 4 };
enum { KVO_IN_F32 = 0, KVO_IN_BF16 = 1 };

typedef struct {
  int format;       /* KVO_Q4, KVO_BF16, KVO_FP8, KVO_Q4_0, KVO_TQ4 */
  int num_kv_heads; /* FP8: 1 */
  int head_dim;     /* Q4/BF16: D; FP8: latent width */
  int rope_dim;     /* FP8 only */
  int page_size;
  int num_pages;
  void* k;          /* Q4: codes; BF16: bf16 rows; FP8: latent e4m3 rows */
  void* k_scale;    /* Q4: fp16 scales; FP8: latent f32 scales */
  void* v;          /* Q4: codes; BF16: bf16 rows; FP8: rope e4m3 rows */
  void* v_scale;    /* Q4: fp16 scales; FP8: rope f32 scales; TQ4: one fp16 scale per row */
  const uint32_t* signs; /* TQ4: rotation sign mask [head_dim / 32] */
} kvo_cache;

/* Row index of (page, head, slot) in every plane. */
static int64_t row_index(const kvo_cache* c, int64_t page, int head, int slot) {
  return (page * c->num_kv_heads + head) * c->page_size + slot;
}

static float load_in(const void* p, int dtype, int64_t i) {
  if (dtype == KVO_IN_F32) return ((const float*)p)[i];
  return kvo_bf16_to_f32(((const uint16_t*)p)[i]);
}

/* Encode one fp8 row of n values (R6).  Writes n codes and returns the scale. */
static float fp8_encode_row(const float* x, int n, uint8_t* codes) {
  float amax = 0.0f;
  for (int i = 0; i < n; i++) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float inv = 448.0f / amax;
  if (amax == 0.0f || !isfinite(inv)) {
    for (int i = 0; i < n; i++) codes[i] = 0;
  } else {
    for (int i = 0; i < n; i++) codes[i] = kvo_f32_to_e4m3(x[i] * inv);
  }
  return amax / 448.0f;
}

/* Store n_tok new tokens.  Q4/BF16: k, v are [n_tok, Hk, D]; FP8: k is
 * [n_tok, D + rope] rows and v is unused.  slot_mapping[t] = page * page_size +
 * offset; a negative slot skips the token.  Returns the number of skipped
 * out-of-range slots. */
int kvo_store(const kvo_cache* c, const void* k, const void* v, int dtype, int64_t n_tok,
              const int32_t* slot_mapping) {
  int bad = 0;
  int D = c->head_dim;
  for (int64_t t = 0; t < n_tok; t++) {
    int32_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if ((int64_t)slot >= (int64_t)c->num_pages * c->page_size) { bad++; continue; }
    int64_t page = slot / c->page_size;
    int off = slot % c->page_size;
    if (c->format == KVO_FP8) {
      int W = D + c->rope_dim;
      float* row = (float*)malloc(sizeof(float) * W);
      for (int i = 0; i < W; i++) row[i] = load_in(k, dtype, t * W + i);
      int64_t r = row_index(c, page, 0, off);
      ((float*)c->k_scale)[r] = fp8_encode_row(row, D, (uint8_t*)c->k + r * D);
      ((float*)c->v_scale)[r] =
          fp8_encode_row(row + D, c->rope_dim, (uint8_t*)c->v + r * c->rope_dim);
      free(row);
      continue;
    }
    for (int hd = 0; hd < c->num_kv_heads; hd++) {
      int64_t r = row_index(c, page, hd, off);
      for (int kv = 0; kv < 2; kv++) {
        const void* src = kv ? v : k;
        float* row = (float*)malloc(sizeof(float) * D);
        for (int i = 0; i < D; i++) row[i] = load_in(src, dtype, (t * c->num_kv_heads + hd) * D + i);
        if (c->format == KVO_BF16) {
          uint16_t* dst = (uint16_t*)(kv ? c->v : c->k) + r * D;
          for (int i = 0; i < D; i++) dst[i] = kvo_f32_to_bf16(row[i]);
        } else if (c->format == KVO_TQ4) {
          uint8_t* dst = (uint8_t*)(kv ? c->v : c->k) + r * (D / 2);
          ((uint16_t*)(kv ? c->v_scale : c->k_scale))[r] = kvo_tq4_quantize_row(row, D, c->signs, dst);
        } else {
          uint8_t* dst = (uint8_t*)(kv ? c->v : c->k) + r * (D / 2);
          uint16_t* sc = (uint16_t*)(kv ? c->v_scale : c->k_scale) + r * (D / 32);
          q4_quantize_row(row, D, dst, sc, c->format == KVO_Q4);
        }
        free(row);
      }
    }
  }
  return bad;
}

/* ------------------------------------------------------------------------- */
/* Attention                                                                  */
/* ------------------------------------------------------------------------- */

/* Key and value vectors of absolute position pos of a sequence with block table
 * bt, KV head hd, as fp64.  Q4 and TQ4 rows are returned in the rotated space they are
 * stored in.  Returns 0 if the block table points outside the pool. */
static int load_kv(const kvo_cache* c, const int32_t* bt, int64_t pos, int hd, double* kvec,
                   double* vvec) {
  int64_t page = bt[pos / c->page_size];
  if (page < 0 || page >= c->num_pages) return 0;
  int off = (int)(pos % c->page_size);
  int D = c->head_dim;
  int64_t r = row_index(c, page, hd, off);
  ensure_tables();
  if (c->format == KVO_Q4 || c->format == KVO_Q4_0) {
    kvo_q4_dequant_row((const uint8_t*)c->k + r * (D / 2), (const uint16_t*)c->k_scale + r * (D / 32),
                       D, kvec);
    kvo_q4_dequant_row((const uint8_t*)c->v + r * (D / 2), (const uint16_t*)c->v_scale + r * (D / 32),
                       D, vvec);
  } else if (c->format == KVO_TQ4) {
    kvo_tq4_dequant_row((const uint8_t*)c->k + r * (D / 2), ((const uint16_t*)c->k_scale)[r], D, kvec);
    kvo_tq4_dequant_row((const uint8_t*)c->v + r * (D / 2), ((const uint16_t*)c->v_scale)[r], D, vvec);
  } else if (c->format == KVO_BF16) {
    for (int i = 0; i < D; i++) {
      kvec[i] = kvo_bf16_to_f32(((const uint16_t*)c->k)[r * D + i]);
      vvec[i] = kvo_bf16_to_f32(((const uint16_t*)c->v)[r * D + i]);
    }
  } else {
    /* FP8 absorbed: key = latent (x Lsc) ++ rope (x Rsc); value = latent (x Lsc). */
    double ls = ((const float*)c->k_scale)[r], rs = ((const float*)c->v_scale)[r];
    for (int i = 0; i < D; i++) {
      double lv = g_e4m3_table[((const uint8_t*)c->k)[r * D + i]] * ls;
      kvec[i] = lv;
      vvec[i] = lv;
    }
    for (int i = 0; i < c->rope_dim; i++)
      kvec[D + i] = g_e4m3_table[((const uint8_t*)c->v)[r * c->rope_dim + i]] * rs;
  }
  return 1;
}

static int key_width(const kvo_cache* c) {
  return c->format == KVO_FP8 ? c->head_dim + c->rope_dim : c->head_dim;
}

/* Prepare the query of one head in the space the cache is stored in: Q4 rotates
 * each 32-group by H (fp64), TQ4 the whole row by its signed transform, the
 * other formats use it as given. */
static void prep_query(const kvo_cache* c, const void* q, int dtype, int64_t off, double* out) {
  int W = key_width(c);
  double* tmp = (double*)malloc(sizeof(double) * W);
  for (int i = 0; i < W; i++) tmp[i] = load_in(q, dtype, off + i);
  if (c->format == KVO_Q4) {
    for (int G = 0; G < W / 32; G++) kvo_hadamard32_f64(tmp + 32 * G, out + 32 * G);
  } else if (c->format == KVO_TQ4) {
    kvo_tq4_rotate_f64(tmp, W, c->signs, 0, out);
  } else {
    memcpy(out, tmp, sizeof(double) * W);
  }
  free(tmp);
}

/* Attention of one query vector over the listed absolute positions.
 * split == 0: single pass, softmax over all keys at once.
 * split == 1: partitions of 512 listed keys (the last one the tail), each giving
 *             (m_p, z_p, acc_p); merged in ascending p by log-sum-exp.
 * Writes the context (value width) to out, rotated back for Q4 and TQ4.
 * Returns 0 on a block-table entry outside the pool. */
static int attend_one(const kvo_cache* c, const int32_t* bt, const double* qv, int hd,
                      const int64_t* pos, int64_t T, double sm_scale, int split, double* out) {
  int W = key_width(c), Dv = c->head_dim;
  double* kvec = (double*)malloc(sizeof(double) * W);
  double* vvec = (double*)malloc(sizeof(double) * Dv);
  double* o = (double*)calloc(Dv, sizeof(double));
  int ok = 1;
  if (T == 0) {
    /* No keys: the context is defined as zero. */
  } else if (!split) {
    double* s = (double*)malloc(sizeof(double) * T);
    double m = -INFINITY;
    for (int64_t j = 0; j < T && ok; j++) {
      ok = load_kv(c, bt, pos[j], hd, kvec, vvec);
      double acc = 0.0;
      for (int i = 0; i < W; i++) acc += qv[i] * kvec[i];
      s[j] = sm_scale * acc;
      if (s[j] > m) m = s[j];
    }
    double z = 0.0;
    for (int64_t j = 0; j < T && ok; j++) {
      load_kv(c, bt, pos[j], hd, kvec, vvec);
      double p = exp(s[j] - m);
      z += p;
      for (int i = 0; i < Dv; i++) o[i] += p * vvec[i];
    }
    for (int i = 0; i < Dv; i++) o[i] /= z;
    free(s);
  } else {
    int64_t P = (T + 511) / 512;
    double* mp = (double*)malloc(sizeof(double) * P);
    double* zp = (double*)malloc(sizeof(double) * P);
    double* ap = (double*)calloc((size_t)P * Dv, sizeof(double));
    for (int64_t p = 0; p < P && ok; p++) {
      int64_t j0 = 512 * p, j1 = j0 + 512 < T ? j0 + 512 : T;
      double m = -INFINITY;
      double* s = (double*)malloc(sizeof(double) * (j1 - j0));
      for (int64_t j = j0; j < j1 && ok; j++) {
        ok = load_kv(c, bt, pos[j], hd, kvec, vvec);
        double acc = 0.0;
        for (int i = 0; i < W; i++) acc += qv[i] * kvec[i];
        s[j - j0] = sm_scale * acc;
        if (s[j - j0] > m) m = s[j - j0];
      }
      double z = 0.0;
      for (int64_t j = j0; j < j1 && ok; j++) {
        load_kv(c, bt, pos[j], hd, kvec, vvec);
        double e = exp(s[j - j0] - m);
        z += e;
        for (int i = 0; i < Dv; i++) ap[p * Dv + i] += e * vvec[i];
      }
      mp[p] = m;
      zp[p] = z;
      free(s);
    }
    if (ok) {
      double M = -INFINITY;
      for (int64_t p = 0; p < P; p++) if (mp[p] > M) M = mp[p];
      double Z = 0.0;
      for (int64_t p = 0; p < P; p++) {
        double w = exp(mp[p] - M);
        Z += w * zp[p];
        for (int i = 0; i < Dv; i++) o[i] += w * ap[p * Dv + i];
      }
      for (int i = 0; i < Dv; i++) o[i] /= Z;
    }
    free(mp); free(zp); free(ap);
  }
  if (c->format == KVO_Q4) {
    for (int G = 0; G < Dv / 32; G++) kvo_hadamard32_f64(o + 32 * G, out + 32 * G);
  } else if (c->format == KVO_TQ4) {
    kvo_tq4_rotate_f64(o, Dv, c->signs, 1, out);
  } else {
    memcpy(out, o, sizeof(double) * Dv);
  }
  free(kvec); free(vvec); free(o);
  return ok;
}

/* Decode attention: for each sequence b and query head h, one query q[b, h, :]
 * (unrotated, dtype as given) attends keys 0 .. seq_lens[b]-1 (dense, sel ==
 * NULL) or the n_sel absolute positions sel[b, :] (gather).  Query head h reads
 * KV head h / (Hq / Hk).  out is [B, Hq, value width] fp64.  Returns 0 on a
 * block-table entry outside the pool. */
int kvo_decode(const kvo_cache* c, const void* q, int dtype, int B, int Hq, const int32_t* seq_lens,
               const int32_t* block_tables, int max_pages, const int32_t* sel, int n_sel,
               double sm_scale, int split, double* out) {
  int W = key_width(c), Dv = c->head_dim;
  int group = Hq / c->num_kv_heads;
  double* qv = (double*)malloc(sizeof(double) * W);
  int ok = 1;
  for (int b = 0; b < B && ok; b++) {
    int64_t T = sel ? n_sel : seq_lens[b];
    int64_t* pos = (int64_t*)malloc(sizeof(int64_t) * (T > 0 ? T : 1));
    for (int64_t j = 0; j < T; j++) pos[j] = sel ? sel[(int64_t)b * n_sel + j] : j;
    for (int h = 0; h < Hq && ok; h++) {
      prep_query(c, q, dtype, ((int64_t)b * Hq + h) * W, qv);
      ok = attend_one(c, block_tables + (int64_t)b * max_pages, qv, h / group, pos, T, sm_scale,
                      split, out + ((int64_t)b * Hq + h) * Dv);
    }
    free(pos);
  }
  free(qv);
  return ok;
}

/* Prefill attention over decoded slots [P1 "What it is", prompt chunks]:
 * query i (absolute position q_start + i) attends keys 0 .. q_start + i.
 * q is [n_q, Hq, key width] unrotated; out is [n_q, Hq, D] fp64, rotated back
 * (key width = D, or D + rope for the fp8 latent rows).
 * Only the listed query rows are computed when rows != NULL (rows[r] indexes
 * 0..n_q-1, out then has n_rows entries).  Returns 0 on a bad block table. */
int kvo_prefill(const kvo_cache* c, const void* q, int dtype, int n_q, int Hq, int64_t q_start,
                const int32_t* block_table, const int32_t* rows, int n_rows, double sm_scale,
                double* out) {
  int W = key_width(c), D = c->head_dim; /* fp8 rows: 576-wide queries, 512-wide outputs */
  int group = Hq / c->num_kv_heads;
  double* qv = (double*)malloc(sizeof(double) * W);
  int count = rows ? n_rows : n_q;
  int ok = 1;
  for (int r = 0; r < count && ok; r++) {
    int i = rows ? rows[r] : r;
    int64_t T = q_start + i + 1;
    int64_t* pos = (int64_t*)malloc(sizeof(int64_t) * T);
    for (int64_t j = 0; j < T; j++) pos[j] = j;
    for (int h = 0; h < Hq && ok; h++) {
      prep_query(c, q, dtype, ((int64_t)i * Hq + h) * W, qv);
      ok = attend_one(c, block_table, qv, h / group, pos, T, sm_scale, 0,
                      out + ((int64_t)r * Hq + h) * D);
    }
    free(pos);
  }
  free(qv);
  return ok;
}

/* Direct fp8 row encoder exposed for pins: codes for n values, returns scale. */
float kvo_fp8_encode_row(const float* x, int n, uint8_t* codes) { return fp8_encode_row(x, n, codes); }

/* ------------------------------------------------------------------------- */
/* Array helpers for the test harness (plain loops over the scalar functions). */
/* ------------------------------------------------------------------------- */
void kvo_f32_to_f16_n(const float* x, uint16_t* y, int64_t n) { for (int64_t i = 0; i < n; i++) y[i] = kvo_f32_to_f16(x[i]); }
void kvo_f32_to_f16_sat_n(const float* x, uint16_t* y, int64_t n) { for (int64_t i = 0; i < n; i++) y[i] = kvo_f32_to_f16_sat(x[i]); }
void kvo_f16_to_f64_n(const uint16_t* x, double* y, int64_t n) { for (int64_t i = 0; i < n; i++) y[i] = kvo_f16_to_f64(x[i]); }
void kvo_f32_to_bf16_n(const float* x, uint16_t* y, int64_t n) { for (int64_t i = 0; i < n; i++) y[i] = kvo_f32_to_bf16(x[i]); }
void kvo_f32_to_e4m3_n(const float* x, uint8_t* y, int64_t n) { for (int64_t i = 0; i < n; i++) y[i] = kvo_f32_to_e4m3(x[i]); }
void kvo_e4m3_to_f64_n(const uint8_t* x, double* y, int64_t n) { for (int64_t i = 0; i < n; i++) y[i] = kvo_e4m3_to_f64(x[i]); }
void kvo_fwht32_f32_n(float* x, int64_t ngroups) { for (int64_t g = 0; g < ngroups; g++) kvo_fwht32_f32(x + 32 * g); }
void kvo_hadamard32_f64_n(const double* x, double* y, int64_t ngroups) {
  for (int64_t g = 0; g < ngroups; g++) kvo_hadamard32_f64(x + 32 * g, y + 32 * g);
}
float kvo_rotation_constant(void) { return (float)(1.0 / sqrt(32.0)); }
