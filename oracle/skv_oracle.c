/*
 * skv_oracle.c -- plain CPU oracle for sparse long-context decode.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * restatement of the method that the CUDA library is checked against.  Only
 * the test suite, the smoke check and the benchmark's CPU-baseline leg load
 * it; the product path never does.  It shares no code, header, table or
 * constant with the CUDA sources.
 *
 * Sources (page title, section):
 *  [P1] "8 agents x 250K context on two 3090s: sparse KV decode with a rank-64
 *       key sketch and a host-RAM tier" -- "What shipped" (sketch, int4 tier,
 *       sinks + tail, shared pick, windowed CLOCK, zero-copy misses).
 *  [P2] "vLLM's Hybrid HiSparse Triples Concurrent Requests on Million-Token
 *       Contexts" -- "Three residency states, one block pool" (fused LRU
 *       resolve) and "What it composes with" (hot buffer = 2 x top-K).
 *  [P3] "You can offload most of Qwen3.8-Flash-Next's KV cache to RAM with
 *       little decode slowdown" (pooled indexer keys, byte arithmetic).
 *  [P4] "3.14M Context on 3x 3090: ..." -- "Why" (sparse threshold
 *       4*block_topk+3), "No Need to Rewrite the Kernel" (row addressing
 *       [token][kv_head][dim]), "What Needs to Stay in VRAM" (pooled keys).
 *
 * Conventions (readings where the pages are silent are listed in the design
 * notes and repeated at each function):
 *  - bf16/fp16/fp8 values are decoded exactly from their bit patterns.
 *  - fp32 arithmetic is done one operation at a time in the loop order stated
 *    at each function.  The file MUST be compiled with -ffp-contract=off so
 *    that no multiply-add is fused on any host architecture.
 *  - Attention is evaluated in fp64 from the dequantised values.
 *
 * Build:  gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fopenmp
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_API __attribute__((visibility("default")))

ORC_API int orc_version(void) { return 1; }

ORC_API int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

ORC_API void orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* Number formats, decoded from their definitions.                           */
/* ------------------------------------------------------------------------ */

/* bfloat16: the upper 16 bits of an IEEE binary32. */
ORC_API float orc_bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
ORC_API double orc_f16_to_f64(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  return s ? -v : v;
}

/*
 * Round a finite double to a binary floating format with `p` significant bits
 * and minimum normal exponent `emin` (round to nearest, ties to even), and
 * return the rounded value as a double.  Overflow handling is the caller's.
 * The rounding step is a single rint() of the value expressed in units of the
 * format's quantum at that binade, which is exact in double for the formats
 * used here (p <= 24).
 */
static double round_to_format(double x, int p, int emin) {
  if (x == 0.0 || !isfinite(x)) return x;
  double a = fabs(x);
  int e2;
  frexp(a, &e2);     /* a = f * 2^e2, f in [0.5, 1) */
  int e = e2 - 1;    /* a in [2^e, 2^(e+1)) */
  if (e < emin) e = emin; /* subnormal range uses the minimum quantum */
  double quantum = ldexp(1.0, e - (p - 1));
  double r = rint(a / quantum) * quantum; /* a/quantum is exact: power of 2 */
  return x < 0 ? -r : r;
}

/* binary32 -> binary16, round to nearest even, IEEE overflow to infinity. */
ORC_API uint16_t orc_f32_to_f16(float f) {
  if (isnan(f)) return 0x7e00;
  uint16_t sign = signbit(f) ? 0x8000 : 0;
  double r = round_to_format((double)f, 11, -14);
  double a = fabs(r);
  if (a >= 65536.0 || isinf(f)) return sign | 0x7c00; /* 65520 rounds here */
  if (a == 0.0) return sign;
  if (a < ldexp(1.0, -14)) /* subnormal: a = m * 2^-24 */
    return sign | (uint16_t)ldexp(a, 24);
  int e2;
  frexp(a, &e2);
  int e = e2 - 1; /* a = (1 + m/1024) * 2^e */
  uint16_t m = (uint16_t)(ldexp(a, 10 - e) - 1024.0);
  return sign | (uint16_t)((e + 15) << 10) | m;
}

/* binary32 -> bfloat16, round to nearest even. */
ORC_API uint16_t orc_f32_to_bf16(float f) {
  if (isnan(f)) return 0x7fc0;
  double r = round_to_format((double)f, 8, -126);
  if (fabs(r) >= ldexp(1.0, 128)) return signbit(f) ? 0xff80 : 0x7f80;
  float rf = (float)r; /* exact: r has <= 8 significant bits */
  uint32_t u;
  memcpy(&u, &rf, 4);
  return (uint16_t)(u >> 16);
}

/* OCP 8-bit float E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3
 * mantissa bits; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN;
 * there are no infinities.  Largest finite value 448. */
ORC_API double orc_fp8_e4m3_to_f64(uint8_t b) {
  int s = (b >> 7) & 1, e = (b >> 3) & 0xf, m = b & 7;
  double v;
  if (e == 15 && m == 7)
    v = NAN;
  else if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/* Two's-complement 4-bit code stored in the low nibble. */
static int nib_to_int(unsigned v) {
  v &= 0xf;
  return v >= 8 ? (int)v - 16 : (int)v;
}

/* Round-half-even to an integer, then clamp. Inputs are finite here. */
static int rint_clamp(float x, int lo, int hi) {
  if (!(x > (float)lo)) return lo; /* also catches -inf */
  if (!(x < (float)hi)) return hi;
  return (int)rintf(x);
}

/* ------------------------------------------------------------------------ */
/* a1: key sketch.  [P1] "What shipped": keys are projected on a frozen       */
/* rank-64 basis and the sketch is stored int4.                              */
/* ------------------------------------------------------------------------ */

/*
 * s[t,h,j] = sum_{i=0}^{d-1} P[i*r + j] * k[t,h,i]   (fp32, i ascending)
 * If c != NULL: x = s / c[h*r+j] (fp32 IEEE division), code = clamp(rint(x),
 * -8, 7), packed two per byte: byte b of a head holds dim 2b in the low nibble
 * and dim 2b+1 in the high nibble; heads follow each other inside a token.
 * Output rows are Hkv*r/2 bytes.  A zero step c gives code 0.
 * Optional outputs: s_out (fp32 [n][Hkv][r]) and x_out (the fp32 ratio s/c
 * before rounding, used by tests to recognise rounding ties).
 */
ORC_API void orc_sketch_project(const uint16_t *keys, int64_t n, int Hkv, int d,
                                int r, const float *P, const float *c,
                                uint8_t *q4_out, float *s_out, float *x_out) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n; t++) {
    for (int h = 0; h < Hkv; h++) {
      const uint16_t *k = keys + (t * Hkv + h) * (int64_t)d;
      for (int j = 0; j < r; j++) {
        float s = 0.0f;
        for (int i = 0; i < d; i++) s = s + P[(int64_t)i * r + j] * orc_bf16_to_f32(k[i]);
        int64_t o = (t * Hkv + h) * (int64_t)r + j;
        if (s_out) s_out[o] = s;
        if (c) {
          float cj = c[h * r + j];
          float x = (cj != 0.0f) ? s / cj : 0.0f;
          if (x_out) x_out[o] = x;
          int code = (cj != 0.0f) ? rint_clamp(x, -8, 7) : 0;
          if (q4_out) {
            uint8_t *byte = q4_out + t * (int64_t)(Hkv * r / 2) + h * (r / 2) + j / 2;
            if ((j & 1) == 0)
              *byte = (uint8_t)((*byte & 0xf0) | (code & 0xf));
            else
              *byte = (uint8_t)((*byte & 0x0f) | ((code & 0xf) << 4));
          }
        }
      }
    }
  }
}

/*
 * a2: query side of the sketch.  One pick per layer is shared by all KV heads
 * ([P1] "What shipped"), read as a sum of the per-head sketch scores; the
 * query heads of one KV head's group (kv_head = g / G, contiguous groups) are
 * summed first:
 *   proj[g][j] = sum_i P[i*r+j] * q[b,g,i]                (fp32, i ascending)
 *   qp[h][j]   = (sum_{g in group h, ascending} proj[g][j]) * c[h*r+j]
 * (the multiplication by c is skipped when c == NULL: fp32 sketch mode).
 * int8 mode (q8_out != NULL): sigma = max_m |qp[m]| / 127 per request (fp32),
 * q8 = clamp(rint(qp / sigma), -127, 127); sigma == 0 gives q8 = 0.
 * Outputs: qp_out fp32 [B][Hkv*r] (always), q8_out int8 [B][Hkv*r],
 * sigma_out fp32 [B], x_out fp32 [B][Hkv*r] = qp/sigma before rounding.
 */
ORC_API void orc_sketch_query(const uint16_t *q, int B, int Hq, int Hkv, int d,
                              int r, const float *P, const float *c, float *qp_out,
                              int8_t *q8_out, float *sigma_out, float *x_out) {
  int G = Hq / Hkv;
  for (int b = 0; b < B; b++) {
    float *qp = qp_out + (int64_t)b * Hkv * r;
    for (int h = 0; h < Hkv; h++) {
      for (int j = 0; j < r; j++) {
        float acc = 0.0f;
        for (int gg = 0; gg < G; gg++) {
          int g = h * G + gg;
          const uint16_t *qg = q + ((int64_t)b * Hq + g) * d;
          float pj = 0.0f;
          for (int i = 0; i < d; i++) pj = pj + P[(int64_t)i * r + j] * orc_bf16_to_f32(qg[i]);
          acc = acc + pj;
        }
        if (c) acc = acc * c[h * r + j];
        qp[h * r + j] = acc;
      }
    }
    if (q8_out) {
      float amax = 0.0f;
      for (int m = 0; m < Hkv * r; m++)
        if (fabsf(qp[m]) > amax) amax = fabsf(qp[m]);
      float sigma = amax / 127.0f;
      if (sigma_out) sigma_out[b] = sigma;
      for (int m = 0; m < Hkv * r; m++) {
        float x = (sigma != 0.0f) ? qp[m] / sigma : 0.0f;
        if (x_out) x_out[(int64_t)b * Hkv * r + m] = x;
        q8_out[(int64_t)b * Hkv * r + m] = (int8_t)((sigma != 0.0f) ? rint_clamp(x, -127, 127) : 0);
      }
    }
  }
}

/*
 * a2': pooled indexer keys.  [P3] and [P4] "What Needs to Stay in VRAM": the
 * indexer keys are pooled per block of `ratio` tokens (compress ratio 4).
 * Reading: the pool is the mean, summed in token order in fp32
 * ((x0 + x1) + x2) + x3, divided by the ratio (exact for 4), rounded to bf16.
 * keys: bf16 [n_blocks*ratio][D]; out: bf16 [n_blocks][D].
 */
ORC_API void orc_pool_keys(const uint16_t *keys, int64_t n_blocks, int D, int ratio,
                           uint16_t *out) {
#pragma omp parallel for schedule(static)
  for (int64_t blk = 0; blk < n_blocks; blk++) {
    for (int i = 0; i < D; i++) {
      float s = orc_bf16_to_f32(keys[(blk * ratio) * (int64_t)D + i]);
      for (int u = 1; u < ratio; u++) s = s + orc_bf16_to_f32(keys[(blk * ratio + u) * (int64_t)D + i]);
      s = s / (float)ratio;
      out[blk * (int64_t)D + i] = orc_f32_to_bf16(s);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* a3: indexer scores and order keys.                                        */
/* ------------------------------------------------------------------------ */

enum { ORC_SKETCH_INT4 = 0, ORC_SKETCH_F32 = 1, ORC_POOLED_BF16 = 2 };

/* Order key: a uint32 whose unsigned order is the score's order.
 * int32 scores: flip the sign bit.  fp32 scores: -0 is treated as +0; for
 * negative values all bits are inverted, otherwise the sign bit is set. */
ORC_API uint32_t orc_order_key_i32(int32_t s) { return (uint32_t)s ^ 0x80000000u; }

ORC_API uint32_t orc_order_key_f32(float s) {
  if (s == 0.0f) s = 0.0f; /* -0 -> +0 */
  uint32_t u;
  memcpy(&u, &s, 4);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

/* Candidate range of request b.  Sketch modes ([P1]): tokens [S, T-W); the
 * sinks and tail are always attended and do not compete (reading: the union
 * is then disjoint and the row count fixed).  Pooled mode ([P4]): every
 * complete block [0, T/ratio). */
static void cand_range(int mode, int64_t T, int ratio, int S, int W, int64_t *lo, int64_t *hi) {
  if (mode == ORC_POOLED_BF16) {
    *lo = 0;
    *hi = T / ratio;
  } else {
    *lo = S;
    *hi = T - W;
    if (*hi < *lo) *hi = *lo;
  }
}

/*
 * INT4: score[t] = sum_{m=0}^{width-1} q8[m] * code(t, m)   (exact integer)
 * F32 : score[t] = sum_m qp[m] * s[t][m]                    (fp32, m ascending)
 * POOLED_BF16: score[blk] = sum_i q_idx[i] * pooled[blk][i] (fp32, i ascending)
 * query: int8 [B][width] | fp32 [B][width] | bf16 [B][width]
 * keys : u8 [B][n_cap][width/2] | fp32 [B][n_cap][width] | bf16 [B][n_cap][width]
 * Outputs (any may be NULL): iscore (int32), fscore (fp32), dscore (fp64 of
 * the same sum, diagnostic), okey (order keys).  Only candidates are written.
 * Returns the number of NaN scores met (an error for the caller).
 */
ORC_API int64_t orc_index_score(int mode, int B, int width, const void *query,
                                const void *keys, int64_t n_cap,
                                const int32_t *lengths, int ratio, int S, int W,
                                int32_t *iscore, float *fscore, double *dscore,
                                uint32_t *okey) {
  int64_t nan_count = 0;
  for (int b = 0; b < B; b++) {
    int64_t lo, hi;
    cand_range(mode, lengths[b], ratio, S, W, &lo, &hi);
#pragma omp parallel for schedule(static) reduction(+ : nan_count)
    for (int64_t t = lo; t < hi; t++) {
      int64_t o = (int64_t)b * n_cap + t;
      if (mode == ORC_SKETCH_INT4) {
        const int8_t *q8 = (const int8_t *)query + (int64_t)b * width;
        const uint8_t *row = (const uint8_t *)keys + o * (width / 2);
        int64_t acc = 0;
        for (int m = 0; m < width; m++) {
          unsigned byte = row[m / 2];
          int code = nib_to_int((m & 1) ? (byte >> 4) : byte);
          acc += (int64_t)q8[m] * code;
        }
        int32_t s = (int32_t)acc;
        if (iscore) iscore[o] = s;
        if (dscore) dscore[o] = (double)acc;
        if (okey) okey[o] = orc_order_key_i32(s);
      } else {
        float acc = 0.0f;
        double dacc = 0.0;
        for (int m = 0; m < width; m++) {
          float qv, kv;
          if (mode == ORC_SKETCH_F32) {
            qv = ((const float *)query)[(int64_t)b * width + m];
            kv = ((const float *)keys)[o * width + m];
          } else {
            qv = orc_bf16_to_f32(((const uint16_t *)query)[(int64_t)b * width + m]);
            kv = orc_bf16_to_f32(((const uint16_t *)keys)[o * width + m]);
          }
          acc = acc + qv * kv;
          dacc += (double)qv * (double)kv;
        }
        if (isnan(acc)) nan_count++;
        if (fscore) fscore[o] = acc;
        if (dscore) dscore[o] = dacc;
        if (okey) okey[o] = orc_order_key_f32(acc);
      }
    }
  }
  return nan_count;
}

/* ------------------------------------------------------------------------ */
/* a4: top-k selection, union with sinks and tail, dense fallback.           */
/* ------------------------------------------------------------------------ */

typedef struct {
  uint32_t key;
  int64_t idx;
} kv_pair;

/* Higher key first; among equal keys the lower index first ([P1] asks for a
 * deterministic selection; lowest index is the tie rule read here). */
static int cmp_desc_key_asc_idx(const void *a, const void *b) {
  const kv_pair *x = (const kv_pair *)a, *y = (const kv_pair *)b;
  if (x->key != y->key) return x->key > y->key ? -1 : 1;
  return (x->idx > y->idx) - (x->idx < y->idx);
}

static int cmp_i64(const void *a, const void *b) {
  int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
  return (x > y) - (x < y);
}

/*
 * Per request b with T = lengths[b] tokens (the current token included):
 * sketch mode (ratio == 1):
 *   if T <= S + W + k: every token 0..T-1 (dense fallback);
 *   else: the k best candidates of [S, T-W) by (key desc, index asc), and the
 *   output is [0, S) ++ picks (ascending) ++ [T-W, T); count = S + k + W.
 * pooled mode (ratio > 1, S = W = 0): with nb = T / ratio complete blocks,
 *   if T <= ratio*k + ratio - 1 ([P4] "Why": 4*block_topk + 3): every token;
 *   else: the k best blocks, each expanded to its `ratio` tokens in ascending
 *   order, then the incomplete last block's tokens [ratio*nb, T).
 * idx_out: int32 [B][max_rows]; count_out: int32 [B].  Returns 0, or -1 if a
 * request needs more than max_rows rows.
 */
ORC_API int orc_topk_select(int B, const uint32_t *okey, int64_t n_cap,
                            const int32_t *lengths, int k, int S, int W, int ratio,
                            int32_t *idx_out, int max_rows, int32_t *count_out) {
  int rc = 0;
  for (int b = 0; b < B; b++) {
    int64_t T = lengths[b];
    int32_t *out = idx_out + (int64_t)b * max_rows;
    int dense = (ratio <= 1) ? (T <= (int64_t)S + W + k) : (T <= (int64_t)ratio * k + ratio - 1);
    if (dense) {
      if (T > max_rows) { rc = -1; count_out[b] = 0; continue; }
      for (int64_t t = 0; t < T; t++) out[t] = (int32_t)t;
      count_out[b] = (int32_t)T;
      continue;
    }
    int64_t lo = (ratio <= 1) ? S : 0;
    int64_t hi = (ratio <= 1) ? T - W : T / ratio;
    int64_t n = hi - lo;
    kv_pair *c = (kv_pair *)malloc(sizeof(kv_pair) * (size_t)n);
    for (int64_t i = 0; i < n; i++) {
      c[i].idx = lo + i;
      c[i].key = okey[(int64_t)b * n_cap + lo + i];
    }
    qsort(c, (size_t)n, sizeof(kv_pair), cmp_desc_key_asc_idx);
    int64_t *pick = (int64_t *)malloc(sizeof(int64_t) * (size_t)k);
    for (int i = 0; i < k; i++) pick[i] = c[i].idx;
    qsort(pick, (size_t)k, sizeof(int64_t), cmp_i64);
    int64_t m = 0;
    if (ratio <= 1) {
      if ((int64_t)S + k + W > max_rows) { rc = -1; count_out[b] = 0; free(c); free(pick); continue; }
      for (int64_t t = 0; t < S; t++) out[m++] = (int32_t)t;
      for (int i = 0; i < k; i++) out[m++] = (int32_t)pick[i];
      for (int64_t t = T - W; t < T; t++) out[m++] = (int32_t)t;
    } else {
      int64_t nb = T / ratio;
      if ((int64_t)ratio * k + (T - ratio * nb) > max_rows) { rc = -1; count_out[b] = 0; free(c); free(pick); continue; }
      for (int i = 0; i < k; i++)
        for (int u = 0; u < ratio; u++) out[m++] = (int32_t)(pick[i] * ratio + u);
      for (int64_t t = ratio * nb; t < T; t++) out[m++] = (int32_t)t;
    }
    count_out[b] = (int32_t)m;
    free(c);
    free(pick);
  }
  return rc;
}

/* ------------------------------------------------------------------------ */
/* KV row encodings.                                                         */
/* ------------------------------------------------------------------------ */

/*
 * int8 rows (reading of the pages' "int8 attention"): one row = D int8 codes
 * and one fp16 scale; scale = fp16(max|x| / 127) (fp32 division, then
 * round-to-nearest-even to fp16), code = clamp(rint(x / scale), -127, 127)
 * with x / scale an fp32 division by the fp16 value.  A zero scale (all-zero
 * row, or an amax too small for fp16) gives all-zero codes.
 * x: bf16 [n][D] -> q: int8 [n][D], scale: fp16 bits [n].
 */
ORC_API void orc_quant_int8_rows(const uint16_t *x, int64_t n, int D, int8_t *q,
                                 uint16_t *scale) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n; t++) {
    const uint16_t *row = x + t * (int64_t)D;
    float amax = 0.0f;
    for (int i = 0; i < D; i++) {
      float a = fabsf(orc_bf16_to_f32(row[i]));
      if (a > amax) amax = a;
    }
    uint16_t sh = orc_f32_to_f16(amax / 127.0f);
    float sf = (float)orc_f16_to_f64(sh);
    scale[t] = sh;
    for (int i = 0; i < D; i++) {
      int v = 0;
      if (sf != 0.0f && isfinite(sf)) v = rint_clamp(orc_bf16_to_f32(row[i]) / sf, -127, 127);
      q[t * (int64_t)D + i] = (int8_t)v;
    }
  }
}

/*
 * int4 host rows ([P1] "What shipped": int4, 64-dim groups, fp16 scales, 272 B
 * per token-head for K and V together).  One encoded K (or V) vector of D
 * dims: D/2 bytes of codes packed as in the sketch (dim 2b low nibble, 2b+1
 * high nibble), then D/64 fp16 group scales, little-endian.  For D = 256 this
 * is 128 + 8 = 136 bytes.  Group scale = fp16(max|x| / 7) over the group's 64
 * values; code = clamp(rint(x / scale), -8, 7); a zero scale gives code 0.
 * x: bf16 [n][D] -> out: u8 [n][D/2 + 2*(D/64)].
 */
ORC_API int orc_int4_row_bytes(int D) { return D / 2 + 2 * (D / 64); }

ORC_API void orc_quant_int4_rows(const uint16_t *x, int64_t n, int D, uint8_t *out) {
  int rb = orc_int4_row_bytes(D);
  int ng = D / 64;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n; t++) {
    const uint16_t *row = x + t * (int64_t)D;
    uint8_t *o = out + t * (int64_t)rb;
    memset(o, 0, (size_t)rb);
    for (int g = 0; g < ng; g++) {
      float amax = 0.0f;
      for (int i = 64 * g; i < 64 * g + 64; i++) {
        float a = fabsf(orc_bf16_to_f32(row[i]));
        if (a > amax) amax = a;
      }
      uint16_t sh = orc_f32_to_f16(amax / 7.0f);
      float sf = (float)orc_f16_to_f64(sh);
      o[D / 2 + 2 * g] = (uint8_t)(sh & 0xff);
      o[D / 2 + 2 * g + 1] = (uint8_t)(sh >> 8);
      for (int i = 64 * g; i < 64 * g + 64; i++) {
        int v = 0;
        if (sf != 0.0f && isfinite(sf)) v = rint_clamp(orc_bf16_to_f32(row[i]) / sf, -8, 7);
        if ((i & 1) == 0)
          o[i / 2] = (uint8_t)((o[i / 2] & 0xf0) | (v & 0xf));
        else
          o[i / 2] = (uint8_t)((o[i / 2] & 0x0f) | ((v & 0xf) << 4));
      }
    }
  }
}

/*
 * int4 -> int8 row ([P1]: host rows are "dequantized back to int8 rows on
 * fetch").  Reading: x_i = code_i * s_g in fp32 (exact), s8 = fp16(max|x| /
 * 127), q8_i = clamp(rint(x_i / s8), -127, 127); a zero s8 gives zero codes.
 * in: one encoded vector (orc_quant_int4_rows layout); out: int8 [D], fp16 s8.
 */
ORC_API void orc_int4_to_int8_row(const uint8_t *in, int D, int8_t *q8, uint16_t *s8) {
  float x[1024];
  float amax = 0.0f;
  for (int i = 0; i < D; i++) {
    int g = i / 64;
    uint16_t sh = (uint16_t)(in[D / 2 + 2 * g] | (in[D / 2 + 2 * g + 1] << 8));
    int code = nib_to_int((i & 1) ? (in[i / 2] >> 4) : in[i / 2]);
    x[i] = (float)code * (float)orc_f16_to_f64(sh);
    if (fabsf(x[i]) > amax) amax = fabsf(x[i]);
  }
  uint16_t sh8 = orc_f32_to_f16(amax / 127.0f);
  float sf = (float)orc_f16_to_f64(sh8);
  *s8 = sh8;
  for (int i = 0; i < D; i++)
    q8[i] = (int8_t)((sf != 0.0f && isfinite(sf)) ? rint_clamp(x[i] / sf, -127, 127) : 0);
}

/* ------------------------------------------------------------------------ */
/* a6: exact attention over the selected rows, fp64.                         */
/* ------------------------------------------------------------------------ */

enum { ORC_KV_BF16 = 0, ORC_KV_INT8 = 1, ORC_KV_FP8 = 2 };

/* Value of element j of head h of pool row `row`. */
static double kv_elem(int kind, const void *pool, const uint16_t *scale,
                      const float *row_scale, int64_t row, int64_t pitch,
                      int Hkv, int h, int dh, int j) {
  int64_t off = row * pitch + (int64_t)h * dh + j;
  if (kind == ORC_KV_BF16) return (double)orc_bf16_to_f32(((const uint16_t *)pool)[off]);
  if (kind == ORC_KV_INT8)
    return (double)((const int8_t *)pool)[off] * orc_f16_to_f64(scale[row * Hkv + h]);
  double s = row_scale ? (double)row_scale[row] : 1.0;
  return orc_fp8_e4m3_to_f64(((const uint8_t *)pool)[off]) * s;
}

/*
 * For request b and query head g (kv head h = g / (Hq/Hkv)):
 *   logit_i = scale * sum_j q[b,g,j] * K(row_i, h, j)
 *   out[b,g,:] = sum_i softmax(logit)_i * V(row_i, h, :)
 * over the count[b] selected rows, row_i = b*req_row_stride + rows[b][i]
 * ([P4] "No Need to Rewrite the Kernel": a row is found by adding an offset to
 * the base, layout [token][kv_head][dim]).
 * K element (row, h, j) = k_pool[row*k_pitch + h*d + j], V element (row, h, j)
 * = v_pool[row*v_pitch + h*dv + j]; int8 rows are multiplied by their fp16
 * scale (k_scale / v_scale, [row][Hkv]); fp8 rows by row_scale[row] (1 if
 * NULL).  For the latent (MLA) layout K and V are the same buffer: the first
 * dv of the d dims are the value.  Empty selection gives a zero output.
 */
ORC_API void orc_attend(int kind, int B, int Hq, int Hkv, int d, int dv,
                        const uint16_t *q, const void *k_pool, const void *v_pool,
                        const uint16_t *k_scale, const uint16_t *v_scale,
                        const float *row_scale, int64_t k_pitch, int64_t v_pitch,
                        int64_t req_row_stride, const int32_t *rows, int max_rows,
                        const int32_t *count, double softmax_scale, double *out) {
  int G = Hq / Hkv;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int b = 0; b < B; b++) {
    for (int g = 0; g < Hq; g++) {
      int h = g / G;
      int n = count[b];
      double *o = out + ((int64_t)b * Hq + g) * dv;
      for (int j = 0; j < dv; j++) o[j] = 0.0;
      if (n <= 0) continue;
      double *logit = (double *)malloc(sizeof(double) * (size_t)n);
      const uint16_t *qg = q + ((int64_t)b * Hq + g) * d;
      double mx = -INFINITY;
      for (int i = 0; i < n; i++) {
        int64_t row = (int64_t)b * req_row_stride + rows[(int64_t)b * max_rows + i];
        double acc = 0.0;
        for (int j = 0; j < d; j++)
          acc += (double)orc_bf16_to_f32(qg[j]) *
                 kv_elem(kind, k_pool, k_scale, row_scale, row, k_pitch, Hkv, h, d, j);
        logit[i] = softmax_scale * acc;
        if (logit[i] > mx) mx = logit[i];
      }
      double l = 0.0;
      for (int i = 0; i < n; i++) {
        double p = exp(logit[i] - mx);
        l += p;
        int64_t row = (int64_t)b * req_row_stride + rows[(int64_t)b * max_rows + i];
        for (int j = 0; j < dv; j++)
          o[j] += p * kv_elem(kind, v_pool, v_scale, row_scale, row, v_pitch, Hkv, h, dv, j);
      }
      for (int j = 0; j < dv; j++) o[j] /= l;
      free(logit);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* a5: resolvers.                                                            */
/* ------------------------------------------------------------------------ */

/*
 * Windowed CLOCK over one request's hot buffer ([P1] "What shipped": the GPU
 * keeps the sketch, sinks, recent tail and a 2.5% hot buffer managed by
 * windowed CLOCK).  Reading:
 *   state: slot_token[Hs] (-1 empty), ref[Hs] (0/1), token_slot[n_tok]
 *   (-1 none), *hand, and use_step[Hs] (the step that last used the slot).
 *   phase 1: every pick that has a slot is a hit: ref = 1, use_step = step
 *            (a slot used this step is never evicted this step -- the window);
 *   phase 2: misses in ascending token order sweep the hand: the slot under
 *            the hand is skipped if used this step; taken if empty or ref == 0
 *            (its old token loses the slot); otherwise its ref is cleared and
 *            the hand moves on.  A taken slot gets the token, ref = 1 and
 *            use_step = step.
 * picks: ascending token ids [n_picks].  Outputs slot_of_pick[n_picks] and
 * miss_of_pick[n_picks] (1 for a miss).  Returns the number of misses, or -1
 * if the sweep cannot finish (more picks than slots).
 */
ORC_API int orc_clock_step(int Hs, int32_t *slot_token, uint8_t *ref, int32_t *use_step,
                           int32_t *token_slot, int32_t *hand, int32_t step,
                           const int32_t *picks, int n_picks, int32_t *slot_of_pick,
                           int32_t *miss_of_pick) {
  if (n_picks > Hs) return -1;
  int misses = 0;
  for (int i = 0; i < n_picks; i++) {
    int32_t s = token_slot[picks[i]];
    if (s >= 0) {
      ref[s] = 1;
      use_step[s] = step;
      slot_of_pick[i] = s;
      miss_of_pick[i] = 0;
    } else {
      slot_of_pick[i] = -1;
      miss_of_pick[i] = 1;
    }
  }
  for (int i = 0; i < n_picks; i++) {
    if (!miss_of_pick[i]) continue;
    int taken = -1;
    for (int64_t guard = 0; guard < 3 * (int64_t)Hs + 3 && taken < 0; guard++) {
      int32_t s = *hand;
      *hand = (*hand + 1) % Hs;
      if (use_step[s] == step) continue;
      if (slot_token[s] < 0 || ref[s] == 0) {
        taken = s;
      } else {
        ref[s] = 0;
      }
    }
    if (taken < 0) return -1;
    if (slot_token[taken] >= 0) token_slot[slot_token[taken]] = -1;
    slot_token[taken] = picks[i];
    token_slot[picks[i]] = taken;
    ref[taken] = 1;
    use_step[taken] = step;
    slot_of_pick[i] = taken;
    misses++;
  }
  return misses;
}

/*
 * Full CLOCK resolve of one request for one layer (host int4 tier):
 * the selection idx[0..n) (ascending) is split into sinks (t < S), tail
 * (t >= T - W) and picks (the rest).  HBM row of a sink: t; of a tail token:
 * S + (t mod W); of a pick: S + W + slot.  Each miss fetches the token's host
 * row (Hkv heads x [K vector | V vector], orc_quant_int4_rows layout, so
 * Hkv * 2 * row_bytes per token) and writes the int8 requantisation
 * (orc_int4_to_int8_row) of every head into the slot's HBM row.
 * HBM pool of the request: k8/v8 int8 [rows][Hkv][D], k_s/v_s fp16 [rows][Hkv].
 * Returns the number of misses, or -1 on failure.
 */
ORC_API int orc_resolve_clock(int64_t T, int S, int W, int Hkv, int D, int Hs,
                              const int32_t *idx, int n, int32_t step,
                              int32_t *slot_token, uint8_t *ref, int32_t *use_step,
                              int32_t *token_slot, int32_t *hand,
                              const uint8_t *host_rows, int8_t *k8, int8_t *v8,
                              uint16_t *k_s, uint16_t *v_s, int32_t *row_out) {
  int32_t *picks = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
  int32_t *pos = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
  int32_t *slot = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
  int32_t *miss = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
  int np = 0;
  for (int i = 0; i < n; i++) {
    int64_t t = idx[i];
    if (t < S)
      row_out[i] = (int32_t)t;
    else if (t >= T - W)
      row_out[i] = (int32_t)(S + (t % W));
    else {
      picks[np] = (int32_t)t;
      pos[np] = i;
      np++;
    }
  }
  int m = orc_clock_step(Hs, slot_token, ref, use_step, token_slot, hand, step, picks,
                         np, slot, miss);
  if (m < 0) {
    free(picks); free(pos); free(slot); free(miss);
    return -1;
  }
  int rb = orc_int4_row_bytes(D);
  for (int p = 0; p < np; p++) {
    int64_t row = S + W + slot[p];
    row_out[pos[p]] = (int32_t)row;
    if (!miss[p]) continue;
    const uint8_t *tok = host_rows + (int64_t)picks[p] * Hkv * 2 * rb;
    for (int h = 0; h < Hkv; h++) {
      orc_int4_to_int8_row(tok + (2 * h) * rb, D, k8 + (row * Hkv + h) * D, &k_s[row * Hkv + h]);
      orc_int4_to_int8_row(tok + (2 * h + 1) * rb, D, v8 + (row * Hkv + h) * D, &v_s[row * Hkv + h]);
    }
  }
  free(picks); free(pos); free(slot); free(miss);
  return m;
}

typedef struct {
  int64_t stamp;
  int32_t slot;
} lru_pair;

static int cmp_lru(const void *a, const void *b) {
  const lru_pair *x = (const lru_pair *)a, *y = (const lru_pair *)b;
  if (x->stamp != y->stamp) return x->stamp < y->stamp ? -1 : 1;
  return (x->slot > y->slot) - (x->slot < y->slot);
}

/*
 * Mixed-residency LRU resolve of one request ([P2] "Three residency states,
 * one block pool": resident tokens are read in place, hot tokens are read and
 * their LRU entry refreshed, a miss copies one row from pinned host memory
 * into an LRU slot; the tail is never evicted; [P2] "What it composes with":
 * the hot buffer holds 2 x top-K rows).  Readings: pages of `page` tokens;
 * block_table[p] >= 0 is the pool page holding resident page p, -1 a null
 * placeholder (host-only page).  Hot slot s is pool row hot_rows[s] when
 * hot_rows is given (a hot-buffer page is an ordinary block leased from the
 * pool: "Three residency states, one block pool"), else hot_base + s.
 * State: stamp[n_slots] (-1 empty), slot_token[n_slots] (-1 none),
 * token_slot[n_tok] (-1 none).
 *   1. resident token: row = block_table[t/page]*page + t%page;
 *   2. token with a hot slot: hit, stamp = step;
 *   3. misses, ascending token order, take the slots not touched this step
 *      with the smallest (stamp, slot index); the old token loses the slot;
 *      the host row (row_bytes bytes at host + t*row_bytes) is copied to the
 *      slot's pool row; stamp = step.
 * pool: u8 [rows][row_bytes].  Returns the number of misses, or -1 when the
 * untouched slots are fewer than the misses.
 */
ORC_API int orc_resolve_lru(const int32_t *idx, int n, int page, const int32_t *block_table,
                            int64_t hot_base, const int32_t *hot_rows, int n_slots, int64_t step, int64_t *stamp,
                            int32_t *slot_token, int32_t *token_slot,
                            const uint8_t *host, uint8_t *pool, int64_t row_bytes,
                            int32_t *row_out) {
  int32_t *mtok = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
  int32_t *mpos = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
  int nm = 0;
  for (int i = 0; i < n; i++) {
    int64_t t = idx[i];
    int32_t bp = block_table[t / page];
    if (bp >= 0) {
      row_out[i] = (int32_t)((int64_t)bp * page + t % page);
    } else if (token_slot[t] >= 0) {
      int32_t s = token_slot[t];
      stamp[s] = step;
      row_out[i] = hot_rows ? hot_rows[s] : (int32_t)(hot_base + s);
    } else {
      mtok[nm] = (int32_t)t;
      mpos[nm] = i;
      nm++;
    }
  }
  lru_pair *cand = (lru_pair *)malloc(sizeof(lru_pair) * (size_t)(n_slots + 1));
  int nc = 0;
  for (int s = 0; s < n_slots; s++)
    if (stamp[s] != step) {
      cand[nc].stamp = stamp[s];
      cand[nc].slot = s;
      nc++;
    }
  if (nc < nm) {
    free(mtok); free(mpos); free(cand);
    return -1;
  }
  qsort(cand, (size_t)nc, sizeof(lru_pair), cmp_lru);
  for (int i = 0; i < nm; i++) {
    int32_t s = cand[i].slot;
    if (slot_token[s] >= 0) token_slot[slot_token[s]] = -1;
    slot_token[s] = mtok[i];
    token_slot[mtok[i]] = s;
    stamp[s] = step;
    int64_t row = hot_rows ? (int64_t)hot_rows[s] : hot_base + s;
    memcpy(pool + row * row_bytes, host + (int64_t)mtok[i] * row_bytes, (size_t)row_bytes);
    row_out[mpos[i]] = (int32_t)row;
  }
  free(mtok); free(mpos); free(cand);
  return nm;
}
