/*
 * QSA oracle: a plain, slow, float64 CPU implementation of the quantized sparse
 * attention layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU
 * baseline call this code.  The library (int8_kv_top_gb300) never includes, links or
 * calls it, and this file includes nothing from the library.
 *
 * Fixed layer shape ("round 6 track b - qsa flash", delivered change; "opus_r9_qsa",
 * what changed): 2 KV groups, 12 query heads per group (query head h reads group
 * h / 12), head dim 256, one fp16 scale per 64 elements of every K and V row
 * ("round 6 track b", delivered change: a half4 of scales per cell).
 *
 * Layouts (row-major, all plain arrays):
 *   q   [T][24][256]  fp16 bits   token t of the call sits at position pos0 + t
 *   kq  [n][2][256]   int8        cache cell c, group g
 *   vq  [n][2][256]   int8
 *   ksc [n][2][4]     fp16 bits   scale of elements 64b..64b+63
 *   vsc [n][2][4]     fp16 bits
 *
 * What is computed, step by step (every function below cites its step):
 *  1. dequantise: k^[c,g,d] = kq[c,g,d] * ksc[c,g,d/64] (exact in float64), same for v^.
 *  2. logits per head: s_h(c) = sm_scale * sum_d q[t,h,d] * k^[c,g,d], for causal cells
 *     c < n_kv(t) = pos0 + t + 1.
 *  3. cell set per (token, group): every causal cell while n_kv <= identity_max
 *     ("round 6 track b", delivered change: identity ids while n_kv <= 2051); otherwise
 *     the topk cells with the largest selection score sum_{h in g} s_h(c), equal scores
 *     going to the lower cell index, listed in ascending cell order.
 *  4. softmax over the set (natural exp, max subtracted), 5. o = sum p * v^.
 *  6. decode partials: the set split into consecutive 64-cell chunks; per chunk and
 *     head m = max s, l = sum exp(s - m), o = sum exp(s - m) v^ (unnormalised), stored
 *     as o[256], m, l with a head stride of 258 values ("round 27 track b - qsa prep and
 *     merge", correctness: head stride 258, chunk stride 6192).
 *  7. merge: M = max_k m_k, L = sum_k l_k exp(m_k - M), out = sum_k exp(m_k - M) o_k / L
 *     ("round 27 track b", correctness: serial L = fma(l[k], e[k], L) over ascending k).
 *  8. quantise (the cache-writing step): per 64-element block a = max |x|,
 *     scale = fp16(a / 127), code = clamp(round_half_away(x / scale), -127, 127); all in
 *     fp32 arithmetic with fp16 rounding to nearest even; a zero scale gives zero codes.
 *
 * Selection is ranked by the EXACT score: every fp16 value is an integer multiple of
 * 2^-24, so 16 * 2^48 * score = sum_b S_b * B_b with S_b = ksc * 2^24 and
 * B_b = sum_{d in b} Qsum_d * kq_d, Qsum_d = sum_h q_hd * 2^24 (int64), all exact in
 * 128-bit integers.  Ordering by this integer orders by the score itself.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define NG 2
#define HPG 12
#define NH 24
#define HD 256
#define BLK 64
#define NB 4
#define PSTRIDE 258
#define CHUNK 64

/* ------------------------------------------------------------ fp16 helpers */

/* IEEE 754 binary16 bits -> double, from the format's definition. */
double oracle_half_to_double(uint16_t h) {
  const int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25);
  return s ? -v : v;
}

/* fp16 value * 2^24 as an exact integer (finite inputs only). */
static int64_t half_to_int24(uint16_t h) {
  const int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  int64_t v = (e == 0) ? (int64_t)m : ((int64_t)(1024 + m) << (e - 1));
  return s ? -v : v;
}

/* float -> fp16 bits, round to nearest, ties to even (finite inputs). */
uint16_t oracle_float_to_half(float f) {
  const double x = (double)f;
  const uint16_t sign = signbit(x) ? 0x8000u : 0u;
  const double a = fabs(x);
  if (a == 0.0) return sign;
  if (a >= 65520.0) return sign | 0x7C00u; /* rounds to infinity */
  int ex;
  frexp(a, &ex);      /* a = f * 2^ex, f in [0.5, 1) */
  int e = ex - 1;     /* a in [2^e, 2^(e+1)) */
  if (e < -14) e = -14;
  double n = rint(ldexp(a, 10 - e)); /* a / 2^(e-10), exact scaling; rint = nearest even */
  if (n >= 2048.0) { n = 1024.0; e += 1; }
  if (e > 15) return sign | 0x7C00u;
  if (n < 1024.0) return sign | (uint16_t)n; /* subnormal (e == -14) */
  return sign | (uint16_t)(((e + 15) << 10) | ((int)n - 1024));
}

/* ------------------------------------------------------------ step 8: quantise */

/* x: [n_rows][256] fp16 bits -> xq [n_rows][256] int8 and xsc [n_rows][4] fp16 bits. */
void oracle_quantize(const uint16_t* x, int64_t n_rows, int8_t* xq, uint16_t* xsc) {
  for (int64_t r = 0; r < n_rows; ++r) {
    for (int b = 0; b < NB; ++b) {
      const uint16_t* xb = x + r * HD + b * BLK;
      float a = 0.0f;
      for (int i = 0; i < BLK; ++i) {
        const float v = fabsf((float)oracle_half_to_double(xb[i]));
        if (v > a) a = v;
      }
      const float ratio = a / 127.0f;
      const uint16_t sh = oracle_float_to_half(ratio);
      const float s = (float)oracle_half_to_double(sh);
      xsc[r * NB + b] = sh;
      for (int i = 0; i < BLK; ++i) {
        int code = 0;
        if (s != 0.0f) {
          const float t = (float)oracle_half_to_double(xb[i]) / s;
          float rq = roundf(t); /* half away from zero */
          if (rq > 127.0f) rq = 127.0f;
          if (rq < -127.0f) rq = -127.0f;
          code = (int)rq;
        }
        xq[r * HD + b * BLK + i] = (int8_t)code;
      }
    }
  }
}

/* ------------------------------------------------------------ steps 1-2 */

/* Step 2 for one head and one cell, float64 (step 1 inline). */
static double logit(const uint16_t* qh, const int8_t* kq, const uint16_t* ksc, int64_t c, int g, double sm_scale) {
  double acc = 0.0;
  for (int d = 0; d < HD; ++d) {
    const double khat = (double)kq[(c * NG + g) * HD + d] * oracle_half_to_double(ksc[(c * NG + g) * NB + d / BLK]);
    acc += oracle_half_to_double(qh[d]) * khat;
  }
  return sm_scale * acc;
}

/* ------------------------------------------------------------ step 3: cell set */

typedef struct {
  __int128 key;
  int32_t idx;
} ranked;

static int cmp_ranked(const void* pa, const void* pb) {
  const ranked* a = (const ranked*)pa;
  const ranked* b = (const ranked*)pb;
  if (a->key != b->key) return (a->key > b->key) ? -1 : 1; /* larger score first */
  return (a->idx < b->idx) ? -1 : (a->idx > b->idx); /* ties: lower index first */
}

typedef struct {
  double key;
  int32_t idx;
} ranked_f64;

static int cmp_ranked_f64(const void* pa, const void* pb) {
  const ranked_f64* a = (const ranked_f64*)pa;
  const ranked_f64* b = (const ranked_f64*)pb;
  if (a->key != b->key) return (a->key > b->key) ? -1 : 1;
  return (a->idx < b->idx) ? -1 : (a->idx > b->idx);
}

static int cmp_i32(const void* pa, const void* pb) {
  const int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a > b) - (a < b);
}

/* Exact selection key of cell c for the token whose 24 query heads start at q_tok. */
__int128 oracle_exact_key(const uint16_t* q_tok, const int8_t* kq, const uint16_t* ksc, int64_t c, int g) {
  __int128 key = 0;
  for (int b = 0; b < NB; ++b) {
    int64_t Bb = 0;
    for (int d = b * BLK; d < (b + 1) * BLK; ++d) {
      int64_t qsum = 0;
      for (int h = 0; h < HPG; ++h) qsum += half_to_int24(q_tok[(g * HPG + h) * HD + d]);
      Bb += qsum * (int64_t)kq[(c * NG + g) * HD + d];
    }
    key += (__int128)half_to_int24(ksc[(c * NG + g) * NB + b]) * (__int128)Bb;
  }
  return key;
}

/* Exact key as two 64-bit halves (for callers without 128-bit integers). */
void oracle_exact_key_parts(const uint16_t* q_tok, const int8_t* kq, const uint16_t* ksc, int64_t c, int g,
                            int64_t* hi, uint64_t* lo) {
  const __int128 k = oracle_exact_key(q_tok, kq, ksc, c, g);
  *hi = (int64_t)(k >> 64);
  *lo = (uint64_t)k;
}

/*
 * Step 3 for one (token, group).  n_kv = number of causal cells.  Writes the set in
 * ascending cell order to cells[] (capacity max(n_kv, topk)), returns its size.
 * *f64_differs (may be NULL) is set to 1 when ranking by the float64 sum of the
 * per-head logits would pick a different set (a diagnostic of near-ties).
 */
int oracle_cell_set(const uint16_t* q_tok, const int8_t* kq, const uint16_t* ksc, int64_t n_kv, int g, int topk,
                    int identity_max, double sm_scale, int32_t* cells, int* f64_differs) {
  if (f64_differs) *f64_differs = 0;
  if (n_kv <= identity_max) {
    for (int64_t c = 0; c < n_kv; ++c) cells[c] = (int32_t)c;
    return (int)n_kv;
  }
  ranked* r = (ranked*)malloc(sizeof(ranked) * (size_t)n_kv);
  for (int64_t c = 0; c < n_kv; ++c) {
    r[c].key = oracle_exact_key(q_tok, kq, ksc, c, g);
    r[c].idx = (int32_t)c;
  }
  qsort(r, (size_t)n_kv, sizeof(ranked), cmp_ranked);
  const int k = (int)(topk < n_kv ? topk : n_kv);
  for (int i = 0; i < k; ++i) cells[i] = r[i].idx;
  qsort(cells, (size_t)k, sizeof(int32_t), cmp_i32);
  free(r);

  if (f64_differs) {
    ranked_f64* rf = (ranked_f64*)malloc(sizeof(ranked_f64) * (size_t)n_kv);
    for (int64_t c = 0; c < n_kv; ++c) {
      double s = 0.0;
      for (int h = 0; h < HPG; ++h) s += logit(q_tok + (g * HPG + h) * HD, kq, ksc, c, g, sm_scale);
      rf[c].key = s;
      rf[c].idx = (int32_t)c;
    }
    qsort(rf, (size_t)n_kv, sizeof(ranked_f64), cmp_ranked_f64);
    int32_t* alt = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
    for (int i = 0; i < k; ++i) alt[i] = rf[i].idx;
    qsort(alt, (size_t)k, sizeof(int32_t), cmp_i32);
    *f64_differs = memcmp(alt, cells, sizeof(int32_t) * (size_t)k) != 0;
    free(alt);
    free(rf);
  }
  return k;
}

/* ------------------------------------------------------------ steps 4-5 */

/* Attention of the group's 12 heads over the given cell set; out [12][256]. */
void oracle_attend(const uint16_t* q_tok, const int8_t* kq, const int8_t* vq, const uint16_t* ksc,
                   const uint16_t* vsc, int g, const int32_t* cells, int n_set, double sm_scale, double* out) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(n_set > 0 ? n_set : 1));
  for (int h = 0; h < HPG; ++h) {
    const uint16_t* qh = q_tok + (g * HPG + h) * HD;
    double mx = -INFINITY;
    for (int i = 0; i < n_set; ++i) {
      s[i] = logit(qh, kq, ksc, cells[i], g, sm_scale);
      if (s[i] > mx) mx = s[i];
    }
    double denom = 0.0;
    for (int i = 0; i < n_set; ++i) {
      s[i] = exp(s[i] - mx);
      denom += s[i];
    }
    double* o = out + h * HD;
    for (int d = 0; d < HD; ++d) o[d] = 0.0;
    for (int i = 0; i < n_set; ++i) {
      const int64_t c = cells[i];
      const double p = s[i] / denom;
      for (int d = 0; d < HD; ++d) {
        const double vhat =
            (double)vq[(c * NG + g) * HD + d] * oracle_half_to_double(vsc[(c * NG + g) * NB + d / BLK]);
        o[d] += p * vhat;
      }
    }
  }
  free(s);
}

/* ------------------------------------------------------------ step 6 */

/* Partials of the group's 12 heads; part [n_chunks][12][258] (o[256], m, l). Returns n_chunks. */
int oracle_partials(const uint16_t* q_tok, const int8_t* kq, const int8_t* vq, const uint16_t* ksc,
                    const uint16_t* vsc, int g, const int32_t* cells, int n_set, double sm_scale, double* part) {
  const int n_chunks = (n_set + CHUNK - 1) / CHUNK;
  for (int k = 0; k < n_chunks; ++k) {
    const int i0 = k * CHUNK, i1 = (i0 + CHUNK < n_set) ? i0 + CHUNK : n_set;
    for (int h = 0; h < HPG; ++h) {
      const uint16_t* qh = q_tok + (g * HPG + h) * HD;
      double s[CHUNK];
      double m = -INFINITY;
      for (int i = i0; i < i1; ++i) {
        s[i - i0] = logit(qh, kq, ksc, cells[i], g, sm_scale);
        if (s[i - i0] > m) m = s[i - i0];
      }
      double* dst = part + ((size_t)k * HPG + h) * PSTRIDE;
      double l = 0.0;
      for (int d = 0; d < HD; ++d) dst[d] = 0.0;
      for (int i = i0; i < i1; ++i) {
        const int64_t c = cells[i];
        const double e = exp(s[i - i0] - m);
        l += e;
        for (int d = 0; d < HD; ++d)
          dst[d] += e * (double)vq[(c * NG + g) * HD + d] * oracle_half_to_double(vsc[(c * NG + g) * NB + d / BLK]);
      }
      dst[HD] = m;
      dst[HD + 1] = l;
    }
  }
  return n_chunks;
}

/* ------------------------------------------------------------ step 7 */

/* Merge of one head's chunks; part_h points at chunk 0 of the head, chunk stride in values. */
static void merge_head(const double* part_h, size_t chunk_stride, int n_chunks, double* out) {
  double M = -INFINITY;
  for (int k = 0; k < n_chunks; ++k) {
    const double m = part_h[k * chunk_stride + HD];
    if (m > M) M = m;
  }
  double L = 0.0;
  for (int k = 0; k < n_chunks; ++k) L += part_h[k * chunk_stride + HD + 1] * exp(part_h[k * chunk_stride + HD] - M);
  for (int d = 0; d < HD; ++d) {
    double acc = 0.0;
    for (int k = 0; k < n_chunks; ++k) acc += exp(part_h[k * chunk_stride + HD] - M) * part_h[k * chunk_stride + d];
    out[d] = acc / L;
  }
}

/* part [N][chunk_cap][24][258] float32, n_chunks [N] -> out [N][24][256] float64. */
void oracle_merge_f32(const float* part, const int32_t* n_chunks, int N, int chunk_cap, double* out) {
  const size_t cs = (size_t)NH * PSTRIDE;
  double* tmp = (double*)malloc(sizeof(double) * (size_t)chunk_cap * PSTRIDE);
  for (int t = 0; t < N; ++t)
    for (int h = 0; h < NH; ++h) {
      for (int k = 0; k < n_chunks[t]; ++k)
        for (int j = 0; j < PSTRIDE; ++j)
          tmp[(size_t)k * PSTRIDE + j] = (double)part[((size_t)t * chunk_cap + k) * cs + (size_t)h * PSTRIDE + j];
      merge_head(tmp, PSTRIDE, n_chunks[t], out + ((size_t)t * NH + h) * HD);
    }
  free(tmp);
}

/* part [n_chunks][12][258] float64 (one group) -> out [12][256]. */
void oracle_merge_group(const double* part, int n_chunks, double* out) {
  for (int h = 0; h < HPG; ++h) merge_head(part + (size_t)h * PSTRIDE, (size_t)HPG * PSTRIDE, n_chunks, out + h * HD);
}

/* ------------------------------------------------------------ output gate */

/*
 * The gate input the pages' evaluator feeds the layer ("round 6 track b - qsa flash",
 * experiment contract: deterministic random int8, scales, query and gate inputs).  The pages
 * give no formula; this oracle takes the plainest reading, an elementwise sigmoid gate on the
 * attention output of every (token, head, dim):  out *= 1 / (1 + exp(-gate)), in float64.
 * out and gate share a layout ([T][24][256]); gate holds fp16 bits.
 */
void oracle_apply_gate(double* out, const uint16_t* gate, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] *= 1.0 / (1.0 + exp(-oracle_half_to_double(gate[i])));
}

/* ------------------------------------------------------------ fused prep */

/*
 * The pages' fused prep (qsa_prep: "round 27 track b - qsa prep and merge", decision and
 * rejected prep fusion: raw rows, their gamma, a norm_rope step, mrope variants; correctness:
 * it writes qcur and the int8 cache kq vq ksc vsc).  The pages name the parts but not their
 * formulas; this oracle takes the plainest readings:
 *  - RMS norm per head row of 256 values with a learned gain:
 *      y_d = x_d / sqrt(mean_d(x^2) + eps) * gamma_d            (q rows use q_gamma, k rows k_gamma)
 *  - rotary position embedding on the normed q and k rows, halves paired (i, i + rd/2) for
 *    i < rd/2 (rd = rotary_dim; dims >= rd untouched), angle theta_i = p * base^(-2 i / rd):
 *      (y_i, y_{i+rd/2}) -> (y_i cos - y_{i+rd/2} sin,  y_{i+rd/2} cos + y_i sin)
 *    with p = pos0 + t; for mrope, pair i takes component c of the token's three positions
 *    pos3[t][c], c = 0, 1, 2 over consecutive frequency sections of sizes sections[0..2];
 *  - v rows are not normed or rotated.
 * Outputs (float64): qcur [T][24][256], kcur [T][2][256].  The cache rows of cell pos0 + t are
 * the quantiser (step 8) applied to fp16(kcur) and to v.
 */
static void prep_row(const uint16_t* x, const double* gamma, double p_or_nan, const int32_t* p3, int rotary_dim,
                     double base, double eps, const int* sections, double* y) {
  double ms = 0.0;
  for (int d = 0; d < HD; ++d) {
    const double v = oracle_half_to_double(x[d]);
    ms += v * v;
  }
  ms /= HD;
  const double r = 1.0 / sqrt(ms + eps);
  for (int d = 0; d < HD; ++d) y[d] = oracle_half_to_double(x[d]) * r * gamma[d];
  const int h = rotary_dim / 2;
  for (int i = 0; i < h; ++i) {
    double p = p_or_nan;
    if (p3) p = (double)p3[i < sections[0] ? 0 : (i < sections[0] + sections[1] ? 1 : 2)];
    const double theta = p * pow(base, -2.0 * i / rotary_dim);
    const double c = cos(theta), sn = sin(theta);
    const double a = y[i], b = y[i + h];
    y[i] = a * c - b * sn;
    y[i + h] = b * c + a * sn;
  }
}

void oracle_prep(const uint16_t* q_raw, const uint16_t* k_raw, const double* q_gamma, const double* k_gamma,
                 const int32_t* pos3, int T, int pos0, double base, int rotary_dim, double eps, const int* sections,
                 double* qcur, double* kcur) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const double p = (double)pos0 + t;
    const int32_t* p3 = pos3 ? pos3 + 3 * t : NULL;
    for (int h = 0; h < NH; ++h)
      prep_row(q_raw + ((size_t)t * NH + h) * HD, q_gamma, p, p3, rotary_dim, base, eps, sections,
               qcur + ((size_t)t * NH + h) * HD);
    for (int g = 0; g < NG; ++g)
      prep_row(k_raw + ((size_t)t * NG + g) * HD, k_gamma, p, p3, rotary_dim, base, eps, sections,
               kcur + ((size_t)t * NG + g) * HD);
  }
}

/* ------------------------------------------------------------ call-level drivers */

/*
 * Prefill for a subset of the call's tokens (toks[i] in [0, T)).  Outputs per listed
 * token i:  out [i][24][256] (float64), ids [i][2][topk] (ascending; rows of identity
 * tokens are filled with -1), n_set [i][2], f64_differs [i][2].
 */
void oracle_prefill(const uint16_t* q, const int8_t* kq, const int8_t* vq, const uint16_t* ksc, const uint16_t* vsc,
                    int T, int pos0, const int32_t* toks, int n_toks, int topk, int identity_max, double sm_scale,
                    double* out, int32_t* ids, int32_t* n_set, int32_t* f64_differs) {
  (void)T;
  const int cap = (identity_max > topk ? identity_max : topk);
#pragma omp parallel for schedule(dynamic, 1)
  for (int w = 0; w < n_toks * NG; ++w) {
    const int i = w / NG, g = w % NG, t = toks[i];
    const int64_t n_kv = (int64_t)pos0 + t + 1;
    const uint16_t* q_tok = q + (size_t)t * NH * HD;
    int32_t* cells = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_kv > cap ? n_kv : cap));
    int differs = 0;
    const int ns = oracle_cell_set(q_tok, kq, ksc, n_kv, g, topk, identity_max, sm_scale, cells,
                                   f64_differs ? &differs : NULL);
    oracle_attend(q_tok, kq, vq, ksc, vsc, g, cells, ns, sm_scale, out + ((size_t)i * NH + g * HPG) * HD);
    int32_t* row = ids + ((size_t)i * NG + g) * topk;
    if (n_kv <= identity_max) {
      for (int j = 0; j < topk; ++j) row[j] = -1;
    } else {
      for (int j = 0; j < topk; ++j) row[j] = (j < ns) ? cells[j] : -1;
    }
    n_set[i * NG + g] = ns;
    if (f64_differs) f64_differs[i * NG + g] = differs;
    free(cells);
  }
}

/*
 * Decode step for N new tokens at positions P..P+N-1 (token t sees n_kv = P + t + 1
 * cells).  Outputs: part [N][chunk_cap][24][258] float64 (slots past a token's chunk
 * count untouched), n_chunks [N], merged out [N][24][256] (step 7 over the partials) and
 * direct [N][24][256] (steps 4-5 over the same set, for the merge identity).
 */
void oracle_decode(const uint16_t* q, const int8_t* kq, const int8_t* vq, const uint16_t* ksc, const uint16_t* vsc,
                   int N, int P, int topk, int identity_max, double sm_scale, int chunk_cap, double* part,
                   int32_t* n_chunks, double* out, double* direct, int32_t* ids) {
  const int cap = (identity_max > topk ? identity_max : topk);
#pragma omp parallel for schedule(dynamic, 1)
  for (int w = 0; w < N * NG; ++w) {
    const int t = w / NG, g = w % NG;
    const int64_t n_kv = (int64_t)P + t + 1;
    const uint16_t* q_tok = q + (size_t)t * NH * HD;
    int32_t* cells = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_kv > cap ? n_kv : cap));
    const int ns = oracle_cell_set(q_tok, kq, ksc, n_kv, g, topk, identity_max, sm_scale, cells, NULL);
    const int nc = (ns + CHUNK - 1) / CHUNK;
    double* gpart = (double*)malloc(sizeof(double) * (size_t)(nc > 0 ? nc : 1) * HPG * PSTRIDE);
    oracle_partials(q_tok, kq, vq, ksc, vsc, g, cells, ns, sm_scale, gpart);
    for (int k = 0; k < nc && k < chunk_cap; ++k)
      for (int h = 0; h < HPG; ++h)
        memcpy(part + (((size_t)t * chunk_cap + k) * NH + g * HPG + h) * PSTRIDE,
               gpart + ((size_t)k * HPG + h) * PSTRIDE, sizeof(double) * PSTRIDE);
    oracle_merge_group(gpart, nc, out + ((size_t)t * NH + g * HPG) * HD);
    oracle_attend(q_tok, kq, vq, ksc, vsc, g, cells, ns, sm_scale, direct + ((size_t)t * NH + g * HPG) * HD);
    if (ids) {
      int32_t* row = ids + ((size_t)t * NG + g) * topk;
      for (int j = 0; j < topk; ++j) row[j] = (n_kv > identity_max && j < ns) ? cells[j] : -1;
    }
    n_chunks[t] = nc;
    free(gpart);
    free(cells);
  }
}
