/*
 * moe_oracle.c -- plain, slow CPU oracle for the fused mixture-of-experts
 * layer forward (routing, permutation, expert MLPs, weighted combine).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the tests, the smoke check and the benchmark's CPU-baseline leg may load
 * it.  It shares no code, header, table or constant with the CUDA library.
 *
 * Sources (page title, section):
 *  - "vLLM Community Traces H20 MoE Scheduling Inefficiency to Expert-Load
 *    Kernel Selection": rows-per-expert estimate ceil(tokens*top_k/experts),
 *    clamped to >= 1, applied after worst-case capacity (para. 3).
 *  - "PR #39593: Fix FlashInfer CUTLASS BF16 + CUDA graphs IMA", section
 *    "Fix": NaN router logits replaced by -FLT_MAX before softmax/sigmoid
 *    and before top-k; top-k returns k distinct ids.  Same page, "Purpose":
 *    the FP8 conversion clamps with fminf/fmaxf, mapping NaN to +-448.
 *  - "Lab notes #6: We tuned vLLM's MoE kernels on an H100", "Method" and
 *    the config-file line: FP8 w8a8 with [128,128] weight block scales.
 *  - OCP 8-bit floating point specification (E4M3: bias 7, max 448, no
 *    infinities, S.1111.111 is NaN) for the e4m3 codec, and IEEE 754
 *    round-to-nearest-even for bfloat16.
 *
 * Readings taken where the pages are silent (each is also listed in the
 * design notes): +-Inf logits clamp to +-FLT_MAX; selection is done on the
 * sanitised logits with ties to the lower expert index; a renormalisation
 * whose denominator is zero or not finite gives 1/k to each pick; the gate
 * projection is rows [0, I) of w13 and the up projection rows [I, 2I);
 * activation FP8 scale = max(amax, 1e-10) / 448 per 128-column group, the
 * clamp is fmaxf(fminf(v, 448), -448) so NaN maps to +448; within one
 * expert, permuted rows keep ascending flat index order (f = t*k + j).
 *
 * Arithmetic: values are dequantised to fp32, every dot product, exp and
 * sum is carried in double.  The one place fp32 is used on purpose is the
 * FP8 activation quantisation, whose codes are an integer decision taken in
 * the precision the method takes it in (fp32 divide, fp32 max).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_DTYPE_F32 0
#define ORACLE_DTYPE_BF16 1
#define ORACLE_DTYPE_FP8 2

/* ------------------------------------------------------------------ */
/* numeric codecs                                                      */
/* ------------------------------------------------------------------ */

/* bfloat16 is the upper half of an IEEE binary32. */
float oracle_bf16_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* IEEE round-to-nearest-even from binary32 to bfloat16; NaN -> quiet NaN. */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if (isnan(f)) return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* OCP E4M3 decode: sign, 4-bit exponent (bias 7), 3-bit mantissa.
 * Exponent field 0 is subnormal (m/8 * 2^-6).  S.1111.111 is NaN; there
 * are no infinities, so S.1111.110 = 448 is the largest finite value. */
float oracle_e4m3_decode(uint8_t c) {
  int s = (c >> 7) & 1;
  int e = (c >> 3) & 15;
  int m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return (float)(s ? -v : v);
}

/* E4M3 encode, round to nearest with ties to the even code, saturating to
 * +-448 (values at or beyond the largest finite magnitude, and infinities,
 * give +-448).  Written as a search over the 127 non-negative finite codes:
 * slow, but each step can be checked by eye against the format.  NaN input
 * gives the NaN code 0x7F (the method never feeds NaN here: it clamps first). */
uint8_t oracle_e4m3_encode(float v) {
  if (isnan(v)) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  int best = 0;
  double best_d = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    double d = fabs((double)oracle_e4m3_decode((uint8_t)c) - a);
    if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_d = d;
    }
  }
  return (uint8_t)(sign | best);
}

/* Per-group FP8 quantisation of n fp32 values in groups of 128 columns:
 * scale = max(amax, 1e-10) / 448 (fp32), code = e4m3(clamp(v / scale)),
 * clamp = fmaxf(fminf(x, 448), -448) so that NaN becomes +448.
 * amax uses fmaxf, which ignores NaN operands. */
void oracle_quant_group128(const float* v, int n, uint8_t* codes, float* scales) {
  for (int g = 0; g * 128 < n; ++g) {
    int lo = g * 128, hi = lo + 128 < n ? lo + 128 : n;
    float amax = 0.0f;
    for (int i = lo; i < hi; ++i) amax = fmaxf(amax, fabsf(v[i]));
    float scale = fmaxf(amax, 1e-10f) / 448.0f;
    scales[g] = scale;
    for (int i = lo; i < hi; ++i) {
      float q = v[i] / scale;
      q = fmaxf(fminf(q, 448.0f), -448.0f);
      codes[i] = oracle_e4m3_encode(q);
    }
  }
}

/* ------------------------------------------------------------------ */
/* step a-3: rows-per-expert estimate                                  */
/* ------------------------------------------------------------------ */

/* est = ceil(T * k / E), clamped to at least 1 (H20 article, para. 3). */
int oracle_estimate(int T, int k, int E) {
  if (E <= 0) return 1;
  long long rows = (long long)T * (long long)k;
  long long est = (rows + E - 1) / E;
  return est < 1 ? 1 : (int)est;
}

/* ------------------------------------------------------------------ */
/* step a-1: NaN-safe routing                                          */
/* ------------------------------------------------------------------ */

/* NaN -> -FLT_MAX (PR #39593, "Fix"); +-Inf -> +-FLT_MAX (reading). */
static float sanitize(float v) {
  if (isnan(v)) return -FLT_MAX;
  if (isinf(v)) return v > 0 ? FLT_MAX : -FLT_MAX;
  return v;
}

typedef struct {
  float v;
  int idx;
} scored_t;

/* value descending, then index ascending: a strict total order, so the
 * library sort's instability does not matter. */
static int cmp_scored(const void* pa, const void* pb) {
  const scored_t* a = (const scored_t*)pa;
  const scored_t* b = (const scored_t*)pb;
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
  return (a->idx > b->idx) - (a->idx < b->idx);
}

/* Route one token: logits row l[E] (fp32 values) -> k ids and k weights.
 * scoring 0 = softmax over all E, 1 = sigmoid per logit; renorm != 0
 * rescales the k picked scores to sum to one. */
static void route_row(const float* l_in, int E, int k, int scoring, int renorm,
                      int32_t* ids, double* w, scored_t* scratch) {
  for (int e = 0; e < E; ++e) {
    scratch[e].v = sanitize(l_in[e]);
    scratch[e].idx = e;
  }
  /* the sort is over the sanitised logits, not over the probabilities */
  qsort(scratch, (size_t)E, sizeof(scored_t), cmp_scored);
  for (int j = 0; j < k; ++j) ids[j] = scratch[j].idx;

  double picked[1024];
  if (scoring == 0) {
    double m = -INFINITY;
    for (int e = 0; e < E; ++e) m = fmax(m, (double)sanitize(l_in[e]));
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += exp((double)sanitize(l_in[e]) - m);
    for (int j = 0; j < k; ++j) picked[j] = exp((double)sanitize(l_in[ids[j]]) - m) / z;
  } else {
    for (int j = 0; j < k; ++j)
      picked[j] = 1.0 / (1.0 + exp(-(double)sanitize(l_in[ids[j]])));
  }
  if (renorm) {
    double den = 0.0;
    for (int j = 0; j < k; ++j) den += picked[j];
    for (int j = 0; j < k; ++j)
      w[j] = (den > 0.0 && isfinite(den)) ? picked[j] / den : 1.0 / (double)k;
  } else {
    for (int j = 0; j < k; ++j) w[j] = picked[j];
  }
}

/* Group-limited routing (PR #39593 "Test Plan" names a grouped top-k
 * whose NaN rows must also give distinct experts; the pages do not define
 * it -- reading): the E experts form n_group contiguous groups of E/n_group;
 * a group's score is its largest sanitised logit; the topk_group best groups
 * (ties to the lower group index) are kept, and top-k runs over the experts
 * of the kept groups only.  Weights as route_row (softmax over all E).
 * Only the kept groups' experts enter the final sort. */
static void route_row_grouped(const float* l_in, int E, int k, int n_group, int topk_group,
                              int scoring, int renorm, int32_t* ids, double* w,
                              scored_t* scratch) {
  const int gs = E / n_group;
  scored_t groups[1024];
  for (int g = 0; g < n_group; ++g) {
    float m = -INFINITY;
    for (int e = g * gs; e < (g + 1) * gs; ++e) m = fmaxf(m, sanitize(l_in[e]));
    groups[g].v = m;
    groups[g].idx = g;
  }
  qsort(groups, (size_t)n_group, sizeof(scored_t), cmp_scored);
  int keep[1024] = {0};
  for (int i = 0; i < topk_group; ++i) keep[groups[i].idx] = 1;
  int n = 0;
  for (int e = 0; e < E; ++e)
    if (keep[e / gs]) {
      scratch[n].v = sanitize(l_in[e]);
      scratch[n].idx = e;
      ++n;
    }
  qsort(scratch, (size_t)n, sizeof(scored_t), cmp_scored);
  for (int j = 0; j < k; ++j) ids[j] = scratch[j].idx;
  double picked[1024];
  if (scoring == 0) {
    double m = -INFINITY;
    for (int e = 0; e < E; ++e) m = fmax(m, (double)sanitize(l_in[e]));
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += exp((double)sanitize(l_in[e]) - m);
    for (int j = 0; j < k; ++j) picked[j] = exp((double)sanitize(l_in[ids[j]]) - m) / z;
  } else {
    for (int j = 0; j < k; ++j)
      picked[j] = 1.0 / (1.0 + exp(-(double)sanitize(l_in[ids[j]])));
  }
  double den = 0.0;
  for (int j = 0; j < k; ++j) den += picked[j];
  for (int j = 0; j < k; ++j)
    w[j] = renorm ? ((den > 0.0 && isfinite(den)) ? picked[j] / den : 1.0 / (double)k)
                  : picked[j];
}

/* Grouped routing of T tokens; requires n_group | E, 1 <= topk_group <=
 * n_group and k <= topk_group * E / n_group.  Returns 0 or -1. */
int oracle_route_grouped(const float* logits, int T, int E, int k, int n_group, int topk_group,
                         int scoring, int renorm, int32_t* ids, double* w) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || n_group < 1 || E % n_group != 0 ||
      topk_group < 1 || topk_group > n_group || k > topk_group * (E / n_group))
    return -1;
  scored_t* scratch = (scored_t*)malloc(sizeof(scored_t) * (size_t)E);
  if (!scratch) return -1;
  for (int t = 0; t < T; ++t)
    route_row_grouped(logits + (size_t)t * E, E, k, n_group, topk_group, scoring, renorm,
                      ids + (size_t)t * k, w + (size_t)t * k, scratch);
  free(scratch);
  return 0;
}

/* Route T tokens.  logits [T, E] fp32 values (bf16 logits are widened
 * exactly by the caller).  ids [T, k], w [T, k].  Returns 0, or -1 on bad
 * sizes (k must be in [1, E], E <= 1024). */
int oracle_route(const float* logits, int T, int E, int k, int scoring, int renorm,
                 int32_t* ids, double* w) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E) return -1;
  scored_t* scratch = (scored_t*)malloc(sizeof(scored_t) * (size_t)E);
  if (!scratch) return -1;
  for (int t = 0; t < T; ++t)
    route_row(logits + (size_t)t * E, E, k, scoring, renorm, ids + (size_t)t * k,
              w + (size_t)t * k, scratch);
  free(scratch);
  return 0;
}

/* ------------------------------------------------------------------ */
/* step a-2: count and permute rows by expert                          */
/* ------------------------------------------------------------------ */

static const int32_t* g_sort_ids; /* key array for cmp_flat (single-threaded) */

static int cmp_flat(const void* pa, const void* pb) {
  int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  int32_t ea = g_sort_ids[a], eb = g_sort_ids[b];
  if (ea != eb) return (ea > eb) - (ea < eb);
  return (a > b) - (a < b);
}

/* ids [R] (R = T*k flat picks, f = t*k + j) -> counts [E], offsets [E+1]
 * (exclusive scan), src [R] (sorted position -> flat index, ordered by
 * expert then by flat index) and pos [R] (flat index -> sorted position,
 * the inverse of src).  Returns -1 if an id is outside [0, E). */
int oracle_permute(const int32_t* ids, int R, int E, int32_t* counts, int32_t* offsets,
                   int32_t* src, int32_t* pos) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int f = 0; f < R; ++f) {
    if (ids[f] < 0 || ids[f] >= E) return -1;
    counts[ids[f]]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  for (int f = 0; f < R; ++f) src[f] = f;
  g_sort_ids = ids;
  qsort(src, (size_t)R, sizeof(int32_t), cmp_flat);
  g_sort_ids = NULL;
  for (int p = 0; p < R; ++p) pos[src[p]] = p;
  return 0;
}

/* ------------------------------------------------------------------ */
/* steps a-4 .. a-7: expert MLPs and the weighted combine              */
/* ------------------------------------------------------------------ */

typedef struct {
  int H, I, dtype;
  const void* w13;
  const float* s13;
  const void* w2;
  const float* s2;
  float e4m3_table[256];
} weights_t;

/* dequantised w13[e][r][h], layout [E, 2I, H]; FP8 block scale
 * s13[e][r/128][h/128], layout [E, 2I/128, H/128] */
static double w13_at(const weights_t* W, int e, int r, int h) {
  size_t i = ((size_t)e * 2 * W->I + r) * W->H + h;
  if (W->dtype == ORACLE_DTYPE_F32) return ((const float*)W->w13)[i];
  if (W->dtype == ORACLE_DTYPE_BF16) return oracle_bf16_to_f32(((const uint16_t*)W->w13)[i]);
  size_t si = ((size_t)e * (2 * W->I / 128) + r / 128) * (W->H / 128) + h / 128;
  return (double)W->e4m3_table[((const uint8_t*)W->w13)[i]] * (double)W->s13[si];
}

/* dequantised w2[e][h][c], layout [E, H, I]; scale s2[e][h/128][c/128] */
static double w2_at(const weights_t* W, int e, int h, int c) {
  size_t i = ((size_t)e * W->H + h) * W->I + c;
  if (W->dtype == ORACLE_DTYPE_F32) return ((const float*)W->w2)[i];
  if (W->dtype == ORACLE_DTYPE_BF16) return oracle_bf16_to_f32(((const uint16_t*)W->w2)[i]);
  size_t si = ((size_t)e * (W->H / 128) + h / 128) * (W->I / 128) + c / 128;
  return (double)W->e4m3_table[((const uint8_t*)W->w2)[i]] * (double)W->s2[si];
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* Quantise a row to FP8 per 128-column group and give back its dequantised
 * value (code value times group scale). */
static void fake_quant_row(const float* v, int n, double* out, uint8_t* codes, float* scales,
                           const float* table) {
  oracle_quant_group128(v, n, codes, scales);
  for (int i = 0; i < n; ++i) out[i] = (double)table[codes[i]] * (double)scales[i / 128];
}

/*
 * The fused MoE layer forward for a list of tokens.
 * n_group > 1 selects group-limited routing (route_row_grouped).
 * Expert parallelism (H20 article, para. 2: the fused-MoE API takes the
 * expert-parallel size and rank): with ep_size > 1 the weights hold only
 * the E / ep_size experts of rank ep_rank (global ids ep_rank*E/ep_size ..
 * +E/ep_size - 1); routing still ranks all E experts, and picks outside the
 * local range contribute nothing, so out is this rank's partial sum.
 *   dtype 0: x [T,H] f32, logits [T,E] f32, w13 [E,2I,H] f32, w2 [E,H,I] f32
 *   dtype 1: x, logits, w13, w2 as bf16 bit patterns (uint16)
 *   dtype 2: x, logits bf16; w13, w2 e4m3 codes with fp32 block scales
 *            s13 [E,2I/128,H/128], s2 [E,H/128,I/128]; activations quantised
 *            per token and 128-column group (x over H, act over I)
 * tokens: n_tokens token indices to compute (NULL: all T, in order).
 * out [n_tokens, H] (double), ids_out [n_tokens, k], w_out [n_tokens, k]
 * (either may be NULL).  Returns 0, or -1 on unsupported sizes.
 */
int oracle_moe_forward(int T, int H, int I, int E, int k, int dtype, int scoring, int renorm,
                       int n_group, int topk_group,
                       int ep_size, int ep_rank, const void* x, const void* logits,
                       const void* w13, const float* s13, const void* w2, const float* s2,
                       const int32_t* tokens, int n_tokens, double* out, int32_t* ids_out,
                       double* w_out) {
  if (T < 0 || H < 1 || I < 1 || E < 1 || E > 1024 || k < 1 || k > E) return -1;
  if (ep_size < 1 || E % ep_size != 0 || ep_rank < 0 || ep_rank >= ep_size) return -1;
  if (n_group < 1 || E % n_group != 0 || topk_group < 1 || topk_group > n_group ||
      k > topk_group * (E / n_group))
    return -1;
  const int e_local = E / ep_size, e_base = ep_rank * e_local;
  if (dtype == ORACLE_DTYPE_FP8 && (H % 128 != 0 || I % 128 != 0)) return -1;
  if (!tokens) n_tokens = T;

  weights_t W;
  W.H = H;
  W.I = I;
  W.dtype = dtype;
  W.w13 = w13;
  W.s13 = s13;
  W.w2 = w2;
  W.s2 = s2;
  for (int c = 0; c < 256; ++c) W.e4m3_table[c] = oracle_e4m3_decode((uint8_t)c);

  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int n = 0; n < n_tokens; ++n) {
    int t = tokens ? tokens[n] : n;
    if (t < 0 || t >= T) {
      bad = 1;
      continue;
    }
    float* lrow = (float*)malloc(sizeof(float) * (size_t)E);
    float* xf = (float*)malloc(sizeof(float) * (size_t)H);
    double* xd = (double*)malloc(sizeof(double) * (size_t)H);
    float* af = (float*)malloc(sizeof(float) * (size_t)I);
    double* ad = (double*)malloc(sizeof(double) * (size_t)I);
    uint8_t* codes = (uint8_t*)malloc((size_t)(H > I ? H : I));
    float* scales = (float*)malloc(sizeof(float) * (size_t)((H > I ? H : I) / 128 + 1));
    scored_t* scratch = (scored_t*)malloc(sizeof(scored_t) * (size_t)E);
    int32_t ids[1024];
    double w[1024];
    double* orow = out + (size_t)n * H;

    /* a-1: route this token */
    for (int e = 0; e < E; ++e) {
      size_t i = (size_t)t * E + e;
      lrow[e] = dtype == ORACLE_DTYPE_F32 ? ((const float*)logits)[i]
                                          : oracle_bf16_to_f32(((const uint16_t*)logits)[i]);
    }
    if (n_group > 1)
      route_row_grouped(lrow, E, k, n_group, topk_group, scoring, renorm, ids, w, scratch);
    else
      route_row(lrow, E, k, scoring, renorm, ids, w, scratch);
    if (ids_out)
      for (int j = 0; j < k; ++j) ids_out[(size_t)n * k + j] = ids[j];
    if (w_out)
      for (int j = 0; j < k; ++j) w_out[(size_t)n * k + j] = w[j];

    /* the token's activation row, dequantised (FP8: quantised first) */
    for (int h = 0; h < H; ++h) {
      size_t i = (size_t)t * H + h;
      xf[h] = dtype == ORACLE_DTYPE_F32 ? ((const float*)x)[i]
                                        : oracle_bf16_to_f32(((const uint16_t*)x)[i]);
    }
    if (dtype == ORACLE_DTYPE_FP8)
      fake_quant_row(xf, H, xd, codes, scales, W.e4m3_table);
    else
      for (int h = 0; h < H; ++h) xd[h] = xf[h];

    for (int h = 0; h < H; ++h) orow[h] = 0.0;
    for (int j = 0; j < k; ++j) {
      int e = ids[j] - e_base; /* index into this rank's weights */
      if (e < 0 || e >= e_local) continue; /* another rank's expert */
      /* a-4, a-5: gate and up projections, SiLU(gate) * up */
      for (int c = 0; c < I; ++c) {
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
          g += xd[h] * w13_at(&W, e, c, h);
          u += xd[h] * w13_at(&W, e, I + c, h);
        }
        ad[c] = silu(g) * u;
      }
      if (dtype == ORACLE_DTYPE_FP8) {
        for (int c = 0; c < I; ++c) af[c] = (float)ad[c];
        fake_quant_row(af, I, ad, codes, scales, W.e4m3_table);
      }
      /* a-6, a-7: down projection, weighted into the token's output */
      for (int h = 0; h < H; ++h) {
        double y = 0.0;
        for (int c = 0; c < I; ++c) y += ad[c] * w2_at(&W, e, h, c);
        orow[h] += w[j] * y;
      }
    }
    free(lrow);
    free(xf);
    free(xd);
    free(af);
    free(ad);
    free(codes);
    free(scales);
    free(scratch);
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* threads                                                             */
/* ------------------------------------------------------------------ */

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
