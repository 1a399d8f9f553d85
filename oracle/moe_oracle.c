/*
 * moe_oracle.c -- plain, slow, CPU oracle of the BF16 Mixture-of-Experts
 * expert block (router -> permute -> grouped gate/up GEMM + SiLU-mul ->
 * grouped down GEMM -> weighted top-k combine / shared-expert gate).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load this library.  The GPU product path
 * never calls it, and the two share no source, header, table or helper.
 *
 * Arithmetic rules (the numeric contract stated in vllm.cpp issue #3094,
 * "Row: BACKEND-ROCM-BF16-MOE", second paragraph, and the bit-exactness rules
 * of vllm.cpp PR #509 "MoE combine/gate ops -- SharedExpertGate, MoeCombine,
 * MoeCombineGate", review rework commit, item 2):
 *   - all math is IEEE-754 binary32, one rounded operation at a time; this
 *     file must be compiled with -ffp-contract=off and without fast-math, so
 *     that no multiply-add is fused and no sum is re-associated;
 *   - bf16 -> f32 widening is exact; f32 -> bf16 narrowing is round to
 *     nearest, ties to even, on the f32 bit pattern (NaN stays NaN);
 *   - every dot product is a sequential sum over the contraction index,
 *     starting from +0.0f, of exact bf16*bf16 products.
 *
 * Readings where the pages are silent are marked READING below.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORA_OK 0
#define ORA_ERR_ARG (-1)
#define ORA_ERR_DTYPE (-2)
#define ORA_ERR_UNSUPPORTED (-3)

#define ORA_F32 0
#define ORA_BF16 1
#define ORA_F16 2

int oracle_abi_version(void) { return 3; }

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* bf16 <-> f32                                                        */
/* ------------------------------------------------------------------ */

static float bf2f(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round to nearest, ties to even, written as the definition: keep the upper
 * half, look at the discarded lower half, round up when it is above one half
 * or exactly one half with an odd kept part.  A carry out of the mantissa
 * moves into the exponent, which is exactly the correct rounding up to the
 * next binade or to infinity.  READING: a NaN stays a NaN (quiet bit set,
 * sign kept); the pages only say that the shared term passes through bf16. */
static uint16_t f2bf(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
    return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t kept = u >> 16;
  uint32_t dropped = u & 0xFFFFu;
  if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;
  return (uint16_t)kept;
}

/* round-trip through bf16: the double rounding of MoeCombineGate's shared term */
static float bf16_round(float f) { return bf2f(f2bf(f)); }

float oracle_bf16_to_f32(uint16_t h) { return bf2f(h); }
uint16_t oracle_f32_to_bf16(float f) { return f2bf(f); }

void oracle_f32_to_bf16_array(const float* src, uint16_t* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i) dst[i] = f2bf(src[i]);
}

/* ------------------------------------------------------------------ */
/* exp and sigmoid                                                      */
/* ------------------------------------------------------------------ */

/* READING: the pages require the sigmoid gate and the combine-gate to be
 * bit-identical across CPU and GPU (PR #509 review and rework commits)
 * but never say which exp.  The exp used there is therefore DEFINED as the
 * binary32 rounding of one fixed double-precision evaluation:
 *   Cody & Waite (1980) argument reduction  x = n*ln2 + r,  |r| <= ln2/2,
 *   with ln2 split in a 32-bit head (n*head is exact for |n| < 2^21) and a
 *   double tail; exp(r) by its Taylor series through r^13 (truncation error
 *   < 4e-18 relative) in Horner form; exact scaling by 2^n; one final
 *   rounding to binary32.
 * Every step is a single IEEE double operation, so any conforming machine
 * that performs the same steps gets the same bits.  The result is within a
 * few double ulps of exp(x), far inside half a binary32 ulp. */
static const double EXP_LOG2E = 0x1.71547652b82fep+0;
static const double EXP_LN2_HEAD = 0x1.62e42fee00000p-1;
static const double EXP_LN2_TAIL = 0x1.a39ef35793c76p-33;
static const double EXP_TAYLOR[14] = {
    /* 1/k!, k = 0..13 */
    0x1.0000000000000p+0, 0x1.0000000000000p+0, 0x1.0000000000000p-1,
    0x1.5555555555555p-3, 0x1.5555555555555p-5, 0x1.1111111111111p-7,
    0x1.6c16c16c16c17p-10, 0x1.a01a01a01a01ap-13, 0x1.a01a01a01a01ap-16,
    0x1.71de3a556c734p-19, 0x1.27e4fb7789f5cp-22, 0x1.ae64567f544e4p-26,
    0x1.1eed8eff8d898p-29, 0x1.6124613a86d09p-33};

float oracle_exp_f32(float x) {
  if (x != x) return x;                      /* NaN */
  if (x > 89.0f) return (float)INFINITY;     /* exp(89) > FLT_MAX */
  if (x < -104.0f) return 0.0f;              /* exp(-104) < 2^-150 */
  double xd = (double)x;
  double n = nearbyint(xd * EXP_LOG2E);      /* ties to even */
  double r = xd - n * EXP_LN2_HEAD;
  r = r - n * EXP_LN2_TAIL;
  double p = EXP_TAYLOR[13];
  for (int k = 12; k >= 0; --k) {
    p = p * r;
    p = p + EXP_TAYLOR[k];
  }
  double y = ldexp(p, (int)n);               /* exact: p*2^n stays normal */
  return (float)y;                           /* the one binary32 rounding */
}

void oracle_exp_f32_array(const float* x, float* y, int64_t n) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_exp_f32(x[i]);
}

/* sigma(g) = 1 / (1 + exp(-g)), two binary32 operations after the exp. */
float oracle_sigmoid_f32(float g) {
  float e = oracle_exp_f32(-g);
  float d = 1.0f + e;
  return 1.0f / d;
}

/* ------------------------------------------------------------------ */
/* dtype-generic element access (f32 and bf16 arms; f16 is refused)    */
/* ------------------------------------------------------------------ */

static float ld(const void* p, int dt, int64_t i) {
  return dt == ORA_F32 ? ((const float*)p)[i] : bf2f(((const uint16_t*)p)[i]);
}

static void st(void* p, int dt, int64_t i, float v) {
  if (dt == ORA_F32)
    ((float*)p)[i] = v;
  else
    ((uint16_t*)p)[i] = f2bf(v);
}

static int dtype_ok(int dt) { return dt == ORA_F32 || dt == ORA_BF16; }

/* sequential f32 dot product of two bf16 vectors (each product is exact) */
static float dot_bf16(const uint16_t* a, const uint16_t* b, int n) {
  float acc = 0.0f;
  for (int i = 0; i < n; ++i) {
    float prod = bf2f(a[i]) * bf2f(b[i]);
    acc = acc + prod;
  }
  return acc;
}

/* ------------------------------------------------------------------ */
/* a1 + a2: ungrouped softmax router, top-k, renormalise                */
/* PR #509 "Honest gaps": only the ungrouped softmax router is in scope;  */
/* grouped / bias-corrected (noaux_tc) forms are refused.                */
/* ------------------------------------------------------------------ */

/* READING: ranking order is descending logit; equal logits (including
 * -0 == +0) go to the lower expert index; NaN ranks below every number. */
static int ranks_above(float a, int ia, float b, int ib) {
  int na = (a != a), nb = (b != b);
  if (na && nb) return ia < ib;
  if (na) return 0;
  if (nb) return 1;
  if (a > b) return 1;
  if (a < b) return 0;
  return ia < ib;
}

/* Select the K best of one row of E logits (rank order) and compute the
 * weights.  READING: selection is on logits (softmax is monotone); with
 * renormalisation the full-softmax denominator cancels, so the weights are
 * the K selected exponentials divided by their own sequential sum. */
static void topk_row(const float* l, int E, int K, int renormalize, int32_t* ids,
                     float* w) {
  int32_t chosen[32] = {0};
  for (int j = 0; j < K; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      int taken = 0;
      for (int q = 0; q < j; ++q)
        if (chosen[q] == e) taken = 1;
      if (taken) continue;
      if (best < 0 || ranks_above(l[e], e, l[best], best)) best = e;
    }
    chosen[j] = best;
    ids[j] = best;
  }
  float m = l[chosen[0]];
  float ex[32];
  for (int j = 0; j < K; ++j) ex[j] = oracle_exp_f32(l[chosen[j]] - m);
  float den = 0.0f;
  if (renormalize) {
    for (int j = 0; j < K; ++j) den = den + ex[j];
  } else {
    for (int e = 0; e < E; ++e) den = den + oracle_exp_f32(l[e] - m);
  }
  for (int j = 0; j < K; ++j) w[j] = ex[j] / den;
}

int oracle_route_topk(const uint16_t* x, const uint16_t* w_router, const float* logit_bias,
                      const uint16_t* w_shared_gate, const float* logits_in, int T, int H,
                      int E, int K, int renormalize, int scoring, int n_group,
                      int32_t* topk_ids, float* topk_w, float* logits_out,
                      float* gate_logit_out) {
  if (scoring != 0 || n_group != 1) return ORA_ERR_UNSUPPORTED;
  if (T < 0 || H <= 0 || E <= 0 || K < 1 || K > E || K > 32) return ORA_ERR_ARG;
  if (!logits_in && (!x || !w_router)) return ORA_ERR_ARG;
  if (w_shared_gate && (!x || !gate_logit_out)) return ORA_ERR_ARG;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    float* row = (float*)malloc(sizeof(float) * (size_t)E);
    for (int e = 0; e < E; ++e) {
      float v;
      if (logits_in) {
        v = logits_in[(int64_t)t * E + e];
      } else {
        v = dot_bf16(x + (int64_t)t * H, w_router + (int64_t)e * H, H);
        if (logit_bias) v = v + logit_bias[e];
      }
      row[e] = v;
      if (logits_out) logits_out[(int64_t)t * E + e] = v;
    }
    topk_row(row, E, K, renormalize, topk_ids + (int64_t)t * K, topk_w + (int64_t)t * K);
    if (w_shared_gate) gate_logit_out[t] = dot_bf16(x + (int64_t)t * H, w_shared_gate, H);
    free(row);
  }
  return ORA_OK;
}

/* ------------------------------------------------------------------ */
/* Router forms the pages name as open gaps (issue #3094 leaves the grouped */
/* and sigmoid routers of DeepSeek-V2 and Dots3 to separate work; PR #509    */
/* "Honest gaps" says its grouped / bias / noaux_tc forms still throw).  The */
/* pages do not define them; READING, after the published DeepSeek-V2 and    */
/* DeepSeek-V3 routers:                                                      */
/*   scores   softmax (scoring 0): selection on the logits, weights as in    */
/*            topk_row; sigmoid (scoring 1): s_e = sigmoid(l_e), the same    */
/*            sigmoid as the shared-expert gate                              */
/*   keys     k_e = s_e + select_bias[e] (sigmoid only; the bias steers the  */
/*            choice, never the weights), else the scores (logits for softmax)*/
/*   groups   E experts in n_group contiguous groups of E / n_group; a       */
/*            group's score is its largest key (group_score 0) or its two    */
/*            largest keys added, largest first (group_score 1); the          */
/*            topk_group best groups (descending, ties to the lower group,   */
/*            NaN last) stay eligible                                        */
/*   choice   the K best keys among eligible experts (descending, ties to     */
/*            the lower id, NaN last)                                        */
/*   weights  sigmoid: w_j = s_j / ((s_0 + s_1) + ... + s_{K-1}) from +0      */
/*            (renormalize 1) or s_j (renormalize 0); softmax: as topk_row    */
/* ------------------------------------------------------------------ */

/* the k-th best (k = 0, 1) key of experts [e0, e1) in ranks_above order */
static float group_score(const float* key, int e0, int e1, int mode) {
  int b0 = -1, b1 = -1;
  for (int e = e0; e < e1; ++e) {
    if (b0 < 0 || ranks_above(key[e], e, key[b0], b0)) {
      b1 = b0;
      b0 = e;
    } else if (b1 < 0 || ranks_above(key[e], e, key[b1], b1)) {
      b1 = e;
    }
  }
  if (mode == 0) return key[b0];
  return key[b0] + key[b1];
}

static void topk_row_ex(const float* l, const float* select_bias, int E, int K, int renormalize,
                        int scoring, int n_group, int topk_group, int gmode, int32_t* ids,
                        float* w) {
  float* key = (float*)malloc(sizeof(float) * (size_t)E);
  float* sc = (float*)malloc(sizeof(float) * (size_t)E);
  unsigned char* ok = (unsigned char*)calloc((size_t)E, 1);
  for (int e = 0; e < E; ++e) {
    sc[e] = scoring == 1 ? oracle_sigmoid_f32(l[e]) : l[e];
    key[e] = select_bias ? sc[e] + select_bias[e] : sc[e];
  }
  /* eligible groups: the topk_group best by group score */
  const int gs = E / n_group;
  float gsc[1024];
  int gchosen[1024];
  for (int g = 0; g < n_group; ++g) gsc[g] = group_score(key, g * gs, g * gs + gs, gmode);
  for (int j = 0; j < topk_group; ++j) {
    int best = -1;
    for (int g = 0; g < n_group; ++g) {
      int taken = 0;
      for (int q = 0; q < j; ++q)
        if (gchosen[q] == g) taken = 1;
      if (taken) continue;
      if (best < 0 || ranks_above(gsc[g], g, gsc[best], best)) best = g;
    }
    gchosen[j] = best;
    for (int e = best * gs; e < best * gs + gs; ++e) ok[e] = 1;
  }
  /* the K best eligible experts */
  int32_t chosen[32] = {0};
  for (int j = 0; j < K; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (!ok[e]) continue;
      int taken = 0;
      for (int q = 0; q < j; ++q)
        if (chosen[q] == e) taken = 1;
      if (taken) continue;
      if (best < 0 || ranks_above(key[e], e, key[best], best)) best = e;
    }
    chosen[j] = best;
    ids[j] = best;
  }
  if (scoring == 1) {
    float den = 0.0f;
    for (int j = 0; j < K; ++j) den = den + sc[chosen[j]];
    for (int j = 0; j < K; ++j) w[j] = renormalize ? sc[chosen[j]] / den : sc[chosen[j]];
  } else {
    float m = l[chosen[0]];
    float ex[32];
    for (int j = 0; j < K; ++j) ex[j] = oracle_exp_f32(l[chosen[j]] - m);
    float den = 0.0f;
    if (renormalize) {
      for (int j = 0; j < K; ++j) den = den + ex[j];
    } else {
      for (int e = 0; e < E; ++e) den = den + oracle_exp_f32(l[e] - m);
    }
    for (int j = 0; j < K; ++j) w[j] = ex[j] / den;
  }
  free(key);
  free(sc);
  free(ok);
}

/* the extended router on given logits (the GEMM part is oracle_route_topk's) */
int oracle_route_topk_ex(const float* logits, const float* select_bias, int T, int E, int K,
                         int renormalize, int scoring, int n_group, int topk_group,
                         int group_score_mode, int32_t* topk_ids, float* topk_w) {
  if (T < 0 || E <= 0 || E > 1024 || K < 1 || K > 32) return ORA_ERR_ARG;
  if (scoring != 0 && scoring != 1) return ORA_ERR_UNSUPPORTED;
  if (select_bias && scoring != 1) return ORA_ERR_UNSUPPORTED;
  if (n_group < 1 || E % n_group != 0 || topk_group < 1 || topk_group > n_group)
    return ORA_ERR_ARG;
  if (group_score_mode != 0 && group_score_mode != 1) return ORA_ERR_ARG;
  if (group_score_mode == 1 && E / n_group < 2) return ORA_ERR_ARG;
  if (K > topk_group * (E / n_group)) return ORA_ERR_ARG;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    topk_row_ex(logits + (int64_t)t * E, select_bias, E, K, renormalize, scoring, n_group,
                topk_group, group_score_mode, topk_ids + (int64_t)t * K, topk_w + (int64_t)t * K);
  return ORA_OK;
}

/* ------------------------------------------------------------------ */
/* a3: permute into expert-contiguous order (stable counting sort)      */
/* The pages' expert path keeps P = T*K permuted bf16 rows of H (PR #509  */
/* review, finding 2) and groups them over                                */
/* expert ids (PR #523 "What changed").  READING: rows of one expert keep */
/* ascending pair order p = t*K + j.                                     */
/* ------------------------------------------------------------------ */

int oracle_permute(const int32_t* topk_ids, const uint16_t* x, int T, int K, int E, int H,
                   int32_t* expert_offsets, int32_t* sorted_pair, int32_t* pair_to_row,
                   uint16_t* x_perm) {
  if (T < 0 || K < 1 || E <= 0 || (x_perm && (!x || H <= 0))) return ORA_ERR_ARG;
  int64_t P = (int64_t)T * K;
  int64_t* cnt = (int64_t*)calloc((size_t)E, sizeof(int64_t));
  int64_t* seen = (int64_t*)calloc((size_t)E, sizeof(int64_t));
  for (int64_t p = 0; p < P; ++p) {
    int32_t e = topk_ids[p];
    if (e < 0 || e >= E) {
      free(cnt);
      free(seen);
      return ORA_ERR_ARG;
    }
    cnt[e] += 1;
  }
  expert_offsets[0] = 0;
  for (int e = 0; e < E; ++e) expert_offsets[e + 1] = (int32_t)(expert_offsets[e] + cnt[e]);
  for (int64_t p = 0; p < P; ++p) {
    int32_t e = topk_ids[p];
    int64_t row = expert_offsets[e] + seen[e];
    seen[e] += 1;
    sorted_pair[row] = (int32_t)p;
    pair_to_row[p] = (int32_t)row;
    if (x_perm) memcpy(x_perm + row * H, x + (p / K) * H, sizeof(uint16_t) * (size_t)H);
  }
  free(cnt);
  free(seen);
  return ORA_OK;
}

/* ------------------------------------------------------------------ */
/* Block-scaled FP8 expert weights (the pages only name                 */
/* kMatmulFp8BlockScaled and kQuantFp8Group as ops of the engine).      */
/* READING, after the published DeepSeek-V3 FP8 weights: each expert's  */
/* weight matrix is stored as FP8 E4M3 codes (the "fn" variant: no      */
/* infinities, S.1111.111 is NaN, largest finite 448) with one f32      */
/* scale per 128 x 128 block of its own rows and columns.  The expert   */
/* GEMMs use w = bf16(f32(code) * scale), one f32 multiply and one RNE  */
/* rounding to bf16, and then the bf16 contract above; activations stay */
/* bf16.                                                                */
/* ------------------------------------------------------------------ */

float oracle_e4m3_to_f32(uint8_t b) {
  const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
  float v;
  if (e == 15 && m == 7) return sign ? -NAN : NAN;
  if (e == 0)
    v = ldexpf((float)m, -9);           /* subnormal: m/8 * 2^-6 */
  else
    v = ldexpf((float)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
  return sign ? -v : v;
}

/* w[g, r, c] = bf16(f32(q[g, r, c]) * scale[g, r / 128, c / 128]) for G matrices
 * of R x C; scale is [G][ceil(R/128)][ceil(C/128)] */
int oracle_dequant_fp8_block(const uint8_t* q, const float* scale, int G, int R, int C,
                             uint16_t* w) {
  if (G < 1 || R < 1 || C < 1 || !q || !scale || !w) return ORA_ERR_ARG;
  const int64_t rb = (R + 127) / 128, cb = (C + 127) / 128;
#pragma omp parallel for schedule(static)
  for (int64_t gr = 0; gr < (int64_t)G * R; ++gr) {
    const int64_t g = gr / R, r = gr % R;
    const float* srow = scale + (g * rb + r / 128) * cb;
    for (int64_t c = 0; c < C; ++c) {
      float v = oracle_e4m3_to_f32(q[gr * C + c]) * srow[c / 128];
      w[gr * C + c] = f2bf(v);
    }
  }
  return ORA_OK;
}

/* ------------------------------------------------------------------ */
/* a4: grouped gate/up GEMM fused with SiLU-and-mul                     */
/* kMoeGroupedGemmBf16GateUpSilu, issue #3094: the GEMM result is cut to  */
/* bf16 ahead of the activation -- both the gate and the up accumulations */
/* are rounded to bf16 before silu(g)*u.  READING: per expert the weight is */
/* [2I, H] with the gate rows first and the up rows after them.          */
/* ------------------------------------------------------------------ */

static float silu_f32(float z) {
  float e = expf(z * -1.0f); /* tolerance-checked only: any exp will do */
  float d = 1.0f + e;
  return z / d;
}

/* one output row; narrow = 0 is a planted mutation used only by tests */
static void gateup_row(const uint16_t* a_row, const uint16_t* w13_g, int H, int I,
                       uint16_t* act_row, int narrow) {
  for (int n = 0; n < I; ++n) {
    float g = dot_bf16(a_row, w13_g + (int64_t)n * H, H);
    float u = dot_bf16(a_row, w13_g + (int64_t)(I + n) * H, H);
    if (narrow) {
      g = bf16_round(g);
      u = bf16_round(u);
    }
    float s = silu_f32(g);
    float v = s * u;
    act_row[n] = f2bf(v);
  }
}

static int group_of_row(const int32_t* off, int G, int64_t r) {
  int lo = 0, hi = G; /* find g with off[g] <= r < off[g+1] */
  if (r < off[0] || r >= off[G]) return -1;
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (off[mid] <= r)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

static int offsets_ok(const int32_t* off, int G, int P) {
  if (!off) return 1;
  if (off[0] < 0) return 0;
  for (int g = 0; g < G; ++g)
    if (off[g + 1] < off[g]) return 0;
  return off[G] <= P;
}

int oracle_gateup_silu(const uint16_t* a, const int32_t* a_row_gather, const uint16_t* w13,
                       const int32_t* group_offsets, int P, int H, int I, int G,
                       const int32_t* rows, int n_rows, uint16_t* act, int narrow) {
  if (P < 0 || H <= 0 || I <= 0 || G <= 0) return ORA_ERR_ARG;
  if (!group_offsets && G != 1) return ORA_ERR_ARG;
  if (!offsets_ok(group_offsets, G, P)) return ORA_ERR_ARG;
  int32_t single[2] = {0, P};
  const int32_t* off = group_offsets ? group_offsets : single;
  int64_t n = rows ? n_rows : (int64_t)off[G] - off[0];
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n; ++i) {
    int64_t r = rows ? rows[i] : off[0] + i;
    int g = group_of_row(off, G, r);
    if (g < 0) continue;
    int64_t src = a_row_gather ? a_row_gather[r] : r;
    gateup_row(a + src * H, w13 + (int64_t)g * 2 * I * H, H, I, act + r * I, narrow);
  }
  return ORA_OK;
}

/* ------------------------------------------------------------------ */
/* a5: grouped down GEMM, routing weight applied once before the store   */
/* kMoeGroupedGemmBf16, issue #3094: the routing weight belongs to the    */
/* down projection, ahead of its store, and the later reduction must not  */
/* apply it a second time.  READING: y = sum_i act*W2 in f32, one f32     */
/* multiply by the pair's weight, one bf16 rounding; the row goes to the  */
/* pair order ([T, K, H]) when row_to_pair is given.                     */
/* ------------------------------------------------------------------ */

static void down_row(const uint16_t* act_row, const uint16_t* w2_g, int I, int H,
                     const float* weight, uint16_t* out_row) {
  for (int n = 0; n < H; ++n) {
    float y = dot_bf16(act_row, w2_g + (int64_t)n * I, I);
    if (weight) y = y * (*weight);
    out_row[n] = f2bf(y);
  }
}

int oracle_down(const uint16_t* act, const uint16_t* w2, const int32_t* group_offsets,
                const float* pair_weight, const int32_t* row_to_pair, int P, int I, int H,
                int G, const int32_t* rows, int n_rows, uint16_t* out) {
  if (P < 0 || H <= 0 || I <= 0 || G <= 0) return ORA_ERR_ARG;
  if (!group_offsets && G != 1) return ORA_ERR_ARG;
  if (!offsets_ok(group_offsets, G, P)) return ORA_ERR_ARG;
  int32_t single[2] = {0, P};
  const int32_t* off = group_offsets ? group_offsets : single;
  int64_t n = rows ? n_rows : (int64_t)off[G] - off[0];
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n; ++i) {
    int64_t r = rows ? rows[i] : off[0] + i;
    int g = group_of_row(off, G, r);
    if (g < 0) continue;
    int64_t dst = row_to_pair ? row_to_pair[r] : r;
    down_row(act + r * I, w2 + (int64_t)g * H * I, I, H, pair_weight ? pair_weight + dst : NULL,
             out + dst * H);
  }
  return ORA_OK;
}

/* ------------------------------------------------------------------ */
/* a7: kMoeCombine                                                       */
/* PR #509 "What changed": weighted top-k expert sum plus an optional     */
/* shared term; review rework item 2: sequential K order, a single store  */
/* rounding, no contraction; routed_scale commit: the f32 scale multiplies */
/* the finished routed sum, then the shared term is added.               */
/* READING: the sum starts from +0.0f; the weight multiply is present     */
/* only when a weight array is given.                                    */
/* ------------------------------------------------------------------ */

int oracle_combine(const void* expert_out, int eo_dtype, const float* w, const void* shared,
                   int sh_dtype, float routed_scale, int T, int K, int H, void* out,
                   int out_dtype) {
  if (!dtype_ok(eo_dtype) || !dtype_ok(out_dtype) || (shared && !dtype_ok(sh_dtype)))
    return ORA_ERR_DTYPE;
  if (T < 0 || K < 1 || H <= 0) return ORA_ERR_ARG;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    for (int c = 0; c < H; ++c) {
      float acc = 0.0f;
      for (int k = 0; k < K; ++k) {
        float v = ld(expert_out, eo_dtype, ((int64_t)t * K + k) * H + c);
        if (w) v = v * w[(int64_t)t * K + k];
        acc = acc + v;
      }
      acc = acc * routed_scale;
      if (shared) acc = acc + ld(shared, sh_dtype, (int64_t)t * H + c);
      st(out, out_dtype, (int64_t)t * H + c, acc);
    }
  }
  return ORA_OK;
}

/* ------------------------------------------------------------------ */
/* a8: kMoeCombineGate                                                   */
/* PR #509 "What changed" + review: combine with the shared-expert sigmoid */
/* gate folded in; the gated shared term is rounded to bf16 and widened   */
/* back before it is added (a double rounding).  READING: routed_scale is */
/* accepted here too and applied to the routed sum before the add.        */
/* ------------------------------------------------------------------ */

int oracle_combine_gate(const void* expert_out, int eo_dtype, const float* w, const void* sd,
                        int sd_dtype, const float* gl, float routed_scale, int T, int K, int H,
                        void* out, int out_dtype) {
  if (!dtype_ok(eo_dtype) || !dtype_ok(sd_dtype) || !dtype_ok(out_dtype)) return ORA_ERR_DTYPE;
  if (T < 0 || K < 1 || H <= 0) return ORA_ERR_ARG;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    float s = oracle_sigmoid_f32(gl[t]);
    for (int c = 0; c < H; ++c) {
      float g = s * ld(sd, sd_dtype, (int64_t)t * H + c);
      float sv = bf16_round(g);
      float acc = 0.0f;
      for (int k = 0; k < K; ++k) {
        float v = ld(expert_out, eo_dtype, ((int64_t)t * K + k) * H + c);
        if (w) v = v * w[(int64_t)t * K + k];
        acc = acc + v;
      }
      acc = acc * routed_scale;
      acc = acc + sv;
      st(out, out_dtype, (int64_t)t * H + c, acc);
    }
  }
  return ORA_OK;
}

/* ------------------------------------------------------------------ */
/* a9: kSharedExpertGate, out[t,c] = sigmoid(gl[t]) * sd[t,c]            */
/* PR #509 "What changed"; f32/bf16 sd, f32/bf16 out (the 4-arm dispatch  */
/* of the review rework), one rounding at the store.                     */
/* ------------------------------------------------------------------ */

int oracle_shared_expert_gate(const void* sd, int sd_dtype, const float* gl, int T, int H,
                              void* out, int out_dtype) {
  if (!dtype_ok(sd_dtype) || !dtype_ok(out_dtype)) return ORA_ERR_DTYPE;
  if (T < 0 || H <= 0) return ORA_ERR_ARG;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    float s = oracle_sigmoid_f32(gl[t]);
    for (int c = 0; c < H; ++c) {
      float v = s * ld(sd, sd_dtype, (int64_t)t * H + c);
      st(out, out_dtype, (int64_t)t * H + c, v);
    }
  }
  return ORA_OK;
}

/* ------------------------------------------------------------------ */
/* The whole expert block for a list of tokens.                          */
/* Each token is routed, each of its K (token, expert) pairs goes through */
/* gate/up + SiLU-mul and the weighted down projection, and the K rows    */
/* are combined with routed_scale; with a shared expert, the shared MLP   */
/* (one group, no routing weight) and its sigmoid gate enter through the  */
/* combine-gate.  A row's arithmetic does not depend on where the permute */
/* puts it, so evaluating token by token gives the same bits as the      */
/* permuted batch.                                                       */
/* ------------------------------------------------------------------ */

int oracle_moe_layer_tokens(const uint16_t* x, const uint16_t* w_router, const float* logit_bias,
                            const uint16_t* w13, const uint16_t* w2,
                            const uint16_t* w_shared_gate, const uint16_t* w13_shared,
                            const uint16_t* w2_shared, int H, int I, int E, int K, int I_shared,
                            float routed_scale, const int32_t* tokens, int n_tokens,
                            int32_t* ids_out, float* w_out, uint16_t* out) {
  if (H <= 0 || I <= 0 || E <= 0 || K < 1 || K > E || K > 32 || n_tokens < 0) return ORA_ERR_ARG;
  int has_shared = (w_shared_gate && w13_shared && w2_shared && I_shared > 0);
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < n_tokens; ++i) {
    const uint16_t* xt = x + (int64_t)tokens[i] * H;
    int32_t ids[32];
    float wts[32];
    float gl = 0.0f;
    oracle_route_topk(xt, w_router, logit_bias, has_shared ? w_shared_gate : NULL, NULL, 1, H, E,
                      K, 1, 0, 1, ids, wts, NULL, has_shared ? &gl : NULL);
    uint16_t* act = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(I > I_shared ? I : I_shared));
    uint16_t* eo = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)K * H);
    for (int j = 0; j < K; ++j) {
      gateup_row(xt, w13 + (int64_t)ids[j] * 2 * I * H, H, I, act, 1);
      down_row(act, w2 + (int64_t)ids[j] * H * I, I, H, &wts[j], eo + (int64_t)j * H);
    }
    uint16_t* o = out + (int64_t)i * H;
    if (has_shared) {
      uint16_t* sd = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)H);
      gateup_row(xt, w13_shared, H, I_shared, act, 1);
      down_row(act, w2_shared, I_shared, H, NULL, sd);
      oracle_combine_gate(eo, ORA_BF16, NULL, sd, ORA_BF16, &gl, routed_scale, 1, K, H, o,
                          ORA_BF16);
      free(sd);
    } else {
      oracle_combine(eo, ORA_BF16, NULL, NULL, ORA_BF16, routed_scale, 1, K, H, o, ORA_BF16);
    }
    if (ids_out) memcpy(ids_out + (int64_t)i * K, ids, sizeof(int32_t) * (size_t)K);
    if (w_out) memcpy(w_out + (int64_t)i * K, wts, sizeof(float) * (size_t)K);
    free(act);
    free(eo);
  }
  return ORA_OK;
}
