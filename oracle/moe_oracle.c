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
 *
 * Parity unpinned at bit level: the exp inside the gate/up SiLU is the C
 * library's expf (the pages fix no exp there), so the GPU's gate/up output is
 * compared with this file's within the GEMM tolerance only; this file's gate/up
 * is itself pinned against float64 within that tolerance.
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

int oracle_abi_version(void) { return 4; }

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

void oracle_sigmoid_f32_array(const float* g, float* y, int64_t n) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) y[i] = oracle_sigmoid_f32(g[i]);
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

/* act = bf16(silu(g) * u) with g and u narrowed to bf16 first; narrow = 0 is
 * a planted mutation used only by tests */
static uint16_t gateup_out(float g, float u, int narrow) {
  if (narrow) {
    g = bf16_round(g);
    u = bf16_round(u);
  }
  float s = silu_f32(g);
  float v = s * u;
  return f2bf(v);
}

/* one output row */
static void gateup_row(const uint16_t* a_row, const uint16_t* w13_g, int H, int I,
                       uint16_t* act_row, int narrow) {
  for (int n = 0; n < I; ++n) {
    float g = dot_bf16(a_row, w13_g + (int64_t)n * H, H);
    float u = dot_bf16(a_row, w13_g + (int64_t)(I + n) * H, H);
    act_row[n] = gateup_out(g, u, narrow);
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

/* ------------------------------------------------------------------ */
/* Keep-quant expert GEMM: kMatmulBTQuant / kMatmulBTQuantGrouped of    */
/* vllm.cpp PR #523 ("What changed"): the expert matmul runs on the     */
/* quantized weights as stored, grouped over the expert ids.  Activations */
/* are quantized to 8-bit blocks (a Q8_0 quantizer for Q8_0 weights, a   */
/* Q8_K one for the K-quant formats) and each block's dot product is an  */
/* exact integer sum.  PR #523 "Evidence" checks it at NMSE <= 5e-4      */
/* against a CPU keep-quant reference.                                   */
/*                                                                      */
/* Weight formats (the GGUF block layouts, stored little-endian):        */
/*   Q8_0: 32 weights in 34 bytes -- fp16 d, int8 q[32]; w = d * q.       */
/*   Q4_K: 256 weights in 144 bytes -- fp16 d, fp16 dmin, 12 bytes of    */
/*         packed 6-bit sub-block scales and mins, 128 bytes of 4-bit    */
/*         codes; sub-block j (32 weights) has w = d*sc_j*q - dmin*m_j.  */
/* READING (activation quantizer; the pages name it but do not define    */
/* it): per block of 32 (Q8_0) or 256 (Q8_K) values,                     */
/*   amax = max |x|,  d = amax / 127,  id = d != 0 ? 1 / d : 0,           */
/*   q = round-half-away(x * id), NaN -> 0, clamped to [-127, 127],      */
/* every operation one binary32 rounding; the Q8_0 block stores d rounded */
/* to fp16 (the Q8_0 format), the Q8_K block keeps the f32 d.  Codes go  */
/* to an int8 [R, K] plane and scales to an f32 [R, K/block] plane.       */
/* READING (float combination): the integer block sums are exact; the    */
/* oracle combines them in double precision, block after block, and     */
/* rounds the row result to binary32 once.                              */
/* ------------------------------------------------------------------ */

#define ORA_Q8_0 1
#define ORA_Q4_K 2

/* fp16 bits -> f32, exact */
static float h2f(uint16_t h) {
  const int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  float v;
  if (e == 31)
    v = m ? NAN : INFINITY;
  else if (e == 0)
    v = ldexpf((float)m, -24);
  else
    v = ldexpf((float)(1024 + m), e - 25);
  return sign ? -v : v;
}

/* f32 -> fp16 bits, round to nearest, ties to even, from the definition:
 * keep the top 11 significant bits (fewer below 2^-14, where the spacing is
 * fixed at 2^-24), then round up when the dropped part is above one half or
 * exactly one half with an odd kept part; a carry moves into the exponent,
 * up to infinity.  NaN gives the quiet NaN 0x7e00 with the sign kept. */
static uint16_t f2h(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  const uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return sign | 0x7E00u;
  if (a == 0x7F800000u) return sign | 0x7C00u;
  const int e = (int)(a >> 23) - 127; /* unbiased exponent (-127 for f32 subnormals) */
  if (e >= 16) return sign | 0x7C00u;
  uint32_t sig; /* significand with the implicit bit */
  int shift;    /* bits dropped to reach the fp16 spacing */
  if (e >= -14) {
    sig = (a & 0x7FFFFFu) | 0x800000u;
    shift = 13;
  } else {
    sig = (e == -127) ? (a & 0x7FFFFFu) : ((a & 0x7FFFFFu) | 0x800000u);
    const int e_eff = (e == -127) ? -126 : e;
    shift = 13 + (-14 - e_eff); /* value = sig * 2^(e_eff-23); fp16 unit 2^-24 */
    if (shift > 31) return sign;
  }
  uint32_t kept = sig >> shift;
  const uint32_t dropped = sig & ((1u << shift) - 1u);
  const uint32_t half = 1u << (shift - 1);
  if (dropped > half || (dropped == half && (kept & 1u))) kept += 1u;
  uint32_t bits;
  if (e >= -14)
    bits = ((uint32_t)(e + 15) << 10) + (kept - 1024u); /* carry reaches the exponent */
  else
    bits = kept; /* subnormal, or 0x400 = the smallest normal after a carry */
  return sign | (uint16_t)bits;
}

float oracle_f16_to_f32(uint16_t h) { return h2f(h); }
uint16_t oracle_f32_to_f16(float f) { return f2h(f); }

static uint16_t le16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

static int q_block(int fmt) { return fmt == ORA_Q8_0 ? 32 : (fmt == ORA_Q4_K ? 256 : 0); }
static int q_block_bytes(int fmt) { return fmt == ORA_Q8_0 ? 34 : (fmt == ORA_Q4_K ? 144 : 0); }

/* Q4_K: the 6-bit scale and min of sub-block j (0..7) from the 12 packed
 * bytes.  Sub-blocks 0-3 keep theirs in the low six bits of bytes j
 * (scale) and j+4 (min); sub-blocks 4-7 take their low four bits from the
 * two nibbles of byte j+4 and their top two bits from the top bits of
 * bytes j-4 (scale) and j (min). */
static void q4k_scale_min(const uint8_t* s, int j, int* sc, int* m) {
  if (j < 4) {
    *sc = s[j] & 63;
    *m = s[j + 4] & 63;
  } else {
    *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
    *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
  }
}

int oracle_q4k_scale_min(const uint8_t* scales12, int j, int32_t* sc_m) {
  if (!scales12 || !sc_m || j < 0 || j > 7) return ORA_ERR_ARG;
  int sc, m;
  q4k_scale_min(scales12, j, &sc, &m);
  sc_m[0] = sc;
  sc_m[1] = m;
  return ORA_OK;
}

/* Q4_K: the 4-bit code of weight k (0..255) of a super-block.  Each group of
 * 64 weights owns 32 bytes of codes: the low nibble of byte i is weight i of
 * the group's first sub-block, the high nibble weight i of its second. */
static int q4k_code(const uint8_t* qs, int k) {
  const int c = k / 64, o = k % 64;
  const uint8_t b = qs[32 * c + (o % 32)];
  return o < 32 ? (b & 15) : (b >> 4);
}

/* rows x K weights in `fmt` blocks -> exact values (double) */
int oracle_dequant_q(const uint8_t* w, int fmt, int64_t rows, int K, double* out) {
  const int blk = q_block(fmt), bb = q_block_bytes(fmt);
  if (!blk || !w || !out || rows < 0 || K <= 0 || K % blk) return ORA_ERR_ARG;
  const int64_t nb = K / blk;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t* p = w + (r * nb + b) * bb;
      double* o = out + r * K + b * blk;
      if (fmt == ORA_Q8_0) {
        const double d = h2f(le16(p));
        for (int i = 0; i < 32; ++i) o[i] = d * (double)(int8_t)p[2 + i];
      } else {
        const double d = h2f(le16(p)), dmin = h2f(le16(p + 2));
        for (int k = 0; k < 256; ++k) {
          int sc, m;
          q4k_scale_min(p + 4, k / 32, &sc, &m);
          o[k] = d * sc * q4k_code(p + 16, k) - dmin * m;
        }
      }
    }
  return ORA_OK;
}

/* activation quantizer (READING above): x bf16 [R, K] -> q int8 [R, K],
 * d f32 [R, K / block] with block 32 (fmt Q8_0) or 256 (fmt Q4_K) */
int oracle_quantize_act_q8(const uint16_t* x, int64_t R, int K, int fmt, int8_t* q, float* d) {
  const int blk = q_block(fmt);
  if (!blk || !x || !q || !d || R < 0 || K <= 0 || K % blk) return ORA_ERR_ARG;
  const int64_t nb = K / blk;
#pragma omp parallel for schedule(static)
  for (int64_t rb = 0; rb < R * nb; ++rb) {
    const uint16_t* xb = x + rb * blk;
    float amax = 0.0f;
    for (int i = 0; i < blk; ++i) {
      const float a = fabsf(bf2f(xb[i]));
      if (a > amax) amax = a;
    }
    const float dd = amax / 127.0f;
    const float id = dd != 0.0f ? 1.0f / dd : 0.0f;
    for (int i = 0; i < blk; ++i) {
      float r = roundf(bf2f(xb[i]) * id);
      if (r != r) r = 0.0f;
      if (r > 127.0f) r = 127.0f;
      if (r < -127.0f) r = -127.0f;
      q[rb * blk + i] = (int8_t)r;
    }
    d[rb] = fmt == ORA_Q8_0 ? h2f(f2h(dd)) : dd;
  }
  return ORA_OK;
}

/* one keep-quant dot product: activation row (codes aq, scales ad) with one
 * weight row of K weights; *abs_out = the sum of the block terms' magnitudes */
static double qdot(const int8_t* aq, const float* ad, const uint8_t* wrow, int fmt, int K,
                   double* abs_out) {
  double y = 0.0, ya = 0.0;
  if (fmt == ORA_Q8_0) {
    for (int b = 0; b < K / 32; ++b) {
      const uint8_t* p = wrow + (int64_t)b * 34;
      int64_t isum = 0;
      for (int i = 0; i < 32; ++i) isum += (int64_t)(int8_t)p[2 + i] * aq[b * 32 + i];
      const double t = (double)h2f(le16(p)) * (double)ad[b] * (double)isum;
      y += t;
      ya += fabs(t);
    }
  } else {
    for (int b = 0; b < K / 256; ++b) {
      const uint8_t* p = wrow + (int64_t)b * 144;
      const int8_t* a = aq + b * 256;
      int64_t s1 = 0, s2 = 0;
      for (int j = 0; j < 8; ++j) {
        int sc, m;
        q4k_scale_min(p + 4, j, &sc, &m);
        int64_t isum = 0, asum = 0;
        for (int i = 0; i < 32; ++i) {
          isum += (int64_t)q4k_code(p + 16, 32 * j + i) * a[32 * j + i];
          asum += a[32 * j + i];
        }
        s1 += sc * isum;
        s2 += m * asum;
      }
      const double dx = ad[b], t1 = (double)h2f(le16(p)) * (double)s1,
                   t2 = (double)h2f(le16(p + 2)) * (double)s2;
      y += dx * (t1 - t2);
      ya += fabs(dx) * (fabs(t1) + fabs(t2));
    }
  }
  if (abs_out) *abs_out = ya;
  return y;
}

static int q_args_ok(int fmt, int K, const int32_t* off, int G, int P) {
  if (!q_block(fmt) || K <= 0 || K % q_block(fmt) || G <= 0 || P < 0) return 0;
  if (!off && G != 1) return 0;
  return offsets_ok(off, G, P);
}

/* plain grouped keep-quant matmul: y[r, n] = sum_k A[src(r), k] * W[g, n, k]
 * for rows r of group g, src(r) = a_row_gather ? a_row_gather[r] / gather_div : r;
 * y (and yabs, the per-element sum of block-term magnitudes) in double */
int oracle_gemm_q(const int8_t* aq, const float* ad, const int32_t* a_row_gather, int gather_div,
                  const uint8_t* w, int fmt, const int32_t* group_offsets, int P, int K, int N,
                  int G, const int32_t* rows, int n_rows, double* y, double* yabs) {
  if (!q_args_ok(fmt, K, group_offsets, G, P) || N <= 0 || !aq || !ad || !w || !y)
    return ORA_ERR_ARG;
  if (a_row_gather && gather_div < 1) return ORA_ERR_ARG;
  int32_t single[2] = {0, P};
  const int32_t* off = group_offsets ? group_offsets : single;
  const int64_t nb = K / q_block(fmt), row_bytes = nb * q_block_bytes(fmt);
  const int64_t n = rows ? n_rows : (int64_t)off[G] - off[0];
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n; ++i) {
    const int64_t r = rows ? rows[i] : off[0] + i;
    const int g = group_of_row(off, G, r);
    if (g < 0) continue;
    const int64_t src = a_row_gather ? a_row_gather[r] / gather_div : r;
    for (int64_t c = 0; c < N; ++c) {
      double ya;
      y[r * N + c] = qdot(aq + src * K, ad + src * nb, w + ((int64_t)g * N + c) * row_bytes, fmt,
                          K, &ya);
      if (yabs) yabs[r * N + c] = ya;
    }
  }
  return ORA_OK;
}

static void gateup_q_row(const int8_t* aq, const float* ad, const uint8_t* w13_g, int fmt, int H,
                         int I, uint16_t* act_row) {
  const int64_t row_bytes = (int64_t)(H / q_block(fmt)) * q_block_bytes(fmt);
  for (int n = 0; n < I; ++n) {
    const float g = (float)qdot(aq, ad, w13_g + n * row_bytes, fmt, H, NULL);
    const float u = (float)qdot(aq, ad, w13_g + (int64_t)(I + n) * row_bytes, fmt, H, NULL);
    act_row[n] = gateup_out(g, u, 1);
  }
}

static void down_q_row(const int8_t* aq, const float* ad, const uint8_t* w2_g, int fmt, int I,
                       int H, const float* weight, uint16_t* out_row) {
  const int64_t row_bytes = (int64_t)(I / q_block(fmt)) * q_block_bytes(fmt);
  for (int n = 0; n < H; ++n) {
    float y = (float)qdot(aq, ad, w2_g + n * row_bytes, fmt, I, NULL);
    if (weight) y = y * (*weight);
    out_row[n] = f2bf(y);
  }
}

/* gate/up with SiLU-and-mul on keep-quant weights: the bf16 gate/up contract
 * (narrowing before the activation) on top of the keep-quant dot products;
 * w13 [G, 2I, H/block] blocks, gate rows first */
int oracle_gateup_silu_q(const int8_t* aq, const float* ad, const int32_t* a_row_gather,
                         int gather_div, const uint8_t* w13, int fmt,
                         const int32_t* group_offsets, int P, int H, int I, int G,
                         const int32_t* rows, int n_rows, uint16_t* act) {
  if (!q_args_ok(fmt, H, group_offsets, G, P) || I <= 0 || !aq || !ad || !w13 || !act)
    return ORA_ERR_ARG;
  if (a_row_gather && gather_div < 1) return ORA_ERR_ARG;
  int32_t single[2] = {0, P};
  const int32_t* off = group_offsets ? group_offsets : single;
  const int64_t nb = H / q_block(fmt), row_bytes = nb * q_block_bytes(fmt);
  const int64_t n = rows ? n_rows : (int64_t)off[G] - off[0];
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n; ++i) {
    const int64_t r = rows ? rows[i] : off[0] + i;
    const int g = group_of_row(off, G, r);
    if (g < 0) continue;
    const int64_t src = a_row_gather ? a_row_gather[r] / gather_div : r;
    gateup_q_row(aq + src * H, ad + src * nb, w13 + (int64_t)g * 2 * I * row_bytes, fmt, H, I,
                 act + r * I);
  }
  return ORA_OK;
}

/* down on keep-quant weights: the bf16 down contract (one f32 weight
 * multiply, one bf16 rounding, scatter to pair order); w2 [G, H, I/block] */
int oracle_down_q(const int8_t* aq, const float* ad, const uint8_t* w2, int fmt,
                  const int32_t* group_offsets, const float* pair_weight,
                  const int32_t* row_to_pair, int P, int I, int H, int G, const int32_t* rows,
                  int n_rows, uint16_t* out) {
  if (!q_args_ok(fmt, I, group_offsets, G, P) || H <= 0 || !aq || !ad || !w2 || !out)
    return ORA_ERR_ARG;
  int32_t single[2] = {0, P};
  const int32_t* off = group_offsets ? group_offsets : single;
  const int64_t nb = I / q_block(fmt), row_bytes = nb * q_block_bytes(fmt);
  const int64_t n = rows ? n_rows : (int64_t)off[G] - off[0];
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n; ++i) {
    const int64_t r = rows ? rows[i] : off[0] + i;
    const int g = group_of_row(off, G, r);
    if (g < 0) continue;
    const int64_t dst = row_to_pair ? row_to_pair[r] : r;
    down_q_row(aq + r * I, ad + r * nb, w2 + (int64_t)g * H * row_bytes, fmt, I, H,
               pair_weight ? pair_weight + dst : NULL, out + dst * H);
  }
  return ORA_OK;
}

/* The whole block with keep-quant expert weights, token by token: the bf16
 * router, then per selected expert the token's row quantized (fmt's
 * activation quantizer), keep-quant gate/up + SiLU-mul, the bf16 act row
 * quantized again, keep-quant down with the routing weight; the shared
 * expert stays bf16; then the combine (or the combine-gate).  The quantizer
 * works on blocks inside one row, so a row's result does not depend on the
 * batch it is computed in. */
int oracle_moe_layer_tokens_q(const uint16_t* x, const uint16_t* w_router,
                              const float* logit_bias, const uint8_t* w13q, const uint8_t* w2q,
                              int fmt, const uint16_t* w_shared_gate, const uint16_t* w13_shared,
                              const uint16_t* w2_shared, int H, int I, int E, int K, int I_shared,
                              float routed_scale, const int32_t* tokens, int n_tokens,
                              int32_t* ids_out, float* w_out, uint16_t* out) {
  if (H <= 0 || I <= 0 || E <= 0 || K < 1 || K > E || K > 32 || n_tokens < 0) return ORA_ERR_ARG;
  const int blk = q_block(fmt);
  if (!blk || H % blk || I % blk) return ORA_ERR_ARG;
  const int has_shared = (w_shared_gate && w13_shared && w2_shared && I_shared > 0);
  const int64_t rb13 = (int64_t)(H / blk) * q_block_bytes(fmt);
  const int64_t rb2 = (int64_t)(I / blk) * q_block_bytes(fmt);
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < n_tokens; ++i) {
    const uint16_t* xt = x + (int64_t)tokens[i] * H;
    int32_t ids[32];
    float wts[32];
    float gl = 0.0f;
    oracle_route_topk(xt, w_router, logit_bias, has_shared ? w_shared_gate : NULL, NULL, 1, H, E,
                      K, 1, 0, 1, ids, wts, NULL, has_shared ? &gl : NULL);
    int8_t* xq = (int8_t*)malloc((size_t)H);
    float* xd = (float*)malloc(sizeof(float) * (size_t)(H / blk));
    int8_t* aq = (int8_t*)malloc((size_t)I);
    float* adv = (float*)malloc(sizeof(float) * (size_t)(I / blk));
    uint16_t* act = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(I > I_shared ? I : I_shared));
    uint16_t* eo = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)K * H);
    oracle_quantize_act_q8(xt, 1, H, fmt, xq, xd);
    for (int j = 0; j < K; ++j) {
      gateup_q_row(xq, xd, w13q + (int64_t)ids[j] * 2 * I * rb13, fmt, H, I, act);
      oracle_quantize_act_q8(act, 1, I, fmt, aq, adv);
      down_q_row(aq, adv, w2q + (int64_t)ids[j] * H * rb2, fmt, I, H, &wts[j],
                 eo + (int64_t)j * H);
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
    free(xq);
    free(xd);
    free(aq);
    free(adv);
    free(act);
    free(eo);
  }
  return ORA_OK;
}

/* Dequantisation of keep-quant weights to bf16, for running them through
 * the bf16 expert GEMMs.  READING (the pages dequantise only implicitly, when
 * keep-quant is off): the value is formed in binary32 and rounded to bf16 once:
 *   Q8_0: bf16(d * q)                          (exact product)
 *   Q4_K: bf16((d * sc_j) * q - dmin * m_j)    (exact products, one rounded
 *                                               subtraction, then the bf16 rounding) */
int oracle_dequant_q_bf16(const uint8_t* w, int fmt, int64_t rows, int K, uint16_t* out) {
  const int blk = q_block(fmt), bb = q_block_bytes(fmt);
  if (!blk || !w || !out || rows < 0 || K <= 0 || K % blk) return ORA_ERR_ARG;
  const int64_t nb = K / blk;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t* p = w + (r * nb + b) * bb;
      uint16_t* o = out + r * K + b * blk;
      if (fmt == ORA_Q8_0) {
        const float d = h2f(le16(p));
        for (int i = 0; i < 32; ++i) o[i] = f2bf(d * (float)(int8_t)p[2 + i]);
      } else {
        const float d = h2f(le16(p)), dmin = h2f(le16(p + 2));
        for (int k = 0; k < 256; ++k) {
          int sc, m;
          q4k_scale_min(p + 4, k / 32, &sc, &m);
          const float t1 = (d * (float)sc) * (float)q4k_code(p + 16, k);
          const float t2 = dmin * (float)m;
          o[k] = f2bf(t1 - t2);
        }
      }
    }
  return ORA_OK;
}
