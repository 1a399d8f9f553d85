/*
 * moe.h -- C ABI of libmoe.so: the BF16 Mixture-of-Experts expert block of an
 * LLM forward pass on one GB300 (sm_103a).
 *
 *   moe_route_topk                     ungrouped softmax router, top-k, renormalise
 *   moe_permute                        tokens -> expert-contiguous rows
 *   moe_grouped_gemm_gateup_silu_bf16  grouped gate/up GEMM fused with SiLU-and-mul
 *   moe_grouped_gemm_down_bf16         grouped down GEMM, routing weight, scatter
 *   moe_combine                        weighted top-k sum (+ optional shared term)
 *   moe_combine_gate                   combine with the shared-expert sigmoid gate
 *   shared_expert_gate                 out = sigmoid(gl) * sd
 *   moe_quantize_act_q8, moe_grouped_gemm_q, moe_grouped_gemm_gateup_silu_q,
 *   moe_grouped_gemm_down_q            keep-quant expert GEMMs (Q8_0 / Q4_K weights)
 *   moe_dequantize_q_bf16              keep-quant weights expanded to bf16
 *
 * Sources (vllm.cpp pages):
 *   [I3094]  issue #3094 "Row: BACKEND-ROCM-BF16-MOE": names the two grouped
 *            BF16 GEMM ops and the numeric contract -- BF16 narrowing of the
 *            gate/up result before activation, routing weight applied before
 *            the down result is stored, reduction without applying the
 *            weights twice.
 *   [PR509]  PR #509 "MoE combine/gate ops -- SharedExpertGate, MoeCombine,
 *            MoeCombineGate": "What changed" (the three formulas), the review
 *            (dtype refusals, production dtype arms, bit-exactness), the
 *            rework commits (sequential K order, single store rounding, no
 *            contraction; routed_scale on the routed sum before the shared
 *            term), "Honest gaps" (the covered router is ungrouped softmax).
 *   [PR523]  PR #509's stacked follow-up #523, "What changed": the expert GEMM
 *            is grouped over expert ids; activation scratch is capture-safe
 *            and never reallocated during reuse; the keep-quant expert GEMMs
 *            run on GGUF weight blocks with 8-bit activation quantizers.
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or synchronises inside a call.  Scratch memory is
 *     a caller-provided workspace sized by the matching *_workspace_size query.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call only enqueues work on it and returns.
 *   - Row-major layouts.  bf16 = IEEE binary32 rounded to nearest even and
 *     truncated to its upper 16 bits.  T tokens, H hidden, I per-expert
 *     intermediate, E experts, K experts per token, P = T*K routed rows.
 *   - Return value: MOE_OK (0) or a negative MOE_ERR_* code; nothing is
 *     enqueued when a call fails its argument checks.  moe_last_error()
 *     returns a thread-local message naming what was refused.
 *   - T = 0 (P = 0) is a legal no-op.  Data pointers must be 16-byte aligned
 *     and H, I multiples of 8 (MOE_ERR_ALIGN otherwise).
 *   - Bit-exact ops (router selection and weights, permute, combine, gate)
 *     give the same bits as the plain sequential definitions in their
 *     comments; the grouped GEMMs accumulate in f32 in tensor-core order.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types */
enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_F16 = 2 /* always refused, see [PR509] review */ };

/* return codes */
enum {
  MOE_OK = 0,
  MOE_ERR_ARG = -1,         /* a size, count or pointer argument is invalid */
  MOE_ERR_DTYPE = -2,       /* dtype other than f32/bf16 (f16 is refused by name) */
  MOE_ERR_UNSUPPORTED = -3, /* a router form outside ungrouped softmax */
  MOE_ERR_ALIGN = -4,       /* pointer not 16-byte aligned or H/I not a multiple of 8 */
  MOE_ERR_WORKSPACE = -5,   /* workspace missing or smaller than the size query */
  MOE_ERR_CUDA = -6,        /* launch or runtime error (message from the CUDA runtime) */
  MOE_ERR_TIMEOUT = -7      /* a device-side wait hit its iteration cap (see moe_device_status) */
};

/* Thread-local message for the last failing call on this thread. */
const char* moe_last_error(void);

/* Library ABI version (bumped on any signature change). */
int moe_abi_version(void);  /* 10 */

/* ------------------------------------------------------------------------
 * moe_route_topk -- ungrouped softmax router ([PR509] "Honest gaps": the
 * router in scope there is ungrouped softmax; grouped / bias-corrected forms
 * are refused).
 *
 *   l[t,e] = sum_h f32(x[t,h]) * f32(w_router[e,h])  (+ logit_bias[e])
 *            f32 accumulation in tensor-core order (not bit-exact vs a
 *            sequential sum; within the dot-product error bound).
 *   Selection: the K largest l[t,:] in descending order; equal logits go to
 *            the lower expert id; NaN ranks below every number.
 *   Weights (renormalize=1): m = l of rank 0, e_j = expf_cr(l_j - m),
 *            S = ((e_0 + e_1) + ...) + e_{K-1} from +0, w_j = e_j / S.
 *            (renormalize=0: S sums expf_cr(l_e - m) over all e in id order.)
 *            expf_cr is the binary32 rounding of a fixed double-precision
 *            evaluation (Cody-Waite reduction with ln2 split in a 32-bit head
 *            and a tail, Taylor series through r^13, scaling by 2^n); its
 *            result is the correctly rounded exp on every input tested.  The
 *            kernels obtain the same bits mostly from binary32 arithmetic (a
 *            table-driven form that declines inputs near a rounding midpoint
 *            and hands them to the double chain): see moe_exp_sigmoid_f32.
 *   Given the same logits (logits_in), ids and weights are bit-exact.
 *
 *   x            bf16 [T,H]        (ignored when logits_in != NULL)
 *   w_router     bf16 [E,H]        (ignored when logits_in != NULL)
 *   logit_bias   f32  [E] or NULL  added to every logit before selection and weights
 *   w_shared_gate bf16 [H] or NULL if set, gate_logit_out[t] = sum_h x[t,h]*wsg[h]
 *   logits_in    f32  [T,E] or NULL: use these logits instead of the GEMM
 *   T >= 0, H > 0 (multiple of 8), 1 <= K <= min(E, 32), E <= 1024
 *   renormalize  1 (the block's path) or 0
 *   scoring      0 = softmax (anything else: MOE_ERR_UNSUPPORTED)
 *   n_group      1 (anything else: MOE_ERR_UNSUPPORTED)
 *   topk_ids     int32 [T,K] out, rank order
 *   topk_w       f32   [T,K] out
 *   logits_out   f32   [T,E] out or NULL
 *   gate_logit_out f32 [T] out; required when w_shared_gate != NULL
 *   workspace    >= moe_route_topk_workspace_size(T, E, K) bytes (may be 0
 *                when logits_in or logits_out is given).  When T*E gives the
 *                logits GEMM fewer tiles than SMs (decode), it splits K into up
 *                to 16 ranges whose partial sums go to the workspace; the
 *                selection adds them in range order, then the bias.  It uses as
 *                many ranges as the workspace holds (one: no split), so a
 *                smaller workspace only costs speed.
 * Errors: MOE_ERR_ARG (T < 0; E outside [1, 1024]; K outside [1, min(E, 32)];
 * renormalize not 0 or 1; NULL topk_ids or topk_w; no x or w_router without
 * logits_in; w_shared_gate without x or gate_logit_out), MOE_ERR_ALIGN (H not a
 * positive multiple of 8 where x is read; x, w_router, w_shared_gate or the
 * workspace not 16-byte aligned), MOE_ERR_UNSUPPORTED (scoring != 0 or
 * n_group != 1; the message points to moe_route_topk_ex), MOE_ERR_WORKSPACE (the
 * logits GEMM runs with neither logits_out nor room for T*E logits),
 * MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
int moe_route_topk(const void* x_bf16, const void* w_router_bf16, const float* logit_bias,
                   const void* w_shared_gate_bf16, const float* logits_in, int T, int H, int E,
                   int K, int renormalize, int scoring, int n_group, int32_t* topk_ids,
                   float* topk_w, float* logits_out, float* gate_logit_out, void* workspace,
                   size_t ws_bytes, void* stream);
size_t moe_route_topk_workspace_size(int T, int E, int K);

/* ------------------------------------------------------------------------
 * moe_route_topk_ex -- the router forms the pages leave open: [I3094] keeps
 * the grouped and sigmoid routers of DeepSeek-V2 and Dots3 out of its scope,
 * and [PR509] "Honest gaps" says its grouped / bias / noaux_tc forms still
 * throw.  The pages do not define them; this follows the published
 * DeepSeek-V2 (softmax, groups scored by their best expert) and DeepSeek-V3
 * (sigmoid scores, selection bias, groups scored by their two best experts)
 * routers.  Logits as in moe_route_topk (GEMM, K split, logit_bias), then:
 *   s_e   = l_e (scoring 0, softmax) or sigmoid(l_e) (scoring 1; the same
 *           binary32 sigmoid as the shared-expert gate)
 *   k_e   = s_e + select_bias[e] (sigmoid only; steers the choice, never
 *           enters a weight), else s_e
 *   groups: E / n_group contiguous experts each; score = best k (group_score
 *           0) or best + second best k (1); the topk_group best groups stay
 *           eligible (descending, ties to the lower group, NaN last)
 *   choice: the K best k among eligible experts (descending, ties to the
 *           lower id, NaN last)
 *   weights: sigmoid: w_j = s_j / ((s_0 + s_1) + ... + s_{K-1}) from +0
 *           (renormalize 1) or s_j (0); softmax: as moe_route_topk
 * Given the same logits, ids and weights are bit-exact.  scoring 0 with
 * n_group 1 and no select_bias is exactly moe_route_topk.
 *   select_bias  f32 [E] or NULL (sigmoid scoring only)
 *   n_group      1..64, divides E; topk_group 1..n_group; group_score 0 or 1
 *                (1 needs groups of at least two experts)
 *   K            <= topk_group * E / n_group (and the limits of moe_route_topk)
 *   the other arguments, outputs, workspace and errors as moe_route_topk;
 *   MOE_ERR_UNSUPPORTED for scoring > 1 or a select_bias with softmax.
 * Errors: those of moe_route_topk, except that scoring 1 and n_group > 1 are
 * accepted; MOE_ERR_UNSUPPORTED (scoring not 0 or 1; a select_bias with softmax
 * scoring), MOE_ERR_ARG (n_group not dividing E or above 64; topk_group outside
 * [1, n_group]; group_score not 0 or 1; two-best group scores with one expert
 * per group; K above the experts of the eligible groups), MOE_ERR_ALIGN
 * (select_bias not 4-byte aligned).
 * ---------------------------------------------------------------------- */
int moe_route_topk_ex(const void* x_bf16, const void* w_router_bf16, const float* logit_bias,
                      const float* select_bias, const void* w_shared_gate_bf16,
                      const float* logits_in, int T, int H, int E, int K, int renormalize,
                      int scoring, int n_group, int topk_group, int group_score,
                      int32_t* topk_ids, float* topk_w, float* logits_out,
                      float* gate_logit_out, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * moe_permute -- stable counting sort of the P = T*K (token, slot) pairs by
 * expert, so each expert's rows are contiguous for the grouped GEMMs ([PR509]
 * review: the expert path keeps P permuted bf16 rows of H; [PR523]:
 * grouped over expert ids).  Rows of one expert keep ascending pair order
 * p = t*K + j.  Bit-exact.
 *
 *   topk_ids       int32 [T,K] in, each in [0,E) (checked on the device:
 *                  out-of-range ids are counted nowhere and raise the device
 *                  status flag MOE_STATUS_BAD_ID)
 *   x              bf16 [T,H] or NULL (indices only)
 *   expert_offsets int32 [E+1] out: exclusive scan of the per-expert counts
 *   sorted_pair    int32 [P] out: sorted_pair[row] = p
 *   pair_to_row    int32 [P] out: inverse of sorted_pair
 *   x_perm         bf16 [P,H] out or NULL: x_perm[row] = x[sorted_pair[row] / K]
 *   T >= 0, 1 <= K <= 32, 1 <= E <= 1024, H multiple of 8 when x != NULL
 *   workspace      >= moe_permute_workspace_size(T, K, E) bytes
 * Errors: MOE_ERR_ARG (T < 0; K outside [1, 32]; E outside [1, 1024]; T*K too
 * large; NULL topk_ids, expert_offsets, sorted_pair or pair_to_row; x_perm
 * without x or H > 0), MOE_ERR_ALIGN (x or x_perm not 16-byte aligned, H not a
 * multiple of 8), MOE_ERR_WORKSPACE (below moe_permute_workspace_size),
 * MOE_ERR_CUDA.  An id outside [0, E) is skipped on the device and sets
 * MOE_STATUS_BAD_ID in the status word (moe_device_status).
 * ---------------------------------------------------------------------- */
int moe_permute(const int32_t* topk_ids, const void* x_bf16, int T, int K, int E, int H,
                int32_t* expert_offsets, int32_t* sorted_pair, int32_t* pair_to_row,
                void* x_perm_bf16, void* workspace, size_t ws_bytes, void* stream);
size_t moe_permute_workspace_size(int T, int K, int E);

/* ------------------------------------------------------------------------
 * moe_permute_noalloc -- moe_permute without a caller-provided workspace, for
 * callers that cannot allocate device memory (no reachable allocator at the
 * call site, or allocation forbidden after start-up).  The pages have no
 * counterpart of this entry point; it exists for those callers only.
 *
 * Same arguments, outputs and bit-exact results as moe_permute, minus the
 * workspace.  The scratch is a fixed array of MOE_PERMUTE_NOALLOC_MAX_SCRATCH
 * bytes inside the library's device memory (held by every GPU that loads the
 * library until the process exits).  The histogram needs 4 bytes per expert
 * for each chunk of 512 pairs, so calls are accepted for
 *   P = T*K <= 512 * floor(2^18 / E)   (131072 pairs at E = 1024, 524288 at
 *                                       E = 256, 1048576 at E = 128)
 * and larger ones are refused with MOE_ERR_WORKSPACE.  The call allocates
 * nothing.  Every call looks up the array's device address on the current
 * device (cudaGetSymbolAddress, a host-side lookup); the first lookup on a
 * device loads the library's device code there, so make the first call on
 * each device before any stream capture.  All calls share the array and it
 * keeps the last call's contents (no state carries over: every entry read is
 * written first); calls whose kernels may overlap on the GPU race on it.
 * ---------------------------------------------------------------------- */
#define MOE_PERMUTE_NOALLOC_MAX_SCRATCH (1 << 20)
int moe_permute_noalloc(const int32_t* topk_ids, const void* x_bf16, int T, int K, int E, int H,
                        int32_t* expert_offsets, int32_t* sorted_pair, int32_t* pair_to_row,
                        void* x_perm_bf16, void* stream);

/* ------------------------------------------------------------------------
 * moe_grouped_gemm_gateup_silu_bf16 -- kMoeGroupedGemmBf16GateUpSilu of
 * [I3094].  For every group g and row r in [group_offsets[g], group_offsets[g+1]):
 *   gate[n] = bf16( sum_h A[r,h] * w13[g, n, h] )        n in [0, I)
 *   up[n]   = bf16( sum_h A[r,h] * w13[g, I + n, h] )
 *   act[r,n] = bf16( silu(f32 gate[n]) * f32 up[n] ),  silu(z) = z / (1 + exp(-z))
 * f32 accumulation on tcgen05 tensor cores; both halves are narrowed to bf16
 * BEFORE the activation, as the numeric contract of [I3094] requires.
 *
 *   a            bf16 [P,H] (rows in group order), or, when a_row_gather is
 *                set, bf16 [a_rows,H] read through a_row_gather
 *   a_rows       rows of `a` when gathering (ignored otherwise)
 *   a_row_gather int32 [P] or NULL: row r of the product reads A row
 *                a_row_gather[r] / gather_div.  With sorted_pair and gather_div = K
 *                this reads every routed row straight from x [T,H] (no x_perm);
 *                extra warps copy the rows into shared memory with 16-byte
 *                cp.async (four per CTA on 128-row single-CTA tiles, one on the
 *                32-row tiles of calls with at most 16 rows per group on
 *                average, two per CTA on CTA-pair tiles).  An index outside
 *                [0, a_rows) reads zeros.  The result is bit-identical to
 *                passing the gathered rows as `a`.  On this GPU the copies
 *                through the SMs' load path are slower than a separate x_perm
 *                pass plus tiled TMA loads on prefill-sized calls; on decode-
 *                sized calls (32-row tiles) the gathered form is as fast and
 *                saves the x_perm pass.
 *   gather_div   >= 1 when gathering (ignored otherwise)
 *   w13          bf16 [G, 2I, H]: gate rows first, then up rows, per group
 *   group_offsets int32 [G+1], non-decreasing, group_offsets[G] <= P;
 *                read on the device (no host round trip); may be NULL when G == 1
 *                (one group of P rows)
 *   act          bf16 [P,I] out; rows outside every group are not written
 *   P >= 0, H > 0 and I > 0 multiples of 64, 1 <= G <= 1024
 *   workspace    >= moe_grouped_gemm_workspace_size(...) bytes (currently 0)
 * Errors: MOE_ERR_ARG (P < 0; a non-positive dimension; G outside [1, 1024];
 * NULL operands; NULL group_offsets with G > 1; gathering with a_rows < 1 or
 * gather_div < 1), MOE_ERR_ALIGN (operands not 16-byte aligned; H or I not a
 * multiple of 8), MOE_ERR_CUDA (tensor-map encoding, shared-memory reservation
 * or launch).  A device-side wait that runs past its limit sets
 * MOE_STATUS_TIMEOUT in the status word (moe_device_status).
 * ---------------------------------------------------------------------- */
int moe_grouped_gemm_gateup_silu_bf16(const void* a_bf16, int a_rows, const int32_t* a_row_gather,
                                      int gather_div, const void* w13_bf16,
                                      const int32_t* group_offsets, int P, int H, int I, int G,
                                      void* act_bf16, void* workspace, size_t ws_bytes,
                                      void* stream);

/* ------------------------------------------------------------------------
 * moe_grouped_gemm_gateup_silu_bf16_staged -- the same op as
 * moe_grouped_gemm_gateup_silu_bf16 on the routed rows of x (kMoeGroupedGemmBf16GateUpSilu
 * of [I3094]), with the row gather of moe_permute folded into the launch:
 *   x_perm[r] = x[sorted_pair[r] / K]   for r in [0, P)   (zeros if that row is
 *                                        outside [0, T))
 *   act = the gate/up result of moe_grouped_gemm_gateup_silu_bf16 on x_perm,
 * bit for bit.  On CTA-pair tiles (prefill-sized batches, moe_set_gemm_pairing)
 * warps of the GEMM launch itself write x_perm, 16 rows at a time, and each tile
 * reads its rows once their chunk is written, so the copy overlaps the GEMM;
 * otherwise a row-gather launch runs first, then the single-CTA tiles.
 *
 *   x            bf16 [T,H]
 *   sorted_pair  int32 [P]: moe_permute's sorted_pair (pair p = t*K + k)
 *   K            >= 1: the divisor that turns a pair into its token row
 *   x_perm       bf16 [P,H] out, 16-byte aligned (written, then read, by this call)
 *   w13, group_offsets, P, H, I, G, act: as for moe_grouped_gemm_gateup_silu_bf16
 *   workspace    >= moe_gateup_staged_workspace_size(P) bytes, 16-byte aligned,
 *                device memory, zero-filled before its first use and then passed
 *                unchanged to every later call (it carries per-chunk ready flags
 *                and the flag value of the last launch, so no reset is needed
 *                between calls).  Calls that may run concurrently need their own.
 * Errors: those of moe_grouped_gemm_gateup_silu_bf16; MOE_ERR_ARG (T < 1 or K < 1,
 * NULL sorted_pair or x_perm, with P > 0), MOE_ERR_ALIGN (x_perm), MOE_ERR_WORKSPACE.
 * A device-side wait that runs past its limit (moe_set_wait_limit_ns), including
 * a tile's wait for its rows, sets MOE_STATUS_TIMEOUT.
 * ---------------------------------------------------------------------- */
size_t moe_gateup_staged_workspace_size(int P);
int moe_grouped_gemm_gateup_silu_bf16_staged(const void* x_bf16, int T, const int32_t* sorted_pair,
                                             int K, void* x_perm_bf16, const void* w13_bf16,
                                             const int32_t* group_offsets, int P, int H, int I,
                                             int G, void* act_bf16, void* workspace,
                                             size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * moe_grouped_gemm_down_bf16 -- kMoeGroupedGemmBf16 of [I3094].  For every
 * group g and row r in it:
 *   y[n] = sum_i act[r,i] * w2[g, n, i]   (f32, tensor cores)
 *   out[dst, n] = bf16( y[n] * pair_weight[dst] )   dst = row_to_pair ? row_to_pair[r] : r
 * The routing weight is applied exactly once, as one f32 multiply before the
 * one bf16 rounding of the store: [I3094] puts the weight on the down result
 * ahead of its store, so a combine after it must not apply it again.
 *
 *   act          bf16 [P,I]
 *   w2           bf16 [G,H,I]
 *   group_offsets int32 [G+1] (as above; NULL allowed when G == 1)
 *   pair_weight  f32 [P] indexed by dst, or NULL (no weight: the shared expert)
 *   row_to_pair  int32 [P] or NULL (store in row order)
 *   out          bf16 [P,H] out (pair order when row_to_pair is set, i.e. [T,K,H])
 *   P >= 0, H > 0 and I > 0 multiples of 64, 1 <= G <= 1024
 * Errors: those of moe_grouped_gemm_gateup_silu_bf16 (no gather here).
 * ---------------------------------------------------------------------- */
int moe_grouped_gemm_down_bf16(const void* act_bf16, const void* w2_bf16,
                               const int32_t* group_offsets, const float* pair_weight,
                               const int32_t* row_to_pair, int P, int I, int H, int G,
                               void* out_bf16, void* workspace, size_t ws_bytes, void* stream);
size_t moe_grouped_gemm_workspace_size(int P, int H, int I, int G);

/* ------------------------------------------------------------------------
 * moe_grouped_gemm_gateup_silu_bf16_shared / moe_grouped_gemm_down_bf16_shared
 * -- the routed expert GEMM and the shared expert's GEMM in ONE launch.
 *
 * The routed half is exactly moe_grouped_gemm_gateup_silu_bf16 over x_perm
 * (no row gather), resp. moe_grouped_gemm_down_bf16 with its routing weight
 * and scatter.  The shared half is the same GEMM over all Ts token rows with
 * the single shared weight matrix and no routing weight: the shared expert of
 * [PR509] (its output sd feeds moe_combine_gate), run as one more group.
 * The shared expert's tiles follow the routed tiles in the one persistent
 * grid's round-robin schedule, so its tensor-bound work fills the ragged last
 * round of the weight-streaming routed tiles instead of a launch of its own.  Every output element
 * is computed by the same tile and K order as in the separate calls, so the
 * results are bit-identical to them.  Always single-CTA 128-row tiles (when
 * one half is empty the call is the plain single-problem one).
 *
 *   gate/up:  xs bf16 [Ts,H], w13s bf16 [1,2Is,H] (gate rows first), acts bf16 [Ts,Is]
 *   down:     acts bf16 [Ts,Is], w2s bf16 [1,H,Is], sd bf16 [Ts,H]
 *   the routed arguments as in the single-problem calls; Is a multiple of 8
 * Errors as the single-problem calls; MOE_ERR_ARG/ALIGN for the shared operands.
 * ---------------------------------------------------------------------- */
int moe_grouped_gemm_gateup_silu_bf16_shared(const void* a_bf16, const void* w13_bf16,
                                             const int32_t* group_offsets, int P, int H, int I,
                                             int G, void* act_bf16, const void* xs_bf16, int Ts,
                                             const void* w13s_bf16, int Is, void* acts_bf16,
                                             void* workspace, size_t ws_bytes, void* stream);
int moe_grouped_gemm_down_bf16_shared(const void* act_bf16, const void* w2_bf16,
                                      const int32_t* group_offsets, const float* pair_weight,
                                      const int32_t* row_to_pair, int P, int I, int H, int G,
                                      void* out_bf16, const void* acts_bf16, int Ts,
                                      const void* w2s_bf16, int Is, void* sd_bf16,
                                      void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * moe_grouped_gemm_gateup_silu_fp8w / moe_grouped_gemm_down_fp8w -- the two
 * expert GEMMs with block-scaled FP8 weights.  The pages name FP8 block-scaled
 * matmul and FP8 group quantisation only as ops of the engine; the format here
 * follows the published DeepSeek-V3 weights: each group's weight matrix is FP8
 * E4M3 codes ("fn" variant: no infinities, largest finite 448) with one f32
 * scale per 128 x 128 block of its own rows and columns.  The GEMM uses
 *   w = bf16( f32(code) * scale )      (one f32 multiply, one RNE rounding)
 * and is then exactly the bf16 call above (same narrowing, weight, scatter,
 * tolerance); activations stay bf16.  Eight converter warps per CTA turn the
 * codes into bf16 tiles in shared memory between the TMA loads and the MMA,
 * so the weights cross HBM at one byte each.
 *   w13_e4m3  uint8 [G, 2I, H] (gate rows first), w13_scale f32 [G, ceil(2I/128), ceil(H/128)]
 *   w2_e4m3   uint8 [G, H, I],                     w2_scale f32 [G, ceil(H/128), ceil(I/128)]
 *   the other arguments as moe_grouped_gemm_gateup_silu_bf16 (x_perm rows, no gather) and
 *   moe_grouped_gemm_down_bf16; the contraction length (H, resp. I) a multiple of 16;
 *   codes 16-byte aligned, scales 4-byte aligned.  Single-CTA tiles (128-wide,
 *   32-row ones when P <= 16 G).  Errors as those calls.
 * ---------------------------------------------------------------------- */
int moe_grouped_gemm_gateup_silu_fp8w(const void* a_bf16, const uint8_t* w13_e4m3,
                                      const float* w13_scale, const int32_t* group_offsets,
                                      int P, int H, int I, int G, void* act_bf16,
                                      void* workspace, size_t ws_bytes, void* stream);
int moe_grouped_gemm_down_fp8w(const void* act_bf16, const uint8_t* w2_e4m3,
                               const float* w2_scale, const int32_t* group_offsets,
                               const float* pair_weight, const int32_t* row_to_pair, int P,
                               int I, int H, int G, void* out_bf16, void* workspace,
                               size_t ws_bytes, void* stream);

/* moe_set_gemm_pairing -- tiling of moe_grouped_gemm_gateup_silu_bf16 (also
 * with gathered or staged rows) and moe_grouped_gemm_down_bf16:
 *   MOE_GEMM_AUTO (default): CTA-pair tiles when P >= 1024, the groups average
 *                    at least 32 rows (P >= 32 G) and G <= 512, single-CTA
 *                    tiles otherwise
 *   MOE_GEMM_SINGLE: one CTA per 128-row x N tile (32-row tiles when P <= 16 G)
 *   MOE_GEMM_PAIR:   CTA-pair tiles for every such call with G <= 512.  A pair
 *                    of SMs runs one tcgen05.mma.cta_group::2 with the group's
 *                    weight rows on the M side (128 per SM) and up to 256 of its
 *                    rows on the N side (N = their count rounded up to 16), so a
 *                    group pads to 16 rows, and each SM stages 16 KB of weights
 *                    plus at most 16 KB of rows per 64-wide K step.  In the
 *                    gate/up GEMM a group's last block of at most 32 rows takes
 *                    two feature blocks per tile (twice the weight rows per step)
 * Results agree up to f32 accumulation order.  The FP8 weight GEMMs and the
 * fused shared-expert launches always use single-CTA tiles.  Values 3 and 4
 * (tilings measured slower and not built) are refused with
 * MOE_ERR_UNSUPPORTED, others with MOE_ERR_ARG.  Process-wide, takes effect at
 * the next launch; returns the previous mode.  Not for use while another
 * thread is launching these GEMMs. */
enum { MOE_GEMM_AUTO = 0, MOE_GEMM_SINGLE = 1, MOE_GEMM_PAIR = 2 };
int moe_set_gemm_pairing(int mode);

/* moe_set_wait_limit_ns -- limit, in nanoseconds of device time, of every
 * pipeline wait inside the bf16 and FP8-weight grouped GEMM kernels (a role
 * waiting for a stage to land or to be freed, or for an accumulator).
 * Default and maximum 10^9 (one second), minimum 1000.  A wait that runs past
 * it raises MOE_STATUS_TIMEOUT in the status word and stops its CTA: the
 * other roles stop at their next wait, the copies and MMAs already in flight
 * are waited for (up to one second each, whatever this limit is), the CTA's
 * tensor memory is freed and the CTA exits, so the device stays usable and the
 * call's output is incomplete.  A short limit lets a caller check this path
 * without a faulty kernel.  Process-wide, takes effect at the next launch.
 * Returns MOE_OK, or MOE_ERR_ARG outside [1000, 10^9]. */
int moe_set_wait_limit_ns(unsigned long long ns);

/* moe_set_pdl -- programmatic dependent launch for every kernel of the
 * library (enable = 1, the default) or plain stream order (0).  With it on,
 * each kernel is allowed to start while the previous kernel in the same
 * stream is still running: its CTAs do their set-up (barrier init, TMEM
 * allocation, descriptor prefetch) early and then wait, on the device, until
 * that kernel has completed before they read or write global memory, so the
 * results are the same either way and only the gaps between kernels shrink.
 * Process-wide, takes effect at the next launch; returns the previous
 * setting (MOE_ERR_ARG unless enable is 0 or 1). */
int moe_set_pdl(int enable);

/* ------------------------------------------------------------------------
 * Keep-quant expert GEMMs -- kMatmulBTQuant / kMatmulBTQuantGrouped of
 * [PR523] ("What changed"): the expert matmul reads the weights as the GGUF
 * blocks they are stored in, grouped over the expert ids; activations are
 * quantized to 8-bit blocks and each block's dot product is an exact integer
 * sum ([PR523] "Evidence" checks the op at NMSE <= 5e-4 against a CPU
 * keep-quant reference).  CUDA-core dp4a kernels: built for decode-class
 * layers, where the weight bytes dominate.
 *
 * Weight formats (qfmt), little-endian blocks along each weight row:
 *   MOE_QFMT_Q8_0  32 weights in 34 bytes: fp16 d, int8 q[32];  w = d * q
 *   MOE_QFMT_Q4_K  256 weights in 144 bytes: fp16 d, fp16 dmin, 12 bytes of
 *                  packed 6-bit scales sc_j and mins m_j, 128 bytes of 4-bit
 *                  codes; sub-block j (32 weights): w = d*sc_j*q - dmin*m_j
 * A weight matrix [G, R, K] is stored as uint8 [G, R, K / block * bytes].
 *
 * moe_quantize_act_q8 -- the activation quantizer: for every block of 32
 * (qfmt Q8_0: Q8_0 activations) or 256 (qfmt Q4_K: Q8_K activations) values
 * of a bf16 row,
 *   amax = max |x| (NaN skipped),  d = amax / 127,  id = d != 0 ? 1 / d : 0,
 *   q = round-half-away-from-zero(x * id), NaN -> 0, clamped to [-127, 127]
 * each a single binary32 operation; the stored scale is d rounded to fp16
 * (Q8_0) or d itself (Q8_K).  Bit-exact.
 *   x       bf16 [R, K], 16-byte aligned; K a multiple of the block
 *   codes   int8 [R, K] out, 16-byte aligned
 *   scales  f32 [R, K / block] out, 4-byte aligned
 *
 * moe_grouped_gemm_q -- the plain grouped op: for every group g and row r in
 * [group_offsets[g], group_offsets[g+1]):
 *   out[r, n] = sum over the blocks b of the row of
 *     Q8_0: d_w[b] * d_x[b] * sum_i q_w[i] * q_x[i]
 *     Q4_K: d_x[b] * (d * sum_j sc_j * sum_i q_ij * q_x,ij  -  dmin * sum_j m_j * sum_i q_x,ij)
 * with exact integer block sums and f32 accumulation over the blocks.
 *   a_codes, a_scales  quantized activations ([a_rows, K], [a_rows, K/block]),
 *                      from moe_quantize_act_q8 with the same qfmt
 *   a_row_gather       int32 [P] or NULL: row r reads activation row
 *                      a_row_gather[r] / gather_div (an index outside
 *                      [0, a_rows) reads zeros); NULL: row r reads row r
 *   w                  uint8 [G, N, K / block * bytes], 16-byte aligned
 *   group_offsets      int32 [G+1], read on the device, values clamped to [0, P];
 *                      NULL allowed when G == 1
 *   out                f32 [P, N]; rows outside every group are not written
 *   P >= 0, N >= 1, K a multiple of 256 and at most 16384, 1 <= G <= 1024
 *
 * moe_grouped_gemm_gateup_silu_q -- the keep-quant gate/up: the sums above for
 * gate rows n and up rows I + n of w13 [G, 2I, H / block * bytes], then the
 * epilogue of moe_grouped_gemm_gateup_silu_bf16 (both narrowed to bf16 before
 * silu(g) * u), act bf16 [P, I].  Same row gather as above.
 *
 * moe_grouped_gemm_down_q -- the keep-quant down projection: the sums above
 * with w2 [G, H, I / block * bytes] and activations [P, I] in row order, then
 * the epilogue of moe_grouped_gemm_down_bf16: one f32 multiply by
 * pair_weight[dst] (when given), one bf16 rounding, stored at row dst =
 * row_to_pair ? row_to_pair[r] : r of out bf16 [P, H] (a dst outside [0, P) is
 * skipped).
 *
 * Errors of the quantizer and the three GEMMs: MOE_ERR_ARG (qfmt, sizes, NULL
 * operands), MOE_ERR_ALIGN (alignment; quantizer K not a multiple of its
 * block; GEMM K not a multiple of 256 or above 16384), MOE_ERR_CUDA.  No
 * workspace.
 *
 * moe_dequantize_q_bf16 -- keep-quant weight rows expanded to bf16, for
 * batches with many rows per expert, which run faster on the bf16 tensor-core
 * GEMMs: each value formed in binary32 and rounded to bf16 once,
 *   Q8_0: bf16(d * q)        Q4_K: bf16((d * sc_j) * q - dmin * m_j)
 * (exact products, one rounded subtraction).  Bit-exact.
 *   w      uint8 [rows, K / block * bytes]: any stack of weight rows, e.g. a
 *          whole [G, R, K] matrix as rows = G * R; Q4_K blocks 16-byte
 *          aligned, Q8_0 blocks 2-byte aligned
 *   qfmt   MOE_QFMT_Q8_0 or MOE_QFMT_Q4_K
 *   rows   >= 0 (0: no-op); K >= 1, a multiple of the block (32 or 256)
 *   out    bf16 [rows, K] out, 16-byte aligned
 * Errors: MOE_ERR_ARG (qfmt, rows < 0, K < 1, NULL operands, more than
 * 2^31 - 1 launch blocks), MOE_ERR_ALIGN (alignment, K not a multiple of the
 * block), MOE_ERR_CUDA.  No workspace.
 * ---------------------------------------------------------------------- */
enum { MOE_QFMT_Q8_0 = 1, MOE_QFMT_Q4_K = 2 };
int moe_quantize_act_q8(const void* x_bf16, int R, int K, int qfmt, int8_t* codes, float* scales,
                        void* stream);
int moe_grouped_gemm_q(const int8_t* a_codes, const float* a_scales, int a_rows,
                       const int32_t* a_row_gather, int gather_div, const uint8_t* w, int qfmt,
                       const int32_t* group_offsets, int P, int K, int N, int G, float* out_f32,
                       void* stream);
int moe_grouped_gemm_gateup_silu_q(const int8_t* a_codes, const float* a_scales, int a_rows,
                                   const int32_t* a_row_gather, int gather_div,
                                   const uint8_t* w13, int qfmt, const int32_t* group_offsets,
                                   int P, int H, int I, int G, void* act_bf16, void* stream);
int moe_grouped_gemm_down_q(const int8_t* a_codes, const float* a_scales, const uint8_t* w2,
                            int qfmt, const int32_t* group_offsets, const float* pair_weight,
                            const int32_t* row_to_pair, int P, int I, int H, int G,
                            void* out_bf16, void* stream);
int moe_dequantize_q_bf16(const uint8_t* w, int qfmt, long long rows, int K, void* out_bf16,
                          void* stream);

/* ------------------------------------------------------------------------
 * moe_combine -- kMoeCombine of [PR509].  Per output element, sequentially:
 *   acc = +0.0f
 *   for k = 0 .. K-1:  acc = acc + (w ? f32(eo[t,k,c]) * w[t,k] : f32(eo[t,k,c]))
 *   acc = acc * routed_scale
 *   if shared: acc = acc + f32(shared[t,c])
 *   out[t,c] = acc rounded once to out_dtype
 * Every operation is a separately rounded binary32 op (no fused multiply-add),
 * so the result is bit-exact against the sequential definition.  In the
 * expert block the down GEMM already applied the weights: pass w = NULL.
 *
 *   expert_out  [T,K,H] f32 or bf16 (eo_dtype)
 *   w           f32 [T,K] or NULL
 *   shared      [T,H] f32 or bf16 (sh_dtype) or NULL
 *   out         [T,H] f32 or bf16 (out_dtype)
 *   T >= 0, 1 <= K <= 64, H > 0 multiple of 8
 * Errors: MOE_ERR_DTYPE (a dtype other than f32 or bf16; f16 is named),
 * MOE_ERR_ARG (T < 0; K outside [1, 64]; H <= 0; T*H too large; NULL expert_out
 * or out), MOE_ERR_ALIGN (H not a multiple of 8; expert_out, shared or out not
 * 16-byte aligned), MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
int moe_combine(const void* expert_out, int eo_dtype, const float* w, const void* shared,
                int sh_dtype, float routed_scale, int T, int K, int H, void* out, int out_dtype,
                void* stream);

/* ------------------------------------------------------------------------
 * moe_combine_gate -- kMoeCombineGate of [PR509]: the combine with the shared
 * expert's sigmoid gate folded in and the gated shared term rounded through
 * bf16 before it is added:
 *   s   = sigmoid(gl[t]) = 1 / (1 + expf_cr(-gl[t]))
 *   sv  = f32( bf16( s * f32(sd[t,c]) ) )
 *   acc = the routed sum of moe_combine (w optional), acc = acc * routed_scale
 *   out[t,c] = (acc + sv) rounded once to out_dtype
 * Bit-exact.  sd f32 or bf16; out f32 or bf16; gl f32 [T].
 * workspace: NULL, or >= moe_gate_workspace_size(T) bytes.  With a workspace
 * the T sigmoids are evaluated first by a small kernel and the stream reads
 * them (faster: each sigmoid is evaluated once, not once per block); without
 * one each block evaluates the sigmoids of its tokens itself.  Same bits.
 * Errors: those of moe_combine (sd and gl required), MOE_ERR_WORKSPACE and
 * MOE_ERR_ALIGN for a workspace below moe_gate_workspace_size or not 16-byte
 * aligned.
 * ---------------------------------------------------------------------- */
int moe_combine_gate(const void* expert_out, int eo_dtype, const float* w, const void* sd,
                     int sd_dtype, const float* gl, float routed_scale, int T, int K, int H,
                     void* out, int out_dtype, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * shared_expert_gate -- kSharedExpertGate of [PR509]:
 *   out[t,c] = sigmoid(gl[t]) * sd[t,c], one rounding to out_dtype.
 * Four dtype arms: sd f32/bf16 x out f32/bf16.  Bit-exact.  workspace as
 * for moe_combine_gate (NULL allowed).
 * Errors: MOE_ERR_DTYPE, MOE_ERR_ARG (T < 0; H <= 0; NULL sd, gl or out),
 * MOE_ERR_ALIGN (H not a multiple of 8; sd or out not 16-byte aligned; the
 * workspace), MOE_ERR_WORKSPACE, MOE_ERR_CUDA.
 * ---------------------------------------------------------------------- */
int shared_expert_gate(const void* sd, int sd_dtype, const float* gl, int T, int H, void* out,
                       int out_dtype, void* workspace, size_t ws_bytes, void* stream);
size_t moe_gate_workspace_size(int T); /* for moe_combine_gate and shared_expert_gate */

/* ------------------------------------------------------------------------
 * Introspection (not on the hot path; these synchronise the device).
 *
 * moe_device_status: reads and optionally clears the library's device status
 * word, a bit set of MOE_STATUS_* raised by kernels (a bounded wait that ran
 * out, an out-of-range expert id).  Returns MOE_OK or MOE_ERR_CUDA.
 *
 * moe_launch_counts: copies the per-kernel launch counters (incremented by
 * each kernel on the device, so they count kernels that actually ran) into
 * counts[0 .. n-1], indexed by MOE_KID_*; returns the number of counters.
 * ---------------------------------------------------------------------- */
enum { MOE_STATUS_TIMEOUT = 1, MOE_STATUS_BAD_ID = 2 };
enum {
  MOE_KID_ROUTE_LOGITS = 0,
  MOE_KID_ROUTE_TOPK = 1,
  MOE_KID_PERMUTE_COUNT = 2,
  MOE_KID_PERMUTE_SCAN = 3,
  MOE_KID_PERMUTE_PLACE = 4,
  MOE_KID_PERMUTE_GATHER = 5,
  MOE_KID_GEMM_GATEUP = 6,
  MOE_KID_GEMM_DOWN = 7,
  MOE_KID_COMBINE = 8,
  MOE_KID_COMBINE_GATE = 9,
  MOE_KID_SHARED_GATE = 10,
  MOE_KID_GATE_SIGMOID = 11,  /* the sigmoid pre-pass of the gate ops (workspace given) */
  MOE_KID_PERMUTE_SMALL = 12, /* count + scan + place in one block (P <= 4096) */
  MOE_KID_QUANT_ACT = 13,     /* moe_quantize_act_q8 */
  MOE_KID_GEMM_Q = 14,        /* moe_grouped_gemm_q */
  MOE_KID_GEMM_Q_GATEUP = 15, /* moe_grouped_gemm_gateup_silu_q */
  MOE_KID_GEMM_Q_DOWN = 16,   /* moe_grouped_gemm_down_q */
  MOE_KID_DEQUANT_Q = 17,     /* moe_dequantize_q_bf16 */
  MOE_KID_EXP_SIGMOID = 18,   /* moe_exp_sigmoid_f32 */
  MOE_KID_COUNT = 20
};
int moe_device_status(int* status_out, int clear);
int moe_launch_counts(unsigned long long* counts, int n);

/* moe_exp_sigmoid_f32 -- the binary32 exp and sigmoid every bit-exact kernel
 * of the library uses (router weights, sigmoid scoring, the shared-expert
 * gate of [PR509], whose rework requires the gate bit-exact), evaluated on a
 * range of bit patterns so that a caller can check them against another
 * implementation of the same definition:
 *   x_i = the binary32 value with bit pattern (first_bits + i) mod 2^32
 *   exp_out[i] = expf_cr(x_i)                       (see moe_route_topk)
 *   sigmoid_out[i] = 1 / (1 + expf_cr(-x_i))        (two binary32 operations)
 * for i in [0, n).  Either output may be NULL; f32 arrays, 4-byte aligned.
 * 0 <= n <= 2^32.  Errors: MOE_ERR_ARG (n outside that range; both outputs
 * NULL), MOE_ERR_ALIGN, MOE_ERR_CUDA. */
int moe_exp_sigmoid_f32(uint32_t first_bits, long long n, float* exp_out, float* sigmoid_out,
                        void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
