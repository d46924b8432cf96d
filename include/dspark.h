/*
 * dspark.h -- C ABI of the GB300 (sm_103a) DSpark verify planner, ragged
 * verify pack, greedy / cap / sampling accept, compact-to-strided scatter and
 * calibration library (libdspark.so).
 *
 * Pages cited below (by title and section):
 *   [AVS]   "DSpark 自适应 Verify 怎样分配候选预算" -- DSpark adaptive
 *           verify: how the candidate budget is allocated
 *   [ROUND] "DeepSeek-V4 DSpark一轮 Draft、Verify、Accept 与 Commit" -- one
 *           DSpark round: draft, verify, accept and commit
 *   [SGL]   "DSpark接入SGLang：用置信度驱动可变长度验证" -- DSpark in SGLang
 *   [TUT]   charlestar.github.io tutorial "DSpark confidence-scheduled
 *           speculative decoding"
 *
 * Conventions shared by every entry point
 *   - Every pointer is DEVICE memory unless its comment says "host".
 *   - The caller owns every buffer; the library allocates nothing.  Scratch
 *     comes from a caller-provided device workspace whose size the matching
 *     *_workspace_bytes() function returns (256-byte aligned pointer).
 *   - All work is enqueued asynchronously on `stream` (a cudaStream_t passed
 *     as void*; NULL = the legacy default stream).  No call synchronises the
 *     host; every result, including the budget, stays in device memory.
 *   - Return value: DSPARK_OK or a negative DSPARK_ERR_* code.  Argument
 *     checks happen on the host before anything is enqueued, so a rejected
 *     call has no effect on the device.
 *   - `status` (device int32[1], zeroed by the caller) collects
 *     DSPARK_STATUS_* bits that the kernels OR in for conditions only the
 *     device can see.  Kernels never trap or assert; their only waits on
 *     memory (the scatter's copy barriers) give up after 200 ms and set
 *     DSPARK_STATUS_TIMEOUT.
 *   - Calls are stateless and thread-safe; concurrent calls must not share
 *     workspaces.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DSPARK_API __attribute__((visibility("default")))
#else
#define DSPARK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- errors */
#define DSPARK_OK               0
#define DSPARK_ERR_INVALID_ARG (-1) /* null pointer, size or range violation */
#define DSPARK_ERR_WORKSPACE   (-2) /* workspace missing, too small or misaligned */
#define DSPARK_ERR_CUDA        (-3) /* a CUDA launch or attribute call failed */
#define DSPARK_ERR_UNSUPPORTED (-4) /* outside the supported envelope (see each call) */

/* device status bits (OR-ed into *status) */
#define DSPARK_STATUS_CAPACITY    1  /* a row count exceeded the buffer's capacity */
#define DSPARK_STATUS_TOKEN_RANGE 2  /* a draft token outside [0, V) */
#define DSPARK_STATUS_NAN_LOGIT   4  /* a NaN in a target-logits row (NaN never wins the argmax) */
#define DSPARK_STATUS_BAD_INPUT   8  /* a NaN confidence logit or a temperature that is not > 0 */
#define DSPARK_STATUS_BAD_LEN     16 /* a verify length / cu_seqlens range outside [1, gamma+1] */
#define DSPARK_STATUS_BAD_COST    32 /* cost table not ascending, or a non-positive / non-finite cost used */
#define DSPARK_STATUS_INFEASIBLE  64 /* no budget in range: budget set to 0 */
#define DSPARK_STATUS_BAD_INDEX   128 /* a packed row's strided destination outside the buffer */
#define DSPARK_STATUS_TIMEOUT     256 /* a kernel's bounded wait gave up (its outputs are incomplete) */
#define DSPARK_STATUS_BAD_TIER    512 /* a shared verify tier below this rank's packed rows */
/* Set only by the bounds-checked build (libdspark_checked.so, compiled with
 * -DDSPARK_CHECKED): an index a kernel computed from data fell outside the
 * buffer (global or shared memory) it addresses; the access was skipped.  It
 * always marks a defect of the library, never of the inputs.  The normal
 * build carries no such checks and never sets it. */
#define DSPARK_STATUS_OUT_OF_BOUNDS 1024

/* Message for a DSPARK_ERR_* code (static string). */
DSPARK_API const char *dspark_strerror(int code);

/* Library version: major*10000 + minor*100 + patch. */
DSPARK_API int dspark_version(void);

/* 1 in the bounds-checked build (see DSPARK_STATUS_OUT_OF_BOUNDS), 0 in the
 * normal one.  The two builds export the same calls with the same results. */
DSPARK_API int dspark_checked_build(void);

/* ---------------------------------------------------------------- planner */

#define DSPARK_COST_SPS_1D   0
#define DSPARK_COST_ADDITIVE 1
#define DSPARK_COST_ADDITIVE_INTERP 2

/* Planner parameters (host struct).  [AVS] §一: ScheduleVerifyLensTopk is
 * bounded by min_verify_len, max_verify_len and survival_eps. */
typedef struct {
    int32_t B;              /* requests in this planner decision, >= 1 */
    int32_t gamma;          /* draft tokens per request, 1..31 */
    float survival_eps;     /* candidates with survival < eps are dropped; in [2^-14, 1] */
    int32_t min_verify_len; /* 1 <= min <= max */
    int32_t max_verify_len; /* <= gamma + 1; depths >= max-1 are never candidates */
    int32_t forced_budget;  /* < 0: budget = argmax theta; >= 0: this budget, clipped to range */
} dspark_plan_params;

/* Step-cost table (host struct pointing at DEVICE arrays M[n], val[n]).
 *   DSPARK_COST_SPS_1D ([AVS] §一 and §四 "1D SpsCostTable"):
 *     theta(b) = tau(b) * SPS(B + b); SPS is a floor lookup -- the sample
 *     with the largest M_j <= B + b, sample 0 below the first -- with no
 *     interpolation.  val = steps per second, must be > 0.
 *   DSPARK_COST_ADDITIVE ([AVS] §一/§四 "Additive SPS"; [TUT] T(bs,K)):
 *     theta(b) = tau(b) / T, T = (bias_ms + alpha_ms) + val[j] with j the
 *     smallest graph tier M_j >= B + b; budgets above the largest tier are
 *     infeasible.  alpha_ms is alpha(B) already evaluated for this B.
 *   DSPARK_COST_ADDITIVE_INTERP ([AVS] §四 "三个关键假设", the third: the
 *     exported additive table interpolates theta(M) linearly at runtime):
 *     T = (bias_ms + alpha_ms) + theta(B + b), with M_j <= M < M_{j+1}
 *     theta(M) = val[j] + (M - M_j) * slope_j, slope_j = (val[j+1] - val[j])
 *     / (M_{j+1} - M_j), in that fp64 order; val[j] at M = M_j; val[0] below
 *     M_0; budgets with B + b above the last sample are infeasible.  Every
 *     budget has its own cost, so theta is evaluated at every in-range
 *     budget (one fp64 division each, on one CTA).
 *   M must be strictly ascending (else DSPARK_STATUS_BAD_COST, all budgets
 *   infeasible).  A used entry whose SPS or T is not a positive finite
 *   number is infeasible and flagged DSPARK_STATUS_BAD_COST. */
typedef struct {
    int32_t kind;          /* DSPARK_COST_SPS_1D, _ADDITIVE or _ADDITIVE_INTERP */
    int32_t n;             /* entries, >= 1 */
    const int32_t *M;      /* device [n]: total verify rows (1-D) or graph tiers (additive) */
    const double *val;     /* device [n]: SPS (steps/s) or token-side cost theta(M) in ms */
    double bias_ms;        /* additive only */
    double alpha_ms;       /* additive only */
} dspark_cost_table;

/* Device scratch of one planner call: about 24 * B * gamma + 4 * B + 25 KB
 * (a completion counter, a 2048-bin histogram of the survivals, candidate
 * ranks, the sorted survivals and their prefix sums, and what passes of one
 * call hand over).  The workspace must be zero-filled
 * once before its first dspark_plan call (cudaMemset); every call that
 * returns DSPARK_OK leaves the histogram zero again, and a call that
 * returns DSPARK_ERR_CUDA after launching clears it on the stream, so the
 * buffer can be passed unchanged to the next call.  Do not reuse it for
 * other data between planner calls. */
DSPARK_API size_t dspark_plan_workspace_bytes(int32_t B, int32_t gamma);

/* The verify planner.  [AVS] §一 (budget by survival, tau, theta, argmax,
 * ScheduleVerifyLensTopk), §二 (STS c = sigmoid(z / T), S_k = prod c);
 * [ROUND] §三 (resolve_verify_token_budget, schedule_layout).
 *   conf_logits  [B, gamma] fp32 row-major: confidence-head logits z
 *   sts_temps    [gamma] fp32: per-depth STS temperature T_k > 0
 *   p, cost      host structs (above); cost->M / cost->val are device arrays
 *   survivals    out [B, gamma] fp32: S_k = prod_{i<=k} sigmoid(z_i / T_i),
 *                fp32 sequential product, 0 where S_k < eps
 *   verify_lens  out [B] int32: 1 (root) + candidates selected for the
 *                request, clamped to [min_verify_len, max_verify_len]
 *   budget       out [1] int32: extra verify rows b (argmax or forced)
 *   tau_theta    out [2] fp64: tau(budget) = B + sum of the budget largest
 *                survivals (exact), theta(budget) (0 if the budget is infeasible)
 * Candidates are ordered by survival descending, then depth ascending,
 * then request id ascending; theta ties go to the smaller budget.
 * Errors: INVALID_ARG (null pointer, B < 1, min/max out of order, cost n < 1
 * or unknown kind); UNSUPPORTED (gamma > 31, B*(gamma+1) > 65536,
 * B*gamma > 16384, eps outside [2^-14, 1]); WORKSPACE (missing, smaller than
 * dspark_plan_workspace_bytes(B, gamma) or not 256-byte aligned); CUDA.
 * Device flags: BAD_INPUT, BAD_COST, INFEASIBLE. */
DSPARK_API int dspark_plan(const float *conf_logits, const float *sts_temps,
                const dspark_plan_params *p /* host */, const dspark_cost_table *cost /* host */,
                float *survivals, int32_t *verify_lens, int32_t *budget, double *tau_theta,
                void *workspace, size_t workspace_bytes, int32_t *status, void *stream);

/* Options of the planner ([AVS] §三, the conditions under which the
 * executed budget departs from the plain plan).  Every field may be left
 * zero / NULL.
 *   conf_generation, req_generation  device [B] int32, both or neither: a
 *       request whose confidences were recorded for another generation of
 *       its pool slot plans with survivals of 1 at every depth (optimistic;
 *       [AVS] §三 "req_generation")
 *   lagged_conf_logits  device [B, gamma] fp32: the budget is chosen from
 *       these (lagged) confidences, then allocated over the current ones by
 *       the same ordering, as with a forced budget ([AVS] §三, overlap
 *       scheduler: lagged confidence sets the budget, the current one the
 *       allocation); tau/theta are reported for the allocation
 *   align_to_tiers  1: graph-tier alignment ([AVS] §三, §五 "paid-padding
 *       reclamation"): with T verify rows at the chosen budget and the
 *       smallest tier >= T, the executed budget takes one more candidate per
 *       spare row of that tier, as long as candidates remain in range; no
 *       tier holds T: unchanged.  Also applies to a forced budget.
 *   host_tiers, n_tiers  host: the tiers for alignment (dspark_plan_ex; the
 *       pack's tiers are used by dspark_plan_pack_ex) */
typedef struct {
    const int32_t *conf_generation;
    const int32_t *req_generation;
    const float *lagged_conf_logits;
    int32_t align_to_tiers;
    const int32_t *host_tiers;
    int32_t n_tiers;
} dspark_plan_options;

/* dspark_plan with options (opt may be NULL: dspark_plan).  Each option adds
 * planner passes over the same workspace: lagged confidences a survival
 * kernel and a pass, alignment a pass.  Errors: those of dspark_plan, and
 * INVALID_ARG for one generation array without the other or alignment
 * without a valid tier list. */
DSPARK_API int dspark_plan_ex(const float *conf_logits, const float *sts_temps,
                   const dspark_plan_params *p /* host */, const dspark_cost_table *cost /* host */,
                   const dspark_plan_options *opt /* host, nullable */, float *survivals,
                   int32_t *verify_lens, int32_t *budget, double *tau_theta, void *workspace,
                   size_t workspace_bytes, int32_t *status, void *stream);

/* ------------------------------------------------------------------ pack */

#define DSPARK_MAX_TIERS 64

/* Front-pack the verify rows and round the total up to a graph tier.
 * [ROUND] §三 (verify ids = [anchor, drafts]; BuildRaggedVerifyWindow /
 * compact_verify_ids), §四 (verify positions); [AVS] §六 (cu_seqlens_q with
 * a leading 0); [SGL] "Ragged verify"; [TUT] "变长批次如何与 CUDA Graph 共存".
 *   anchor [B], draft [B, gamma], prefix_lens [B], verify_lens [B]: int32
 *   host_tiers   host [n_tiers] ascending graph tiers (n_tiers <= 64; 0 = no
 *                rounding)
 *   capacity     rows available in each packed_* buffer
 *   packed_ids/pos/req/src  out [capacity] int32.  Row cu[r]+j (j < len_r):
 *                id = anchor[r] (j = 0) or draft[r][j-1]; pos = prefix_lens[r]
 *                + j; req = r; src = r*(gamma+1) + j (row in the strided
 *                [B, gamma+1] layout).  Rows [total, padded) are pad rows
 *                (0, 0, -1, -1); rows >= padded are not written.
 *   cu_seqlens   out [B+1] int32, cu[0] = 0
 *   totals       out [2] int32: {total, padded}
 * A length outside [1, gamma+1] is clamped and flagged BAD_LEN; rows past
 * capacity are dropped and flagged CAPACITY, as is a total above the
 * largest tier (then padded = total).
 * Errors: INVALID_ARG (null pointer, B < 1, gamma outside 1..31, capacity
 * < 0, n_tiers outside 0..64, tiers not ascending); CUDA. */
DSPARK_API int dspark_pack_verify(const int32_t *anchor, const int32_t *draft, const int32_t *prefix_lens,
                       const int32_t *verify_lens, int32_t B, int32_t gamma,
                       const int32_t *host_tiers /* host */, int32_t n_tiers, int32_t capacity,
                       int32_t *packed_ids, int32_t *packed_pos, int32_t *packed_req,
                       int32_t *packed_src, int32_t *cu_seqlens, int32_t *totals,
                       int32_t *status, void *stream);

/* dspark_plan followed by dspark_pack_verify on the planner's verify_lens,
 * in fewer launches: for cost tables of at most 6143 entries (interpolated:
 * 2048 samples) the planner's last kernel, which runs on one CTA, also packs
 * the window (one launch and one dependency wait fewer per step); larger
 * tables run the two calls' kernels back to back.
 * Arguments and outputs are those of the two calls (the planner's
 * workspace, which must be zero-filled once, serves both); the pages'
 * planner and pack are the same two steps ([AVS] §一, §五-§六; [ROUND]
 * §三).  Errors: those of dspark_plan, then of dspark_pack_verify's
 * arguments (checked before anything is launched). */
DSPARK_API int dspark_plan_pack(const float *conf_logits, const float *sts_temps,
                     const dspark_plan_params *p /* host */, const dspark_cost_table *cost /* host */,
                     float *survivals, int32_t *verify_lens, int32_t *budget, double *tau_theta,
                     const int32_t *anchor, const int32_t *draft, const int32_t *prefix_lens,
                     const int32_t *host_tiers /* host */, int32_t n_tiers, int32_t capacity,
                     int32_t *packed_ids, int32_t *packed_pos, int32_t *packed_req,
                     int32_t *packed_src, int32_t *cu_seqlens, int32_t *totals,
                     void *workspace, size_t workspace_bytes, int32_t *status, void *stream);

/* Scratch of one sampling accept: per-(CTA, row) softmax partials for up
 * to max_rows target rows and B*gamma draft rows, and B+1 offsets. */
DSPARK_API size_t dspark_sampling_workspace_bytes(int32_t max_rows, int32_t B, int32_t gamma);

/* Speculative sampling accept, compact mode ([ROUND] §五 AcceptSampling
 * with chain speculative sampling; [AVS] §一: a draft drawn from q is
 * accepted with probability min(1, p/q)).  The pages leave the rule to the
 * speculative algorithm; this is the textbook one:
 *   p_j = softmax(target row cu[r] + j), q_j = softmax(draft row r*gamma+j)
 *   draft j (token x) is accepted iff u_accept[r][j] * q_j(x) < p_j(x); the
 *   chain stops at the first rejection (correct_len = j)
 *   bonus: inverse-CDF draw with u_bonus[r] -- the smallest token whose
 *   cumulative weight exceeds u * W -- from max(0, p_j - q_j) after a
 *   rejection (from p_j when that residual's mass is below 2^-20), else from the last
 *   row's p; then num_accepted / commit_lens / new_seq_lens / out_tokens as
 *   dspark_greedy_accept.
 *   target_logits  [max_rows, ld_t] bf16 or fp32, draft_logits [B*gamma,
 *                  ld_d] of the same dtype: the proposal logits that produced
 *                  each draft (after any correction)
 *   u_accept [B, gamma], u_bonus [B]: fp32 uniforms in [0, 1) (the caller's
 *                  random numbers)
 * Softmax sums are fp32 per thread and fp64 beyond, the bonus weights are
 * summed exactly in units of 2^-40: a decision can differ from an exact
 * evaluation only within ~1e-6 relative of its threshold.  NaN logits weigh
 * 0 (DSPARK_STATUS_NAN_LOGIT); a draft token outside [0, V) is rejected
 * (TOKEN_RANGE); a bad cu range gives the greedy defaults (BAD_LEN).
 * Errors: INVALID_ARG (null pointer, dtype, B < 1, gamma outside 1..31,
 * V < 1, a stride below V, max_rows < 0); UNSUPPORTED (B > 4096 or
 * V > 2^20); WORKSPACE; CUDA. */
DSPARK_API int dspark_sampling_accept(const void *target_logits, int32_t dtype, int64_t ld_t,
                           int32_t V, int32_t max_rows, const int32_t *cu_seqlens,
                           const void *draft_logits, int64_t ld_d, const int32_t *draft,
                           const int32_t *prefix_lens /* nullable with new_seq_lens */,
                           int32_t B, int32_t gamma, const float *u_accept,
                           const float *u_bonus, int32_t *num_accepted, int32_t *bonus,
                           int32_t *commit_lens, int32_t *new_seq_lens /* nullable */,
                           int32_t *out_tokens, void *workspace, size_t workspace_bytes,
                           int32_t *status, void *stream);

/* dspark_sampling_accept with the draft rows' softmax normalizers supplied
 * by the caller -- the drafting step's sampler has them -- so that the
 * draft rows are not streamed to normalise them (only the target rows are;
 * a rejected request's draft row is still read for the residual bonus):
 *   draft_lse  [B*gamma] fp32 (nullable: dspark_sampling_accept):
 *              log(sum_y exp(z_y)) of draft row r*gamma + j (natural log);
 *              q_j(x) = exp(z_x - draft_lse[r*gamma + j]).  Read for the
 *              tested drafts only.  A non-finite value makes that row's q
 *              zero everywhere.
 * Everything else, including the workspace size, as dspark_sampling_accept. */
DSPARK_API int dspark_sampling_accept_ex(const void *target_logits, int32_t dtype, int64_t ld_t,
                           int32_t V, int32_t max_rows, const int32_t *cu_seqlens,
                           const void *draft_logits, int64_t ld_d, const float *draft_lse,
                           const int32_t *draft, const int32_t *prefix_lens, int32_t B,
                           int32_t gamma, const float *u_accept, const float *u_bonus,
                           int32_t *num_accepted, int32_t *bonus, int32_t *commit_lens,
                           int32_t *new_seq_lens, int32_t *out_tokens, void *workspace,
                           size_t workspace_bytes, int32_t *status, void *stream);

/* ScatterCompactToStrided ([ROUND] §三): after the target forward over the
 * compact verify rows, copy packed row i (i < totals[0]) to row
 * packed_src[i] = r*(gamma+1) + j of the [B x (gamma+1)] strided buffer, so
 * that the accept can address rows by fixed position (cap-accept); pad rows
 * and the strided rows no request selected are left untouched.
 *   src          device [max_rows, ld_src] rows of `width` elements of
 *                elem_bytes (2: bf16 logits or hidden states, 4: fp32)
 *   packed_src   device [max_rows] int32, the pack's output
 *   totals       device [>= 1] int32, totals[0] = real packed rows (clamped
 *                to [0, max_rows])
 *   dst          device [dst_rows, ld_dst], strides in elements
 * TMA bulk copies (16 KB segments staged in shared memory) when both
 * buffers, both strides and the row size are 16-byte multiples, else 2-byte
 * copies.  A destination outside [0, dst_rows) is skipped and flagged
 * DSPARK_STATUS_BAD_INDEX; DSPARK_STATUS_TIMEOUT if a copy did not complete
 * within 200 ms (that CTA then copies nothing more: the rows it had left are
 * not written).
 * Errors: INVALID_ARG (null pointer, elem_bytes not 2 or 4, width < 1, a
 * stride below width, negative row counts); CUDA. */
DSPARK_API int dspark_scatter_compact_to_strided(const void *src, int64_t ld_src, int32_t width,
                                      int32_t elem_bytes, const int32_t *packed_src,
                                      const int32_t *totals, int32_t max_rows, void *dst,
                                      int64_t ld_dst, int32_t dst_rows, int32_t *status,
                                      void *stream);

/* dspark_scatter_compact_to_strided with the limit of one pipeline wait of
 * the TMA path in the caller's hands (no counterpart on the pages: failure
 * detection).
 *   wait_limit_ns  < 0: 200 ms (the default); 0: each wait tests its copy
 *                  once, so a copy not yet landed at the first test gives
 *                  up -- how the tests exercise the give-up path.
 * A CTA that gives up flags DSPARK_STATUS_TIMEOUT, issues nothing more,
 * waits (up to 200 ms each, whatever wait_limit_ns) for the loads it still
 * has in flight and for its stores, and exits; the call returns normally and
 * the rows that CTA had left are not written.  The 2-byte path has no waits. */
DSPARK_API int dspark_scatter_compact_to_strided_ex(const void *src, int64_t ld_src,
                                      int32_t width, int32_t elem_bytes,
                                      const int32_t *packed_src, const int32_t *totals,
                                      int32_t max_rows, void *dst, int64_t ld_dst,
                                      int32_t dst_rows, int64_t wait_limit_ns, int32_t *status,
                                      void *stream);

/* The verify tier shared by data-parallel ranks.  [AVS] §六 "DP / DeepEP
 * 是第二层复杂度" (each rank's local verify tier is gathered and the
 * DP-global max token tier is what every rank replays); [SGL] "Ragged
 * verify" (under DP attention the ranks share one tier, the largest any rank
 * needs).  Each rank packs its own requests (dspark_pack_verify or
 * dspark_plan_pack: totals[1] = its local tier), the ranks take the max of
 * totals[1] (one int32 MAX all-reduce, e.g. NCCL, on the step's stream), and
 * this call pads the rank's window to the result:
 *   pad_to       device [1] int32: the shared tier.  May point at totals + 1
 *                (the all-reduce done in place).
 *   capacity     rows of the packed_* buffers
 *   packed_*     device [capacity], the pack's outputs; rows
 *                [totals[0], min(*pad_to, capacity)) become pad rows (id 0,
 *                position 0, request -1, source -1), other rows untouched
 *   totals       device [2] in/out: totals[0] (real rows) is read,
 *                totals[1] = *pad_to is written
 * A shared tier below totals[0] changes nothing and flags
 * DSPARK_STATUS_BAD_TIER; one above capacity writes up to capacity and flags
 * DSPARK_STATUS_CAPACITY.  No host synchronisation.
 * Errors: INVALID_ARG (null pointer, capacity < 0); CUDA. */
DSPARK_API int dspark_pad_to_tier(const int32_t *pad_to, int32_t capacity, int32_t *packed_ids,
                                  int32_t *packed_pos, int32_t *packed_req, int32_t *packed_src,
                                  int32_t *totals, int32_t *status, void *stream);

/* dspark_plan_pack with options (see dspark_plan_options; alignment uses
 * the pack's tiers). */
DSPARK_API int dspark_plan_pack_ex(const float *conf_logits, const float *sts_temps,
                        const dspark_plan_params *p /* host */,
                        const dspark_cost_table *cost /* host */,
                        const dspark_plan_options *opt /* host, nullable */, float *survivals,
                        int32_t *verify_lens, int32_t *budget, double *tau_theta,
                        const int32_t *anchor, const int32_t *draft, const int32_t *prefix_lens,
                        const int32_t *host_tiers /* host */, int32_t n_tiers, int32_t capacity,
                        int32_t *packed_ids, int32_t *packed_pos, int32_t *packed_req,
                        int32_t *packed_src, int32_t *cu_seqlens, int32_t *totals,
                        void *workspace, size_t workspace_bytes, int32_t *status, void *stream);

/* ---------------------------------------------------------------- accept */

#define DSPARK_DTYPE_BF16 0
#define DSPARK_DTYPE_F32  1

/* Scratch of one accept call over at most max_rows rows. */
DSPARK_API size_t dspark_accept_workspace_bytes(int32_t max_rows, int32_t V);

/* Compact-mode greedy accept.  [ROUND] §五 "Greedy" (target_predict =
 * argmax(target_logits); correct_len = leading drafts equal to the target
 * chain; bonus from the last valid input row; no acceptance past the first
 * mismatch), FinalizeAcceptLens and BuildOutTokens.
 *   logits       [max_rows, ld] bf16 or fp32 (dtype), row stride ld >= V
 *                elements; 16-byte aligned base and ld*elem % 16 == 0 take
 *                the vector path, anything else a scalar path.  Device
 *                memory, or pinned host memory (device-accessible at the
 *                same address under unified addressing): the kernels then
 *                read the packed rows over the host link, with no copy step
 *   cu_seqlens   [B+1]: request r owns packed rows [cu[r], cu[r+1]); rows
 *                = min(cu[B], max_rows) rows are read (CAPACITY if cu[B] >
 *                max_rows)
 *   draft        [B, gamma]; prefix_lens [B] (may be NULL iff new_seq_lens is)
 *   argmax       out [max_rows] (nullable): argmax of every row < rows --
 *                lowest index of the largest non-NaN value, -0 == +0, 0 for
 *                a row with nothing above -inf
 *   num_accepted out [B]: correct_len = first j < L-1 with argmax(row
 *                cu[r]+j) != draft[r][j], else L-1 (L = cu[r+1]-cu[r])
 *   bonus        out [B]: argmax of row cu[r] + correct_len
 *   commit_lens  out [B]: correct_len + 1
 *   new_seq_lens out [B] (nullable): prefix_lens + commit_lens
 *   out_tokens   out [B, gamma+1]: drafts, -1 in column gamma, then the
 *                bonus written at column correct_len
 * A request whose range is empty, longer than gamma+1 or beyond rows gets
 * correct 0, bonus -1, commit 0 (flag BAD_LEN).  Device flags also:
 * TOKEN_RANGE, NAN_LOGIT, CAPACITY.
 * Errors: INVALID_ARG (null pointer, B < 1, gamma outside 1..31, V < 1,
 * ld < V, max_rows < 0, unknown dtype, new_seq_lens without prefix_lens);
 * WORKSPACE; CUDA. */
DSPARK_API int dspark_greedy_accept(const void *logits, int32_t dtype, int64_t ld, int32_t V,
                         int32_t max_rows, const int32_t *cu_seqlens, const int32_t *draft,
                         const int32_t *prefix_lens, int32_t B, int32_t gamma, int32_t *argmax,
                         int32_t *num_accepted, int32_t *bonus, int32_t *commit_lens,
                         int32_t *new_seq_lens, int32_t *out_tokens, void *workspace,
                         size_t workspace_bytes, int32_t *status, void *stream);

/* cap-accept: verify the full block, commit only the window.  [AVS] §三
 * (capped_correct_len = min(raw_correct_len, verify_len - 1)), §五
 * "cap-accept"; [SGL] "三种 verify mode" (commits equal compact's and the
 * full-verify acceptance ceiling is exposed).
 *   logits       [B*(gamma+1), ld] strided verify rows, row r*(gamma+1)+j
 *   verify_lens  [B] (clamped to [1, gamma+1], flag BAD_LEN)
 *   outputs as dspark_greedy_accept, with L = gamma+1 for the raw count:
 *   num_accepted = capped; bonus = argmax of row r*(gamma+1) + capped
 *   ceiling      out [B]: raw correct_len over the full block
 *   totals       out [2] int32: {sum commit_lens, sum (ceiling + 1)}
 * Errors as dspark_greedy_accept. */
DSPARK_API int dspark_cap_accept(const void *logits, int32_t dtype, int64_t ld, int32_t V,
                      const int32_t *verify_lens, const int32_t *draft,
                      const int32_t *prefix_lens, int32_t B, int32_t gamma, int32_t *argmax,
                      int32_t *num_accepted, int32_t *bonus, int32_t *commit_lens,
                      int32_t *new_seq_lens, int32_t *out_tokens, int32_t *ceiling,
                      int32_t *totals, void *workspace, size_t workspace_bytes,
                      int32_t *status, void *stream);

/* ------------------------------------------------ allocation-free accept */

#define DSPARK_STATIC_MAX_ROWS 32768

/* dspark_greedy_accept without a workspace.  The pages have no counterpart:
 * this exists for callers that cannot allocate device memory (embeddings
 * that only pass in buffers they own, runtimes whose device memory is fixed
 * at start-up and that forbid cudaMalloc afterwards).
 *   Arguments, outputs and device flags are those of dspark_greedy_accept,
 *   minus workspace / workspace_bytes.
 *   Scratch: a file-scope device array of (4096 + 32768 + 1) * 8 bytes
 *   rounded up to 256 (~300 KB) that every GPU loading this library holds
 *   until the process exits.  max_rows may be at most DSPARK_STATIC_MAX_ROWS
 *   (else DSPARK_ERR_UNSUPPORTED, nothing enqueued); a device row count
 *   cu_seqlens[B] above max_rows is clamped to max_rows and flags
 *   DSPARK_STATUS_CAPACITY, as in dspark_greedy_accept.
 *   The first call on a device looks up the array's device address with
 *   cudaGetSymbolAddress (and so loads the module on that device) and keeps
 *   it for the life of the process; make that first call on each device
 *   before any stream capture.  cudaDeviceReset unloads the module and makes
 *   the kept address stale: a process that resets a device must not call
 *   this function on that device afterwards.
 *   Every call shares the one array: calls whose kernels may overlap on the
 *   GPU (different streams without ordering) race on it.  The array keeps the
 *   last call's contents; nothing in it needs clearing, because every slot a
 *   call reads is written earlier in the same call.
 *   Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
DSPARK_API int dspark_greedy_accept_static(const void *logits, int32_t dtype, int64_t ld, int32_t V,
                         int32_t max_rows, const int32_t *cu_seqlens, const int32_t *draft,
                         const int32_t *prefix_lens, int32_t B, int32_t gamma, int32_t *argmax,
                         int32_t *num_accepted, int32_t *bonus, int32_t *commit_lens,
                         int32_t *new_seq_lens, int32_t *out_tokens, int32_t *status,
                         void *stream);

/* ------------------------------------------------------------ calibration
 *
 * STS recorder, calibration statistics and the sequential temperature fit.
 *   [AVS] §二 "但 SGLang STS 校准的不是同一个 soft target" (the recorder's
 *   label: prefix_mask = positions < num_correct_drafts) and "STS
 *   更像运行时语义桥" (c_i = sigmoid(z_i / T_i); the fitter picks a
 *   temperature position by position, keeping the cumulative survival of the
 *   positions already fitted, by lowest ECE); §七 A (per-position and
 *   cumulative calibration, ECE, Brier).  [TUT] "为什么置信度必须校准"
 *   (ECE = sum_b |I_b|/n |acc(I_b) - conf(I_b)|), "截短会制造观测盲区"
 *   (positions past a compact window are censored), "置信度质量" (by depth;
 *   reliability diagram; ECE, Brier score or log loss).
 *
 * A recorded sample is one request of one step: its confidence logits
 * z[gamma] (fp32), `correct` = drafts accepted and `tested` = drafts the
 * target checked.  Definitions used by the statistics and the fit:
 *   - tested is clamped to [0, gamma] and correct to [0, tested] (BAD_LEN);
 *   - depth k is observed iff k < tested; its label is y_k = (k < correct);
 *   - flavour 0 (cumulative): prediction S_k = c_0 * ... * c_k (fp32, left
 *     to right, c as in dspark_plan), over observed samples; flavour 1
 *     (per-position): prediction c_k over observed samples with correct >= k
 *     (the prefix survived through k-1); a NaN prediction is left out;
 *   - n_bins equal-width bins over [0, 1]: bin = min(floor(p*n_bins),
 *     n_bins-1); each confidence enters the bin sums as floor(p * 2^32), so
 *     the bin sums are exact integers and ECE = sum_b |L_b 2^32 - C_b| /
 *     (n 2^32) is exact up to its final rounding (within 2^-32 of the
 *     real-number ECE);
 *   - Brier = mean (p - y)^2 and log loss = mean -[y ln p + (1-y) ln(1-p)]
 *     with p clamped to [2^-24, 1 - 2^-24]; each term is evaluated as a pair
 *     of floats (Brier to ~2^-47 relative, the log term to ~2^-43 absolute)
 *     and the sums end in fp64 (deterministic for a given GPU; within ~1e-13
 *     of a sequential fp64 sum);
 *   - a flavour/depth with no sample reports n = 0 and zeros. */

/* STS-calibrated confidences c[r][k] = sigmoid(conf_logits[r][k] /
 * sts_temps[k]) ([AVS] §二, c_i = sigmoid(z_i / T_i)), elementwise over
 * [n_rows, gamma] fp32 -- the same values the planner multiplies into its
 * survivals: IEEE fp32 division, then the fp64 formula 1 / (1 + exp(-t))
 * rounded once to fp32 (evaluated in fp32 arithmetic wherever that
 * certifies the same rounding).  Flags BAD_INPUT for a NaN logit or a
 * temperature that is not > 0.  Errors: INVALID_ARG (null pointer, n_rows <
 * 0, gamma < 1); CUDA. */
DSPARK_API int dspark_sts_confidence(const float *conf_logits, const float *sts_temps,
                                     int64_t n_rows, int32_t gamma, float *conf_out,
                                     int32_t *status, void *stream);

/* Append the selected requests of one step to ring buffers of recorded
 * samples, and optionally write the step's greedy prefix mask.
 *   conf_logits  [B, gamma] fp32 confidence logits of the step
 *   num_correct  [B] accepted drafts (num_accepted of the compact accept, or
 *                the cap-accept ceiling with verify_lens NULL)
 *   verify_lens  [B] (nullable): tested = verify_len - 1, verify_len clamped
 *                to [1, gamma+1] (BAD_LEN); NULL = the full block was tested
 *   select       [B] uint8 (nullable): record request r iff select[r] != 0;
 *                NULL records every request
 *   rec_logits   [capacity, gamma] fp32, rec_correct / rec_tested
 *                [capacity] int32: the ring; the i-th selected request of the
 *                call (request order) goes to slot (*cursor + i) % capacity;
 *                num_correct is stored clamped to [0, tested] (BAD_LEN)
 *   cursor       device uint64[1], advanced by the number selected (so a
 *                captured graph can record every step); when one call
 *                selects more than capacity requests only the last capacity
 *                are written (CAPACITY)
 *   prefix_mask  [B, gamma] uint8 (nullable): (k < clamped num_correct)
 * One CTA; any B.  Errors: INVALID_ARG (null required pointer, B < 1, gamma
 * outside 1..31, capacity < 1); CUDA. */
DSPARK_API int dspark_sts_record(const float *conf_logits, const int32_t *num_correct,
                                 const int32_t *verify_lens, const uint8_t *select, int32_t B,
                                 int32_t gamma, float *rec_logits, int32_t *rec_correct,
                                 int32_t *rec_tested, int64_t capacity, uint64_t *cursor,
                                 uint8_t *prefix_mask, int32_t *status, void *stream);

/* Workspace of dspark_calibration_stats (independent of N); 0 for gamma
 * outside 1..31 or n_bins outside 1..32.  Zero-fill it once before its first
 * use: every call leaves it zeroed again. */
DSPARK_API size_t dspark_calibration_workspace_bytes(int32_t gamma, int32_t n_bins);

/* Calibration of N recorded samples under temperatures sts_temps, by depth.
 *   rec_logits [N, gamma] fp32, rec_correct / rec_tested [N] int32 (may be
 *              NULL when N == 0)
 *   sts_temps  [gamma] fp32 (a value that is not > 0 flags BAD_INPUT and is
 *              used as given)
 *   hist       out [2][gamma][n_bins][3] uint64 (nullable): per flavour,
 *              depth and bin -- count, label sum, confidence sum in 2^-32
 *              units (a reliability diagram)
 *   metrics    out [2][gamma][4] fp64: n, ECE, Brier, log loss
 * Device flags: BAD_INPUT (NaN logit anywhere, temperature not > 0),
 * BAD_LEN.  Errors: INVALID_ARG (null required pointer, N outside
 * 0..2^31-1, gamma outside 1..31, n_bins outside 1..32); WORKSPACE; CUDA. */
DSPARK_API int dspark_calibration_stats(const float *rec_logits, const int32_t *rec_correct,
                                        const int32_t *rec_tested, int64_t N, int32_t gamma,
                                        const float *sts_temps, int32_t n_bins, uint64_t *hist,
                                        double *metrics, void *workspace,
                                        size_t workspace_bytes, int32_t *status, void *stream);

/* Workspace of dspark_sts_fit; 0 outside the envelope.  Zero-fill it once
 * before its first use: every call leaves the part that must be zero zeroed
 * again. */
DSPARK_API size_t dspark_sts_fit_workspace_bytes(int64_t N, int32_t n_temps, int32_t n_bins);

/* Sequential temperature scaling fit.  For depth k = 0, 1, ..., gamma-1 and
 * every grid temperature T_j: the cumulative survival S_k = S_{k-1} *
 * sigmoid(z_k / T_j), with S_{k-1} under the temperatures already chosen,
 * is scored by its ECE (flavour 0 above) over the samples observed at depth
 * k; the lowest ECE * n * 2^32 (an exact integer) wins, ties to the lower
 * grid index.  A depth with no observed sample gets T = 1 and choice -1.
 *   rec_*         as in dspark_calibration_stats (NULL allowed when N == 0)
 *   temp_grid     HOST [n_temps] fp32, each positive and finite
 *   sts_temps_out out [gamma] fp32: the fitted temperatures (grid values)
 *   choice        out [gamma] int32: grid index per depth, -1 = none
 *   ece_curve     out [gamma][n_temps] fp64 (nullable): ECE of every candidate
 *   n_obs         out [gamma] int64 (nullable): samples observed per depth
 * gamma launches (one per depth), N * n_temps fp32-rounded fp64 sigmoids
 * each.  Device flags: BAD_INPUT (NaN logit), BAD_LEN.  Errors: INVALID_ARG
 * (null required pointer, N outside 0..2^31-1, gamma outside 1..31, n_temps outside
 * 1..256, a grid value not positive and finite, n_bins outside 1..32);
 * WORKSPACE; CUDA. */
DSPARK_API int dspark_sts_fit(const float *rec_logits, const int32_t *rec_correct,
                              const int32_t *rec_tested, int64_t N, int32_t gamma,
                              const float *temp_grid /* host */, int32_t n_temps, int32_t n_bins,
                              float *sts_temps_out, int32_t *choice, double *ece_curve,
                              int64_t *n_obs, void *workspace, size_t workspace_bytes,
                              int32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
