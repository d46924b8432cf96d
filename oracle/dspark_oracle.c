/*
 * dspark_oracle.c -- plain, slow, single-threaded CPU oracle for the DSpark
 * verify planner, ragged verify pack, greedy / cap-accept, the scatter of
 * compact rows back to the strided layout, speculative sampling accept, and
 * the calibration side (STS recorder, reliability statistics, sequential
 * temperature fit).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file.  The product path (the CUDA
 * library) never links, calls or executes it, and it shares no code, header,
 * table or helper with that path.
 *
 * Every function restates a definition from the pages it cites, in the order
 * the pages give the steps, with no blocking, fusion or reordering:
 *
 *   [AVS]   "DSpark 自适应 Verify 怎样分配候选预算" (DSpark adaptive verify:
 *           how the candidate budget is allocated), akiyangdev.github.io
 *   [ROUND] "DeepSeek-V4 DSpark一轮 Draft、Verify、Accept 与 Commit" (one
 *           DSpark round: draft, verify, accept and commit), akiyangdev.github.io
 *   [SGL]   "DSpark接入SGLang：用置信度驱动可变长度验证" (DSpark in SGLang:
 *           confidence-driven variable-length verify), yingzheng.com review
 *   [TUT]   charlestar.github.io tutorial "DSpark confidence-scheduled
 *           speculative decoding"
 *
 * Arithmetic: STS division and the survival product in IEEE fp32 (the
 * planner's tensors are fp32 on the pages), the sigmoid in fp64 rounded once
 * to fp32, the tau prefix sum and theta in fp64.  Build with
 * -ffp-contract=off so that no multiply-add is fused.
 *
 * Readings of points the pages leave open (each also listed in the design
 * notes):
 *   R1 sigmoid precision: c = (float)(1 / (1 + exp(-(double)t))).
 *   R2 depths k >= max_verify_len-1 cannot be verified and are not budget
 *      candidates.
 *   R3 tau is summed in fp64; with every kept survival >= 2^-14 and
 *      B + B*gamma <= 2^16 every partial sum is exact.
 *   R4 1-D SPS lookup below the first sample uses sample 0; additive lookup
 *      above the largest tier is infeasible; an entry whose SPS or total step
 *      time is not a positive finite number is infeasible and flagged.
 *   R5 argmax ties go to the smaller budget; a forced budget is clipped to
 *      the largest in-range budget.
 *   R6 clamps to [min_verify_len, max_verify_len] are applied after the
 *      top-b selection.
 *   R7 argmax over a logits row: the lowest index of the largest non-NaN
 *      value, -0 equal to +0; a row with no value above -inf returns 0.
 *   R8 out_tokens[r][gamma] is -1 before the bonus scatter; pad rows carry
 *      id 0, position 0, request -1, source -1.
 *   R29 the interpolated additive table (kind 2): theta(M) linear between
 *      samples in the fp64 order val_j + (M - M_j) * slope_j; val_0 below
 *      the first sample; budgets above the last sample are infeasible.
 *
 * Parity pins: every function below is pinned in the oracle's CPU tests
 * against the pages' worked examples, closed forms or brute force.
 */

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* status flags (the library's device status word uses the same bit values,
 * which are part of the call interface) */
#define ORC_ST_CAPACITY    1
#define ORC_ST_TOKEN_RANGE 2
#define ORC_ST_NAN_LOGIT   4
#define ORC_ST_BAD_INPUT   8
#define ORC_ST_BAD_LEN     16
#define ORC_ST_BAD_COST    32
#define ORC_ST_INFEASIBLE  64
#define ORC_ST_BAD_INDEX   128
#define ORC_ST_BAD_TIER    512

/* ------------------------------------------------------------------ STS */

/* One STS-calibrated conditional confidence: c = sigmoid(z / T).
 * [AVS] §二 "STS 更像运行时语义桥" (runtime formula c_i = sigmoid(z_i / T_i)). */
float orc_sts(float z, float T)
{
    float t = z / T;                               /* fp32 IEEE division */
    double c = 1.0 / (1.0 + exp(-(double)t));      /* reading R1 */
    return (float)c;
}

/* c[r][k] = orc_sts(z[r][k], T[k]) over [n, gamma]; NaN logits and
 * temperatures that are not > 0 flag BAD_INPUT. */
void orc_sts_rows(const float *z, const float *T, int64_t n, int gamma, float *c, int *status)
{
    for (int k = 0; k < gamma; ++k)
        if (!(T[k] > 0.0f)) *status |= ORC_ST_BAD_INPUT;
    for (int64_t i = 0; i < n; ++i)
        for (int k = 0; k < gamma; ++k) {
            float zk = z[(size_t)i * gamma + k];
            if (zk != zk) *status |= ORC_ST_BAD_INPUT;
            c[(size_t)i * gamma + k] = orc_sts(zk, T[k]);
        }
}

/* Prefix survivals S_k = prod_{i<=k} c_i per request, in sequential order.
 * [AVS] §一 (same-request survival is a cumulative product) and §二 (S_k);
 * [TUT] "接受是一件前缀事件" (prefix survival table).
 * s_raw receives the product itself; s_out the product with values below
 * survival_eps set to 0 ([AVS] §三, sixth deviation: eps treats tiny
 * survivals as 0). */
void orc_survival(const float *z, const float *T, int B, int gamma, float eps,
                  float *s_raw, float *s_out, int *status)
{
    for (int k = 0; k < gamma; ++k)
        if (!(T[k] > 0.0f)) *status |= ORC_ST_BAD_INPUT;
    for (int r = 0; r < B; ++r) {
        float run = 0.0f;
        for (int k = 0; k < gamma; ++k) {
            float zk = z[(size_t)r * gamma + k];
            if (zk != zk) *status |= ORC_ST_BAD_INPUT;
            float c = orc_sts(zk, T[k]);
            run = (k == 0) ? c : run * c;
            s_raw[(size_t)r * gamma + k] = run;
            s_out[(size_t)r * gamma + k] = (run >= eps) ? run : 0.0f;
        }
    }
}

/* ---------------------------------------------------------------- plan */

typedef struct { float s; int k; int r; } orc_cand;

/* Global order of candidates: survival descending; equal survivals go to the
 * earlier position, then to the lower request id.  [AVS] §一 (sort from high
 * to low; ties prefer the earlier position, then the request number). */
static int orc_cand_cmp(const void *a, const void *b)
{
    const orc_cand *x = (const orc_cand *)a, *y = (const orc_cand *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    if (x->k != y->k) return x->k < y->k ? -1 : 1;
    if (x->r != y->r) return x->r < y->r ? -1 : 1;
    return 0;
}

/* theta(b) for one budget.  [AVS] §一: 1-D table theta = tau(b) * SPS(B+b);
 * additive table theta = tau(b) / T(B, B+b).  [AVS] §四 "1D SpsCostTable"
 * (floor lookup, no interpolation) and "Additive SPS" (T = bias + alpha(B) +
 * theta(M)); [TUT] "调度器要比较期望收益与边际成本" (M = bs + K).
 * kind 1 looks theta(M) up at the smallest graph tier >= M; kind 2 is the
 * exported additive table's runtime linear interpolation of theta(M)
 * ([AVS] §四 "三个关键假设", the third): with M_j <= M < M_{j+1},
 * theta(M) = val_j + (M - M_j) * slope_j, slope_j = (val_{j+1} - val_j) /
 * (M_{j+1} - M_j), in that fp64 order; val_j itself at M = M_j; val_0 below
 * M_0 and infeasible above the last sample (reading R29).
 * Returns 1 if b is feasible and writes theta; sets *bad when the entry used
 * holds an invalid value (reading R4). */
static int orc_theta(double tau, int B, int b, int kind, int n, const int32_t *M,
                     const double *val, double bias, double alpha, double *theta, int *bad)
{
    long Mv = (long)B + b;
    if (kind == 0) {
        int j = -1;
        for (int i = 0; i < n; ++i)
            if (M[i] <= Mv) j = i;
        if (j < 0) j = 0;
        double sps = val[j];
        if (!(sps > 0.0) || !isfinite(sps)) { *bad = 1; return 0; }
        *theta = tau * sps;
        return 1;
    } else if (kind == 1) {
        int j = -1;
        for (int i = 0; i < n; ++i)
            if (M[i] >= Mv) { j = i; break; }
        if (j < 0) return 0;                       /* above the largest tier */
        double T = (bias + alpha) + val[j];
        if (!(T > 0.0) || !isfinite(T)) { *bad = 1; return 0; }
        *theta = tau / T;
        return 1;
    } else {
        if (Mv > M[n - 1]) return 0;               /* above the last sample */
        double th;
        if (Mv <= M[0]) {
            th = val[0];
        } else {
            int j = 0;                             /* last sample with M_j <= Mv */
            for (int i = 0; i < n; ++i)
                if (M[i] <= Mv) j = i;
            if (M[j] == Mv) {
                th = val[j];
            } else {
                double slope = (val[j + 1] - val[j]) / (double)(M[j + 1] - M[j]);
                th = val[j] + (double)(Mv - M[j]) * slope;
            }
        }
        double T = (bias + alpha) + th;
        if (!(T > 0.0) || !isfinite(T)) { *bad = 1; return 0; }
        *theta = tau / T;
        return 1;
    }
}

/* Budget choice and ScheduleVerifyLensTopk from given survivals (s_raw as
 * produced by orc_survival, i.e. before the eps zeroing).
 *   [AVS] §一: tau(b) = B + sum_{i<=b} s_i over survivals sorted descending;
 *   budget = argmax_b theta(b); ScheduleVerifyLensTopk hands the budget to
 *   requests by the same order; verify_len = root + selected candidates,
 *   bounded by min/max_verify_len and survival_eps.
 * tau_curve / theta_curve / feasible (each of size B*gamma+1) and n_kept are
 * optional diagnostics.  Returns the number of kept candidates. */
int orc_plan_from_survivals(const float *s_raw, int B, int gamma, float eps, int min_len,
                            int max_len, int forced, int kind, int n, const int32_t *M,
                            const double *val, double bias, double alpha, int32_t *verify_lens,
                            int32_t *budget_out, double *tau_theta, double *tau_curve,
                            double *theta_curve, uint8_t *feasible_curve, int *status)
{
    size_t NT = (size_t)B * gamma;
    orc_cand *cand = (orc_cand *)malloc(sizeof(orc_cand) * (NT ? NT : 1));
    double *tau = (double *)malloc(sizeof(double) * (NT + 1));
    double *theta = (double *)malloc(sizeof(double) * (NT + 1));
    uint8_t *feas = (uint8_t *)malloc(NT + 1);
    int32_t *cnt = (int32_t *)calloc((size_t)B, sizeof(int32_t));

    /* candidates: s >= eps (eps drop) and a verifiable depth (reading R2) */
    int N = 0;
    for (int r = 0; r < B; ++r)
        for (int k = 0; k < gamma; ++k) {
            float s = s_raw[(size_t)r * gamma + k];
            if (k < max_len - 1 && s >= eps) {
                cand[N].s = s; cand[N].k = k; cand[N].r = r; ++N;
            }
        }
    qsort(cand, (size_t)N, sizeof(orc_cand), orc_cand_cmp);

    /* tau(b) = B + sum of the b largest survivals, fp64, sequential (R3) */
    tau[0] = (double)B;
    for (int b = 1; b <= N; ++b) tau[b] = tau[b - 1] + (double)cand[b - 1].s;

    /* the cost table must list strictly ascending M */
    int table_ok = n >= 1;
    for (int i = 1; i < n; ++i)
        if (!(M[i] > M[i - 1])) table_ok = 0;
    if (!table_ok) *status |= ORC_ST_BAD_COST;

    int bad = 0;
    for (int b = 0; b <= N; ++b) {
        theta[b] = 0.0;
        feas[b] = table_ok ? (uint8_t)orc_theta(tau[b], B, b, kind, n, M, val, bias, alpha,
                                                &theta[b], &bad)
                           : 0;
    }
    if (bad) *status |= ORC_ST_BAD_COST;

    int budget;
    if (forced < 0) {
        double best = -INFINITY;
        budget = -1;
        for (int b = 0; b <= N; ++b)
            if (feas[b] && theta[b] > best) { best = theta[b]; budget = b; }
        if (budget < 0) { budget = 0; *status |= ORC_ST_INFEASIBLE; }
    } else {
        long b_hi = N;
        if (kind != 0 && n >= 1) {
            long top = (long)M[n - 1] - B;
            if (top < b_hi) b_hi = top;
        }
        if (!table_ok) b_hi = -1;
        if (b_hi < 0) { budget = 0; *status |= ORC_ST_INFEASIBLE; }
        else budget = forced < b_hi ? forced : (int)b_hi;
    }

    for (int i = 0; i < budget; ++i) cnt[cand[i].r] += 1;
    for (int r = 0; r < B; ++r) {
        int len = 1 + cnt[r];
        if (len < min_len) len = min_len;
        if (len > max_len) len = max_len;
        verify_lens[r] = len;
    }
    *budget_out = budget;
    tau_theta[0] = tau[budget];
    tau_theta[1] = feas[budget] ? theta[budget] : 0.0;

    if (tau_curve) memcpy(tau_curve, tau, sizeof(double) * (size_t)(N + 1));
    if (theta_curve) memcpy(theta_curve, theta, sizeof(double) * (size_t)(N + 1));
    if (feasible_curve) memcpy(feasible_curve, feas, (size_t)(N + 1));

    free(cand); free(tau); free(theta); free(feas); free(cnt);
    return N;
}

/* The whole planner: STS + survival, then budget and verify_lens. */
int orc_plan(const float *z, const float *T, int B, int gamma, float eps, int min_len,
             int max_len, int forced, int kind, int n, const int32_t *M, const double *val,
             double bias, double alpha, float *survivals, int32_t *verify_lens,
             int32_t *budget, double *tau_theta, int *status)
{
    size_t NT = (size_t)B * gamma;
    float *s_raw = (float *)malloc(sizeof(float) * (NT ? NT : 1));
    orc_survival(z, T, B, gamma, eps, s_raw, survivals, status);
    int N = orc_plan_from_survivals(s_raw, B, gamma, eps, min_len, max_len, forced, kind, n, M,
                                    val, bias, alpha, verify_lens, budget, tau_theta, NULL, NULL,
                                    NULL, status);
    free(s_raw);
    return N;
}

/* ---------------------------------------------------------------- pack */

/* Front-pack each request's anchor + selected draft prefix into compact
 * verify rows with cu_seqlens, then round the packed total up to the
 * smallest captured graph tier.
 *   [ROUND] §三 (verify ids = [anchor, draft...]; compact ragged layout;
 *   BuildRaggedVerifyWindow / compact_verify_ids), §四 (positions of the
 *   verify window); [AVS] §六 (cu_seqlens_q = [0, 2, 3, 7] for lens
 *   [2, 1, 4]); [SGL] "Ragged verify" (front-pack, round to the nearest
 *   captured tier); [TUT] "变长批次如何与 CUDA Graph 共存" (37 -> 40 etc.).
 * Row cu[r]+j: id = anchor[r] for j = 0, else draft[r][j-1];
 * position = prefix_lens[r] + j; request = r; source = r*(gamma+1) + j. */
void orc_pack(const int32_t *anchor, const int32_t *draft, const int32_t *prefix,
              const int32_t *lens, int B, int gamma, const int32_t *tiers, int n_tiers,
              int capacity, int32_t *ids, int32_t *pos, int32_t *req, int32_t *src,
              int32_t *cu, int32_t *totals, int *status)
{
    cu[0] = 0;
    for (int r = 0; r < B; ++r) {
        int L = lens[r];
        if (L < 1 || L > gamma + 1) {
            *status |= ORC_ST_BAD_LEN;
            L = L < 1 ? 1 : gamma + 1;
        }
        cu[r + 1] = cu[r] + L;
        for (int j = 0; j < L; ++j) {
            int dst = cu[r] + j;
            if (dst >= capacity) { *status |= ORC_ST_CAPACITY; continue; }
            ids[dst] = (j == 0) ? anchor[r] : draft[(size_t)r * gamma + (j - 1)];
            pos[dst] = prefix[r] + j;
            req[dst] = r;
            src[dst] = r * (gamma + 1) + j;
        }
    }
    int total = cu[B];
    int padded = total;
    if (n_tiers > 0) {
        int found = 0;
        for (int i = 0; i < n_tiers; ++i)
            if (tiers[i] >= total) { padded = tiers[i]; found = 1; break; }
        if (!found) *status |= ORC_ST_CAPACITY;
    }
    for (int i = total; i < padded; ++i) {
        if (i >= capacity) { *status |= ORC_ST_CAPACITY; break; }
        ids[i] = 0; pos[i] = 0; req[i] = -1; src[i] = -1;
    }
    totals[0] = total;
    totals[1] = padded;
}

/* Data-parallel ranks replay one shared verify tier: each rank's local tier
 * (the pack's padded total) is gathered and the largest taken, and every
 * rank pads its window to that tier.  [AVS] §六 "DP / DeepEP 是第二层复杂度"
 * (local verify tier -> DP gather -> DP-global max token tier); [SGL]
 * "Ragged verify" (under DP attention all ranks share one tier, the largest
 * any rank needs).  Reading R30: after the rank-local pack, rows
 * [totals[0], pad_to) become pad rows (id 0, position 0, request -1, source
 * -1; reading R13) and totals[1] = pad_to; rows at or past capacity are not
 * written and flag CAPACITY; a shared tier below the rank's real total
 * changes nothing and flags BAD_TIER. */
void orc_pad_to_tier(int pad_to, int capacity, int32_t *ids, int32_t *pos, int32_t *req,
                     int32_t *src, int32_t *totals, int *status)
{
    const int total = totals[0];
    if (pad_to < total) { *status |= ORC_ST_BAD_TIER; return; }
    for (int i = total; i < pad_to; ++i) {
        if (i >= capacity) { *status |= ORC_ST_CAPACITY; break; }
        ids[i] = 0; pos[i] = 0; req[i] = -1; src[i] = -1;
    }
    totals[1] = pad_to;
}

/* -------------------------------------------------------------- accept */

static float orc_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* target_predict = argmax(target_logits) per row ([ROUND] §五 "Greedy"),
 * with the tie and NaN conventions of reading R12. */
void orc_argmax_rows_f32(const float *x, int64_t ld, int V, int rows, int32_t *am, int *status)
{
    for (int i = 0; i < rows; ++i) {
        const float *row = x + (size_t)i * (size_t)ld;
        float best = -INFINITY;
        int idx = 0;
        for (int v = 0; v < V; ++v) {
            float f = row[v];
            if (f != f) { *status |= ORC_ST_NAN_LOGIT; continue; }
            if (f > best) { best = f; idx = v; }
        }
        am[i] = idx;
    }
}

void orc_argmax_rows_bf16(const uint16_t *x, int64_t ld, int V, int rows, int32_t *am, int *status)
{
    for (int i = 0; i < rows; ++i) {
        const uint16_t *row = x + (size_t)i * (size_t)ld;
        float best = -INFINITY;
        int idx = 0;
        for (int v = 0; v < V; ++v) {
            float f = orc_bf16_to_f32(row[v]);
            if (f != f) { *status |= ORC_ST_NAN_LOGIT; continue; }
            if (f > best) { best = f; idx = v; }
        }
        am[i] = idx;
    }
}

static void orc_check_tokens(const int32_t *draft, int B, int gamma, int V, int *status)
{
    for (size_t i = 0; i < (size_t)B * gamma; ++i)
        if (draft[i] < 0 || draft[i] >= V) { *status |= ORC_ST_TOKEN_RANGE; return; }
}

/* Shared tail of both accept modes for one request: given the accepted draft
 * count and the bonus, FinalizeAcceptLens and BuildOutTokens.
 *   [ROUND] §五: commit_lens = correct_len + 1; new_seq_lens = prefix_lens +
 *   commit_lens; out_tokens[:, :gamma] = drafts, then the bonus is scattered
 *   at column correct_len. */
static void orc_finish(int r, int correct, int bonus_tok, const int32_t *draft,
                       const int32_t *prefix, int gamma, int32_t *num_acc, int32_t *bonus,
                       int32_t *commit, int32_t *new_seq, int32_t *out)
{
    num_acc[r] = correct;
    bonus[r] = bonus_tok;
    commit[r] = correct + 1;
    if (new_seq) new_seq[r] = prefix[r] + correct + 1;
    for (int j = 0; j < gamma; ++j) out[(size_t)r * (gamma + 1) + j] = draft[(size_t)r * gamma + j];
    out[(size_t)r * (gamma + 1) + gamma] = -1;
    out[(size_t)r * (gamma + 1) + correct] = bonus_tok;
}

/* Compact-mode greedy accept over argmax rows of the packed window.
 *   [ROUND] §五 "Greedy": correct_len counts the leading drafts equal to the
 *   target chain's argmax; bonus is the prediction of the last valid input
 *   row; no acceptance past the first mismatch ([AVS] §二, prefix_mask;
 *   [TUT] "一次推测解码究竟节省了什么").
 * Request r owns packed rows [cu[r], cu[r+1]); L = cu[r+1]-cu[r] rows verify
 * L-1 drafts.  A request whose range is empty, longer than gamma+1 or past
 * `rows` is flagged BAD_LEN and gets correct 0, bonus -1, commit 0. */
void orc_greedy_finalize(const int32_t *am, int rows, const int32_t *cu, const int32_t *draft,
                         const int32_t *prefix, int B, int gamma, int V, int32_t *num_acc,
                         int32_t *bonus, int32_t *commit, int32_t *new_seq, int32_t *out,
                         int *status)
{
    orc_check_tokens(draft, B, gamma, V, status);
    for (int r = 0; r < B; ++r) {
        int lo = cu[r], hi = cu[r + 1], L = hi - lo;
        if (lo < 0 || hi > rows || L < 1 || L > gamma + 1) {
            *status |= ORC_ST_BAD_LEN;
            num_acc[r] = 0; bonus[r] = -1; commit[r] = 0;
            if (new_seq) new_seq[r] = prefix[r];
            for (int j = 0; j < gamma; ++j)
                out[(size_t)r * (gamma + 1) + j] = draft[(size_t)r * gamma + j];
            out[(size_t)r * (gamma + 1) + gamma] = -1;
            continue;
        }
        int correct = L - 1;
        for (int j = 0; j < L - 1; ++j)
            if (am[lo + j] != draft[(size_t)r * gamma + j]) { correct = j; break; }
        orc_finish(r, correct, am[lo + correct], draft, prefix, gamma, num_acc, bonus, commit,
                   new_seq, out);
    }
}

/* cap-accept: the full block is verified (rows r*(gamma+1)+j), the raw
 * acceptance is the ceiling, and only the window commits:
 * capped = min(raw, verify_len - 1).
 *   [AVS] §三 "Cap 本身也没有破坏这个推导" and §五 "cap-accept" (lens
 *   [2,1,4] at width 4 cap the drafts to [1,0,3]); [SGL] "三种 verify mode"
 *   (same commits as compact, exposes the acceptance ceiling).
 * totals[0] = sum of commit_lens, totals[1] = sum of (ceiling + 1). */
void orc_cap_finalize(const int32_t *am, const int32_t *lens, const int32_t *draft,
                      const int32_t *prefix, int B, int gamma, int V, int32_t *num_acc,
                      int32_t *bonus, int32_t *commit, int32_t *new_seq, int32_t *out,
                      int32_t *ceiling, int32_t *totals, int *status)
{
    orc_check_tokens(draft, B, gamma, V, status);
    int sum_commit = 0, sum_ceiling = 0;
    for (int r = 0; r < B; ++r) {
        int base = r * (gamma + 1);
        int raw = gamma;
        for (int j = 0; j < gamma; ++j)
            if (am[base + j] != draft[(size_t)r * gamma + j]) { raw = j; break; }
        int len = lens[r];
        if (len < 1 || len > gamma + 1) {
            *status |= ORC_ST_BAD_LEN;
            len = len < 1 ? 1 : gamma + 1;
        }
        int capped = raw < len - 1 ? raw : len - 1;
        orc_finish(r, capped, am[base + capped], draft, prefix, gamma, num_acc, bonus, commit,
                   new_seq, out);
        ceiling[r] = raw;
        sum_commit += capped + 1;
        sum_ceiling += raw + 1;
    }
    totals[0] = sum_commit;
    totals[1] = sum_ceiling;
}


/* ScatterCompactToStrided ([ROUND] §三): after the target forward, packed
 * row i (i < min(total, max_rows)) goes back to row src_of[i] =
 * r*(gamma+1) + j of the [B x (gamma+1)] strided layout; every other strided
 * row is left as it was.  Rows are row_bytes bytes, strides in bytes.  A
 * destination outside [0, dst_rows) is skipped and flagged. */
void orc_scatter_rows(const unsigned char *src, long long ld_src, long long row_bytes,
                      const int32_t *src_of, int total, int max_rows, unsigned char *dst,
                      long long ld_dst, int dst_rows, int *status)
{
    int rows = total < 0 ? 0 : (total > max_rows ? max_rows : total);
    for (int i = 0; i < rows; ++i) {
        int d = src_of[i];
        if (d < 0 || d >= dst_rows) {
            *status |= ORC_ST_BAD_INDEX;
            continue;
        }
        for (long long b = 0; b < row_bytes; ++b)
            dst[(long long)d * ld_dst + b] = src[(long long)i * ld_src + b];
    }
}

/* ------------------------------------------------------------ sampling
 *
 * Speculative sampling accept: [ROUND] §五 names
 * the path (AcceptSampling: chain speculative sampling over the draft's
 * proposal probabilities -- the corrected ones that actually produced the
 * drafts -- and the target probabilities, giving correct_len and the bonus)
 * and leaves the rule to the speculative algorithm; [AVS] §一 states its
 * classic form: a draft x drawn from q is accepted with probability
 * min(1, p(x)/q(x)), so the mean acceptance is sum_x min(p, q) = 1 - TV.
 * Written out here as the textbook rule: accept draft j iff u_j * q_j(x) <
 * p_j(x); at the first rejection the bonus is drawn from the residual
 * max(0, p_j - q_j) (normalised); when every draft is accepted, from the
 * last row's p.  The draws are inverse-CDF draws with one uniform per
 * request: the smallest token whose cumulative weight exceeds u * W.  A
 * residual of total mass below 2^-20 (p == q up to the precision any
 * implementation of the softmax sums resolves) is read as empty: draw from
 * p.
 *
 * Arithmetic: logits are fp32 (bf16 widened exactly); m = the row's largest
 * non-NaN logit; e_y = expf(z_y - m) in fp32 (NaN logits weigh 0 and are
 * flagged); S = sum of e_y in fp64 in index order; p_y = e_y / S in fp64.
 */

/* m and S of one row (S in fp64, index order). */
static double orc_row_norm(const float *z, int V, float *m_out, int *status)
{
    float m = -INFINITY;
    for (int y = 0; y < V; ++y) {
        if (z[y] != z[y]) { *status |= ORC_ST_NAN_LOGIT; continue; }
        if (z[y] > m) m = z[y];
    }
    double S = 0.0;
    for (int y = 0; y < V; ++y)
        if (z[y] == z[y]) S += (double)expf(z[y] - m);
    *m_out = m;
    return S;
}

static double orc_prob(const float *z, int y, float m, double S)
{
    if (z[y] != z[y] || !(S > 0.0)) return 0.0;
    return (double)expf(z[y] - m) / S;
}

void orc_sampling_accept(const float *tgt, int64_t ld_t, int V, int rows_avail, const int32_t *cu,
                         const float *dft, int64_t ld_d, const int32_t *draft,
                         const int32_t *prefix, int B, int gamma, const float *u_acc,
                         const float *u_bonus, int32_t *num_acc, int32_t *bonus,
                         int32_t *commit, int32_t *new_seq, int32_t *out, int *status)
{
    orc_check_tokens(draft, B, gamma, V, status);
    /* NaN logits are flagged in every packed target row and in every draft
     * row a test of a valid request reads, whether or not the chain gets
     * there */
    for (int i = 0; i < rows_avail; ++i)
        for (int y = 0; y < V; ++y)
            if (tgt[(size_t)i * (size_t)ld_t + y] != tgt[(size_t)i * (size_t)ld_t + y])
                *status |= ORC_ST_NAN_LOGIT;
    for (int r = 0; r < B; ++r) {
        const int lo = cu[r], hi = cu[r + 1], L = hi - lo;
        if (lo < 0 || hi > rows_avail || L < 1 || L > gamma + 1) continue;
        for (int j = 0; j < L - 1; ++j)
            for (int y = 0; y < V; ++y) {
                const float z = dft[((size_t)r * gamma + j) * (size_t)ld_d + y];
                if (z != z) *status |= ORC_ST_NAN_LOGIT;
            }
    }
    double *w = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    for (int r = 0; r < B; ++r) {
        const int lo = cu[r], hi = cu[r + 1], L = hi - lo;
        if (lo < 0 || hi > rows_avail || L < 1 || L > gamma + 1) {
            *status |= ORC_ST_BAD_LEN;
            num_acc[r] = 0;
            bonus[r] = -1;
            commit[r] = 0;
            if (new_seq) new_seq[r] = prefix[r];
            for (int j = 0; j < gamma; ++j) out[(size_t)r * (gamma + 1) + j] = draft[(size_t)r * gamma + j];
            out[(size_t)r * (gamma + 1) + gamma] = -1;
            continue;
        }
        /* acceptance, draft by draft; the chain stops at the first rejection */
        int correct = L - 1;
        for (int j = 0; j < L - 1; ++j) {
            const int x = draft[(size_t)r * gamma + j];
            const float *zt = tgt + (size_t)(lo + j) * (size_t)ld_t;
            const float *zd = dft + ((size_t)r * gamma + j) * (size_t)ld_d;
            float mt, md;
            const double St = orc_row_norm(zt, V, &mt, status);
            const double Sd = orc_row_norm(zd, V, &md, status);
            double p = 0.0, q = 0.0;
            if (x >= 0 && x < V) {
                p = orc_prob(zt, x, mt, St);
                q = orc_prob(zd, x, md, Sd);
            }
            if (!((double)u_acc[(size_t)r * gamma + j] * q < p)) { correct = j; break; }
        }
        /* the bonus: residual of row `correct` after a rejection, else p of the last row */
        const float *zt = tgt + (size_t)(lo + correct) * (size_t)ld_t;
        float mt, md = 0.0f;
        const double St = orc_row_norm(zt, V, &mt, status);
        const int rejected = correct < L - 1;
        const float *zd = rejected ? dft + ((size_t)r * gamma + correct) * (size_t)ld_d : NULL;
        const double Sd = rejected ? orc_row_norm(zd, V, &md, status) : 0.0;
        double W = 0.0;
        for (int y = 0; y < V; ++y) {
            double p = orc_prob(zt, y, mt, St);
            double v = p;
            if (rejected) {
                v = p - orc_prob(zd, y, md, Sd);
                if (v < 0.0) v = 0.0;
            }
            w[y] = v;
            W += v;
        }
        if (!(W >= 0x1p-20)) { /* p == q (a mass below 2^-20 counts as empty): draw from p */
            W = 0.0;
            for (int y = 0; y < V; ++y) { w[y] = orc_prob(zt, y, mt, St); W += w[y]; }
        }
        const double target = (double)u_bonus[r] * W;
        int tok = -1, last_pos = -1;
        double C = 0.0;
        for (int y = 0; y < V; ++y) {
            if (w[y] > 0.0) last_pos = y;
            C += w[y];
            if (C > target) { tok = y; break; }
        }
        if (tok < 0) tok = last_pos;
        orc_finish(r, correct, tok, draft, prefix, gamma, num_acc, bonus, commit, new_seq, out);
    }
    free(w);
}

/* --------------------------------------------------------- calibration
 *
 * STS recorder, calibration statistics and the sequential temperature
 * fitter.
 *
 *   [AVS] §二 "但 SGLang STS 校准的不是同一个 soft target": the recorder
 *         labels a recorded step with the greedy prefix mask, position k is 1
 *         iff k < num_correct_drafts (a later chance match after the first
 *         mismatch stays 0).
 *   [AVS] §二 "STS 更像运行时语义桥": c_i = sigmoid(z_i / T_i), S_k = prod
 *         c_i; the fitter searches a temperature position by position,
 *         keeping the cumulative survival of the positions already fitted,
 *         and takes for the current position the temperature of lowest ECE.
 *   [TUT] "为什么置信度必须校准": ECE = sum_b |I_b|/n |acc(I_b) - conf(I_b)|
 *         over confidence bins; the label of position k only means something
 *         when the positions before it survived.
 *   [TUT] "截短会制造观测盲区": a compact verify that stops at position L
 *         leaves the later positions unobserved (censored), unless the chain
 *         already broke inside the window.
 *   [AVS] §七 A and [TUT] "置信度质量": per-position and cumulative
 *         calibration, ECE, Brier score or log loss, by depth, with a
 *         reliability diagram.
 *
 * Readings of what the pages leave open:
 *   R24 a recorded sample is (z[gamma], correct, tested): tested = drafts
 *       the target checked (verify_len - 1; gamma for a full block).  Depth
 *       k is observed iff k < tested; label y_k = (k < correct).  A depth
 *       past the window stays unobserved even when the chain broke inside it
 *       (its label is then known to be 0): keeping those samples would keep
 *       them only when their label is 0, the selection bias the truncation
 *       passage warns of.  Out-of-range values are clamped (tested to [0,
 *       gamma], correct to [0, tested]) and flagged BAD_LEN.
 *   R25 cumulative flavour at depth k: prediction S_k, over observed
 *       samples; per-position flavour: prediction c_k, over samples with k <
 *       tested and correct >= k (tested and the prefix survived).  A NaN
 *       prediction leaves the sample out.
 *   R26 n_bins equal-width bins over [0, 1]: bin = min(floor(p*n_bins),
 *       n_bins-1).  Confidences enter the bin sums floored to multiples of
 *       2^-32, so every sum is an exact integer and ECE*n*2^32 =
 *       sum_b |L_b*2^32 - C_b| is an exact integer (ECE within 2^-32 of the
 *       real-number value).  Brier = mean (p - y)^2; log loss = mean
 *       -[y ln p + (1-y) ln(1-p)] with p clamped to [2^-24, 1 - 2^-24]; both
 *       summed in fp64.  A flavour with no sample reports n = 0 and zeros.
 *   R27 the fitter chooses from a caller's grid of temperatures; the lowest
 *       ECE*n*2^32 wins, ties to the lower grid index; a depth with no
 *       observed sample takes T = 1 and choice -1.
 *   R28 recorder: selected rows are appended in request order at slots
 *       (cursor + i) mod capacity and the cursor advances by their count;
 *       when one call selects more than capacity rows, only the last
 *       capacity of them are written (CAPACITY).
 */

#define ORC_Q32 4294967296.0  /* 2^32 */

/* tested and correct of one recorded sample, clamped (reading R24) */
static void orc_sample_lens(int32_t correct, int32_t tested, int gamma, int *c_out, int *t_out,
                            int *status)
{
    int t = tested, c = correct;
    if (t < 0 || t > gamma) {
        *status |= ORC_ST_BAD_LEN;
        t = t < 0 ? 0 : gamma;
    }
    if (c < 0 || c > t) {
        *status |= ORC_ST_BAD_LEN;
        c = c < 0 ? 0 : t;
    }
    *c_out = c;
    *t_out = t;
}

/* The recorder ([AVS] §二; reading R28).  tested = verify_len - 1 (every
 * draft when verify_lens is NULL: a full verify or the cap-accept ceiling);
 * verify_len is clamped to [1, gamma+1] and correct to [0, tested] (BAD_LEN).
 * prefix_mask (nullable) [B, gamma] gets (k < correct) for every request. */
void orc_sts_record(const float *z, const int32_t *correct, const int32_t *verify_lens,
                    const uint8_t *select, int B, int gamma, float *rec_z, int32_t *rec_correct,
                    int32_t *rec_tested, int64_t capacity, uint64_t *cursor, uint8_t *prefix_mask,
                    int *status)
{
    int64_t count = 0;
    for (int r = 0; r < B; ++r)
        if (!select || select[r]) ++count;
    if (count > capacity) *status |= ORC_ST_CAPACITY;
    int64_t i = 0;
    for (int r = 0; r < B; ++r) {
        int tested = gamma;
        if (verify_lens) {
            int L = verify_lens[r];
            if (L < 1 || L > gamma + 1) {
                *status |= ORC_ST_BAD_LEN;
                L = L < 1 ? 1 : gamma + 1;
            }
            tested = L - 1;
        }
        int c = correct[r];
        if (c < 0 || c > tested) {
            *status |= ORC_ST_BAD_LEN;
            c = c < 0 ? 0 : tested;
        }
        if (prefix_mask)
            for (int k = 0; k < gamma; ++k) prefix_mask[(size_t)r * gamma + k] = (uint8_t)(k < c);
        if (select && !select[r]) continue;
        /* appended one after the other: a later row overwrites an earlier
         * one on the same slot */
        uint64_t slot = (*cursor + (uint64_t)i) % (uint64_t)capacity;
        for (int k = 0; k < gamma; ++k) rec_z[slot * (uint64_t)gamma + k] = z[(size_t)r * gamma + k];
        rec_correct[slot] = c;
        rec_tested[slot] = tested;
        ++i;
    }
    *cursor += (uint64_t)count;
}

/* Reliability statistics of n (prediction, label) pairs ([TUT]
 * "为什么置信度必须校准", "置信度质量"; reading R26).
 *   hist    [n_bins][3]: count, label sum, confidence sum in 2^-32 units
 *   metrics [4]: n, ECE, Brier, log loss
 * Returns ECE*n*2^32 as an exact integer. */
uint64_t orc_reliability(const float *p, const uint8_t *y, int64_t n, int n_bins, uint64_t *hist,
                         double *metrics)
{
    memset(hist, 0, sizeof(uint64_t) * 3 * (size_t)n_bins);
    double brier = 0.0, logloss = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double pd = (double)p[i];
        int b = (int)floor(pd * n_bins);
        if (b > n_bins - 1) b = n_bins - 1;
        hist[3 * b + 0] += 1;
        hist[3 * b + 1] += y[i] ? 1 : 0;
        hist[3 * b + 2] += (uint64_t)floor(pd * ORC_Q32);
        double d = pd - (y[i] ? 1.0 : 0.0);
        brier += d * d;
        double pc = pd < 0x1p-24 ? 0x1p-24 : (pd > 1.0 - 0x1p-24 ? 1.0 - 0x1p-24 : pd);
        logloss += y[i] ? -log(pc) : -log(1.0 - pc);
    }
    /* ECE: sum over bins of |I_b|/n |acc - conf| = |L_b - C_b 2^-32| / n */
    uint64_t E = 0;
    for (int b = 0; b < n_bins; ++b) {
        uint64_t L = hist[3 * b + 1] << 32, C = hist[3 * b + 2];
        E += L > C ? L - C : C - L;
    }
    metrics[0] = (double)n;
    metrics[1] = n ? (double)E / ((double)n * ORC_Q32) : 0.0;
    metrics[2] = n ? brier / (double)n : 0.0;
    metrics[3] = n ? logloss / (double)n : 0.0;
    return E;
}

/* Calibration of recorded samples under temperatures T[gamma], by depth and
 * flavour ([AVS] §七 A; [TUT] "置信度质量"; readings R24-R26).
 *   hist    [2][gamma][n_bins][3], metrics [2][gamma][4]; flavour 0 = the
 *   cumulative survival S_k against the prefix label, flavour 1 = the
 *   per-position c_k given that the prefix survived. */
void orc_calib_stats(const float *z, const int32_t *correct, const int32_t *tested, int64_t N,
                     int gamma, const float *T, int n_bins, uint64_t *hist, double *metrics,
                     int *status)
{
    for (int k = 0; k < gamma; ++k)
        if (!(T[k] > 0.0f)) *status |= ORC_ST_BAD_INPUT;
    float *S = (float *)malloc(sizeof(float) * (size_t)(N ? N : 1));
    float *c = (float *)malloc(sizeof(float) * (size_t)(N ? N : 1));
    int *cor = (int *)malloc(sizeof(int) * (size_t)(N ? N : 1));
    int *tst = (int *)malloc(sizeof(int) * (size_t)(N ? N : 1));
    float *p = (float *)malloc(sizeof(float) * (size_t)(N ? N : 1));
    uint8_t *y = (uint8_t *)malloc((size_t)(N ? N : 1));
    for (int64_t i = 0; i < N; ++i) orc_sample_lens(correct[i], tested[i], gamma, &cor[i], &tst[i], status);
    for (int k = 0; k < gamma; ++k) {
        for (int64_t i = 0; i < N; ++i) {
            float zk = z[(size_t)i * gamma + k];
            if (zk != zk) *status |= ORC_ST_BAD_INPUT;
            c[i] = orc_sts(zk, T[k]);
            S[i] = (k == 0) ? c[i] : S[i] * c[i];
        }
        for (int f = 0; f < 2; ++f) {
            int64_t n = 0;
            for (int64_t i = 0; i < N; ++i) {
                int take;
                float pi = f == 0 ? S[i] : c[i];
                if (f == 0) take = k < tst[i];
                else take = k < tst[i] && cor[i] >= k;
                if (!take || pi != pi) continue;
                p[n] = pi;
                y[n] = (uint8_t)(k < cor[i]);
                ++n;
            }
            orc_reliability(p, y, n, n_bins, hist + ((size_t)f * gamma + k) * 3 * (size_t)n_bins,
                            metrics + ((size_t)f * gamma + k) * 4);
        }
    }
    free(S); free(c); free(cor); free(tst); free(p); free(y);
}

/* Sequential temperature scaling fit ([AVS] §二 "STS 更像运行时语义桥";
 * readings R24-R27).  For depth k = 0, 1, ...: for every grid temperature
 * T_j, the cumulative survival S_k = S_{k-1} * sigmoid(z_k / T_j) (S_{k-1}
 * from the temperatures already chosen) is scored by its ECE against the
 * prefix label over the samples observed at depth k; the lowest wins.
 *   T_fit [gamma], choice [gamma], ece_curve [gamma][J] (nullable), n_obs
 *   [gamma] (nullable).  The grid must hold positive finite values. */
void orc_sts_fit(const float *z, const int32_t *correct, const int32_t *tested, int64_t N,
                 int gamma, const float *grid, int J, int n_bins, float *T_fit, int32_t *choice,
                 double *ece_curve, int64_t *n_obs, int *status)
{
    float *S = (float *)malloc(sizeof(float) * (size_t)(N ? N : 1));
    int *cor = (int *)malloc(sizeof(int) * (size_t)(N ? N : 1));
    int *tst = (int *)malloc(sizeof(int) * (size_t)(N ? N : 1));
    float *p = (float *)malloc(sizeof(float) * (size_t)(N ? N : 1));
    uint8_t *y = (uint8_t *)malloc((size_t)(N ? N : 1));
    uint64_t *hist = (uint64_t *)malloc(sizeof(uint64_t) * 3 * (size_t)n_bins);
    double met[4];
    for (int64_t i = 0; i < N; ++i) {
        orc_sample_lens(correct[i], tested[i], gamma, &cor[i], &tst[i], status);
        S[i] = 1.0f;
    }
    for (int k = 0; k < gamma; ++k) {
        uint64_t best = 0;
        int jbest = -1;
        int64_t n = 0;
        for (int j = 0; j < J; ++j) {
            n = 0;
            for (int64_t i = 0; i < N; ++i) {
                float zk = z[(size_t)i * gamma + k];
                if (j == 0 && zk != zk) *status |= ORC_ST_BAD_INPUT;
                if (!(k < tst[i])) continue;     /* past the window: censored */
                float c = orc_sts(zk, grid[j]);
                float pi = (k == 0) ? c : S[i] * c;
                if (pi != pi) continue;
                p[n] = pi;
                y[n] = (uint8_t)(k < cor[i]);
                ++n;
            }
            uint64_t E = orc_reliability(p, y, n, n_bins, hist, met);
            if (ece_curve) ece_curve[(size_t)k * J + j] = met[1];
            if (n > 0 && (jbest < 0 || E < best)) { best = E; jbest = j; }
        }
        if (n_obs) n_obs[k] = n;
        float Tk = jbest >= 0 ? grid[jbest] : 1.0f;
        T_fit[k] = Tk;
        choice[k] = jbest;
        /* keep this depth's survival for the next one */
        for (int64_t i = 0; i < N; ++i) {
            float c = orc_sts(z[(size_t)i * gamma + k], Tk);
            S[i] = (k == 0) ? c : S[i] * c;
        }
    }
    free(S); free(cor); free(tst); free(p); free(y); free(hist);
}
