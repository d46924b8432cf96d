// plan.cu -- the DSpark verify planner on sm_103a.
//
// Pages (by title and section):
//   [AVS] "DSpark 自适应 Verify 怎样分配候选预算" (DSpark adaptive verify:
//         how the candidate budget is allocated)
//   [TUT] charlestar.github.io tutorial "DSpark confidence-scheduled
//         speculative decoding"
//
// Two kernels:
//   survival_kernel  one warp per request, lane k = depth: STS
//                    c_k = sigmoid(z_k / T_k) ([AVS] §二) and the prefix
//                    survival S_k = prod_{i<=k} c_i ([AVS] §一) as a
//                    left-to-right chain of fp32 products, so that every
//                    S_k is the same float as a sequential loop gives.  The
//                    sigmoid runs in fp64 (CUDA's exp is called) and is
//                    rounded once to fp32.  fp64 is slow on this part, so
//                    the B*gamma sigmoids are spread over many SMs.
//   budget_kernel    one 1024-thread CTA, everything in shared memory:
//                    (1) 28-bit candidate keys, ascending key = descending
//                        survival, dropped candidates last;
//                    (2) stable LSD radix sort, 4 passes x 7 bits, ranks
//                        from warp match_any, per-warp histograms;
//                    (3) tau(b) = B + sum of the b largest survivals
//                        ([AVS] §一) as an exact int64 fixed-point scan
//                        (every kept survival is a multiple of 2^-37, and
//                        B + B*gamma <= 2^16 keeps every partial sum below
//                        2^53, so converting to fp64 is exact and equals
//                        any-order fp64 summation);
//                    (4) theta(b) = tau(b)*SPS(B+b) or tau(b)/T(B,B+b)
//                        ([AVS] §一, §四; [TUT] T(bs,K) = bias + alpha(bs)
//                        + theta(M)).  The cost is constant over each table
//                        entry's range of M while tau strictly increases,
//                        so only the right end of each entry's range can
//                        be the first maximiser: one candidate per entry;
//                    (5) budget = first argmax (or the forced budget);
//                    (6) ScheduleVerifyLensTopk ([AVS] §一): the budget
//                        largest candidates in (survival desc, depth asc,
//                        request asc) order are those strictly above the
//                        budget-th survival v*, plus the first ties at v*
//                        in (depth, request) order; each request counts
//                        its own, then clamps to [min, max] verify_len.

#include "dspark_common.cuh"

#include <cmath>

namespace dspark {

constexpr int kSurvThreads = 256;
constexpr int kBudgetThreads = 1024;
constexpr int kBudgetWarps = kBudgetThreads / 32;
constexpr int kRadixBits = 7;
constexpr int kRadix = 1 << kRadixBits;
constexpr int kRadixPasses = 4;             // 28 bits >= the 27-bit keys
constexpr int kHistStride = kRadix + 1;     // pad: fewer bank conflicts in the scan
constexpr int kMaxCandidates = 24576;       // B*gamma limit of the one-CTA planner
constexpr int kMaxItemsPerThread = kMaxCandidates / kBudgetThreads;  // 24
constexpr uint32_t kOneBits = 0x3F800000u;  // bits of 1.0f
constexpr uint32_t kDroppedKey = 0x07FFFFFFu;
constexpr int kMinExpBiased = 113;          // 2^-14: the smallest allowed eps

// ------------------------------------------------------------- survival

__global__ void __launch_bounds__(kSurvThreads)
survival_kernel(const float *__restrict__ z, const float *__restrict__ T, int B, int gamma,
                float eps, float *__restrict__ s_out, int32_t *__restrict__ status) {
    pdl_trigger();
    const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= B) return;  // warp-uniform
    const bool active = lane < gamma;
    float c = 1.0f;
    bool bad = false;
    if (active) {
        const float zk = z[(size_t)r * gamma + lane];
        const float tk = T[lane];
        bad = (zk != zk) || !(tk > 0.0f);
        const float t = __fdiv_rn(zk, tk);                      // IEEE fp32 division
        const double e = exp(-(double)t);                       // CUDA's fp64 exp
        c = __double2float_rn(__ddiv_rn(1.0, __dadd_rn(1.0, e)));
    }
    // S_k = S_{k-1} * c_k strictly left to right (a gamma-step chain).
    float s = c;
    for (int k = 1; k < gamma; ++k) {
        const float prev = __shfl_sync(kFullMask, s, k - 1);
        if (lane == k) s = __fmul_rn(prev, c);
    }
    if (active) s_out[(size_t)r * gamma + lane] = (s >= eps) ? s : 0.0f;
    if (__any_sync(kFullMask, bad) && lane == 0) flag(status, DSPARK_STATUS_BAD_INPUT);
}

// --------------------------------------------------------------- budget

struct CostArgs {
    int kind, n;
    const int32_t *M;
    const double *val;
    double bias, alpha;
};

struct PlanArgs {
    const float *surv;  // [B, gamma], eps-zeroed survivals
    int B, gamma, N;
    float eps;
    int min_len, max_len, forced;
    CostArgs cost;
    int32_t *verify_lens, *budget;
    double *tau_theta;
    int32_t *status;
};

__device__ __forceinline__ uint32_t key_of(float s, bool kept) {
    return kept ? (kOneBits - __float_as_uint(s)) : kDroppedKey;
}

// survival of a kept key as an exact multiple of 2^-37
__device__ __forceinline__ long long fixed_of_key(uint32_t key) {
    if (key == kDroppedKey) return 0;
    const uint32_t bits = kOneBits - key;
    const uint32_t e = bits >> 23;
    const long long mant = (long long)((bits & 0x7FFFFFu) | 0x800000u);
    return mant << (e - kMinExpBiased);
}

__device__ __forceinline__ double tau_of(int B, long long P) {
    return __ll2double_rn(((long long)B << 37) + P) * 0x1p-37;  // exact
}

// Shared-memory layout of the budget kernel.
struct BudgetSmem {
    uint32_t hist[kBudgetWarps * kHistStride];
    long long scan64[40];
    int scan32[40];
    double best_theta[kBudgetWarps];
    int best_b[kBudgetWarps];
    int n_kept, budget, e_star, table_bad;
    float v_star;
    uint32_t key_or, key_and;
};

__device__ __forceinline__ bool theta_better(double ta, int ba, double tb, int bb) {
    return ta > tb || (ta == tb && ba < bb);
}

// Stable LSD radix sort of N 28-bit keys; returns the buffer holding the
// sorted keys (A or Bf).  Items are assigned warp-contiguously: warp w owns
// [w*ipw, (w+1)*ipw) and handles it in rounds of 32 consecutive items, so a
// key's rank inside its warp (earlier rounds, then lower lanes) plus the
// (digit-major, warp-minor) histogram prefix is a stable position.
__device__ uint32_t *radix_sort(uint32_t *A, uint32_t *Bf, int N, BudgetSmem &sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ipt = (N + kBudgetThreads - 1) / kBudgetThreads;
    const int ipw = ipt * 32;
    const unsigned lt = lanemask_lt();
    uint32_t *src = A, *dst = Bf;
    const uint32_t varying = sm.key_or ^ sm.key_and;
    for (int pass = 0; pass < kRadixPasses; ++pass) {
        const int shift = pass * kRadixBits;
        if (((varying >> shift) & (kRadix - 1)) == 0) continue;  // digit constant: skip
        for (int i = tid; i < kBudgetWarps * kHistStride; i += kBudgetThreads) sm.hist[i] = 0;
        __syncthreads();
        uint32_t *h = sm.hist + warp * kHistStride;
        int rank[kMaxItemsPerThread];
#pragma unroll
        for (int i = 0; i < kMaxItemsPerThread; ++i) {
            if (i < ipt) {
                const int idx = warp * ipw + i * 32 + lane;
                const bool valid = idx < N;
                const uint32_t d = valid ? (src[idx] >> shift) & (kRadix - 1) : 0xFFFFu;
                const unsigned peers = __match_any_sync(kFullMask, d);
                const uint32_t base = valid ? h[d] : 0u;
                __syncwarp();
                if (valid && lane == __ffs(peers) - 1) h[d] = base + __popc(peers);
                __syncwarp();
                rank[i] = (int)base + __popc(peers & lt);
            }
        }
        __syncthreads();
        // exclusive scan of the histogram in (digit, warp) order
        {
            const int d = tid >> 3, w0 = (tid & 7) * 4;
            uint32_t v[4], local = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                v[q] = sm.hist[(w0 + q) * kHistStride + d];
                local += v[q];
            }
            int total;
            int off = block_exclusive_scan<int>((int)local, sm.scan32, &total);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                sm.hist[(w0 + q) * kHistStride + d] = (uint32_t)off;
                off += (int)v[q];
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kMaxItemsPerThread; ++i) {
            if (i < ipt) {
                const int idx = warp * ipw + i * 32 + lane;
                if (idx < N) {
                    const uint32_t key = src[idx];
                    const uint32_t d = (key >> shift) & (kRadix - 1);
                    dst[h[d] + rank[i]] = key;
                }
            }
        }
        __syncthreads();
        uint32_t *t = src;
        src = dst;
        dst = t;
    }
    return src;
}

__global__ void __launch_bounds__(kBudgetThreads, 1) budget_kernel(PlanArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BudgetSmem &sm = *reinterpret_cast<BudgetSmem *>(smem_raw);
    unsigned char *buf = smem_raw + ((sizeof(BudgetSmem) + 15) & ~size_t(15));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.B, G = a.gamma, N = a.N;

    pdl_trigger();
    if (tid == 0) {
        sm.key_or = 0u;
        sm.key_and = 0xFFFFFFFFu;
        sm.table_bad = 0;
    }
    pdl_wait();  // survivals come from survival_kernel
    __syncthreads();

    // (1) keys in depth-major order e = k*B + r (coalesced reads of [B, gamma])
    uint32_t *A = reinterpret_cast<uint32_t *>(buf);
    uint32_t *Bf = A + N;
    int kept_local = 0;
    uint32_t kor = 0u, kand = 0xFFFFFFFFu;
    for (int i = tid; i < N; i += kBudgetThreads) {
        const int r = i / G, k = i - r * G;
        const float s = a.surv[i];
        const bool kept = (k < a.max_len - 1) && (s >= a.eps);
        const uint32_t key = key_of(s, kept);
        A[k * B + r] = key;
        kept_local += kept ? 1 : 0;
        kor |= key;
        kand &= key;
    }
    kor = __reduce_or_sync(kFullMask, kor);
    kand = __reduce_and_sync(kFullMask, kand);
    if (lane == 0) {
        atomicOr(&sm.key_or, kor);
        atomicAnd(&sm.key_and, kand);
    }
    const int n_kept = block_sum<int>(kept_local, sm.scan32);  // contains __syncthreads

    // (2) sort
    const uint32_t *sorted = radix_sort(A, Bf, N, sm);

    // (3) P[i] = sum of the i largest survivals, fixed point 2^-37 (P[0] = 0)
    const int ipt = (N + kBudgetThreads - 1) / kBudgetThreads;
    long long *P = reinterpret_cast<long long *>(buf);
    {
        uint32_t kreg[kMaxItemsPerThread];
        long long local = 0;
#pragma unroll
        for (int i = 0; i < kMaxItemsPerThread; ++i) {
            const int idx = tid * ipt + i;
            kreg[i] = (i < ipt && idx < N) ? sorted[idx] : kDroppedKey;
            local += fixed_of_key(kreg[i]);
        }
        long long tot;
        long long run = block_exclusive_scan<long long>(local, sm.scan64, &tot);  // syncs: reads done
#pragma unroll
        for (int i = 0; i < kMaxItemsPerThread; ++i) {
            const int idx = tid * ipt + i;
            if (i < ipt && idx < N) {
                run += fixed_of_key(kreg[i]);
                P[idx + 1] = run;
            }
        }
        if (tid == 0) P[0] = 0;
    }
    __syncthreads();

    // (4) theta at the right end of every table entry's range of budgets
    const CostArgs &c = a.cost;
    const long long Bl = B;
    long long b_top = n_kept;  // largest in-range budget
    if (c.kind == DSPARK_COST_ADDITIVE) b_top = min(b_top, (long long)c.M[c.n - 1] - Bl);
    double my_theta = -INFINITY;
    int my_b = 0x7FFFFFFF;
    bool my_bad_cost = false, my_bad_table = false;
    const double fixed_cost = __dadd_rn(c.bias, c.alpha);
    for (int j = tid; j < c.n; j += kBudgetThreads) {
        if (j > 0 && !(c.M[j] > c.M[j - 1])) my_bad_table = true;
        long long loM, hiM;
        if (c.kind == DSPARK_COST_SPS_1D) {
            loM = (j == 0) ? LLONG_MIN / 4 : (long long)c.M[j];
            hiM = (j == c.n - 1) ? LLONG_MAX / 4 : (long long)c.M[j + 1] - 1;
        } else {
            loM = (j == 0) ? LLONG_MIN / 4 : (long long)c.M[j - 1] + 1;
            hiM = (long long)c.M[j];
        }
        const long long blo = max(loM - Bl, 0LL);
        const long long bhi = min(hiM - Bl, b_top);
        if (blo > bhi) continue;
        const int b = (int)bhi;
        const double tau = tau_of(B, P[b]);
        double theta;
        if (c.kind == DSPARK_COST_SPS_1D) {
            const double sps = c.val[j];
            if (!(sps > 0.0) || !isfinite(sps)) { my_bad_cost = true; continue; }
            theta = __dmul_rn(tau, sps);
        } else {
            const double Tm = __dadd_rn(fixed_cost, c.val[j]);
            if (!(Tm > 0.0) || !isfinite(Tm)) { my_bad_cost = true; continue; }
            theta = __ddiv_rn(tau, Tm);
        }
        if (theta > -INFINITY && theta_better(theta, b, my_theta, my_b)) {
            my_theta = theta;
            my_b = b;
        }
    }
    // block argmax (theta desc, b asc)
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const double ot = __shfl_down_sync(kFullMask, my_theta, d);
        const int ob = __shfl_down_sync(kFullMask, my_b, d);
        if (theta_better(ot, ob, my_theta, my_b)) {
            my_theta = ot;
            my_b = ob;
        }
    }
    if (lane == 0) {
        sm.best_theta[warp] = my_theta;
        sm.best_b[warp] = my_b;
    }
    const int any_bad_cost = __syncthreads_or(my_bad_cost);
    const int any_bad_table = __syncthreads_or(my_bad_table);
    if (tid == 0) {
        double bt = -INFINITY;
        int bb = 0x7FFFFFFF;
        for (int w = 0; w < kBudgetWarps; ++w)
            if (theta_better(sm.best_theta[w], sm.best_b[w], bt, bb)) {
                bt = sm.best_theta[w];
                bb = sm.best_b[w];
            }
        int st = 0;
        if (any_bad_cost || any_bad_table) st |= DSPARK_STATUS_BAD_COST;
        int budget;
        double theta_out = 0.0;
        if (a.forced < 0) {
            if (any_bad_table || bb == 0x7FFFFFFF) {
                budget = 0;
                st |= DSPARK_STATUS_INFEASIBLE;
            } else {
                budget = bb;
                theta_out = bt;
            }
        } else {
            const long long bh = any_bad_table ? -1 : b_top;
            if (bh < 0) {
                budget = 0;
                st |= DSPARK_STATUS_INFEASIBLE;
            } else {
                budget = (int)min((long long)a.forced, bh);
                // theta at the forced budget: the entry that covers M = B + budget
                const long long Mv = Bl + budget;
                int j = -1;
                if (c.kind == DSPARK_COST_SPS_1D) {
                    for (int i = 0; i < c.n; ++i)
                        if (c.M[i] <= Mv) j = i;
                    if (j < 0) j = 0;
                    const double sps = c.val[j];
                    if (sps > 0.0 && isfinite(sps)) theta_out = __dmul_rn(tau_of(B, P[budget]), sps);
                } else {
                    for (int i = c.n - 1; i >= 0; --i)
                        if (c.M[i] >= Mv) j = i;
                    if (j >= 0) {
                        const double Tm = __dadd_rn(fixed_cost, c.val[j]);
                        if (Tm > 0.0 && isfinite(Tm))
                            theta_out = __ddiv_rn(tau_of(B, P[budget]), Tm);
                    }
                }
            }
        }
        if (st) flag(a.status, st);
        sm.budget = budget;
        sm.n_kept = n_kept;
        a.budget[0] = budget;
        a.tau_theta[0] = tau_of(B, P[budget]);
        a.tau_theta[1] = theta_out;
        // the budget-th survival v* and how many candidates lie strictly above it
        if (budget > 0) {
            const long long mstar = P[budget] - P[budget - 1];
            int lo = 0, hi = budget - 1;
            while (lo < hi) {  // first index whose value equals v* (values descend)
                const int mid = (lo + hi) >> 1;
                if (P[mid + 1] - P[mid] > mstar) lo = mid + 1;
                else hi = mid;
            }
            sm.e_star = budget - lo;  // ties to take, temporarily
            sm.v_star = (float)(__ll2double_rn(mstar) * 0x1p-37);
        } else {
            sm.e_star = 0;
            sm.v_star = INFINITY;
        }
    }
    __syncthreads();

    // (6) the m-th tied candidate in (depth, request) order: e = k*B + r
    const int budget = sm.budget;
    const float vstar = sm.v_star;
    const int m_ties = sm.e_star;
    __syncthreads();
    if (budget > 0) {
        int cnt = 0;
        const int e0 = tid * ipt, e1 = min(e0 + ipt, N);
        for (int e = e0; e < e1; ++e) {
            const int k = e / B, r = e - k * B;
            const float s = a.surv[(size_t)r * G + k];
            cnt += (k < a.max_len - 1 && s >= a.eps && s == vstar) ? 1 : 0;
        }
        int total;
        int before = block_exclusive_scan<int>(cnt, sm.scan32, &total);
        if (before < m_ties && m_ties <= before + cnt) {
            for (int e = e0; e < e1; ++e) {
                const int k = e / B, r = e - k * B;
                const float s = a.surv[(size_t)r * G + k];
                if (k < a.max_len - 1 && s >= a.eps && s == vstar) {
                    if (++before == m_ties) {
                        sm.e_star = e;
                        break;
                    }
                }
            }
        }
        __syncthreads();
    }
    const int e_star = sm.e_star;
    for (int r = tid; r < B; r += kBudgetThreads) {
        int cnt = 0;
        if (budget > 0) {
            for (int k = 0; k < G && k < a.max_len - 1; ++k) {
                const float s = a.surv[(size_t)r * G + k];
                if (!(s >= a.eps)) break;  // survivals do not increase along a request
                if (s > vstar || (s == vstar && k * B + r <= e_star)) ++cnt;
            }
        }
        a.verify_lens[r] = min(max(1 + cnt, a.min_len), a.max_len);
    }
}

size_t budget_smem_bytes(int N) {
    return ((sizeof(BudgetSmem) + 15) & ~size_t(15)) + (size_t)8 * (N + 1);
}

}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_plan_workspace_bytes(int32_t B, int32_t gamma) {
    (void)B;
    (void)gamma;
    return 0;  // the whole planner state lives in shared memory
}

extern "C" int dspark_plan(const float *conf_logits, const float *sts_temps,
                           const dspark_plan_params *p, const dspark_cost_table *cost,
                           float *survivals, int32_t *verify_lens, int32_t *budget,
                           double *tau_theta, void *workspace, size_t workspace_bytes,
                           int32_t *status, void *stream) {
    (void)workspace;
    (void)workspace_bytes;
    if (!conf_logits || !sts_temps || !p || !cost || !survivals || !verify_lens || !budget ||
        !tau_theta || !status)
        return DSPARK_ERR_INVALID_ARG;
    if (p->B < 1 || p->gamma < 1) return DSPARK_ERR_INVALID_ARG;
    if (p->gamma > 31) return DSPARK_ERR_UNSUPPORTED;
    if ((long long)p->B * (p->gamma + 1) > 65536) return DSPARK_ERR_UNSUPPORTED;
    if ((long long)p->B * p->gamma > kMaxCandidates) return DSPARK_ERR_UNSUPPORTED;
    if (p->survival_eps != p->survival_eps) return DSPARK_ERR_INVALID_ARG;
    if (!(p->survival_eps >= 0x1p-14f) || !(p->survival_eps <= 1.0f)) return DSPARK_ERR_UNSUPPORTED;
    if (p->min_verify_len < 1 || p->min_verify_len > p->max_verify_len ||
        p->max_verify_len > p->gamma + 1)
        return DSPARK_ERR_INVALID_ARG;
    if (cost->kind != DSPARK_COST_SPS_1D && cost->kind != DSPARK_COST_ADDITIVE)
        return DSPARK_ERR_INVALID_ARG;
    if (cost->n < 1 || !cost->M || !cost->val) return DSPARK_ERR_INVALID_ARG;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int B = p->B, G = p->gamma, N = B * G;
    const int sblocks = (B * 32 + kSurvThreads - 1) / kSurvThreads;
    survival_kernel<<<sblocks, kSurvThreads, 0, s>>>(conf_logits, sts_temps, B, G,
                                                     p->survival_eps, survivals, status);
    if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;

    PlanArgs a;
    a.surv = survivals;
    a.B = B;
    a.gamma = G;
    a.N = N;
    a.eps = p->survival_eps;
    a.min_len = p->min_verify_len;
    a.max_len = p->max_verify_len;
    a.forced = p->forced_budget;
    a.cost = CostArgs{cost->kind, cost->n, cost->M, cost->val, cost->bias_ms, cost->alpha_ms};
    a.verify_lens = verify_lens;
    a.budget = budget;
    a.tau_theta = tau_theta;
    a.status = status;
    const size_t smem = budget_smem_bytes(N);
    if (ensure_smem(reinterpret_cast<const void *>(budget_kernel), (int)budget_smem_bytes(kMaxCandidates), 0) !=
        cudaSuccess)
        return DSPARK_ERR_CUDA;
    if (launch_pdl(budget_kernel, dim3(1), dim3(kBudgetThreads), smem, s, a) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    return DSPARK_OK;
}
