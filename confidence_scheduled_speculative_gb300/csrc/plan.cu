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

constexpr int kSurvThreads = 64;  // 2 requests per CTA: spreads the fp64 sigmoids over many SMs
constexpr int kBudgetThreads = 1024;
constexpr int kBudgetWarps = kBudgetThreads / 32;
constexpr int kRadixBits = 7;
constexpr int kRadix = 1 << kRadixBits;
constexpr int kRadixPasses = 4;             // 28 bits >= the 27-bit keys
constexpr int kHistStride = kRadix + 1;     // pad: fewer bank conflicts in the scan
constexpr int kMaxCandidates = 16384;       // B*gamma limit of the one-CTA planner
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

// inverse of fixed_of_key for a kept survival
__device__ __forceinline__ uint32_t key_of_fixed(long long m) {
    const float s = (float)(__ll2double_rn(m) * 0x1p-37);  // exact
    return kOneBits - __float_as_uint(s);
}

__device__ __forceinline__ double tau_of(int B, long long P) {
    return __ll2double_rn(((long long)B << 37) + P) * 0x1p-37;  // exact
}

// Shared-memory header of the budget kernel; the key and prefix arrays follow.
struct BudgetSmem {
    uint32_t hist[kBudgetWarps * kHistStride];
    long long scan64[40];
    int scan32[40];
    double best_theta[kBudgetWarps];
    int best_b[kBudgetWarps];
    int budget, e_star, table_bad;
    uint32_t key_star;
    uint32_t key_or, key_and;
};

__device__ __forceinline__ bool theta_better(double ta, int ba, double tb, int bb) {
    return ta > tb || (ta == tb && ba < bb);
}

// Stable LSD radix sort of N 28-bit keys, IPT keys per thread.  Warp w owns
// items [w*32*IPT, (w+1)*32*IPT) and ranks them in rounds of 32 consecutive
// items, so (earlier rounds, lower lanes) before it within the warp plus the
// (digit-major, warp-minor) histogram prefix is a stable position.  The first
// executed pass reads `src` (left intact) and writes A; later passes
// alternate A and Bf.  Passes whose digit is the same for every key are
// skipped.  Returns the buffer that holds the sorted keys.
template <int IPT>
__device__ const uint32_t *radix_sort(const uint32_t *src, uint32_t *A, uint32_t *Bf, int N,
                                      BudgetSmem &sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lt = lanemask_lt();
    const uint32_t varying = sm.key_or ^ sm.key_and;
    uint32_t *dst = A;
    const int base_idx = warp * 32 * IPT + lane;
    for (int pass = 0; pass < kRadixPasses; ++pass) {
        const int shift = pass * kRadixBits;
        if (((varying >> shift) & (kRadix - 1)) == 0) continue;
        for (int i = tid; i < kBudgetWarps * kHistStride; i += kBudgetThreads) sm.hist[i] = 0;
        uint32_t key[IPT];
#pragma unroll
        for (int i = 0; i < IPT; ++i) {
            const int idx = base_idx + i * 32;
            key[i] = idx < N ? src[idx] : 0u;
        }
        __syncthreads();
        uint32_t *h = sm.hist + warp * kHistStride;
        int rank[IPT];
#pragma unroll
        for (int i = 0; i < IPT; ++i) {
            const bool valid = base_idx + i * 32 < N;
            const uint32_t d = valid ? (key[i] >> shift) & (kRadix - 1) : 0xFFFFu;
            const unsigned peers = __match_any_sync(kFullMask, d);
            const uint32_t base = valid ? h[d] : 0u;
            __syncwarp();
            if (valid && lane == __ffs(peers) - 1) h[d] = base + __popc(peers);
            __syncwarp();
            rank[i] = (int)base + __popc(peers & lt);
        }
        __syncthreads();
        {   // exclusive scan of the histogram in (digit, warp) order
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
        for (int i = 0; i < IPT; ++i)
            if (base_idx + i * 32 < N) dst[h[(key[i] >> shift) & (kRadix - 1)] + rank[i]] = key[i];
        __syncthreads();
        src = dst;
        dst = (dst == A) ? Bf : A;
    }
    return src;
}

template <int IPT>
__global__ void __launch_bounds__(kBudgetThreads, 1) budget_kernel(PlanArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BudgetSmem &sm = *reinterpret_cast<BudgetSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.B, G = a.gamma, N = a.N;
    // U: unsorted keys in (depth, request) order e = k*B + r; A/Bf: sort
    // buffers; P (prefix sums, N+1 int64) overlays A..Bf once sorted.
    uint32_t *U = reinterpret_cast<uint32_t *>(smem_raw + ((sizeof(BudgetSmem) + 15) & ~size_t(15)));
    const int Nu = (N + 3) & ~3;
    uint32_t *A = U + Nu;
    uint32_t *Bf = A + Nu;
    long long *P = reinterpret_cast<long long *>(A);
    const CostArgs &c = a.cost;

    pdl_trigger();
    // the cost table is written before the step: fetch it while waiting
    int Mj = 0, Mprev = 0, Mnext = 0;
    double vj = 0.0;
    if (tid < c.n) {
        Mj = __ldg(c.M + tid);
        vj = __ldg(c.val + tid);
        if (tid > 0) Mprev = __ldg(c.M + tid - 1);
        if (tid < c.n - 1) Mnext = __ldg(c.M + tid + 1);
    }
    if (tid == 0) {
        sm.key_or = 0u;
        sm.key_and = 0xFFFFFFFFu;
    }
    pdl_wait();  // survivals come from survival_kernel

    // (1) keys (coalesced reads of the row-major survivals)
    int kept_local = 0;
    uint32_t kor = 0u, kand = 0xFFFFFFFFu;
    {
        float sv[IPT];
#pragma unroll
        for (int q = 0; q < IPT; ++q) {
            const int i = q * kBudgetThreads + tid;
            sv[q] = i < N ? a.surv[i] : 0.0f;
        }
#pragma unroll
        for (int q = 0; q < IPT; ++q) {
            const int i = q * kBudgetThreads + tid;
            if (i < N) {
                const int r = i / G, k = i - r * G;
                const bool kept = (k < a.max_len - 1) && (sv[q] >= a.eps);
                const uint32_t key = key_of(sv[q], kept);
                U[k * B + r] = key;
                kept_local += kept ? 1 : 0;
                kor |= key;
                kand &= key;
            }
        }
    }
    kor = __reduce_or_sync(kFullMask, kor);
    kand = __reduce_and_sync(kFullMask, kand);
    __syncthreads();  // key_or / key_and initialised
    if (lane == 0) {
        atomicOr(&sm.key_or, kor);
        atomicAnd(&sm.key_and, kand);
    }
    const int n_kept = block_sum<int>(kept_local, sm.scan32);  // syncs

    // (2) sort
    const uint32_t *sorted = radix_sort<IPT>(U, A, Bf, N, sm);

    // (3) P[i] = sum of the i largest survivals in units of 2^-37 (P[0] = 0)
    {
        uint32_t kreg[IPT];
        long long local = 0;
#pragma unroll
        for (int i = 0; i < IPT; ++i) {
            const int idx = tid * IPT + i;
            kreg[i] = idx < N ? sorted[idx] : kDroppedKey;
            local += fixed_of_key(kreg[i]);
        }
        long long tot;
        long long run = block_exclusive_scan<long long>(local, sm.scan64, &tot);  // reads done
#pragma unroll
        for (int i = 0; i < IPT; ++i) {
            const int idx = tid * IPT + i;
            if (idx < N) {
                run += fixed_of_key(kreg[i]);
                P[idx + 1] = run;
            }
        }
        if (tid == 0) P[0] = 0;
    }
    __syncthreads();

    // (4) theta at the last budget of every table entry's range of M = B + b
    const long long Bl = B;
    long long b_top = n_kept;  // largest in-range budget
    if (c.kind == DSPARK_COST_ADDITIVE) b_top = min(b_top, (long long)__ldg(c.M + c.n - 1) - Bl);
    const double fixed_cost = __dadd_rn(c.bias, c.alpha);
    double my_theta = -INFINITY;
    int my_b = 0x7FFFFFFF;
    bool my_bad_cost = false, my_bad_table = false;
    for (int j = tid; j < c.n; j += kBudgetThreads) {
        if (j >= kBudgetThreads) {
            Mj = __ldg(c.M + j);
            vj = __ldg(c.val + j);
            Mprev = __ldg(c.M + j - 1);
            Mnext = j < c.n - 1 ? __ldg(c.M + j + 1) : 0;
        }
        if (j > 0 && !(Mj > Mprev)) my_bad_table = true;
        long long loM, hiM;
        if (c.kind == DSPARK_COST_SPS_1D) {
            loM = (j == 0) ? LLONG_MIN / 4 : (long long)Mj;
            hiM = (j == c.n - 1) ? LLONG_MAX / 4 : (long long)Mnext - 1;
        } else {
            loM = (j == 0) ? LLONG_MIN / 4 : (long long)Mprev + 1;
            hiM = (long long)Mj;
        }
        const long long blo = max(loM - Bl, 0LL);
        const long long bhi = min(hiM - Bl, b_top);
        if (blo > bhi) continue;
        const int b = (int)bhi;
        const double tau = tau_of(B, P[b]);
        double theta;
        if (c.kind == DSPARK_COST_SPS_1D) {
            if (!(vj > 0.0) || !isfinite(vj)) { my_bad_cost = true; continue; }
            theta = __dmul_rn(tau, vj);
        } else {
            const double Tm = __dadd_rn(fixed_cost, vj);
            if (!(Tm > 0.0) || !isfinite(Tm)) { my_bad_cost = true; continue; }
            theta = __ddiv_rn(tau, Tm);
        }
        if (theta > -INFINITY && theta_better(theta, b, my_theta, my_b)) {
            my_theta = theta;
            my_b = b;
        }
    }
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
    if (warp == 0) {
        double bt = sm.best_theta[lane];
        int bb = sm.best_b[lane];
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            const double ot = __shfl_down_sync(kFullMask, bt, d);
            const int ob = __shfl_down_sync(kFullMask, bb, d);
            if (theta_better(ot, ob, bt, bb)) {
                bt = ot;
                bb = ob;
            }
        }
        if (lane == 0) {
            int st = (any_bad_cost || any_bad_table) ? DSPARK_STATUS_BAD_COST : 0;
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
                    // theta at the forced budget: binary search for the entry covering B + budget
                    const long long Mv = Bl + budget;
                    int lo = 0, hi = c.n;  // first index with M > Mv (1-D) / M >= Mv (additive)
                    while (lo < hi) {
                        const int mid = (lo + hi) >> 1;
                        const long long Mm = __ldg(c.M + mid);
                        const bool right = (c.kind == DSPARK_COST_SPS_1D) ? (Mm > Mv) : (Mm >= Mv);
                        if (right) hi = mid;
                        else lo = mid + 1;
                    }
                    if (c.kind == DSPARK_COST_SPS_1D) {
                        const int j = lo > 0 ? lo - 1 : 0;
                        const double sps = __ldg(c.val + j);
                        if (sps > 0.0 && isfinite(sps)) theta_out = __dmul_rn(tau_of(B, P[budget]), sps);
                    } else if (lo < c.n) {
                        const double Tm = __dadd_rn(fixed_cost, __ldg(c.val + lo));
                        if (Tm > 0.0 && isfinite(Tm)) theta_out = __ddiv_rn(tau_of(B, P[budget]), Tm);
                    }
                }
            }
            if (st) flag(a.status, st);
            sm.budget = budget;
            sm.key_star = budget > 0 ? key_of_fixed(P[budget] - P[budget - 1]) : 0u;
            a.budget[0] = budget;
            a.tau_theta[0] = tau_of(B, P[budget]);
            a.tau_theta[1] = theta_out;
        }
    }
    __syncthreads();

    // (5) ScheduleVerifyLensTopk: candidates strictly above the budget-th
    // survival, plus the first m ties at it in (depth, request) order
    const int budget = sm.budget;
    const uint32_t kstar = sm.key_star;
    int e_star = -1;
    if (budget > 0) {
        int gt = 0, tie = 0;
#pragma unroll
        for (int i = 0; i < IPT; ++i) {
            const int e = tid * IPT + i;
            const uint32_t key = e < N ? U[e] : kDroppedKey;
            gt += key < kstar ? 1 : 0;
            tie += key == kstar ? 1 : 0;
        }
        int total;
        const int excl = block_exclusive_scan<int>((gt << 15) | tie, sm.scan32, &total);
        const int m = budget - (total >> 15);  // ties to take (>= 1)
        int before = excl & 0x7FFF;
        if (before < m && m <= before + tie) {
#pragma unroll
            for (int i = 0; i < IPT; ++i) {
                const int e = tid * IPT + i;
                if (e < N && U[e] == kstar && ++before == m) sm.e_star = e;
            }
        }
        __syncthreads();
        e_star = sm.e_star;
    }
    const int kmax = min(G, a.max_len - 1);
    for (int r = tid; r < B; r += kBudgetThreads) {
        int cnt = 0;
        for (int k = 0; k < kmax; ++k) {
            const int e = k * B + r;
            const uint32_t key = U[e];
            cnt += (key < kstar || (key == kstar && e <= e_star)) ? 1 : 0;
        }
        a.verify_lens[r] = min(max(1 + cnt, a.min_len), a.max_len);
    }
}

size_t budget_smem_bytes(int N) {
    const size_t Nu = (size_t)((N + 3) & ~3);
    return ((sizeof(BudgetSmem) + 15) & ~size_t(15)) + 12 * Nu + 16;
}

template <int IPT>
cudaError_t launch_budget(const PlanArgs &a, cudaStream_t s) {
    const size_t smem = budget_smem_bytes(a.N);
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(budget_kernel<IPT>),
                                (int)budget_smem_bytes(IPT * kBudgetThreads), IPT);
    if (e != cudaSuccess) return e;
    return launch_pdl(budget_kernel<IPT>, dim3(1), dim3(kBudgetThreads), smem, s, a);
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
    const int ipt = (N + kBudgetThreads - 1) / kBudgetThreads;
    cudaError_t e;
    if (ipt <= 1) e = launch_budget<1>(a, s);
    else if (ipt <= 2) e = launch_budget<2>(a, s);
    else if (ipt <= 4) e = launch_budget<4>(a, s);
    else if (ipt <= 8) e = launch_budget<8>(a, s);
    else e = launch_budget<16>(a, s);
    if (e != cudaSuccess) return DSPARK_ERR_CUDA;
    return DSPARK_OK;
}
