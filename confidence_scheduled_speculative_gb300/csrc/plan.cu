// plan.cu -- the DSpark verify planner on sm_103a.
//
// Pages (by title and section):
//   [AVS] "DSpark 自适应 Verify 怎样分配候选预算" (DSpark adaptive verify:
//         how the candidate budget is allocated)
//   [TUT] charlestar.github.io tutorial "DSpark confidence-scheduled
//         speculative decoding"
//
// The survival kernel, then one of four planner kernels by cost table:
// select_kernel (at most 31 entries), dense_select_kernel (up to 6143
// entries, not interpolated) and interp_select_kernel (interpolated, up to
// 2048 samples) run on one CTA and are described at their definitions;
// rank_kernel takes the rest:
//   survival_kernel  one warp per request, lane k = depth: STS
//                    c_k = sigmoid(z_k / T_k) ([AVS] §二) and the prefix
//                    survival S_k = prod_{i<=k} c_i ([AVS] §一), each lane
//                    multiplying c_0..c_k left to right in fp32 so that S_k is
//                    the same float a sequential loop gives.  The sigmoid
//                    runs in fp64 (CUDA's exp is called) and is rounded once
//                    to fp32; fp64 is slow on this part, so the B*gamma
//                    sigmoids are spread over B/2 CTAs.
//   rank_kernel      the global order of [AVS] §一 -- survival descending,
//                    then depth ascending, then request ascending -- as one
//                    rank per candidate, computed over the whole GPU: a
//                    request's survivals never increase with depth, so its
//                    keys form a sorted run, and a candidate's rank is its
//                    own depth plus, for every other request, a 5-step binary
//                    search in that request's run (ties resolved by depth,
//                    then request).  The candidate's survival goes to
//                    position rank of a sorted array.  The last CTA to finish
//                    (atomic ticket; nothing waits) then
//                    (a) scans tau(b) = B + sum of the b largest survivals
//                        ([AVS] §一) as an exact int64 fixed-point sum (every
//                        kept survival is a multiple of 2^-37 and B + B*gamma
//                        <= 2^16 keeps every partial sum below 2^53, so the
//                        fp64 value, built with integer operations, equals
//                        any-order fp64 summation);
//                    (b) evaluates theta(b) = tau(b)*SPS(B+b) or
//                        tau(b)/T(B,B+b) ([AVS] §一, §四; [TUT] T(bs,K) =
//                        bias + alpha(bs) + theta(M)) once per cost-table
//                        entry, at the last budget of the entry's range of M
//                        (the cost is constant there and tau strictly
//                        increases, so no other budget of the range can be
//                        the first maximiser); candidates compare by their
//                        fp64 bit patterns, so fp64 arithmetic is limited to
//                        the defined product or quotient;
//                    (c) takes budget = first argmax (or the forced budget);
//                    (d) ScheduleVerifyLensTopk ([AVS] §一): a request's
//                        selected candidates are its ranks below the budget,
//                        clamped to [min, max] verify_len.

#include "dspark_common.cuh"

#include <cfloat>
#include <climits>
#include <cmath>

namespace dspark {

constexpr int kSurvThreads = 64;  // 2 requests per CTA: spreads the fp64 sigmoids over many SMs
constexpr int kRankThreads = 1024;
constexpr int kRankWarps = kRankThreads / 32;
constexpr int kRankMinPerCta = 4;  // candidates per CTA below which the rank grid shrinks
constexpr int kMaxCandidates = 16384;       // B*gamma limit of the planner
constexpr int kInterpPer = (kMaxCandidates + kRankThreads) / kRankThreads;  // budgets per thread
constexpr int kScanReg = 4;  // kept candidates per thread held in registers by the prefix scan
constexpr uint32_t kOneBits = 0x3F800000u;  // bits of 1.0f
constexpr uint32_t kDroppedKey = 0x07FFFFFFu;
constexpr int kMinExpBiased = 113;          // 2^-14: the smallest allowed eps
constexpr int kNoRank = 0x7FFFFFFF;

// The select path ranks candidates inside the top-11-bit bins of their keys:
// survival_kernel counts the kept keys (and adds their fixed-point
// survivals) per bin, select_kernel reads and clears the bins.
constexpr int kHistShift = 16;               // bin = key >> 16 of a 27-bit key
constexpr int kHistBins = 2048;              // kept keys use bins 0..1792

// Planner scratch in the caller's workspace.
struct PlanScratch {
    unsigned int ticket;  // CTAs of rank_kernel done
    unsigned int pad[3];
    // single-CTA paths: kept keys per top bin and their fixed-point survival
    // sums; zero between calls (the planner kernel clears what
    // survival_kernel added)
    unsigned int hcount[kHistBins];
    unsigned long long hsum[kHistBins];
    // followed by the rank path's int32 rank[N] | int64 sorted[N] |
    // int64 prefix[N+1]
};
static_assert(offsetof(PlanScratch, hcount) % 16 == 0 && offsetof(PlanScratch, hsum) % 16 == 0,
              "histogram rows are read as 16-byte vectors");

__host__ __device__ inline size_t plan_rank_offset() { return (sizeof(PlanScratch) + 255) & ~size_t(255); }
__host__ __device__ inline size_t plan_sorted_offset(int N) {
    return plan_rank_offset() + (((size_t)N * 4 + 15) & ~size_t(15));
}
__host__ __device__ inline size_t plan_prefix_offset(int N) {
    return plan_sorted_offset(N) + (size_t)N * 8;
}
// Between the passes of one call (dspark_plan_ex): the lagged pass's
// budget, the tier-filled budget, and the lengths / tau-theta / survivals a
// pass computes that the caller does not receive.
struct PassScratch {
    int32_t lagged_budget, exec_budget, pass_budget, pad;
    double pass_tau_theta[2];
};
__host__ __device__ inline size_t plan_pass_offset(int B, int N) {
    return (plan_prefix_offset(N) + (size_t)(N + 1) * 8 + 255) & ~size_t(255);
}
__host__ __device__ inline size_t plan_pass_lens_offset(int B, int N) {
    return plan_pass_offset(B, N) + 256;
}
__host__ __device__ inline size_t plan_pass_surv_offset(int B, int N) {
    return (plan_pass_lens_offset(B, N) + (size_t)B * 4 + 255) & ~size_t(255);
}
__host__ __device__ inline size_t plan_scratch_bytes(int B, int N) {
    return plan_pass_surv_offset(B, N) + (size_t)N * 4;
}

template <typename T>
__host__ __device__ __forceinline__ T *scratch_at(PlanScratch *sc, size_t off) {
    return reinterpret_cast<T *>(reinterpret_cast<unsigned char *>(sc) + off);
}

// Keys order the candidates: a kept survival s in [2^-14, 1] maps to
// bits(1.0f) - bits(s), a 27-bit integer that grows as s shrinks; dropped
// candidates map to the largest 27-bit value.
__device__ __forceinline__ uint32_t key_of(float s, bool kept) {
    return kept ? (kOneBits - __float_as_uint(s)) : kDroppedKey;
}

// survival of a kept key as an exact multiple of 2^-37
__device__ __forceinline__ long long fixed_of_key(uint32_t key) {
    const uint32_t bits = kOneBits - key;
    const uint32_t e = bits >> 23;
    const long long mant = (long long)((bits & 0x7FFFFFu) | 0x800000u);
    return mant << (e - kMinExpBiased);
}

// ------------------------------------------------------------- survival

__global__ void __launch_bounds__(kSurvThreads)
survival_kernel(const float *__restrict__ z, const float *__restrict__ T, int B, int gamma,
                float eps, int kmax, bool bin_keys, const int32_t *__restrict__ conf_gen,
                const int32_t *__restrict__ req_gen, float *__restrict__ s_out,
                int32_t *__restrict__ status, PlanScratch *__restrict__ scratch) {
    // launched early behind the previous kernel (programmatic dependent
    // launch): wait for it before touching any input or output, then let the
    // planner pass launch (its pre-wait loads of step inputs and the cost
    // table then run after every earlier kernel has completed)
    pdl_wait();
    pdl_trigger();
    // the rank kernel's ticket starts at zero (only that kernel uses it)
    if (!bin_keys && blockIdx.x == 0 && threadIdx.x == 0) scratch->ticket = 0u;
    const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= B) return;  // warp-uniform
    const bool active = lane < gamma;
    // a request whose pool slot was reused since its confidences were
    // recorded falls back to survivals of 1 ([AVS] §三, req_generation)
    const bool stale = conf_gen && __ldg(conf_gen + r) != __ldg(req_gen + r);
    float c = 1.0f;
    bool bad = false;
    if (active && !stale) {
        const float zk = z[(size_t)r * gamma + lane];
        const float tk = T[lane];
        bad = (zk != zk) || !(tk > 0.0f);
        c = sts_confidence(zk, tk);
    }
    // S_k = (((c_0 c_1) c_2) ... c_k): every lane gathers c_0..c_k and multiplies
    // them strictly left to right.
    float s = __shfl_sync(kFullMask, c, 0);
    for (int k = 1; k < gamma; ++k) {
        const float ck = __shfl_sync(kFullMask, c, k);
        if (k <= lane) s = __fmul_rn(s, ck);
    }
    if (active) s_out[(size_t)r * gamma + lane] = (s >= eps) ? s : 0.0f;
    if (__any_sync(kFullMask, bad) && lane == 0) flag(status, DSPARK_STATUS_BAD_INPUT);
    if (bin_keys && active && lane < kmax && s >= eps) {  // select path: bin the kept key
        const uint32_t key = key_of(s, true);
        const uint32_t bin = key >> kHistShift;
        if (in_bounds(bin, kHistBins, status)) {
            atomicAdd(&scratch->hcount[bin], 1u);
            atomicAdd(&scratch->hsum[bin], (unsigned long long)fixed_of_key(key));
        }
    }
}

// ---------------------------------------------------------------- rank

struct CostArgs {
    int kind, n;
    const int32_t *M;
    const double *val;
    double bias, alpha;
};

// Pack of the verify window fused into select_kernel (dspark_plan_pack):
// the arguments of dspark_pack_verify, verify_lens being the planner's.
struct PackArgs {
    bool on;
    const int32_t *anchor, *draft, *prefix;
    TierArgs tiers;
    int capacity;
    int32_t *ids, *pos, *req, *src, *cu, *totals;
};

struct PlanArgs {
    const float *surv;  // [B, gamma], eps-zeroed survivals
    int B, gamma, N;
    int P2;  // gamma rounded up to a power of two (run length in shared memory)
    float eps;
    int min_len, max_len, forced;
    CostArgs cost;
    int32_t *verify_lens, *budget;
    double *tau_theta;
    int32_t *status;
    PlanScratch *scratch;
    PackArgs pk;
    const int32_t *forced_dev;  // device forced budget (a previous pass's), read after the wait
    bool more_passes;           // another pass over the same survivals follows: the select
                                // path keeps the bins, the rank path resets its ticket and
                                // accumulators for it
    TierArgs align;             // align.n > 0: write the tier-filled budget to *exec_budget
    int32_t *exec_budget;
};

// The forced budget of this pass: from device memory when a previous pass
// chose it, else the caller's.  Call after the dependency wait.
__device__ __forceinline__ int resolve_forced(const PlanArgs &a) {
    return a.forced_dev ? *a.forced_dev : a.forced;
}

// Graph-tier alignment ([AVS] §三, §五 "paid-padding reclamation"): with
// `total` verify rows at budget b (b <= b_top), the rows up to the smallest
// tier >= total are paid for anyway; the executed budget takes one more
// candidate per spare row, within the candidates that are in range.  No tier
// holds the total: b.
__device__ __forceinline__ int aligned_budget(const TierArgs &t, int b, int total, long long b_top) {
    if (t.n <= 0 || b_top < 0) return b;
    bool no_tier;
    const int tier = tier_round_up(t, total, &no_tier);
    if (no_tier) return b;
    return (int)min((long long)b + (tier - total), b_top);
}

// tau = (B * 2^37 + P) * 2^-37 as an fp64 built with integer operations:
// the value is below 2^53 units, so it is exactly representable.
__device__ __forceinline__ double tau_of(int B, long long P) {
    const unsigned long long x = ((unsigned long long)B << 37) + (unsigned long long)P;
    const int msb = 63 - __clzll((long long)x);  // >= 37 since B >= 1
    const unsigned long long mant = (x << (52 - msb)) & ((1ull << 52) - 1);
    const unsigned long long bits = ((unsigned long long)(msb - 37 + 1023) << 52) | mant;
    return __longlong_as_double((long long)bits);
}

__device__ __forceinline__ bool cand_better(long long ka, int ba, long long kb, int bb) {
    return ka > kb || (ka == kb && ba < bb);
}

// The first maximiser over a warp: the largest key (-1: none), ties to the
// smaller budget; every lane receives it with the winner's P and C.  32-bit
// warp reductions (a loop of 64-bit shuffles and compares took ~8000 cycles
// here).
__device__ __forceinline__ void warp_first_max(long long &key, int &b, unsigned long long &P,
                                               unsigned long long &C) {
    const unsigned long long uk = key >= 0 ? (unsigned long long)key + 1ull : 0ull;
    const unsigned hi = (unsigned)(uk >> 32), lo = (unsigned)uk;
    const unsigned mhi = __reduce_max_sync(kFullMask, hi);
    const unsigned mlo = __reduce_max_sync(kFullMask, hi == mhi ? lo : 0u);
    const bool top = hi == mhi && lo == mlo;
    const unsigned bmin = __reduce_min_sync(kFullMask, top ? (unsigned)b : 0x7FFFFFFFu);
    const unsigned win = __ballot_sync(kFullMask, top && (unsigned)b == bmin);
    const int src = __ffs(win) - 1;
    P = __shfl_sync(kFullMask, P, src);
    C = __shfl_sync(kFullMask, C, src);
    key = (long long)((((unsigned long long)mhi << 32) | mlo) - 1ull);
    b = (int)bmin;
}

// Number of keys < key in each of four runs of P2 keys (a power of two,
// at most 32; runs padded past gamma with the largest key): log2(P2) + 1
// branch-free probes per run, the four probe chains interleaved.  The
// caller ignores the result for a run index at or past B (probed as run 0).
__device__ __forceinline__ void run_lower_bound4(const uint32_t *K, int S, int P2, int B,
                                                 uint32_t key, int q0, int lb[4]) {
    const uint32_t *run[4];
    int pos[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int q = q0 + 32 * u;
        run[u] = K + (q < B ? q : 0) * S;
        pos[u] = 0;
    }
#pragma unroll
    for (int step = 16; step > 0; step >>= 1) {
        if (step < P2) {  // uniform: the steps P2/2, ..., 1
#pragma unroll
            for (int u = 0; u < 4; ++u) pos[u] += (run[u][pos[u] + step - 1] < key) ? step : 0;
        }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) lb[u] = pos[u] + ((run[u][pos[u]] < key) ? 1 : 0);
}

// Shared state of the rank kernel.
struct RankSmem {
    long long scan64[40];
    int scan32[40];
    long long best_key[kRankWarps];
    int best_b[kRankWarps];
    long long best_P[kRankWarps];                // P at each warp's best budget
    float fixed32;                              // bias + alpha as a float
    double fixed_cost;                          // bias + alpha
    int order_bad;                              // interpolated table: samples out of order
    int budget, last, n_kept, forced;
    unsigned int theta_floor;  // interpolated table: a lower bound of the largest theta (float bits)
    int n_icand;               // interpolated table: budgets left for the fp64 definition
    int icand_b[kRankThreads], icand_seg[kRankThreads];
    long long b_top;
};

// Keys live in shared memory request-major, each run padded to P2 keys with
// the largest key and laid out with an odd stride, so the 32 lanes of a warp
// probing 32 different runs hit 32 different banks.
__host__ __device__ inline int run_stride(int P2) { return P2 + 1; }

__device__ void finish_plan(const PlanArgs &a, RankSmem &sm);

// Dynamic shared memory of rank_kernel: RankSmem | region R.  R holds the
// keys while the CTAs rank; the last CTA then reuses it for the prefix sums
// P[0..N] (int64) of a table that is not interpolated or, for an
// interpolated table, for the float tau of every budget.
__host__ __device__ inline size_t rank_head_bytes() { return (sizeof(RankSmem) + 15) & ~size_t(15); }
__host__ __device__ inline size_t rank_region_bytes(int B, int S, int N, int kind) {
    size_t r = (size_t)4 * B * S;
    if (kind != DSPARK_COST_ADDITIVE_INTERP && (size_t)8 * (N + 1) > r) r = (size_t)8 * (N + 1);
    return (r + 15) & ~size_t(15);
}

__device__ __forceinline__ int sat_int(long long x) {
    return x > INT_MAX ? INT_MAX : (x < INT_MIN ? INT_MIN : (int)x);
}

// The range of budgets whose M = B + b uses table entry j, clipped to
// [0, b_top]; returns its last budget, or -1 if the range is empty.
__device__ __forceinline__ int entry_last_budget(const CostArgs &c, int j, int Mj, int Mprev,
                                                 int Mnext, long long Bl, long long b_top) {
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
    return blo > bhi ? -1 : (int)bhi;
}

// Entry j's range of budgets [x, y] whose M = B + b looks it up, before the
// clip to the largest in-range budget (saturated to int); order_bad is set
// when M_j does not exceed M_{j-1}.
__device__ __forceinline__ int2 entry_range_from(int kind, int n, int j, long long Mp,
                                                 long long Mj, long long Mn, long long Bl,
                                                 bool &order_bad) {
    if (j > 0 && !(Mj > Mp)) order_bad = true;
    long long lo, hi;
    if (kind == DSPARK_COST_SPS_1D) {
        lo = j == 0 ? 0 : max(Mj - Bl, 0LL);
        hi = j == n - 1 ? (long long)INT_MAX : Mn - 1 - Bl;
    } else {
        lo = j == 0 ? 0 : max(Mp + 1 - Bl, 0LL);
        hi = Mj - Bl;
    }
    return make_int2(sat_int(lo), sat_int(hi));
}

__global__ void __launch_bounds__(kRankThreads, 1) rank_kernel(PlanArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    RankSmem &sm = *reinterpret_cast<RankSmem *>(smem_raw);
    uint32_t *K = reinterpret_cast<uint32_t *>(smem_raw + rank_head_bytes());
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.B, G = a.gamma, N = a.N, P2 = a.P2, S = run_stride(P2);
    const CostArgs &c = a.cost;
    bool order_bad = false;
    int32_t *rank_out = scratch_at<int32_t>(a.scratch, plan_rank_offset());
    long long *sorted = scratch_at<long long>(a.scratch, plan_sorted_offset(N));

    pdl_trigger();
    // the cost table is written before the step: fetch it while waiting
    const bool interp = c.kind == DSPARK_COST_ADDITIVE_INTERP;
    const int Mlast = __ldg(c.M + c.n - 1);
    // interpolated table: its order, checked while the survivals are on the way
    if (interp)
        for (int j = tid + 1; j < c.n; j += kRankThreads)
            if (!(__ldg(c.M + j) > __ldg(c.M + j - 1))) order_bad = true;
    pdl_wait();  // survivals come from survival_kernel
    const int forced = resolve_forced(a);

    // every CTA holds all keys: run r = K[r*S .. r*S + P2)
    int kept_local = 0;
    for (int i0 = tid; i0 < N; i0 += 4 * kRankThreads) {
        float sv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kRankThreads;
            sv[u] = i < N ? a.surv[i] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kRankThreads;
            if (i < N) {
                const int r = i / G;
                const int k = i - r * G;
                const bool kept = (k < a.max_len - 1) && (sv[u] >= a.eps);
                if (in_bounds((long long)r * S + k, (long long)B * S, a.status))
                    K[r * S + k] = key_of(sv[u], kept);
                kept_local += kept ? 1 : 0;
            }
        }
    }
    const int pad = P2 - G;
    for (int j = tid; j < B * pad; j += kRankThreads) {
        const int r = j / pad;
        if (in_bounds((long long)r * S + G + (j - r * pad), (long long)B * S, a.status))
            K[r * S + G + (j - r * pad)] = kDroppedKey;
    }
    const int n_kept = block_sum<int>(kept_local, sm.scan32);  // syncs
    const int any_order_bad = __syncthreads_or(order_bad);
    long long b_top = n_kept;  // largest in-range budget
    if (c.kind != DSPARK_COST_SPS_1D) b_top = min(b_top, (long long)Mlast - (long long)B);
    // fp64 operations and conversions share GB300's small fp64 unit: once per CTA
    if (tid == 0) {
        sm.fixed_cost = __dadd_rn(c.bias, c.alpha);
        sm.fixed32 = (float)sm.fixed_cost;
        sm.order_bad = any_order_bad;
        sm.n_kept = n_kept;
        sm.b_top = b_top;
        sm.forced = forced;
    }
    __syncthreads();

    // ranks: one warp per candidate, lanes over the other requests' runs
    // candidate x goes to CTA x mod grid (warps 0, 1, ... in turn), so every
    // SM of the grid gets its share even when there are few candidates
    const int nwarps = gridDim.x * kRankWarps;
    for (int x = blockIdx.x + gridDim.x * warp; x < N; x += nwarps) {
        const int r = x / G;
        const int k = x - r * G;
        const uint32_t key = K[r * S + k];
        if (key == kDroppedKey) {  // warp-uniform
            if (lane == 0) rank_out[x] = kNoRank;
            continue;
        }
        int cnt = 0;
        // four runs per lane at a time, so their probe chains overlap
        for (int q0 = lane; q0 < B; q0 += 4 * 32) {
            int lb[4];
            run_lower_bound4(K, S, P2, B, key, q0, lb);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int q = q0 + 32 * u;
                if (q >= B || q == r) continue;
                // keys equal to this one in run q sit at depths lb, lb+1, ...;
                // those at a smaller depth, or at the same depth of a lower
                // request, come first (order: survival desc, depth, request)
                const uint32_t *run = K + q * S;
                const int lim = k + (q < r ? 1 : 0);
                int cq = lb[u];
                for (int d = lb[u]; d < lim && run[d] == key; ++d) ++cq;
                cnt += cq;
            }
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) cnt += __shfl_xor_sync(kFullMask, cnt, d);
        const int rk = k + cnt;  // own request: exactly the k shallower depths come first
        const long long m = fixed_of_key(key);
        if (lane == 0) {
            rank_out[x] = rk;
            if (in_bounds(rk, N, a.status)) sorted[rk] = m;
        }
    }

    // the last CTA to finish completes the plan: the ranks and sorted values
    // are made visible before the ticket
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned t = atomicAdd(&a.scratch->ticket, 1u);
        sm.last = (t == gridDim.x - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!sm.last) return;
    __threadfence();
    finish_plan(a, sm);
    if (a.more_passes && tid == 0) a.scratch->ticket = 0u;  // zero for the next pass
}

// T(B, M) of the interpolated additive table at M = Mv <= M_{n-1}
// ([AVS] §四, the exported table's runtime linear interpolation of theta(M)):
// val_j + (Mv - M_j) * slope_j with slope_j = (val_{j+1} - val_j) /
// (M_{j+1} - M_j) in that fp64 order, val_j at Mv = M_j, val_0 below M_0.
// False when T is not a positive finite number.  j = the last sample with
// M_j <= Mv, or -1 when Mv <= M_0 (interp_cost below finds it).
// tM / tV: the table's samples and values, in shared or global memory.
__device__ __forceinline__ bool interp_cost_at(const int32_t *tM, const double *tV, int n,
                                               long long Mv, int j, double fixed_cost, double &T) {
    double th;
    if (j < 0) {
        th = tV[0];
    } else {
        const int lo = j;
        const long long Mj = tM[lo];
        const double vj = tV[lo];
        if (Mj == Mv || lo + 1 >= n) {  // the second: only a table out of order gets here
            th = vj;
        } else {
            const long long Mn = tM[lo + 1];
            const double slope = __ddiv_rn(__dsub_rn(tV[lo + 1], vj), (double)(Mn - Mj));
            th = __dadd_rn(vj, __dmul_rn((double)(Mv - Mj), slope));
        }
    }
    T = __dadd_rn(fixed_cost, th);
    return T > 0.0 && isfinite(T);
}

__device__ __forceinline__ bool interp_cost(const CostArgs &c, long long Mv, double fixed_cost,
                                            double &T) {
    int j = -1;
    if (Mv > (long long)__ldg(c.M)) {
        int lo = 0, hi = c.n - 1;  // the last sample with M_j <= Mv
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((long long)__ldg(c.M + mid) <= Mv) lo = mid;
            else hi = mid - 1;
        }
        j = lo;
    }
    return interp_cost_at(c.M, c.val, c.n, Mv, j, fixed_cost, T);
}

// The key region of the rank kernel's shared memory (after RankSmem), reused
// by the last CTA for the float tau of every budget of an interpolated table.
__device__ __forceinline__ float *interp_tau_smem(RankSmem &sm) {
    return reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(&sm) +
                                     ((sizeof(RankSmem) + 15) & ~size_t(15)));
}

// x as a float for 0 <= x < 2^23, from its bits (no conversion instruction)
__device__ __forceinline__ float small_int_float(int x) {
    return __fsub_rn(__int_as_float(0x4B000000 | x), 8388608.0f);
}

// tau = B + P 2^-37 as a float, truncated (relative error below 2^-23), by
// integer operations only
__device__ __forceinline__ float tau_float(int B, long long P) {
    const unsigned long long x = ((unsigned long long)B << 37) + (unsigned long long)P;
    const int msb = 63 - __clzll((long long)x);  // >= 37
    const unsigned mant = (unsigned)((x >> (msb - 23)) & 0x7fffffull);
    return __uint_as_float(((unsigned)(msb - 37 + 127) << 23) | mant);
}

// fp32 view of the interpolated table for a walk over increasing budgets:
// the segment [M_j, M_{j+1}) holding M = B + b (j = -1 below M_0), loaded
// once per segment crossed.
struct InterpWalk {
    const int32_t *tM;  // the table, in shared or global memory
    const double *tV;
    const float *tV32;  // its values as floats, or null (converted here)
    int n;
    int seg = -2;
    long long Mj = 0, Mn = 0;
    float vj = 0.0f, slope = 0.0f, mag_v = 0.0f;

    __device__ InterpWalk(const int32_t *M, const double *V, const float *V32, int count)
        : tM(M), tV(V), tV32(V32), n(count) {}

    __device__ float value(int j) const { return tV32 ? tV32[j] : (float)tV[j]; }

    __device__ void load(int j) {
        seg = j;
        const int jj = j < 0 ? 0 : j;
        Mj = tM[jj];
        vj = value(jj);
        if (j >= 0 && j + 1 < n) {
            Mn = tM[j + 1];
            const float vn = value(j + 1);
            const long long dM = Mn - Mj;
            slope = __fdiv_rn(vn - vj, dM < (1 << 23) ? small_int_float((int)dM) : (float)dM);
            mag_v = fabsf(vj) + fabsf(vn);
        } else {
            Mn = j < 0 ? Mj + 1 : LLONG_MAX;  // below M_0: up to M_0 inclusive
            slope = 0.0f;
            mag_v = fabsf(vj);
        }
    }

    // Bounds lo <= tau/T <= hi of theta(b) from fp32 arithmetic: the real
    // quotient of the fp64 definition's tau and T lies inside, with room for
    // its final rounding.  The fp32 T differs from the fp64 T by less than
    // 2^-20 times the sum of the magnitudes it is built from (conversions,
    // the slope's subtraction and division, the FMA and the add each
    // contribute at most 2^-23 of one of them).  False when that bound
    // cannot show T > 0 or a value is not finite in fp32: the caller then
    // evaluates the budget in fp64.  Budgets must come in increasing order.
    // the segment of M = Mv, by binary search
    __device__ void init(long long Mv) {
        if (Mv <= (long long)tM[0]) {
            load(-1);
            return;
        }
        int l = 0, h = n - 1;  // the last sample with M_j <= Mv
        while (l < h) {
            const int mid = (l + h + 1) >> 1;
            if ((long long)tM[mid] <= Mv) l = mid;
            else h = mid - 1;
        }
        load(l);
    }

    __device__ bool bounds(int B, long long b, float tau32, float fixed32, float &lo, float &hi) {
        const long long Mv = (long long)B + b;
        while (Mv >= Mn && seg + 1 < n) load(seg + 1);
        const long long dv = Mv - Mj;  // in [0, M_{j+1} - M_j)
        const float d = seg < 0 ? 0.0f : (dv < (1 << 23) ? small_int_float((int)dv) : (float)dv);
        const float th = fmaf(d, slope, vj);
        const float T = fixed32 + th;
        const float err = 0x1p-20f * (fabsf(fixed32) + mag_v + fabsf(d * slope));
        if (!(isfinite(T) && isfinite(err)) || !(T - err > 0.0f)) return false;
        float rT, rTe;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rT) : "f"(T));
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rTe) : "f"(T - err));
        const float q = tau32 * rT;
        const float rel = 0x1p-19f + 2.0f * err * rTe;
        lo = q * (1.0f - rel);
        hi = q * (1.0f + rel);
        return isfinite(hi);
    }
};

// fp32 bounds lo <= theta <= hi of a dense-table entry's theta (the value
// of the fp64 definition: tau * SPS, or tau / (bias + alpha + theta(M))),
// from tau as a float (truncated: relative error below 2^-23) and the
// entry's value as a float.  1-D: the fp32 product is within 2^-21 of the
// fp64 one, inside the 2^-20 margins.  Additive: the bounds of InterpWalk.
// False when fp32 cannot bound theta (a value or the product not a normal
// finite float, or T not shown positive): the caller then evaluates the fp64
// definition, which also flags invalid values.
__device__ __forceinline__ bool dense_theta_bounds(int kind, float tau32, float v32,
                                                   float fixed32, float &lo, float &hi) {
    if (kind == DSPARK_COST_SPS_1D) {
        if (!(v32 >= FLT_MIN) || !(v32 <= FLT_MAX)) return false;
        const float est = tau32 * v32;
        if (!(est >= FLT_MIN) || !(est <= FLT_MAX)) return false;
        lo = est * (1.0f - 0x1p-20f);
        hi = est * (1.0f + 0x1p-20f);
        return hi <= FLT_MAX;
    }
    const float T = fixed32 + v32;
    const float err = 0x1p-20f * (fabsf(fixed32) + fabsf(v32));
    if (!(isfinite(T) && isfinite(err)) || !(T - err > 0.0f)) return false;
    float rT, rTe;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rT) : "f"(T));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rTe) : "f"(T - err));
    const float q = tau32 * rT;
    const float rel = 0x1p-19f + 2.0f * err * rTe;
    lo = q * (1.0f - rel);
    hi = q * (1.0f + rel);
    return isfinite(hi) && lo >= 0.0f;
}

__device__ void finish_plan(const PlanArgs &a, RankSmem &sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.B, G = a.gamma;
    const CostArgs &c = a.cost;
    const int n_kept = sm.n_kept;
    const long long b_top = sm.b_top;
    const int forced = sm.forced;
    const int32_t *rank_in = scratch_at<int32_t>(a.scratch, plan_rank_offset());
    const long long *sorted = scratch_at<long long>(a.scratch, plan_sorted_offset(a.N));
    // the prefix sums: in shared memory (the key region) for a table that
    // is not interpolated, in the workspace for an interpolated one
    unsigned char *smem = reinterpret_cast<unsigned char *>(&sm);
    const bool interp = c.kind == DSPARK_COST_ADDITIVE_INTERP;
    const bool dense = !interp;
    long long *P = dense ? reinterpret_cast<long long *>(smem + rank_head_bytes())
                         : scratch_at<long long>(a.scratch, plan_prefix_offset(a.N));
    // P holds N + 1 sums; the float taus of an interpolated table fill the
    // key region's B * (P2 + 1) words
    const long long nP = (long long)a.N + 1, nT = (long long)B * run_stride(a.P2);
    auto load_P = [&](long long b) -> long long {
        if (!in_bounds(b, nP, a.status)) return 0;
        return dense ? P[b] : __ldcg(P + b);
    };
    auto dense_P = [&](long long b) -> long long {  // P in shared memory
        return in_bounds(b, nP, a.status) ? P[b] : 0;
    };

    // (a) P[i] = sum of the i largest survivals in units of 2^-37 (P[0] =
    // 0), a blocked scan
    {
        const int per = (n_kept + kRankThreads - 1) / kRankThreads;  // <= kScanPer
        const int lo = tid * per, hi = min(lo + per, n_kept);
        // the thread's chunk (up to kScanReg in registers, all in flight at once)
        long long v[kScanReg];
        long long local = 0;
#pragma unroll
        for (int u = 0; u < kScanReg; ++u) v[u] = lo + u < hi ? __ldcg(sorted + lo + u) : 0;
        for (int i = lo + kScanReg; i < hi; ++i) local += __ldcg(sorted + i);
#pragma unroll
        for (int u = 0; u < kScanReg; ++u) local += v[u];
        long long tot;
        long long run = block_exclusive_scan<long long>(local, sm.scan64, &tot);
        // interpolated table: tau of every budget as a float as well, in the
        // key region of shared memory (free once the ranks are out; it holds
        // B * (gamma + 1) >= n_kept + 1 words)
        float *tauf = interp_tau_smem(sm);
        const bool want_f = interp;
#pragma unroll
        for (int u = 0; u < kScanReg; ++u) {
            if (lo + u < hi) {
                run += v[u];
                if (in_bounds(lo + u + 1, nP, a.status)) P[lo + u + 1] = run;
                if (want_f && in_bounds(lo + u + 1, nT, a.status)) tauf[lo + u + 1] = tau_float(B, run);
            }
        }
        for (int i = lo + kScanReg; i < hi; ++i) {
            run += __ldcg(sorted + i);
            if (in_bounds(i + 1, nP, a.status)) P[i + 1] = run;
            if (want_f && in_bounds(i + 1, nT, a.status)) tauf[i + 1] = tau_float(B, run);
        }
        if (tid == 0) {
            P[0] = 0;
            if (want_f) tauf[0] = tau_float(B, 0);
        }
        __syncthreads();
    }

    // (b) theta: at every budget of an interpolated table, else at the last
    // budget of every table entry's range of M = B + b
    const double fixed_cost = sm.fixed_cost;
    long long my_key = -1, my_P = 0;
    int my_b = 0x7FFFFFFF;
    bool my_bad_cost = false, my_bad_table = false;
    if (interp) {
        // The cost changes with every budget.  fp32 bounds of theta at every
        // in-range budget first; the fp64 definition is then evaluated only
        // where the bounds cannot exclude the maximum (or cannot show T > 0):
        // a budget whose upper bound is below the largest lower bound cannot
        // be the first maximiser.
        if (sm.order_bad) my_bad_table = true;  // checked in the prologue
        const int32_t *tM = c.M;
        const double *tV = c.val;
        const float *tV32 = nullptr;  // values converted as the walk reads them
        const float fixed32 = sm.fixed32;
        if (tid == 0) {
            sm.theta_floor = 0u;
            sm.n_icand = 0;
        }
        __syncthreads();
        auto exact = [&](long long b, int seg) {
            double Tm;
            if (!interp_cost_at(tM, tV, c.n, (long long)B + b, seg, fixed_cost, Tm)) {
                my_bad_cost = true;
                return;
            }
            const long long Pb = in_bounds(b, nP, a.status) ? __ldcg(P + b) : 0;
            const double theta = __ddiv_rn(tau_of(B, Pb), Tm);
            const long long kk = __double_as_longlong(theta);
            if (cand_better(kk, (int)b, my_key, my_b)) {
                my_key = kk;
                my_b = (int)b;
                my_P = Pb;
            }
        };
        // each thread walks a contiguous range of at most kInterpPer budgets;
        // its tau values are loaded together, once
        const int per = (int)((b_top + kRankThreads) / kRankThreads);
        const long long b0 = (long long)tid * per;
        const int cnt = (int)max(0LL, min(b0 + per, b_top + 1) - b0);
        const float *tauf = interp_tau_smem(sm);  // tau of every budget, from the scan
        auto tau_at = [&](long long b) -> float {
            return in_bounds(b, nT, a.status) ? tauf[b] : 0.0f;
        };
        InterpWalk wk0(tM, tV, tV32, c.n);
        if (cnt > 0) wk0.init((long long)B + b0);
        float my_floor = 0.0f;
        InterpWalk wk = wk0;
#pragma unroll
        for (int i = 0; i < kInterpPer; ++i) {
            if (i >= cnt) break;
            float lo, hi;
            if (wk.bounds(B, b0 + i, tau_at(b0 + i), fixed32, lo, hi)) {
                my_floor = fmaxf(my_floor, lo);
            } else {
                exact(b0 + i, wk.seg);  // uncertain sign of T, or not finite in fp32
                if (my_b == (int)(b0 + i))
                    my_floor = fmaxf(my_floor, (float)__longlong_as_double(my_key) * (1.0f - 0x1p-20f));
            }
        }
        // non-negative floats order like their bits: one atomic per warp
        const unsigned wfloor = __reduce_max_sync(kFullMask, __float_as_uint(my_floor));
        if (lane == 0) atomicMax(&sm.theta_floor, wfloor);
        __syncthreads();
        const float floor_all = __uint_as_float(sm.theta_floor);
        // the budgets the bounds cannot exclude sit next to each other: list
        // them and give each its own thread for the fp64 definition
        wk = wk0;
#pragma unroll
        for (int i = 0; i < kInterpPer; ++i) {
            if (i >= cnt) break;
            float lo, hi;
            if (wk.bounds(B, b0 + i, tau_at(b0 + i), fixed32, lo, hi) && hi >= floor_all) {
                const int slot = atomicAdd(&sm.n_icand, 1);
                if (slot < kRankThreads) {
                    sm.icand_b[slot] = (int)(b0 + i);
                    sm.icand_seg[slot] = wk.seg;
                } else {
                    exact(b0 + i, wk.seg);  // more than a thread each
                }
            }
        }
        __syncthreads();
        if (tid < min(sm.n_icand, kRankThreads)) exact(sm.icand_b[tid], sm.icand_seg[tid]);
    }
    if (dense) {
        // every entry's theta bounded in fp32 first; the fp64 definition
        // runs only where the bounds cannot exclude the first maximiser (a
        // budget whose upper bound is below the largest lower bound cannot
        // be it), or cannot bound theta at all
        // entry j's last budget b (false when its range holds none) and value
        auto entry = [&](int j, int &b, float &v32) -> bool {
            const int Mj = __ldg(c.M + j);
            const int Mprev = j > 0 ? __ldg(c.M + j - 1) : 0;
            const int Mnext = j < c.n - 1 ? __ldg(c.M + j + 1) : 0;
            if (j > 0 && !(Mj > Mprev)) my_bad_table = true;
            b = entry_last_budget(c, j, Mj, Mprev, Mnext, B, b_top);
            v32 = (float)__ldg(c.val + j);
            return b >= 0;
        };
        auto exact = [&](int j, int b) {
            const double vj = __ldg(c.val + j);
            const long long Pb = dense_P(b);
            const double tau = tau_of(B, Pb);
            double theta;
            if (c.kind == DSPARK_COST_SPS_1D) {
                if (!(vj > 0.0) || !isfinite(vj)) { my_bad_cost = true; return; }
                theta = __dmul_rn(tau, vj);
            } else {
                const double Tm = __dadd_rn(fixed_cost, vj);
                if (!(Tm > 0.0) || !isfinite(Tm)) { my_bad_cost = true; return; }
                theta = __ddiv_rn(tau, Tm);
            }
            const long long kk = __double_as_longlong(theta);
            if (cand_better(kk, b, my_key, my_b)) {
                my_key = kk;
                my_b = b;
                my_P = Pb;
            }
        };
        if (tid == 0) sm.theta_floor = 0u;
        __syncthreads();
        const float fixed32 = sm.fixed32;
        float my_floor = 0.0f, my_top = -1.0f;
        for (int j = tid; j < c.n; j += kRankThreads) {
            int b;
            float v32, lo, hi;
            if (!entry(j, b, v32)) continue;
            if (dense_theta_bounds(c.kind, tau_float(B, dense_P(b)), v32, fixed32, lo, hi)) {
                my_floor = fmaxf(my_floor, lo);
                my_top = fmaxf(my_top, hi);
            } else {
                exact(j, b);
                if (my_b == b)  // its exact theta is itself a lower bound of the maximum
                    my_floor = fmaxf(my_floor,
                                     (float)__longlong_as_double(my_key) * (1.0f - 0x1p-20f));
            }
        }
        // non-negative floats order like their bits: one atomic per warp
        const unsigned wfloor = __reduce_max_sync(kFullMask, __float_as_uint(my_floor));
        if (lane == 0) atomicMax(&sm.theta_floor, wfloor);
        __syncthreads();
        const float floor_all = __uint_as_float(sm.theta_floor);
        if (my_top >= floor_all) {  // only threads holding a possible maximiser
            for (int j = tid; j < c.n; j += kRankThreads) {
                int b;
                float v32, lo, hi;
                if (entry(j, b, v32) &&
                    dense_theta_bounds(c.kind, tau_float(B, dense_P(b)), v32, fixed32, lo, hi) &&
                    hi >= floor_all)
                    exact(j, b);
            }
        }
    }
    {
        unsigned long long P = (unsigned long long)my_P, unused = 0ull;
        warp_first_max(my_key, my_b, P, unused);
        my_P = (long long)P;
    }
    if (lane == 0) {
        sm.best_key[warp] = my_key;
        sm.best_b[warp] = my_b;
        sm.best_P[warp] = my_P;
    }
    const int any_bad_cost = __syncthreads_or(my_bad_cost);
    const int any_bad_table = __syncthreads_or(my_bad_table);
    if (warp == 0) {
        long long bk = lane < kRankWarps ? sm.best_key[lane] : -1;
        int bb = lane < kRankWarps ? sm.best_b[lane] : 0x7FFFFFFF;
        long long bP = lane < kRankWarps ? sm.best_P[lane] : 0;
        {
            unsigned long long P = (unsigned long long)bP, unused = 0ull;
            warp_first_max(bk, bb, P, unused);
            bP = (long long)P;
        }
        if (lane == 0) {
            int st = (any_bad_cost || any_bad_table) ? DSPARK_STATUS_BAD_COST : 0;
            int budget;
            long long Pbud = 0;
            double theta_out = 0.0;
            if (forced < 0) {
                if (any_bad_table || bb == 0x7FFFFFFF) {
                    budget = 0;
                    st |= DSPARK_STATUS_INFEASIBLE;
                } else {
                    budget = bb;
                    theta_out = __longlong_as_double(bk);
                }
            } else {
                const long long bh = any_bad_table ? -1 : b_top;
                if (bh < 0) {
                    budget = 0;
                    st |= DSPARK_STATUS_INFEASIBLE;
                } else {
                    budget = (int)min((long long)forced, bh);
                }
            }
            // P at the budget: carried with the best candidate, or the scan's
            if (budget > 0) Pbud = forced < 0 ? bP : load_P(budget);
            if (forced >= 0 && budget == (int)min((long long)forced, b_top) && b_top >= 0 &&
                !any_bad_table) {
                // theta at the forced budget: the entry covering M = B + budget
                const long long Mv = (long long)B + budget;
                double Ti;
                if (interp && interp_cost(c, Mv, fixed_cost, Ti))
                    theta_out = __ddiv_rn(tau_of(B, Pbud), Ti);
                int lo = 0, hi = interp ? 0 : c.n;  // first index with M > Mv (1-D) / M >= Mv (additive)
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
                    if (sps > 0.0 && isfinite(sps)) theta_out = __dmul_rn(tau_of(B, Pbud), sps);
                } else if (!interp && lo < c.n) {
                    const double Tm = __dadd_rn(fixed_cost, __ldg(c.val + lo));
                    if (Tm > 0.0 && isfinite(Tm)) theta_out = __ddiv_rn(tau_of(B, Pbud), Tm);
                }
            }
            if (st) flag(a.status, st);
            sm.budget = budget;
            a.budget[0] = budget;
            a.tau_theta[0] = tau_of(B, Pbud);
            a.tau_theta[1] = theta_out;
        }
    }
    __syncthreads();

    // (d) a request's selected candidates are its ranks below the budget
    const int budget = sm.budget;
    const int kmax = min(G, a.max_len - 1);
    int lens_sum = 0;
    for (int r = tid; r < B; r += kRankThreads) {
        int cnt = 0;
#pragma unroll 8
        for (int k = 0; k < kmax; ++k) cnt += __ldcg(rank_in + r * G + k) < budget ? 1 : 0;
        const int L = min(max(1 + cnt, a.min_len), a.max_len);
        a.verify_lens[r] = L;
        lens_sum += L;
    }
    if (a.align.n > 0) {  // the tier-filled budget for the next pass
        const int total = block_sum<int>(lens_sum, sm.scan32);
        if (tid == 0) *a.exec_budget = aligned_budget(a.align, budget, total, b_top);
    }
}

size_t rank_smem_bytes(int B, int P2, int N, int kind) {
    return rank_head_bytes() + rank_region_bytes(B, run_stride(P2), N, kind);
}

int pow2_at_least(int g) {
    int p = 1;
    while (p < g) p <<= 1;
    return p;
}

// largest shared-memory request over every (B, gamma) with B*gamma <= kMaxCandidates
size_t rank_smem_max() {
    size_t m = 0;
    for (int g = 1; g <= 31; ++g) {
        const int B = kMaxCandidates / g;
        const size_t v = rank_smem_bytes(B, pow2_at_least(g), B * g, DSPARK_COST_SPS_1D);
        m = v > m ? v : m;
    }
    return m;
}

// ------------------------------------------------------------- select
//
// Cost tables with at most kMaxSelect entries (the graph-tier tables) need
// tau only at a handful of candidate budgets b_j (the last budget of each
// entry's range, and the forced budget), so one CTA finds, for every b_j at
// once, the b_j-th candidate of the global order and the fixed-point sum of
// the survivals up to it:
//   (1) survival_kernel has counted the kept keys per top-11-bit bin; a
//       block scan of the 2048 bins and a 32-way search per candidate give
//       the bin holding its threshold and its rank inside that bin;
//   (2) inside the bins, candidates order by the composite C = key*2^14 + e
//       with e = k*B + r (depth-major position: key ascending is survival
//       descending, then depth, then request), unique per candidate.  The
//       candidates of the marked bins are gathered; when they are few, each
//       one's rank among them is counted directly, otherwise four radix
//       passes over C's low 30 bits (8, 8, 7, 7 bits) find each threshold;
//   (3) theta at every candidate and the budget, as in rank_kernel;
//   (4) a request's survivals never increase with depth, so its C grows with
//       depth and its selected candidates are those up to its first C above
//       C*: the thread holding that position writes the verify length.
// Each thread holds IPT consecutive candidates of the request-major order.

constexpr int kMaxSelect = 31;  // + the forced budget: one warp each of the 32
constexpr int kSelSlots = kMaxSelect + 1;  // table entries + the forced budget
constexpr int kSelThreads = 1024;
constexpr int kRadixBins = 256;
constexpr int kGather = 512;  // gathered candidates ranked by counting
constexpr unsigned long long kNoComposite = ~0ull;

constexpr int kStage = 24576;  // int32 step inputs the fused pack stages in shared memory

struct SelSmem {
    union {
        struct {  // steps (1)-(2)
            unsigned int cum[kHistBins];                       // inclusive key counts by top bin
            unsigned long long csum[kHistBins];                // fixed-point sums of the bins before
            unsigned int H[2][kSelSlots][kRadixBins];          // radix pass counts (two buffers)
            unsigned long long part[kSelSlots][32];            // per-warp partial sums (radix path)
            unsigned long long LC[kGather], LF[kGather];       // gathered composites and survivals
            unsigned long long SC[kGather], SF[kGather];       // the same in composite order
        };
        int lens_s[kMaxCandidates];  // steps (4)-(5): verify length, then first packed row
    };
    int32_t stage[kStage];  // fused pack: anchor [B] | prefix_lens [B] | draft [B, gamma]
    unsigned int binmask[kHistBins / 32];              // top bins holding some threshold
    uint32_t lastkey[kSelThreads];                     // last key of each thread's candidates
    unsigned int wc[32];
    unsigned long long ws[32];
    int scan32[40];
    unsigned long long prefix[kSelSlots];  // high bits of C*_j fixed so far (radix path)
    unsigned long long psum[kSelSlots];    // fixed-point survivals before the current prefix
    unsigned long long P[kSelSlots];       // fixed-point sum of the b_j largest survivals
    unsigned long long cthr[kSelSlots];    // C*_j
    int cand_b[kSelSlots];                 // candidate budget (-1: entry unused)
    int rem[kSelSlots];                    // rank still to find under the prefix (1-based)
    int dbin[kSelSlots];                   // top bin holding C*_j
    int hcnt[kSelSlots];                   // candidates in that bin
    double val_s[kMaxSelect];
    double div_s[kMaxSelect];              // theta divisor T of entry j (additive tables)
    int ok_s[kMaxSelect];                  // entry j's SPS or T is a positive finite number
    int32_t M_s[kMaxSelect];
    int n_gather, bad_table, budget_s;
    unsigned long long cstar;  // C* of the chosen budget (kNoComposite: none)
    // dense_select_kernel
    unsigned int d_floor;      // the largest lower bound of theta (float bits)
    int d_ncand, d_marked;     // entries left after the bounds; keys in their bins
    int d_nruns;               // runs whose bound reaches the floor
    int d_runs[kSelThreads];   // their threads
    double d_fixed;            // bias + alpha
    float d_fixed_lo, d_fixed_hi;  // rounded down and up to float
    float d_fixed32;               // rounded to the nearest float (interp_select_kernel)
    unsigned long long d_fP, d_fC;  // P and C* at the forced budget
    int d_item[32];                 // entry of each threshold slot (-1: the forced budget)
    long long d_bkey[32];           // per-warp first maximiser
    int d_bb[32];
    unsigned long long d_bP[32], d_bC[32];
};

__device__ __forceinline__ unsigned long long composite(uint32_t key, int e) {
    return ((unsigned long long)key << 14) | (unsigned)e;
}

__device__ __forceinline__ void zero_rows(unsigned int (*H)[kRadixBins], int rows) {
    uint4 *h = reinterpret_cast<uint4 *>(&H[0][0]);
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < rows * kRadixBins / 4; i += kSelThreads) h[i] = z;
}

// Four radix passes over the low 30 bits of C for every active slot (rem >=
// 1, prefix = its top bin), then the fixed-point survivals of its bin below
// C*_j; leaves P[j] and cthr[j].  Used when many candidates share the marked
// bins.  Only 32-bit shared atomics: equal digits are common here (ties), and
// same-address 64-bit shared additions serialise badly.
template <int IPT>
__device__ void radix_thresholds(const PlanArgs &a, SelSmem &sm, const uint32_t (&key)[IPT],
                                 int r0, int k0, int nc) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.B, G = a.gamma;
    zero_rows(sm.H[0], nc);
    if (warp < nc && lane == 0) sm.prefix[warp] = (unsigned long long)sm.dbin[warp];
    __syncthreads();
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int sh = pass == 0 ? 22 : pass == 1 ? 14 : pass == 2 ? 7 : 0;
        const int w = pass < 2 ? 8 : 7;
        const int cur = pass & 1;
        // the histogram row of slot `warp`: the first active slot with its prefix
        int myrow = -1;
        if (warp < nc && sm.rem[warp] >= 1) {
            const unsigned long long pw = sm.prefix[warp];
            for (int j = 0; j <= warp; ++j)
                if (sm.rem[j] >= 1 && sm.prefix[j] == pw) {
                    myrow = j;
                    break;
                }
        }
        {   // this thread's candidates in order; equal (row, digit) runs add at once
            int run_row = -1;
            unsigned run_d = 0u, run_c = 0u;
            int r = r0, k = k0;
#pragma unroll
            for (int u = 0; u < IPT; ++u) {
                const uint32_t kk = key[u];
                const uint32_t bin = kk >> kHistShift;
                if (kk != kDroppedKey && ((sm.binmask[bin >> 5] >> (bin & 31)) & 1u)) {
                    const unsigned long long C = composite(kk, k * B + r);
                    const unsigned long long hi = C >> (sh + w);
                    int row = -1;
                    for (int j = 0; j < nc; ++j)
                        if (sm.rem[j] >= 1 && sm.prefix[j] == hi) {
                            row = j;
                            break;
                        }
                    if (row >= 0) {
                        const unsigned dg = (unsigned)(C >> sh) & ((1u << w) - 1u);
                        if (row == run_row && dg == run_d) {
                            ++run_c;
                        } else {
                            if (run_row >= 0 && in_bounds(run_row * kRadixBins + (int)run_d,
                                                          kSelSlots * kRadixBins, a.status))
                                atomicAdd(&sm.H[cur][run_row][run_d], run_c);
                            run_row = row;
                            run_d = dg;
                            run_c = 1u;
                        }
                    }
                }
                if (++k == G) {
                    k = 0;
                    ++r;
                }
            }
            if (run_row >= 0 && in_bounds(run_row * kRadixBins + (int)run_d,
                                          kSelSlots * kRadixBins, a.status))
                atomicAdd(&sm.H[cur][run_row][run_d], run_c);
        }
        __syncthreads();
        // warp j: the digit where the running count reaches rem_j.  Meanwhile
        // the other buffer is cleared.
        if (myrow >= 0) {
            const int per = (1 << w) / 32;
            const unsigned *hc = sm.H[cur][myrow];
            unsigned local = 0u;
            for (int q = 0; q < per; ++q) local += hc[lane * per + q];
            unsigned incl = local;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const unsigned o = __shfl_up_sync(kFullMask, incl, d);
                if (lane >= d) incl += o;
            }
            const int want = sm.rem[warp];
            const int fl = __ffs(__ballot_sync(kFullMask, (int)incl >= want)) - 1;
            if (lane == fl) {
                int run = (int)(incl - local);
                int dg = lane * per;
                for (int q = 0; q < per; ++q) {
                    const int cnt = (int)hc[lane * per + q];
                    if (run + cnt >= want) {
                        dg = lane * per + q;
                        break;
                    }
                    run += cnt;
                }
                sm.prefix[warp] = (sm.prefix[warp] << w) | (unsigned long long)dg;
                sm.rem[warp] = want - run;
            }
        }
        if (pass < 3) zero_rows(sm.H[cur ^ 1], nc);
        __syncthreads();
    }
    // the prefix is now C*_j; add the survivals of its bin below it: per-warp
    // partial sums, then warp j adds its 32 partials
    for (int j = 0; j < nc; ++j) {
        if (sm.cand_b[j] < 1) continue;  // uniform
        const unsigned long long cj = sm.prefix[j];
        const uint32_t dj = (uint32_t)sm.dbin[j];
        unsigned long long acc = 0ull;
        int r = r0, k = k0;
#pragma unroll
        for (int u = 0; u < IPT; ++u) {
            const uint32_t kk = key[u];
            if (kk != kDroppedKey && (kk >> kHistShift) == dj && composite(kk, k * B + r) < cj)
                acc += (unsigned long long)fixed_of_key(kk);
            if (++k == G) {
                k = 0;
                ++r;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFullMask, acc, o);
        if (lane == 0) sm.part[j][warp] = acc;
    }
    __syncthreads();
    if (warp < nc && sm.cand_b[warp] >= 1) {
        unsigned long long acc = sm.part[warp][lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFullMask, acc, o);
        if (lane == 0) {
            sm.cthr[warp] = sm.prefix[warp];
            sm.P[warp] = sm.psum[warp] + acc +
                         (unsigned long long)fixed_of_key((uint32_t)(sm.prefix[warp] >> 14));
        }
    }
}

// Step (5) of select_kernel when the pack is fused: the ragged verify window
// of dspark_pack_verify from the lengths in shared memory ([ROUND] §三,
// [AVS] §五-§六, [SGL] "Ragged verify"): cu_seqlens = exclusive scan of the
// lengths, row cu[r]+j = (j == 0 ? anchor[r] : draft[r][j-1]) at position
// prefix[r]+j, rounded up to the smallest graph tier with pad rows
// (id 0, position 0, request -1, source -1).  A block scan gives each
// request its first row; then each thread writes whole packed rows (stores
// coalesced across the warp), reading anchor / prefix / draft from their
// copy in shared memory, started before the dependency wait (when
// B*(gamma+2) <= kStage).  The planner's lengths are always in [1, gamma+1].
//
// The staging copies (stage_async) are 4-byte cp.async copies global ->
// shared: issuing one does not hold the thread, so the staging's loads run
// past the dependency wait instead of in front of it; each thread waits for
// its own copies (stage_wait) before the barrier that precedes the pack.
__device__ __forceinline__ void stage_async(int32_t *dst, const int32_t *src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}

__device__ __forceinline__ void stage_wait() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void select_pack(const PlanArgs &a, SelSmem &sm, bool staged) {
    const int tid = threadIdx.x;
    const int B = a.B, G = a.gamma, capacity = a.pk.capacity;
    const int32_t *__restrict__ anchor = a.pk.anchor;
    const int32_t *__restrict__ draft = a.pk.draft;
    const int32_t *__restrict__ prefix = a.pk.prefix;
    int32_t *__restrict__ ids = a.pk.ids;
    int32_t *__restrict__ pos = a.pk.pos;
    int32_t *__restrict__ req = a.pk.req;
    int32_t *__restrict__ src = a.pk.src;
    int32_t *__restrict__ cu = a.pk.cu;
    const int per = (B + kSelThreads - 1) / kSelThreads;
    const int q0 = min(tid * per, B), q1 = min(q0 + per, B);
    int mine = 0;
    for (int q = q0; q < q1; ++q) mine += sm.lens_s[q];
    int total;
    int off = block_exclusive_scan<int>(mine, sm.scan32, &total);
    // lens_s becomes the first packed row of each request (strictly
    // increasing: every length is >= 1)
    for (int q = q0; q < q1; ++q) {
        const int L = sm.lens_s[q];
        sm.lens_s[q] = off;
        cu[q + 1] = off + L;
        off += L;
    }
    bool no_tier;
    const int padded = tier_round_up(a.pk.tiers, total, &no_tier);
    __syncthreads();
    // one packed row per thread (coalesced stores); its request by binary
    // search over the first rows
    const int rows = min(total, capacity);
    for (int dst = tid; dst < rows; dst += kSelThreads) {
        int lo = 0, hi = B - 1;  // the last request whose first row is <= dst
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sm.lens_s[mid] <= dst) lo = mid;
            else hi = mid - 1;
        }
        const int j = dst - sm.lens_s[lo];
        if (!in_bounds(j, G + 1, a.status) || !in_bounds(dst, capacity, a.status)) continue;
        int tok, pre;
        if (staged) {
            tok = j == 0 ? sm.stage[lo] : sm.stage[2 * B + lo * G + j - 1];
            pre = sm.stage[B + lo];
        } else {
            tok = j == 0 ? __ldg(anchor + lo) : __ldg(draft + (size_t)lo * G + j - 1);
            pre = __ldg(prefix + lo);
        }
        ids[dst] = tok;
        pos[dst] = pre + j;
        req[dst] = lo;
        src[dst] = lo * (G + 1) + j;
    }
    const int pad_end = min(padded, capacity);
    for (int i = total + tid; i < pad_end; i += kSelThreads) {
        ids[i] = 0;
        pos[i] = 0;
        req[i] = -1;
        src[i] = -1;
    }
    if (tid == 0) {
        cu[0] = 0;
        a.pk.totals[0] = total;
        a.pk.totals[1] = padded;
        if (total > capacity || no_tier || padded > capacity) flag(a.status, DSPARK_STATUS_CAPACITY);
    }
}

// Step (3) of select_kernel, run by warp 0: theta at every candidate budget,
// the first maximiser (or the forced budget) and the plan's scalar outputs.
// Lane j < n holds entry j's candidate and lane n the forced budget's slot;
// every choice is a warp vote or a shuffle, so lane 0 only stores.
__device__ __forceinline__ void select_theta(const PlanArgs &a, SelSmem &sm, long long b_top,
                                             int forced) {
    const int lane = threadIdx.x & 31;
    const int B = a.B, n = a.cost.n;
    const bool sps = a.cost.kind == DSPARK_COST_SPS_1D;
    const int b = lane <= n ? sm.cand_b[lane] : -1;  // slot n: -1 unless forced
    const double tau = tau_of(B, b > 0 ? (long long)sm.P[lane] : 0);
    const unsigned long long cthr = (lane <= n && b > 0) ? sm.cthr[lane] : kNoComposite;
    // the entry whose theta the lane evaluates; for the forced budget the
    // entry covering M = B + budget (1-D: the last M_j <= M, else the first
    // entry; additive: the first M_j >= M, else none)
    int e = lane < n ? lane : -1;
    if (forced >= 0) {
        const long long Mv = (long long)B + __shfl_sync(kFullMask, b, n);
        const long long Mi = lane < n ? (long long)sm.M_s[lane] : 0;
        const unsigned m = __ballot_sync(kFullMask, lane < n && (sps ? Mi <= Mv : Mi >= Mv));
        const int jf = sps ? (m ? 31 - __clz((int)m) : 0) : __ffs((int)m) - 1;
        if (lane == n) e = jf;
    }
    const bool ok = e >= 0 && sm.ok_s[e] != 0;
    double theta = 0.0;
    if (b >= 0 && ok) theta = sps ? __dmul_rn(tau, sm.val_s[e]) : __ddiv_rn(tau, sm.div_s[e]);
    const bool cand = lane < n && b >= 0 && ok;
    const bool bad_cost = lane < n && b >= 0 && !ok;
    // first maximiser: theta >= 0, so its bits order like the values;
    // +1 leaves 0 for "no candidate"; ties go to the smaller budget
    int my_b;
    long long my_key;
    {
        const unsigned long long uk = cand ? (unsigned long long)__double_as_longlong(theta) + 1ull : 0ull;
        const unsigned hi = (unsigned)(uk >> 32), lo = (unsigned)uk;
        const unsigned mhi = __reduce_max_sync(kFullMask, hi);
        const unsigned mlo = __reduce_max_sync(kFullMask, hi == mhi ? lo : 0u);
        const bool top = cand && hi == mhi && lo == mlo;
        my_b = (int)__reduce_min_sync(kFullMask, top ? (unsigned)b : 0x7FFFFFFFu);
        my_key = (long long)((((unsigned long long)mhi << 32) | mlo) - 1ull);
    }
    const bool any_bad_cost = __any_sync(kFullMask, bad_cost);
    const bool bad_table = sm.bad_table != 0;
    int slot = -1;  // -1: infeasible
    if (forced < 0) {
        if (!bad_table && my_b != 0x7FFFFFFF)  // the first entry with the chosen budget
            slot = __ffs((int)__ballot_sync(kFullMask, lane < n && b == my_b)) - 1;
    } else if (!bad_table && b_top >= 0) {
        slot = n;
    }
    const int src = slot < 0 ? 0 : slot;
    const int budget = slot < 0 ? 0 : __shfl_sync(kFullMask, b, src);
    const double tau_s = __shfl_sync(kFullMask, tau, src);
    const unsigned long long cthr_s = __shfl_sync(kFullMask, cthr, src);
    const double theta_f = __shfl_sync(kFullMask, theta, n);
    if (lane == 0) {
        int st = (any_bad_cost || bad_table) ? DSPARK_STATUS_BAD_COST : 0;
        if (slot < 0) st |= DSPARK_STATUS_INFEASIBLE;
        if (st) flag(a.status, st);
        const bool chosen = budget > 0;  // and slot >= 0
        sm.cstar = chosen ? cthr_s : kNoComposite;
        sm.budget_s = budget;
        a.budget[0] = budget;
        a.tau_theta[0] = slot < 0 ? tau_of(B, 0) : tau_s;
        a.tau_theta[1] = slot < 0 ? 0.0 : (forced < 0 ? __longlong_as_double(my_key) : theta_f);
    }
}

// (1) of select_kernel and dense_select_kernel, after the dependency wait:
// the thread's two bins (cleared for the next call, unless a later pass of
// the same call reads them), its keys, and the block scan of the bins into
// inclusive counts (cum) and exclusive fixed-point sums (csum).  Returns the
// number of kept candidates.
template <int IPT>
__device__ __forceinline__ int select_bins(const PlanArgs &a, SelSmem &sm, uint32_t (&key)[IPT]) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.gamma, N = a.N;
    const int kmax = a.max_len - 1;
    const int i0 = tid * IPT;
    const int k0 = i0 - (i0 / G) * G;
    unsigned int h0, h1;
    unsigned long long s0, s1;
    {
        uint2 *hc = reinterpret_cast<uint2 *>(a.scratch->hcount) + tid;
        ulonglong2 *hs = reinterpret_cast<ulonglong2 *>(a.scratch->hsum) + tid;
        const uint2 cv = *hc;
        const ulonglong2 sv = *hs;
        h0 = cv.x;
        h1 = cv.y;
        s0 = sv.x;
        s1 = sv.y;
        if (!a.more_passes) {
            *hc = make_uint2(0u, 0u);
            *hs = make_ulonglong2(0ull, 0ull);
        }
    }
    {
        float sv[IPT];
#pragma unroll
        for (int u = 0; u < IPT; ++u) sv[u] = i0 + u < N ? a.surv[i0 + u] : 0.0f;
        int k = k0;
#pragma unroll
        for (int u = 0; u < IPT; ++u) {
            key[u] = key_of(sv[u], i0 + u < N && k < kmax && sv[u] >= a.eps);
            if (++k == G) k = 0;
        }
        sm.lastkey[tid] = key[IPT - 1];
    }
    // block scan of the bins: inclusive counts, exclusive sums
    int n_kept;
    {
        unsigned ci = h0 + h1;
        unsigned long long si = s0 + s1;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned oc = __shfl_up_sync(kFullMask, ci, d);
            const unsigned long long os = __shfl_up_sync(kFullMask, si, d);
            if (lane >= d) {
                ci += oc;
                si += os;
            }
        }
        if (lane == 31) {
            sm.wc[warp] = ci;
            sm.ws[warp] = si;
        }
        __syncthreads();
        // every warp scans the 32 warp totals itself (no second barrier)
        const unsigned w = sm.wc[lane];
        const unsigned long long wsum = sm.ws[lane];
        unsigned wi = w;
        unsigned long long wsi = wsum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned oc = __shfl_up_sync(kFullMask, wi, d);
            const unsigned long long os = __shfl_up_sync(kFullMask, wsi, d);
            if (lane >= d) {
                wi += oc;
                wsi += os;
            }
        }
        n_kept = (int)__shfl_sync(kFullMask, wi, 31);
        const unsigned wex = __shfl_sync(kFullMask, wi - w, warp);
        const unsigned long long wsex = __shfl_sync(kFullMask, wsi - wsum, warp);
        const unsigned cex = wex + ci - (h0 + h1);
        const unsigned long long sex = wsex + si - (s0 + s1);
        sm.cum[2 * tid] = cex + h0;
        sm.cum[2 * tid + 1] = cex + h0 + h1;
        sm.csum[2 * tid] = sex;
        sm.csum[2 * tid + 1] = sex + s0;
    }
    __syncthreads();
    return n_kept;
}

// Threshold slot `slot` (one warp, every lane calls) takes candidate budget
// b: the top bin holding its threshold, its rank inside the bin (rem, from
// 1), the bin's count and the fixed-point sum of the bins before; the bin is
// marked for the gather.  b < 1: no threshold.
__device__ __forceinline__ void slot_setup(SelSmem &sm, int slot, int lane, int b,
                                           int32_t *status) {
    int rem = 0, d = 0, cnt = 0;
    unsigned long long ps = 0ull;
    if (b >= 1) {  // b <= n_kept = cum[2047]
        const unsigned ub = (unsigned)b;
        // lane 31 always votes (cum[2047] = n_kept >= b); the clamps only keep
        // the indices inside the table
        const int l1 = max(__ffs(__ballot_sync(kFullMask, sm.cum[64 * lane + 63] >= ub)) - 1, 0);
        const int base = 64 * l1;
        const int l2 = max(__ffs(__ballot_sync(kFullMask, sm.cum[base + 2 * lane + 1] >= ub)) - 1, 0);
        d = base + 2 * l2;
        if (sm.cum[d] < ub) ++d;
        const int before = d > 0 ? (int)sm.cum[d - 1] : 0;
        rem = b - before;
        cnt = (int)sm.cum[d] - before;
        ps = sm.csum[d];
        if (lane == 0 && in_bounds(d, kHistBins, status))
            atomicOr(&sm.binmask[d >> 5], 1u << (d & 31));
    }
    if (lane == 0) {
        sm.cand_b[slot] = b;
        sm.rem[slot] = rem;
        sm.dbin[slot] = d;
        sm.hcnt[slot] = cnt;
        sm.psum[slot] = ps;
        sm.P[slot] = 0ull;
        sm.cthr[slot] = kNoComposite;
    }
}

// Gather the candidates of the marked bins into LC (composites) and LF
// (fixed-point survivals), in no particular order; sm.n_gather counts them
// all, the first kGather are stored.
template <int IPT>
__device__ __forceinline__ void gather_marked(const PlanArgs &a, SelSmem &sm,
                                              const uint32_t (&key)[IPT], int r0, int k0) {
    const int lane = threadIdx.x & 31;
    const int B = a.B, G = a.gamma;
    int r = r0, k = k0;
#pragma unroll
    for (int u = 0; u < IPT; ++u) {
        const uint32_t kk = key[u];
        const uint32_t bin = kk >> kHistShift;
        const bool take = kk != kDroppedKey && ((sm.binmask[bin >> 5] >> (bin & 31)) & 1u);
        const unsigned vote = __ballot_sync(kFullMask, take);
        if (vote) {
            int base = 0;
            if (lane == 0) base = atomicAdd(&sm.n_gather, __popc(vote));
            base = __shfl_sync(kFullMask, base, 0);
            const int pos = base + __popc(vote & lanemask_lt());
            if (take && pos < kGather) {
                sm.LC[pos] = composite(kk, k * B + r);
                sm.LF[pos] = (unsigned long long)fixed_of_key(kk);
            }
        }
        if (++k == G) {
            k = 0;
            ++r;
        }
    }
}

// The m <= kGather gathered candidates in composite order: SC / SF (rank of
// each by counting; composites are unique).
__device__ __forceinline__ void rank_gathered(SelSmem &sm, int m, int32_t *status) {
    for (int i = threadIdx.x; i < m; i += kSelThreads) {
        const unsigned long long ci = sm.LC[i];
        int pos = 0;
        for (int y = 0; y < m; ++y) pos += sm.LC[y] < ci ? 1 : 0;
        if (!in_bounds(pos, m, status)) continue;
        sm.SC[pos] = ci;
        sm.SF[pos] = sm.LF[i];
    }
}

// (2) of select_kernel for the nc slots set up by slot_setup: gather the
// candidates of the marked bins; C*_j and P_j of every active slot go to
// sm.cthr and sm.P.  Ends with a barrier.
template <int IPT>
__device__ __forceinline__ void slot_thresholds(const PlanArgs &a, SelSmem &sm,
                                                const uint32_t (&key)[IPT], int r0, int k0,
                                                int nc) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    gather_marked<IPT>(a, sm, key, r0, k0);
    __syncthreads();
    const int m = sm.n_gather;
    if (m <= kGather) {
        rank_gathered(sm, m, a.status);
        __syncthreads();
        // warp j: its bin starts after the gathered candidates of the marked
        // bins below it; C*_j is the rem_j-th of its bin
        if (warp < nc) {
            const int d = sm.dbin[warp], rem = sm.rem[warp];
            if (rem >= 1) {
                int below = 0;
                if (lane < nc) {
                    const int dl = sm.dbin[lane];
                    bool first = sm.rem[lane] >= 1 && dl < d;
                    for (int i = 0; i < lane && first; ++i)
                        if (sm.rem[i] >= 1 && sm.dbin[i] == dl) first = false;
                    below = first ? sm.hcnt[lane] : 0;
                }
                const int start = __reduce_add_sync(kFullMask, below);
                // the bin's candidates are all gathered: start + rem <= m
                const bool in = in_bounds(start + rem - 1, m, a.status);
                unsigned long long part = 0ull;
                for (int q = lane; in && q < rem; q += 32) part += sm.SF[start + q];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(kFullMask, part, o);
                if (lane == 0 && in) {
                    sm.cthr[warp] = sm.SC[start + rem - 1];
                    sm.P[warp] = sm.psum[warp] + part;
                }
            }
        }
    } else {
        radix_thresholds<IPT>(a, sm, key, r0, k0, nc);
    }
    __syncthreads();
}

// (4)-(5) of select_kernel and dense_select_kernel, once sm.cstar and
// sm.budget_s are set.  ScheduleVerifyLensTopk: request r selects its
// candidates with C <= C*, a prefix of its depths; the thread holding the
// first depth past that prefix (or the last depth) writes 1 + its length,
// clamped.  Then the tier-filled budget for a next pass and the fused pack.
template <int IPT>
__device__ __forceinline__ void select_finish(const PlanArgs &a, SelSmem &sm,
                                              const uint32_t (&key)[IPT], long long b_top,
                                              bool staged) {
    const int tid = threadIdx.x;
    const int B = a.B, G = a.gamma, N = a.N;
    const int i0 = tid * IPT;
    const int r0 = i0 / G, k0 = i0 - r0 * G;
    const unsigned long long cstar = sm.cstar;
    {
        int r = r0, k = k0;
        bool prev_in = false;  // the previous depth of the same request is selected
        if (tid > 0 && k0 > 0) {
            const uint32_t pk = sm.lastkey[tid - 1];
            prev_in = cstar != kNoComposite && pk != kDroppedKey &&
                      composite(pk, (k0 - 1) * B + r0) <= cstar;
        }
#pragma unroll
        for (int u = 0; u < IPT; ++u) {
            if (i0 + u < N) {
                const uint32_t kk = key[u];
                const bool in = cstar != kNoComposite && kk != kDroppedKey &&
                                composite(kk, k * B + r) <= cstar;
                int len = -1;
                if (!in && (k == 0 || prev_in)) len = k;  // first depth not selected
                if (in && k == G - 1) len = G;            // every depth selected
                if (len >= 0 && in_bounds(r, B, a.status)) {
                    const int L = min(max(1 + len, a.min_len), a.max_len);
                    a.verify_lens[r] = L;
                    sm.lens_s[r] = L;
                }
                prev_in = in;
            }
            if (++k == G) {
                k = 0;
                ++r;
                prev_in = false;
            }
        }
    }
    if (a.align.n > 0) {  // the tier-filled budget for the next pass
        __syncthreads();
        int mine = 0;
        for (int r = tid; r < B; r += kSelThreads) mine += sm.lens_s[r];
        const int total = block_sum<int>(mine, sm.scan32);
        if (tid == 0) *a.exec_budget = aligned_budget(a.align, sm.budget_s, total, b_top);
    }
    if (a.pk.on) {
        if (staged) stage_wait();
        __syncthreads();
        select_pack(a, sm, staged);
    }
}

template <int IPT>
__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(PlanArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SelSmem &sm = *reinterpret_cast<SelSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.B, G = a.gamma, N = a.N;
    const CostArgs &c = a.cost;
    const int nc = c.n + 1;
    const int i0 = tid * IPT;
    const int r0 = i0 / G, k0 = i0 - r0 * G;  // request and depth of this thread's first candidate

    pdl_trigger();
    // while the survivals are computed: warp j fetches cost entry j (for its
    // budget range); warp 0 fetches entry `lane` and prepares its theta
    // divisor, so that only the product or quotient is left for later
    int Mj = 0, Mprev = 0, Mnext = 0;
    if (warp < c.n) {
        Mj = __ldg(c.M + warp);
        Mprev = warp > 0 ? __ldg(c.M + warp - 1) : 0;
        Mnext = warp < c.n - 1 ? __ldg(c.M + warp + 1) : 0;
    }
    const int Mlast = __ldg(c.M + c.n - 1);
    if (warp == 0) {
        bool bad_entry = false;
        if (lane < c.n) {
            const int m = __ldg(c.M + lane);
            const double v = __ldg(c.val + lane);
            bad_entry = lane > 0 && !(m > __ldg(c.M + lane - 1));
            double Tm = 0.0;
            bool ok;
            if (c.kind == DSPARK_COST_SPS_1D) {
                ok = v > 0.0 && isfinite(v);
            } else {
                Tm = __dadd_rn(__dadd_rn(c.bias, c.alpha), v);
                ok = Tm > 0.0 && isfinite(Tm);
            }
            sm.val_s[lane] = v;
            sm.div_s[lane] = Tm;
            sm.ok_s[lane] = ok ? 1 : 0;
            sm.M_s[lane] = m;
        }
        const bool bt = __any_sync(kFullMask, bad_entry);
        if (lane == 0) sm.bad_table = bt ? 1 : 0;
    }
    if (tid < kHistBins / 32) sm.binmask[tid] = 0u;
    if (tid == 0) sm.n_gather = 0;
    // the fused pack's step inputs are not written by the planner: start
    // their copies now, while the survivals are computed
    const bool staged = a.pk.on && (long long)B * (G + 2) <= kStage;
    if (staged) {
        for (int i = tid; i < B; i += kSelThreads) {
            stage_async(sm.stage + i, a.pk.anchor + i);
            stage_async(sm.stage + B + i, a.pk.prefix + i);
        }
        for (int i = tid; i < N; i += kSelThreads)
            if (in_bounds(2 * B + i, kStage, a.status)) stage_async(sm.stage + 2 * B + i, a.pk.draft + i);
    }
    pdl_wait();  // survivals and bins come from survival_kernel
    const int forced = resolve_forced(a);

    // (1) bins, keys, scan
    uint32_t key[IPT];
    const int n_kept = select_bins<IPT>(a, sm, key);
    long long b_top = n_kept;  // largest in-range budget
    if (c.kind == DSPARK_COST_ADDITIVE) b_top = min(b_top, (long long)Mlast - (long long)B);

    // warp j: candidate budget b_j, the top bin holding its threshold and
    // its rank inside the bin
    if (warp < nc) {
        int b;
        if (warp < c.n) b = entry_last_budget(c, warp, Mj, Mprev, Mnext, B, b_top);
        else b = (forced >= 0 && b_top >= 0) ? (int)min((long long)forced, b_top) : -1;
        slot_setup(sm, warp, lane, b, a.status);
    }
    __syncthreads();

    // (2) thresholds of the candidate budgets
    slot_thresholds<IPT>(a, sm, key, r0, k0, nc);

    // (3) theta at every candidate (all in warp 0) and the budget
    if (warp == 0) select_theta(a, sm, b_top, forced);
    __syncthreads();

    // (4)-(5) lengths, tier-filled budget, pack
    select_finish<IPT>(a, sm, key, b_top, staged);
}

// ------------------------------------------------------------ dense select
//
// Dense cost tables (more than kMaxSelect entries, at most kDenseMaxEntries,
// not interpolated; the 1-D SPS table with an entry per M) on one CTA,
// without ranking every candidate.  The bins of select_kernel give P exactly
// at every bin edge, and bound it inside a bin:
//   (1) as in select_kernel: bins, keys, their scan;
//   (2) entry j's last budget b_j falls in the bin d holding the b_j-th
//       kept key; each of the r = b_j - cum[d-1] keys of that bin up to it
//       survives between the bin's smallest and largest survival (and the
//       bin's other keys between the same), so tau(b_j) lies in an interval
//       and theta_j between fp32 bounds computed with directed rounding
//       (which bound the fp64 definition as well).  Each thread holds a
//       contiguous run of entries: the run's last entry (its largest tau)
//       gives a lower bound, and the largest over the CTA is a floor of the
//       maximum; the run as a whole is bounded above by that tau with the
//       run's largest SPS (smallest cost);
//   (3) the runs whose bound reaches the floor are listed and every entry
//       of theirs is bounded by a thread of its own; an entry whose upper
//       bound is below the floor cannot be the first maximiser.  The entries left (in the workloads, a handful) and the
//       forced budget mark their bins.  When those bins hold at most kGather
//       keys, the keys are gathered, ordered by composite and prefix-summed
//       (both by counting): the exact P and C* of every entry left follow,
//       and theta in fp64 as in the other paths; the first maximiser wins;
//   (4) otherwise (bins crowded by near-equal survivals) the entries left
//       take select_kernel's threshold slots, 32 at a time (radix passes
//       inside crowded bins);
//   (5) lengths, tier-filled budget and pack as in select_kernel.
// The table is staged in shared memory before the dependency wait (each
// entry's range of budgets and its value rounded down to a float, and each
// run's value range), in the region the select path stages the pack's
// inputs in; the fused pack reads its inputs from global memory instead.

// entries of the stage: range int2 + value float + candidate list int
constexpr int kDenseMaxEntries = (kStage * 4 - 16) / 16;
constexpr int kDensePer = (kDenseMaxEntries + kSelThreads - 1) / kSelThreads;  // entries a thread

struct DenseStage {
    int2 *range;  // entry j's budgets [x, y] whose M = B + b looks it up (before the clip to
                  // b_top); for an entry left by step (3): its last budget and that bin
    float *f32;   // its value rounded down to a float
    int *list;    // entries left by step (3)
};

__device__ __forceinline__ DenseStage dense_stage(SelSmem &sm, int n) {
    unsigned char *p = reinterpret_cast<unsigned char *>(sm.stage);
    return DenseStage{reinterpret_cast<int2 *>(p), reinterpret_cast<float *>(p + (size_t)8 * n),
                      reinterpret_cast<int *>(p + (size_t)12 * n)};
}

// the largest kept key: survivals are at least 2^-14
constexpr uint32_t kMaxKeptKey = kOneBits - ((uint32_t)kMinExpBiased << 23);

// An upper bound of a value whose float rounded down is v_lo: one float ulp
// up (the smallest positive float above 0).
__device__ __forceinline__ float value_hi(float v_lo) {
    return v_lo == 0.0f ? __int_as_float(1) : __fmaf_ru(fabsf(v_lo), 0x1p-23f, v_lo);
}

// B + P 2^-37 rounded down and up to floats, by integer operations
// (tau_float truncates; one ulp more when bits were dropped)
__device__ __forceinline__ void tau_float_rd_ru(int B, long long P, float &lo, float &hi) {
    const unsigned long long x = ((unsigned long long)B << 37) + (unsigned long long)P;
    const int msb = 63 - __clzll((long long)x);  // >= 37
    const unsigned bits = ((unsigned)(msb - 37 + 127) << 23) | (unsigned)((x >> (msb - 23)) & 0x7fffffull);
    lo = __uint_as_float(bits);
    hi = __uint_as_float(bits + ((x & ((1ull << (msb - 23)) - 1ull)) ? 1u : 0u));
}


// The bin of budget b >= 1: the first whose inclusive count reaches b
// (cum[kHistBins-1] = n_kept >= b).
__device__ __forceinline__ int bin_of_budget(const SelSmem &sm, int b) {
    int lo = 0, hi = kHistBins - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (sm.cum[mid] >= (unsigned)b) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

// Bin d marked for the gather; its first marker adds the bin's keys to
// d_marked.
__device__ __forceinline__ void mark_bin(SelSmem &sm, int d, int32_t *status) {
    if (!in_bounds(d, kHistBins, status)) return;
    const unsigned bit = 1u << (d & 31);
    if (!(atomicOr(&sm.binmask[d >> 5], bit) & bit))
        atomicAdd(&sm.d_marked, (int)(sm.cum[d] - (d > 0 ? sm.cum[d - 1] : 0u)));
}

// tau(b) = B + P 2^-37 in fp32 with directed rounding (bounds of the fp64
// definition too: rd32(x) <= rn64(x) <= ru32(x) for every real x).  tau(b)
// lies in [B + c0 + r s_lo, B + c0 + r s_hi] and in [B + c1 - (cnt - r) s_hi,
// B + c1 - (cnt - r) s_lo], with c0 and c1 the fixed-point sums before and
// after b's bin d, cnt the bin's keys, s_lo and s_hi its smallest and largest
// survival (exact floats) and r = b - cum[d-1].  b = 0: tau = B exactly.
__device__ __forceinline__ void tau_interval(const SelSmem &sm, int B, int b, int d, float &t_lo,
                                             float &t_hi, int32_t *status) {
    t_lo = t_hi = (float)B;
    if (b < 1 || !in_bounds(d + 1, kHistBins, status)) return;
    const int before = d > 0 ? (int)sm.cum[d - 1] : 0;
    const int cnt = (int)sm.cum[d] - before;
    const uint32_t last = (((uint32_t)d + 1) << kHistShift) - 1;
    const float s_hi = __uint_as_float(kOneBits - ((uint32_t)d << kHistShift));
    const float s_lo = __uint_as_float(kOneBits - (last < kMaxKeptKey ? last : kMaxKeptKey));
    float b0_lo, b0_hi, b1_lo, b1_hi;
    tau_float_rd_ru(B, (long long)sm.csum[d], b0_lo, b0_hi);
    tau_float_rd_ru(B, (long long)sm.csum[d + 1], b1_lo, b1_hi);
    const float r = (float)(b - before), rest = (float)(cnt - (b - before));
    t_lo = fmaxf(__fmaf_rd(r, s_lo, b0_lo), __fmaf_rd(-rest, s_hi, b1_lo));
    t_hi = fminf(__fmaf_ru(r, s_hi, b0_hi), __fmaf_ru(-rest, s_lo, b1_hi));
}

// Each of the m <= kGather gathered candidates' rank and the inclusive
// fixed-point sum of the survivals up to it, both by counting: SC / SF in
// composite order.
__device__ __forceinline__ void rank_gathered_prefix(SelSmem &sm, int m, int32_t *status) {
    for (int i = threadIdx.x; i < m; i += kSelThreads) {
        const unsigned long long ci = sm.LC[i];
        int pos = 0;
        unsigned long long sum = 0ull;
        for (int y = 0; y < m; ++y) {
            const bool le = sm.LC[y] <= ci;
            pos += le ? 1 : 0;
            sum += le ? sm.LF[y] : 0ull;
        }
        if (!in_bounds(pos - 1, m, status)) continue;
        sm.SC[pos - 1] = ci;
        sm.SF[pos - 1] = sum;
    }
}

// P and C* at budget b >= 1 in bin d, from SC / SF when every key of the bin
// is among the m gathered: the bin's keys start where the composites reach
// the bin (its number is the composite's top bits).
__device__ __forceinline__ bool exact_at_budget(const SelSmem &sm, int m, int b, int d,
                                                unsigned long long &P, unsigned long long &C,
                                                int32_t *status) {
    const int r = b - (d > 0 ? (int)sm.cum[d - 1] : 0);
    const unsigned long long first = (unsigned long long)d << (kHistShift + 14);
    int lo = 0, hi = m;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (sm.SC[mid] < first) lo = mid + 1;
        else hi = mid;
    }
    const int idx = lo + r - 1;
    if (!in_bounds(idx, m, status) || !in_bounds(lo, m, status)) return false;
    P = sm.csum[d] + sm.SF[idx] - (lo > 0 ? sm.SF[lo - 1] : 0ull);
    C = sm.SC[idx];
    return true;
}

// The first maximiser over the block, left in every lane of warp 0 (the
// other warps keep their own); true when any thread's `bad` is set.
// Contains a barrier: every thread of the block calls it.
__device__ __forceinline__ bool block_first_max(SelSmem &sm, long long &key, int &b,
                                                unsigned long long &P, unsigned long long &C,
                                                bool bad) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    warp_first_max(key, b, P, C);
    if (lane == 0) {
        sm.d_bkey[warp] = key;
        sm.d_bb[warp] = b;
        sm.d_bP[warp] = P;
        sm.d_bC[warp] = C;
    }
    const bool any_bad = __syncthreads_or(bad) != 0;
    if (warp == 0) {
        key = sm.d_bkey[lane];
        b = sm.d_bb[lane];
        P = sm.d_bP[lane];
        C = sm.d_bC[lane];
        warp_first_max(key, b, P, C);
    }
    return any_bad;
}


// Crowded bins (step (4) of the dense and interp paths): the K items left
// (item i's budget from budget_of(i)), then the forced budget b_forced when
// it is >= 1, take select_kernel's threshold slots 32 at a time; eval(i, b,
// P, C) runs in warp 0's lane of item i's slot, and the forced budget's P and
// C* go to sm.d_fP / sm.d_fC.  Every thread of the block calls it.
template <int IPT, class BudgetOf, class Eval>
__device__ __forceinline__ void threshold_rounds(const PlanArgs &a, SelSmem &sm,
                                                 const uint32_t (&key)[IPT], int r0, int k0,
                                                 int K, int b_forced, BudgetOf budget_of,
                                                 Eval eval) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = K + (b_forced >= 1 ? 1 : 0);
    for (int base = 0; base < T; base += 32) {  // uniform
        const int nc = min(32, T - base);
        if (tid < kHistBins / 32) sm.binmask[tid] = 0u;
        if (tid == 0) sm.n_gather = 0;
        __syncthreads();
        if (warp < nc) {
            const int item = base + warp;
            slot_setup(sm, warp, lane, item < K ? budget_of(item) : b_forced, a.status);
            if (lane == 0) sm.d_item[warp] = item < K ? item : -1;
        }
        __syncthreads();
        slot_thresholds<IPT>(a, sm, key, r0, k0, nc);
        if (warp == 0 && lane < nc) {
            const int b = sm.cand_b[lane], item = sm.d_item[lane];
            const unsigned long long P = b >= 1 ? sm.P[lane] : 0ull;
            const unsigned long long C = b >= 1 ? sm.cthr[lane] : kNoComposite;
            if (item >= 0) {
                eval(item, b, P, C);
            } else {
                sm.d_fP = P;
                sm.d_fC = C;
            }
        }
        __syncthreads();
    }
}

// The plan's decision and scalar outputs on the dense and interp paths, in
// lane 0 of warp 0 after block_first_max: the first maximiser (key, b, P,
// C), or the forced budget (its P and C* in sm.d_fP / sm.d_fC, theta from
// forced_theta(budget, tau)); sets sm.cstar and sm.budget_s for the lengths.
template <class ForcedTheta>
__device__ __forceinline__ void write_decision(const PlanArgs &a, SelSmem &sm, long long key,
                                               int b, unsigned long long P, unsigned long long C,
                                               bool any_bad_cost, bool bad_table, int forced,
                                               int b_forced, ForcedTheta forced_theta) {
    int st = (any_bad_cost || bad_table) ? DSPARK_STATUS_BAD_COST : 0;
    int budget = 0;
    unsigned long long Pbud = 0ull, cstar = kNoComposite;
    double theta_out = 0.0;
    if (forced < 0) {
        if (bad_table || b == 0x7FFFFFFF) {
            st |= DSPARK_STATUS_INFEASIBLE;
        } else {
            budget = b;
            theta_out = __longlong_as_double(key);
            if (budget > 0) {
                Pbud = P;
                cstar = C;
            }
        }
    } else if (b_forced < 0) {
        st |= DSPARK_STATUS_INFEASIBLE;
    } else {
        budget = b_forced;
        if (budget > 0) {
            Pbud = sm.d_fP;
            cstar = sm.d_fC;
        }
        theta_out = forced_theta(budget, tau_of(a.B, (long long)Pbud));
    }
    if (st) flag(a.status, st);
    sm.cstar = cstar;
    sm.budget_s = budget;
    a.budget[0] = budget;
    a.tau_theta[0] = tau_of(a.B, (long long)Pbud);
    a.tau_theta[1] = theta_out;
}


template <int IPT>
__global__ void __launch_bounds__(kSelThreads, 1) dense_select_kernel(PlanArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SelSmem &sm = *reinterpret_cast<SelSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.B, G = a.gamma;
    const CostArgs &c = a.cost;
    const int n = c.n;
    const int i0 = tid * IPT;
    const int r0 = i0 / G, k0 = i0 - r0 * G;
    const DenseStage ds = dense_stage(sm, n);

    // each thread a contiguous run of entries (their budgets and bins do
    // not decrease along it)
    const int per = (n + kSelThreads - 1) / kSelThreads;  // <= kDensePer
    const int j0 = min(tid * per, n), j1 = min(j0 + per, n);

    pdl_trigger();
    // while the survivals are computed: every entry's range of budgets (the
    // 64-bit arithmetic of entry_last_budget, before the clip) and its value
    // as a float; the run's loads are all issued first
    bool order_bad = false;
    // the run's smallest staged value and largest upper bound of a value
    // (NaN when a value is NaN), for the run's bound after the wait
    float run_vmin = INFINITY, run_vmax = 0.0f;
    {
        long long Mv[kDensePer + 2];  // M_{j0-1} .. M_{j0+kDensePer}
        double vv[kDensePer];
#pragma unroll
        for (int u = 0; u < kDensePer + 2; ++u) {
            const int j = j0 - 1 + u;
            Mv[u] = (u <= j1 - j0 + 1 && j >= 0 && j < n) ? __ldg(c.M + j) : 0;
        }
#pragma unroll
        for (int u = 0; u < kDensePer; ++u) vv[u] = j0 + u < j1 ? __ldg(c.val + j0 + u) : 0.0;
#pragma unroll
        for (int u = 0; u < kDensePer; ++u) {
            const int j = j0 + u;
            if (j < j1 && in_bounds(j, kDenseMaxEntries, a.status)) {
                ds.range[j] = entry_range_from(c.kind, n, j, Mv[u], Mv[u + 1], Mv[u + 2], B,
                                               order_bad);
                const float v_lo = __double2float_rd(vv[u]);
                ds.f32[j] = v_lo;
                run_vmin = fminf(run_vmin, v_lo);
                run_vmax = (v_lo != v_lo || run_vmax != run_vmax) ? v_lo + run_vmax
                                                                  : fmaxf(run_vmax, value_hi(v_lo));
            }
        }
    }
    const int Mlast = __ldg(c.M + n - 1);
    if (tid < kHistBins / 32) sm.binmask[tid] = 0u;
    if (tid == 0) {
        sm.n_gather = 0;
        sm.d_floor = 0u;
        sm.d_ncand = 0;
        sm.d_marked = 0;
        sm.d_nruns = 0;
        sm.d_fixed = __dadd_rn(c.bias, c.alpha);
        sm.d_fixed_lo = __double2float_rd(sm.d_fixed);
        sm.d_fixed_hi = __double2float_ru(sm.d_fixed);
        sm.d_fP = 0ull;
        sm.d_fC = kNoComposite;
    }
    pdl_wait();  // survivals and bins come from survival_kernel
    const int forced = resolve_forced(a);

    // (1) bins, keys, scan (its barriers publish the prologue's stores)
    uint32_t key[IPT];
    const int n_kept = select_bins<IPT>(a, sm, key);
    const bool bad_table = __syncthreads_or(order_bad) != 0;
    long long b_top = n_kept;  // largest in-range budget
    if (c.kind == DSPARK_COST_ADDITIVE) b_top = min(b_top, (long long)Mlast - (long long)B);
    const int b_top32 = (int)max(min(b_top, (long long)INT_MAX), -1LL);
    const double fixed_cost = sm.d_fixed;
    const float fixed_lo = sm.d_fixed_lo, fixed_hi = sm.d_fixed_hi;
    const bool has_forced = forced >= 0 && b_top >= 0 && !bad_table;
    const int b_forced = has_forced ? (int)min((long long)forced, b_top) : -1;

    // entry j's last budget b (false: its range holds none)
    auto entry_b = [&](int j, int &b) -> bool {
        const int2 r = ds.range[j];
        b = min(r.y, b_top32);
        return b >= r.x;
    };
    // the fp64 definition of entry j's cost is a positive finite number
    auto cost_ok = [&](int j) -> bool {
        const double vj = __ldg(c.val + j);
        if (c.kind == DSPARK_COST_SPS_1D) return vj > 0.0 && isfinite(vj);
        const double Tm = __dadd_rn(fixed_cost, vj);
        return Tm > 0.0 && isfinite(Tm);
    };
    // the staged value v rounded down and an upper bound one float ulp up;
    // the cost's bounds (SPS: v; additive: bias + alpha + v); false when
    // fp32 cannot bound theta (the fp64 cost is then checked)
    auto cost_bounds = [&](int j, float &k_lo, float &k_hi) -> bool {
        const float v_lo = ds.f32[j];
        const float v_hi = value_hi(v_lo);
        if (c.kind == DSPARK_COST_SPS_1D) {
            k_lo = v_lo;
            k_hi = v_hi;
            return v_lo > 0.0f && v_hi < INFINITY;  // SPS must be positive: 0 is flagged
        }
        k_lo = __fadd_rd(fixed_lo, v_lo);
        k_hi = __fadd_ru(fixed_hi, v_hi);
        return k_lo > 0.0f && k_hi < INFINITY;
    };
    // theta's bounds from tau's and the cost's
    auto theta_lo = [&](float t_lo, float k_lo, float k_hi) -> float {
        return c.kind == DSPARK_COST_SPS_1D ? __fmul_rd(t_lo, k_lo) : __fdiv_rd(t_lo, k_hi);
    };
    auto theta_hi = [&](float t_hi, float k_lo, float k_hi) -> float {
        return c.kind == DSPARK_COST_SPS_1D ? __fmul_ru(t_hi, k_hi) : __fdiv_ru(t_hi, k_lo);
    };

    // (2) per run: the last entry with a budget (the run's largest tau) is
    // bounded and its lower bound feeds the floor; the whole run is bounded
    // above by that tau with the run's largest SPS (smallest cost)
    int jl = -1;            // the run's last entry with a budget
    float run_hi = 0.0f;    // upper bound of theta over the run (NaN: none)
    if (!bad_table) {
        int bl = 0;
        for (int j = j1 - 1; j >= j0 && jl < 0; --j)
            if (entry_b(j, bl)) jl = j;
        float my_floor = 0.0f;
        if (jl >= 0) {
            // every budget of the run is at most bl: tau(bl) bounds them all;
            // the cost's bounds over the run from the prologue's value range
            // (over every entry of the run, a superset of those with a budget)
            float t_lo, t_hi, k_lo, k_hi, kr_lo, kr_hi;
            tau_interval(sm, B, bl, bl >= 1 ? bin_of_budget(sm, bl) : 0, t_lo, t_hi, a.status);
            if (cost_bounds(jl, k_lo, k_hi)) my_floor = theta_lo(t_lo, k_lo, k_hi);
            bool run_bounded;
            if (c.kind == DSPARK_COST_SPS_1D) {
                kr_lo = run_vmin;
                kr_hi = run_vmax;
                run_bounded = run_vmin > 0.0f && run_vmax < INFINITY;
            } else {
                kr_lo = __fadd_rd(fixed_lo, run_vmin);
                kr_hi = __fadd_ru(fixed_hi, run_vmax);
                run_bounded = kr_lo > 0.0f && kr_hi < INFINITY;
            }
            run_hi = run_bounded ? theta_hi(t_hi, kr_lo, kr_hi) : __int_as_float(0x7fffffff);
        }
        // non-negative floats order like their bits: one atomic per warp
        const unsigned wfloor = __reduce_max_sync(kFullMask, __float_as_uint(my_floor));
        if (lane == 0) atomicMax(&sm.d_floor, wfloor);
    }
    __syncthreads();
    const float floor_all = __uint_as_float(sm.d_floor);

    // (3) the runs that can hold the maximum are listed; then every entry
    // of theirs gets a thread and its own bounds: those whose upper bound
    // reaches the floor (or that fp32 cannot bound) are left, with their
    // budget and bin written over their stage range
    if (jl >= 0 && !(run_hi < floor_all)) {
        const int k = atomicAdd(&sm.d_nruns, 1);
        if (in_bounds(k, kSelThreads, a.status)) sm.d_runs[k] = tid;
    }
    __syncthreads();
    const int n_runs = min(sm.d_nruns, kSelThreads);
    bool my_bad_cost = false;
    for (int e = tid; e < n_runs * per; e += kSelThreads) {
        const int r = e / per;
        const int j = sm.d_runs[r] * per + (e - r * per);  // the run's thread t holds [t * per, ...)
        if (j >= n) continue;  // the table's last run is short
        int b;
        if (!entry_b(j, b)) continue;
        const int d = b >= 1 ? bin_of_budget(sm, b) : 0;
        float k_lo, k_hi;
        if (cost_bounds(j, k_lo, k_hi)) {
            float t_lo, t_hi;
            tau_interval(sm, B, b, d, t_lo, t_hi, a.status);
            if (theta_hi(t_hi, k_lo, k_hi) < floor_all) continue;
        } else if (!cost_ok(j)) {  // flagged; never a maximiser
            my_bad_cost = true;
            continue;
        }
        ds.range[j] = make_int2(b, d);
        const int slot = atomicAdd(&sm.d_ncand, 1);
        if (in_bounds(slot, n, a.status)) ds.list[slot] = j;
        if (b >= 1) mark_bin(sm, d, a.status);
    }
    if (tid == 0 && b_forced >= 1) mark_bin(sm, bin_of_budget(sm, b_forced), a.status);
    __syncthreads();
    const int K = min(sm.d_ncand, n);
    // the first candidate value of each thread's exact evaluation, in flight
    // while the bins are gathered
    const double v_first = tid < K ? __ldg(c.val + ds.list[tid]) : 0.0;

    long long my_key = -1;
    int my_b = 0x7FFFFFFF;
    unsigned long long my_P = 0ull, my_C = kNoComposite;
    // exact theta of entry j (value vj) at budget b with P, C*: the first
    // maximiser
    auto evaluate = [&](int j, double vj, int b, unsigned long long P, unsigned long long C) {
        const double tau = tau_of(B, (long long)P);
        double theta;
        if (c.kind == DSPARK_COST_SPS_1D) {
            if (!(vj > 0.0) || !isfinite(vj)) {
                my_bad_cost = true;
                return;
            }
            theta = __dmul_rn(tau, vj);
        } else {
            const double Tm = __dadd_rn(fixed_cost, vj);
            if (!(Tm > 0.0) || !isfinite(Tm)) {
                my_bad_cost = true;
                return;
            }
            theta = __ddiv_rn(tau, Tm);
        }
        const long long kk = __double_as_longlong(theta);  // positive: orders like the values
        if (cand_better(kk, b, my_key, my_b)) {
            my_key = kk;
            my_b = b;
            my_P = P;
            my_C = C;
        }
    };

    if (sm.d_marked <= kGather) {
        // (3) the marked bins' candidates in composite order, prefix-summed
        gather_marked<IPT>(a, sm, key, r0, k0);
        __syncthreads();
        const int m = min(sm.n_gather, kGather);
        rank_gathered_prefix(sm, m, a.status);
        __syncthreads();
        auto exact_at = [&](int b, int d, unsigned long long &P, unsigned long long &C) -> bool {
            return exact_at_budget(sm, m, b, d, P, C, a.status);
        };
        for (int i = tid; i < K; i += kSelThreads) {
            const int j = ds.list[i];
            const double vj = i == tid ? v_first : __ldg(c.val + j);
            const int2 bd = ds.range[j];
            unsigned long long P = 0ull, C = kNoComposite;
            if (bd.x >= 1 && !exact_at(bd.x, bd.y, P, C)) continue;
            evaluate(j, vj, bd.x, P, C);
        }
        if (tid == 0 && b_forced >= 1) {
            unsigned long long P, C;
            if (exact_at(b_forced, bin_of_budget(sm, b_forced), P, C)) {
                sm.d_fP = P;
                sm.d_fC = C;
            }
        }
    } else {
        // (4) crowded bins: the entries left, then the forced budget
        threshold_rounds<IPT>(
            a, sm, key, r0, k0, K, b_forced, [&](int i) { return ds.range[ds.list[i]].x; },
            [&](int i, int b, unsigned long long P, unsigned long long C) {
                const int j = ds.list[i];
                evaluate(j, __ldg(c.val + j), b, P, C);
            });
    }

    // the first maximiser over the block (in warp 0), the decision
    const bool any_bad_cost = block_first_max(sm, my_key, my_b, my_P, my_C, my_bad_cost);
    if (warp == 0 && lane == 0)
        write_decision(a, sm, my_key, my_b, my_P, my_C, any_bad_cost, bad_table, forced,
                       b_forced, [&](int budget, double tau) -> double {
                           // theta at the forced budget: the entry covering M = B + budget
                           const long long Mv = (long long)B + budget;
                           int lo = 0, hi = n;  // first M > Mv (1-D) / M >= Mv (additive)
                           while (lo < hi) {
                               const int mid = (lo + hi) >> 1;
                               const long long Mm = __ldg(c.M + mid);
                               const bool right = (c.kind == DSPARK_COST_SPS_1D) ? (Mm > Mv) : (Mm >= Mv);
                               if (right) hi = mid;
                               else lo = mid + 1;
                           }
                           if (c.kind == DSPARK_COST_SPS_1D) {
                               const double sps = __ldg(c.val + (lo > 0 ? lo - 1 : 0));
                               return sps > 0.0 && isfinite(sps) ? __dmul_rn(tau, sps) : 0.0;
                           }
                           if (lo >= n) return 0.0;
                           const double Tm = __dadd_rn(fixed_cost, __ldg(c.val + lo));
                           return Tm > 0.0 && isfinite(Tm) ? __ddiv_rn(tau, Tm) : 0.0;
                       });
    __syncthreads();

    // (5) lengths, tier-filled budget, pack (its inputs from global memory)
    select_finish<IPT>(a, sm, key, b_top, false);
}

// ------------------------------------------------------ interpolated select
//
// Interpolated additive tables ([AVS] §四: theta(M) read between the exported
// samples by linear interpolation, so every budget has its own cost and is a
// candidate) of at most kInterpMaxSamples samples, on one CTA, as
// dense_select_kernel plans dense tables, with budgets in the place of the
// table's entries:
//   (1) bins, keys, their scan;
//   (2) each thread holds a contiguous run of the budgets 0..b_top; tau's
//       interval at the run's last budget (the run's largest tau) and the
//       cost in fp32 (InterpWalk: T with its error bound, a reciprocal with
//       margins) at the run's ends and at the samples inside it (where the
//       piecewise-linear cost takes its minimum) bound theta over the run;
//       the last budget's lower bound feeds the floor;
//   (3) the runs reaching the floor are listed and each of their budgets is
//       bounded by a thread of its own; the budgets left (or that fp32
//       cannot bound, whose cost is checked in fp64) mark their bins;
//   (4) exact P and C* from the gathered bins (or the threshold slots when
//       they are crowded), T in fp64 from the samples and theta = tau / T;
//       the first maximiser wins;
//   (5) lengths, tier-filled budget and pack as in select_kernel.
// The samples (M as int32, the value as a float) are staged in shared memory
// before the dependency wait, then the list of budgets left.

constexpr int kInterpMaxSamples = 2048;
static_assert(8 * kInterpMaxSamples + 4 * (kMaxCandidates + 1) <= 4 * kStage,
              "samples and the budget list fit the stage");

// T(B, M) of the interpolated table at M = Mv from the staged samples (the
// segment by binary search; the fp64 values from global memory), as
// interp_cost: false when T is not a positive finite number.
__device__ __forceinline__ bool interp_cost_staged(const int32_t *sM, const double *val, int n,
                                                   long long Mv, double fixed_cost, double &T) {
    int j = -1;
    if (Mv > (long long)sM[0]) {
        int lo = 0, hi = n - 1;  // the last sample with M_j <= Mv
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((long long)sM[mid] <= Mv) lo = mid;
            else hi = mid - 1;
        }
        j = lo;
    }
    return interp_cost_at(sM, val, n, Mv, j, fixed_cost, T);
}

template <int IPT>
__global__ void __launch_bounds__(kSelThreads, 1) interp_select_kernel(PlanArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SelSmem &sm = *reinterpret_cast<SelSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.B, G = a.gamma;
    const CostArgs &c = a.cost;
    const int n = c.n;
    const int i0 = tid * IPT;
    const int r0 = i0 / G, k0 = i0 - r0 * G;
    int32_t *sM = sm.stage;
    float *sV = reinterpret_cast<float *>(sm.stage + n);
    int *list = sm.stage + 2 * n;  // budgets left by step (3)

    pdl_trigger();
    // while the survivals are computed: the samples, their order
    bool order_bad = false;
    for (int j = tid; j < n; j += kSelThreads) {
        if (!in_bounds(j, kInterpMaxSamples, a.status)) break;
        const int m = __ldg(c.M + j);
        sM[j] = m;
        sV[j] = (float)__ldg(c.val + j);
        if (j > 0 && !(m > __ldg(c.M + j - 1))) order_bad = true;
    }
    const int Mlast = __ldg(c.M + n - 1);
    if (tid < kHistBins / 32) sm.binmask[tid] = 0u;
    if (tid == 0) {
        sm.n_gather = 0;
        sm.d_floor = 0u;
        sm.d_ncand = 0;
        sm.d_marked = 0;
        sm.d_nruns = 0;
        sm.d_fixed = __dadd_rn(c.bias, c.alpha);
        sm.d_fixed32 = (float)sm.d_fixed;  // bias + alpha as a float (InterpWalk's bounds)
        sm.d_fP = 0ull;
        sm.d_fC = kNoComposite;
    }
    pdl_wait();  // survivals and bins come from survival_kernel
    const int forced = resolve_forced(a);

    // (1) bins, keys, scan (its barriers publish the prologue's stores)
    uint32_t key[IPT];
    const int n_kept = select_bins<IPT>(a, sm, key);
    const bool bad_table = __syncthreads_or(order_bad) != 0;
    const long long b_top = min((long long)n_kept, (long long)Mlast - (long long)B);
    const double fixed_cost = sm.d_fixed;
    const float fixed32 = sm.d_fixed32;
    const bool has_forced = forced >= 0 && b_top >= 0 && !bad_table;
    const int b_forced = has_forced ? (int)min((long long)forced, b_top) : -1;
    const int nb = (bad_table || b_top < 0) ? 0 : (int)b_top + 1;  // the budgets 0..b_top
    const int per = (nb + kSelThreads - 1) / kSelThreads;
    const int b0 = min(tid * per, nb), b1 = min(b0 + per, nb);

    // (2) the run's bound and the floor
    float run_hi = 0.0f;  // upper bound of theta over the run (NaN: none)
    {
        float my_floor = 0.0f;
        if (b0 < b1) {
            const int bl = b1 - 1;
            float t_lo, t_hi;
            tau_interval(sm, B, bl, bl >= 1 ? bin_of_budget(sm, bl) : 0, t_lo, t_hi, a.status);
            // theta <= tau(bl) / T over the run, and T (linear between the
            // samples, constant below the first) is smallest at an end of
            // the run or at a sample inside it: bounded at those only
            InterpWalk wk(sM, c.val, sV, n);
            wk.init((long long)B + b0);
            bool bounded = true;
            float lo, hi;
            auto at = [&](int b) {
                if (wk.bounds(B, b, t_hi, fixed32, lo, hi)) run_hi = fmaxf(run_hi, hi);
                else bounded = false;
            };
            at(b0);
            // the samples after b0's segment up to bl, in order (the table is
            // ascending here); at most n steps
            for (int q = wk.seg + 1; q < n && (long long)sM[q] <= (long long)B + bl; ++q) {
                const int bs = sM[q] - B;
                if (bs > b0) at(bs);
            }
            if (bl > b0) at(bl);
            if (!bounded) run_hi = __int_as_float(0x7fffffff);
            if (wk.bounds(B, bl, t_lo, fixed32, lo, hi)) my_floor = lo;
        }
        // non-negative floats order like their bits: one atomic per warp
        const unsigned wfloor = __reduce_max_sync(kFullMask, __float_as_uint(my_floor));
        if (lane == 0) atomicMax(&sm.d_floor, wfloor);
    }
    __syncthreads();
    const float floor_all = __uint_as_float(sm.d_floor);

    // (3) the runs that can hold the maximum, then each of their budgets
    if (b0 < b1 && !(run_hi < floor_all)) {
        const int k = atomicAdd(&sm.d_nruns, 1);
        if (in_bounds(k, kSelThreads, a.status)) sm.d_runs[k] = tid;
    }
    __syncthreads();
    const int n_runs = min(sm.d_nruns, kSelThreads);
    bool my_bad_cost = false;
    for (int e = tid; e < n_runs * per; e += kSelThreads) {
        const int r = e / per;
        const int b = sm.d_runs[r] * per + (e - r * per);  // the run's thread t holds [t * per, ...)
        if (b >= nb) continue;  // the last run is short
        const int d = b >= 1 ? bin_of_budget(sm, b) : 0;
        float t_lo, t_hi, lo, hi;
        tau_interval(sm, B, b, d, t_lo, t_hi, a.status);
        InterpWalk wk(sM, c.val, sV, n);
        wk.init((long long)B + b);
        if (wk.bounds(B, b, t_hi, fixed32, lo, hi)) {
            if (hi < floor_all) continue;
        } else {
            double T;
            if (!interp_cost_staged(sM, c.val, n, (long long)B + b, fixed_cost, T)) {
                my_bad_cost = true;  // flagged; never a maximiser
                continue;
            }
        }
        const int slot = atomicAdd(&sm.d_ncand, 1);
        if (in_bounds(slot, kMaxCandidates + 1, a.status)) list[slot] = b;
        if (b >= 1) mark_bin(sm, d, a.status);
    }
    if (tid == 0 && b_forced >= 1) mark_bin(sm, bin_of_budget(sm, b_forced), a.status);
    __syncthreads();
    const int K = min(sm.d_ncand, kMaxCandidates + 1);

    long long my_key = -1;
    int my_b = 0x7FFFFFFF;
    unsigned long long my_P = 0ull, my_C = kNoComposite;
    // exact theta at budget b with P, C*: the first maximiser
    auto evaluate = [&](int b, unsigned long long P, unsigned long long C) {
        double T;
        if (!interp_cost_staged(sM, c.val, n, (long long)B + b, fixed_cost, T)) {
            my_bad_cost = true;
            return;
        }
        const double theta = __ddiv_rn(tau_of(B, (long long)P), T);
        const long long kk = __double_as_longlong(theta);  // positive: orders like the values
        if (cand_better(kk, b, my_key, my_b)) {
            my_key = kk;
            my_b = b;
            my_P = P;
            my_C = C;
        }
    };

    if (sm.d_marked <= kGather) {
        // (4) the marked bins' candidates in composite order, prefix-summed
        gather_marked<IPT>(a, sm, key, r0, k0);
        __syncthreads();
        const int m = min(sm.n_gather, kGather);
        rank_gathered_prefix(sm, m, a.status);
        __syncthreads();
        for (int i = tid; i < K; i += kSelThreads) {
            const int b = list[i];
            unsigned long long P = 0ull, C = kNoComposite;
            if (b >= 1 && !exact_at_budget(sm, m, b, bin_of_budget(sm, b), P, C, a.status)) continue;
            evaluate(b, P, C);
        }
        if (tid == 0 && b_forced >= 1) {
            unsigned long long P, C;
            if (exact_at_budget(sm, m, b_forced, bin_of_budget(sm, b_forced), P, C, a.status)) {
                sm.d_fP = P;
                sm.d_fC = C;
            }
        }
    } else {
        // (4) crowded bins: the budgets left, then the forced budget
        threshold_rounds<IPT>(
            a, sm, key, r0, k0, K, b_forced, [&](int i) { return list[i]; },
            [&](int, int b, unsigned long long P, unsigned long long C) { evaluate(b, P, C); });
    }

    // the first maximiser over the block (in warp 0), the decision
    const bool any_bad_cost = block_first_max(sm, my_key, my_b, my_P, my_C, my_bad_cost);
    if (warp == 0 && lane == 0)
        write_decision(a, sm, my_key, my_b, my_P, my_C, any_bad_cost, bad_table, forced,
                       b_forced, [&](int budget, double tau) -> double {
                           // theta at the forced budget: the cost interpolated at M = B + budget
                           double Ti;
                           return interp_cost_staged(sM, c.val, n, (long long)B + budget,
                                                     fixed_cost, Ti)
                                      ? __ddiv_rn(tau, Ti) : 0.0;
                       });
    __syncthreads();

    // (5) lengths, tier-filled budget, pack (its inputs from global memory)
    select_finish<IPT>(a, sm, key, b_top, false);
}

// The select kernels launch with the largest dynamic shared memory a CTA
// may have, more than SelSmem needs, so that their one CTA has an SM to
// itself: with 56 registers a thread, 1024 threads leave room for one CTA of
// the argmax kernel, and a step whose planner shared its SM with the
// previous step's argmax took 102 us instead of 90 in the chained bench
// loop (dsv4_like).
constexpr size_t kSelLaunchSmem = 227 * 1024;
static_assert(sizeof(SelSmem) <= kSelLaunchSmem, "SelSmem fits the launch");
size_t select_smem_bytes() { return kSelLaunchSmem; }


// Which planner kernel takes a cost table: select_kernel for at most
// kMaxSelect entries, dense_select_kernel for more (at most
// kDenseMaxEntries), interp_select_kernel for interpolated tables of at most
// kInterpMaxSamples samples, rank_kernel for the rest.
enum class PlanPath { kSelect, kDense, kInterp, kRank };

PlanPath plan_path(const dspark_cost_table *cost) {
    if (cost->kind == DSPARK_COST_ADDITIVE_INTERP)
        return cost->n <= kInterpMaxSamples ? PlanPath::kInterp : PlanPath::kRank;
    if (cost->n <= kMaxSelect) return PlanPath::kSelect;
    return cost->n <= kDenseMaxEntries ? PlanPath::kDense : PlanPath::kRank;
}

template <int IPT>
cudaError_t launch_select(const PlanArgs &a, PlanPath path, cudaStream_t s) {
    // shared-memory attribute slots: 1-5 select, 10-14 dense, 15-19 interp
    const int slot = (IPT == 1 ? 1 : IPT == 2 ? 2 : IPT == 4 ? 3 : IPT == 8 ? 4 : 5) +
                     (path == PlanPath::kDense ? 9 : path == PlanPath::kInterp ? 14 : 0);
    void (*kernel)(PlanArgs) = path == PlanPath::kDense    ? dense_select_kernel<IPT>
                               : path == PlanPath::kInterp ? interp_select_kernel<IPT>
                                                           : select_kernel<IPT>;
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(kernel), (int)select_smem_bytes(), slot);
    if (e != cudaSuccess) return e;
    return launch_pdl(kernel, dim3(1), dim3(kSelThreads), select_smem_bytes(), s, a);
}

}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_plan_workspace_bytes(int32_t B, int32_t gamma) {
    if (B < 1 || gamma < 1) return 256;
    return (plan_scratch_bytes(B, B * gamma) + 255) & ~size_t(255);
}

namespace {

// Argument checks of dspark_plan; DSPARK_OK when the call may proceed.
int check_plan(const float *conf_logits, const float *sts_temps, const dspark_plan_params *p,
               const dspark_cost_table *cost, float *survivals, int32_t *verify_lens,
               int32_t *budget, double *tau_theta, void *workspace, size_t workspace_bytes,
               int32_t *status) {
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
    if (cost->kind != DSPARK_COST_SPS_1D && cost->kind != DSPARK_COST_ADDITIVE &&
        cost->kind != DSPARK_COST_ADDITIVE_INTERP)
        return DSPARK_ERR_INVALID_ARG;
    if (cost->n < 1 || !cost->M || !cost->val) return DSPARK_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < dspark_plan_workspace_bytes(p->B, p->gamma) ||
        !aligned(workspace, 256))
        return DSPARK_ERR_WORKSPACE;
    return DSPARK_OK;
}

// One planner pass over survivals already computed, on the kernel plan_path
// chose.
int launch_pass(PlanArgs a, PlanPath path, cudaStream_t s) {
    if (path != PlanPath::kRank) {
        const int ipt = (a.N + kSelThreads - 1) / kSelThreads;
        cudaError_t e;
        if (ipt <= 1) e = launch_select<1>(a, path, s);
        else if (ipt <= 2) e = launch_select<2>(a, path, s);
        else if (ipt <= 4) e = launch_select<4>(a, path, s);
        else if (ipt <= 8) e = launch_select<8>(a, path, s);
        else e = launch_select<16>(a, path, s);
        if (e == cudaSuccess) return DSPARK_OK;
        // the bins survival_kernel filled must not reach the next call
        cudaMemsetAsync(&a.scratch->hcount[0], 0,
                        sizeof(a.scratch->hcount) + sizeof(a.scratch->hsum), s);
        return DSPARK_ERR_CUDA;
    }
    a.pk.on = false;
    const size_t smem = rank_smem_bytes(a.B, a.P2, a.N, a.cost.kind);
    if (ensure_smem(reinterpret_cast<const void *>(rank_kernel), (int)rank_smem_max(), 0) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    // ranking is issue-bound: at least a few candidates per CTA, else every
    // SM (one CTA each)
    int grid = (a.N + kRankMinPerCta - 1) / kRankMinPerCta;
    grid = grid < 1 ? 1 : (grid > sm_count() ? sm_count() : grid);
    return launch_pdl(rank_kernel, dim3(grid), dim3(kRankThreads), smem, s, a) == cudaSuccess
               ? DSPARK_OK
               : DSPARK_ERR_CUDA;
}

// The planner's launches.  Without options: survival_kernel, then one
// pass.  opt->lagged_conf_logits: a first survival + pass on the lagged
// confidences chooses the budget, and the pass on the current ones
// allocates it ([AVS] §三: lagged confidence sets the budget, the current
// one the allocation).  opt->align_to_tiers: a pass chooses the budget and
// the tier-filled budget, and a last pass allocates that.  pk.on: the last
// pass also packs the verify window (the select path in the same kernel,
// the rank path with the pack kernel after it).
int run_plan(const float *conf_logits, const float *sts_temps, const dspark_plan_params *p,
             const dspark_cost_table *cost, const dspark_plan_options *opt, float *survivals,
             int32_t *verify_lens, int32_t *budget, double *tau_theta, void *workspace,
             int32_t *status, const PackArgs &pk, const TierArgs &align, cudaStream_t s) {
    const int B = p->B, G = p->gamma, N = B * G;
    PlanScratch *scratch = static_cast<PlanScratch *>(workspace);
    PassScratch *ps = scratch_at<PassScratch>(scratch, plan_pass_offset(B, N));
    int32_t *pass_lens = scratch_at<int32_t>(scratch, plan_pass_lens_offset(B, N));
    float *lagged_surv = scratch_at<float>(scratch, plan_pass_surv_offset(B, N));
    // one-CTA select (few candidate budgets, a dense table bounded per
    // entry, an interpolated table bounded per budget), else the rank path
    const PlanPath path = plan_path(cost);
    const bool select = path != PlanPath::kRank;  // the survival kernel bins the keys
    const int32_t *conf_gen = opt ? opt->conf_generation : nullptr;
    const int32_t *req_gen = opt ? opt->req_generation : nullptr;
    const bool lagged = opt && opt->lagged_conf_logits;
    const int sblocks = (B * 32 + kSurvThreads - 1) / kSurvThreads;

    PlanArgs a;
    a.B = B;
    a.gamma = G;
    a.N = N;
    a.P2 = pow2_at_least(G);
    a.eps = p->survival_eps;
    a.min_len = p->min_verify_len;
    a.max_len = p->max_verify_len;
    a.forced = p->forced_budget;
    a.cost = CostArgs{cost->kind, cost->n, cost->M, cost->val, cost->bias_ms, cost->alpha_ms};
    a.status = status;
    a.scratch = scratch;
    a.pk = PackArgs{};
    a.pk.on = false;
    a.forced_dev = nullptr;
    a.more_passes = false;
    a.align.n = 0;
    a.exec_budget = nullptr;
    // outputs of a pass whose results only the next pass reads
    a.verify_lens = pass_lens;
    a.budget = &ps->pass_budget;
    a.tau_theta = ps->pass_tau_theta;

    int rc;
    if (lagged) {
        if (launch_pdl(survival_kernel, dim3(sblocks), dim3(kSurvThreads), 0, s,
                       opt->lagged_conf_logits, sts_temps, B, G, p->survival_eps,
                       p->max_verify_len - 1, select, conf_gen, req_gen, lagged_surv, status,
                       scratch) != cudaSuccess)
            return DSPARK_ERR_CUDA;
        a.surv = lagged_surv;
        a.budget = &ps->lagged_budget;
        if ((rc = launch_pass(a, path, s)) != DSPARK_OK) return rc;
        a.budget = &ps->pass_budget;
        a.forced_dev = &ps->lagged_budget;
    }
    if (launch_pdl(survival_kernel, dim3(sblocks), dim3(kSurvThreads), 0, s, conf_logits,
                   sts_temps, B, G, p->survival_eps, p->max_verify_len - 1, select, conf_gen,
                   req_gen, survivals, status, scratch) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    a.surv = survivals;
    if (align.n > 0) {
        a.more_passes = true;
        a.align = align;
        a.exec_budget = &ps->exec_budget;
        if ((rc = launch_pass(a, path, s)) != DSPARK_OK) return rc;
        a.more_passes = false;
        a.align.n = 0;
        a.exec_budget = nullptr;
        a.forced_dev = &ps->exec_budget;
    }
    a.verify_lens = verify_lens;
    a.budget = budget;
    a.tau_theta = tau_theta;
    a.pk = pk;
    if ((rc = launch_pass(a, path, s)) != DSPARK_OK) return rc;
    if (!select && pk.on &&
        launch_pack(true, pk.anchor, pk.draft, pk.prefix, verify_lens, B, G, pk.tiers, pk.capacity,
                    pk.ids, pk.pos, pk.req, pk.src, pk.cu, pk.totals, status, s) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    return DSPARK_OK;
}

// Checks of the options; DSPARK_OK when they may be used.
int check_options(const dspark_plan_options *opt, TierArgs *align, const int32_t *pack_tiers,
                  int32_t pack_n_tiers) {
    align->n = 0;
    if (!opt) return DSPARK_OK;
    if ((opt->conf_generation == nullptr) != (opt->req_generation == nullptr))
        return DSPARK_ERR_INVALID_ARG;
    if (opt->align_to_tiers) {
        const int32_t *t = pack_tiers ? pack_tiers : opt->host_tiers;
        const int32_t n = pack_tiers ? pack_n_tiers : opt->n_tiers;
        if (n < 1 || !load_tiers(t, n, align)) return DSPARK_ERR_INVALID_ARG;
    }
    return DSPARK_OK;
}

}  // namespace

extern "C" int dspark_plan(const float *conf_logits, const float *sts_temps,
                           const dspark_plan_params *p, const dspark_cost_table *cost,
                           float *survivals, int32_t *verify_lens, int32_t *budget,
                           double *tau_theta, void *workspace, size_t workspace_bytes,
                           int32_t *status, void *stream) {
    return dspark_plan_ex(conf_logits, sts_temps, p, cost, nullptr, survivals, verify_lens,
                          budget, tau_theta, workspace, workspace_bytes, status, stream);
}

extern "C" int dspark_plan_ex(const float *conf_logits, const float *sts_temps,
                              const dspark_plan_params *p, const dspark_cost_table *cost,
                              const dspark_plan_options *opt, float *survivals,
                              int32_t *verify_lens, int32_t *budget, double *tau_theta,
                              void *workspace, size_t workspace_bytes, int32_t *status,
                              void *stream) {
    int rc = check_plan(conf_logits, sts_temps, p, cost, survivals, verify_lens, budget,
                        tau_theta, workspace, workspace_bytes, status);
    if (rc != DSPARK_OK) return rc;
    TierArgs align;
    if ((rc = check_options(opt, &align, nullptr, 0)) != DSPARK_OK) return rc;
    PackArgs pk = {};
    pk.on = false;
    return run_plan(conf_logits, sts_temps, p, cost, opt, survivals, verify_lens, budget,
                    tau_theta, workspace, status, pk, align, static_cast<cudaStream_t>(stream));
}

extern "C" int dspark_plan_pack(const float *conf_logits, const float *sts_temps,
                                const dspark_plan_params *p, const dspark_cost_table *cost,
                                float *survivals, int32_t *verify_lens, int32_t *budget,
                                double *tau_theta, const int32_t *anchor, const int32_t *draft,
                                const int32_t *prefix_lens, const int32_t *host_tiers,
                                int32_t n_tiers, int32_t capacity, int32_t *packed_ids,
                                int32_t *packed_pos, int32_t *packed_req, int32_t *packed_src,
                                int32_t *cu_seqlens, int32_t *totals, void *workspace,
                                size_t workspace_bytes, int32_t *status, void *stream) {
    return dspark_plan_pack_ex(conf_logits, sts_temps, p, cost, nullptr, survivals, verify_lens,
                               budget, tau_theta, anchor, draft, prefix_lens, host_tiers, n_tiers,
                               capacity, packed_ids, packed_pos, packed_req, packed_src,
                               cu_seqlens, totals, workspace, workspace_bytes, status, stream);
}

extern "C" int dspark_plan_pack_ex(const float *conf_logits, const float *sts_temps,
                                   const dspark_plan_params *p, const dspark_cost_table *cost,
                                   const dspark_plan_options *opt, float *survivals,
                                   int32_t *verify_lens, int32_t *budget, double *tau_theta,
                                   const int32_t *anchor, const int32_t *draft,
                                   const int32_t *prefix_lens, const int32_t *host_tiers,
                                   int32_t n_tiers, int32_t capacity, int32_t *packed_ids,
                                   int32_t *packed_pos, int32_t *packed_req, int32_t *packed_src,
                                   int32_t *cu_seqlens, int32_t *totals, void *workspace,
                                   size_t workspace_bytes, int32_t *status, void *stream) {
    int rc = check_plan(conf_logits, sts_temps, p, cost, survivals, verify_lens, budget,
                        tau_theta, workspace, workspace_bytes, status);
    if (rc != DSPARK_OK) return rc;
    if (!anchor || !draft || !prefix_lens || !packed_ids || !packed_pos || !packed_req ||
        !packed_src || !cu_seqlens || !totals || capacity < 0)
        return DSPARK_ERR_INVALID_ARG;
    PackArgs pk = {};
    if (!load_tiers(host_tiers, n_tiers, &pk.tiers)) return DSPARK_ERR_INVALID_ARG;
    TierArgs align;
    if ((rc = check_options(opt, &align, host_tiers, n_tiers)) != DSPARK_OK) return rc;
    pk.on = true;
    pk.anchor = anchor;
    pk.draft = draft;
    pk.prefix = prefix_lens;
    pk.capacity = capacity;
    pk.ids = packed_ids;
    pk.pos = packed_pos;
    pk.req = packed_req;
    pk.src = packed_src;
    pk.cu = cu_seqlens;
    pk.totals = totals;
    return run_plan(conf_logits, sts_temps, p, cost, opt, survivals, verify_lens, budget,
                    tau_theta, workspace, status, pk, align, static_cast<cudaStream_t>(stream));
}
