// calib.cu -- STS recorder, calibration statistics and the sequential
// temperature fit on sm_103a.
//
// Pages (by title and section):
//   [AVS] "DSpark 自适应 Verify 怎样分配候选预算" §二 (the STS recorder labels
//         a step with the greedy prefix mask, position k set iff k <
//         num_correct_drafts; the fitter searches a temperature position by
//         position, keeping the cumulative survival of the positions already
//         fitted, and takes the one of lower ECE), §七 A (per-position and
//         cumulative calibration, ECE, Brier)
//   [TUT] charlestar.github.io tutorial, "为什么置信度必须校准" (binned ECE;
//         a position's label only means something once the earlier
//         positions survived), "截短会制造观测盲区" (positions past a compact
//         window are censored), "置信度质量" (reliability diagram, ECE,
//         Brier score or log loss, by depth)
//
// A recorded sample is (z[gamma], correct, tested): tested = drafts the
// target checked, correct = accepted drafts among them.  Depth k is observed
// iff k < tested (a depth past the window stays out even when the chain broke
// inside it: keeping it only when its label is known to be 0 would bias the
// labels).  Label y_k = (k < correct).  Two flavours per depth: the
// cumulative survival S_k over observed samples, and the conditional c_k over
// observed samples whose prefix survived through k-1 (correct >= k).
//
// Bins and exact sums.  A confidence p (an fp32 in [0, 1]) enters as q =
// floor(p * 2^32), an integer (p * 2^32 is exact in fp32); its bin is
// min(q * n_bins >> 32, n_bins - 1), which equals floor(p * n_bins) (for p >=
// 2^-8 q is p * 2^32 itself, below it both are 0).  Bin counts, label counts
// and confidence sums are integers added with integer atomics, so they and
// ECE * n * 2^32 = sum_b |L_b 2^32 - C_b| do not depend on the order in which
// the GPU adds them.  Brier and log-loss terms are float pairs (the square
// exact to ~2^-47, -ln p to ~2^-43 absolute), summed as float pairs over a
// warp tree and within a warp's slot, then in fp64 over warps and CTAs in
// order: deterministic, within ~1e-13 of a sequential fp64 sum.
//
// Kernels
//   sts_record_kernel  one CTA: block scans number the selected requests,
//                      rows land at (cursor + i) mod capacity, coalesced
//                      element copies; the cursor lives on the device, so
//                      a captured graph can record every step.
//   calib_stats_kernel each thread holds two samples in registers over the
//                      depth loop (the fp32 survival product runs left to
//                      right); per (flavour, depth) a sample's bin gets
//                      count + (label << 32) and its confidence by shared
//                      atomics, its Brier and log-loss terms add to float
//                      pairs that one warp reduction per depth and pass
//                      folds into the warp's slot; CTAs add their
//                      histograms to a global one with u64 atomics and the
//                      last CTA (atomic ticket, no waiting) turns it into
//                      the metrics.
//   sts_fit_kernel     one launch per depth (programmatic serialization
//                      chains them).  A CTA stages a tile of 256 samples --
//                      z_k, the survival S_{k-1} under the temperatures
//                      already chosen (updated in place in the workspace),
//                      the label and whether the sample counts -- then every
//                      thread owns one grid temperature (and one phase of the
//                      tile when there are fewer than 256 candidates) and
//                      adds each sample's p = S_{k-1} * c(z_k, T_j) to bins
//                      private to the thread (shared memory, [bin][thread]
//                      layout: no atomics, no bank conflicts).  The CTA
//                      folds its phases into global per-candidate histograms
//                      with atomics; the last CTA scores every candidate
//                      (exact integer ECE), picks the lowest (ties to the
//                      lower index) and clears the histograms for the next
//                      depth.  The work is N * J sigmoids per depth, four
//                      interleaved per thread over tiles compacted to the
//                      samples that count: the kernel is bound by
//                      instruction issue, not by memory.
//
// No kernel waits on another CTA: the last-CTA tickets never spin.

#include "dspark_common.cuh"

namespace dspark {

constexpr int kRecThreads = 512;
constexpr int kStatsThreads = 256;
constexpr int kStatsWarps = kStatsThreads / 32;
constexpr int kStatsMaxCtas = 1024;
constexpr int kFitThreads = 256;
constexpr int kFitTile = 256;  // samples staged per step
constexpr int kMaxBins = 32;
constexpr int kMaxTemps = 256;
constexpr int kMaxGamma = 31;
constexpr long long kMaxSamples = 0x7fffffffLL;  // bin counters of a CTA or thread are 32-bit
constexpr double kQ32 = 4294967296.0;

// q = floor(p * 2^32) for p in [0, 1], from the bits of p: p = 1.f * 2^e
// gives (1.f * 2^23) shifted by e + 9 (integer work only; float-to-integer
// conversions run on the fp64 unit)
__device__ __forceinline__ unsigned long long conf_q(float p) {
    const unsigned bits = __float_as_uint(p);
    const int sh = (int)(bits >> 23) - 127 + 9;  // e + 9; p in [0, 1] is never negative
    const unsigned long long m = (unsigned long long)((bits & 0x007fffffu) | 0x00800000u);
    if (sh >= 0) return m << sh;                  // e >= -9 (p = 1: 2^23 << 9)
    return sh > -24 ? m >> (-sh) : 0ull;          // below 2^-32 (and +0, subnormals): 0
}

// --- float-pair terms of the Brier score and the log loss (no fp64 in the
// per-sample work: GB300's fp64 unit is 1/64 of its fp32 rate)

// (p - y)^2 as hi + lo (relative error ~2^-47)
__device__ __forceinline__ void brier_pair(float p, bool y, float &hi, float &lo) {
    float dh, dl;
    two_sum(p, y ? -1.0f : 0.0f, dh, dl);
    hi = __fmul_rn(dh, dh);
    lo = fmaf(dh, dh, -hi);
    lo = fmaf(__fmul_rn(2.0f, dh), dl, lo);
}

// -ln q for q = qh + ql in [2^-24, 1] (absolute error ~2^-43): a float
// estimate y0 of ln q, then ln q = y0 + ln(1 + w) with w = q e^{-y0} - 1
// (|w| < 2^-20, so w - w^2/2 leaves an error below 2^-60).
__device__ __forceinline__ void neglog_pair(float qh, float ql, float &hi, float &lo) {
    const float y0 = __logf(qh);
    float eh, el;
    exp_pair(-y0, eh, el);
    const float ph = __fmul_rn(qh, eh);
    float pl = fmaf(qh, eh, -ph);
    pl = fmaf(qh, el, fmaf(ql, eh, pl));
    const float w = __fadd_rn(__fsub_rn(ph, 1.0f), pl);  // ph - 1 is exact
    const float l1 = __fsub_rn(w, __fmul_rn(__fmul_rn(0.5f, w), w));
    two_sum(-y0, -l1, hi, lo);
}

// hi + lo summed over the warp (every lane gets the sum)
__device__ __forceinline__ void warp_sum_pair(float &hi, float &lo) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float oh = __shfl_xor_sync(kFullMask, hi, o), ol = __shfl_xor_sync(kFullMask, lo, o);
        float s, e;
        two_sum(hi, oh, s, e);
        e = __fadd_rn(e, __fadd_rn(lo, ol));
        fast_two_sum(s, e, hi, lo);
    }
}

// (ah, al) += hi + lo, all float pairs
__device__ __forceinline__ void acc_pair(float &ah, float &al, float hi, float lo) {
    float s, e;
    two_sum(ah, hi, s, e);
    e = __fadd_rn(e, __fadd_rn(al, lo));
    fast_two_sum(s, e, ah, al);
}

// acc (a float pair in shared memory) += hi + lo
__device__ __forceinline__ void add_pair(float *acc, float hi, float lo) {
    float s, e;
    two_sum(acc[0], hi, s, e);
    e = __fadd_rn(e, __fadd_rn(acc[1], lo));
    fast_two_sum(s, e, acc[0], acc[1]);
}

__device__ __forceinline__ int conf_bin(unsigned long long q, int M) {
    const unsigned long long b = (q * (unsigned long long)M) >> 32;
    return b < (unsigned long long)(M - 1) ? (int)b : M - 1;
}

// tested clamped to [0, gamma], correct to [0, tested]
__device__ __forceinline__ bool sample_lens(int32_t correct, int32_t tested, int gamma, int &c,
                                            int &t) {
    bool bad = false;
    t = tested;
    c = correct;
    if (t < 0 || t > gamma) {
        bad = true;
        t = t < 0 ? 0 : gamma;
    }
    if (c < 0 || c > t) {
        bad = true;
        c = c < 0 ? 0 : t;
    }
    return bad;
}

// |L 2^32 - C| summed over the bins of one histogram [M][3]
__device__ __forceinline__ unsigned long long ece_numerator(const unsigned long long *h, int M,
                                                            unsigned long long *n_out) {
    unsigned long long E = 0, n = 0;
    for (int b = 0; b < M; ++b) {
        const unsigned long long cnt = __ldcg(h + 3 * b), L = __ldcg(h + 3 * b + 1) << 32,
                                 C = __ldcg(h + 3 * b + 2);
        n += cnt;
        E += L > C ? L - C : C - L;
    }
    *n_out = n;
    return E;
}

__device__ __forceinline__ double ece_of(unsigned long long E, unsigned long long n) {
    return n ? __ddiv_rn((double)E, __dmul_rn((double)n, kQ32)) : 0.0;
}

// ------------------------------------------------------------------ recorder

struct RecordArgs {
    const float *z;
    const int32_t *correct;
    const int32_t *verify_lens;  // nullable: the full block was verified
    const uint8_t *select;       // nullable: every request
    int B, gamma;
    float *rec_z;
    int32_t *rec_correct, *rec_tested;
    long long capacity;
    unsigned long long *cursor;
    uint8_t *mask;  // nullable
    int32_t *status;
};

__global__ void __launch_bounds__(kRecThreads) sts_record_kernel(RecordArgs a) {
    __shared__ int scan_tmp[33];
    __shared__ long long slot_s[kRecThreads];
    __shared__ int corr_s[kRecThreads];
    __shared__ unsigned long long off_s, first_s;
    __shared__ long long count_s;
    pdl_trigger();
    pdl_wait();  // num_correct / verify_lens come from the accept
    const int tid = threadIdx.x, G = a.gamma;
    const unsigned long long cap = (unsigned long long)a.capacity;
    // selected rows in all; a second pass over `select` only when the
    // requests span more than one chunk
    long long count = a.B;
    if (a.select && a.B > kRecThreads) {
        int mine = 0;
        for (int r = tid; r < a.B; r += kRecThreads) mine += a.select[r] ? 1 : 0;
        count = block_sum<int>(mine, scan_tmp);
    }
    bool bad_len = false;
    long long base = 0;
    for (int r0 = 0; r0 < a.B; r0 += kRecThreads) {
        const int rows = min(kRecThreads, a.B - r0);
        const int nel = rows * G;
        // every load of the chunk is issued before the scan
        float zr[kMaxGamma];
#pragma unroll
        for (int i = 0; i < kMaxGamma; ++i) {
            const int e = tid + i * kRecThreads;
            if (i < G && e < nel) zr[i] = a.z[(size_t)r0 * G + e];
        }
        const int r = r0 + tid;
        int tested = G, c = 0;
        bool sel = false;
        if (r < a.B) {
            c = a.correct[r];
            sel = !a.select || a.select[r];
            if (a.verify_lens) {
                int L = a.verify_lens[r];
                if (L < 1 || L > G + 1) {
                    bad_len = true;
                    L = L < 1 ? 1 : G + 1;
                }
                tested = L - 1;
            }
            if (c < 0 || c > tested) {
                bad_len = true;
                c = c < 0 ? 0 : tested;
            }
        }
        int tot;
        const int pre = block_exclusive_scan<int>(sel ? 1 : 0, scan_tmp, &tot);
        if (r0 == 0 && tid == 0) {
            const long long n = (a.select && a.B <= kRecThreads) ? tot : count;
            // more rows than slots: only the last `capacity` are written
            const unsigned long long skip =
                n > a.capacity ? (unsigned long long)(n - a.capacity) : 0ull;
            count_s = n;
            first_s = skip;
            off_s = (*a.cursor % cap + skip % cap) % cap;  // slot of row `skip`
        }
        __syncthreads();
        count = count_s;
        const unsigned long long first = first_s;
        const unsigned long long i = (unsigned long long)(base + pre);
        long long slot = -1;
        if (sel && i >= first) {
            unsigned long long s = off_s + (i - first);  // i - first < capacity
            slot = (long long)(s >= cap ? s - cap : s);
            if (in_bounds(slot, a.capacity, a.status)) {
                a.rec_correct[slot] = c;
                a.rec_tested[slot] = tested;
            } else {
                slot = -1;
            }
        }
        slot_s[tid] = slot;
        corr_s[tid] = c;
        __syncthreads();
#pragma unroll
        for (int i2 = 0; i2 < kMaxGamma; ++i2) {
            const int e = tid + i2 * kRecThreads;
            if (i2 < G && e < nel) {
                const int rr = e / G, k = e - rr * G;
                const long long sl = slot_s[rr];
                if (sl >= 0) a.rec_z[(size_t)sl * G + k] = zr[i2];
                if (a.mask) a.mask[(size_t)r0 * G + e] = (uint8_t)(k < corr_s[rr]);
            }
        }
        __syncthreads();
        base += tot;
    }
    if (__syncthreads_or(bad_len) && tid == 0) flag(a.status, DSPARK_STATUS_BAD_LEN);
    if (tid == 0) {
        *a.cursor += (unsigned long long)count;
        if (count > a.capacity) flag(a.status, DSPARK_STATUS_CAPACITY);
    }
}

// -------------------------------------------------------------------- STS

// c[r][k] = sigmoid(z[r][k] / T[k]), elementwise over a grid-stride loop.
__global__ void __launch_bounds__(256) sts_confidence_kernel(const float *z, const float *T,
                                                             long long n, int gamma, float *c,
                                                             int32_t *status) {
    pdl_trigger();
    pdl_wait();
    bool bad = false;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float zi = z[i], Ti = __ldg(T + i % gamma);
        bad |= (zi != zi) || !(Ti > 0.0f);
        c[i] = sts_confidence(zi, Ti);
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag(status, DSPARK_STATUS_BAD_INPUT);
}

// --------------------------------------------------------------- statistics

struct StatsArgs {
    const float *z;
    const int32_t *correct, *tested;
    long long N;
    int gamma, M;
    const float *T;
    unsigned long long *hist_ws;   // [2][gamma][M][3], all zero between calls
    double *part_ws;               // [gridDim.x][2][gamma][2]
    unsigned int *ticket;          // zero between calls
    unsigned long long *hist_out;  // nullable
    double *metrics;               // [2][gamma][4]
    int32_t *status;
};

// One (prediction, label) of flavour f at depth k: the bin of the CTA's
// histogram gets count + (label << 32) and floor(p 2^32) by shared atomics;
// the Brier and log-loss terms add to the thread's float pairs acc[0..3].
__device__ __forceinline__ void stats_add(unsigned long long *hs, float *acc, int f, int k,
                                          float p, bool y, int G, int M, int32_t *status) {
    const unsigned long long q = conf_q(p);
    const int bin = conf_bin(q, M);
    if (in_bounds(bin, M, status)) {
        unsigned long long *h = hs + ((size_t)(f * G + k) * M + bin) * 2;
        atomicAdd(h, 1ull + ((unsigned long long)y << 32));
        atomicAdd(h + 1, q);
    }
    float th, tl;
    brier_pair(p, y, th, tl);
    acc_pair(acc[0], acc[1], th, tl);
    const float pc = fminf(fmaxf(p, 0x1p-24f), 1.0f - 0x1p-24f);
    float qh = pc, ql = 0.0f;
    if (!y) two_sum(1.0f, -pc, qh, ql);  // 1 - pc exactly
    neglog_pair(qh, ql, th, tl);
    acc_pair(acc[2], acc[3], th, tl);
}

constexpr int kStatsR = 2;  // samples per thread held across the depth loop

__global__ void __launch_bounds__(kStatsThreads) calib_stats_kernel(StatsArgs a) {
    // [2][gamma][M][2]: count + (label count << 32), confidence sum
    extern __shared__ __align__(16) unsigned long long hs[];
    __shared__ float wsum[kStatsWarps][2 * kMaxGamma * 4];  // float pairs
    __shared__ float T_s[kMaxGamma];
    __shared__ bool last_s;
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = a.gamma, M = a.M;
    const int HS = 2 * G * M * 2;
    for (int i = threadIdx.x; i < HS; i += kStatsThreads) hs[i] = 0;
    for (int i = threadIdx.x; i < kStatsWarps * 2 * kMaxGamma * 4; i += kStatsThreads)
        (&wsum[0][0])[i] = 0.0f;
    pdl_wait();
    if (threadIdx.x < G) T_s[threadIdx.x] = a.T[threadIdx.x];
    __syncthreads();
    bool bad_in = blockIdx.x == 0 && threadIdx.x < G && !(T_s[threadIdx.x] > 0.0f);
    bool bad_len = false;
    const long long per_pass = (long long)kStatsThreads * kStatsR;
    for (long long base = (long long)blockIdx.x * per_pass; base < a.N;
         base += (long long)gridDim.x * per_pass) {
        // this thread's samples, kept in registers over the depths
        int cor[kStatsR], tst[kStatsR];
        float S[kStatsR];
#pragma unroll
        for (int r = 0; r < kStatsR; ++r) {
            const long long n = base + r * kStatsThreads + threadIdx.x;
            cor[r] = tst[r] = 0;  // tested 0: never observed
            S[r] = 1.0f;
            if (n < a.N) bad_len |= sample_lens(a.correct[n], a.tested[n], G, cor[r], tst[r]);
        }
        for (int k = 0; k < G; ++k) {
            float acc[8];  // per flavour: Brier pair, log-loss pair
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
            bool any = false;
#pragma unroll
            for (int r = 0; r < kStatsR; ++r) {
                const long long n = base + r * kStatsThreads + threadIdx.x;
                const float zk = n < a.N ? a.z[n * G + k] : 0.0f;
                if (zk != zk) bad_in = true;
                if (k >= tst[r]) continue;  // the window did not reach depth k
                const float c = sts_confidence(zk, T_s[k]);
                S[r] = (k == 0) ? c : __fmul_rn(S[r], c);
                const bool y = k < cor[r];
                if (S[r] == S[r]) stats_add(hs, acc, 0, k, S[r], y, G, M, a.status);
                if (cor[r] >= k && c == c) stats_add(hs, acc + 4, 1, k, c, y, G, M, a.status);
                any = true;
            }
            if (__any_sync(kFullMask, any)) {
#pragma unroll
                for (int i = 0; i < 8; i += 2) warp_sum_pair(acc[i], acc[i + 1]);
                if (lane == 0) {
                    float *w = wsum[warp];
                    add_pair(w + k * 4, acc[0], acc[1]);
                    add_pair(w + k * 4 + 2, acc[2], acc[3]);
                    add_pair(w + (kMaxGamma + k) * 4, acc[4], acc[5]);
                    add_pair(w + (kMaxGamma + k) * 4 + 2, acc[6], acc[7]);
                }
            }
        }
    }
    if (__syncthreads_or(bad_in) && threadIdx.x == 0) flag(a.status, DSPARK_STATUS_BAD_INPUT);
    if (__syncthreads_or(bad_len) && threadIdx.x == 0) flag(a.status, DSPARK_STATUS_BAD_LEN);
    // to the global [2][gamma][M][3] histogram: count, label count, confidence sum
    for (int i = threadIdx.x; i < 2 * G * M; i += kStatsThreads) {
        const unsigned long long cl = hs[2 * i], conf = hs[2 * i + 1];
        if (cl) {
            atomicAdd(a.hist_ws + 3 * i, cl & 0xffffffffull);
            atomicAdd(a.hist_ws + 3 * i + 1, cl >> 32);
            atomicAdd(a.hist_ws + 3 * i + 2, conf);
        }
    }
    // this CTA's Brier / log-loss sums, warps in order; slot (f*G + k)*2 + s
    for (int i = threadIdx.x; i < 4 * G; i += kStatsThreads) {
        const int f = i / (2 * G), k = (i >> 1) % G, s = i & 1;
        double v = 0.0;
        for (int w = 0; w < kStatsWarps; ++w) {
            const float *pr = &wsum[w][(f * kMaxGamma + k) * 4 + 2 * s];
            v += (double)pr[0] + (double)pr[1];
        }
        a.part_ws[(size_t)blockIdx.x * (4 * G) + i] = v;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last_s = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last_s) return;
    __threadfence();
    for (int fk = threadIdx.x; fk < 2 * G; fk += kStatsThreads) {
        unsigned long long n;
        const unsigned long long E = ece_numerator(a.hist_ws + (size_t)fk * M * 3, M, &n);
        double br = 0.0, ll = 0.0;
        for (unsigned c = 0; c < gridDim.x; ++c) {
            br += __ldcg(a.part_ws + (size_t)c * (4 * G) + 2 * fk);
            ll += __ldcg(a.part_ws + (size_t)c * (4 * G) + 2 * fk + 1);
        }
        double *m = a.metrics + (size_t)fk * 4;
        m[0] = (double)n;
        m[1] = ece_of(E, n);
        m[2] = n ? __ddiv_rn(br, (double)n) : 0.0;
        m[3] = n ? __ddiv_rn(ll, (double)n) : 0.0;
    }
    __syncthreads();
    const int HN = 2 * G * M * 3;
    for (int i = threadIdx.x; i < HN; i += kStatsThreads) {
        const unsigned long long v = __ldcg(a.hist_ws + i);
        if (a.hist_out) a.hist_out[i] = v;
        a.hist_ws[i] = 0;
    }
    if (threadIdx.x == 0) *a.ticket = 0;
}

// ---------------------------------------------------------------------- fit

struct FitState {
    unsigned int ticket;
    int32_t pad;
    int32_t choice[kMaxGamma + 1];  // the grid index chosen per depth (-1: none)
};

struct FitArgs {
    const float *z;
    const int32_t *correct, *tested;
    long long N;
    int gamma, k, J, M, P;     // P = sample phases per tile (kFitThreads / J)
    float *S;                  // [N] survival of the depths already fitted
    unsigned long long *hist;  // [J][M][3], all zero between depths
    FitState *st;
    float *T_out;
    int32_t *choice_out;
    double *ece_curve;  // nullable [gamma][J]
    long long *n_obs;   // nullable [gamma]
    int32_t *status;
    float grid[kMaxTemps];
};

__global__ void __launch_bounds__(kFitThreads) sts_fit_kernel(const __grid_constant__ FitArgs a) {
    extern __shared__ __align__(16) unsigned char fsm[];
    __shared__ float z_s[kFitTile], sp_s[kFitTile];
    __shared__ unsigned char y_s[kFitTile];  // labels of the compacted samples
    __shared__ int scan_tmp[33];
    __shared__ unsigned long long e_s[kMaxTemps];
    __shared__ bool last_s;
    const int M = a.M, J = a.J, P = a.P, k = a.k, G = a.gamma;
    // private bins, [bin][thread]: confidence sums, and count + (label
    // count << 32) in one word
    unsigned long long *bconf = reinterpret_cast<unsigned long long *>(fsm);
    unsigned long long *bcl = bconf + (size_t)M * kFitThreads;
    pdl_trigger();
    const int tid = threadIdx.x;
    for (int i = tid; i < M * kFitThreads; i += kFitThreads) {
        bconf[i] = 0;
        bcl[i] = 0;
    }
    const int j = tid % J, ph = tid / J;
    const bool worker = ph < P;
    const float Tj = a.grid[worker ? j : 0];
    pdl_wait();  // the previous depth chose its temperature and updated S
    float Tprev = 1.0f;
    if (k > 0) {
        const int cp = __ldcg(&a.st->choice[k - 1]);
        Tprev = cp >= 0 ? a.grid[cp] : 1.0f;
    }
    bool bad_in = false, bad_len = false;
    const long long ntiles = (a.N + kFitTile - 1) / kFitTile;
    for (long long t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const long long n = t * kFitTile + tid;
        unsigned char fl = 0;
        float zk = 0.0f, sp = 1.0f;
        if (n < a.N) {
            int cor, tst;
            const bool bl = sample_lens(a.correct[n], a.tested[n], G, cor, tst);
            if (k == 0) bad_len |= bl;
            zk = a.z[n * G + k];
            if (zk != zk) bad_in = true;
            if (k < tst) {
                // S_{k-1} under the chosen temperatures; only samples whose
                // window reaches k need it, now or at any later depth
                if (k > 0) {
                    const float cprev = sts_confidence(a.z[n * G + k - 1], Tprev);
                    sp = (k == 1) ? cprev : __fmul_rn(a.S[n], cprev);
                    a.S[n] = sp;
                }
                if (zk == zk && sp == sp) fl = 1;
            }
            if (k < cor) fl |= 2;
        }
        // the samples that count, packed to the front of the tile
        int n_in;
        const int pos = block_exclusive_scan<int>(fl & 1, scan_tmp, &n_in);
        if ((fl & 1) && in_bounds(pos, kFitTile, a.status)) {
            z_s[pos] = zk;
            sp_s[pos] = sp;
            y_s[pos] = fl >> 1;
        }
        __syncthreads();
        if (worker) {
            // bins private to this thread; four samples at a time so that
            // their dependent float-pair chains interleave
            auto add = [&](int s, float c) {
                const float p = (k == 0) ? c : __fmul_rn(sp_s[s], c);
                const unsigned long long q = conf_q(p);
                const int bin = conf_bin(q, M);
                if (!in_bounds(bin, M, a.status)) return;
                const int idx = bin * kFitThreads + tid;
                bcl[idx] += 1ull + ((unsigned long long)y_s[s] << 32);
                bconf[idx] += q;
            };
            int s = ph;
            for (; s + 3 * P < n_in; s += 4 * P) {
                float t[4], c[4];
                bool ok[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) t[u] = __fdiv_rn(z_s[s + u * P], Tj);
#pragma unroll
                for (int u = 0; u < 4; ++u) ok[u] = sigmoid_f32(t[u], c[u]);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (!ok[u]) c[u] = sigmoid_f64(t[u]);
#pragma unroll
                for (int u = 0; u < 4; ++u) add(s + u * P, c[u]);
            }
            for (; s < n_in; s += P) add(s, sts_confidence(z_s[s], Tj));
        }
        __syncthreads();
    }
    if (__syncthreads_or(bad_in) && tid == 0) flag(a.status, DSPARK_STATUS_BAD_INPUT);
    if (__syncthreads_or(bad_len) && tid == 0) flag(a.status, DSPARK_STATUS_BAD_LEN);
    // fold the phases of each candidate and publish
    for (int pair = tid; pair < J * M; pair += kFitThreads) {
        const int jj = pair % J, b = pair / J;
        unsigned long long cnt = 0, lab = 0, conf = 0;
        for (int q = 0; q < P; ++q) {
            const int idx = b * kFitThreads + q * J + jj;
            cnt += bcl[idx] & 0xffffffffull;
            lab += bcl[idx] >> 32;
            conf += bconf[idx];
        }
        if (cnt) {
            unsigned long long *h = a.hist + ((size_t)jj * M + b) * 3;
            atomicAdd(h, cnt);
            atomicAdd(h + 1, lab);
            atomicAdd(h + 2, conf);
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) last_s = atomicAdd(&a.st->ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last_s) return;
    __threadfence();
    unsigned long long n = 0;
    if (tid < J) {
        const unsigned long long E = ece_numerator(a.hist + (size_t)tid * M * 3, M, &n);
        e_s[tid] = E;
        if (a.ece_curve) a.ece_curve[(size_t)k * J + tid] = ece_of(E, n);
    }
    __syncthreads();
    if (tid == 0) {  // n: samples counted at this depth (the same for every candidate)
        int best = -1;
        unsigned long long bestE = 0;
        if (n > 0)
            for (int jj = 0; jj < J; ++jj)
                if (best < 0 || e_s[jj] < bestE) {
                    best = jj;
                    bestE = e_s[jj];
                }
        a.st->choice[k] = best;
        a.choice_out[k] = best;
        a.T_out[k] = best >= 0 ? a.grid[best] : 1.0f;
        if (a.n_obs) a.n_obs[k] = (long long)n;
        a.st->ticket = 0;
    }
    for (int i = tid; i < J * M * 3; i += kFitThreads) a.hist[i] = 0;
}

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

size_t stats_hist_bytes(int gamma, int M) { return align256((size_t)2 * gamma * M * 3 * 8); }

size_t fit_hist_bytes(int J, int M) { return align256((size_t)J * M * 3 * 8); }

}  // namespace dspark

using namespace dspark;

extern "C" int dspark_sts_record(const float *conf_logits, const int32_t *num_correct,
                                 const int32_t *verify_lens, const uint8_t *select, int32_t B,
                                 int32_t gamma, float *rec_logits, int32_t *rec_correct,
                                 int32_t *rec_tested, int64_t capacity, uint64_t *cursor,
                                 uint8_t *prefix_mask, int32_t *status, void *stream) {
    if (!conf_logits || !num_correct || !rec_logits || !rec_correct || !rec_tested || !cursor ||
        !status)
        return DSPARK_ERR_INVALID_ARG;
    if (B < 1 || gamma < 1 || gamma > kMaxGamma || capacity < 1) return DSPARK_ERR_INVALID_ARG;
    RecordArgs a;
    a.z = conf_logits;
    a.correct = num_correct;
    a.verify_lens = verify_lens;
    a.select = select;
    a.B = B;
    a.gamma = gamma;
    a.rec_z = rec_logits;
    a.rec_correct = rec_correct;
    a.rec_tested = rec_tested;
    a.capacity = capacity;
    a.cursor = reinterpret_cast<unsigned long long *>(cursor);
    a.mask = prefix_mask;
    a.status = status;
    const cudaError_t e = launch_pdl(sts_record_kernel, dim3(1), dim3(kRecThreads), 0,
                                     static_cast<cudaStream_t>(stream), a);
    return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

extern "C" int dspark_sts_confidence(const float *conf_logits, const float *sts_temps,
                                    int64_t n_rows, int32_t gamma, float *conf_out,
                                    int32_t *status, void *stream) {
    if (!sts_temps || !status) return DSPARK_ERR_INVALID_ARG;
    if (n_rows < 0 || gamma < 1) return DSPARK_ERR_INVALID_ARG;
    if (n_rows > 0 && (!conf_logits || !conf_out)) return DSPARK_ERR_INVALID_ARG;
    const long long n = (long long)n_rows * gamma;
    if (n == 0) return DSPARK_OK;
    long long g = (n + 255) / 256;
    const long long cap = (long long)sm_count() * 8;
    g = g < cap ? g : cap;
    const cudaError_t e = launch_pdl(sts_confidence_kernel, dim3((unsigned)g), dim3(256), 0,
                                     static_cast<cudaStream_t>(stream), conf_logits, sts_temps, n,
                                     (int)gamma, conf_out, status);
    return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

extern "C" size_t dspark_calibration_workspace_bytes(int32_t gamma, int32_t n_bins) {
    if (gamma < 1 || gamma > kMaxGamma || n_bins < 1 || n_bins > kMaxBins) return 0;
    return stats_hist_bytes(gamma, n_bins) + 256 +
           align256((size_t)kStatsMaxCtas * 4 * gamma * sizeof(double));
}

extern "C" int dspark_calibration_stats(const float *rec_logits, const int32_t *rec_correct,
                                        const int32_t *rec_tested, int64_t N, int32_t gamma,
                                        const float *sts_temps, int32_t n_bins, uint64_t *hist,
                                        double *metrics, void *workspace,
                                        size_t workspace_bytes, int32_t *status, void *stream) {
    if (!sts_temps || !metrics || !status) return DSPARK_ERR_INVALID_ARG;
    if (N > 0 && (!rec_logits || !rec_correct || !rec_tested)) return DSPARK_ERR_INVALID_ARG;
    if (N < 0 || N > kMaxSamples || gamma < 1 || gamma > kMaxGamma || n_bins < 1 ||
        n_bins > kMaxBins)
        return DSPARK_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < dspark_calibration_workspace_bytes(gamma, n_bins) ||
        !aligned(workspace, 256))
        return DSPARK_ERR_WORKSPACE;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    StatsArgs a;
    a.z = rec_logits;
    a.correct = rec_correct;
    a.tested = rec_tested;
    a.N = N;
    a.gamma = gamma;
    a.M = n_bins;
    a.T = sts_temps;
    a.hist_ws = reinterpret_cast<unsigned long long *>(ws);
    a.ticket = reinterpret_cast<unsigned int *>(ws + stats_hist_bytes(gamma, n_bins));
    a.part_ws = reinterpret_cast<double *>(ws + stats_hist_bytes(gamma, n_bins) + 256);
    a.hist_out = reinterpret_cast<unsigned long long *>(hist);
    a.metrics = metrics;
    a.status = status;
    const int smem = 2 * gamma * n_bins * 2 * 8;
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(calib_stats_kernel), smem, 7);
    if (e != cudaSuccess) return DSPARK_ERR_CUDA;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, calib_stats_kernel, kStatsThreads,
                                                      (size_t)smem);
    if (e != cudaSuccess) return DSPARK_ERR_CUDA;
    const long long tiles = (N + kStatsThreads * kStatsR - 1) / (kStatsThreads * kStatsR);
    long long g = (long long)sm_count() * (occ > 0 ? occ : 1);
    g = g < tiles ? g : tiles;
    g = g < kStatsMaxCtas ? g : kStatsMaxCtas;
    g = g < 1 ? 1 : g;
    e = launch_pdl(calib_stats_kernel, dim3((unsigned)g), dim3(kStatsThreads), (size_t)smem,
                   static_cast<cudaStream_t>(stream), a);
    return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

extern "C" size_t dspark_sts_fit_workspace_bytes(int64_t N, int32_t n_temps, int32_t n_bins) {
    if (N < 0 || N > kMaxSamples || n_temps < 1 || n_temps > kMaxTemps || n_bins < 1 || n_bins > kMaxBins) return 0;
    return align256(sizeof(FitState)) + fit_hist_bytes(n_temps, n_bins) +
           align256((size_t)N * sizeof(float));
}

extern "C" int dspark_sts_fit(const float *rec_logits, const int32_t *rec_correct,
                              const int32_t *rec_tested, int64_t N, int32_t gamma,
                              const float *temp_grid, int32_t n_temps, int32_t n_bins,
                              float *sts_temps_out, int32_t *choice, double *ece_curve,
                              int64_t *n_obs, void *workspace, size_t workspace_bytes,
                              int32_t *status, void *stream) {
    if (!temp_grid || !sts_temps_out || !choice || !status) return DSPARK_ERR_INVALID_ARG;
    if (N > 0 && (!rec_logits || !rec_correct || !rec_tested)) return DSPARK_ERR_INVALID_ARG;
    if (N < 0 || N > kMaxSamples || gamma < 1 || gamma > kMaxGamma || n_temps < 1 ||
        n_temps > kMaxTemps || n_bins < 1 || n_bins > kMaxBins)
        return DSPARK_ERR_INVALID_ARG;
    for (int i = 0; i < n_temps; ++i)  // the grid is host memory
        if (!(temp_grid[i] > 0.0f) || !(temp_grid[i] < INFINITY)) return DSPARK_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < dspark_sts_fit_workspace_bytes(N, n_temps, n_bins) ||
        !aligned(workspace, 256))
        return DSPARK_ERR_WORKSPACE;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    FitArgs a;
    a.z = rec_logits;
    a.correct = rec_correct;
    a.tested = rec_tested;
    a.N = N;
    a.gamma = gamma;
    a.J = n_temps;
    a.M = n_bins;
    a.P = kFitThreads / n_temps;
    a.st = reinterpret_cast<FitState *>(ws);
    a.hist = reinterpret_cast<unsigned long long *>(ws + align256(sizeof(FitState)));
    a.S = reinterpret_cast<float *>(ws + align256(sizeof(FitState)) +
                                    fit_hist_bytes(n_temps, n_bins));
    a.T_out = sts_temps_out;
    a.choice_out = choice;
    a.ece_curve = ece_curve;
    a.n_obs = reinterpret_cast<long long *>(n_obs);
    a.status = status;
    for (int i = 0; i < kMaxTemps; ++i) a.grid[i] = i < n_temps ? temp_grid[i] : 1.0f;
    const int smem = n_bins * kFitThreads * 16;
    cudaError_t e = ensure_smem(reinterpret_cast<const void *>(sts_fit_kernel), smem, 8);
    if (e != cudaSuccess) return DSPARK_ERR_CUDA;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sts_fit_kernel, kFitThreads,
                                                      (size_t)smem);
    if (e != cudaSuccess) return DSPARK_ERR_CUDA;
    const long long tiles = (N + kFitTile - 1) / kFitTile;
    long long g = (long long)sm_count() * (occ > 0 ? occ : 1);
    g = g < tiles ? g : tiles;
    g = g < 1 ? 1 : g;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int k = 0; k < gamma; ++k) {
        a.k = k;
        e = launch_pdl(sts_fit_kernel, dim3((unsigned)g), dim3(kFitThreads), (size_t)smem, s, a);
        if (e != cudaSuccess) return DSPARK_ERR_CUDA;
    }
    return DSPARK_OK;
}
