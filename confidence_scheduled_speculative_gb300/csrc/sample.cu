// sample.cu -- speculative sampling accept (compact mode) on sm_103a.
//
// Pages (by title and section):
//   [ROUND] "DeepSeek-V4 DSpark一轮 Draft、Verify、Accept 与 Commit", §五
//           (AcceptSampling: chain speculative sampling over the draft's
//           proposal probabilities -- the corrected ones that produced the
//           drafts -- and the target probabilities, giving correct_len and
//           the bonus; then FinalizeAcceptLens / BuildOutTokens as in the
//           greedy path)
//   [AVS]   "DSpark 自适应 Verify 怎样分配候选预算", §一 (a draft drawn from q
//           is accepted with probability min(1, p/q); mean acceptance
//           sum min(p, q) = 1 - TV)
//
// The rule, as the pages' classic form: draft j of request r (token x) is
// accepted iff u_j * q_j(x) < p_j(x), p_j = softmax of packed target row
// cu[r] + j, q_j = softmax of draft row r*gamma + j; at the first rejection
// the bonus is the inverse-CDF draw (uniform u_bonus[r]) from the residual
// max(0, p_j - q_j), normalised; when every draft is accepted, from the
// last row's p.  An empty residual (p == q; in practice a total mass below
// 2^-20, the precision of the softmax sums) draws from p.
//
// Two kernels:
//   softmax_norm_kernel  HBM-bound: for every packed target row and every
//     draft row some test reads (j < len - 1), the row max m and S = sum
//     exp(z - m).  The target rows, then the draft rows in (request, depth)
//     order, form one list of "virtual rows", flattened into 16-byte chunks
//     and split into one equal contiguous range per CTA of a persistent grid
//     (as the greedy argmax does); each warp leaves a partial (m, S) of
//     each (CTA, row) piece, so no block barrier separates one row from the
//     next; at its end the CTA folds each piece's warp partials into one at
//     slot CTA + row.  Per thread an online max / sum of exps (hardware
//     ex2), float-pair sums per warp and piece; the accept kernel combines
//     a row's partials in fp64.
//   sampling_accept_kernel  one thread-block cluster of S CTAs per request
//     (S up to 8, as many as fill the GPU in one wave).  Every CTA combines
//     the partials of the request's rows and runs the acceptance tests (warp
//     0, one lane per draft), so each knows the bonus row; the residual (or
//     p) of that row is then summed in rounds of 512 tokens (16 per lane),
//     each warp of the cluster owning one contiguous range of rounds.  The
//     CTAs swap their slice totals through distributed shared memory; the
//     CTA whose slice holds u * W finds the round and the token in it and
//     writes the request's results.
//   Every weight is quantized per lane and round to a multiple of 2^-40 and
//   summed as an integer, so the draw does not depend on how the rounds are
//   split among warps and CTAs.
// Sums of exps are fp32 per thread and fp64 beyond, so p and q agree with
// an fp64 index-order evaluation to about 1e-6 relative: decisions can
// differ from such an evaluation only when u * q and p (or u * W and a
// cumulative weight) are that close.

#include "dspark_common.cuh"
#include "logits.cuh"

namespace dspark {

constexpr int kNormThreads = 256;
constexpr int kNormCtasPerSm = 4;
constexpr int kNormUnroll = 4;
constexpr int kSampThreads = 256;
constexpr int kSampWarps = kSampThreads / 32;
constexpr int kSampMaxB = 4096;   // cu_seqlens staged in shared memory by every CTA
constexpr int kSampMaxCtas = 4096;
constexpr int kSampMaxV = 1 << 20;
constexpr int kTokLane = 16;                  // tokens of one lane in a round of the bonus draw
constexpr int kRound = 32 * kTokLane;         // tokens of one warp-round
constexpr int kMaxRounds = kSampMaxV / kRound / kSampWarps;  // rounds per warp (one CTA per request)
constexpr int kSampMaxCluster = 8;            // CTAs sharing one request's bonus draw
constexpr int kSampCtasPerSm = 4;             // resident accept CTAs per SM (launch bound)
constexpr int kBonusChunks = 4;               // 16-byte target chunks in flight per lane

constexpr int kNormWarps = kNormThreads / 32;

// One warp's share of one (CTA, row) piece.
struct __align__(16) NormPartial {
    float m;       // largest logit the warp read (-inf: none)
    float sh, sl;  // sum of exp(z - m) over them, as a float pair sh + sl
    float pad;
};

struct SampArgs {
    const void *tgt;
    long long ld_t;  // elements
    const void *dft;
    long long ld_d;
    const float *draft_lse;  // [B*gamma] the draft rows' log-sum-exp, or null (normalised here)
    int V, B, gamma, max_rows;
    const int32_t *cu, *draft, *prefix;
    const float *u_acc, *u_bonus;
    int32_t *num_acc, *bonus, *commit, *new_seq, *out, *status;
    NormPartial *part;    // [kSampMaxCtas + max_rows + B*gamma + 1]: one per (CTA, row) piece
    NormPartial *part_w;  // [(kSampMaxCtas + max_rows + B*gamma + 1) * kNormWarps]: per warp
    int32_t *dcu;       // [B+1] first virtual draft row of each request (written by CTA 0)
    int grid;           // normalizer grid size
    int split;          // CTAs (one thread-block cluster) per request in the accept kernel
};

// Partial slots: one per (CTA, virtual row) piece, CTA c < kSampMaxCtas and
// virtual row v < max_rows + B*gamma.
__device__ __forceinline__ long long samp_slots(const SampArgs &a) {
    return (long long)kSampMaxCtas + a.max_rows + (long long)a.B * a.gamma + 1;
}

__device__ __forceinline__ int samp_rows(const SampArgs &a) {
    const int r = a.cu[a.B];
    return r < 0 ? 0 : (r > a.max_rows ? a.max_rows : r);
}

// A request reads packed rows [lo, hi) with 1 <= hi - lo <= gamma + 1.
__device__ __forceinline__ bool samp_valid(int lo, int hi, int rows, int gamma) {
    return lo >= 0 && hi <= rows && hi - lo >= 1 && hi - lo <= gamma + 1;
}

constexpr float kLog2e = 1.4426950408889634f;

// A residual max(0, p - q) of total mass below 2^-20 -- under the precision
// of the softmax sums -- is empty: the bonus is drawn from p.  (2^20 units
// of 2^-40.)
constexpr unsigned long long kEmptyResidual = 1ull << 20;

// 2^x by the hardware approximation (relative error about 2^-22).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Online (max, sum of exps) of one value; NaN counts as -inf.
__device__ __forceinline__ void norm_take(float z, float &m, float &s) {
    if (z > m) {
        s = s * __expf(m - z) + 1.0f;
        m = z;
    } else if (z > -INFINITY) {
        s += __expf(z - m);
    }
}

// A chunk holding a NaN: value by value, NaN skipped (rare path).
template <typename T>
__device__ __noinline__ void norm_chunk_nan(uint4 v, float &m, float &s) {
#pragma unroll
    for (int e = 0; e < Elem<T>::kPerChunk; ++e) norm_take(Elem<T>::at(v, e), m, s);
}

// One 16-byte chunk into the thread's running (m, s): the chunk max (NaN-
// propagating, packed for bf16), one rescale, then exp(z - m) =
// 2^(z*log2e - m*log2e) with one FMA and one ex2 per value.
template <typename T>
__device__ __forceinline__ void norm_chunk(const uint4 &v, float &m, float &s, bool &nan) {
    const float cm = Elem<T>::chunk_max(v);
    if (cm != cm) {
        nan = true;
        norm_chunk_nan<T>(v, m, s);
        return;
    }
    if (cm > m) {
        s *= ex2((m - cm) * kLog2e);
        m = cm;
    }
    if (m > -INFINITY) {
        const float ml = m * kLog2e;
#pragma unroll
        for (int e = 0; e < Elem<T>::kPerChunk; ++e) s += ex2(fmaf(Elem<T>::at(v, e), kLog2e, -ml));
    }
}

// Warp-wide combine of the lanes' (m, s); lane 0 writes the warp's partial
// of the piece.  The sums travel as float pairs (hi + lo, error-free
// additions): no fp64 instruction in the streaming kernel (GB300's fp64
// unit is small), no block barrier between pieces.
__device__ __forceinline__ void norm_warp(float m, float s, NormPartial *dst, bool store) {
    float M = m;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, d));
    float th = (m > -INFINITY) ? s * ex2((m - M) * kLog2e) : 0.0f, tl = 0.0f;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const float oh = __shfl_xor_sync(kFullMask, th, d), ol = __shfl_xor_sync(kFullMask, tl, d);
        float h, e;
        two_sum(th, oh, h, e);
        e = __fadd_rn(e, __fadd_rn(tl, ol));
        fast_two_sum(h, e, th, tl);
    }
    if ((threadIdx.x & 31) == 0 && store) *dst = NormPartial{M, th, tl, 0.0f};
}

// Warp-wide fold of one partial per lane (lanes past the piece's warps hold
// m = -inf, s = 0); lane 0 writes the result.
__device__ __forceinline__ void norm_fold(const NormPartial &p, NormPartial *dst, bool store) {
    float M = p.m;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, d));
    float th = 0.0f, tl = 0.0f;
    if (p.m > -INFINITY) {
        const float e = ex2((p.m - M) * kLog2e);  // 1 for the largest
        th = __fmul_rn(p.sh, e);
        tl = fmaf(p.sh, e, -th);  // the product's rounding error
        tl = fmaf(p.sl, e, tl);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const float oh = __shfl_xor_sync(kFullMask, th, d), ol = __shfl_xor_sync(kFullMask, tl, d);
        float h, e;
        two_sum(th, oh, h, e);
        e = __fadd_rn(e, __fadd_rn(tl, ol));
        fast_two_sum(h, e, th, tl);
    }
    if ((threadIdx.x & 31) == 0 && store) *dst = NormPartial{M, th, tl, 0.0f};
}

// Virtual row v: a packed target row (v < rows) or the draft row of the
// (v - rows)-th draft a test reads, in (request, depth) order; dcu[r] is the
// first such draft of request r.  Returns the element offset of the row in
// its buffer and whether it is a draft row.
__device__ __forceinline__ long long virtual_row(const SampArgs &a, const int32_t *dcu, int rows,
                                                 int v, bool &is_draft) {
    if (v < rows) {
        is_draft = false;
        return (long long)v * a.ld_t;
    }
    is_draft = true;
    const int d = v - rows;
    int lo = 0, hi = a.B - 1;  // the last request whose first draft row is <= d
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (dcu[mid] <= d) lo = mid;
        else hi = mid - 1;
    }
    const int j = d - dcu[lo];  // < its number of tested drafts <= gamma
    return ((long long)lo * a.gamma + j) * a.ld_d;
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kNormThreads, kNormCtasPerSm) softmax_norm_kernel(SampArgs a) {
    extern __shared__ int32_t dcu[];  // [B+1]
    __shared__ int scan32[40];
    constexpr int EPC = VEC ? Elem<T>::kPerChunk : 1;
    const int tid = threadIdx.x;
    const int B = a.B, G = a.gamma;

    pdl_wait();  // cu_seqlens and the logits come from the kernels before
    // the accept kernel launches once every CTA is past its wait, so it may
    // read cu_seqlens and the logits in its prologue
    pdl_trigger();
    const int rows = samp_rows(a);
    if (blockIdx.x == 0 && tid == 0 && a.cu[B] > a.max_rows) flag(a.status, DSPARK_STATUS_CAPACITY);
    // the tested drafts of each valid request, scanned: dcu
    {
        const int per = (B + kNormThreads - 1) / kNormThreads;
        const int q0 = min(tid * per, B), q1 = min(q0 + per, B);
        int mine = 0;
        for (int q = q0; q < q1; ++q) {
            const int lo = a.cu[q], hi = a.cu[q + 1];
            mine += samp_valid(lo, hi, rows, G) ? hi - lo - 1 : 0;
        }
        int total;
        int off = block_exclusive_scan<int>(mine, scan32, &total);
        for (int q = q0; q < q1; ++q) {
            dcu[q] = off;
            const int lo = a.cu[q], hi = a.cu[q + 1];
            off += samp_valid(lo, hi, rows, G) ? hi - lo - 1 : 0;
        }
        if (tid == 0) dcu[B] = total;
        __syncthreads();
        if (blockIdx.x == 0)
            for (int q = tid; q <= B; q += kNormThreads) a.dcu[q] = dcu[q];
    }
    // the tested draft rows too, unless the caller gave their normalizers
    const int VR = rows + (a.draft_lse ? 0 : dcu[B]);
    const int cpr = (a.V + EPC - 1) / EPC;  // chunks per row, the last maybe partial
    const int full = a.V / EPC;
    const long long W = (long long)VR * cpr;
    const long long per = div_nonneg(W + a.grid - 1, a.grid);
    const long long q0 = (long long)blockIdx.x * per;
    const long long q1 = min(q0 + per, W);
    bool nan = false;
    for (long long q = q0; q < q1;) {
        const int v = (int)div_nonneg(q, cpr);
        const int c0 = (int)(q - (long long)v * cpr);
        const long long seg_end = min(q1, (long long)(v + 1) * cpr);
        const int c1 = c0 + (int)(seg_end - q);
        bool is_draft;
        const long long row_off = virtual_row(a, dcu, rows, v, is_draft);  // every thread
        const T *row = reinterpret_cast<const T *>(is_draft ? a.dft : a.tgt) + row_off;
        float m = -INFINITY, s = 0.0f;
        if (VEC) {
            const uint4 *row4 = reinterpret_cast<const uint4 *>(row);
            const int cf = min(c1, full);
            int c = c0 + tid;
            for (; c + (kNormUnroll - 1) * kNormThreads < cf; c += kNormUnroll * kNormThreads) {
                uint4 x[kNormUnroll];
#pragma unroll
                for (int u = 0; u < kNormUnroll; ++u) x[u] = ld_stream16(row4 + c + u * kNormThreads);
#pragma unroll
                for (int u = 0; u < kNormUnroll; ++u) norm_chunk<T>(x[u], m, s, nan);
            }
            for (; c < cf; c += kNormThreads) norm_chunk<T>(ld_stream16(row4 + c), m, s, nan);
            // the row's partial last chunk, element by element
            if (c1 > full && tid == 0)
                for (int e = full * EPC; e < a.V; ++e) {
                    const float z = Elem<T>::load(row + e);
                    nan |= z != z;
                    norm_take(z, m, s);
                }
        } else {
            for (int e = c0 + tid; e < c1; e += kNormThreads) {
                const float z = Elem<T>::load(row + e);
                nan |= z != z;
                norm_take(z, m, s);
            }
        }
        const bool in = in_bounds(blockIdx.x + v, samp_slots(a), a.status);
        norm_warp(m, s, a.part_w + (size_t)(blockIdx.x + v) * kNormWarps + (tid >> 5), in);
        q = seg_end;
    }
    if (__syncthreads_or(nan) && tid == 0) flag(a.status, DSPARK_STATUS_NAN_LOGIT);
    // the warps' partials of each piece of this CTA, folded into one (warp
    // j % kNormWarps folds piece j; lane w reads warp w's partial)
    if (q0 < q1) {
        const int v0 = (int)div_nonneg(q0, cpr), v1 = (int)div_nonneg(q1 - 1, cpr);
        const int lane = tid & 31;
        for (int v = v0 + (tid >> 5); v <= v1; v += kNormWarps) {
            NormPartial p = NormPartial{-INFINITY, 0.0f, 0.0f, 0.0f};
            const bool in = in_bounds(blockIdx.x + v, samp_slots(a), a.status);
            if (lane < kNormWarps && in) p = a.part_w[(size_t)(blockIdx.x + v) * kNormWarps + lane];
            norm_fold(p, a.part + blockIdx.x + v, in);
        }
    }
}

// ---------------------------------------------------- acceptance and bonus

// (M, S) of virtual row v from the partials of the CTAs that covered it.
__device__ __forceinline__ void row_stats(const SampArgs &a, long long cpr, long long per,
                                          int v, float &M, double &S) {
    const NormPartial *part = a.part;
    const long long q_first = (long long)v * cpr;
    const int c_lo = (int)div_nonneg(q_first, per), c_hi = (int)div_nonneg(q_first + cpr - 1, per);
    M = -INFINITY;
    S = 0.0;
    if (!in_bounds(c_hi + v, samp_slots(a), a.status)) return;
    for (int c = c_lo; c <= c_hi; ++c) M = fmaxf(M, part[c + v].m);
    if (M > -INFINITY)
        for (int c = c_lo; c <= c_hi; ++c) {
            const NormPartial p = part[c + v];
            if (p.m > -INFINITY) S += ((double)p.sh + (double)p.sl) * (double)__expf(p.m - M);
        }
}

// Weights of the bonus draw are summed exactly as integers in units of 2^-40:
// q = w * 2^40 rounded to the nearest integer, ties to even, from the bits of
// the (exact) float product -- the value a round-to-nearest conversion
// gives, without the conversion instruction (it runs on the fp64 unit).
__device__ __forceinline__ unsigned long long quantize(float w) {
    if (!(w > 0.0f)) return 0ull;
    const unsigned bits = __float_as_uint(w * 1099511627776.0f);
    const int e = (int)(bits >> 23) - 127;
    const unsigned long long m = (unsigned long long)((bits & 0x7fffffu) | 0x800000u);
    if (e >= 64) return ~0ull;         // saturates, as the conversion does
    if (e >= 23) return m << (e - 23);
    if (e < -1) return 0ull;           // below 1/2
    const int sh = 23 - e;             // 1..24
    const unsigned long long q = m >> sh, rem = m & ((1ull << sh) - 1), half = 1ull << (sh - 1);
    return q + ((rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull);
}

struct BonusRow {
    const void *t;  // target row
    const void *d;  // draft row (residual) or null (p)
    float mt, md;   // row maxima, times log2(e)
    float inv_st, inv_sd;
};

// Weight of one token of the bonus draw from its target (and draft) logit;
// a NaN logit weighs 0.
__device__ __forceinline__ float weight_of(const BonusRow &b, float zt, float zd) {
    float w = (zt == zt) ? __fmul_rn(ex2(fmaf(zt, kLog2e, -b.mt)), b.inv_st) : 0.0f;
    if (b.d) {
        const float q = (zd == zd) ? __fmul_rn(ex2(fmaf(zd, kLog2e, -b.md)), b.inv_sd) : 0.0f;
        w = fmaxf(__fsub_rn(w, q), 0.0f);
    }
    return w;
}

// The 16-byte chunks of the kTokLane tokens one lane handles in a round.
template <typename T>
struct LaneChunks {
    static constexpr int NC = kTokLane / Elem<T>::kPerChunk;
    uint4 t[NC], d[NC];
};

// Issue the loads of tokens y0 .. y0 + kTokLane - 1 when the rows are
// aligned and every token is in range; false selects the token-by-token
// path.
// HAS_D: the draft row is read too (b.d is not null).
template <typename T, bool HAS_D>
__device__ __forceinline__ bool lane_load(const BonusRow &b, int y0, int V, bool vec,
                                          LaneChunks<T> &c) {
    constexpr int NC = LaneChunks<T>::NC;
    if (!vec || y0 + kTokLane > V) return false;
    const uint4 *pt = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(b.t) + y0);
#pragma unroll
    for (int i = 0; i < NC; ++i) c.t[i] = ld_stream16(pt + i);
    if (HAS_D) {
        const uint4 *pd = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(b.d) + y0);
#pragma unroll
        for (int i = 0; i < NC; ++i) c.d[i] = ld_stream16(pd + i);
    }
    return true;
}

// The weights of the lane's tokens y0 .. y0 + kTokLane - 1 (0 past V): from
// the loaded chunks when they hold no NaN, otherwise token by token.
template <typename T>
__device__ __forceinline__ void lane_weights(const BonusRow &b, int y0, int V, bool loaded,
                                             const LaneChunks<T> &c, float (&w)[kTokLane]) {
    constexpr int E = Elem<T>::kPerChunk, NC = LaneChunks<T>::NC;
    if (loaded) {
        bool nan = false;
#pragma unroll
        for (int i = 0; i < NC; ++i) {
            const float mt = Elem<T>::chunk_max(c.t[i]);
            nan |= mt != mt;
            if (b.d) {
                const float md = Elem<T>::chunk_max(c.d[i]);
                nan |= md != md;
            }
        }
        if (!nan) {
            if (b.d) {
#pragma unroll
                for (int e = 0; e < kTokLane; ++e) {
                    const float p = __fmul_rn(ex2(fmaf(Elem<T>::at(c.t[e / E], e % E), kLog2e, -b.mt)), b.inv_st);
                    const float q = __fmul_rn(ex2(fmaf(Elem<T>::at(c.d[e / E], e % E), kLog2e, -b.md)), b.inv_sd);
                    w[e] = fmaxf(__fsub_rn(p, q), 0.0f);
                }
            } else {
#pragma unroll
                for (int e = 0; e < kTokLane; ++e)
                    w[e] = __fmul_rn(ex2(fmaf(Elem<T>::at(c.t[e / E], e % E), kLog2e, -b.mt)), b.inv_st);
            }
            return;
        }
    }
    const T *rt = reinterpret_cast<const T *>(b.t);
    const T *rd = reinterpret_cast<const T *>(b.d);
#pragma unroll
    for (int e = 0; e < kTokLane; ++e) {
        const int y = y0 + e;
        w[e] = y < V ? weight_of(b, Elem<T>::load(rt + y), rd ? Elem<T>::load(rd + y) : 0.0f) : 0.0f;
    }
}

// A lane's round total: the fp32 sum of its weights in token order (at most
// kTokLane = 16), quantized once (below 2^45 units).
__device__ __forceinline__ unsigned long long lane_total(const float (&w)[kTokLane]) {
    float acc = 0.0f;
#pragma unroll
    for (int e = 0; e < kTokLane; ++e) acc = __fadd_rn(acc, w[e]);
    return quantize(acc);
}

// The same total straight from the loaded chunks (the weights are added as
// they are made, in the same order, so the sum is lane_total's).
template <typename T, bool HAS_D>
__device__ __forceinline__ unsigned long long lane_total_of(const BonusRow &b, int y0, int V,
                                                           bool loaded, const LaneChunks<T> &c) {
    constexpr int E = Elem<T>::kPerChunk, NC = LaneChunks<T>::NC;
    if (loaded) {
        bool nan = false;
#pragma unroll
        for (int i = 0; i < NC; ++i) {
            const float mt = Elem<T>::chunk_max(c.t[i]);
            nan |= mt != mt;
            if (HAS_D) {
                const float md = Elem<T>::chunk_max(c.d[i]);
                nan |= md != md;
            }
        }
        if (!nan) {
            float acc = 0.0f;
            if (HAS_D) {
#pragma unroll
                for (int e = 0; e < kTokLane; ++e) {
                    const float p = __fmul_rn(ex2(fmaf(Elem<T>::at(c.t[e / E], e % E), kLog2e, -b.mt)), b.inv_st);
                    const float q = __fmul_rn(ex2(fmaf(Elem<T>::at(c.d[e / E], e % E), kLog2e, -b.md)), b.inv_sd);
                    acc = __fadd_rn(acc, fmaxf(__fsub_rn(p, q), 0.0f));
                }
            } else {
#pragma unroll
                for (int e = 0; e < kTokLane; ++e)
                    acc = __fadd_rn(acc, __fmul_rn(ex2(fmaf(Elem<T>::at(c.t[e / E], e % E), kLog2e, -b.mt)), b.inv_st));
            }
            return quantize(acc);
        }
    }
    float w[kTokLane];
    lane_weights<T>(b, y0, V, false, c, w);
    return lane_total(w);
}

// The warp's sum of the lanes' round totals: each total is split at bit 22
// into two parts below 2^23, so that 32 of each sum exactly in a 32-bit warp
// reduction.
__device__ __forceinline__ unsigned long long warp_round_total(unsigned long long q) {
    const unsigned lo = __reduce_add_sync(kFullMask, (unsigned)q & 0x3FFFFFu);
    const unsigned hi = __reduce_add_sync(kFullMask, (unsigned)(q >> 22));
    return ((unsigned long long)hi << 22) + lo;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(kFullMask, v, d);
    return v;
}

// ---- the thread-block cluster of one request (PTX: %cluster_ctarank,
// barrier.cluster, mapa + ld.shared::cluster)

__device__ __forceinline__ unsigned cluster_rank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster: writes before it (shared memory
// included) are visible to the whole cluster after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of a cluster barrier: every CTA arrives early, so that by
// the wait every CTA of the cluster is known to run (the condition for
// touching another CTA's shared memory).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Store a 64-bit value at the same shared-memory offset in the CTA of the
// given cluster rank.
__device__ __forceinline__ void st_cluster_u64(void *local, unsigned rank, unsigned long long v) {
    const unsigned a = (unsigned)__cvta_generic_to_shared(local);
    unsigned ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(ra), "l"(v) : "memory");
}

// This CTA's share of the bonus draw's round sums: the request's rounds
// (kRound tokens each, in token order) are cut into one contiguous range of
// rpw rounds per warp of the cluster, CTA rank q holding warps q*kSampWarps..;
// rsum[w * rpw + k] = round k of warp w (0 past the row).
template <typename T, bool HAS_D>
__device__ __forceinline__ void bonus_rounds(const BonusRow &b, int V, bool vec, int q, int rpw,
                                             unsigned long long *rsum, int32_t *status) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // rounds in flight per lane: kBonusChunks 16-byte chunks of the rows read
    constexpr int U = kBonusChunks / (LaneChunks<T>::NC * (HAS_D ? 2 : 1)) > 0
                          ? kBonusChunks / (LaneChunks<T>::NC * (HAS_D ? 2 : 1)) : 1;
    const int first = (q * kSampWarps + warp) * rpw;     // first round of this warp
    for (int k0 = 0; k0 < rpw; k0 += U) {
        LaneChunks<T> c[U];
        bool ld[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            ld[u] = k0 + u < rpw &&
                    lane_load<T, HAS_D>(b, (first + k0 + u) * kRound + lane * kTokLane, V, vec, c[u]);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (k0 + u < rpw) {  // warp-uniform
                const unsigned long long t = warp_round_total(
                    lane_total_of<T, HAS_D>(b, (first + k0 + u) * kRound + lane * kTokLane, V, ld[u], c[u]));
                if (lane == 0 && in_bounds(warp * rpw + k0 + u, kSampWarps * kMaxRounds, status))
                    rsum[warp * rpw + k0 + u] = t;
            }
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kSampThreads, kSampCtasPerSm) sampling_accept_kernel(SampArgs a, int epc, bool vec) {
    __shared__ unsigned long long rsum[kSampWarps * kMaxRounds];  // this CTA's round sums
    __shared__ BonusRow brow;
    __shared__ int s_correct;
    __shared__ unsigned long long s_tot[kSampMaxCluster];  // slice totals, written by the cluster
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = a.split;
    const int r = blockIdx.x / S;
    const int q = (int)cluster_rank();  // == blockIdx.x % S
    const int G = a.gamma, V = a.V;
    // drafts and uniforms are step inputs: fetch them before the wait
    const int dj = (warp == 0 && lane < G) ? __ldg(a.draft + (size_t)r * G + lane) : -1;
    const float uj = (warp == 0 && lane < G) ? __ldg(a.u_acc + (size_t)r * G + lane) : 1.0f;
    // cu_seqlens and the logits were written before the normalizer passed
    // its wait, which precedes this grid's launch: the tested logits are
    // fetched (from HBM) while the normalizer finishes
    const int rows = min(max(__ldcg(a.cu + a.B), 0), a.max_rows);
    const int lo = __ldcg(a.cu + r), hi = __ldcg(a.cu + r + 1), L = hi - lo;
    float zt = 0.0f, zd = 0.0f;  // the two logits lane j's test reads
    float lse = 0.0f;            // the caller's normalizer of draft row j
    if (warp == 0 && samp_valid(lo, hi, rows, G) && lane < L - 1) {
        if (dj >= 0 && dj < V) {
            zt = Elem<T>::load(reinterpret_cast<const T *>(a.tgt) + (long long)(lo + lane) * a.ld_t + dj);
            zd = Elem<T>::load(reinterpret_cast<const T *>(a.dft) + ((long long)r * G + lane) * a.ld_d + dj);
        }
        if (a.draft_lse) lse = __ldg(a.draft_lse + (size_t)r * G + lane);
    }
    pdl_trigger();
    pdl_wait();  // partials and dcu come from softmax_norm_kernel

    if (q == 0 && warp == 0 && __any_sync(kFullMask, lane < G && (dj < 0 || dj >= V)) && lane == 0)
        flag(a.status, DSPARK_STATUS_TOKEN_RANGE);
    if (!samp_valid(lo, hi, rows, G)) {  // the whole cluster leaves here
        if (q != 0) return;
        if (tid == 0) {
            flag(a.status, DSPARK_STATUS_BAD_LEN);
            a.num_acc[r] = 0;
            a.bonus[r] = -1;
            a.commit[r] = 0;
            if (a.new_seq) a.new_seq[r] = __ldg(a.prefix + r);
        }
        if (warp == 0 && lane <= G) a.out[(size_t)r * (G + 1) + lane] = lane < G ? dj : -1;
        return;
    }
    cluster_arrive_relaxed();  // waited for before the first remote store
    const int D = a.draft_lse ? 0 : a.dcu[a.B];  // the normaliser's virtual draft rows
    const long long cpr = (V + epc - 1) / epc;
    const long long W = (long long)(rows + D) * cpr;
    const long long per = div_nonneg(W + a.grid - 1, a.grid);
    const int vd0 = rows + a.dcu[r];  // virtual row of this request's first tested draft

    // (1) acceptance tests, in every CTA of the cluster (each needs the
    // bonus row).  Lane j: the statistics of target row lo + j (j < L: the
    // tests and any bonus row) and of draft row j (j < L - 1), all in
    // parallel; lane j < L - 1 tests draft j.
    if (warp == 0) {
        const bool has_t = lane < L, has_d = lane < L - 1;
        const bool tok_ok = dj >= 0 && dj < V;
        float mt = -INFINITY, md = -INFINITY;
        double st = 0.0, sd = 0.0;
        if (has_t) row_stats(a, cpr, per, lo + lane, mt, st);
        if (has_d) {
            if (!a.draft_lse) {
                row_stats(a, cpr, per, vd0 + lane, md, sd);
            } else if (isfinite(lse)) {  // q = exp(z - lse): "max" lse, sum 1
                md = lse;
                sd = 1.0;
            }
        }
        const float inv_t = st > 0.0 ? (float)(1.0 / st) : 0.0f;
        const float inv_d = sd > 0.0 ? (float)(1.0 / sd) : 0.0f;
        bool accept = true;
        if (has_d) {
            accept = false;
            if (tok_ok) {
                // p = et / st, q = ed / sd; u q < p  <=>  u ed st < et sd
                const double et = (zt == zt && st > 0.0) ? (double)__expf(zt - mt) : 0.0;
                const double ed = (zd == zd && sd > 0.0) ? (double)__expf(zd - md) : 0.0;
                accept = et > 0.0 && (ed == 0.0 || (double)uj * ed * st < et * sd);
            }
        }
        const unsigned rej = __ballot_sync(kFullMask, !accept);
        const int correct = rej ? __ffs(rej) - 1 : L - 1;
        const float bmt = __shfl_sync(kFullMask, mt, correct), bit = __shfl_sync(kFullMask, inv_t, correct);
        const float bmd = __shfl_sync(kFullMask, md, correct), bid = __shfl_sync(kFullMask, inv_d, correct);
        if (lane == 0) {
            s_correct = correct;
            const bool rejected = correct < L - 1;
            brow.t = reinterpret_cast<const T *>(a.tgt) + (long long)(lo + correct) * a.ld_t;
            brow.d = rejected ? reinterpret_cast<const T *>(a.dft) + ((long long)r * G + correct) * a.ld_d
                              : nullptr;
            brow.mt = bmt * kLog2e;
            brow.md = rejected ? bmd * kLog2e : 0.0f;
            brow.inv_st = bit;
            brow.inv_sd = rejected ? bid : 0.0f;
        }
    }
    __syncthreads();
    const int correct = s_correct;
    BonusRow b = brow;

    // (2) the bonus draw.  Round sums of the quantized weights over this
    // CTA's slice of the vocabulary; the slice totals are exchanged through
    // the cluster's shared memory, so every CTA knows the total W and the
    // weight before its slice.  An empty residual draws from p (the whole
    // cluster takes the same decision from the same W).
    const int R = (V + kRound - 1) / kRound;
    const int rpw = (R + S * kSampWarps - 1) / (S * kSampWarps);  // <= kMaxRounds
    const int nt = kSampWarps * rpw;
    unsigned long long Wq = 0ull, before = 0ull, slice = 0ull;
    for (int attempt = 0; attempt < 2; ++attempt) {
        if (attempt > 0) cluster_sync();  // every CTA has read the previous totals
        if (b.d) bonus_rounds<T, true>(b, V, vec, q, rpw, rsum, a.status);
        else bonus_rounds<T, false>(b, V, vec, q, rpw, rsum, a.status);
        if (attempt == 0) cluster_wait();  // every CTA of the cluster runs
        __syncthreads();
        if (warp == 0) {  // this slice's total into slot q of every CTA of the cluster
            unsigned long long m = 0ull;
            for (int i = lane; i < nt; i += 32) m += rsum[i];
            m = warp_sum_u64(m);
            if (lane < S) st_cluster_u64(&s_tot[q], (unsigned)lane, m);
        }
        cluster_sync();  // s_tot holds every slice total, in rank order
        Wq = 0ull;
        before = 0ull;
        for (int i = 0; i < S; ++i) {
            const unsigned long long t = s_tot[i];
            before += i < q ? t : 0ull;
            Wq += t;
        }
        slice = s_tot[q];
        if (!(Wq < kEmptyResidual && b.d != nullptr)) break;
        b.d = nullptr;  // p == q within the sums' precision: draw from p
    }
    const unsigned long long target = (unsigned long long)((double)__ldg(a.u_bonus + r) * (double)Wq);
    const bool owner = target >= before && target - before < slice;
    // the CTA whose slice holds u * W writes the request's results; when no
    // slice holds it (W = 0), rank 0 does, with no bonus token
    if (!owner && !(q == 0 && !(target < Wq))) return;

    // (3) warp 0 of the writing CTA: the round, then the token within it;
    // then FinalizeAcceptLens and BuildOutTokens
    if (warp == 0) {
        int round = -1;
        unsigned long long pre = 0ull;
        if (owner) {
            const unsigned long long lt = target - before;  // within this slice
            const int nb = (nt + 31) / 32;
            unsigned long long mine = 0ull;
            for (int i = lane * nb; i < min(nt, (lane + 1) * nb); ++i) mine += rsum[i];
            unsigned long long incl = mine;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const unsigned long long o = __shfl_up_sync(kFullMask, incl, d);
                if (lane >= d) incl += o;
            }
            const unsigned found = __ballot_sync(kFullMask, incl > lt);
            if (found) {
                const int fl = __ffs(found) - 1;
                if (lane == fl) {
                    unsigned long long c = incl - mine;
                    for (int i = lane * nb; i < min(nt, (lane + 1) * nb); ++i) {
                        if (c + rsum[i] > lt) {
                            round = i;
                            break;
                        }
                        c += rsum[i];
                    }
                    pre = c;
                }
                round = __shfl_sync(kFullMask, round, fl);
                pre = __shfl_sync(kFullMask, pre, fl);
            }
        }
        int tok = -1;
        if (round >= 0) {
            const unsigned long long lt = target - before;
            const int rw = round / rpw, k = round - rw * rpw;
            const int y0 = ((q * kSampWarps + rw) * rpw + k) * kRound + lane * kTokLane;
            LaneChunks<T> c;
            const bool ld = b.d ? lane_load<T, true>(b, y0, V, vec, c) : lane_load<T, false>(b, y0, V, vec, c);
            float w[kTokLane];
            lane_weights<T>(b, y0, V, ld, c, w);
            const unsigned long long mine = lane_total(w);
            unsigned long long incl = mine;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const unsigned long long o = __shfl_up_sync(kFullMask, incl, d);
                if (lane >= d) incl += o;
            }
            const unsigned found = __ballot_sync(kFullMask, pre + incl > lt);
            if (found) {
                const int fl = __ffs(found) - 1;
                if (lane == fl) {
                    // the same fp32 running sum as lane_total, quantized per prefix
                    const unsigned long long base = pre + incl - mine;
                    float acc = 0.0f;
                    for (int e = 0; e < kTokLane; ++e) {
                        acc = __fadd_rn(acc, w[e]);
                        if (base + quantize(acc) > lt) {
                            tok = y0 + e;
                            break;
                        }
                    }
                }
                tok = __shfl_sync(kFullMask, tok, fl);
            }
        }
        if (lane == 0) {
            a.num_acc[r] = correct;
            a.bonus[r] = tok;
            a.commit[r] = correct + 1;
            if (a.new_seq) a.new_seq[r] = __ldg(a.prefix + r) + correct + 1;
        }
        if (lane < G) a.out[(size_t)r * (G + 1) + lane] = lane == correct ? tok : dj;
        else if (lane == G) a.out[(size_t)r * (G + 1) + G] = G == correct ? tok : -1;
    }
}

size_t samp_partial_bytes(int max_rows, int B, int gamma) {
    const size_t slots = (size_t)kSampMaxCtas + (size_t)max_rows + (size_t)B * gamma + 1;
    return (slots * (1 + kNormWarps) * sizeof(NormPartial) + 255) & ~size_t(255);
}

// launch_pdl in thread-block clusters of `cluster` CTAs along x (gridDim.x
// a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, int cluster, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename T>
cudaError_t launch_sampling(const SampArgs &a, bool vec, cudaStream_t s) {
    const size_t smem = (size_t)(a.B + 1) * sizeof(int32_t);
    cudaError_t e = vec ? launch_pdl(softmax_norm_kernel<T, true>, dim3(a.grid), dim3(kNormThreads), smem, s, a)
                        : launch_pdl(softmax_norm_kernel<T, false>, dim3(a.grid), dim3(kNormThreads), smem, s, a);
    if (e != cudaSuccess) return e;
    const int epc = vec ? Elem<T>::kPerChunk : 1;
    return launch_pdl_cluster(sampling_accept_kernel<T>, dim3(a.B * a.split), dim3(kSampThreads), 0, s,
                              a.split, a, epc, vec);
}

}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_sampling_workspace_bytes(int32_t max_rows, int32_t B, int32_t gamma) {
    if (max_rows < 0) max_rows = 0;
    if (B < 0) B = 0;
    if (gamma < 0) gamma = 0;
    return samp_partial_bytes(max_rows, B, gamma) + ((((size_t)B + 1) * 4 + 255) & ~size_t(255));
}

extern "C" int dspark_sampling_accept_ex(const void *target_logits, int32_t dtype, int64_t ld_t,
                                         int32_t V, int32_t max_rows, const int32_t *cu_seqlens,
                                         const void *draft_logits, int64_t ld_d,
                                         const float *draft_lse, const int32_t *draft,
                                         const int32_t *prefix_lens, int32_t B,
                                      int32_t gamma, const float *u_accept, const float *u_bonus,
                                      int32_t *num_accepted, int32_t *bonus, int32_t *commit_lens,
                                      int32_t *new_seq_lens, int32_t *out_tokens, void *workspace,
                                      size_t workspace_bytes, int32_t *status, void *stream) {
    if (!target_logits || !cu_seqlens || !draft_logits || !draft || !u_accept || !u_bonus ||
        !num_accepted || !bonus || !commit_lens || !out_tokens || !status)
        return DSPARK_ERR_INVALID_ARG;
    if (new_seq_lens && !prefix_lens) return DSPARK_ERR_INVALID_ARG;
    if (dtype != DSPARK_DTYPE_BF16 && dtype != DSPARK_DTYPE_F32) return DSPARK_ERR_INVALID_ARG;
    if (B < 1 || gamma < 1 || gamma > 31 || V < 1 || ld_t < V || ld_d < V || max_rows < 0)
        return DSPARK_ERR_INVALID_ARG;
    if (B > kSampMaxB || V > kSampMaxV) return DSPARK_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < dspark_sampling_workspace_bytes(max_rows, B, gamma) ||
        !aligned(workspace, 256))
        return DSPARK_ERR_WORKSPACE;
    const long long esize = dtype == DSPARK_DTYPE_BF16 ? 2 : 4;
    SampArgs a;
    a.tgt = target_logits;
    a.ld_t = ld_t;
    a.dft = draft_logits;
    a.ld_d = ld_d;
    a.draft_lse = draft_lse;
    a.V = V;
    a.B = B;
    a.gamma = gamma;
    a.max_rows = max_rows;
    a.cu = cu_seqlens;
    a.draft = draft;
    a.prefix = prefix_lens;
    a.u_acc = u_accept;
    a.u_bonus = u_bonus;
    a.num_acc = num_accepted;
    a.bonus = bonus;
    a.commit = commit_lens;
    a.new_seq = new_seq_lens;
    a.out = out_tokens;
    a.status = status;
    a.part = static_cast<NormPartial *>(workspace);
    {
        const size_t slots = (size_t)kSampMaxCtas + (size_t)max_rows + (size_t)B * gamma + 1;
        a.part_w = a.part + slots;
    }
    a.dcu = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(workspace) +
                                        samp_partial_bytes(max_rows, B, gamma));
    const int g = sm_count() * kNormCtasPerSm;
    a.grid = g < 1 ? 1 : (g > kSampMaxCtas ? kSampMaxCtas : g);
    // the accept kernel: as many CTAs per request as stay resident together
    // (one wave), at most one cluster's worth
    const int split = sm_count() * kSampCtasPerSm / B;
    a.split = split < 1 ? 1 : (split > kSampMaxCluster ? kSampMaxCluster : split);
    const bool vec = aligned(target_logits, 16) && aligned(draft_logits, 16) &&
                     (ld_t * esize) % 16 == 0 && (ld_d * esize) % 16 == 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = dtype == DSPARK_DTYPE_BF16 ? launch_sampling<__nv_bfloat16>(a, vec, s)
                                                     : launch_sampling<float>(a, vec, s);
    return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

extern "C" int dspark_sampling_accept(const void *target_logits, int32_t dtype, int64_t ld_t,
                                      int32_t V, int32_t max_rows, const int32_t *cu_seqlens,
                                      const void *draft_logits, int64_t ld_d,
                                      const int32_t *draft, const int32_t *prefix_lens, int32_t B,
                                      int32_t gamma, const float *u_accept, const float *u_bonus,
                                      int32_t *num_accepted, int32_t *bonus, int32_t *commit_lens,
                                      int32_t *new_seq_lens, int32_t *out_tokens, void *workspace,
                                      size_t workspace_bytes, int32_t *status, void *stream) {
    return dspark_sampling_accept_ex(target_logits, dtype, ld_t, V, max_rows, cu_seqlens,
                                     draft_logits, ld_d, nullptr, draft, prefix_lens, B, gamma,
                                     u_accept, u_bonus, num_accepted, bonus, commit_lens,
                                     new_seq_lens, out_tokens, workspace, workspace_bytes, status,
                                     stream);
}
