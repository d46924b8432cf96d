// pack.cu -- ragged verify pack on sm_103a.
//
// Pages (by title and section):
//   [ROUND] "DeepSeek-V4 DSpark一轮 Draft、Verify、Accept 与 Commit", §三
//           (verify ids = [anchor, draft tokens]; compact ragged layout built
//           by BuildRaggedVerifyWindow / compact_verify_ids), §四 (verify
//           positions)
//   [AVS]   "DSpark 自适应 Verify 怎样分配候选预算", §五 (compact rows
//           A0 A1 | B0 | C0 C1 C2 C3), §六 (cu_seqlens_q = [0,2,3,7])
//   [SGL]   "DSpark接入SGLang：用置信度驱动可变长度验证", "Ragged verify"
//           (front-pack into a compact buffer, round the total up to the
//           nearest captured tier)
//
// One warp per request, lane j = row j of the request (gamma+1 <= 32).  Each
// CTA covers 8 requests; it obtains the packed offset of its first request
// and the packed total (needed for the pad rows) from one block scan over
// all lengths (B is at most a few thousand, so every CTA re-reading
// verify_lens is cheaper than a separate scan kernel).  Token ids and
// positions are fetched before waiting on the planner.

#include "dspark_common.cuh"

namespace dspark {

constexpr int kPackThreads = 256;
constexpr int kPackReqPerCta = kPackThreads / 32;

__device__ __forceinline__ int clamp_len(int L, int gamma, bool &bad) {
    if (L < 1 || L > gamma + 1) {
        bad = true;
        return L < 1 ? 1 : gamma + 1;
    }
    return L;
}

__global__ void __launch_bounds__(kPackThreads)
pack_kernel(const int32_t *__restrict__ anchor, const int32_t *__restrict__ draft,
            const int32_t *__restrict__ prefix, const int32_t *__restrict__ lens, int B, int gamma,
            TierArgs tiers, int capacity, int32_t *__restrict__ ids, int32_t *__restrict__ pos,
            int32_t *__restrict__ req, int32_t *__restrict__ src, int32_t *__restrict__ cu,
            int32_t *__restrict__ totals, int32_t *__restrict__ status, bool in_chain) {
    __shared__ long long scan64[40];
    __shared__ int offs[kPackReqPerCta];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = blockIdx.x * kPackReqPerCta;
    const int r = r0 + warp;

    pdl_trigger();
    // token ids and prefix lengths are step inputs (not written by the
    // planner): behind the planner, fetch them while it finishes; called on
    // its own, after the wait (they may be outputs of the kernel before, e.g.
    // the bonus tokens and new sequence lengths of an accept)
    int tok = 0, pre = 0;
    auto fetch = [&]() {
        if (r < B) {
            pre = __ldg(prefix + r);
            if (lane == 0) tok = __ldg(anchor + r);
            else if (lane <= gamma) tok = __ldg(draft + (size_t)r * gamma + lane - 1);
        }
    };
    if (in_chain) fetch();
    pdl_wait();  // verify_lens come from the planner
    if (!in_chain) fetch();

    // total packed rows and the rows before this CTA's first request, in one
    // block scan of (total << 32 | before)
    long long both = 0;
    bool bad = false;
    for (int q = tid; q < B; q += kPackThreads) {
        const long long L = clamp_len(__ldg(lens + q), gamma, bad);
        both += (L << 32) | (q < r0 ? L : 0);
    }
    long long sum;
    block_exclusive_scan<long long>(both, scan64, &sum);
    const int total = (int)(sum >> 32), before = (int)(sum & 0xFFFFFFFFll);
    if (__syncthreads_or(bad) && tid == 0 && blockIdx.x == 0) flag(status, DSPARK_STATUS_BAD_LEN);

    bool b2 = false;
    const int L = r < B ? clamp_len(__ldg(lens + r), gamma, b2) : 0;
    if (warp == 0) {
        bool b3 = false;
        const int Lw = (r0 + lane < B && lane < kPackReqPerCta) ? clamp_len(__ldg(lens + r0 + lane), gamma, b3) : 0;
        int incl = Lw;
#pragma unroll
        for (int d = 1; d < kPackReqPerCta; d <<= 1) {
            const int o = __shfl_up_sync(kFullMask, incl, d);
            if (lane >= d) incl += o;
        }
        if (lane < kPackReqPerCta) offs[lane] = before + incl - Lw;
    }
    __syncthreads();

    bool over = false;
    if (r < B) {
        const int off = offs[warp];
        if (lane == 0 && in_bounds(r + 1, (long long)B + 1, status)) cu[r + 1] = off + L;
        if (lane < L) {
            const int dst = off + lane;
            if (dst < capacity && in_bounds(dst, capacity, status)) {
                ids[dst] = tok;
                pos[dst] = pre + lane;
                req[dst] = r;
                src[dst] = r * (gamma + 1) + lane;
            } else {
                over = true;
            }
        }
    }

    // graph-tier round-up and pad rows
    bool no_tier;
    const int padded = tier_round_up(tiers, total, &no_tier);
    const int pad_end = min(padded, capacity);
    for (int i = total + blockIdx.x * kPackThreads + tid; i < pad_end; i += gridDim.x * kPackThreads) {
        ids[i] = 0;
        pos[i] = 0;
        req[i] = -1;
        src[i] = -1;
    }
    if (blockIdx.x == 0 && tid == 0) {
        cu[0] = 0;
        totals[0] = total;
        totals[1] = padded;
        if (no_tier || padded > capacity) over = true;
    }
    if (__syncthreads_or(over) && tid == 0) flag(status, DSPARK_STATUS_CAPACITY);
}

// The data-parallel shared tier ([AVS] §六: local verify tier -> DP gather
// -> DP-global max token tier; [SGL] "Ragged verify": DP ranks share the
// largest tier any rank needs).  After the rank-local pack and the max over
// ranks, rows [totals[0], pad_to) become pad rows and totals[1] = pad_to.
// Starting from the real total (not the local padded end) rewrites the
// local pad rows with the same values, and lets pad_to alias totals + 1 (an
// in-place all-reduce).  A grid-stride loop over at most `capacity` rows.
__global__ void __launch_bounds__(kPackThreads)
pad_tier_kernel(const int32_t *pad_to, int capacity, int32_t *__restrict__ ids,
                int32_t *__restrict__ pos, int32_t *__restrict__ req, int32_t *__restrict__ src,
                int32_t *totals, int32_t *status) {
    pdl_trigger();
    pdl_wait();  // totals from the pack, pad_to from the collective
    const int total = __ldcg(totals);
    const int P = __ldcg(pad_to);  // when pad_to is totals + 1, the store below rewrites P
    if (P < total) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag(status, DSPARK_STATUS_BAD_TIER);
        return;
    }
    const int end = min(P, capacity);
    for (int i = total + blockIdx.x * kPackThreads + threadIdx.x; i < end;
         i += gridDim.x * kPackThreads) {
        ids[i] = 0;
        pos[i] = 0;
        req[i] = -1;
        src[i] = -1;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        totals[1] = P;
        if (P > capacity) flag(status, DSPARK_STATUS_CAPACITY);
    }
}

bool load_tiers(const int32_t *host_tiers, int32_t n_tiers, TierArgs *out) {
    if (n_tiers < 0 || n_tiers > DSPARK_MAX_TIERS || (n_tiers > 0 && !host_tiers)) return false;
    out->n = n_tiers;
    for (int i = 0; i < n_tiers; ++i) {
        out->t[i] = host_tiers[i];
        if (i > 0 && !(out->t[i] > out->t[i - 1])) return false;
    }
    for (int i = n_tiers; i < DSPARK_MAX_TIERS; ++i) out->t[i] = 0;
    return true;
}

cudaError_t launch_pack(bool in_chain, const int32_t *anchor, const int32_t *draft,
                        const int32_t *prefix,
                        const int32_t *lens, int B, int gamma, const TierArgs &tiers,
                        int capacity, int32_t *ids, int32_t *pos, int32_t *req, int32_t *src,
                        int32_t *cu, int32_t *totals, int32_t *status, cudaStream_t stream) {
    const int grid = (B + kPackReqPerCta - 1) / kPackReqPerCta;
    return launch_pdl(pack_kernel, dim3(grid), dim3(kPackThreads), 0, stream, anchor, draft,
                      prefix, lens, B, gamma, tiers, capacity, ids, pos, req, src, cu, totals,
                      status, in_chain);
}

}  // namespace dspark

using namespace dspark;

extern "C" int dspark_pack_verify(const int32_t *anchor, const int32_t *draft,
                                  const int32_t *prefix_lens, const int32_t *verify_lens, int32_t B,
                                  int32_t gamma, const int32_t *host_tiers, int32_t n_tiers,
                                  int32_t capacity, int32_t *packed_ids, int32_t *packed_pos,
                                  int32_t *packed_req, int32_t *packed_src, int32_t *cu_seqlens,
                                  int32_t *totals, int32_t *status, void *stream) {
    if (!anchor || !draft || !prefix_lens || !verify_lens || !packed_ids || !packed_pos ||
        !packed_req || !packed_src || !cu_seqlens || !totals || !status)
        return DSPARK_ERR_INVALID_ARG;
    if (B < 1 || gamma < 1 || gamma > 31 || capacity < 0) return DSPARK_ERR_INVALID_ARG;
    if ((long long)B * (gamma + 1) > 0x7FFFFFFF) return DSPARK_ERR_INVALID_ARG;
    TierArgs t;
    if (!load_tiers(host_tiers, n_tiers, &t)) return DSPARK_ERR_INVALID_ARG;
    if (launch_pack(false, anchor, draft, prefix_lens, verify_lens, B, gamma, t, capacity, packed_ids,
                    packed_pos, packed_req, packed_src, cu_seqlens, totals, status,
                    static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    return DSPARK_OK;
}

extern "C" int dspark_pad_to_tier(const int32_t *pad_to, int32_t capacity, int32_t *packed_ids,
                                  int32_t *packed_pos, int32_t *packed_req,
                                  int32_t *packed_src, int32_t *totals, int32_t *status,
                                  void *stream) {
    if (!pad_to || !packed_ids || !packed_pos || !packed_req || !packed_src || !totals ||
        !status)
        return DSPARK_ERR_INVALID_ARG;
    if (capacity < 0) return DSPARK_ERR_INVALID_ARG;
    // enough CTAs for 4 rows a thread, at most two per SM
    const int want = (capacity + 4 * kPackThreads - 1) / (4 * kPackThreads);
    const int grid = max(1, min(want, 2 * sm_count()));
    if (launch_pdl(pad_tier_kernel, dim3(grid), dim3(kPackThreads), 0,
                   static_cast<cudaStream_t>(stream), pad_to, (int)capacity, packed_ids,
                   packed_pos, packed_req, packed_src, totals, status) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    return DSPARK_OK;
}
