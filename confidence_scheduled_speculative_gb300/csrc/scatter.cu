// scatter.cu -- ScatterCompactToStrided on sm_103a.
//
// Pages (by title and section):
//   [ROUND] "DeepSeek-V4 DSpark一轮 Draft、Verify、Accept 与 Commit", §三
//           (after the target forward over the compact verify rows,
//           ScatterCompactToStrided puts the logits and hidden states back
//           into the [bs x stride] layout so that the accept addresses rows
//           by fixed position; verify_lens still bound which rows are valid)
//
// Packed row i < totals[0] goes to row packed_src[i] = r*(gamma+1) + j of
// the strided buffer; pad rows and strided rows no request selected are not
// touched.  A pure copy: rows x row_bytes read once and written once, so the
// bound is HBM bandwidth.
//
// Aligned rows (bases, strides and row size multiples of 16 bytes) move by
// TMA bulk copies: the rows are cut into 16 KB segments, each CTA of a
// persistent grid takes one equal contiguous range of segments (the work
// per CTA does not depend on the ragged row count, which only the device
// knows), and one thread runs a 4-stage pipeline -- cp.async.bulk global ->
// shared completing on an mbarrier, then cp.async.bulk shared -> global --
// so 64 KB per CTA are in flight with no per-element instructions.  A
// pipeline wait on an mbarrier gives up after wait_ns (200 ms unless the
// caller sets it) and flags DSPARK_STATUS_TIMEOUT; the CTA then copies
// nothing more, waits (up to 200 ms each) for the loads it still has in
// flight and for its stores, and exits.  Other rows are copied 2 bytes at a
// time by all threads.

#include "dspark_common.cuh"
#include "bulk.cuh"

namespace dspark {

constexpr int kScatterThreads = 256;    // 2-byte path
constexpr int kBulkCtasPerSm = 3;       // 64 KB of stages each
constexpr int kBulkStages = 4;
constexpr int kBulkSeg = 16384;         // bytes per bulk copy

struct ScatterArgs {
    const unsigned char *src;
    long long ld_src;  // bytes between source rows
    unsigned char *dst;
    long long ld_dst;  // bytes between destination rows
    long long row_bytes;
    const int32_t *packed_src;
    const int32_t *totals;
    int max_rows, dst_rows;
    unsigned long long wait_ns;  // limit of one pipeline wait
    int32_t *status;
};

__device__ __forceinline__ int scatter_rows_of(const ScatterArgs &a) {
    const int rows = *a.totals;
    return rows < 0 ? 0 : (rows > a.max_rows ? a.max_rows : rows);
}

// Segment t of the CTA's range: source row, byte offset and size (a
// multiple of 16: row_bytes is).
__device__ __forceinline__ void bulk_segment(const ScatterArgs &a, long long spr, long long t,
                                             int &r, long long &off, int &bytes) {
    r = (int)(t / spr);
    off = (t - (long long)r * spr) * kBulkSeg;
    const long long rem = a.row_bytes - off;
    bytes = (int)(rem < kBulkSeg ? rem : kBulkSeg);
}

__global__ void __launch_bounds__(32) scatter_bulk_kernel(ScatterArgs a) {
    extern __shared__ __align__(128) unsigned char stage_buf[];
    __shared__ __align__(8) unsigned long long bar[kBulkStages];
    pdl_trigger();
    if (threadIdx.x != 0) return;  // one thread drives the copy engine
    pdl_wait();  // packed_src / totals come from the pack, the rows from the forward
    const int rows = scatter_rows_of(a);
    const long long spr = (a.row_bytes + kBulkSeg - 1) / kBulkSeg;  // segments per row
    const long long T = (long long)rows * spr;
    const long long per = (T + gridDim.x - 1) / gridDim.x;
    const long long t0 = (long long)blockIdx.x * per;
    const long long n = max(0LL, min(t0 + per, T) - t0);
    for (int s = 0; s < kBulkStages; ++s) mbar_init(smem_addr(&bar[s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");

    uint32_t inflight = 0;  // bit s: a load into stage s is issued and not yet waited for
    auto load = [&](long long i) {
        int r, bytes;
        long long off;
        bulk_segment(a, spr, t0 + i, r, off, bytes);
        const int s = (int)(i % kBulkStages);
        inflight |= 1u << s;
        bulk_load(smem_addr(stage_buf + (size_t)s * kBulkSeg), a.src + (long long)r * a.ld_src + off,
                  (uint32_t)bytes, smem_addr(&bar[s]));
    };
    bool bad = false, timeout = false;
    uint32_t phase = 0;  // bit s: the parity stage s waits for next
    for (long long i = 0; i < min(n, (long long)kBulkStages); ++i) load(i);
    for (long long i = 0; i < n; ++i) {
        const int s = (int)(i % kBulkStages);
        if (!mbar_wait(smem_addr(&bar[s]), (phase >> s) & 1u, a.wait_ns)) {
            timeout = true;
            break;
        }
        inflight &= ~(1u << s);
        phase ^= 1u << s;
        int r, bytes;
        long long off;
        bulk_segment(a, spr, t0 + i, r, off, bytes);
        const int d = __ldg(a.packed_src + r);
        if (d < 0 || d >= a.dst_rows) {
            bad = true;
        } else {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                         ::"l"(a.dst + (long long)d * a.ld_dst + off),
                         "r"(smem_addr(stage_buf + (size_t)s * kBulkSeg)), "r"(bytes)
                         : "memory");
        }
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        if (i + kBulkStages < n) {
            // the store just issued read stage s: refill it after that
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            load(i + kBulkStages);
        }
    }
    if (timeout) {  // let the loads still in flight land before the CTA exits
        for (int s = 0; s < kBulkStages; ++s)
            if ((inflight >> s) & 1u) mbar_wait(smem_addr(&bar[s]), (phase >> s) & 1u);
        flag(a.status, DSPARK_STATUS_TIMEOUT);
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    if (bad) flag(a.status, DSPARK_STATUS_BAD_INDEX);
}

// Rows that are not 16-byte aligned: 2-byte copies (every row size is even:
// bf16 or fp32 elements), the flattened rows split evenly over the grid.
__global__ void __launch_bounds__(kScatterThreads) scatter_rows_kernel(ScatterArgs a) {
    pdl_trigger();
    pdl_wait();
    const int rows = scatter_rows_of(a);
    const long long cpr = a.row_bytes / 2;
    const long long W = (long long)rows * cpr;
    const long long per = (W + gridDim.x - 1) / gridDim.x;
    const long long q0 = (long long)blockIdx.x * per;
    const long long q1 = min(q0 + per, W);
    bool bad = false;
    for (long long q = q0; q < q1;) {
        const int r = (int)(q / cpr);
        const long long c0 = q - (long long)r * cpr;
        const long long seg_end = min(q1, (long long)(r + 1) * cpr);
        const long long c1 = c0 + (seg_end - q);
        const int d = __ldg(a.packed_src + r);
        if (d < 0 || d >= a.dst_rows) {
            bad = true;
        } else {
            const unsigned short *s =
                reinterpret_cast<const unsigned short *>(a.src + (long long)r * a.ld_src);
            unsigned short *t = reinterpret_cast<unsigned short *>(a.dst + (long long)d * a.ld_dst);
            for (long long c = c0 + threadIdx.x; c < c1; c += kScatterThreads) t[c] = __ldg(s + c);
        }
        q = seg_end;
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag(a.status, DSPARK_STATUS_BAD_INDEX);
}

}  // namespace dspark

using namespace dspark;

extern "C" int dspark_scatter_compact_to_strided_ex(const void *src, int64_t ld_src,
                                                    int32_t width, int32_t elem_bytes,
                                                    const int32_t *packed_src,
                                                    const int32_t *totals, int32_t max_rows,
                                                    void *dst, int64_t ld_dst, int32_t dst_rows,
                                                    int64_t wait_limit_ns, int32_t *status,
                                                    void *stream) {
    if (!src || !dst || !packed_src || !totals || !status) return DSPARK_ERR_INVALID_ARG;
    if (elem_bytes != 2 && elem_bytes != 4) return DSPARK_ERR_INVALID_ARG;
    if (width < 1 || ld_src < width || ld_dst < width || max_rows < 0 || dst_rows < 0)
        return DSPARK_ERR_INVALID_ARG;
    ScatterArgs a;
    a.src = static_cast<const unsigned char *>(src);
    a.dst = static_cast<unsigned char *>(dst);
    a.ld_src = ld_src * elem_bytes;
    a.ld_dst = ld_dst * elem_bytes;
    a.row_bytes = (long long)width * elem_bytes;
    a.packed_src = packed_src;
    a.totals = totals;
    a.max_rows = max_rows;
    a.dst_rows = dst_rows;
    a.wait_ns = wait_limit_ns < 0 ? kWaitLimitNs : (unsigned long long)wait_limit_ns;
    a.status = status;
    // TMA bulk copies need 16-byte aligned addresses and sizes
    const bool bulk = aligned(src, 16) && aligned(dst, 16) && a.ld_src % 16 == 0 &&
                      a.ld_dst % 16 == 0 && a.row_bytes % 16 == 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (bulk) {
        const int smem = kBulkStages * kBulkSeg;
        e = ensure_smem(reinterpret_cast<const void *>(scatter_bulk_kernel), smem, 6);
        if (e == cudaSuccess)
            e = launch_pdl(scatter_bulk_kernel, dim3(sm_count() * kBulkCtasPerSm), dim3(32),
                           (size_t)smem, s, a);
    } else {
        e = launch_pdl(scatter_rows_kernel, dim3(sm_count() * 4), dim3(kScatterThreads), 0, s, a);
    }
    return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

extern "C" int dspark_scatter_compact_to_strided(const void *src, int64_t ld_src, int32_t width,
                                                 int32_t elem_bytes, const int32_t *packed_src,
                                                 const int32_t *totals, int32_t max_rows,
                                                 void *dst, int64_t ld_dst, int32_t dst_rows,
                                                 int32_t *status, void *stream) {
    return dspark_scatter_compact_to_strided_ex(src, ld_src, width, elem_bytes, packed_src, totals,
                                                max_rows, dst, ld_dst, dst_rows, -1, status,
                                                stream);
}
