// accept.cu -- greedy accept (compact mode) and cap-accept on sm_103a.
//
// Pages (by title and section):
//   [ROUND] "DeepSeek-V4 DSpark一轮 Draft、Verify、Accept 与 Commit", §五
//           (AcceptGreedy: target_predict = argmax(target_logits); correct_len
//           counts the leading drafts equal to the target chain; bonus comes
//           from the last valid input row; FinalizeAcceptLens: commit_lens =
//           correct_len + 1, new_seq_lens = prefix_lens + commit_lens;
//           BuildOutTokens: copy the drafts, scatter the bonus at correct_len)
//   [AVS]   "DSpark 自适应 Verify 怎样分配候选预算", §三 (capped_correct_len =
//           min(raw_correct_len, verify_len - 1)), §五 "cap-accept"
//   [SGL]   "DSpark接入SGLang：用置信度驱动可变长度验证", "三种 verify mode"
//           (cap-accept commits what compact commits and exposes the
//           full-verify acceptance ceiling)
//
// The argmax over the vocabulary is the whole cost: rows * V * 2 bytes of
// bf16 read once from HBM.  It is a streaming reduction, not a contraction,
// so no tensor cores: the design goal is HBM bandwidth.
//
// argmax_kernel  persistent grid of (SMs x kCtasPerSm) CTAs.  The rows are
//   flattened into 16-byte chunks and cut into one equal contiguous range per
//   CTA, so every CTA streams the same number of bytes whatever the ragged
//   row count (which only the device knows: cu_seqlens[B]).  A CTA's range
//   crosses at most a few row boundaries; for each (CTA c, row r) piece it
//   writes one partial (max, lowest index) to slot c + r, which is unique
//   because c + r increases by at least one from one piece to the next.
//   Inner loop: kUnroll independent 16-byte non-allocating loads with a
//   256-byte L2 prefetch per thread in flight (7 CTAs x 256 threads x 4 per
//   SM: of the launch shapes measured on dsv4_like, 4 to 8 CTAs x 4 to 12
//   loads, this one streamed fastest, 6.80 TB/s back to back); each chunk is reduced by a packed bf16x2 NaN-propagating max
//   (5 instructions for 8 values) and folded into a running (max, first
//   chunk holding it) with one compare and two selects -- no divergent
//   per-element path.  After the block reduction the winning chunk is read
//   once more to find the first element equal to the max (-0 == +0).  A
//   chunk holding a NaN takes a rare path that skips the NaN and flags it.
// finalize kernels  one warp per request, lane j = verify row j: combine the
//   partials of the row, compare with draft j, ballot the mismatches; the
//   first set bit is correct_len (no acceptance after the first mismatch).

#include "dspark_common.cuh"
#include "logits.cuh"

#include <atomic>


namespace dspark {

constexpr int kArgmaxThreads = 256;
constexpr int kCtasPerSm = 7;
constexpr int kUnroll = 4;
constexpr int kMaxCtas = 4096;
constexpr int kFinalWarps = 8;

struct Partial {
    float v;
    int i;
};

// Partial slots of a workspace for max_rows rows: slot c + r of CTA c < kMaxCtas
// and row r < max_rows.
__host__ __device__ __forceinline__ long long partial_slots(int max_rows) {
    return (long long)kMaxCtas + (max_rows > 0 ? max_rows : 0) + 1;
}

struct ArgmaxArgs {
    const void *logits;
    long long ld;
    int V;
    int rows_host;           // used when rows_dev is null
    const int32_t *rows_dev;  // cu_seqlens + B (compact mode)
    int max_rows;
    Partial *partial;
    int32_t *status;
    int32_t *zero_totals;  // cap-accept totals, zeroed here before the finalize adds
};

__device__ __forceinline__ int device_rows(const int32_t *rows_dev, int rows_host, int max_rows) {
    if (!rows_dev) return rows_host;
    const int r = *rows_dev;
    return r < 0 ? 0 : (r > max_rows ? max_rows : r);
}

// One chunk into the running (best value, first chunk holding it).  The
// element index is recovered once per row segment, so the common path is
// branch-free: compare, two selects.
template <typename T>
__device__ __forceinline__ void chunk_step(const uint4 &v, int cc, float &best, int &bchunk,
                                           bool &nan) {
    float m = Elem<T>::chunk_max(v);
    if (m != m) {
        nan = true;
        m = chunk_max_nonnan<T>(v);
    }
    const bool up = m > best;
    best = up ? m : best;
    bchunk = up ? cc : bchunk;
}

// Scan the full 16-byte chunks [c0, c1) of one row.
template <typename T>
__device__ __forceinline__ void scan_chunks(const uint4 *row4, int c0, int c1, float &best,
                                            int &bchunk, bool &nan) {
    int c = c0 + (int)threadIdx.x;
    for (; c + (kUnroll - 1) * kArgmaxThreads < c1; c += kUnroll * kArgmaxThreads) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream16_pf(row4 + c + u * kArgmaxThreads);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) chunk_step<T>(v[u], c + u * kArgmaxThreads, best, bchunk, nan);
    }
    for (; c < c1; c += kArgmaxThreads) chunk_step<T>(ld_stream16_pf(row4 + c), c, best, bchunk, nan);
}

// Scalar scan of elements [e0, e1) (unaligned rows).
template <typename T>
__device__ __forceinline__ void scan_scalar(const T *row, int e0, int e1, float &best, int &bidx,
                                            bool &nan) {
    int e = e0 + (int)threadIdx.x;
    for (; e + (kUnroll - 1) * kArgmaxThreads < e1; e += kUnroll * kArgmaxThreads) {
        float f[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) f[u] = Elem<T>::load(row + e + u * kArgmaxThreads);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) take(f[u], e + u * kArgmaxThreads, best, bidx, nan);
    }
    for (; e < e1; e += kArgmaxThreads) take(Elem<T>::load(row + e), e, best, bidx, nan);
}

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

// Block-wide (max value, lowest index); the result is valid in thread 0.
__device__ __forceinline__ void block_best(float &best, int &bidx, float *red_v, int *red_i) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const float ov = __shfl_down_sync(kFullMask, best, d);
        const int oi = __shfl_down_sync(kFullMask, bidx, d);
        if (better(ov, oi, best, bidx)) {
            best = ov;
            bidx = oi;
        }
    }
    if (lane == 0) {
        red_v[warp] = best;
        red_i[warp] = bidx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kArgmaxThreads / 32; ++w)
            if (better(red_v[w], red_i[w], best, bidx)) {
                best = red_v[w];
                bidx = red_i[w];
            }
    }
    __syncthreads();
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kArgmaxThreads, kCtasPerSm) argmax_kernel(ArgmaxArgs a) {
    __shared__ float red_v[kArgmaxThreads / 32];
    __shared__ int red_i[kArgmaxThreads / 32];
    constexpr int EPC = VEC ? Elem<T>::kPerChunk : 1;

    pdl_wait();  // cu_seqlens / logits come from the kernels before
    // the finalize launches once every CTA is past its wait, so it may read
    // what the kernels before wrote (cu_seqlens, verify_lens) in its prologue
    pdl_trigger();
    const int rows = device_rows(a.rows_dev, a.rows_host, a.max_rows);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (a.rows_dev && *a.rows_dev > a.max_rows) flag(a.status, DSPARK_STATUS_CAPACITY);
        if (a.zero_totals) {
            a.zero_totals[0] = 0;
            a.zero_totals[1] = 0;
        }
    }
    const int cpr = (a.V + EPC - 1) / EPC;  // chunks per row, the last one maybe partial
    const int full = a.V / EPC;             // full chunks per row
    const long long W = (long long)rows * cpr;
    const long long per = div_nonneg(W + gridDim.x - 1, gridDim.x);
    const long long q0 = (long long)blockIdx.x * per;
    const long long q1 = min(q0 + per, W);
    bool nan = false;
    for (long long q = q0; q < q1;) {
        const int r = (int)div_nonneg(q, cpr);
        const int c0 = (int)(q - (long long)r * cpr);
        const long long seg_end = min(q1, (long long)(r + 1) * cpr);
        const int c1 = c0 + (int)(seg_end - q);
        const T *row = reinterpret_cast<const T *>(a.logits) + (long long)r * a.ld;
        float best = -INFINITY;
        int bidx;
        if (VEC) {
            int bchunk = c0;
            scan_chunks<T>(reinterpret_cast<const uint4 *>(row), c0, min(c1, full), best, bchunk,
                           nan);
            block_best(best, bchunk, red_v, red_i);  // lowest chunk holding the max
            if (threadIdx.x == 0) {
                bidx = c0 * EPC;
                if (best > -INFINITY) {
                    // first element of that chunk equal to the max (-0 == +0)
                    const uint4 v = ld_stream16_pf(reinterpret_cast<const uint4 *>(row) + bchunk);
                    bidx = bchunk * EPC + EPC - 1;
#pragma unroll
                    for (int e = EPC - 1; e >= 0; --e)
                        if (Elem<T>::at(v, e) == best) bidx = bchunk * EPC + e;
                }
                // the row's partial last chunk, element by element
                for (int e = full * EPC; c1 > full && e < a.V; ++e)
                    take(Elem<T>::load(row + e), e, best, bidx, nan);
            }
        } else {
            bidx = c0;
            scan_scalar<T>(row, c0, c1, best, bidx, nan);
            block_best(best, bidx, red_v, red_i);
        }
        if (threadIdx.x == 0 && in_bounds(blockIdx.x + r, partial_slots(a.max_rows), a.status))
            a.partial[blockIdx.x + r] = Partial{best, bidx};
        q = seg_end;
    }
    if (__syncthreads_or(nan) && threadIdx.x == 0) flag(a.status, DSPARK_STATUS_NAN_LOGIT);
}

struct FinalArgs {
    int rows_host;
    const int32_t *rows_dev;
    int max_rows, V, epc, grid;
    const Partial *partial;
    const int32_t *cu;    // greedy: cu_seqlens [B+1]
    const int32_t *lens;  // cap: verify_lens [B]
    const int32_t *draft, *prefix;
    int B, gamma;
    int32_t *argmax, *num_acc, *bonus, *commit, *new_seq, *out, *ceiling, *totals, *status;
};

// The argmax CTAs [c_lo, c_hi] whose ranges hold a piece of row `row`
// (integer divisions only: the finalize kernels take them before their
// dependency wait).
__device__ __forceinline__ void row_ctas(int row, long long cpr, long long per, int &c_lo,
                                         int &c_hi) {
    const long long q_first = (long long)row * cpr;
    c_lo = (int)div_nonneg(q_first, per);
    c_hi = (int)div_nonneg(q_first + cpr - 1, per);
}

// The argmax of row `row` from the partials of CTAs [c_lo, c_hi].
__device__ __forceinline__ int row_argmax_in(const Partial *partial, int row, int c_lo, int c_hi,
                                             int max_rows, int32_t *status) {
    if (!in_bounds(c_hi + row, partial_slots(max_rows), status)) return 0;
    // the first two partials (a row usually spans one or two CTAs) are
    // loaded together
    const Partial p0 = partial[c_lo + row];
    const Partial p1 = c_hi > c_lo ? partial[c_lo + 1 + row] : Partial{-INFINITY, 0x7FFFFFFF};
    float bv = p0.v;
    int bi = p0.i;
    if (better(p1.v, p1.i, bv, bi)) {
        bv = p1.v;
        bi = p1.i;
    }
    for (int c = c_lo + 2; c <= c_hi; ++c) {
        const Partial p = partial[c + row];
        if (better(p.v, p.i, bv, bi)) {
            bv = p.v;
            bi = p.i;
        }
    }
    return bi;
}

__device__ __forceinline__ int row_argmax(const Partial *partial, int row, long long cpr,
                                          long long per, int max_rows, int32_t *status) {
    int c_lo, c_hi;
    row_ctas(row, cpr, per, c_lo, c_hi);
    return row_argmax_in(partial, row, c_lo, c_hi, max_rows, status);
}

// per-row argmax output (every row < rows), grid-stride over all threads
__device__ __forceinline__ void write_argmax(const FinalArgs &a, int rows, long long cpr, long long per) {
    if (!a.argmax || per <= 0) return;
    const int nthreads = gridDim.x * blockDim.x;
    for (int row = blockIdx.x * blockDim.x + threadIdx.x; row < rows; row += nthreads)
        a.argmax[row] = row_argmax(a.partial, row, cpr, per, a.max_rows, a.status);
}

// BuildOutTokens and FinalizeAcceptLens for request r (lane 0 writes the
// scalars; pre = prefix_lens[r], fetched by lane 0 before the dependency wait)
__device__ __forceinline__ void finish(const FinalArgs &a, int r, int lane, int correct, int bon,
                                       int dj, int pre) {
    const int g = a.gamma;
    if (lane == 0) {
        a.num_acc[r] = correct;
        a.bonus[r] = bon;
        a.commit[r] = correct + 1;
        if (a.new_seq) a.new_seq[r] = pre + correct + 1;
    }
    if (lane < g) a.out[(size_t)r * (g + 1) + lane] = (lane == correct) ? bon : dj;
    else if (lane == g) a.out[(size_t)r * (g + 1) + g] = (g == correct) ? bon : -1;
}

__global__ void __launch_bounds__(kFinalWarps * 32) greedy_finalize_kernel(FinalArgs a) {
    // the next kernel may launch now: this library's kernels read nothing
    // this one writes before their own dependency wait
    pdl_trigger();
    const int rq = blockIdx.x * kFinalWarps + (threadIdx.x >> 5);
    const int ln = threadIdx.x & 31;
    // drafts and prefix lengths are step inputs, and cu_seqlens was written
    // before any argmax CTA passed its wait (which precedes this grid's
    // launch): fetch them while the argmax finishes, from L2
    const int dj = (rq < a.B && ln < a.gamma) ? __ldg(a.draft + (size_t)rq * a.gamma + ln) : -1;
    const int pre = (a.new_seq && rq < a.B && ln == 0) ? __ldg(a.prefix + rq) : 0;
    const int rows = a.rows_dev ? min(max(__ldcg(a.rows_dev), 0), a.max_rows) : a.rows_host;
    const int lo = rq < a.B ? __ldcg(a.cu + rq) : 0, hi = rq < a.B ? __ldcg(a.cu + rq + 1) : 0;
    const long long cpr = (a.V + a.epc - 1) / a.epc;
    const long long W = (long long)rows * cpr;
    const long long per = div_nonneg(W + a.grid - 1, a.grid);
    const int lane = ln;
    const int r = rq;
    const int g = a.gamma;
    const int L = hi - lo;
    const bool valid = r < a.B && lo >= 0 && hi <= rows && L >= 1 && L <= g + 1;
    const bool mine = valid && lane < L;  // this lane's row: lo + lane
    int c_lo = 0, c_hi = 0;
    if (mine) row_ctas(lo + lane, cpr, per, c_lo, c_hi);
    pdl_wait();
    // the request's row argmaxes first, so that their partial loads and the
    // argmax output pass's are in flight together
    const int am = mine ? row_argmax_in(a.partial, lo + lane, c_lo, c_hi, a.max_rows, a.status) : 0;
    write_argmax(a, rows, cpr, per);

    if (r >= a.B) return;  // warp-uniform
    if (__any_sync(kFullMask, lane < g && (dj < 0 || dj >= a.V)) && lane == 0)
        flag(a.status, DSPARK_STATUS_TOKEN_RANGE);
    if (!valid) {
        if (lane == 0) {
            a.num_acc[r] = 0;
            a.bonus[r] = -1;
            a.commit[r] = 0;
            if (a.new_seq) a.new_seq[r] = pre;
            flag(a.status, DSPARK_STATUS_BAD_LEN);
        }
        if (lane < g) a.out[(size_t)r * (g + 1) + lane] = dj;
        else if (lane == g) a.out[(size_t)r * (g + 1) + g] = -1;
        return;
    }
    const unsigned mism = __ballot_sync(kFullMask, lane < L - 1 && am != dj);
    const int correct = mism ? __ffs(mism) - 1 : L - 1;
    const int bon = __shfl_sync(kFullMask, am, correct);
    finish(a, r, lane, correct, bon, dj, pre);
}

__global__ void __launch_bounds__(kFinalWarps * 32) cap_finalize_kernel(FinalArgs a) {
    __shared__ int sums[2];
    pdl_trigger();  // as in greedy_finalize_kernel
    const int rq = blockIdx.x * kFinalWarps + (threadIdx.x >> 5);
    const int ln = threadIdx.x & 31;
    const int dj0 = (rq < a.B && ln < a.gamma) ? __ldg(a.draft + (size_t)rq * a.gamma + ln) : -1;
    const int pre = (a.new_seq && rq < a.B && ln == 0) ? __ldg(a.prefix + rq) : 0;
    const int len0 = rq < a.B ? __ldcg(a.lens + rq) : 0;  // written before the argmax's wait
    const int rows = a.rows_host;
    const long long cpr = (a.V + a.epc - 1) / a.epc;
    const long long W = (long long)rows * cpr;
    const long long per = div_nonneg(W + a.grid - 1, a.grid);
    const int lane = ln;
    const int r = rq;
    const int g = a.gamma;
    const bool mine = r < a.B && lane <= g;  // this lane's row: r*(gamma+1) + lane
    int c_lo = 0, c_hi = 0;
    if (mine) row_ctas(r * (g + 1) + lane, cpr, per, c_lo, c_hi);
    pdl_wait();
    // the request's row argmaxes first (their loads in flight with the
    // argmax output pass's)
    const int am0 = mine ? row_argmax_in(a.partial, r * (g + 1) + lane, c_lo, c_hi, a.max_rows,
                                         a.status)
                         : 0;
    write_argmax(a, rows, cpr, per);
    if (threadIdx.x == 0) sums[0] = sums[1] = 0;
    __syncthreads();

    if (r < a.B) {
        const int dj = dj0;
        if (__any_sync(kFullMask, lane < g && (dj < 0 || dj >= a.V)) && lane == 0)
            flag(a.status, DSPARK_STATUS_TOKEN_RANGE);
        const int am = am0;
        const unsigned mism = __ballot_sync(kFullMask, lane < g && am != dj);
        const int raw = mism ? __ffs(mism) - 1 : g;
        int len = len0;
        if (len < 1 || len > g + 1) {
            if (lane == 0) flag(a.status, DSPARK_STATUS_BAD_LEN);
            len = len < 1 ? 1 : g + 1;
        }
        const int capped = min(raw, len - 1);
        const int bon = __shfl_sync(kFullMask, am, capped);
        finish(a, r, lane, capped, bon, dj, pre);
        if (lane == 0) {
            a.ceiling[r] = raw;
            atomicAdd(&sums[0], capped + 1);
            atomicAdd(&sums[1], raw + 1);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        atomicAdd(&a.totals[0], sums[0]);
        atomicAdd(&a.totals[1], sums[1]);
    }
}

int argmax_grid() {
    const int g = sm_count() * kCtasPerSm;
    return g < 1 ? 1 : (g > kMaxCtas ? kMaxCtas : g);
}

template <typename T>
cudaError_t launch_argmax(const ArgmaxArgs &a, bool vec, int grid, cudaStream_t s) {
    if (vec) return launch_pdl(argmax_kernel<T, true>, dim3(grid), dim3(kArgmaxThreads), 0, s, a);
    return launch_pdl(argmax_kernel<T, false>, dim3(grid), dim3(kArgmaxThreads), 0, s, a);
}

int run_accept(const void *logits, int dtype, long long ld, int V, int max_rows, int rows_host,
               const int32_t *rows_dev, FinalArgs f, bool cap, void *ws, size_t ws_bytes,
               cudaStream_t s) {
    if (!ws || ws_bytes < dspark_accept_workspace_bytes(max_rows, V) || !aligned(ws, 256))
        return DSPARK_ERR_WORKSPACE;
    const size_t esize = dtype == DSPARK_DTYPE_BF16 ? 2 : 4;
    const bool vec = aligned(logits, 16) && ((ld * (long long)esize) % 16 == 0);
    const int grid = argmax_grid();
    ArgmaxArgs a;
    a.logits = logits;
    a.ld = ld;
    a.V = V;
    a.rows_host = rows_host;
    a.rows_dev = rows_dev;
    a.max_rows = max_rows;
    a.partial = static_cast<Partial *>(ws);
    a.status = f.status;
    a.zero_totals = cap ? f.totals : nullptr;
    cudaError_t e = dtype == DSPARK_DTYPE_BF16 ? launch_argmax<__nv_bfloat16>(a, vec, grid, s)
                                               : launch_argmax<float>(a, vec, grid, s);
    if (e != cudaSuccess) return DSPARK_ERR_CUDA;
    f.rows_host = rows_host;
    f.rows_dev = rows_dev;
    f.max_rows = max_rows;
    f.V = V;
    f.epc = vec ? (int)(16 / esize) : 1;
    f.grid = grid;
    f.partial = a.partial;
    const int fgrid = (f.B + kFinalWarps - 1) / kFinalWarps;
    e = cap ? launch_pdl(cap_finalize_kernel, dim3(fgrid), dim3(kFinalWarps * 32), 0, s, f)
            : launch_pdl(greedy_finalize_kernel, dim3(fgrid), dim3(kFinalWarps * 32), 0, s, f);
    return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

int check_common(const void *logits, int dtype, long long ld, int V, const int32_t *draft,
                 const int32_t *prefix, int B, int gamma, const int32_t *num_acc,
                 const int32_t *bonus, const int32_t *commit, const int32_t *new_seq,
                 const int32_t *out, const int32_t *status) {
    if (!logits || !draft || !num_acc || !bonus || !commit || !out || !status)
        return DSPARK_ERR_INVALID_ARG;
    if (new_seq && !prefix) return DSPARK_ERR_INVALID_ARG;
    if (dtype != DSPARK_DTYPE_BF16 && dtype != DSPARK_DTYPE_F32) return DSPARK_ERR_INVALID_ARG;
    if (B < 1 || gamma < 1 || gamma > 31 || V < 1 || ld < V) return DSPARK_ERR_INVALID_ARG;
    return DSPARK_OK;
}

}  // namespace dspark

using namespace dspark;

extern "C" size_t dspark_accept_workspace_bytes(int32_t max_rows, int32_t V) {
    (void)V;
    if (max_rows < 0) max_rows = 0;
    const size_t n = (size_t)partial_slots(max_rows);
    return (n * sizeof(Partial) + 255) & ~size_t(255);
}

extern "C" int dspark_greedy_accept(const void *logits, int32_t dtype, int64_t ld, int32_t V,
                                    int32_t max_rows, const int32_t *cu_seqlens,
                                    const int32_t *draft, const int32_t *prefix_lens, int32_t B,
                                    int32_t gamma, int32_t *argmax, int32_t *num_accepted,
                                    int32_t *bonus, int32_t *commit_lens, int32_t *new_seq_lens,
                                    int32_t *out_tokens, void *workspace, size_t workspace_bytes,
                                    int32_t *status, void *stream) {
    int rc = check_common(logits, dtype, ld, V, draft, prefix_lens, B, gamma, num_accepted, bonus,
                          commit_lens, new_seq_lens, out_tokens, status);
    if (rc != DSPARK_OK) return rc;
    if (!cu_seqlens || max_rows < 0) return DSPARK_ERR_INVALID_ARG;
    FinalArgs f = {};
    f.cu = cu_seqlens;
    f.draft = draft;
    f.prefix = prefix_lens;
    f.B = B;
    f.gamma = gamma;
    f.argmax = argmax;
    f.num_acc = num_accepted;
    f.bonus = bonus;
    f.commit = commit_lens;
    f.new_seq = new_seq_lens;
    f.out = out_tokens;
    f.status = status;
    return run_accept(logits, dtype, ld, V, max_rows, 0, cu_seqlens + B, f, false, workspace,
                      workspace_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" int dspark_cap_accept(const void *logits, int32_t dtype, int64_t ld, int32_t V,
                                 const int32_t *verify_lens, const int32_t *draft,
                                 const int32_t *prefix_lens, int32_t B, int32_t gamma,
                                 int32_t *argmax, int32_t *num_accepted, int32_t *bonus,
                                 int32_t *commit_lens, int32_t *new_seq_lens, int32_t *out_tokens,
                                 int32_t *ceiling, int32_t *totals, void *workspace,
                                 size_t workspace_bytes, int32_t *status, void *stream) {
    int rc = check_common(logits, dtype, ld, V, draft, prefix_lens, B, gamma, num_accepted, bonus,
                          commit_lens, new_seq_lens, out_tokens, status);
    if (rc != DSPARK_OK) return rc;
    if (!verify_lens || !ceiling || !totals) return DSPARK_ERR_INVALID_ARG;
    if ((long long)B * (gamma + 1) > 0x7FFFFFFF) return DSPARK_ERR_INVALID_ARG;
    const int rows = B * (gamma + 1);
    FinalArgs f = {};
    f.lens = verify_lens;
    f.draft = draft;
    f.prefix = prefix_lens;
    f.B = B;
    f.gamma = gamma;
    f.argmax = argmax;
    f.num_acc = num_accepted;
    f.bonus = bonus;
    f.commit = commit_lens;
    f.new_seq = new_seq_lens;
    f.out = out_tokens;
    f.ceiling = ceiling;
    f.totals = totals;
    f.status = status;
    return run_accept(logits, dtype, ld, V, rows, rows, nullptr, f, true, workspace,
                      workspace_bytes, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------- allocation-free variant
//
// dspark_greedy_accept_static: the same compact-mode greedy accept, for
// callers that cannot allocate device memory -- an embedding that hands over
// only tensors it owns, or a runtime whose device memory is fixed at start-up
// and which forbids cudaMalloc afterwards.  Its scratch (the per-CTA partials
// of the argmax) lives in the file-scope array below instead of a caller
// workspace.  Every GPU that loads this library holds the array (about
// 300 KB) until the process exits.

namespace dspark {

constexpr int kStaticMaxRows = 32768;  // largest max_rows the static scratch serves
// partial slots, rounded up to whole 256-byte blocks like a workspace
constexpr int kStaticSlots = ((kMaxCtas + kStaticMaxRows + 1) + 31) / 32 * 32;

static __device__ __align__(256) Partial g_static_partials[kStaticSlots];

namespace {
constexpr int kMaxStaticDevices = 64;
std::atomic<Partial *> g_static_ptr[kMaxStaticDevices];
}  // namespace

// Device address of g_static_partials on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is taken
// once per device with cudaGetSymbolAddress (which also loads this module
// on that device) and kept for the life of the process; a cudaDeviceReset
// unloads the module, so the kept address is then stale.
static cudaError_t static_partials(Partial **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxStaticDevices) return cudaErrorInvalidDevice;
    Partial *p = g_static_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_static_partials);
        if (e != cudaSuccess) return e;
        g_static_ptr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace dspark

extern "C" int dspark_greedy_accept_static(const void *logits, int32_t dtype, int64_t ld,
                                           int32_t V, int32_t max_rows,
                                           const int32_t *cu_seqlens, const int32_t *draft,
                                           const int32_t *prefix_lens, int32_t B, int32_t gamma,
                                           int32_t *argmax, int32_t *num_accepted,
                                           int32_t *bonus, int32_t *commit_lens,
                                           int32_t *new_seq_lens, int32_t *out_tokens,
                                           int32_t *status, void *stream) {
    static_assert(sizeof(g_static_partials) % 256 == 0, "whole 256-byte blocks");
    int rc = check_common(logits, dtype, ld, V, draft, prefix_lens, B, gamma, num_accepted, bonus,
                          commit_lens, new_seq_lens, out_tokens, status);
    if (rc != DSPARK_OK) return rc;
    if (!cu_seqlens || max_rows < 0) return DSPARK_ERR_INVALID_ARG;
    if (max_rows > kStaticMaxRows) return DSPARK_ERR_UNSUPPORTED;
    Partial *partial = nullptr;
    if (static_partials(&partial) != cudaSuccess) return DSPARK_ERR_CUDA;
    FinalArgs f = {};
    f.cu = cu_seqlens;
    f.draft = draft;
    f.prefix = prefix_lens;
    f.B = B;
    f.gamma = gamma;
    f.argmax = argmax;
    f.num_acc = num_accepted;
    f.bonus = bonus;
    f.commit = commit_lens;
    f.new_seq = new_seq_lens;
    f.out = out_tokens;
    f.status = status;
    // the array stands in for the workspace: every slot the finalize reads
    // is written earlier in the same call, so nothing needs clearing
    return run_accept(logits, dtype, ld, V, max_rows, 0, cu_seqlens + B, f, false, partial,
                      sizeof(g_static_partials), static_cast<cudaStream_t>(stream));
}
