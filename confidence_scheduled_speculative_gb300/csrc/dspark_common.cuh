// dspark_common.cuh -- device helpers and host plumbing shared by the
// library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/dspark.h"
#include "sigmoid.cuh"

namespace dspark {

constexpr unsigned kFullMask = 0xffffffffu;

// Set a status bit from device code.  Kernels never trap: every condition a
// kernel can detect is reported here and the host decides.
__device__ __forceinline__ void flag(int32_t *status, int bit) { atomicOr(status, bit); }

// Bounds-checked build (-DDSPARK_CHECKED, built as libdspark_checked.so):
// the kernels pass each index they compute from data through in_bounds()
// before the global or shared-memory access it addresses.  An index outside
// [0, n) flags DSPARK_STATUS_OUT_OF_BOUNDS and the access is skipped.  Every
// such index is in range by construction once the inputs have passed their
// own checks, so a flag marks a defect of the library.  In the normal build
// in_bounds() is the constant true and the compiler removes it.
#ifdef DSPARK_CHECKED
constexpr bool kCheckedBuild = true;
#else
constexpr bool kCheckedBuild = false;
#endif

__device__ __forceinline__ bool in_bounds(long long i, long long n, int32_t *status) {
    if (!kCheckedBuild || (i >= 0 && i < n)) return true;
    flag(status, DSPARK_STATUS_OUT_OF_BOUNDS);
    return false;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start before its predecessor finishes;
// it must wait here before touching the predecessor's outputs.  Without the
// attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// STS-calibrated conditional confidence c = sigmoid(z / T) ([AVS] §二, the
// runtime formula c_i = sigmoid(z_i / T_i)): IEEE fp32 division, then the
// fp64 sigmoid 1 / (1 + exp(-t)) with CUDA's exp, rounded once to fp32 --
// computed in fp32 arithmetic where that certifies the same rounding
// (sigmoid.cuh).  The planner's survivals and the calibration statistics and
// fit all go through this one function, so a fitted temperature scores
// exactly the survivals the planner will compute.
__device__ __forceinline__ float sts_confidence(float z, float T) {
    const float t = __fdiv_rn(z, T);  // IEEE fp32 division
    float c;
    if (sigmoid_f32(t, c)) return c;
    return sigmoid_f64(t);
}

// Block-wide exclusive scan over blockDim.x threads (a multiple of 32, at
// most 1024).  `warp_tot` is shared scratch of at least 32 entries.  Returns
// the exclusive prefix of `v`; *total receives the block total.  Contains
// __syncthreads(): every thread of the block must call it.
template <typename T>
__device__ T block_exclusive_scan(T v, T *warp_tot, T *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    T incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        T o = __shfl_up_sync(kFullMask, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        T w = lane < nwarps ? warp_tot[lane] : T(0);
        T wi = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            T o = __shfl_up_sync(kFullMask, wi, d);
            if (lane >= d) wi += o;
        }
        if (lane < nwarps) warp_tot[lane] = wi - w;  // exclusive warp offsets
        if (lane == 31) warp_tot[32] = wi;            // block total
    }
    __syncthreads();
    T res = warp_tot[warp] + incl - v;
    *total = warp_tot[32];
    __syncthreads();
    return res;
}

// Graph tiers of the verify window (ascending), passed by value.
struct TierArgs {
    int n;
    int32_t t[DSPARK_MAX_TIERS];
};

// The packed total rounded up to the smallest tier >= total ([SGL] "Ragged
// verify"); no tiers: the total itself.  *no_tier is set when every tier is
// below the total (the window cannot be replayed; flagged as CAPACITY).
__device__ __forceinline__ int tier_round_up(const TierArgs &tiers, int total, bool *no_tier) {
    *no_tier = false;
    if (tiers.n <= 0) return total;
    for (int i = 0; i < tiers.n; ++i)
        if (tiers.t[i] >= total) return tiers.t[i];
    *no_tier = true;
    return total;
}

// Block-wide sum (all threads receive it).  `scratch` >= 33 entries.
template <typename T>
__device__ T block_sum(T v, T *scratch) {
    T total;
    block_exclusive_scan<T>(v, scratch, &total);
    return total;
}

}  // namespace dspark

// ---------------------------------------------------------------- host side
namespace dspark {

// Streaming multiprocessor count of the current device (cached per device).
int sm_count();

// Host-side check and copy of a tier list (ascending, at most
// DSPARK_MAX_TIERS); false when it is invalid.
bool load_tiers(const int32_t *host_tiers, int32_t n_tiers, TierArgs *out);

// The pack kernel on `stream` (pack.cu), launched after the planner with
// programmatic serialization.  in_chain: launched behind this library's
// planner pass, whose chain began after every earlier kernel completed, so
// the kernel may fetch the step inputs before its dependency wait.
cudaError_t launch_pack(bool in_chain, const int32_t *anchor, const int32_t *draft, const int32_t *prefix,
                        const int32_t *lens, int B, int gamma, const TierArgs &tiers,
                        int capacity, int32_t *ids, int32_t *pos, int32_t *req, int32_t *src,
                        int32_t *cu, int32_t *totals, int32_t *status, cudaStream_t stream);

// Raise a kernel's dynamic shared-memory limit once per device.
cudaError_t ensure_smem(const void *kernel, int bytes, int slot);

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// x / d for non-negative x and positive d, in 32-bit arithmetic when both
// fit (a 64-bit division is a long software sequence on the GPU).
__device__ __forceinline__ long long div_nonneg(long long x, long long d) {
    if (((unsigned long long)x | (unsigned long long)d) <= 0xFFFFFFFFull)
        return (long long)((unsigned)x / (unsigned)d);
    return x / d;
}

// Launch with the programmatic stream-serialization attribute so that the
// kernel's prologue overlaps its predecessor on the stream (the kernel calls
// pdl_wait() before reading what the predecessor wrote).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace dspark
