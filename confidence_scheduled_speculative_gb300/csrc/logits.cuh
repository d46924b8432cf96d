// logits.cuh -- reading rows of target / draft logits (bf16 or fp32) on
// sm_103a: 16-byte streaming loads and per-chunk element access, shared by
// the greedy accept (accept.cu) and the sampling accept (sample.cu).
#pragma once

#include <cuda_bf16.h>

#include "dspark_common.cuh"

namespace dspark {

__device__ __forceinline__ uint4 ld_stream16(const uint4 *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// The same with a 256-byte L2 prefetch per access (the argmax's pure row
// stream: 6.58 against 6.50 TB/s back to back on dsv4_like).
__device__ __forceinline__ uint4 ld_stream16_pf(const uint4 *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ void take(float f, int idx, float &best, int &bidx, bool &nan) {
    if (f != f) nan = true;
    else if (f > best) {
        best = f;
        bidx = idx;
    }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <typename T>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kPerChunk = 8;
    __device__ static float load(const __nv_bfloat16 *p) {
        return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(p)) << 16);
    }
    __device__ static float at(const uint4 &v, int e) {
        const uint32_t w = e < 2 ? v.x : (e < 4 ? v.y : (e < 6 ? v.z : v.w));
        return (e & 1) ? bf16_hi(w) : bf16_lo(w);
    }
    // Largest value of the chunk; NaN if the chunk holds a NaN.  Packed
    // bf16x2 NaN-propagating max: 5 instructions for 8 values.
    __device__ static float chunk_max(const uint4 &v) {
        __nv_bfloat162 a, b, c, d;
        *reinterpret_cast<uint32_t *>(&a) = v.x;
        *reinterpret_cast<uint32_t *>(&b) = v.y;
        *reinterpret_cast<uint32_t *>(&c) = v.z;
        *reinterpret_cast<uint32_t *>(&d) = v.w;
        __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
        const uint32_t mw = *reinterpret_cast<uint32_t *>(&m);
        __nv_bfloat162 sw;
        *reinterpret_cast<uint32_t *>(&sw) = __byte_perm(mw, 0u, 0x1032);
        m = __hmax2_nan(m, sw);
        return bf16_lo(*reinterpret_cast<uint32_t *>(&m));
    }
};
template <>
struct Elem<float> {
    static constexpr int kPerChunk = 4;
    __device__ static float load(const float *p) { return __ldg(p); }
    __device__ static float at(const uint4 &v, int e) {
        const uint32_t w = e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w));
        return __uint_as_float(w);
    }
    __device__ static float chunk_max(const uint4 &v) {
        const float f0 = __uint_as_float(v.x), f1 = __uint_as_float(v.y);
        const float f2 = __uint_as_float(v.z), f3 = __uint_as_float(v.w);
        const bool nan = (f0 != f0) | (f1 != f1) | (f2 != f2) | (f3 != f3);
        return nan ? __uint_as_float(0x7FC00000u) : fmaxf(fmaxf(f0, f1), fmaxf(f2, f3));
    }
};

// Largest non-NaN value of a chunk that holds a NaN (rare path).
template <typename T>
__device__ __noinline__ float chunk_max_nonnan(uint4 v) {
    float m = -INFINITY;
#pragma unroll
    for (int e = 0; e < Elem<T>::kPerChunk; ++e) {
        const float f = Elem<T>::at(v, e);
        if (f > m) m = f;
    }
    return m;
}

}  // namespace dspark
