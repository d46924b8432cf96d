// api.cu -- error strings, version and the per-device host caches shared by
// the library's entry points.

#include "dspark_common.cuh"

#include <atomic>

namespace dspark {

namespace {
constexpr int kMaxDevices = 64;
constexpr int kMaxSmemSlots = 24;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_smem_done[kMaxDevices][kMaxSmemSlots];
}  // namespace

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return 1;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t ensure_smem(const void *kernel, int bytes, int slot) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || slot < 0 || slot >= kMaxSmemSlots)
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (g_smem_done[dev][slot].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) g_smem_done[dev][slot].store(bytes, std::memory_order_release);
    return e;
}

}  // namespace dspark

extern "C" const char *dspark_strerror(int code) {
    switch (code) {
        case DSPARK_OK: return "ok";
        case DSPARK_ERR_INVALID_ARG: return "invalid argument";
        case DSPARK_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
        case DSPARK_ERR_CUDA: return "CUDA launch or attribute call failed";
        case DSPARK_ERR_UNSUPPORTED: return "outside the supported envelope";
        default: return "unknown dspark error";
    }
}

extern "C" int dspark_version(void) { return 100; }

extern "C" int dspark_checked_build(void) { return dspark::kCheckedBuild ? 1 : 0; }
