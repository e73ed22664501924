// host_common.h -- host-side helpers of the C ABI: device queries cached per
// device, the sm_103 architecture check, launch-status mapping, alignment.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

#include "../../include/mxfp8moe.h"

namespace mx {
namespace host {

constexpr int kMaxDevices = 64;

inline int current_device() {
    int d = 0;
    cudaGetDevice(&d);
    return d;
}

inline int num_sms() {
    static std::atomic<int> cache[kMaxDevices];
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices) return 148;
    int v = cache[d].load(std::memory_order_relaxed);
    if (v == 0) {
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d);
        if (v <= 0) v = 148;
        cache[d].store(v, std::memory_order_relaxed);
    }
    return v;
}

// The kernels are built for sm_103a only: refuse other devices up front.
// Also make sure the device's primary context is current in the calling host
// thread (a fresh thread, e.g. an autograd worker that has issued no CUDA call
// yet, has none, and encoding a TMA descriptor needs one).
inline mxfp8_status_t check_arch() {
    static std::atomic<int> cache[kMaxDevices];  // 0 unknown, 1 ok, 2 wrong arch
    static thread_local int bound = -1;
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices) return MXFP8_ERR_ARCH;
    if (bound != d) {
        if (cudaSetDevice(d) != cudaSuccess) return MXFP8_ERR_LAUNCH;
        bound = d;
    }
    int v = cache[d].load(std::memory_order_relaxed);
    if (v == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess)
            return MXFP8_ERR_LAUNCH;
        v = (major == 10 && minor == 3) ? 1 : 2;
        cache[d].store(v, std::memory_order_relaxed);
    }
    return v == 1 ? MXFP8_OK : MXFP8_ERR_ARCH;
}

inline mxfp8_status_t last_launch_status() {
    return cudaGetLastError() == cudaSuccess ? MXFP8_OK : MXFP8_ERR_LAUNCH;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuTensorMapEncodeTiled, looked up through the runtime (no -lcuda needed).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_relaxed);
    if (!f) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f = reinterpret_cast<EncodeTiledFn>(ptr);
            fn.store(f, std::memory_order_relaxed);
        }
    }
    return f;
}

// Raise a kernel's dynamic shared-memory limit once per device.
inline bool ensure_smem(const void* func, int bytes, std::atomic<int>* flags) {
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices) return false;
    if (flags[d].load(std::memory_order_relaxed)) return true;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    flags[d].store(1, std::memory_order_relaxed);
    return true;
}

}  // namespace host
}  // namespace mx
