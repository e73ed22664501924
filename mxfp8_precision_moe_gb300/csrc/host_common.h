// host_common.h -- host-side helpers of the C ABI: device queries cached per
// device, the sm_103 architecture check, launch-status mapping, alignment.
#pragma once

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
inline mxfp8_status_t check_arch() {
    static std::atomic<int> cache[kMaxDevices];  // 0 unknown, 1 ok, 2 wrong arch
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices) return MXFP8_ERR_ARCH;
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

}  // namespace host
}  // namespace mx
