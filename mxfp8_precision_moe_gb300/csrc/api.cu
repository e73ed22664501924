// api.cu -- size helpers, status strings and the bounded-wait self-test of the
// C ABI declared in include/mxfp8moe.h.

#include "common.cuh"
#include "host_common.h"

namespace mx {

// One thread waits on an mbarrier that nothing ever arrives on, through the
// same bounded wait the GEMM uses; it must give up after limit_ns and record
// MXFP8_ERR_TIMEOUT instead of hanging.
__global__ void wait_timeout_probe_kernel(int32_t* dev_status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_bounded<true>(&bar, 0, limit_ns, &abort_flag, dev_status);
    __syncthreads();
}

}  // namespace mx

using namespace mx;

extern "C" size_t mxfp8_scale_bytes(int64_t rows, int64_t K, int32_t G, int scale_layout) {
    if (rows < 0 || K < 0 || K % 32) return 0;
    if (scale_layout == MXFP8_SCALES_COMPACT) return (size_t)(rows * (K / 32));
    const int64_t g = G > 1 ? G : 1;
    return (size_t)(((rows + 127) / 128 + g) * 128 * ((K + 127) / 128) * 4);
}

extern "C" size_t mxfp8_scale_bytes_colgroups(int64_t R, int64_t M, int32_t G) {
    if (R < 0 || M < 0) return 0;
    const int64_t g = G > 1 ? G : 1;
    return (size_t)(((R + 127) / 128) * 128 * ((M + 127) / 128 + g) * 4);
}

extern "C" const char* mxfp8_status_string(mxfp8_status_t s) {
    switch (s) {
        case MXFP8_OK: return "ok";
        case MXFP8_ERR_NULL: return "a required pointer is NULL";
        case MXFP8_ERR_SHAPE: return "invalid shape";
        case MXFP8_ERR_ALIGN: return "size or pointer alignment requirement violated";
        case MXFP8_ERR_LAYOUT: return "invalid direction / scale layout";
        case MXFP8_ERR_ARCH: return "device is not sm_103 (GB300)";
        case MXFP8_ERR_LAUNCH: return "CUDA launch failed";
        case MXFP8_ERR_OFFSETS: return "invalid group offsets (device-detected)";
        case MXFP8_ERR_TIMEOUT: return "bounded wait timed out (device-detected)";
        case MXFP8_ERR_DRIVER: return "TMA descriptor encoding failed";
    }
    return "unknown status";
}

extern "C" mxfp8_status_t mxfp8_debug_wait_timeout(int32_t* dev_status, uint64_t limit_ns, mxfp8_stream_t stream) {
    if (!dev_status) return MXFP8_ERR_NULL;
    if (limit_ns == 0 || limit_ns > 10000000000ull) return MXFP8_ERR_SHAPE;
    if (mxfp8_status_t a = host::check_arch(); a != MXFP8_OK) return a;
    wait_timeout_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(dev_status, limit_ns);
    return host::last_launch_status();
}
