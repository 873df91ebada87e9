// sc_common.cu -- status codes, error messages, device checks, defaults.
#include <cstdio>
#include <cstring>
#include <mutex>

#include "sc_internal.h"

namespace sc {

namespace {
thread_local char g_last_error[512] = {0};

constexpr int kMaxDevices = 64;
// 0 = unknown, 1 = supported, 2 = unsupported
int g_device_state[kMaxDevices] = {0};
std::mutex g_device_mutex;
}  // namespace

int fail(int status, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

int ok() {
    g_last_error[0] = '\0';
    return SC_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(SC_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int check_device(int* device_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (device_out) *device_out = dev;
    if (dev < 0 || dev >= kMaxDevices) return fail(SC_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lock(g_device_mutex);
    if (g_device_state[dev] == 1) return SC_OK;
    if (g_device_state[dev] == 2)
        return fail(SC_ERR_UNSUPPORTED, "device %d is not an sm_103 GPU with cluster launch", dev);
    int major = 0, minor = 0, cluster = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute(major)");
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute(minor)");
    if ((e = cudaDeviceGetAttribute(&cluster, cudaDevAttrClusterLaunch, dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute(cluster)");
    if (major != 10 || minor != 3 || !cluster) {
        g_device_state[dev] = 2;
        return fail(SC_ERR_UNSUPPORTED,
                    "device %d has compute capability %d.%d; this library is built for sm_103a", dev,
                    major, minor);
    }
    g_device_state[dev] = 1;
    return SC_OK;
}

const char* last_error_text() { return g_last_error; }

}  // namespace sc

extern "C" {

int sc_params_default(sc_params* p) {
    if (!p) return sc::fail(SC_ERR_NULL, "p is NULL");
    std::memset(p, 0, sizeof *p);
    p->K_max = 128;
    p->is_mode = SC_IS_NONE;
    p->tis_max = 2.0f;
    p->mis_min = 0.5f;
    p->mis_max = 5.0f;
    p->centering = 1;
    p->inv_temperature = 1.0f;
    p->grad_scale = 1.0f;
    p->cluster_size = 0;
    p->threads = 0;
    p->stages = 0;
    p->clip_low = 0.2f;
    p->clip_high = 0.3f;
    p->flag_layout = 0;
    p->wait_limit_us = 0;
    p->test_stall = 0;
    return sc::ok();
}

const char* sc_status_string(int status) {
    switch (status) {
        case SC_OK: return "ok";
        case SC_ERR_NULL: return "null pointer";
        case SC_ERR_ALIGN: return "misaligned pointer or stride";
        case SC_ERR_SHAPE: return "size out of range";
        case SC_ERR_ARG: return "invalid argument";
        case SC_ERR_CUDA: return "CUDA error";
        case SC_ERR_UNSUPPORTED: return "unsupported device";
        default: return "unknown status";
    }
}

const char* sc_last_error(void) { return sc::last_error_text(); }

int sc_abi_version(void) { return 106; }

}  // extern "C"
