// sc_internal.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstdarg>

#include "../../include/sc.h"

namespace sc {

// Records a message for sc_last_error() and returns `status`.
int fail(int status, const char* fmt, ...);
// Clears the thread's last-error message and returns SC_OK.
int ok();
// Maps a CUDA error to SC_ERR_CUDA with a message naming `what`.
int cuda_fail(cudaError_t e, const char* what);
// Checks that the current device can run sm_103a code with clusters.
// Caches the answer per device.  Returns SC_OK or an error status.
int check_device(int* device_out);

inline bool aligned(const void* p, unsigned a) {
    return (reinterpret_cast<unsigned long long>(p) % a) == 0;
}

}  // namespace sc
