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

// C[M, N] = A . B on the tensor cores (sc_gemm.cu): A [M][K] (a_mn = 0) or
// [K][M] (a_mn = 1), B [N][K] (b_mn = 0) or [K][N] (b_mn = 1), bf16; C
// row-major, c_mode 0 bf16, 1 FP32, 2 FP32 added to C.  m_fastest orders the
// output tiles so that consecutive ones share B's tile (1) or A's (0).
// Checks its arguments; returns SC_OK or an error status (no message reset).
// k_splits > 1 (c_mode 1 only) splits each tile's K range over that many
// tiles; split s stores its rows at C row s * round_up(M, 128) + m.
int gemm_bf16(const uint16_t* A, long long lda, int a_mn, const uint16_t* B, long long ldb, int b_mn, void* C,
              long long ldc, int c_mode, long long M, long long N, long long K, int m_fastest, uint32_t* status,
              cudaStream_t stream, int k_splits);
// bf16 C = A . B with K split `k_splits` ways through FP32 slices in acc
// (k_splits x split_slice_rows(M) rows of ldacc floats), summed in slice order.
long long split_slice_rows(long long M);
int gemm_bf16_split(const uint16_t* A, long long lda, int a_mn, const uint16_t* B, long long ldb, int b_mn,
                    uint16_t* C, long long ldc, float* acc, long long ldacc, long long M, long long N, long long K,
                    int m_fastest, int k_splits, uint32_t* status, cudaStream_t stream);
// K splits (1..8) whose tiles come closest to whole waves over `sms` SMs.
int best_k_splits(long long M, long long N, long long K, int sms);
// SMs of the current device.
int sm_count(int* out);

inline bool aligned(const void* p, unsigned a) {
    return (reinterpret_cast<unsigned long long>(p) % a) == 0;
}

}  // namespace sc
