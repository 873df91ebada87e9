// sc_advantages.cu -- GRPO group advantages (one warp per group), the
// per-rollout mean of the clipped GRPO baseline (advantage / valid tokens),
// and the batch loss grad_scale * sum_t loss_t of the fused call.
//
// Follows the "Training" section of the Agent Lightning "Score Centering"
// docs page (rollout-level advantages with group standard-deviation
// normalisation) and section 4 of the devotd.net release note (rewards stay
// fractional FP32, no overflow in the denominator, mean-only variant).
//
// Statistics are taken in FP64 with two passes (mean, then the centred sum of
// squares), so squares of large FP32 rewards cannot overflow.  A group whose
// rewards are all equal is detected exactly (min == max) and gets A = 0
// without any division.
#include <cmath>

#include "sc_internal.h"

namespace sc {
namespace {

__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ float warp_min_f32(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ float warp_max_f32(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Grid: one 32-thread block per group.
__global__ void __launch_bounds__(32) group_adv_kernel(const float* rewards, int group_size,
                                                       int normalize_std, float eps, float* adv) {
    // No early trigger of the next grid (griddepcontrol.launch_dependents): the
    // fused call that follows is a persistent grid of clusters, and launched
    // while these CTAs still hold SMs, part of its clusters started late
    // (measured: 16384 x 248320 rows 3.08 -> 5.05 ms, 65536 x 151936 7.30 ->
    // 12.38 ms), while the early start saves it under 5 us.
    const int lane = threadIdx.x;
    const long long base = static_cast<long long>(blockIdx.x) * group_size;
    const float* r = rewards + base;
    float mn = INFINITY, mx = -INFINITY;
    double sum = 0.0;
    for (int i = lane; i < group_size; i += 32) {
        const float v = r[i];
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
        sum += static_cast<double>(v);
    }
    mn = warp_min_f32(mn);
    mx = warp_max_f32(mx);
    sum = warp_sum_f64(sum);
    if (mn == mx) {  // all equal (also a group of one)
        for (int i = lane; i < group_size; i += 32) adv[base + i] = 0.0f;
        return;
    }
    const double mean = sum / group_size;
    double ss = 0.0;
    for (int i = lane; i < group_size; i += 32) {
        const double d = static_cast<double>(r[i]) - mean;
        ss += d * d;
    }
    ss = warp_sum_f64(ss);
    const double denom = sqrt(ss / (group_size - 1)) + static_cast<double>(eps);
    // Each lane reads and writes only its own indices, so adv may alias rewards.
    for (int i = lane; i < group_size; i += 32) {
        const double d = static_cast<double>(r[i]) - mean;
        adv[base + i] = static_cast<float>(normalize_std ? d / denom : d);
    }
}

// Valid tokens per response: rows of one response are mostly consecutive, so
// the lanes of a warp that share a response index add their count once.
__global__ void response_count_kernel(const int32_t* row_response, long long T, int n_resp, int32_t* counts) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long t0 = static_cast<long long>(blockIdx.x) * blockDim.x; t0 < T; t0 += stride) {
        const long long t = t0 + threadIdx.x;
        const int r = t < T ? row_response[t] : -1;
        const bool valid = r >= 0 && r < n_resp;
        const unsigned active = __ballot_sync(0xFFFFFFFFu, valid);
        if (valid) {
            const unsigned same = __match_any_sync(active, r);
            const int lane = threadIdx.x & 31;
            if ((same & ((1u << lane) - 1u)) == 0u) atomicAdd(counts + r, __popc(same));
        }
    }
}

__global__ void rollout_mean_kernel(const float* adv, const int32_t* counts, int n_resp, float* out) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r < n_resp) {
        const int c = counts[r];
        out[r] = c > 0 ? adv[r] / static_cast<float>(c) : 0.0f;
    }
}

// The batch loss: grad_scale * sum of the rows' token losses (the first field
// of each 64-byte diagnostics record), the docs' global generated-token
// reduction when grad_scale = 1 / N_tokens.  One CTA, so the order of the
// additions is fixed: thread i sums rows i, i + 512, ... in FP64, then a
// pairwise tree over the 512 partial sums; one rounding to FP32 at the end.
constexpr int kLossThreads = 512;
__global__ void __launch_bounds__(kLossThreads) batch_loss_kernel(const float* diag_words, long long T,
                                                                  float grad_scale, float* out) {
    __shared__ double part[kLossThreads];
    double s = 0.0;
    for (long long t = threadIdx.x; t < T; t += kLossThreads) s += static_cast<double>(diag_words[16 * t]);
    part[threadIdx.x] = s;
    __syncthreads();
    for (int h = kLossThreads / 2; h > 0; h >>= 1) {
        if (static_cast<int>(threadIdx.x) < h) part[threadIdx.x] += part[threadIdx.x + h];
        __syncthreads();
    }
    if (threadIdx.x == 0) *out = static_cast<float>(static_cast<double>(grad_scale) * part[0]);
}

}  // namespace
}  // namespace sc

extern "C" int sc_batch_loss(const sc_row_diag* diag, long long T, float grad_scale, float* loss_out,
                             sc_stream_t stream) {
    using namespace sc;
    if (T < 0) return fail(SC_ERR_SHAPE, "T = %lld < 0", T);
    if (!loss_out) return fail(SC_ERR_NULL, "loss_out is NULL");
    if (T > 0 && !diag) return fail(SC_ERR_NULL, "diag is NULL with T > 0");
    if (!std::isfinite(grad_scale)) return fail(SC_ERR_ARG, "grad_scale must be finite");
    if (!aligned(diag, 16) || !aligned(loss_out, 4))
        return fail(SC_ERR_ALIGN, "diag must be 16-byte aligned, loss_out 4-byte aligned");
    int dev = 0;
    int st = check_device(&dev);
    if (st != SC_OK) return st;
    batch_loss_kernel<<<1, kLossThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const float*>(diag), T, grad_scale, loss_out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "batch_loss_kernel launch");
    return ok();
}

extern "C" int sc_group_advantages(const float* rewards, int n_groups, int group_size,
                                   int normalize_std, float eps, float* adv_out, sc_stream_t stream) {
    using namespace sc;
    if (n_groups < 0) return fail(SC_ERR_SHAPE, "n_groups = %d < 0", n_groups);
    if (group_size < 1 || group_size > 65536)
        return fail(SC_ERR_SHAPE, "group_size = %d outside 1..65536", group_size);
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return fail(SC_ERR_ARG, "eps must be finite and >= 0");
    if (n_groups == 0) return ok();
    if (!rewards || !adv_out) return fail(SC_ERR_NULL, "rewards or adv_out is NULL");
    if (!aligned(rewards, 4) || !aligned(adv_out, 4))
        return fail(SC_ERR_ALIGN, "rewards and adv_out must be 4-byte aligned");
    const char* r0 = reinterpret_cast<const char*>(rewards);
    const char* a0 = reinterpret_cast<const char*>(adv_out);
    const long long bytes = 4LL * n_groups * group_size;
    if (r0 != a0 && r0 < a0 + bytes && a0 < r0 + bytes)
        return fail(SC_ERR_ARG, "adv_out partially overlaps rewards");
    int dev = 0;
    int st = check_device(&dev);
    if (st != SC_OK) return st;
    group_adv_kernel<<<n_groups, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        rewards, group_size, normalize_std ? 1 : 0, eps, adv_out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "group_adv_kernel launch");
    return ok();
}

extern "C" int sc_rollout_mean_advantages(const float* adv, const int32_t* row_response, long long T, int n_resp,
                                          int32_t* counts_out, float* adv_out, sc_stream_t stream) {
    using namespace sc;
    if (T < 0) return fail(SC_ERR_SHAPE, "T = %lld < 0", T);
    if (n_resp < 0) return fail(SC_ERR_SHAPE, "n_resp = %d < 0", n_resp);
    if (n_resp == 0) return ok();
    if (!adv || !counts_out || !adv_out) return fail(SC_ERR_NULL, "adv, counts_out and adv_out are required");
    if (T > 0 && !row_response) return fail(SC_ERR_NULL, "row_response is NULL with T > 0");
    if (!aligned(adv, 4) || !aligned(row_response, 4) || !aligned(counts_out, 4) || !aligned(adv_out, 4))
        return fail(SC_ERR_ALIGN, "arrays must be 4-byte aligned");
    int dev = 0;
    int st = check_device(&dev);
    if (st != SC_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(counts_out, 0, sizeof(int32_t) * static_cast<size_t>(n_resp), s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(counts)");
    if (T > 0) {
        const long long want = (T + 255) / 256;
        const int blocks = static_cast<int>(want < 1024 ? want : 1024);
        response_count_kernel<<<blocks, 256, 0, s>>>(row_response, T, n_resp, counts_out);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "response_count_kernel launch");
    }
    rollout_mean_kernel<<<(n_resp + 255) / 256, 256, 0, s>>>(adv, counts_out, n_resp, adv_out);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "rollout_mean_kernel launch");
    return ok();
}
