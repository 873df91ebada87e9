// sc_lmhead.cu -- the LM head followed by score centering, over row blocks.
//
// The trainer's logits are z = H W^T (H [T, d] hidden states, W [V, d] the LM
// head, both bf16; the products accumulated in FP32 and the logits rounded to
// bf16, as a BF16 trainer holds them).  Score centering (the Agent Lightning
// docs page "Score Centering", section "Score Centering") gives the gradient g
// of the batch loss with respect to z; z's linearity then gives
//     dH = g W,   dW = g^T H.
// The full [T, V] logits are never held: the rows go through in blocks of
// block_rows, each block
//   1. z_b = H_b W^T          tensor-core GEMM (sc_gemm.cu), FP32 accumulate -> bf16
//   2. g_b from z_b           the fused score-centering kernel, in place
//   3. dH_b = g_b W           tensor-core GEMM, W read N-major, -> bf16 (K = V
//                             split into FP32 slices summed in a fixed order
//                             when the output tiles are too few for the SMs)
//   4. dW  (+)= g_b^T H_b     tensor-core GEMM, g read M-major, FP32 (stored by
//                             block 0, added by the tensor-store engine after)
// all on the caller's stream, so only one [block_rows, V] buffer is needed.
// Every step is this library's own kernel.
#include <cmath>
#include <cstring>

#include "sc_internal.h"

namespace sc {
namespace {

constexpr size_t kScHeader = 256;  // the fused kernel's workspace (SC_WORKSPACE_BYTES), padded

inline size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }
inline long long row_stride_for(int V) { return (static_cast<long long>(V) + 7) / 8 * 8; }

}  // namespace
}  // namespace sc

namespace sc {
namespace {

// K splits of the dH = g W product for blocks of n rows (its n/128 x d/256
// output tiles are few next to the SMs): the count that fills whole waves
// best on the current device (148 SMs assumed without one).
int dh_splits(long long n, int d, int V) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
        (void)cudaGetLastError();  // (no device here: a size query only)
        sms = 148;
    }
    return best_k_splits(n, d, V, sms);
}

// FP32 rows the workspace holds for the split dH of blocks of Tb rows.
long long dh_acc_rows(long long Tb, int d, int V) {
    const int s = dh_splits(Tb, d, V);
    return s > 1 ? s * split_slice_rows(Tb) : 0;
}

}  // namespace
}  // namespace sc

extern "C" size_t sc_lmhead_workspace_bytes(long long block_rows, int V, int d) {
    using namespace sc;
    if (block_rows < 1 || V < 1 || d < 1) return 0;
    const size_t acc = static_cast<size_t>(dh_acc_rows(block_rows, d, V)) * static_cast<size_t>(d) * 4;
    return kScHeader + round_up(static_cast<size_t>(block_rows) * row_stride_for(V) * 2, 256) + round_up(acc, 256);
}

extern "C" int sc_lmhead_forward_backward(const uint16_t* hidden, const uint16_t* w, long long T, int d, int V,
                                          const int32_t* rec_ids, const float* rec_logprobs, const int32_t* rec_count,
                                          const int32_t* sampled_id, const float* rollout_logprob,
                                          const int32_t* row_response, const float* adv, int n_resp,
                                          const sc_params* p, long long block_rows, uint16_t* dhidden, float* dw,
                                          float* logp_out, sc_row_diag* diag_out, uint32_t* status_dev,
                                          void* workspace, size_t workspace_bytes, sc_stream_t stream) {
    using namespace sc;
    if (!p) return fail(SC_ERR_NULL, "params is NULL");
    if (T < 0) return fail(SC_ERR_SHAPE, "T = %lld < 0", T);
    if (d < 8 || d % 8 != 0 || d > (1 << 20)) return fail(SC_ERR_SHAPE, "d = %d must be a multiple of 8 in 8..2^20", d);
    if (V < 1 || V > (1 << 20)) return fail(SC_ERR_SHAPE, "V = %d outside 1..2^20", V);
    if (block_rows < 1) return fail(SC_ERR_SHAPE, "block_rows = %lld < 1", block_rows);
    {   // the score-centering parameters and V, checked before anything is launched
        const int pst = sc_plan_query(V, p, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
        if (pst != SC_OK && pst != SC_ERR_CUDA && pst != SC_ERR_UNSUPPORTED) return pst;
    }
    if (T == 0) return ok();
    if (!hidden || !w || !dhidden || !dw || !workspace || !sampled_id || !row_response || !logp_out)
        return fail(SC_ERR_NULL, "hidden, w, dhidden, dw, workspace, sampled_id, row_response and logp_out are required");
    if (n_resp > 0 && !adv) return fail(SC_ERR_NULL, "adv is NULL with n_resp > 0");
    if (p->K_max > 0 && (!rec_ids || !rec_logprobs))
        return fail(SC_ERR_NULL, "rec_ids and rec_logprobs are required when K_max > 0");
    if (p->is_mode != SC_IS_NONE && !rollout_logprob)
        return fail(SC_ERR_NULL, "is_mode tis/mis/clip needs rollout_logprob");
    if (!aligned(hidden, 16) || !aligned(w, 16) || !aligned(dhidden, 16) || !aligned(dw, 16) ||
        !aligned(workspace, 256))
        return fail(SC_ERR_ALIGN, "hidden, w, dhidden and dw must be 16-byte aligned, workspace 256-byte aligned");
    const long long Tb = block_rows < T ? block_rows : T;
    if (workspace_bytes < sc_lmhead_workspace_bytes(Tb, V, d))
        return fail(SC_ERR_SHAPE, "workspace holds %zu bytes, %zu needed", workspace_bytes,
                    sc_lmhead_workspace_bytes(Tb, V, d));
    int dev = 0;
    int st = check_device(&dev);
    if (st != SC_OK) return st;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    void* sc_ws = ws;
    uint16_t* zbuf = reinterpret_cast<uint16_t*>(ws + kScHeader);
    const long long Vs = row_stride_for(V);
    float* acc = reinterpret_cast<float*>(ws + kScHeader + round_up(static_cast<size_t>(Tb) * Vs * 2, 256));
    const long long acc_rows = dh_acc_rows(Tb, d, V);
    const int K = p->K_max;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (long long t0 = 0; t0 < T; t0 += Tb) {
        const long long n = T - t0 < Tb ? T - t0 : Tb;
        const uint16_t* Hb = hidden + t0 * d;
        // 1. z_b [n x V] = H_b [n x d] . W^T: both operands K-major; consecutive
        //    tiles share W's tile (read once from HBM per block)
        st = gemm_bf16(Hb, d, 0, w, d, 0, zbuf, Vs, 0, n, V, d, 1, status_dev, s, 1);
        if (st != SC_OK) return st;
        // 2. the score-centered gradient of the block, in place
        st = sc_center_forward_backward(zbuf, n, V, Vs, K ? rec_ids + t0 * K : nullptr,
                                        K ? rec_logprobs + t0 * K : nullptr, rec_count ? rec_count + t0 : nullptr,
                                        sampled_id + t0, rollout_logprob ? rollout_logprob + t0 : nullptr,
                                        row_response + t0, adv, n_resp, p, zbuf, Vs, logp_out + t0,
                                        diag_out ? diag_out + t0 : nullptr, status_dev, sc_ws, stream);
        if (st != SC_OK) return st;
        // 3. dH_b [n x d] = g_b [n x V] . W [V x d]: W read N-major; K = V split
        //    when the n/128 x d/256 output tiles would leave SMs idle
        int splits = dh_splits(n, d, V);  // (a shorter last block: as many as its slices fit)
        if (splits > 1 && splits * split_slice_rows(n) > acc_rows)
            splits = static_cast<int>(acc_rows / split_slice_rows(n));
        st = gemm_bf16_split(zbuf, Vs, 0, w, d, 1, dhidden + t0 * d, d, acc, d, n, d, V, 1, splits > 1 ? splits : 1,
                             status_dev, s);
        if (st != SC_OK) return st;
        // 4. dW [V x d] (+)= g_b^T [V x n] . H_b [n x d]: g read M-major, H_b N-major;
        //    consecutive tiles share g's tile
        st = gemm_bf16(zbuf, Vs, 1, Hb, d, 1, dw, d, t0 == 0 ? 1 : 2, V, d, n, 0, status_dev, s, 1);
        if (st != SC_OK) return st;
    }
    return ok();
}
