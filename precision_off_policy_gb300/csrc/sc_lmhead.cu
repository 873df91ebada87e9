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
//   1. z_b = H_b W^T          cuBLASLt, bf16 x bf16 -> FP32 accumulate -> bf16
//   2. g_b from z_b           the fused score-centering kernel, in place
//   3. dH_b = g_b W           cuBLASLt, -> bf16
//   4. dW  += g_b^T H_b       cuBLASLt, FP32 accumulator (overwritten by block 0)
// all on the caller's stream, so only one [block_rows, V] buffer is needed.
// The matrix products are plain dense GEMMs on the tensor cores (cuBLASLt's
// kernels); every other step is this library's own kernel.
#include <cublasLt.h>

#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "sc_internal.h"

namespace sc {
namespace {

constexpr size_t kLtWorkspace = size_t(32) << 20;  // cuBLASLt's scratch, taken from the caller's workspace
constexpr size_t kScHeader = 256;                   // the fused kernel's workspace (SC_WORKSPACE_BYTES), padded

inline size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }
inline long long row_stride_for(int V) { return (static_cast<long long>(V) + 7) / 8 * 8; }

int lt_fail(cublasStatus_t s, const char* what) {
    return fail(SC_ERR_CUDA, "%s: cuBLASLt status %d", what, static_cast<int>(s));
}

// One GEMM shape (column-major, as cuBLASLt sees the row-major operands).
struct GemmKey {
    int dev;
    int ta, tb;                      // transposes of A and B
    long long m, n, k, lda, ldb, ldc;
    int ctype;                       // 0: bf16 output, 1: FP32 output
    bool operator<(const GemmKey& o) const {
        return std::tie(dev, ta, tb, m, n, k, lda, ldb, ldc, ctype) <
               std::tie(o.dev, o.ta, o.tb, o.m, o.n, o.k, o.lda, o.ldb, o.ldc, o.ctype);
    }
};
struct GemmPlan {
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t a = nullptr, b = nullptr, c = nullptr;
    cublasLtMatmulAlgo_t algo;
};

std::mutex g_lt_mutex;
std::map<int, cublasLtHandle_t> g_lt_handle;
std::map<GemmKey, GemmPlan> g_gemm_plans;

int lt_handle(int dev, cublasLtHandle_t* out) {
    auto it = g_lt_handle.find(dev);
    if (it == g_lt_handle.end()) {
        cublasLtHandle_t h = nullptr;
        const cublasStatus_t s = cublasLtCreate(&h);
        if (s != CUBLAS_STATUS_SUCCESS) return lt_fail(s, "cublasLtCreate");
        it = g_lt_handle.emplace(dev, h).first;
    }
    *out = it->second;
    return SC_OK;
}

int gemm_plan(const GemmKey& key, cublasLtHandle_t h, const GemmPlan** out) {
    auto it = g_gemm_plans.find(key);
    if (it != g_gemm_plans.end()) {
        *out = &it->second;
        return SC_OK;
    }
    GemmPlan P;
    cublasStatus_t s = cublasLtMatmulDescCreate(&P.op, CUBLAS_COMPUTE_32F, CUDA_R_32F);
    if (s != CUBLAS_STATUS_SUCCESS) return lt_fail(s, "cublasLtMatmulDescCreate");
    const cublasOperation_t ta = key.ta ? CUBLAS_OP_T : CUBLAS_OP_N, tb = key.tb ? CUBLAS_OP_T : CUBLAS_OP_N;
    cublasLtMatmulDescSetAttribute(P.op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof ta);
    cublasLtMatmulDescSetAttribute(P.op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof tb);
    const long long ar = key.ta ? key.k : key.m, ac = key.ta ? key.m : key.k;
    const long long br = key.tb ? key.n : key.k, bc = key.tb ? key.k : key.n;
    const cudaDataType_t ct = key.ctype ? CUDA_R_32F : CUDA_R_16BF;
    if ((s = cublasLtMatrixLayoutCreate(&P.a, CUDA_R_16BF, ar, ac, key.lda)) != CUBLAS_STATUS_SUCCESS ||
        (s = cublasLtMatrixLayoutCreate(&P.b, CUDA_R_16BF, br, bc, key.ldb)) != CUBLAS_STATUS_SUCCESS ||
        (s = cublasLtMatrixLayoutCreate(&P.c, ct, key.m, key.n, key.ldc)) != CUBLAS_STATUS_SUCCESS)
        return lt_fail(s, "cublasLtMatrixLayoutCreate");
    cublasLtMatmulPreference_t pref = nullptr;
    if ((s = cublasLtMatmulPreferenceCreate(&pref)) != CUBLAS_STATUS_SUCCESS)
        return lt_fail(s, "cublasLtMatmulPreferenceCreate");
    const size_t ws = kLtWorkspace;
    cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws, sizeof ws);
    cublasLtMatmulHeuristicResult_t res;
    int found = 0;
    s = cublasLtMatmulAlgoGetHeuristic(h, P.op, P.a, P.b, P.c, P.c, pref, 1, &res, &found);
    cublasLtMatmulPreferenceDestroy(pref);
    if (s != CUBLAS_STATUS_SUCCESS) return lt_fail(s, "cublasLtMatmulAlgoGetHeuristic");
    if (found < 1) return fail(SC_ERR_UNSUPPORTED, "cuBLASLt has no algorithm for a %lld x %lld x %lld GEMM",
                               key.m, key.n, key.k);
    P.algo = res.algo;
    *out = &g_gemm_plans.emplace(key, P).first->second;
    return SC_OK;
}

int gemm(int dev, cublasLtHandle_t h, int ta, int tb, long long m, long long n, long long k, const void* A,
         long long lda, const void* B, long long ldb, void* C, long long ldc, int ctype, float beta, void* lt_ws,
         cudaStream_t stream) {
    const GemmPlan* P = nullptr;
    const int st = gemm_plan(GemmKey{dev, ta, tb, m, n, k, lda, ldb, ldc, ctype}, h, &P);
    if (st != SC_OK) return st;
    const float alpha = 1.0f;
    const cublasStatus_t s = cublasLtMatmul(h, P->op, &alpha, A, P->a, B, P->b, &beta, C, P->c, C, P->c, &P->algo,
                                            lt_ws, kLtWorkspace, stream);
    if (s != CUBLAS_STATUS_SUCCESS) return lt_fail(s, "cublasLtMatmul");
    return SC_OK;
}

}  // namespace
}  // namespace sc

extern "C" size_t sc_lmhead_workspace_bytes(long long block_rows, int V) {
    using namespace sc;
    if (block_rows < 1 || V < 1) return 0;
    return kScHeader + kLtWorkspace + round_up(static_cast<size_t>(block_rows) * row_stride_for(V) * 2, 256);
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
    if (workspace_bytes < sc_lmhead_workspace_bytes(Tb, V))
        return fail(SC_ERR_SHAPE, "workspace holds %zu bytes, %zu needed", workspace_bytes,
                    sc_lmhead_workspace_bytes(Tb, V));
    int dev = 0;
    int st = check_device(&dev);
    if (st != SC_OK) return st;
    cublasLtHandle_t h = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_lt_mutex);
        st = lt_handle(dev, &h);
    }
    if (st != SC_OK) return st;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    void* sc_ws = ws;
    void* lt_ws = ws + kScHeader;
    uint16_t* zbuf = reinterpret_cast<uint16_t*>(ws + kScHeader + kLtWorkspace);
    const long long Vs = row_stride_for(V);
    const int K = p->K_max;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (long long t0 = 0; t0 < T; t0 += Tb) {
        const long long n = T - t0 < Tb ? T - t0 : Tb;
        const uint16_t* Hb = hidden + t0 * d;
        // 1. z_b^T [V x n] = W [V x d] . H_b^T: column-major A = W^T (d x V) transposed, B = H_b^T (d x n)
        {
            std::lock_guard<std::mutex> lock(g_lt_mutex);
            st = gemm(dev, h, 1, 0, V, n, d, w, d, Hb, d, zbuf, Vs, 0, 0.0f, lt_ws, s);
        }
        if (st != SC_OK) return st;
        // 2. the score-centered gradient of the block, in place
        st = sc_center_forward_backward(zbuf, n, V, Vs, K ? rec_ids + t0 * K : nullptr,
                                        K ? rec_logprobs + t0 * K : nullptr, rec_count ? rec_count + t0 : nullptr,
                                        sampled_id + t0, rollout_logprob ? rollout_logprob + t0 : nullptr,
                                        row_response + t0, adv, n_resp, p, zbuf, Vs, logp_out + t0,
                                        diag_out ? diag_out + t0 : nullptr, status_dev, sc_ws, stream);
        if (st != SC_OK) return st;
        {
            std::lock_guard<std::mutex> lock(g_lt_mutex);
            // 3. dH_b^T [d x n] = W^T (d x V) . g_b^T (V x n)
            st = gemm(dev, h, 0, 0, d, n, V, w, d, zbuf, Vs, dhidden + t0 * d, d, 0, 0.0f, lt_ws, s);
            // 4. dW^T [d x V] (+)= H_b^T (d x n) . g_b (n x V)
            if (st == SC_OK)
                st = gemm(dev, h, 0, 1, d, V, n, Hb, d, zbuf, Vs, dw, d, 1, t0 == 0 ? 0.0f : 1.0f, lt_ws, s);
        }
        if (st != SC_OK) return st;
    }
    return ok();
}
