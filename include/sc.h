/*
 * sc.h -- C ABI of the GB300 (sm_103a) score-centering library.
 *
 * Score centering is the correction of the Agent Lightning docs page "Score
 * Centering", section "Score Centering": for every generated position the
 * sampler records its top-K candidate ids with their log-probabilities; the
 * trainer scores the current policy p over the full vocabulary at the rollout
 * temperature and minimises the token loss
 *
 *     -sg(A) * [ log p_a - sum_{v in H} sg(q_v - rho p_v) log p_v ],
 *     rho = max(1 - Q_H, 1e-6) / max(1 - P_H, 1e-6),
 *     P_H = sum_{v in H} p_v,  Q_H = sum_{v in H} q_v,
 *
 * whose gradient with respect to the raw logits z (x = z / T) is
 *
 *     g_v = grad_scale * (1/T) * (-A) * ( [v == a] - mu_hat_v ),
 *     mu_hat_v = s p_v + [v in H] (q_v - rho p_v),   s = 1 - Q_H + rho P_H,
 *
 * i.e. the recorded head keeps the sampler's probabilities and the
 * unrecorded tail is taken proportional to the current policy.
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller.  The library
 *     allocates no memory at run time.  It keeps a small per-process cache of
 *     launch plans and one 256-byte static device array per GPU, which only
 *     sc_center_forward_backward_noalloc uses.  The fused call takes a small
 *     caller-owned workspace (see SC_WORKSPACE_BYTES).
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     Argument errors are detected on the host before anything is launched
 *     and returned as a status code; nothing is written in that case.
 *   - Data errors found while the kernel runs (bad ids, bad counts, a wait
 *     that ran out) are reported per row in the diagnostics' `flags` and,
 *     OR-ed together, in the optional device status word, which the caller
 *     reads after synchronising the stream.
 *   - bf16 values travel as their raw 16-bit patterns (uint16_t).
 *   - Entry points are thread-safe; calls that share output buffers and run
 *     concurrently on different streams race on those buffers.
 */
#ifndef SC_H
#define SC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* sc_stream_t;

/* ---- status codes ---------------------------------------------------- */
#define SC_OK 0
#define SC_ERR_NULL 1        /* a required pointer is NULL                     */
#define SC_ERR_ALIGN 2       /* a pointer or row stride breaks its alignment   */
#define SC_ERR_SHAPE 3       /* a size is out of the supported range           */
#define SC_ERR_ARG 4         /* a parameter value is invalid                   */
#define SC_ERR_CUDA 5        /* the CUDA runtime reported an error             */
#define SC_ERR_UNSUPPORTED 6 /* the current device cannot run this library     */

/* ---- device status word bits (OR-ed by the kernels) ------------------- */
#define SC_STATUS_DATA 0x1u             /* some row carried a data-error flag    */
#define SC_STATUS_TIMEOUT_LOAD 0x2u     /* a bulk-copy wait ran out (about 1 s)  */
#define SC_STATUS_TIMEOUT_EXCHANGE 0x4u /* a cluster exchange wait ran out       */

/* ---- per-row flag bits (sc_row_diag.flags) ---------------------------- */
#define SC_FLAG_MASKED 0x1u        /* padding row: row_response < 0             */
#define SC_FLAG_BAD_ID 0x2u        /* a recorded id outside [0, V) was ignored   */
#define SC_FLAG_DUP_ID 0x4u        /* a repeated recorded id was ignored         */
#define SC_FLAG_BAD_SAMPLED 0x8u   /* sampled id outside [0, V): row zeroed      */
#define SC_FLAG_BAD_COUNT 0x10u    /* rec_count outside [0, K_max]: clamped      */
#define SC_FLAG_BAD_RESPONSE 0x20u /* row_response >= n_resp: row zeroed         */
#define SC_FLAG_CLAMP_PI 0x40u     /* 1 - P_H < 1e-6: denominator clamped        */
#define SC_FLAG_CLAMP_MU 0x80u     /* 1 - Q_H < 1e-6: numerator clamped          */
#define SC_FLAG_IS_TRUNC 0x100u    /* tis: weight truncated at tis_max           */
#define SC_FLAG_IS_REJECT 0x200u   /* mis: weight outside [mis_min, mis_max]     */
#define SC_FLAG_CLIPPED 0x400u     /* clip: the clipped term is the minimum       */
#define SC_FLAG_DATA_ERRORS (SC_FLAG_BAD_ID | SC_FLAG_DUP_ID | SC_FLAG_BAD_SAMPLED | \
                             SC_FLAG_BAD_COUNT | SC_FLAG_BAD_RESPONSE)

/* Importance weighting modes: the `is_mode` setting (none / tis / mis) of the
 * settings table in the docs' "Score Centering" section.  w = exp(log p_a -
 * rollout logprob).  tis weights the token by min(w, tis_max); mis weights it
 * by w inside [mis_min, mis_max] and by 0 outside.
 * SC_IS_CLIP is the clipped GRPO baseline of the page's "Training" section
 * (`grpo` preset): token loss -min(w A, clamp(w, 1 - clip_low, 1 + clip_high) A)
 * with rollout_logprob holding the old policy's log-probability; the gradient
 * is the policy gradient weighted by w where the unclipped term is the
 * minimum and 0 where the clipped one is (SC_FLAG_CLIPPED).  It requires
 * centering = 0.  Its per-rollout mean loss comes from the advantages of
 * sc_rollout_mean_advantages. */
#define SC_IS_NONE 0
#define SC_IS_TIS 1
#define SC_IS_MIS 2
#define SC_IS_CLIP 3

/* Parameters of sc_center_forward_backward.  Defaults (sc_params_default):
 * the docs' settings table -- K = 128, is_mode none, tis_max 2.0,
 * mis_min 0.5, mis_max 5.0, centering on -- at temperature 1, scale 1, and
 * the `grpo` preset's clip widths 0.2 / 0.3. */
typedef struct sc_params {
    int K_max;             /* row length of rec_ids / rec_logprobs, 0..1024     */
    int is_mode;           /* SC_IS_NONE, SC_IS_TIS, SC_IS_MIS or SC_IS_CLIP     */
    float tis_max;         /* > 0                                               */
    float mis_min;         /* 0 <= mis_min <= mis_max                            */
    float mis_max;
    int centering;         /* 1: score centering; 0: plain (weighted) score      */
    float inv_temperature; /* 1 / rollout temperature, finite, > 0               */
    float grad_scale;      /* multiplies every gradient element, e.g. 1 / N_tok */
    int cluster_size;      /* CTAs sharing one row: 0 = automatic, else 1..16   */
    int threads;           /* streaming threads per CTA (plus three warps: row
                              scalars, bulk copies, zero rows):
                              0 = automatic, else 128, 256, 384 or 512          */
    int stages;            /* rows in flight per CTA: 0 = automatic, else 1..4   */
    float clip_low;        /* SC_IS_CLIP: ratio floor 1 - clip_low, 0 <= low < 1 */
    float clip_high;       /* SC_IS_CLIP: ratio ceiling 1 + clip_high, >= 0      */
    int flag_layout;       /* how a CTA marks the recorded ids of its slice in
                              shared memory: 0 = automatic, SC_FLAGS_ENTRY or
                              SC_FLAGS_VECTOR                                   */
    int wait_limit_us;     /* how long any wait inside the kernel (a bulk copy,
                              a peer's record, a hand-off between its warps)
                              may take before the launch gives up and sets
                              SC_STATUS_TIMEOUT_*: 0 = 1 s, else 1..60000000 us.
                              The final wait for bulk copies in flight before
                              a CTA exits always allows 1 s.                    */
    int test_stall;        /* test hook, 0 in normal use.  1: every CTA leaves
                              out the bulk copy of the first chunk of its first
                              row, so the waits for it run out: the launch ends
                              early with SC_STATUS_TIMEOUT_LOAD and its outputs
                              are incomplete, with no fault and the context
                              usable.  It exercises the failure path.           */
} sc_params;

/* Recorded-id flag layouts (sc_params.flag_layout).  SC_FLAGS_ENTRY keeps one
 * bit per vocabulary entry of the slice: the fastest lookup.  SC_FLAGS_VECTOR
 * keeps one bit per 8-entry vector plus, for the few flagged vectors, their
 * 8-bit entry masks in vector order behind a per-word count of the flags
 * before it: 15-20 KB less shared memory per CTA at the large vocabularies,
 * so that a smaller cluster still fits two CTAs to an SM, for two more
 * dependent shared-memory loads on a flagged vector.  The automatic choice
 * takes, under each layout, the smallest cluster whose CTAs fit two to an SM
 * and keeps the one with more CTAs resident on the GPU (SC_FLAGS_ENTRY on a
 * tie). */
#define SC_FLAGS_ENTRY 1
#define SC_FLAGS_VECTOR 2

/* Per-row diagnostics, 64 bytes.  Masked and error rows hold zeros and their
 * flags.  loss is the unscaled token loss; the batch loss whose gradient is
 * grad_out is grad_scale * sum(loss). */
typedef struct sc_row_diag {
    float loss;        /* -A_w [log p_a - sum_H c_v log p_v]                    */
    float logp_a;      /* log p_a (same as logp_out)                            */
    float P_H;         /* current mass on the recorded ids                      */
    float tail_pi;     /* 1 - P_H, accumulated directly over the unrecorded ids */
    float Q_H;         /* recorded (sampler) mass                               */
    float tail_mu;     /* 1 - Q_H                                               */
    float rho;         /* max(1-Q_H,1e-6) / max(1-P_H,1e-6)                     */
    float s;           /* 1 - Q_H + rho P_H (1 when centering is off)           */
    float entropy;     /* -sum p log p                                          */
    float k3;          /* exp(d) - 1 - d, d = log p_a - rollout logprob         */
    float is_weight;   /* importance weight applied to A (1 for none)           */
    float row_sum;     /* sum of the row's FP32 gradient before bf16 rounding   */
    float adv;         /* the row's advantage A before the importance weight    */
    int32_t n_valid_k; /* recorded ids used                                     */
    uint32_t flags;    /* SC_FLAG_* bits                                        */
    uint32_t reserved;
} sc_row_diag;

/*
 * The batch loss of a fused call: grad_scale * sum_t diag[t].loss, the docs'
 * global generated-token reduction ("Score Centering" page, section
 * "Training": the loss summed over every generated token of the batch and
 * divided by their number) when grad_scale = 1 / N_tokens.  Its gradient with
 * respect to the logits is the grad_out of the same call.
 *
 * diag     : sc_row_diag [T] written by sc_center_forward_backward (device,
 *            16-byte aligned); masked and error rows hold loss 0.
 * loss_out : one FP32 value (device), written.
 * The sum runs in one fixed order (FP64 partial sums over rows t = i mod 512,
 * then a pairwise tree), rounded to FP32 once, so repeated calls give the
 * same bits.  T == 0 writes 0.  Asynchronous on `stream`.
 * Errors: SC_ERR_SHAPE (T < 0), SC_ERR_NULL, SC_ERR_ARG (grad_scale not
 * finite), SC_ERR_ALIGN, SC_ERR_UNSUPPORTED, SC_ERR_CUDA.
 */
int sc_batch_loss(const sc_row_diag* diag, long long T, float grad_scale, float* loss_out, sc_stream_t stream);

/*
 * Sampler-side capture of the top K behaviour probabilities (docs page
 * "Score Centering", section "Score Centering": each generated position
 * records the top K probabilities of the sampling call, with their original
 * normalisation).  The behaviour distribution is mu = softmax(z * inv_t)
 * over the V sampler logits, or, with top_p < 1, that distribution
 * restricted to its nucleus -- the shortest prefix of the entries sorted by
 * probability whose preceding mass is below top_p -- and renormalised.
 * Entries are ordered by z, larger first, equal values by lower id.
 *
 * logits       : FP32 [T, logits_stride] sampler logits (device), 16-byte
 *                aligned, logits_stride % 4 == 0, >= V; each row holds at
 *                least one finite value (-inf entries carry no mass).
 * ids_out      : int32 [T, K] the recorded ids, row t at t * K; entries past
 *                the row's count hold -1.
 * logprobs_out : FP32 [T, K] log mu of those ids (0 past the count).
 * count_out    : int32 [T] min(K, V, nucleus size), or NULL.
 * workspace    : SC_WORKSPACE_BYTES of device memory, 16-byte aligned, zero
 *                before its first use, or NULL.  With it, the rows after each
 *                thread group's first are handed out at run time from a
 *                counter there (rows whose nucleus reaches far below the top
 *                entries cost more passes, and the groups that drew them take
 *                fewer rows); the launch leaves it zero again when it
 *                completes.  It may be the workspace of the fused call on the
 *                same stream (the two use different words of it).  NULL: every
 *                row dealt at launch.
 * K            : 1..1024.  inv_temperature finite > 0.  top_p in (0, 1].
 * Asynchronous on `stream`; nothing is allocated.  Every sum is taken in a
 * fixed order (on the one-pass path that almost every row takes, FP32 sums of
 * 24 terms added to a compensated FP32 sum per thread; 2^-40 fixed point where
 * the nucleus reaches below the top entries and on the exact path), so the
 * results do not depend on how the rows are scheduled; log mu is within
 * 2e-6 (1 + |log mu|) of its FP64 value.
 * Errors: SC_ERR_SHAPE (T < 0, V outside 1..2^24, K, stride), SC_ERR_ARG,
 * SC_ERR_NULL, SC_ERR_ALIGN, SC_ERR_UNSUPPORTED, SC_ERR_CUDA.
 */
int sc_topk_capture(const float* logits, long long T, int V, long long logits_stride, float inv_temperature,
                    int K, float top_p, int32_t* ids_out, float* logprobs_out, int32_t* count_out,
                    void* workspace, sc_stream_t stream);

/* Fills *p with the defaults above.  Returns SC_OK or SC_ERR_NULL. */
int sc_params_default(sc_params* p);

/*
 * GRPO group advantages (docs "Score Centering" page, section "Training":
 * rollout-level advantages with group standard-deviation normalisation; the
 * devotd.net release note, section 4: rewards stay fractional, no overflow in
 * the denominator, and the paper's mean-only variant).
 *
 *   A_i = (r_i - mean_g) / (std_g + eps)   (normalize_std = 1)
 *   A_i =  r_i - mean_g                    (normalize_std = 0)
 *
 * rewards : FP32 [n_groups * group_size], group-major (group g holds
 *           rewards[g*group_size .. (g+1)*group_size)).
 * adv_out : FP32 [n_groups * group_size]; may alias rewards exactly.
 * std is the unbiased (n - 1) sample std, computed in FP64 with two passes;
 * a group whose rewards are all equal (including a group of one) gets
 * exactly 0.  n_groups == 0 is a no-op.
 * Errors: SC_ERR_NULL (pointer NULL with n_groups > 0), SC_ERR_SHAPE
 * (n_groups < 0, group_size < 1 or > 65536), SC_ERR_ARG (eps negative or
 * not finite, partial overlap), SC_ERR_ALIGN (pointer not 4-byte aligned),
 * SC_ERR_UNSUPPORTED, SC_ERR_CUDA.
 */
int sc_group_advantages(const float* rewards, int n_groups, int group_size, int normalize_std,
                        float eps, float* adv_out, sc_stream_t stream);

/*
 * Per-rollout mean loss (the `grpo` preset of the docs page's "Training"
 * section): each response's advantage divided by its number of valid tokens,
 * so that grad_scale = 1 / n_resp then averages per-rollout token means.
 *
 * adv          : FP32 [n_resp] advantages (device).
 * row_response : int32 [T] response index of each row; rows with an index
 *                outside [0, n_resp) count for no response.
 * counts_out   : int32 [n_resp] valid tokens per response (device, written).
 * adv_out      : FP32 [n_resp] adv[r] / counts[r], 0 where counts[r] == 0;
 *                may equal adv.
 * Asynchronous on `stream` (two kernels and a memset; nothing allocated).
 * Errors: SC_ERR_NULL, SC_ERR_SHAPE (T or n_resp negative), SC_ERR_ALIGN,
 * SC_ERR_UNSUPPORTED, SC_ERR_CUDA.
 */
int sc_rollout_mean_advantages(const float* adv, const int32_t* row_response, long long T, int n_resp,
                               int32_t* counts_out, float* adv_out, sc_stream_t stream);

/*
 * Score-centered forward and backward over T token rows (docs "Score
 * Centering" page, section "Score Centering"; one fused kernel).
 *
 * logits          : bf16 [T, logits_stride], the first V entries of each row
 *                   are the trainer's raw logits; 16-byte aligned,
 *                   logits_stride % 8 == 0, logits_stride >= V.  Any
 *                   values: -inf entries carry no mass (a NaN makes the
 *                   row's results NaN).
 * rec_ids         : int32 [T, K_max] recorded candidate ids (top-K of the
 *                   sampler); entries past rec_count[t] are ignored.
 * rec_logprobs    : FP32 [T, K_max] their sampler log-probabilities, in
 *                   their original normalisation (their sum may be below 1).
 * rec_count       : int32 [T] number of recorded ids per row, or NULL for
 *                   K_max everywhere.
 * sampled_id      : int32 [T] the sampled token a (may lie outside H).
 * rollout_logprob : FP32 [T] the sampler's own log-probability of a, or
 *                   NULL (then k3 = 0; is_mode must be SC_IS_NONE).
 * row_response    : int32 [T] response index of each row, -1 for padding.
 * adv             : FP32 [n_resp] the responses' advantages A.
 * grad_out        : bf16 [T, grad_stride], written for every row (zeros for
 *                   padding and error rows), round-to-nearest-even; 16-byte
 *                   aligned, grad_stride % 8 == 0.  May equal `logits` (in
 *                   place) when grad_stride == logits_stride; any other
 *                   overlap is rejected.  Entries past V are not touched.
 * logp_out        : FP32 [T] log p_a (0 for padding and error rows).
 * diag_out        : sc_row_diag [T] or NULL.
 * status_dev      : one device uint32 or NULL; SC_STATUS_* bits are OR-ed
 *                   into it (the caller clears it).
 * workspace       : SC_WORKSPACE_BYTES of device memory, 16-byte aligned,
 *                   all zero before its first use.  It holds the counter from
 *                   which the launch hands rows out to its thread-block
 *                   clusters at run time (the clusters that run ahead take
 *                   more rows), and the launch leaves it zero again when it
 *                   completes, so consecutive calls on one stream can share
 *                   one workspace.  Calls that may run at the same time (other
 *                   streams) need workspaces of their own; after a launch that
 *                   did not complete (a CUDA error), zero it again.
 * Recorded ids outside [0, V) are ignored, and a repeated id is ignored
 * after its first occurrence; both set row flags.
 * Errors: SC_ERR_NULL, SC_ERR_ALIGN, SC_ERR_SHAPE (T < 0, V < 1,
 * V > 1048576, K_max outside 0..1024, n_resp < 0, strides < V), SC_ERR_ARG
 * (bad parameter values or overlap), SC_ERR_UNSUPPORTED, SC_ERR_CUDA.
 * T == 0 is a no-op (the workspace is not touched).
 */
#define SC_WORKSPACE_BYTES 64
int sc_center_forward_backward(const uint16_t* logits, long long T, int V, long long logits_stride,
                               const int32_t* rec_ids, const float* rec_logprobs,
                               const int32_t* rec_count, const int32_t* sampled_id,
                               const float* rollout_logprob, const int32_t* row_response,
                               const float* adv, int n_resp, const sc_params* p, uint16_t* grad_out,
                               long long grad_stride, float* logp_out, sc_row_diag* diag_out,
                               uint32_t* status_dev, void* workspace, sc_stream_t stream);

/*
 * The same call for callers that cannot allocate device memory.  (The docs
 * pages have no counterpart: this is a property of the library, not of the
 * method.)
 *
 * Some callers receive their input and output buffers and nothing else -- a
 * plugin inside another framework whose memory planner has already placed
 * every buffer, or an embedded runtime that reserves all of its device memory
 * up front -- so they cannot provide the workspace above.  This entry point
 * takes the same arguments as sc_center_forward_backward except the
 * workspace, and computes the same outputs.  It allocates nothing: its
 * workspace is a fixed 256-byte array inside the library, held in device
 * memory on every GPU that loads the library until the process exits.
 *   - The first call on a device looks up that array's device address on
 *     the current device (cudaGetSymbolAddress); make that first call before
 *     any stream capture.
 *   - Every call clears the workspace on `stream` before its launch, so a
 *     failed earlier call does not leave it dirty.
 *   - All calls share the one array: calls whose launches may overlap on the
 *     GPU (different streams without ordering between them) race on it and
 *     give wrong results.  Serialise them, or use sc_center_forward_backward
 *     with a workspace per stream.
 *   - The workspace a call needs does not depend on T, V or K_max; a call
 *     would be refused (SC_ERR_SHAPE) only if SC_WORKSPACE_BYTES exceeded the
 *     array's 256 bytes.
 * Errors: as sc_center_forward_backward; on an argument error nothing but the
 * library's own array is written.
 */
int sc_center_forward_backward_noalloc(const uint16_t* logits, long long T, int V, long long logits_stride,
                                       const int32_t* rec_ids, const float* rec_logprobs,
                                       const int32_t* rec_count, const int32_t* sampled_id,
                                       const float* rollout_logprob, const int32_t* row_response,
                                       const float* adv, int n_resp, const sc_params* p, uint16_t* grad_out,
                                       long long grad_stride, float* logp_out, sc_row_diag* diag_out,
                                       uint32_t* status_dev, sc_stream_t stream);

/*
 * The LM head followed by score centering, in row blocks (the next step of
 * the path: the trainer's logits come from its LM head, z = H W^T).
 *
 * hidden      : bf16 [T, d] hidden states H, rows contiguous (d % 8 == 0),
 *               16-byte aligned.
 * w           : bf16 [V, d] the LM head W, 16-byte aligned.
 * rec_ids ... p : as sc_center_forward_backward, for the T rows.
 * block_rows  : rows per block; only one [block_rows, V] block of logits is
 *               ever held (in the workspace).
 * dhidden     : bf16 [T, d], written: dH = g W, g the score-centered gradient
 *               of grad_scale * sum(loss) with respect to z.
 * dw          : FP32 [V, d], written (not accumulated across calls):
 *               dW = g^T H.
 * logp_out, diag_out, status_dev : as sc_center_forward_backward.
 * workspace   : sc_lmhead_workspace_bytes(block_rows, V, d) bytes of device
 *               memory, 256-byte aligned; its first SC_WORKSPACE_BYTES must
 *               be zero before the first call (they are left zero, as for
 *               sc_center_forward_backward).  It holds the block of logits
 *               (bf16 [block_rows, V rounded up to 8]) and, when dH's
 *               output tiles are too few for the SMs (block_rows / 128 x
 *               d / 256 tiles), FP32 slices of dH's partial products over
 *               parts of the vocabulary, summed in a fixed order.  Its size
 *               depends on the current device's SM count.  Calls that may run
 *               at the same time need workspaces of their own.
 * Per block: z_b = H_b W^T (sc_gemm_bf16: FP32 accumulation, bf16 logits),
 * the fused score-centering kernel in place, dH_b = g_b W and dW (+)= g_b^T
 * H_b (sc_gemm_bf16, FP32 accumulation; dW stored by the first block and
 * added to by the others); all asynchronous on `stream`.
 * Errors: as sc_center_forward_backward, plus SC_ERR_SHAPE (d not a multiple
 * of 8, block_rows < 1, workspace too small).  T == 0 is a no-op.
 */
/*
 * Dense bf16 GEMM on the tensor cores: the LM head's three products
 * (z = H W^T, dH = g W, dW = g^T H) run on it.
 *
 *     C[M, N] = A[M, K] . B[K, N]    (FP32 accumulation)
 *
 * A       : bf16, a_layout 0: stored [M][K] (K contiguous, row stride lda);
 *           a_layout 1: stored [K][M] (M contiguous, row stride lda).
 * B       : bf16, b_layout 0: stored [N][K] (row stride ldb); b_layout 1:
 *           stored [K][N].
 * C       : row-major [M][N], row stride ldc; c_mode SC_GEMM_BF16 writes bf16
 *           (round to nearest even), SC_GEMM_FP32 writes FP32, SC_GEMM_FP32_ADD
 *           adds the FP32 product to what C holds.
 * All pointers device, 16-byte aligned; row strides multiples of 16 bytes
 * and at least the row length.  Sizes 1..2^31.  status_dev (nullable): a
 * device word into which SC_STATUS_TIMEOUT_LOAD is OR-ed if a wait inside
 * the kernel ran out.  Asynchronous on `stream`; nothing is allocated.
 * Errors: SC_ERR_NULL, SC_ERR_ALIGN, SC_ERR_SHAPE, SC_ERR_ARG,
 * SC_ERR_UNSUPPORTED, SC_ERR_CUDA.
 */
#define SC_GEMM_BF16 0
#define SC_GEMM_FP32 1
#define SC_GEMM_FP32_ADD 2
int sc_gemm_bf16(const uint16_t* A, long long lda, int a_layout, const uint16_t* B, long long ldb, int b_layout,
                 void* C, long long ldc, int c_mode, long long M, long long N, long long K, uint32_t* status_dev,
                 sc_stream_t stream);

size_t sc_lmhead_workspace_bytes(long long block_rows, int V, int d);
int sc_lmhead_forward_backward(const uint16_t* hidden, const uint16_t* w, long long T, int d, int V,
                               const int32_t* rec_ids, const float* rec_logprobs, const int32_t* rec_count,
                               const int32_t* sampled_id, const float* rollout_logprob,
                               const int32_t* row_response, const float* adv, int n_resp, const sc_params* p,
                               long long block_rows, uint16_t* dhidden, float* dw, float* logp_out,
                               sc_row_diag* diag_out, uint32_t* status_dev, void* workspace,
                               size_t workspace_bytes, sc_stream_t stream);

/* Launch plan the library would use for a vocabulary of V and these
 * parameters on the current device (no launch).  Any output pointer may be
 * NULL.  cluster_size: CTAs per row; threads: per CTA; slice: vocabulary
 * entries per CTA; smem_bytes: dynamic shared memory per CTA;
 * max_clusters: clusters resident at once (the persistent grid size);
 * flag_layout: SC_FLAGS_ENTRY or SC_FLAGS_VECTOR.
 * Errors: as sc_center_forward_backward for V, K_max and p. */
int sc_plan_query(int V, const sc_params* p, int* cluster_size, int* threads, int* slice,
                  int* smem_bytes, int* max_clusters, int* flag_layout);

/* Short text for a status code. */
const char* sc_status_string(int status);

/* Text of the last error returned on this thread ("" if none). */
const char* sc_last_error(void);

/* ABI version: 100 * major + minor. */
int sc_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SC_H */
