// sc_center.cu -- fused score-centered forward/backward over [T, V] bf16 logits.
//
// Implements the token loss of the Agent Lightning docs page "Score
// Centering", section "Score Centering":
//   P_H = sum_H p_v,  Q_H = sum_H q_v,  rho = max(1-Q_H,1e-6)/max(1-P_H,1e-6),
//   loss = -sg(A) [log p_a - sum_H sg(q_v - rho p_v) log p_v],
// and its gradient with respect to the raw logits,
//   g_v = scale (1/T) (-A) ([v==a] - mu_hat_v),
//   mu_hat_v = s p_v + [v in H](q_v - rho p_v),  s = 1 - Q_H + rho P_H,
// plus log p_a and per-row diagnostics (the section's K3, entropy, masses).
//
// GB300 design.  One row is shared by a cluster of C CTAs; CTA r owns the
// vocabulary slice [r*S, min((r+1)*S, V)).  Each CTA is warp-specialised.
//
// * The producer warp walks the cluster's rows ahead of the consumers.  Per
//   row it fills a slot of a small metadata ring: the row's scalars and, for
//   valid rows, the compact list of recorded ids that fall in this CTA's
//   slice (repeats dropped, q = exp(logprob) precomputed) with a bitmap of the
//   16-byte vectors that hold them.  It then starts 1-D bulk copies (TMA
//   engine) of the logit slice into the data stage, 4 KiB chunk by chunk, each
//   as soon as the previous row's write pass has released that chunk.
// * The consumer warps, per row of the ring:
//   0. padding / error rows: write the zero gradient slice and move on;
//   1. max pass on packed bf16 pairs as chunks land, while consumer warp 0
//      reads the owned recorded ids' logits and overwrites them in shared
//      memory with -2^100 (the max is exact either way: warp 0 contributes
//      the values it overwrites);
//   2. warp 0 reduces the owned recorded ids (mass, entropy term, sum of
//      q y, the recorded mass as an error-free FP32 pair with its largest
//      term apart) while all warps run the exp pass: the unrecorded mass
//      sum_{v not in H} e^{x_v - m} accumulates directly (no 1 - P_H
//      cancellation), with the entropy term;
//   3. exchange: each CTA sends one 64-byte record to every CTA of the
//      cluster with st.async stores that complete as transaction bytes on the
//      receiver's mbarrier; warp 0 merges the C records into the row scalars
//      (LSE, P_H, Q_H, rho, s, loss, k3, importance weight) in O(C), the same
//      way in every CTA;
//   4. write pass: p_v is recomputed from shared memory and g_v = beta p_v
//      streams to global memory with 16-byte stores and an evict-first L2
//      hint; the <= K+1 special entries (recorded ids and the sampled token)
//      are patched in registers via the per-vector bitmap.
// Every logit is read from HBM once and every gradient written once.  The
// grid is persistent (as many clusters as fit).  Every wait is bounded
// (about 1 s) and reports through the status word.
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "sc_device.cuh"
#include "sc_internal.h"

namespace sc {
namespace {

constexpr int kMaxCluster = 16;
constexpr int kMaxChunks = 16;
constexpr int kMaxStages = 4;             // data stages
constexpr int kMaxMeta = kMaxStages + 1;  // metadata ring slots
constexpr int kMaxK = 1024;
constexpr int kMaxV = 1 << 20;
constexpr int kMaxSmem = 232448;          // 227 KiB of dynamic shared memory per CTA
constexpr int kChunkVecTarget = 256;      // 16-byte vectors per bulk copy (4 KiB)
constexpr uint16_t kSentinel = 0xF180u;   // bf16 -2^100: marks recorded ids in shared memory
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kTailFloor = 1e-6f;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;
constexpr uint32_t kFull = 0xFFFFFFFFu;

// One row as the producer hands it to the consumers.
struct RowMeta {
    long long t;      // row index; -1 ends the consumers' loop
    uint32_t zflags;  // nonzero: padding or error row (zero gradient)
    int sa;           // sampled id
    int nown;         // recorded ids of this CTA's slice in the compact list
    int a_li;         // local index of a in this slice, -1 if another CTA owns it
    uint32_t flags;   // row flags found by the producer (count, repeats, out of range)
    float A, rl;      // advantage, rollout logprob
    int pad[3];
};
static_assert(sizeof(RowMeta) == 48, "RowMeta layout");

// One CTA's contribution to a row, exchanged across the cluster (64 bytes).
// y' values are relative to this CTA's own slice maximum m (y' = (z - m) kscale).
struct Partial {
    float m;            // slice maximum of z (-inf for an empty slice)
    float S1, S2;       // unrecorded entries: sum 2^y', sum 2^y' y'
    float rs;           // FP32 gradient sum of this slice for the previous valid row
    float lH, EH;       // recorded ids owned here: sum 2^y', sum 2^y' y'
    float QY;           // sum q_k y'_k over the owned recorded ids
    float qo_hi, qo_lo; // sum of q_k over them except the largest one (double-float)
    float qbest;        // the largest q_k owned here (0 if none)
    int kbest;          // its position k (INT_MAX if none)
    int nval;           // owned recorded ids used
    uint32_t flags;     // row flags found by this CTA's producer
    float ya;           // y' of the sampled token, if this CTA owns it
    int has_a;
    float omq;          // 1 - qbest, from its log-probability (-expm1)
};
static_assert(sizeof(Partial) == 64, "partial record is 64 bytes");

struct Layout {
    int stage_bytes;  // bytes of one data stage (128-aligned)
    int list_cap;     // entries of one owned list (K_max)
    int nwords;       // bitmap words of one slice
    int off_meta, off_list_li, off_list_lp, off_list_k, off_bitmap, off_bars, off_part, off_mine, off_frs,
        off_fixz, off_fixv, off_red, off_scal, total;
};

struct KArgs {
    const uint16_t* logits;
    const int32_t* ids;
    const float* lps;
    const int32_t* cnt;
    const int32_t* sampled;
    const float* rollout;
    const int32_t* resp;
    const float* adv;
    uint16_t* grad;
    float* logp;
    sc_row_diag* diag;
    uint32_t* status;
    long long T, lstride, gstride;
    int V, K_max, n_resp;
    int is_mode, centering;
    float tis_max, mis_min, mis_max, inv_t, grad_scale;
    int C, S, ncv, NB, MS;
    Layout L;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
__device__ __forceinline__ uint16_t f_to_bf_bits(float x) {
    return static_cast<uint16_t>(pack_bf16x2(x, 0.0f) & 0xFFFFu);
}
__device__ __forceinline__ void status_or(uint32_t* st, uint32_t bits) {
    if (st) atomicOr(st, bits);
}

// Largest recorded probability with the mass of the others, merged
// commutatively (ties go to the lower k) so a butterfly gives every lane the
// same bits.  The others' mass is kept as an unevaluated FP32 pair.
struct HeadMass {
    float q;
    int k;
    float omq;  // 1 - q of the winner, accurate near q = 1
    float oh, ol;
};
__device__ __forceinline__ HeadMass head_merge(const HeadMass& a, const HeadMass& b) {
    const bool b_wins = b.q > a.q || (b.q == a.q && b.k < a.k);
    HeadMass r;
    r.q = b_wins ? b.q : a.q;
    r.k = b_wins ? b.k : a.k;
    r.omq = b_wins ? b.omq : a.omq;
    const float lq = b_wins ? a.q : b.q;
    float s, e;
    two_sum(a.oh, b.oh, s, e);
    const float ol = (a.ol + b.ol) + e;
    float s2, e2;
    two_sum(s, lq, s2, e2);
    r.oh = s2;
    r.ol = ol + e2;
    return r;
}
__device__ __forceinline__ HeadMass head_shfl(const HeadMass& h, int off) {
    HeadMass o;
    o.q = __shfl_xor_sync(kFull, h.q, off);
    o.k = __shfl_xor_sync(kFull, h.k, off);
    o.omq = __shfl_xor_sync(kFull, h.omq, off);
    o.oh = __shfl_xor_sync(kFull, h.oh, off);
    o.ol = __shfl_xor_sync(kFull, h.ol, off);
    return o;
}

// Barriers.  Data stage d: kChunkFull + i (copy of chunk i landed, tx bytes),
// kChunkFree + i (every consumer warp is done with chunk i).  Meta slot s:
// kMetaFull (producer wrote it), kMetaFree (consumers are done with it).
constexpr int kChunkFull = 0;
constexpr int kChunkFree = kMaxChunks;
constexpr int kBarsPerStage = 2 * kMaxChunks;
constexpr int kMetaBase = kMaxStages * kBarsPerStage;
constexpr int kMetaFull = 0;
constexpr int kMetaFree = 1;
constexpr int kXBase = kMetaBase + 2 * kMaxMeta;
constexpr int kNumBars = kXBase + 2;

// Resident CTAs per SM the register allocation must allow (shared memory
// allows about this many at the automatic plan's slice sizes).
constexpr int min_blocks(int NC) { return NC <= 128 ? 6 : (NC <= 256 ? 4 : (NC <= 384 ? 3 : 2)); }

template <int NC>
__global__ void __launch_bounds__(NC + 32, min_blocks(NC)) center_kernel(const __grid_constant__ KArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int NCW = NC / 32;  // consumer warps; warp NCW is the producer
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t crank = cluster_ctarank();
    const uint32_t cid = cluster_id_x();
    const uint32_t ncl = num_clusters_x();
    const int C = a.C, K_max = a.K_max, NB = a.NB, MS = a.MS;
    const Layout& L = a.L;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.off_bars);
    RowMeta* meta = reinterpret_cast<RowMeta*>(smem + L.off_meta);         // [MS]
    int* list_li = reinterpret_cast<int*>(smem + L.off_list_li);           // [MS][list_cap]
    float* list_lp = reinterpret_cast<float*>(smem + L.off_list_lp);       // [MS][list_cap]
    int* list_k = reinterpret_cast<int*>(smem + L.off_list_k);             // [MS][list_cap]
    uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem + L.off_bitmap);   // [MS][nwords]
    Partial* part = reinterpret_cast<Partial*>(smem + L.off_part);         // [2][C]
    Partial* mine = reinterpret_cast<Partial*>(smem + L.off_mine);         // staging of this CTA's record
    float2* frs = reinterpret_cast<float2*>(smem + L.off_frs);             // [kMaxCluster]
    float* fix_z = reinterpret_cast<float*>(smem + L.off_fixz);            // [list_cap]
    float* fix_v = reinterpret_cast<float*>(smem + L.off_fixv);            // [list_cap]
    float* red = reinterpret_cast<float*>(smem + L.off_red);               // [4][NCW]
    float* scal = reinterpret_cast<float*>(smem + L.off_scal);             // [8]
    int* scal_i = reinterpret_cast<int*>(scal);
    auto data_bar = [&](int d, int i) { return smem_addr(&bars[d * kBarsPerStage + i]); };
    auto meta_bar = [&](int s, int i) { return smem_addr(&bars[kMetaBase + 2 * s + i]); };
    const uint32_t xbar0 = smem_addr(&bars[kXBase]);

    const int lo = static_cast<int>(crank) * a.S;
    const int hi = min(lo + a.S, a.V);
    const int n = max(hi - lo, 0);
    const int n8 = n & ~7, nvb = n8 >> 3, tail = n - n8, nv = nvb + (tail ? 1 : 0);
    const int nchunks = (nvb + a.ncv - 1) / a.ncv;
    const int cap = L.list_cap, nwords = L.nwords;
    const float kscale = a.inv_t * kLog2e;
    const uint64_t pol = l2_policy_evict_first();     // last use: gradient stores, write-pass reads
    const uint64_t pol_keep = l2_policy_evict_last(); // slice copies, read again by the write pass

    if (tid == 0) {
        for (int d = 0; d < NB; ++d)
            for (int i = 0; i < kMaxChunks; ++i) {
                mbar_init(data_bar(d, kChunkFull + i), 1u);
                mbar_init(data_bar(d, kChunkFree + i), static_cast<uint32_t>(NCW));
            }
        for (int s = 0; s < MS; ++s) {
            mbar_init(meta_bar(s, kMetaFull), 1u);
            mbar_init(meta_bar(s, kMetaFree), 1u);
        }
        mbar_init(xbar0, 1u);  // exchange: own expect_tx arrive + peers' st.async bytes
        mbar_init(xbar0 + 8, 1u);
        fence_mbar_init_cluster();
    }
    for (int i = tid; i < MS * nwords; i += NC + 32) bitmap[i] = 0u;
    cluster_sync_all();  // every CTA's barriers exist before peers signal them

    long long t_last = -1;  // consumers: last valid row (for the final row sum)
    float rs_last = 0.0f;   // consumer thread 0: this CTA's share of its sum
    bool aborted = false;

    if (warp == NCW) {
        // ================= producer warp =================
        uint32_t nmeta = 0, ndata = 0;
        bool stop = false;
        for (long long base = cid; base < a.T && !stop; base += 32LL * ncl) {
            const long long tl = base + static_cast<long long>(lane) * ncl;
            const bool in = tl < a.T;
            int resp_l = -1, sa_l = 0;
            if (in) {
                resp_l = __ldg(a.resp + tl);
                sa_l = __ldg(a.sampled + tl);
            }
            uint32_t zf = 0;
            if (in) {
                if (resp_l < 0)
                    zf = SC_FLAG_MASKED;
                else if (resp_l >= a.n_resp)
                    zf = SC_FLAG_BAD_RESPONSE;
                else if (sa_l < 0 || sa_l >= a.V)
                    zf = SC_FLAG_BAD_SAMPLED;
            }
            const unsigned inmask = __ballot_sync(kFull, in);
            for (int j = 0; j < 32 && ((inmask >> j) & 1u); ++j) {
                const long long t = base + static_cast<long long>(j) * ncl;
                const uint32_t zfj = __shfl_sync(kFull, zf, j);
                const int rj = __shfl_sync(kFull, resp_l, j);
                const int sj = __shfl_sync(kFull, sa_l, j);
                const int ms = static_cast<int>(nmeta % MS);
                if (nmeta >= static_cast<uint32_t>(MS) &&
                    !mbar_wait_bounded(meta_bar(ms, kMetaFree), ((nmeta / MS) - 1u) & 1u, kWaitLimitNs)) {
                    if (lane == 0) status_or(a.status, SC_STATUS_TIMEOUT_LOAD);
                    stop = true;
                    break;
                }
                RowMeta* mt = meta + ms;
                if (zfj) {  // padding or error row: the consumers write zeros
                    if (lane == 0) {
                        mt->t = t;
                        mt->zflags = zfj;
                        mt->sa = sj;
                        mt->nown = 0;
                        mt->a_li = -1;
                        mt->flags = 0;
                        mt->A = 0.0f;
                        mt->rl = 0.0f;
                        mbar_arrive(meta_bar(ms, kMetaFull));
                    }
                    ++nmeta;
                    continue;
                }
                // ---- recorded ids of this slice: compact list, repeats dropped ----
                // (row scalars loaded first so their latency overlaps the list)
                const float row_A = __ldg(a.adv + rj);
                const float row_rl = a.rollout ? __ldg(a.rollout + t) : 0.0f;
                int cnt = a.cnt ? __ldg(a.cnt + t) : K_max;
                uint32_t flags = 0;
                if (cnt < 0 || cnt > K_max) {
                    flags |= SC_FLAG_BAD_COUNT;
                    cnt = cnt < 0 ? 0 : K_max;
                }
                int* li_s = list_li + ms * cap;
                float* lp_s = list_lp + ms * cap;
                int* k_s = list_k + ms * cap;
                uint32_t* bm = bitmap + ms * nwords;
                for (int w = lane; w < nwords; w += 32) bm[w] = 0u;  // the slot's previous bits
                __syncwarp();
                const long long kb = t * static_cast<long long>(K_max);
                int nown = 0;
                bool bad = false, dup = false;
                for (int kb0 = 0; kb0 < cnt; kb0 += 128) {
                    int idr[4];
                    float lpr[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {  // four rounds of loads in flight together
                        const int k = kb0 + 32 * r + lane;
                        idr[r] = k < cnt ? __ldg(a.ids + kb + k) : -1;
                        lpr[r] = k < cnt ? __ldg(a.lps + kb + k) : 0.0f;
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int k = kb0 + 32 * r + lane;
                        const bool kin = k < cnt;
                        const int id = idr[r];
                        bad = bad || (kin && (id < 0 || id >= a.V));
                        const bool owned = kin && id >= lo && id < hi;
                        const unsigned same = __match_any_sync(kFull, owned ? id : -1 - lane);
                        bool keep = owned && (same & lanemask_lt()) == 0u;
                        if (keep)  // repeats of an earlier round
                            for (int e = 0; e < nown; ++e)
                                if (li_s[e] == id - lo) {
                                    keep = false;
                                    break;
                                }
                        dup = dup || (owned && !keep);
                        const unsigned km = __ballot_sync(kFull, keep);
                        if (keep) {
                            const int pos = nown + __popc(km & lanemask_lt());
                            li_s[pos] = id - lo;
                            lp_s[pos] = lpr[r];
                            k_s[pos] = k;
                            atomicOr(&bm[(id - lo) >> 8], 1u << (((id - lo) >> 3) & 31));
                        }
                        nown += __popc(km);
                        __syncwarp();
                    }
                }
                if (__any_sync(kFull, dup)) flags |= SC_FLAG_DUP_ID;
                if (crank == 0 && __any_sync(kFull, bad)) flags |= SC_FLAG_BAD_ID;
                const int a_li = (sj >= lo && sj < hi) ? sj - lo : -1;
                if (lane == 0) {
                    if (a_li >= 0) atomicOr(&bm[a_li >> 8], 1u << ((a_li >> 3) & 31));
                    mt->t = t;
                    mt->zflags = 0;
                    mt->sa = sj;
                    mt->nown = nown;
                    mt->a_li = a_li;
                    mt->flags = flags;
                    mt->A = row_A;
                    mt->rl = row_rl;
                }
                // ---- logit slice: chunk by chunk as the stage's slots free up ----
                if (lane == 0) {
                    const int ds = static_cast<int>(ndata % NB);
                    const bool reuse = ndata >= static_cast<uint32_t>(NB);
                    const uint32_t fpar = ((ndata / NB) - 1u) & 1u;
                    uint16_t* bufst = reinterpret_cast<uint16_t*>(smem + ds * L.stage_bytes);
                    const uint16_t* lrow = a.logits + t * a.lstride + lo;
                    const uint32_t bs = smem_addr(bufst);
                    for (int i = 0; i < nchunks; ++i) {
                        if (reuse && !mbar_wait_bounded(data_bar(ds, kChunkFree + i), fpar, kWaitLimitNs)) {
                            status_or(a.status, SC_STATUS_TIMEOUT_LOAD);
                            for (int i2 = 0; i2 < i; ++i2)  // started copies land before the CTA leaves
                                (void)mbar_wait_bounded(data_bar(ds, kChunkFull + i2), (ndata / NB) & 1u,
                                                        kWaitLimitNs);
                            stop = true;
                            break;
                        }
                        fence_proxy_async_smem();
                        const int v0 = i * a.ncv, v1 = min(v0 + a.ncv, nvb);
                        const uint32_t bytes = static_cast<uint32_t>(v1 - v0) * 16u;
                        mbar_expect_tx(data_bar(ds, kChunkFull + i), bytes);
                        bulk_load(bs + 16u * v0, lrow + 8 * v0, bytes, data_bar(ds, kChunkFull + i), pol_keep);
                    }
                }
                stop = __shfl_sync(kFull, static_cast<int>(stop), 0) != 0;
                if (stop) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(meta_bar(ms, kMetaFull));  // release: slot contents
                ++nmeta;
                ++ndata;
            }
        }
        if (!stop) {  // end marker for the consumers
            const int ms = static_cast<int>(nmeta % MS);
            bool ok = true;
            if (nmeta >= static_cast<uint32_t>(MS))
                ok = mbar_wait_bounded(meta_bar(ms, kMetaFree), ((nmeta / MS) - 1u) & 1u, kWaitLimitNs);
            if (ok) {
                if (lane == 0) {
                    meta[ms].t = -1;
                    mbar_arrive(meta_bar(ms, kMetaFull));
                }
            } else if (lane == 0) {
                status_or(a.status, SC_STATUS_TIMEOUT_LOAD);
            }
        }
        // copies still in flight land before the CTA can exit (bounded again)
        if (lane == 0) {
            const uint32_t f0 = ndata > static_cast<uint32_t>(NB) ? ndata - NB : 0u;
            for (uint32_t f = f0; f < ndata; ++f)
                for (int i = 0; i < nchunks; ++i)
                    (void)mbar_wait_bounded(data_bar(f % NB, kChunkFull + i), (f / NB) & 1u, kWaitLimitNs);
        }
        __syncwarp();
    } else {
        // ================= consumer warps =================
        uint32_t nmeta = 0, ndata = 0;
        float rs_prev = 0.0f;
        long long t_prev = -1;
        for (;;) {
            const int ms = static_cast<int>(nmeta % MS);
            const bool got = mbar_wait_bounded(meta_bar(ms, kMetaFull), (nmeta / MS) & 1u, kWaitLimitNs);
            if (named_bar_or(NC, !got)) {
                if (tid == 0) status_or(a.status, SC_STATUS_TIMEOUT_LOAD);
                aborted = true;
                break;
            }
            const RowMeta m = meta[ms];
            if (m.t < 0) break;
            const long long t = m.t;
            uint16_t* grow = a.grad + t * a.gstride + lo;
            if (m.zflags) {  // ---- padding or error row: zero gradient ----
                for (int j = tid; j < nvb; j += NC) st_global_v4_hint(grow + 8 * j, 0u, 0u, 0u, 0u, pol);
                if (tid < tail) grow[n8 + tid] = 0;
                if (crank == 0 && tid == 0) {
                    a.logp[t] = 0.0f;
                    if (a.diag) {  // zeros and the flags, as four 16-byte stores
                        float4* dp = reinterpret_cast<float4*>(a.diag + t);
                        const float4 z4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        dp[0] = z4;
                        dp[1] = z4;
                        dp[2] = z4;
                        dp[3] = make_float4(0.0f, 0.0f, __uint_as_float(m.zflags), 0.0f);
                    }
                    if (m.zflags & SC_FLAG_DATA_ERRORS) status_or(a.status, SC_STATUS_DATA);
                }
                named_bar(NC);  // every consumer is done with the slot
                if (tid == 0) mbar_arrive(meta_bar(ms, kMetaFree));
                ++nmeta;
                continue;
            }
            const int ds = static_cast<int>(ndata % NB);
            const uint32_t fpar = (ndata / NB) & 1u;
            const uint32_t par = ndata & 1u;
            const uint32_t xph = (ndata >> 1) & 1u;
            const uint32_t xb = xbar0 + 8u * par;
            uint16_t* buf = reinterpret_cast<uint16_t*>(smem + ds * L.stage_bytes);
            const uint32_t buf_s = smem_addr(buf);
            const int* li_s = list_li + ms * cap;
            const float* lp_s = list_lp + ms * cap;
            const int* k_s = list_k + ms * cap;
            const uint32_t* bm = bitmap + ms * nwords;
            const int nown = m.nown;

            // ---- 1. max pass (warps 1..) and owned recorded ids (warp 0) -------
            float m_loc = -INFINITY;
            bool timed_out = false;
            float zav = 0.0f;  // warp 0: z of the sampled token if owned here
            if (warp == 0) {
                if (tail) {  // entries past the last whole vector, padded with the sentinel
                    const uint16_t* lrow = a.logits + t * a.lstride + lo;
                    if (lane < 8) buf[n8 + lane] = lane < tail ? lrow[n8 + lane] : kSentinel;
                    __syncwarp();
                }
                for (int i = 0; i < nchunks && !timed_out; ++i)
                    timed_out = !mbar_wait_bounded(data_bar(ds, kChunkFull + i), fpar, kWaitLimitNs);
                timed_out = __any_sync(kFull, timed_out);
                if (!timed_out) {
                    if (lane < tail) m_loc = bf_to_f(buf[n8 + lane]);
                    if (m.a_li >= 0) zav = bf_to_f(buf[m.a_li]);  // before any entry is overwritten
                    __syncwarp();
                    for (int e = lane; e < nown; e += 32) {
                        const int li = li_s[e];
                        const float z = bf_to_f(buf[li]);
                        fix_z[e] = z;
                        m_loc = fmaxf(m_loc, z);
                        buf[li] = kSentinel;
                    }
                    // bytes this CTA receives for the row: one record from every CTA
                    if (lane == 0) mbar_expect_tx(xb, static_cast<uint32_t>(sizeof(Partial)) * C);
                }
            } else {
                uint32_t mx2 = 0xFF80FF80u;  // (-inf, -inf)
                for (int i = 0; i < nchunks && !timed_out; ++i) {
                    const int v0 = i * a.ncv, v1 = min(v0 + a.ncv, nvb);
                    if (!mbar_wait_bounded(data_bar(ds, kChunkFull + i), fpar, kWaitLimitNs)) {
                        timed_out = true;
                        break;
                    }
#pragma unroll 4
                    for (int j = v0 + tid - 32; j < v1; j += NC - 32) {
                        const uint4 w = lds128(buf_s + 16u * j);
                        mx2 = bmax2(mx2, bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w)));
                    }
                }
                m_loc = fmaxf(bf_lo(mx2), bf_hi(mx2));
            }
            m_loc = warp_max(m_loc);
            if (lane == 0) red[warp] = m_loc;
            if (named_bar_or(NC, timed_out)) {
                if (tid == 0) status_or(a.status, SC_STATUS_TIMEOUT_LOAD);
                aborted = true;
                break;
            }
            m_loc = red[0];
#pragma unroll
            for (int w = 1; w < NCW; ++w) m_loc = fmaxf(m_loc, red[w]);
            const float o_c = m_loc * kscale;

            // ---- 2. owned recorded ids (warp 0), then the exp pass (all) --------
            if (warp == 0) {
                float lH = 0.0f, EH = 0.0f, QY = 0.0f;
                int nval = 0;
                HeadMass hm{0.0f, 0x7FFFFFFF, 1.0f, 0.0f, 0.0f};
                for (int e = lane; e < nown; e += 32) {
                    const float y = fmaf(fix_z[e], kscale, -o_c);
                    const float ev = ex2(y);
                    lH += ev;
                    EH = fmaf(ev, y, EH);
                    const float lp = lp_s[e];
                    const float q = expf(lp);
                    QY = fmaf(q, y, QY);
                    ++nval;
                    hm = head_merge(hm, HeadMass{q, k_s[e], -expm1f(lp), 0.0f, 0.0f});
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    lH += __shfl_xor_sync(kFull, lH, off);
                    EH += __shfl_xor_sync(kFull, EH, off);
                    QY += __shfl_xor_sync(kFull, QY, off);
                    nval += __shfl_xor_sync(kFull, nval, off);
                    hm = head_merge(hm, head_shfl(hm, off));
                }
                if (lane == 0) {
                    Partial& p = *mine;
                    p.m = m_loc;
                    p.rs = rs_prev;
                    p.lH = lH;
                    p.EH = EH;
                    p.QY = QY;
                    p.qo_hi = hm.oh;
                    p.qo_lo = hm.ol;
                    p.qbest = hm.q;
                    p.kbest = hm.k;
                    p.nval = nval;
                    p.flags = m.flags;
                    p.ya = m.a_li >= 0 ? fmaf(zav, kscale, -o_c) : 0.0f;
                    p.has_a = m.a_li >= 0 ? 1 : 0;
                    p.omq = hm.omq;
                }
            }
            // four independent accumulator pairs keep the FADD/FFMA chains short
            float s1a = 0.0f, s1b = 0.0f, s1c = 0.0f, s1d = 0.0f;
            float s2a = 0.0f, s2b = 0.0f, s2c = 0.0f, s2d = 0.0f;
#pragma unroll 2
            for (int j = tid; j < nv; j += NC) {
                const uint4 w = lds128(buf_s + 16u * j);
                float y0 = fmaf(bf_lo(w.x), kscale, -o_c), y1 = fmaf(bf_hi(w.x), kscale, -o_c);
                float e0 = ex2(y0), e1 = ex2(y1);
                s1a += e0 + e1;
                s2a = fmaf(e0, y0, fmaf(e1, y1, s2a));
                y0 = fmaf(bf_lo(w.y), kscale, -o_c);
                y1 = fmaf(bf_hi(w.y), kscale, -o_c);
                e0 = ex2(y0);
                e1 = ex2(y1);
                s1b += e0 + e1;
                s2b = fmaf(e0, y0, fmaf(e1, y1, s2b));
                y0 = fmaf(bf_lo(w.z), kscale, -o_c);
                y1 = fmaf(bf_hi(w.z), kscale, -o_c);
                e0 = ex2(y0);
                e1 = ex2(y1);
                s1c += e0 + e1;
                s2c = fmaf(e0, y0, fmaf(e1, y1, s2c));
                y0 = fmaf(bf_lo(w.w), kscale, -o_c);
                y1 = fmaf(bf_hi(w.w), kscale, -o_c);
                e0 = ex2(y0);
                e1 = ex2(y1);
                s1d += e0 + e1;
                s2d = fmaf(e0, y0, fmaf(e1, y1, s2d));
            }
            float s1t = (s1a + s1b) + (s1c + s1d);
            float s2t = (s2a + s2b) + (s2c + s2d);
            s1t = warp_sum(s1t);
            s2t = warp_sum(s2t);
            if (lane == 0) {
                red[NCW + warp] = s1t;
                red[2 * NCW + warp] = s2t;
            }
            named_bar(NC);
            // The slice in shared memory has served its two passes: hand it back so
            // the next row streams in during the exchange and the write pass, which
            // reads the logits again from L2.
            if (lane == 0)
                for (int i = 0; i < nchunks; ++i) mbar_arrive(data_bar(ds, kChunkFree + i));

            // ---- 3. cluster exchange and row scalars (warp 0) -------------------
            if (warp == 0) {
                if (lane == 0) {
                    float S1 = 0.0f, S2 = 0.0f;
                    for (int w = 0; w < NCW; ++w) {
                        S1 += red[NCW + w];
                        S2 += red[2 * NCW + w];
                    }
                    mine->S1 = S1;
                    mine->S2 = S2;
                }
                __syncwarp();
                if (lane < C) {  // lane r sends this CTA's record to CTA r
                    const uint32_t src = smem_addr(mine);
                    const uint32_t dst = map_to_rank(smem_addr(part + static_cast<int>(par) * C + crank), lane);
                    const uint32_t rb = map_to_rank(xb, lane);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 v = lds128(src + 16u * q);
                        st_async_v4(dst + 16u * q, v.x, v.y, v.z, v.w, rb);
                    }
                }
                const bool ok = mbar_wait_cluster_bounded(xb, xph, kWaitLimitNs);
                if (!__all_sync(kFull, ok)) {
                    if (lane == 0) {
                        status_or(a.status, SC_STATUS_TIMEOUT_EXCHANGE);
                        scal_i[4] = 1;
                    }
                } else {
                    // lane r < C holds CTA r's record; the others hold neutral values
                    const Partial* pp = part + static_cast<int>(par) * C;
                    const bool have = lane < C;
                    const uint32_t pa = smem_addr(pp + (have ? lane : 0));
                    const uint4 r0 = lds128(pa), r1 = lds128(pa + 16u), r2 = lds128(pa + 32u), r3 = lds128(pa + 48u);
                    struct {
                        float m, S1, S2, lH, EH, QY, qo_hi, qo_lo, qbest, ya, omq;
                        int kbest, nval, has_a;
                        uint32_t flags;
                    } P;
                    P.m = have ? __uint_as_float(r0.x) : -INFINITY;
                    P.S1 = have ? __uint_as_float(r0.y) : 0.0f;
                    P.S2 = have ? __uint_as_float(r0.z) : 0.0f;
                    P.lH = have ? __uint_as_float(r1.x) : 0.0f;
                    P.EH = have ? __uint_as_float(r1.y) : 0.0f;
                    P.QY = have ? __uint_as_float(r1.z) : 0.0f;
                    P.qo_hi = have ? __uint_as_float(r1.w) : 0.0f;
                    P.qo_lo = have ? __uint_as_float(r2.x) : 0.0f;
                    P.qbest = have ? __uint_as_float(r2.y) : 0.0f;
                    P.kbest = have ? static_cast<int>(r2.z) : 0x7FFFFFFF;
                    P.nval = have ? static_cast<int>(r2.w) : 0;
                    P.flags = have ? r3.x : 0u;
                    P.ya = have ? __uint_as_float(r3.y) : 0.0f;
                    P.has_a = have ? static_cast<int>(r3.z) : 0;
                    P.omq = have ? __uint_as_float(r3.w) : 1.0f;
                    const float mg = warp_max(P.m);
                    const float o = mg * kscale;
                    const bool live = P.m > -INFINITY;
                    const float d = live ? P.m * kscale - o : 0.0f;
                    const float f = live ? ex2(d) : 0.0f;
                    float lT = f * P.S1;
                    float ET = f * fmaf(d, P.S1, P.S2);
                    float lH = f * P.lH;
                    float EH = f * fmaf(d, P.lH, P.EH);
                    float QYg = 0.0f;
                    if (P.nval > 0) QYg = fmaf(d, (P.qbest + P.qo_hi) + P.qo_lo, P.QY);
                    float ya = P.has_a ? P.ya + d : 0.0f;
                    int nval = P.nval;
                    uint32_t flags = P.flags;
                    HeadMass hm{P.qbest, P.kbest, P.omq, P.qo_hi, P.qo_lo};
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        lT += __shfl_xor_sync(kFull, lT, off);
                        ET += __shfl_xor_sync(kFull, ET, off);
                        lH += __shfl_xor_sync(kFull, lH, off);
                        EH += __shfl_xor_sync(kFull, EH, off);
                        QYg += __shfl_xor_sync(kFull, QYg, off);
                        ya += __shfl_xor_sync(kFull, ya, off);
                        nval += __shfl_xor_sync(kFull, nval, off);
                        flags |= __shfl_xor_sync(kFull, flags, off);
                        hm = head_merge(hm, head_shfl(hm, off));
                    }
                    // 1 - Q_H without cancellation: (1 - q_max), taken from its
                    // log-probability, minus the others' mass
                    float tail_mu = 1.0f, Q_H = 0.0f;
                    if (nval > 0) {
                        tail_mu = (hm.omq - hm.oh) - hm.ol;
                        Q_H = (hm.q + hm.oh) + hm.ol;
                    }
                    const float l = lT + lH;
                    const float log2l = log2f(l);
                    const float P_H = lH / l;
                    const float tail_pi = lT / l;
                    const float rho = fmaxf(tail_mu, kTailFloor) / fmaxf(tail_pi, kTailFloor);
                    if (tail_pi < kTailFloor) flags |= SC_FLAG_CLAMP_PI;
                    if (tail_mu < kTailFloor) flags |= SC_FLAG_CLAMP_MU;
                    const float s = a.centering ? tail_mu + rho * P_H : 1.0f;
                    const float dsr = a.centering ? tail_mu - rho * tail_pi : 0.0f;  // s - rho
                    const float logp_a = (ya - log2l) * kLn2;
                    float wt = 1.0f, k3 = 0.0f;
                    if (a.rollout) {
                        const float dd = logp_a - m.rl;
                        k3 = expm1f(dd) - dd;
                        const float w = expf(dd);
                        if (a.is_mode == SC_IS_TIS) {
                            if (w > a.tis_max) {
                                wt = a.tis_max;
                                flags |= SC_FLAG_IS_TRUNC;
                            } else {
                                wt = w;
                            }
                        } else if (a.is_mode == SC_IS_MIS) {
                            if (w >= a.mis_min && w <= a.mis_max) {
                                wt = w;
                            } else {
                                wt = 0.0f;
                                flags |= SC_FLAG_IS_REJECT;
                            }
                        }
                    }
                    const float A = m.A;
                    const float Aw = A * wt;
                    // sum_H c log p = sum_H q log p - rho sum_H p log p, each from the
                    // merged sums: log p_k = (y_k - log2 l) ln 2.
                    float csum = 0.0f;
                    if (a.centering && nval > 0) {
                        const float qlogp = kLn2 * fmaf(-log2l, Q_H, QYg);
                        const float plogp = kLn2 * fmaf(-log2l, lH, EH) / l;
                        csum = fmaf(-rho, plogp, qlogp);
                    }
                    const float loss = -Aw * (logp_a - csum);
                    const float entropy = kLn2 * (log2l - (ET + EH) / l);
                    const float alpha = -a.grad_scale * a.inv_t * Aw;
                    const float beta = -alpha * s;
                    for (int e = lane; e < nown; e += 32) {  // gradient at the owned recorded ids
                        const float p = ex2(fmaf(fix_z[e], kscale, -o) - log2l);
                        const float mu = a.centering ? fmaf(dsr, p, expf(lp_s[e])) : p;
                        fix_v[e] = alpha * ((li_s[e] == m.a_li ? 1.0f : 0.0f) - mu);
                    }
                    if (lane == 0) {
                        scal[0] = o + log2l;
                        scal[1] = beta;
                        scal[2] = alpha * (1.0f - s * ex2(ya - log2l));  // g_a when a is unrecorded
                        scal_i[4] = 0;
                        if (crank == 0) {
                            a.logp[t] = logp_a;
                            if (a.diag) {  // the record in field order, as four 16-byte stores
                                float4* dp = reinterpret_cast<float4*>(a.diag + t);
                                dp[0] = make_float4(loss, logp_a, P_H, tail_pi);
                                dp[1] = make_float4(Q_H, tail_mu, rho, s);
                                dp[2] = make_float4(entropy, k3, wt, 0.0f);
                                dp[3] = make_float4(A, __int_as_float(nval), __uint_as_float(flags), 0.0f);
                                if (t_prev >= 0) {  // the previous row's sum rode in with this exchange
                                    float rsum = 0.0f;
                                    for (int r = 0; r < C; ++r) rsum += pp[r].rs;
                                    a.diag[t_prev].row_sum = rsum;
                                }
                            }
                            if (flags & SC_FLAG_DATA_ERRORS) status_or(a.status, SC_STATUS_DATA);
                        }
                    }
                }
            }
            named_bar(NC);
            if (scal_i[4]) {
                aborted = true;
                break;
            }

            // ---- 4. write pass: g = beta p, patched at recorded ids and a ----------
            const float bw = scal[0];
            const float beta = scal[1];
            const float g_a_free = scal[2];
            const int a_li = m.a_li;
            const uint16_t* lrow = a.logits + t * a.lstride + lo;
            float rs = 0.0f;
#pragma unroll 2
            for (int j = tid; j < nvb; j += NC) {
                const uint4 w = ldg_v4_hint(lrow + 8 * j, pol);
                float g0 = beta * ex2(fmaf(bf_lo(w.x), kscale, -bw));
                float g1 = beta * ex2(fmaf(bf_hi(w.x), kscale, -bw));
                float g2 = beta * ex2(fmaf(bf_lo(w.y), kscale, -bw));
                float g3 = beta * ex2(fmaf(bf_hi(w.y), kscale, -bw));
                float g4 = beta * ex2(fmaf(bf_lo(w.z), kscale, -bw));
                float g5 = beta * ex2(fmaf(bf_hi(w.z), kscale, -bw));
                float g6 = beta * ex2(fmaf(bf_lo(w.w), kscale, -bw));
                float g7 = beta * ex2(fmaf(bf_hi(w.w), kscale, -bw));
                const uint32_t word = bm[j >> 5];  // same word for the whole warp
                if (word != 0u && ((word >> (j & 31)) & 1u)) {
                    auto patch = [&](int q, float v) {
                        g0 = q == 0 ? v : g0;
                        g1 = q == 1 ? v : g1;
                        g2 = q == 2 ? v : g2;
                        g3 = q == 3 ? v : g3;
                        g4 = q == 4 ? v : g4;
                        g5 = q == 5 ? v : g5;
                        g6 = q == 6 ? v : g6;
                        g7 = q == 7 ? v : g7;
                    };
                    if ((a_li >> 3) == j) patch(a_li & 7, g_a_free);
                    for (int e = 0; e < nown; ++e) {
                        const int li = li_s[e];
                        if ((li >> 3) == j) patch(li & 7, fix_v[e]);
                    }
                }
                rs += ((g0 + g1) + (g2 + g3)) + ((g4 + g5) + (g6 + g7));
                st_global_v4_hint(grow + 8 * j, pack_bf16x2(g0, g1), pack_bf16x2(g2, g3), pack_bf16x2(g4, g5),
                                  pack_bf16x2(g6, g7), pol);
            }
            if (tail && tid == 0) {
                for (int q = 0; q < tail; ++q) {
                    const int li = n8 + q;
                    float g = li == a_li ? g_a_free : beta * ex2(fmaf(bf_to_f(lrow[li]), kscale, -bw));
                    for (int e = 0; e < nown; ++e)
                        if (li_s[e] == li) g = fix_v[e];
                    rs += g;
                    grow[li] = f_to_bf_bits(g);
                }
            }
            rs = warp_sum(rs);
            if (lane == 0) red[3 * NCW + warp] = rs;
            named_bar(NC);
            if (tid == 0) {
                float tot = 0.0f;
                for (int w = 0; w < NCW; ++w) tot += red[3 * NCW + w];
                rs_prev = tot;
                mbar_arrive(meta_bar(ms, kMetaFree));  // the slot's list and bitmap are free
            }
            t_prev = t;
            ++nmeta;
            ++ndata;
        }
        t_last = t_prev;
        rs_last = rs_prev;
    }

    // The row sum of the last valid row goes to CTA 0 over DSMEM; the final
    // cluster barrier also keeps every CTA's shared memory alive until no
    // peer can still write to it.
    if (tid == 0 && a.diag && t_last >= 0 && !aborted) {
        const uint32_t fs = smem_addr(frs + crank);
        st_cluster_v2(map_to_rank(fs, 0), __float_as_uint(rs_last), 0u);
    }
    cluster_sync_all();
    if (crank == 0 && tid == 0 && a.diag && t_last >= 0 && !aborted) {
        float rsum = 0.0f;
        for (int r = 0; r < C; ++r) rsum += frs[r].x;
        a.diag[t_last].row_sum = rsum;
    }
}

// ---- host side ----------------------------------------------------------

inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

struct Plan {
    int C, NC, S, ncv, NB, MS;
    Layout L;
};

Layout make_layout(int S, int K_max, int NC, int NB, int MS, int C) {
    Layout L;
    L.stage_bytes = round_up(S * 2, 128);
    L.list_cap = K_max > 0 ? K_max : 1;
    L.nwords = (S / 8 + 31) / 32;
    int off = NB * L.stage_bytes;
    auto take = [&](int bytes) {
        const int o = off;
        off = round_up(off + bytes, 16);
        return o;
    };
    L.off_meta = take(MS * static_cast<int>(sizeof(RowMeta)));
    L.off_list_li = take(MS * L.list_cap * 4);
    L.off_list_lp = take(MS * L.list_cap * 4);
    L.off_list_k = take(MS * L.list_cap * 4);
    L.off_bitmap = take(MS * L.nwords * 4);
    L.off_bars = take(kNumBars * 8);
    L.off_part = take(2 * C * static_cast<int>(sizeof(Partial)));
    L.off_mine = take(static_cast<int>(sizeof(Partial)));
    L.off_frs = take(kMaxCluster * 8);
    L.off_fixz = take(L.list_cap * 4);
    L.off_fixv = take(L.list_cap * 4);
    L.off_red = take(4 * (NC / 32) * 4);
    L.off_scal = take(8 * 4);
    L.total = off;
    return L;
}

// Automatic plan: about 40 KiB of logits per CTA (clusters of up to 16
// CTAs), one data stage whose 4 KiB chunks are recycled as the write pass
// frees them, a two-slot metadata ring, 256 compute threads (128 for small
// slices).  For the 151936-entry vocabulary: 8 CTAs x 18992 entries.
int make_plan(int V, int K_max, int req_cluster, int req_threads, int req_stages, Plan* out) {
    const int NB = req_stages > 0 ? req_stages : 1;
    const int MS = NB + 1;
    int C = req_cluster;
    auto threads_for = [&](int S) { return req_threads > 0 ? req_threads : (S >= 8192 ? 256 : 128); };
    if (C <= 0) {
        C = static_cast<int>((2LL * V + 40959) / 40960);
        C = C < 1 ? 1 : (C > kMaxCluster ? kMaxCluster : C);
        while (C > 1 && static_cast<long long>(C - 1) * round_up((V + C - 1) / C, 8) >= V) --C;
    }
    const int S = round_up((V + C - 1) / C, 8);
    const int NC = threads_for(S);
    const Layout L = make_layout(S, K_max, NC, NB, MS, C);
    if (L.total > kMaxSmem)
        return fail(SC_ERR_SHAPE,
                    "V = %d with cluster size %d and %d stages needs %d bytes of shared memory per CTA", V, C,
                    NB, L.total);
    const int nvb = S / 8;
    int nch = (nvb + kChunkVecTarget - 1) / kChunkVecTarget;
    nch = nch < 1 ? 1 : (nch > kMaxChunks ? kMaxChunks : nch);
    out->C = C;
    out->NC = NC;
    out->S = S;
    out->NB = NB;
    out->MS = MS;
    // a whole number of 32-vector groups per chunk keeps each warp's bitmap word uniform
    out->ncv = round_up((nvb + nch - 1) / nch, 32);
    if (out->ncv < 32) out->ncv = 32;
    out->L = L;
    return SC_OK;
}

using KernelFn = void (*)(KArgs);

KernelFn kernel_for(int NC) {
    switch (NC) {
        case 128: return center_kernel<128>;
        case 256: return center_kernel<256>;
        case 384: return center_kernel<384>;
        case 512: return center_kernel<512>;
        default: return nullptr;
    }
}

std::mutex g_plan_mutex;
std::map<std::tuple<int, int>, int> g_attr_set;                     // (device, NC)
std::map<std::tuple<int, int, int, int>, int> g_max_clusters;      // (device, NC, C, smem)

// Sets the kernel's shared-memory and cluster attributes and returns the
// number of clusters that can be resident at once.
int prepare_kernel(int dev, const Plan& P, int* max_clusters) {
    KernelFn fn = kernel_for(P.NC);
    if (!fn) return fail(SC_ERR_ARG, "threads = %d is not one of 128, 256, 384, 512", P.NC);
    std::lock_guard<std::mutex> lock(g_plan_mutex);
    cudaError_t e;
    auto key = std::make_tuple(dev, P.NC);
    if (g_attr_set.find(key) == g_attr_set.end()) {
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic smem)");
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(non-portable cluster)");
        g_attr_set[key] = 1;
    }
    auto ckey = std::make_tuple(dev, P.NC, P.C, P.L.total);
    auto cit = g_max_clusters.find(ckey);
    if (cit != g_max_clusters.end()) {
        *max_clusters = cit->second;
        return SC_OK;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(P.C, 1, 1);
    cfg.blockDim = dim3(P.NC + 32, 1, 1);
    cfg.dynamicSmemBytes = P.L.total;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = P.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(fn), &cfg);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
    if (n <= 0)
        return fail(SC_ERR_SHAPE, "a cluster of %d CTAs with %d bytes of shared memory does not fit",
                    P.C, P.L.total);
    g_max_clusters[ckey] = n;
    *max_clusters = n;
    return SC_OK;
}

int check_params(int V, const sc_params* p) {
    if (!p) return fail(SC_ERR_NULL, "params is NULL");
    if (V < 1 || V > kMaxV) return fail(SC_ERR_SHAPE, "V = %d outside 1..%d", V, kMaxV);
    if (p->K_max < 0 || p->K_max > kMaxK)
        return fail(SC_ERR_SHAPE, "K_max = %d outside 0..%d", p->K_max, kMaxK);
    if (!(p->inv_temperature > 0.0f) || !std::isfinite(p->inv_temperature) || p->inv_temperature > 1e4f)
        return fail(SC_ERR_ARG, "inv_temperature must be finite and in (0, 1e4]");
    if (!std::isfinite(p->grad_scale)) return fail(SC_ERR_ARG, "grad_scale must be finite");
    if (p->is_mode < SC_IS_NONE || p->is_mode > SC_IS_MIS) return fail(SC_ERR_ARG, "is_mode = %d", p->is_mode);
    if (p->is_mode == SC_IS_TIS && !(p->tis_max > 0.0f && std::isfinite(p->tis_max)))
        return fail(SC_ERR_ARG, "tis_max must be finite and > 0");
    if (p->is_mode == SC_IS_MIS &&
        !(p->mis_min >= 0.0f && p->mis_min <= p->mis_max && std::isfinite(p->mis_max)))
        return fail(SC_ERR_ARG, "need 0 <= mis_min <= mis_max < inf");
    if (p->centering != 0 && p->centering != 1) return fail(SC_ERR_ARG, "centering must be 0 or 1");
    if (p->cluster_size < 0 || p->cluster_size > kMaxCluster)
        return fail(SC_ERR_ARG, "cluster_size = %d outside 0..%d", p->cluster_size, kMaxCluster);
    if (p->threads != 0 && !kernel_for(p->threads))
        return fail(SC_ERR_ARG, "threads = %d is not 0, 128, 256, 384 or 512", p->threads);
    if (p->stages < 0 || p->stages > kMaxStages)
        return fail(SC_ERR_ARG, "stages = %d outside 0..%d", p->stages, kMaxStages);
    return SC_OK;
}

}  // namespace
}  // namespace sc

extern "C" int sc_plan_query(int V, const sc_params* p, int* cluster_size, int* threads, int* slice,
                             int* smem_bytes, int* max_clusters) {
    using namespace sc;
    int st = check_params(V, p);
    if (st != SC_OK) return st;
    Plan P;
    st = make_plan(V, p->K_max, p->cluster_size, p->threads, p->stages, &P);
    if (st != SC_OK) return st;
    int dev = 0;
    st = check_device(&dev);
    if (st != SC_OK) return st;
    int mc = 0;
    st = prepare_kernel(dev, P, &mc);
    if (st != SC_OK) return st;
    if (cluster_size) *cluster_size = P.C;
    if (threads) *threads = P.NC;
    if (slice) *slice = P.S;
    if (smem_bytes) *smem_bytes = P.L.total;
    if (max_clusters) *max_clusters = mc;
    return ok();
}

extern "C" int sc_center_forward_backward(const uint16_t* logits, long long T, int V,
                                          long long logits_stride, const int32_t* rec_ids,
                                          const float* rec_logprobs, const int32_t* rec_count,
                                          const int32_t* sampled_id, const float* rollout_logprob,
                                          const int32_t* row_response, const float* adv, int n_resp,
                                          const sc_params* p, uint16_t* grad_out, long long grad_stride,
                                          float* logp_out, sc_row_diag* diag_out, uint32_t* status_dev,
                                          sc_stream_t stream) {
    using namespace sc;
    int st = check_params(V, p);
    if (st != SC_OK) return st;
    if (T < 0) return fail(SC_ERR_SHAPE, "T = %lld < 0", T);
    if (n_resp < 0) return fail(SC_ERR_SHAPE, "n_resp = %d < 0", n_resp);
    if (logits_stride < V || grad_stride < V)
        return fail(SC_ERR_SHAPE, "row strides (%lld, %lld) must be >= V = %d", logits_stride, grad_stride, V);
    if (p->is_mode != SC_IS_NONE && !rollout_logprob)
        return fail(SC_ERR_NULL, "is_mode tis/mis needs rollout_logprob");
    if (T == 0) return ok();
    if (!logits || !sampled_id || !row_response || !grad_out || !logp_out)
        return fail(SC_ERR_NULL, "logits, sampled_id, row_response, grad_out and logp_out are required");
    if (n_resp > 0 && !adv) return fail(SC_ERR_NULL, "adv is NULL with n_resp > 0");
    if (p->K_max > 0 && (!rec_ids || !rec_logprobs))
        return fail(SC_ERR_NULL, "rec_ids and rec_logprobs are required when K_max > 0");
    if (!aligned(logits, 16) || !aligned(grad_out, 16))
        return fail(SC_ERR_ALIGN, "logits and grad_out must be 16-byte aligned");
    if (logits_stride % 8 != 0 || grad_stride % 8 != 0)
        return fail(SC_ERR_ALIGN, "row strides must be multiples of 8 elements");
    if (!aligned(rec_ids, 4) || !aligned(rec_logprobs, 4) || !aligned(rec_count, 4) ||
        !aligned(sampled_id, 4) || !aligned(rollout_logprob, 4) || !aligned(row_response, 4) ||
        !aligned(adv, 4) || !aligned(logp_out, 4) || !aligned(diag_out, 16) || !aligned(status_dev, 4))
        return fail(SC_ERR_ALIGN, "metadata arrays must be 4-byte aligned and diag_out 16-byte aligned");
    {
        const char* l0 = reinterpret_cast<const char*>(logits);
        const char* g0 = reinterpret_cast<const char*>(grad_out);
        const long long lb = 2LL * ((T - 1) * logits_stride + V);
        const long long gb = 2LL * ((T - 1) * grad_stride + V);
        const bool same = (l0 == g0) && (logits_stride == grad_stride);
        if (!same && l0 < g0 + gb && g0 < l0 + lb)
            return fail(SC_ERR_ARG, "grad_out overlaps logits other than exactly (in place)");
    }
    Plan P;
    st = make_plan(V, p->K_max, p->cluster_size, p->threads, p->stages, &P);
    if (st != SC_OK) return st;
    int dev = 0;
    st = check_device(&dev);
    if (st != SC_OK) return st;
    int mc = 0;
    st = prepare_kernel(dev, P, &mc);
    if (st != SC_OK) return st;
    const long long G = T < mc ? T : mc;

    KArgs ka;
    std::memset(&ka, 0, sizeof ka);
    ka.logits = logits;
    ka.ids = rec_ids;
    ka.lps = rec_logprobs;
    ka.cnt = rec_count;
    ka.sampled = sampled_id;
    ka.rollout = rollout_logprob;
    ka.resp = row_response;
    ka.adv = adv;
    ka.grad = grad_out;
    ka.logp = logp_out;
    ka.diag = diag_out;
    ka.status = status_dev;
    ka.T = T;
    ka.lstride = logits_stride;
    ka.gstride = grad_stride;
    ka.V = V;
    ka.K_max = p->K_max;
    ka.n_resp = n_resp;
    ka.is_mode = p->is_mode;
    ka.centering = p->centering;
    ka.tis_max = p->tis_max;
    ka.mis_min = p->mis_min;
    ka.mis_max = p->mis_max;
    ka.inv_t = p->inv_temperature;
    ka.grad_scale = p->grad_scale;
    ka.C = P.C;
    ka.S = P.S;
    ka.ncv = P.ncv;
    ka.NB = P.NB;
    ka.MS = P.MS;
    ka.L = P.L;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(G * P.C), 1, 1);
    cfg.blockDim = dim3(P.NC + 32, 1, 1);
    cfg.dynamicSmemBytes = P.L.total;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = P.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel_for(P.NC), ka);
    if (e != cudaSuccess) return cuda_fail(e, "center_kernel launch");
    return ok();
}
