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
// * The row warp walks the cluster's rows ahead of the others: the first
//   seven eighths of the rows dealt round robin, the rest handed out at run
//   time from a counter in the caller's workspace (CTA 0 takes each row and
//   passes its index to its peers through their shared memory).  Padding and
//   error rows go to the zero warp's queue.  For every valid row it fills a
//   slot of a metadata ring, up to three rows ahead -- the row's scalars and
//   the compact list of recorded ids that fall in this CTA's slice (repeats
//   dropped), with flags marking them (one bit per entry, or one bit per
//   8-entry vector with the flagged vectors' masks).
// * The copy warp takes the valid rows from that ring and starts 1-D bulk
//   copies (TMA engine) of each logit slice into shared memory, chunk by
//   chunk, each as soon as the streaming warps have released that chunk.
// * The streaming warps take each row through two passes over the slice in
//   shared memory.  Phase A: with one exponent offset (the largest logit of the
//   slice's first vectors), sum 2^y and its entropy term over the unrecorded
//   entries (recorded ids are skipped through the flags, so the unrecorded
//   mass accumulates directly, with no 1 - P_H cancellation); each warp sends
//   its 16-byte partial to every CTA of the cluster the moment it is done
//   (st.async stores that complete as transaction bytes on the receiver's
//   mbarrier).  Then, once the cluster has the row scalars, the write pass:
//   g_v = beta p_v with 16-byte stores and no special cases, handing every
//   chunk back to the copy warp as soon as it is written, so the next row
//   streams into the stage while this one is written.
// * The scalar warp does the per-row serial work off the streaming path.
//   While phase A runs it picks up the recorded ids' logits from the slice,
//   sums them relative to their own offset and sends this CTA's 64-byte record
//   (those sums, the recorded probabilities, the sampled token's logit, the
//   previous row's gradient sum) to every CTA of the cluster.  The C records
//   land on their own mbarrier and are merged lane-parallel (a butterfly: the
//   same bits in every CTA) while the streaming partials are still on their
//   way; once the last partial has landed, the short critical merge (the row
//   maximum, one summed value) gives the row scalars the write pass needs (LSE,
//   P_H, Q_H, rho, s, importance weight), published at once, then the loss, k3
//   and entropy, and it patches the previous row's special entries (recorded
//   ids and the sampled token) with their own gradients.
// * The zero warp writes the queued zero rows (padding and error rows) and
//   their log p_a and diagnostics, so the row warp never waits on them.
// Every logit is read from HBM once and every gradient written once.  The
// grid is persistent (as many clusters as fit).  Every wait is bounded (about
// 1 s) and reports through the status word.
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
constexpr int kMaxStages = 4;  // data stages
constexpr int kMetaSlots = 4;  // metadata ring: rows in the write pass, in phase A, and two prefetched
// Exchange buffers.  Two suffice: a CTA sends its partials of row j + 2 only
// after it has merged row j + 1, which took every peer's partials of row
// j + 1, and a peer sends those only after its write pass of row j, which
// follows its own merge (its reads) of row j.
constexpr int kXBufs = 2;
constexpr int kMaxK = 1024;
constexpr int kMaxV = 1 << 20;
constexpr int kMaxSmem = 232448;        // 227 KiB of dynamic shared memory per CTA
constexpr int kTwoPerSmBytes = 114688;  // dynamic shared memory that still fits two CTAs on an SM
constexpr int kChunkVecTarget = 2048;   // 16-byte vectors per bulk copy (32 KiB; measured best of 8-128 KiB)
constexpr int kGrab = 8;                // grab ring: rows CTA 0 may hand out ahead of its peers
constexpr int kZq = 16;                 // zero queue: zero rows the row warp may queue ahead
constexpr long long kDynamicShare = 8;  // 1 / (share of the rows handed out at run time; measured best of 3..20)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kTailFloor = 1e-6f;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // default limit of a bounded wait
constexpr unsigned long long kDrainLimitNs = 1000000000ull;  // bulk copies in flight before a CTA leaves
constexpr uint32_t kFull = 0xFFFFFFFFu;

// One valid row as the row warp hands it to the copy warp and the consumers.
struct RowMeta {
    long long t;     // row index; -1 ends the consumers' loop
    int sa;          // sampled id
    int nown;        // recorded ids of this CTA's slice in the compact list
    int a_li;        // local index of a in this slice, -1 if another CTA owns it
    uint32_t flags;  // row flags found by the row warp (count, repeats, out of range)
    float A, rl;     // advantage, rollout logprob
    // this slice's recorded ids, from their log-probabilities alone
    float qbest;     // the largest q (0 if none)
    float omq;       // 1 - qbest, from its log-probability
    float oh, ol;    // the sum of the other q (double-float)
    int kbest;       // position k of qbest (INT_MAX if none)
    int pad[3];
};
static_assert(sizeof(RowMeta) == 64, "RowMeta layout");

// What a row's exchange carries to every CTA of the cluster.  Each streaming
// warp sends its phase-A sums over its share of the unrecorded entries as soon
// as it has them (16 bytes); y' values are relative to the warp's offset m
// (y' = (z - m) kscale).
struct WarpPart {
    float m;       // the warp's exponent offset in z (-inf: nothing summed)
    float S1, S2;  // sum 2^y', sum 2^y' y'
    float pad;
};
static_assert(sizeof(WarpPart) == 16, "warp partial is 16 bytes");
// The scalar warp sends the rest of the CTA's contribution (64 bytes), which
// needs only the slice: the recorded ids owned here relative to their own
// offset, their probabilities, the logit of the sampled token, and the
// finished gradient sum of the previous row.
struct CtaRec {
    float m;            // offset of the recorded ids' sums in z (-inf: none)
    float lH, EH;       // recorded ids owned here: sum 2^y', sum 2^y' y'
    float QY;           // sum q_k y'_k over them
    float rs;           // FP32 gradient sum of this slice for the previous row
    float qo_hi, qo_lo; // sum of q_k over them except the largest one (double-float)
    float qbest;        // the largest q_k owned here (0 if none)
    int kbest;          // its position k (INT_MAX if none)
    int nval;           // owned recorded ids used
    uint32_t flags;     // row flags found by this CTA's row warp
    float za;           // logit of the sampled token, if this CTA owns it
    int has_a;
    float omq;          // 1 - qbest, from its log-probability (-expm1)
    int pad[2];
};
static_assert(sizeof(CtaRec) == 64, "CTA record is 64 bytes");

struct Layout {
    int stage_bytes;  // bytes of one data stage (128-aligned)
    int list_cap;     // entries of one owned list (K_max)
    int nwords;       // flag words of one slice (a bit per entry, or per 8-entry vector)
    int mwords;       // mask words of one slot (per-vector flags: four 8-bit masks a word)
    int off_meta, off_list_li, off_list_q, off_bitmap, off_vpre, off_vmask, off_bars, off_wpart, off_rec, off_frs,
        off_fixz, off_fixv, off_zav, off_rsw, off_scal, off_flag, off_grab, off_zq, off_zqf, off_ticket, total;
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
    unsigned long long* ws;  // [0]: rows handed out after T_static, [1]: CTAs that have finished
    long long T_static;      // rows dealt round robin before the hand-out starts (a multiple of the clusters)
    long long T, lstride, gstride;
    int V, K_max, n_resp;
    int is_mode, centering;
    float tis_max, mis_min, mis_max, inv_t, grad_scale, clip_lo, clip_hi;
    unsigned long long wait_ns;  // limit of every bounded wait but the final drains of bulk copies
    int stall;                   // test hook: the first bulk copy of each CTA is left out
    int C, S, ncv, NB;
    Layout L;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {  // exact: the same in every lane
    float r;
    asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ uint16_t f_to_bf_bits(float x) {
    return static_cast<uint16_t>(pack_bf16x2(x, 0.0f) & 0xFFFFu);
}
__device__ __forceinline__ void status_or(uint32_t* st, uint32_t bits) {
    if (st) atomicOr(st, bits);
}

// Running (max, sum 2^y, sum 2^y y) triples, y relative to max * kscale.
// Merging rescales both sides to the larger maximum; an empty side (m = -inf)
// contributes nothing.  The merge is commutative, so a butterfly leaves every
// lane with the same bits.
struct Mass {
    float m, s1, s2;
};
__device__ __forceinline__ Mass mass_merge(const Mass& a, const Mass& b, float kscale) {
    const float m = fmaxf(a.m, b.m);
    Mass r;
    r.m = m;
    r.s1 = 0.0f;
    r.s2 = 0.0f;
    if (a.m > -INFINITY) {
        const float d = (a.m - m) * kscale;
        const float f = ex2(d);
        r.s1 = f * a.s1;
        r.s2 = f * fmaf(d, a.s1, a.s2);
    }
    if (b.m > -INFINITY) {
        const float d = (b.m - m) * kscale;
        const float f = ex2(d);
        r.s1 = fmaf(f, b.s1, r.s1);
        r.s2 = fmaf(f, fmaf(d, b.s1, b.s2), r.s2);
    }
    return r;
}
__device__ __forceinline__ Mass mass_shfl(const Mass& x, int off) {
    return Mass{__shfl_xor_sync(kFull, x.m, off), __shfl_xor_sync(kFull, x.s1, off),
                __shfl_xor_sync(kFull, x.s2, off)};
}

// Largest recorded probability with the mass of the others, merged
// commutatively (ties go to the lower k).  The others' mass is kept as an
// unevaluated FP32 pair.
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

// Barriers.  Meta slot s: kMetaFull (row warp wrote it), kMetaFree (its row
// is written).  Exchange buffer x: kXRec (a row's C records) and kXPart (its
// C x warps partials), each the own expect_tx arrive + every CTA's bytes.  kWDone[p]: every streaming warp
// finished the write pass of a row of parity p.  kSReady[p]: the row scalars of
// a row of parity p are published.  Grab ring slot g: kGrabFull (the row index
// from CTA 0 landed, tx bytes), kGrabFree (in CTA 0: every CTA of the cluster
// has read it).  Zero queue slot z: kZqFull (row warp wrote it), kZqFree (the
// zero warp took it).  Ticket s: the row index of a valid row is in ticket
// slot s (row warp, before its metadata work).  Then, per data stage d: kChunkFull + i (copy of chunk i
// landed, tx bytes), kChunkFree + i (every streaming warp is done with chunk i);
// only the plan's stages take space.
constexpr int kMetaBase = 0;
constexpr int kMetaFull = 0;
constexpr int kMetaFree = 1;
constexpr int kXRec = kMetaBase + 2 * kMetaSlots;
constexpr int kXPart = kXRec + kXBufs;
constexpr int kWDone = kXPart + kXBufs;
constexpr int kSReady = kWDone + 2;
constexpr int kGrabBase = kSReady + 2;
constexpr int kZqBase = kGrabBase + 2 * kGrab;
constexpr int kTicketBase = kZqBase + 2 * kZq;
constexpr int kDataBase = kTicketBase + kMetaSlots;
constexpr int kChunkFull = 0;
constexpr int kChunkFree = kMaxChunks;
constexpr int kBarsPerStage = 2 * kMaxChunks;
constexpr int num_bars(int NB) { return kDataBase + NB * kBarsPerStage; }

// Threads of a CTA besides the NC streaming threads: the scalar, row, zero
// and copy warps.
constexpr int kAuxThreads = 128;
// Resident CTAs per SM the register allocation must allow.
constexpr int min_blocks(int NC) { return NC <= 128 ? 4 : 2; }

// VF: recorded-id flags one bit per 8-entry vector (with the flagged vectors'
// masks) instead of one bit per entry.
template <int NC, bool VF>
__global__ void __launch_bounds__(NC + kAuxThreads, min_blocks(NC)) center_kernel(const __grid_constant__ KArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int NCW = NC / 32;  // streaming warps; warp NCW: row scalars; NCW + 1: rows; NCW + 2: zero rows; NCW + 3: copies
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t crank = cluster_ctarank();
    const uint32_t cid = cluster_id_x();
    const uint32_t ncl = num_clusters_x();
    const int C = a.C, K_max = a.K_max, NB = a.NB;
    const Layout& L = a.L;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.off_bars);
    RowMeta* meta = reinterpret_cast<RowMeta*>(smem + L.off_meta);         // [kMetaSlots]
    int* list_li = reinterpret_cast<int*>(smem + L.off_list_li);           // [kMetaSlots][cap]
    float* list_q = reinterpret_cast<float*>(smem + L.off_list_q);         // [kMetaSlots][cap] q = e^lp
    uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem + L.off_bitmap);   // [kMetaSlots][nwords] flags
    uint16_t* vpre = reinterpret_cast<uint16_t*>(smem + L.off_vpre);        // VF: [kMetaSlots][nwords]
    uint32_t* vmask = reinterpret_cast<uint32_t*>(smem + L.off_vmask);      // VF: [kMetaSlots][mwords]
    WarpPart* wpart = reinterpret_cast<WarpPart*>(smem + L.off_wpart);    // [kXBufs][C][NCW]
    CtaRec* crec = reinterpret_cast<CtaRec*>(smem + L.off_rec);            // [kXBufs][C]
    float2* frs = reinterpret_cast<float2*>(smem + L.off_frs);             // [kMaxCluster]
    float* fix_z = reinterpret_cast<float*>(smem + L.off_fixz);            // [2][cap] recorded logits
    float* fix_v = reinterpret_cast<float*>(smem + L.off_fixv);            // [2][cap] their gradients
    float* zav = reinterpret_cast<float*>(smem + L.off_zav);               // [2] logit of a
    float* rsw = reinterpret_cast<float*>(smem + L.off_rsw);               // [2][NCW] warp row sums
    float* scal = reinterpret_cast<float*>(smem + L.off_scal);             // [2][4] row scalars
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.off_flag);
    volatile uint32_t* copied = reinterpret_cast<volatile uint32_t*>(smem + L.off_flag + 4);  // rows with all copies started
    long long* grab_ring = reinterpret_cast<long long*>(smem + L.off_grab);  // [kGrab] row indices from CTA 0
    long long* zq_t = reinterpret_cast<long long*>(smem + L.off_zq);        // [kZq] zero rows
    uint32_t* zq_f = reinterpret_cast<uint32_t*>(smem + L.off_zqf);         // [kZq] their flags
    long long* ticket = reinterpret_cast<long long*>(smem + L.off_ticket);  // [kMetaSlots] valid rows' indices
    auto data_bar = [&](int d, int i) { return smem_addr(&bars[kDataBase + d * kBarsPerStage + i]); };
    auto meta_bar = [&](int s, int i) { return smem_addr(&bars[kMetaBase + 2 * s + i]); };
    auto xrec = [&](int x) { return smem_addr(&bars[kXRec + x]); };
    auto xpart = [&](int x) { return smem_addr(&bars[kXPart + x]); };
    auto wdone = [&](int p) { return smem_addr(&bars[kWDone + p]); };
    auto sready = [&](int p) { return smem_addr(&bars[kSReady + p]); };
    auto grab_full = [&](int g) { return smem_addr(&bars[kGrabBase + 2 * g]); };
    auto grab_free = [&](int g) { return smem_addr(&bars[kGrabBase + 2 * g + 1]); };
    auto zq_full = [&](int z) { return smem_addr(&bars[kZqBase + 2 * z]); };
    auto zq_free = [&](int z) { return smem_addr(&bars[kZqBase + 2 * z + 1]); };
    auto ticket_bar = [&](int s) { return smem_addr(&bars[kTicketBase + s]); };

    const int lo = static_cast<int>(crank) * a.S;
    const int hi = min(lo + a.S, a.V);
    const int n = max(hi - lo, 0);
    const int n8 = n & ~7, nvb = n8 >> 3, tail = n - n8;
    const int nchunks = (nvb + a.ncv - 1) / a.ncv;
    const int cap = L.list_cap, nwords = L.nwords, mwords = L.mwords;
    const float kscale = a.inv_t * kLog2e;
    const unsigned long long wait_ns = a.wait_ns;
    const uint64_t pol = l2_policy_evict_first();      // last use: gradient stores, write-pass reads
    const uint64_t pol_keep = l2_policy_evict_normal();  // slice copies (measured: evict-first is slower)

    if (tid == 0) {
        for (int d = 0; d < NB; ++d)
            for (int i = 0; i < kMaxChunks; ++i) {
                mbar_init(data_bar(d, kChunkFull + i), 1u);
                mbar_init(data_bar(d, kChunkFree + i), static_cast<uint32_t>(NCW));
            }
        for (int s = 0; s < kMetaSlots; ++s) {
            mbar_init(meta_bar(s, kMetaFull), 1u);
            mbar_init(meta_bar(s, kMetaFree), 1u);
            mbar_init(ticket_bar(s), 1u);
            meta[s].nown = 0;
        }
        for (int x = 0; x < kXBufs; ++x) {
            mbar_init(xrec(x), 1u);
            mbar_init(xpart(x), 1u);
        }
        for (int p = 0; p < 2; ++p) {
            mbar_init(wdone(p), static_cast<uint32_t>(NCW));
            mbar_init(sready(p), 1u);
        }
        for (int g = 0; g < kGrab; ++g) {
            mbar_init(grab_full(g), 1u);
            mbar_init(grab_free(g), static_cast<uint32_t>(C));
        }
        for (int z = 0; z < kZq; ++z) {
            mbar_init(zq_full(z), 1u);
            mbar_init(zq_free(z), 1u);
        }
        for (int r = 0; r < kMaxCluster; ++r) frs[r] = make_float2(0.0f, 0.0f);
        *abort_flag = 0;
        *copied = 0u;
        fence_mbar_init_cluster();
    }
    for (int i = tid; i < kMetaSlots * nwords; i += NC + kAuxThreads) bitmap[i] = 0u;
    // Launched with programmatic stream serialisation: everything above touches
    // only shared memory and may overlap the previous kernel in the stream; no
    // global input is read before that kernel has completed.
    grid_dependency_wait();
    cluster_sync_all();  // every CTA's barriers exist before peers signal them

    // Any role that gives up raises the flag; the others see it at their next
    // row and leave too (their waits are bounded in any case).
    auto give_up = [&](uint32_t bits) {
        if (lane == 0) {
            status_or(a.status, bits);
            *abort_flag = 1;
        }
    };
    auto flag_up = [&]() { return __any_sync(kFull, *abort_flag != 0); };

    // scalar warp state kept for the final row-sum flush
    bool clean_end = false;
    uint32_t nrows = 0;
    float fin_rs1 = 0.0f;
    long long t_m1 = -1;    // row index of the row before the current one
    float corr_m1 = 0.0f;   // its row-sum correction for the patched entries

    // The write pass stores g = beta p everywhere; once it is done with row r,
    // the scalar warp overwrites the recorded ids and a with their own values.
    auto patch_row = [&](uint32_t r, long long t) {
        const int sl = static_cast<int>(r % kMetaSlots);
        const int q = static_cast<int>(r & 1u);
        const int* li = list_li + sl * cap;
        const float* fv = fix_v + q * cap;
        const int nown = meta[sl].nown, a_li = meta[sl].a_li;
        uint16_t* grow = a.grad + t * a.gstride + lo;
        bool a_rec = false;
        for (int e = lane; e < nown; e += 32) {
            const int l = li[e];
            a_rec = a_rec || l == a_li;
            grow[l] = f_to_bf_bits(fv[e]);
        }
        a_rec = __any_sync(kFull, a_rec);
        if (lane == 0 && a_li >= 0 && !a_rec) grow[a_li] = f_to_bf_bits(scal[4 * q + 2]);
    };

    if (warp == NCW + 1) {
        // ================= row warp: rows, zero queue, metadata =================
        // Rows [0, T_static) are dealt round robin (row cid + k * ncl).  The rest
        // are handed out at run time: CTA 0 of the cluster takes the next one
        // from the launch's counter (workspace; the following take is always in
        // flight) and sends it to every CTA of the cluster through a grab ring in
        // their shared memory, so the clusters that have run ahead take more of
        // the last rows and all finish together.  Rows with a response get a
        // metadata slot (the copy warp starts their slice copies); zero rows (padding, bad
        // response or sampled id) go to the zero warp's queue, so their stores
        // never hold up the row warp.
        uint32_t nfill = 0, ng = 0, nz = 0;
        bool stop = false;
        long long t_static = cid;
        // The cluster's first row is known at launch: all its inputs are loaded
        // at once (the streaming warps wait on its metadata; later rows are built
        // ahead of need).  If it is padding only these loads were spent.
        const long long t_first = t_static < a.T_static ? t_static : -1;
        int f_rj = -1, f_sj = 0, f_cnt = K_max, f_id[4];
        float f_rl = 0.0f, f_lp[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            f_id[r] = -1;
            f_lp[r] = 0.0f;
        }
        if (t_first >= 0) {
            f_rj = __ldg(a.resp + t_first);
            f_sj = __ldg(a.sampled + t_first);
            if (a.cnt) f_cnt = __ldg(a.cnt + t_first);
            if (a.rollout) f_rl = __ldg(a.rollout + t_first);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int k = 32 * r + lane;
                if (k < K_max) {  // (in bounds whatever the row's count)
                    f_id[r] = __ldg(a.ids + t_first * static_cast<long long>(K_max) + k);
                    f_lp[r] = __ldg(a.lps + t_first * static_cast<long long>(K_max) + k);
                }
            }
        }
        unsigned long long pend = 0;  // CTA 0, lane 0: the counter value of the take in flight
        bool pending = false;
        for (;;) {
            if (flag_up()) {
                stop = true;
                break;
            }
            long long t;
            if (t_static < a.T_static) {
                t = t_static;
                t_static += ncl;
            } else {
                const int g = static_cast<int>(ng % kGrab);
                if (crank == 0) {
                    // every CTA has read this slot's previous row (bounded wait)
                    bool ok = true;
                    if (ng >= static_cast<uint32_t>(kGrab))
                        ok = mbar_wait_cluster_bounded(grab_free(g), ((ng / kGrab) - 1u) & 1u, wait_ns);
                    if (!__all_sync(kFull, ok)) {
                        give_up(SC_STATUS_TIMEOUT_LOAD);
                        stop = true;
                        break;
                    }
                    // A run-time row is taken only once every published row has had
                    // its copies started: a row taken early is one that a cluster
                    // further ahead could have finished first (measured: one row of
                    // look-ahead lengthens the 4096-row batch's tail by ~1.5 us).
                    bool paced = true;
                    {
                        const unsigned long long t0 = global_timer_ns();
                        while (nfill > *copied) {
                            if (global_timer_ns() - t0 > wait_ns) {
                                paced = false;
                                break;
                            }
                            __nanosleep(128);
                        }
                    }
                    if (!__all_sync(kFull, paced)) {
                        give_up(SC_STATUS_TIMEOUT_LOAD);
                        stop = true;
                        break;
                    }
                    unsigned long long tg = 0;
                    if (lane == 0) {
                        tg = static_cast<unsigned long long>(a.T_static) + (pending ? pend : atomicAdd(a.ws, 1ull));
                        pending = tg < static_cast<unsigned long long>(a.T);
                        if (pending) pend = atomicAdd(a.ws, 1ull);  // the next take, in flight
                    }
                    tg = __shfl_sync(kFull, tg, 0);
                    if (lane < C)
                        st_async_v2(map_to_rank(smem_addr(grab_ring + g), lane), static_cast<uint32_t>(tg),
                                    static_cast<uint32_t>(tg >> 32), map_to_rank(grab_full(g), lane));
                }
                if (lane == 0) mbar_expect_tx(grab_full(g), 8u);
                if (!__all_sync(kFull, mbar_wait_cluster_bounded(grab_full(g), (ng / kGrab) & 1u, wait_ns))) {
                    give_up(SC_STATUS_TIMEOUT_LOAD);
                    stop = true;
                    break;
                }
                const unsigned long long tu = static_cast<unsigned long long>(grab_ring[g]);
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(map_to_rank(grab_free(g), 0));  // slot read
                ++ng;
                if (tu >= static_cast<unsigned long long>(a.T)) break;  // no rows left
                t = static_cast<long long>(tu);
            }
            const bool first = t == t_first;
            const int rj = first ? f_rj : __ldg(a.resp + t);
            const int sj = first ? f_sj : __ldg(a.sampled + t);  // (both loads in flight together)
            uint32_t zf = 0;
            if (rj < 0) {
                zf = SC_FLAG_MASKED;
            } else if (rj >= a.n_resp) {
                zf = SC_FLAG_BAD_RESPONSE;
            } else if (sj < 0 || sj >= a.V) {
                zf = SC_FLAG_BAD_SAMPLED;
            }
            if (zf) {  // zero row: to the zero warp's queue
                const int z = static_cast<int>(nz % kZq);
                if (nz >= static_cast<uint32_t>(kZq) &&
                    !__all_sync(kFull, mbar_wait_bounded(zq_free(z), ((nz / kZq) - 1u) & 1u, wait_ns))) {
                    give_up(SC_STATUS_TIMEOUT_LOAD);
                    stop = true;
                    break;
                }
                if (lane == 0) {
                    zq_t[z] = t;
                    zq_f[z] = zf;
                    mbar_arrive(zq_full(z));  // release: the slot
                }
                ++nz;
                continue;
            }
            const int ms = static_cast<int>(nfill % kMetaSlots);
            if (nfill >= static_cast<uint32_t>(kMetaSlots) &&
                !mbar_wait_bounded(meta_bar(ms, kMetaFree), ((nfill / kMetaSlots) - 1u) & 1u, wait_ns)) {
                if (lane == 0) status_or(a.status, SC_STATUS_TIMEOUT_LOAD);
                stop = true;
                break;
            }
            // the row's index to the copy warp, which can start the slice's copies
            // while the metadata is built (the slot's previous row is written)
            if (lane == 0) {
                ticket[ms] = t;
                mbar_arrive(ticket_bar(ms));  // release: the ticket
            }
            // ---- recorded ids of this slice: compact list, repeats dropped ----
            // (row scalars loaded first so their latency overlaps the list)
            const float row_A = __ldg(a.adv + rj);
            const float row_rl = first ? f_rl : (a.rollout ? __ldg(a.rollout + t) : 0.0f);
            int cnt = first ? f_cnt : (a.cnt ? __ldg(a.cnt + t) : K_max);
            uint32_t flags = 0;
            if (cnt < 0 || cnt > K_max) {
                flags |= SC_FLAG_BAD_COUNT;
                cnt = cnt < 0 ? 0 : K_max;
            }
            int* li_s = list_li + ms * cap;
            float* q_s = list_q + ms * cap;
            uint32_t* bm = bitmap + ms * nwords;
            uint16_t* pre = vpre + ms * nwords;
            uint32_t* mk = vmask + ms * mwords;
            {  // clear the flags of the slot's previous row (whole words: they are all its own)
                const int old = meta[ms].nown;
                for (int e = lane; e < old; e += 32) bm[li_s[e] >> (VF ? 8 : 5)] = 0u;
                if constexpr (VF)
                    for (int w = lane; w < mwords; w += 32) mk[w] = 0u;
            }
            __syncwarp();
            const long long kb = t * static_cast<long long>(K_max);
            int nown = 0;
            bool bad = false, dup = false;
            HeadMass hm{0.0f, 0x7FFFFFFF, 1.0f, 0.0f, 0.0f};  // the kept ids' q, merged
            for (int kb0 = 0; kb0 < cnt; kb0 += 128) {
                int idr[4];
                float lpr[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {  // four rounds of loads in flight together
                    const int k = kb0 + 32 * r + lane;
                    if (first && kb0 == 0) {
                        idr[r] = f_id[r];
                        lpr[r] = f_lp[r];
                    } else {
                        idr[r] = k < cnt ? __ldg(a.ids + kb + k) : -1;
                        lpr[r] = k < cnt ? __ldg(a.lps + kb + k) : 0.0f;
                    }
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
                        const float q = expf(lpr[r]);
                        li_s[pos] = id - lo;
                        q_s[pos] = q;
                        hm = head_merge(hm, HeadMass{q, k, -expm1f(lpr[r]), 0.0f, 0.0f});
                        if constexpr (VF)
                            atomicOr(&bm[(id - lo) >> 8], 1u << (((id - lo) >> 3) & 31));
                        else
                            atomicOr(&bm[(id - lo) >> 5], 1u << ((id - lo) & 31));
                    }
                    nown += __popc(km);
                    __syncwarp();
                }
            }
            if constexpr (VF) {
                if (nown > 0) {
                    // rank of each flagged vector among the slice's flagged vectors, in
                    // vector order: per flag word, the flags of the words before it
                    // (each lane counts a run of consecutive words, one warp scan)
                    const int wb = (nwords + 31) >> 5;
                    const int w0 = min(lane * wb, nwords), w1 = min(w0 + wb, nwords);
                    int nf = 0;
                    for (int w = w0; w < w1; ++w) nf += __popc(bm[w]);
                    int inc = nf;
#pragma unroll
                    for (int d = 1; d < 32; d <<= 1) {
                        const int y = __shfl_up_sync(kFull, inc, d);
                        if (lane >= d) inc += y;
                    }
                    int run = inc - nf;
                    for (int w = w0; w < w1; ++w) {
                        pre[w] = static_cast<uint16_t>(run);
                        run += __popc(bm[w]);
                    }
                    __syncwarp();
                    // each recorded entry's bit in its vector's mask (ranks < nown <= cap)
                    for (int e = lane; e < nown; e += 32) {
                        const int x = li_s[e], v = x >> 3;
                        const int r = pre[v >> 5] + __popc(bm[v >> 5] & ((1u << (v & 31)) - 1u));
                        atomicOr(&mk[r >> 2], (1u << (x & 7)) << (8 * (r & 3)));
                    }
                    __syncwarp();
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) hm = head_merge(hm, head_shfl(hm, off));
            if (__any_sync(kFull, dup)) flags |= SC_FLAG_DUP_ID;
            if (crank == 0 && __any_sync(kFull, bad)) flags |= SC_FLAG_BAD_ID;
            const int a_li = (sj >= lo && sj < hi) ? sj - lo : -1;
            if (lane == 0) {
                RowMeta* mt = meta + ms;
                mt->t = t;
                mt->sa = sj;
                mt->nown = nown;
                mt->a_li = a_li;
                mt->flags = flags;
                mt->A = row_A;
                mt->rl = row_rl;
                mt->qbest = hm.q;
                mt->omq = hm.omq;
                mt->oh = hm.oh;
                mt->ol = hm.ol;
                mt->kbest = hm.k;
            }
            // Published for the copy warp (which starts the slice's copies) and
            // the consumers, usually rows before they need it.
            __syncwarp();
            if (lane == 0) mbar_arrive(meta_bar(ms, kMetaFull));  // release: slot contents
            ++nfill;
        }
        {  // end marker for the zero warp (it leaves on its own if the queue stalls)
            const int z = static_cast<int>(nz % kZq);
            bool ok = true;
            if (nz >= static_cast<uint32_t>(kZq))
                ok = mbar_wait_bounded(zq_free(z), ((nz / kZq) - 1u) & 1u, wait_ns);
            if (__all_sync(kFull, ok) && lane == 0) {
                zq_t[z] = -1;
                mbar_arrive(zq_full(z));
            }
        }
        if (!stop) {  // end marker for the consumers
            const int ms = static_cast<int>(nfill % kMetaSlots);
            bool ok = true;
            if (nfill >= static_cast<uint32_t>(kMetaSlots))
                ok = mbar_wait_bounded(meta_bar(ms, kMetaFree), ((nfill / kMetaSlots) - 1u) & 1u, wait_ns);
            if (ok) {
                if (lane == 0) {
                    meta[ms].t = -1;
                    mbar_arrive(meta_bar(ms, kMetaFull));
                    ticket[ms] = -1;
                    mbar_arrive(ticket_bar(ms));
                }
            } else if (lane == 0) {
                status_or(a.status, SC_STATUS_TIMEOUT_LOAD);
            }
        }
    } else if (warp == NCW + 3) {
        // ================= copy warp: each valid row's slice into the stage =================
        // Takes the valid rows' indices in the row warp's order from the ticket
        // ring (published before their metadata is built) and starts the
        // slice's 1-D bulk copies chunk by chunk, each the moment the write pass
        // of the row before hands that chunk back.  The row warp's metadata work
        // (dependent global loads, padding rows in between) never sits between
        // a freed chunk and its refill.
        uint32_t nfill = 0;
        bool stop = false;
        for (;; ++nfill) {
            if (flag_up()) break;
            const int ms = static_cast<int>(nfill % kMetaSlots);
            if (!__all_sync(kFull, mbar_wait_bounded(ticket_bar(ms), (nfill / kMetaSlots) & 1u, wait_ns))) {
                give_up(SC_STATUS_TIMEOUT_LOAD);
                break;
            }
            const long long t = ticket[ms];  // read before the slot can be refilled (its row is not written yet)
            if (t < 0) break;                // end of the stream
            if (lane == 0) {
                const int ds = static_cast<int>(nfill % NB);
                const bool reuse = nfill >= static_cast<uint32_t>(NB);
                const uint32_t fpar = ((nfill / NB) - 1u) & 1u;
                const uint16_t* lrow = a.logits + t * a.lstride + lo;
                const uint32_t bs = smem_addr(smem + ds * L.stage_bytes);
                for (int i = 0; i < nchunks; ++i) {
                    if (reuse &&
                        !mbar_wait_bounded(data_bar(ds, kChunkFree + i), fpar, wait_ns)) {
                        for (int i2 = 0; i2 < i; ++i2)  // started copies land before the CTA leaves
                            (void)mbar_wait_bounded(data_bar(ds, kChunkFull + i2), (nfill / NB) & 1u,
                                                    kDrainLimitNs);
                        stop = true;
                        break;
                    }
                    // test hook: the first chunk of the first row is never copied,
                    // so every wait for it runs out (the failure path, with no fault)
                    if (a.stall && nfill == 0u && i == 0) continue;
                    fence_proxy_async_smem();
                    const int v0 = i * a.ncv, v1 = min(v0 + a.ncv, nvb);
                    const uint32_t bytes = static_cast<uint32_t>(v1 - v0) * 16u;
                    mbar_expect_tx(data_bar(ds, kChunkFull + i), bytes);
                    bulk_load(bs + 16u * v0, lrow + 8 * v0, bytes, data_bar(ds, kChunkFull + i), pol_keep);
                }
            }
            stop = __shfl_sync(kFull, static_cast<int>(stop), 0) != 0;
            if (stop) {
                give_up(SC_STATUS_TIMEOUT_LOAD);
                break;
            }
            if (lane == 0) *copied = nfill + 1u;
        }
        // copies still in flight land before the CTA can exit (bounded again)
        if (lane == 0) {
            const uint32_t f0 = nfill > static_cast<uint32_t>(NB) ? nfill - NB : 0u;
            for (uint32_t f = f0; f < nfill; ++f)
                for (int i = 0; i < nchunks; ++i)
                    if (!(a.stall && f == 0u && i == 0))  // (the copy the test hook left out)
                        (void)mbar_wait_bounded(data_bar(f % NB, kChunkFull + i), (f / NB) & 1u, kDrainLimitNs);
        }
        __syncwarp();
    } else if (warp == NCW + 2) {
        // ================= zero warp: zero rows from the row warp's queue =================
        for (uint32_t iz = 0;; ++iz) {
            const int z = static_cast<int>(iz % kZq);
            if (!__all_sync(kFull, mbar_wait_bounded(zq_full(z), (iz / kZq) & 1u, wait_ns))) {
                give_up(SC_STATUS_TIMEOUT_LOAD);
                break;
            }
            const long long t = zq_t[z];
            const uint32_t zf = zq_f[z];
            __syncwarp();
            if (t < 0) break;
            uint16_t* grow = a.grad + t * a.gstride + lo;
            for (int v = lane; v < nvb; v += 32) st_global_v4_hint(grow + 8 * v, 0u, 0u, 0u, 0u, pol);
            if (lane < tail) grow[n8 + lane] = 0;
            if (crank == 0 && lane == 0) {
                a.logp[t] = 0.0f;
                if (a.diag) {  // zeros and the flags, as four 16-byte stores
                    float4* dp = reinterpret_cast<float4*>(a.diag + t);
                    const float4 z4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    dp[0] = z4;
                    dp[1] = z4;
                    dp[2] = z4;
                    dp[3] = make_float4(0.0f, 0.0f, __uint_as_float(zf), 0.0f);
                }
                if (zf & SC_FLAG_DATA_ERRORS) status_or(a.status, SC_STATUS_DATA);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(zq_free(z));
        }
    } else if (warp == NCW) {
        // ================= scalar warp: records, exchange, row scalars =================
        for (uint32_t j = 0;; ++j) {
            if (flag_up()) break;
            const int p = static_cast<int>(j & 1u);
            const int ms = static_cast<int>(j % kMetaSlots);
            const int xi = static_cast<int>(j % kXBufs);
            // ---- while the streaming warps run phase A of row j: the recorded ids'
            // and a's logits and the recorded ids' sums relative to their maximum ----
            if (!__all_sync(kFull, mbar_wait_bounded(meta_bar(ms, kMetaFull), (j / kMetaSlots) & 1u, wait_ns))) {
                give_up(SC_STATUS_TIMEOUT_LOAD);
                break;
            }
            const RowMeta m = meta[ms];
            const int* li_s = list_li + ms * cap;
            const float* q_s = list_q + ms * cap;
            const float* fz = fix_z + p * cap;
            const int nown = m.nown, a_li = m.a_li;
            float Mo = -INFINITY, lH = 0.0f, EH = 0.0f, QY = 0.0f;
            auto head_sums = [&](float o_c) {  // owned recorded ids relative to o_c
                lH = 0.0f;
                EH = 0.0f;
                QY = 0.0f;
                for (int e = lane; e < nown; e += 32) {
                    const float y = fmaf(fz[e], kscale, -o_c);
                    const float ev = ex2(y);
                    lH += ev;
                    EH = fmaf(ev, y, EH);
                    QY = fmaf(q_s[e], y, QY);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    lH += __shfl_xor_sync(kFull, lH, off);
                    EH += __shfl_xor_sync(kFull, EH, off);
                    QY += __shfl_xor_sync(kFull, QY, off);
                }
            };
            if (m.t >= 0) {
                // The owned recorded ids' logits and a's, straight from global memory
                // (coherent loads: the gradient may alias the logits, but this row is
                // written only after its scalars): the record then waits for none of
                // the slice's copies and its merge is done before phase A ends.
                const uint16_t* lrow = a.logits + m.t * a.lstride + lo;
                float* fzw = fix_z + p * cap;
                float zmax = -INFINITY;
                for (int e = lane; e < nown; e += 32) {
                    const float z = bf_to_f(lrow[li_s[e]]);
                    fzw[e] = z;
                    zmax = fmaxf(zmax, z);
                }
                zmax = warp_max(zmax);
                if (lane == 0 && a_li >= 0) zav[p] = bf_to_f(lrow[a_li]);
                __syncwarp();
                Mo = zmax;  // the recorded ids' sums are relative to their own maximum
                if (Mo > -INFINITY) {
                    head_sums(Mo * kscale);
                } else if (nown > 0) {
                    // every recorded logit here is -inf: their sums carry the
                    // infinities (relative to 0), not a row offset of -inf
                    head_sums(0.0f);
                }
            }
            // ---- the write pass of row j - 1 is done in every streaming warp: its
            // row sum is complete (it rides with this row's record), and its special
            // entries can be patched once the scalars of row j are out ----
            float rs1 = 0.0f;
            if (j >= 1) {
                const bool wd = mbar_wait_bounded(wdone(static_cast<int>((j - 1) & 1u)), ((j - 1) >> 1) & 1u, wait_ns);
                if (!__all_sync(kFull, wd)) {
                    give_up(SC_STATUS_TIMEOUT_LOAD);
                    break;
                }
                rs1 = warp_sum(lane < NCW ? rsw[((j - 1) & 1u) * NCW + lane] : 0.0f) + corr_m1;
            }
            auto finish_prev = [&]() {
                if (j >= 1) {
                    patch_row(j - 1, t_m1);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(meta_bar(static_cast<int>((j - 1) % kMetaSlots), kMetaFree));
                }
            };
            if (m.t < 0) {  // end of the stream: the last row's sum goes to CTA 0 below
                finish_prev();
                fin_rs1 = rs1;
                nrows = j;
                clean_end = true;
                break;
            }
            // ---- this CTA's record of row j, to every CTA of the cluster (the
            // streaming warps send their own partials as they finish phase A) ----
            if (lane == 0) {
                mbar_expect_tx(xrec(xi), static_cast<uint32_t>(C * static_cast<int>(sizeof(CtaRec))));
                mbar_expect_tx(xpart(xi), static_cast<uint32_t>(C * NCW * static_cast<int>(sizeof(WarpPart))));
            }
            if (lane < C) {  // lane r sends the record to CTA r
                const uint32_t dst = map_to_rank(smem_addr(crec + xi * C + static_cast<int>(crank)), lane);
                const uint32_t rb = map_to_rank(xrec(xi), lane);
                const float za = a_li >= 0 ? zav[p] : 0.0f;
                st_async_v4(dst, __float_as_uint(Mo), __float_as_uint(lH), __float_as_uint(EH), __float_as_uint(QY), rb);
                st_async_v4(dst + 16u, __float_as_uint(rs1), __float_as_uint(m.oh), __float_as_uint(m.ol),
                            __float_as_uint(m.qbest), rb);
                st_async_v4(dst + 32u, static_cast<uint32_t>(m.kbest), static_cast<uint32_t>(nown), m.flags,
                            __float_as_uint(za), rb);
                st_async_v4(dst + 48u, a_li >= 0 ? 1u : 0u, __float_as_uint(m.omq), 0u, 0u, rb);
            }
            // ---- the C records of row j, usually in before phase A ends: merged
            // relative to their own largest offset Mh while the streaming partials
            // are still on their way.  Lane r < C takes the record of CTA r and a
            // butterfly of commutative steps sums the lanes, so every lane of every
            // CTA ends with the same bits. ----
            if (!__all_sync(kFull, mbar_wait_cluster_bounded(xrec(xi), (j / kXBufs) & 1u, wait_ns))) {
                give_up(SC_STATUS_TIMEOUT_EXCHANGE);
                break;
            }
            {
                const CtaRec* rp = crec + xi * C;
                // Every group of RP lanes (the power of two >= C) holds the C records,
                // lane r of a group record r, so log2(RP) butterfly steps leave the
                // same sums in every lane.
                const int RP = C <= 1 ? 1 : C <= 2 ? 2 : C <= 4 ? 4 : C <= 8 ? 8 : 16;
                const int rl = lane & (RP - 1);
                uint4 r0 = make_uint4(__float_as_uint(-INFINITY), 0u, 0u, 0u), r1 = make_uint4(0u, 0u, 0u, 0u),
                      r2 = make_uint4(0x7FFFFFFFu, 0u, 0u, 0u), r3 = make_uint4(0u, __float_as_uint(1.0f), 0u, 0u);
                if (rl < C) {
                    const uint32_t pa = smem_addr(rp + rl);
                    r0 = lds128(pa);
                    r1 = lds128(pa + 16u);
                    r2 = lds128(pa + 32u);
                    r3 = lds128(pa + 48u);
                }
                const float Hm = __uint_as_float(r0.x);
                const float Mh = warp_max(Hm);
                const int Pnval = static_cast<int>(r2.y);
                const float PlH = __uint_as_float(r0.y), PEH = __uint_as_float(r0.z), PQY = __uint_as_float(r0.w);
                const float Pqb = __uint_as_float(r1.w), Poh = __uint_as_float(r1.y), Pol = __uint_as_float(r1.z);
                float lH1 = 0.0f, EH1 = 0.0f, QY1 = 0.0f;
                if (Hm > -INFINITY) {
                    const float d = (Hm - Mh) * kscale;
                    const float f = ex2(d);
                    lH1 = f * PlH;
                    EH1 = f * fmaf(d, PlH, PEH);
                    if (Pnval > 0) QY1 = fmaf(d, (Pqb + Poh) + Pol, PQY);
                } else if (Pnval > 0) {  // (recorded logits of -inf: their infinities)
                    EH1 = PEH;
                    QY1 = PQY;
                }
                HeadMass hm{Pqb, static_cast<int>(r2.x), __uint_as_float(r3.y), Poh, Pol};
                for (int off = 1; off < RP; off <<= 1) {
                    lH1 += __shfl_xor_sync(kFull, lH1, off);
                    EH1 += __shfl_xor_sync(kFull, EH1, off);
                    QY1 += __shfl_xor_sync(kFull, QY1, off);
                    hm = head_merge(hm, head_shfl(hm, off));
                }
                const int nval = __reduce_add_sync(kFull, lane < RP ? Pnval : 0);  // one group's records
                uint32_t flags = __reduce_or_sync(kFull, r2.z);
                // the logit of a: only its owner's lane has nonzero bits
                const bool has_a = __reduce_or_sync(kFull, r3.x) != 0u;
                const float za = __uint_as_float(__reduce_or_sync(kFull, r3.x ? r2.w : 0u));
                // 1 - Q_H without cancellation: (1 - q_max), taken from its
                // log-probability, minus the others' mass
                float tail_mu = 1.0f, Q_H = 0.0f;
                if (nval > 0) {
                    tail_mu = (hm.omq - hm.oh) - hm.ol;
                    Q_H = (hm.q + hm.oh) + hm.ol;
                }
                // the previous row's sum, in CTA order (the order the end-of-stream
                // flush adds the last row's in)
                float rsum = 0.0f;
                for (int r = 0; r < C; ++r) rsum += rp[r].rs;

                // ---- the streaming partials of row j: the row scalars ----
                if (!__all_sync(kFull, mbar_wait_cluster_bounded(xpart(xi), (j / kXBufs) & 1u, wait_ns))) {
                    give_up(SC_STATUS_TIMEOUT_EXCHANGE);
                    break;
                }
                const WarpPart* wp = wpart + xi * C * NCW;
                const int NP = C * NCW;
                float mx = Mh;
                float lT = 0.0f, ET = 0.0f;
                if (NP <= 32) {  // (the usual case) one partial a lane, loaded once
                    const uint4 w = lane < NP ? lds128(smem_addr(wp + lane))
                                              : make_uint4(__float_as_uint(-INFINITY), 0u, 0u, 0u);
                    const float Pm = __uint_as_float(w.x);
                    const float o1 = warp_max(fmaxf(mx, Pm)) * kscale;
                    if (Pm > -INFINITY) {
                        const float d = Pm * kscale - o1;
                        const float f = ex2(d);
                        const float S1 = __uint_as_float(w.y), S2 = __uint_as_float(w.z);
                        lT = f * S1;
                        ET = f * fmaf(d, S1, S2);
                    }
                    mx = o1;
                } else if (NP <= 64) {  // (clusters of 5 to 8) two partials a lane, both loaded at once
                    const uint4 w0 = lds128(smem_addr(wp + lane));
                    const uint4 w1 = lane + 32 < NP ? lds128(smem_addr(wp + lane + 32))
                                                    : make_uint4(__float_as_uint(-INFINITY), 0u, 0u, 0u);
                    const float P0 = __uint_as_float(w0.x), P1 = __uint_as_float(w1.x);
                    const float o1 = warp_max(fmaxf(mx, fmaxf(P0, P1))) * kscale;
                    if (P0 > -INFINITY) {
                        const float d = P0 * kscale - o1;
                        const float f = ex2(d);
                        const float S1 = __uint_as_float(w0.y), S2 = __uint_as_float(w0.z);
                        lT = f * S1;
                        ET = f * fmaf(d, S1, S2);
                    }
                    if (P1 > -INFINITY) {
                        const float d = P1 * kscale - o1;
                        const float f = ex2(d);
                        const float S1 = __uint_as_float(w1.y), S2 = __uint_as_float(w1.z);
                        lT = fmaf(f, S1, lT);
                        ET = fmaf(f, fmaf(d, S1, S2), ET);
                    }
                    mx = o1;
                } else {
                    for (int q = lane; q < NP; q += 32) mx = fmaxf(mx, wp[q].m);
                    const float o1 = warp_max(mx) * kscale;
                    for (int q = lane; q < NP; q += 32) {
                        const uint4 w = lds128(smem_addr(wp + q));
                        const float Pm = __uint_as_float(w.x);
                        if (Pm > -INFINITY) {
                            const float d = Pm * kscale - o1;
                            const float f = ex2(d);
                            const float S1 = __uint_as_float(w.y), S2 = __uint_as_float(w.z);
                            lT = fmaf(f, S1, lT);
                            ET = fmaf(f, fmaf(d, S1, S2), ET);
                        }
                    }
                    mx = o1;
                }
                const float o = mx;  // the row's offset, scaled
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) lT += __shfl_xor_sync(kFull, lT, off);
                // the recorded ids' sums moved from Mh to the row offset
                const float dH = Mh > -INFINITY ? Mh * kscale - o : 0.0f;
                const float fH = Mh > -INFINITY ? ex2(dH) : 0.0f;
                const float lHg = fH * lH1;
                const float ya = has_a ? fmaf(za, kscale, -o) : 0.0f;
                // First what the write pass needs (bw, beta), published at once;
                // the diagnostics and the recorded ids' own gradients after.
                // (the MUFU logarithm and one correctly rounded reciprocal: a few ulp
                // on this path, which every later value of the row shares)
                const float l = lT + lHg;
                const float log2l = __log2f(l);
                const float inv_l = __frcp_rn(l);
                const float P_H = lHg * inv_l;
                const float tail_pi = lT * inv_l;
                const float rho = fmaxf(tail_mu, kTailFloor) * __frcp_rn(fmaxf(tail_pi, kTailFloor));
                const float s = a.centering ? tail_mu + rho * P_H : 1.0f;
                const float logp_a = (ya - log2l) * kLn2;
                const float dd = a.rollout ? logp_a - m.rl : 0.0f;
                // importance weight: w = exp(d) clipped, truncated or masked by mode
                const float A = m.A;
                const float w = a.is_mode != SC_IS_NONE ? expf(dd) : 1.0f;
                float wt = w;
                float wc = w;  // clipped GRPO: the clipped ratio
                if (a.is_mode == SC_IS_TIS) {
                    if (w > a.tis_max) {
                        wt = a.tis_max;
                        flags |= SC_FLAG_IS_TRUNC;
                    }
                } else if (a.is_mode == SC_IS_MIS) {
                    if (!(w >= a.mis_min && w <= a.mis_max)) {
                        wt = 0.0f;
                        flags |= SC_FLAG_IS_REJECT;
                    }
                } else if (a.is_mode == SC_IS_CLIP) {
                    // -min(w A, w_c A): the ratio's gradient where the unclipped
                    // term is the minimum, none where the clipped one is
                    wc = fminf(fmaxf(w, a.clip_lo), a.clip_hi);
                    if (!(wc == w || w * A < wc * A)) {
                        wt = 0.0f;
                        flags |= SC_FLAG_CLIPPED;
                    }
                }
                const float Aw = A * wt;
                const float alpha = -a.grad_scale * a.inv_t * Aw;
                const float beta = -alpha * s;
                const float bw = o + log2l;
                if (lane == 0) {  // (the one writer arrives: its stores are released with it)
                    scal[4 * p + 0] = bw;
                    scal[4 * p + 1] = beta;
                    mbar_arrive(sready(p));
                }
                finish_prev();  // the previous row's special entries, off the critical path

                // the rest of the sums
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ET += __shfl_xor_sync(kFull, ET, off);
                float EHg = EH1, QYg = QY1;
                if (Mh > -INFINITY) {
                    EHg = fH * fmaf(dH, lH1, EH1);
                    if (nval > 0) QYg = fmaf(dH, Q_H, QY1);
                }
                if (tail_pi < kTailFloor) flags |= SC_FLAG_CLAMP_PI;
                if (tail_mu < kTailFloor) flags |= SC_FLAG_CLAMP_MU;
                const float dsr = a.centering ? tail_mu - rho * tail_pi : 0.0f;  // s - rho
                const float k3 = a.rollout ? expm1f(dd) - dd : 0.0f;
                // sum_H c log p = sum_H q log p - rho sum_H p log p, each from the
                // merged sums: log p_k = (y_k - log2 l) ln 2.
                float csum = 0.0f;
                if (a.centering && nval > 0) {
                    const float qlogp = kLn2 * fmaf(-log2l, Q_H, QYg);
                    const float plogp = kLn2 * fmaf(-log2l, lHg, EHg) * inv_l;
                    csum = fmaf(-rho, plogp, qlogp);
                }
                const float loss = a.is_mode == SC_IS_CLIP ? -fminf(w * A, wc * A) : -Aw * (logp_a - csum);
                const float entropy = kLn2 * (log2l - (ET + EHg) * inv_l);
                const float g_a_free = alpha * (1.0f - s * ex2(ya - log2l));  // g_a when a is unrecorded
                // gradient at the owned recorded ids, and how far it is from the
                // beta p the write pass stores there (the row sum's correction)
                float* fv = fix_v + p * cap;
                float corr = 0.0f;
                bool a_rec = false;
                for (int e = lane; e < nown; e += 32) {
                    const float pe = ex2(fmaf(fz[e], kscale, -o) - log2l);
                    const float mu = a.centering ? fmaf(dsr, pe, q_s[e]) : pe;
                    const bool is_a = li_s[e] == a_li;
                    const float g = alpha * ((is_a ? 1.0f : 0.0f) - mu);
                    fv[e] = g;
                    corr += g - beta * ex2(fmaf(fz[e], kscale, -bw));
                    a_rec = a_rec || is_a;
                }
                corr = warp_sum(corr);
                if (a_li >= 0 && !__any_sync(kFull, a_rec))
                    corr += g_a_free - beta * ex2(fmaf(zav[p], kscale, -bw));
                corr_m1 = corr;
                if (lane == 0) {
                    scal[4 * p + 2] = g_a_free;  // read back by this warp when it patches the row
                    if (crank == 0) {
                        a.logp[m.t] = logp_a;
                        if (a.diag) {  // the record in field order, as four 16-byte stores
                            float4* dp = reinterpret_cast<float4*>(a.diag + m.t);
                            dp[0] = make_float4(loss, logp_a, P_H, tail_pi);
                            dp[1] = make_float4(Q_H, tail_mu, rho, s);
                            dp[2] = make_float4(entropy, k3, wt, 0.0f);
                            dp[3] = make_float4(A, __int_as_float(nval), __uint_as_float(flags), 0.0f);
                            // the records of row j carried the row sums of row j - 1
                            if (j >= 1) a.diag[t_m1].row_sum = rsum;
                        }
                        if (flags & SC_FLAG_DATA_ERRORS) status_or(a.status, SC_STATUS_DATA);
                    }
                }
            }
            t_m1 = m.t;
        }
    } else {
        // ================= streaming warps: phase A of row i, then its write pass =================
        for (uint32_t i = 0;; ++i) {
            if (flag_up()) break;
            const int ms = static_cast<int>(i % kMetaSlots);
            const bool got =
                mbar_wait_bounded(meta_bar(ms, kMetaFull), (i / kMetaSlots) & 1u, wait_ns);
            if (!__all_sync(kFull, got)) {
                give_up(SC_STATUS_TIMEOUT_LOAD);
                break;
            }
            const RowMeta m = meta[ms];
            if (m.t < 0) break;  // end of the stream: every row of this warp is written
            const int p = static_cast<int>(i & 1u);
            const int ds = static_cast<int>(i % NB);  // the row's data stage
            const uint32_t buf_s = smem_addr(smem + ds * L.stage_bytes);
            {
                // ------------- phase A: one pass over the slice in shared memory -------------
                const uint32_t fpar = (i / NB) & 1u;
                const uint32_t* bm = bitmap + ms * nwords;
                const uint16_t* pre = vpre + ms * nwords;
                const uint32_t* mk = vmask + ms * mwords;
                // VF: the recorded entries (8 bits) of a flagged vector j, fw its flag word
                auto rec_mask = [&](int j, uint32_t fw) {
                    const int r = pre[j >> 5] + __popc(fw & ((1u << (j & 31)) - 1u));
                    return (mk[r >> 2] >> (8 * (r & 3))) & 0xFFu;
                };
                auto rec_bits = [&](int j) -> uint32_t {  // the recorded entries of any vector j
                    if constexpr (VF) {
                        const uint32_t fw = bm[j >> 5];
                        return ((fw >> (j & 31)) & 1u) ? rec_mask(j, fw) : 0u;
                    } else {
                        return (bm[j >> 2] >> (8 * (j & 3))) & 0xFFu;
                    }
                };
                // The exponent offset is the largest logit among the slice's first 32
                // vectors -- every warp reads the same ones and reduces them the same
                // way, so the whole CTA shares it without a barrier -- fixed for the
                // whole pass: no running maximum to keep up to date, and the warp's
                // sums add up plainly.  Entries far above it would overflow 2^y, so a
                // thread whose sums come out too large or not finite redoes its own
                // vectors exactly (its maximum first).  Vectors holding a recorded id
                // take the rare per-entry path.
                bool timed_out = false;
                // The slice stays in its stage after the pass: the write pass reads
                // it again, and the scalar warp took the recorded ids' logits from it.
                float mz = -INFINITY;
                if (nchunks > 0) {  // (waits decided warp-wide)
                    timed_out = !__all_sync(kFull, mbar_wait_bounded(data_bar(ds, kChunkFull), fpar, wait_ns));
                    if (!timed_out && lane < nvb) {
                        const uint4 w = lds128(buf_s + 16u * lane);
                        const uint32_t mx = bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w));
                        mz = fmaxf(bf_lo(mx), bf_hi(mx));
                    }
                }
                mz = warp_max(mz);
                const bool fast = mz > -INFINITY;
                const float o = fast ? mz * kscale : 0.0f;
                // packed pairs: sum 2^y and sum 2^y y over the unrecorded entries
                const f2_t K2 = f2_pack(kscale, kscale), NO2 = f2_pack(-o, -o);
                f2_t S1a = 0ull, S1b = 0ull, S2a = 0ull, S2b = 0ull;
                float s1x = 0.0f, s2x = 0.0f;  // entries taken one by one
                for (int c = 0; c < nchunks && !timed_out; ++c) {
                    if (!__all_sync(kFull, mbar_wait_bounded(data_bar(ds, kChunkFull + c), fpar, wait_ns))) {
                        timed_out = true;
                        break;
                    }
                    const int v1 = min((c + 1) * a.ncv, nvb);
#pragma unroll 2
                    for (int j = c * a.ncv + tid; j < v1; j += NC) {
                        const uint4 w = lds128(buf_s + 16u * j);
                        uint32_t rbits, fw = 0u;
                        if constexpr (VF) {
                            fw = bm[j >> 5];
                            rbits = (fw >> (j & 31)) & 1u;  // nonzero: look up the mask below
                        } else {
                            rbits = (bm[j >> 2] >> (8 * (j & 3))) & 0xFFu;
                        }
                        if (rbits == 0u) {
                            f2_t y = f2_fma(bf2_to_f2(w.x), K2, NO2);
                            f2_t e = f2_ex2(y);
                            S1a = f2_add(S1a, e);
                            S2a = f2_fma(e, y, S2a);
                            y = f2_fma(bf2_to_f2(w.y), K2, NO2);
                            e = f2_ex2(y);
                            S1b = f2_add(S1b, e);
                            S2b = f2_fma(e, y, S2b);
                            y = f2_fma(bf2_to_f2(w.z), K2, NO2);
                            e = f2_ex2(y);
                            S1a = f2_add(S1a, e);
                            S2a = f2_fma(e, y, S2a);
                            y = f2_fma(bf2_to_f2(w.w), K2, NO2);
                            e = f2_ex2(y);
                            S1b = f2_add(S1b, e);
                            S2b = f2_fma(e, y, S2b);
                        } else {
                            if constexpr (VF) rbits = rec_mask(j, fw);
                            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float z = (q & 1) ? bf_hi(ww[q >> 1]) : bf_lo(ww[q >> 1]);
                                if (!((rbits >> q) & 1u)) {
                                    const float y = fmaf(z, kscale, -o);
                                    const float e = ex2(y);
                                    s1x += e;
                                    s2x = fmaf(e, y, s2x);
                                }
                            }
                        }
                    }
                }
                if (tail && tid == 0 && !timed_out) {  // entries past the last whole vector
                    const uint16_t* lrow = a.logits + m.t * a.lstride + lo;
                    const uint32_t tb = rec_bits(nvb);
                    for (int q = 0; q < tail; ++q) {
                        const int li = n8 + q;
                        if (!((tb >> q) & 1u)) {
                            const float y = fmaf(bf_to_f(lrow[li]), kscale, -o);
                            const float e = ex2(y);
                            s1x += e;
                            s2x = fmaf(e, y, s2x);
                        }
                    }
                }
                const f2_t S1 = f2_add(S1a, S1b), S2 = f2_add(S2a, S2b);
                Mass ms_acc{mz, (f2_lo(S1) + f2_hi(S1)) + s1x, (f2_lo(S2) + f2_hi(S2)) + s2x};
                const bool ok = fast && ms_acc.s1 <= 0x1p100f && fabsf(ms_acc.s2) <= 0x1p110f;
                if (!timed_out && !ok) {
                    // exact: this thread's maximum, then its sums relative to it (also
                    // the path of -inf logits, whose 0 * -inf made the fast sums NaN)
                    // (from the slice in its stage, which stays there until the write pass)
                    float mx = -INFINITY;
                    for (int j = tid; j < nvb; j += NC) {
                        const uint4 w = lds128(buf_s + 16u * j);
                        const uint32_t m2 = bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w));
                        mx = fmaxf(mx, fmaxf(bf_lo(m2), bf_hi(m2)));
                    }
                    float s1 = 0.0f, s2 = 0.0f;
                    if (mx > -INFINITY) {
                        const float ox = mx * kscale;
                        for (int j = tid; j < nvb; j += NC) {
                            const uint4 w = lds128(buf_s + 16u * j);
                            const uint32_t rbits = rec_bits(j);
                            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                if ((rbits >> q) & 1u) continue;
                                // (clamped so that a -inf logit adds 0, not 0 * -inf)
                                const float y = fmaxf(
                                    fmaf((q & 1) ? bf_hi(ww[q >> 1]) : bf_lo(ww[q >> 1]), kscale, -ox), -1024.0f);
                                const float e = ex2(y);
                                s1 += e;
                                s2 = fmaf(e, y, s2);
                            }
                        }
                    }
                    ms_acc = Mass{mx, s1, s2};
                    if (tail && tid == 0) {  // the tail again, relative to this maximum
                        const uint16_t* lrow = a.logits + m.t * a.lstride + lo;
                        const uint32_t tb = rec_bits(nvb);
                        for (int q = 0; q < tail; ++q) {
                            const int li = n8 + q;
                            if (!((tb >> q) & 1u))
                                ms_acc = mass_merge(ms_acc, Mass{bf_to_f(lrow[li]), 1.0f, 0.0f}, kscale);
                        }
                    }
                }
                if (__any_sync(kFull, timed_out)) {
                    give_up(SC_STATUS_TIMEOUT_LOAD);
                    break;
                }
                if (__all_sync(kFull, ok)) {  // one offset for the whole warp: plain sums
                    ms_acc.s1 = warp_sum(ms_acc.s1);
                    ms_acc.s2 = warp_sum(ms_acc.s2);
                } else {
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
                        ms_acc = mass_merge(ms_acc, mass_shfl(ms_acc, off), kscale);
                }
                // this warp's partial to every CTA of the cluster (lane r to CTA r)
                if (lane < C) {
                    const int xi = static_cast<int>(i % kXBufs);
                    const uint32_t dst =
                        map_to_rank(smem_addr(wpart + (xi * C + static_cast<int>(crank)) * NCW + warp), lane);
                    st_async_v4(dst, __float_as_uint(ms_acc.m), __float_as_uint(ms_acc.s1), __float_as_uint(ms_acc.s2),
                                0u, map_to_rank(xpart(xi), lane));
                }
            }
            {
                // ---- write pass of row i, once the cluster has its row scalars: g = beta p
                // (the special entries are patched by the scalar warp afterwards), the
                // slice read from its stage, every chunk handed back to the copy warp
                // as soon as this warp is done with it (the next row streams into it
                // while this one is written) ----
                const uint32_t ip = i;
                const int pp = p;
                const uint16_t* lrow = a.logits + m.t * a.lstride + lo;
                uint16_t* grow = a.grad + m.t * a.gstride + lo;
                const bool ready = mbar_wait_bounded(sready(pp), (ip >> 1) & 1u, wait_ns);
                if (!__all_sync(kFull, ready)) {
                    give_up(SC_STATUS_TIMEOUT_EXCHANGE);
                    break;
                }
                const float bw = scal[4 * pp + 0];
                const float beta = scal[4 * pp + 1];
                float rs = 0.0f;
                const f2_t K2 = f2_pack(kscale, kscale), NBW2 = f2_pack(-bw, -bw), BETA2 = f2_pack(beta, beta);
                f2_t RS = 0ull;
                auto emit = [&](int j, const uint4& w) {  // 8 gradients from 8 logits, in packed pairs
                    const f2_t g0 = f2_mul(f2_ex2(f2_fma(bf2_to_f2(w.x), K2, NBW2)), BETA2);
                    const f2_t g1 = f2_mul(f2_ex2(f2_fma(bf2_to_f2(w.y), K2, NBW2)), BETA2);
                    const f2_t g2 = f2_mul(f2_ex2(f2_fma(bf2_to_f2(w.z), K2, NBW2)), BETA2);
                    const f2_t g3 = f2_mul(f2_ex2(f2_fma(bf2_to_f2(w.w), K2, NBW2)), BETA2);
                    RS = f2_add(RS, f2_add(f2_add(g0, g1), f2_add(g2, g3)));
                    st_global_v4_hint(grow + 8 * j, pack_bf16x2(f2_lo(g0), f2_hi(g0)), pack_bf16x2(f2_lo(g1), f2_hi(g1)),
                                      pack_bf16x2(f2_lo(g2), f2_hi(g2)), pack_bf16x2(f2_lo(g3), f2_hi(g3)), pol);
                };
                for (int c = 0; c < nchunks; ++c) {
                    const int v1 = min((c + 1) * a.ncv, nvb);
#pragma unroll 2
                    for (int j = c * a.ncv + tid; j < v1; j += NC) emit(j, lds128(buf_s + 16u * j));
                    __syncwarp();
                    if (lane == 0) mbar_arrive(data_bar(ds, kChunkFree + c));
                }
                if (tail && tid == 0) {
                    for (int q = 0; q < tail; ++q) {
                        const int li = n8 + q;
                        const float g = beta * ex2(fmaf(bf_to_f(lrow[li]), kscale, -bw));
                        rs += g;
                        grow[li] = f_to_bf_bits(g);
                    }
                }
                rs = warp_sum(rs + (f2_lo(RS) + f2_hi(RS)));
                if (lane == 0) rsw[pp * NCW + warp] = rs;
                __syncwarp();
                if (lane == 0) mbar_arrive(wdone(pp));
            }
        }
    }

    // The row sums of the last two rows go to CTA 0 over DSMEM (the earlier
    // ones rode with later records); the final cluster barrier also keeps
    // every CTA's shared memory alive until no peer can still write to it.
    if (warp == NCW && lane == 0 && a.diag && clean_end)
        st_cluster_v2(map_to_rank(smem_addr(frs + crank), 0), __float_as_uint(fin_rs1), 0u);
    cluster_sync_all();
    if (crank == 0 && warp == NCW && lane == 0 && a.diag && clean_end) {
        float s1 = 0.0f;
        for (int r = 0; r < C; ++r) s1 += frs[r].x;
        if (nrows >= 1) a.diag[t_m1].row_sum = s1;
    }
    // The last CTA to finish leaves the workspace zeroed for the next launch
    // (every CTA is past its last row hand-out by now).
    if (tid == 0) {
        __threadfence();
        const unsigned long long done = atomicAdd(a.ws + 1, 1ull);
        if (done == static_cast<unsigned long long>(gridDim.x) - 1ull) {
            atomicExch(a.ws, 0ull);
            atomicExch(a.ws + 1, 0ull);
        }
    }
}

// ---- host side ----------------------------------------------------------

inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

struct Plan {
    int C, NC, S, ncv, NB;
    bool VF;  // recorded-id flags per 8-entry vector (else per entry)
    Layout L;
};

Layout make_layout(int S, int K_max, int NC, int NB, int C, bool vf) {
    Layout L;
    L.stage_bytes = round_up(S * 2, 128);
    L.list_cap = K_max > 0 ? K_max : 1;
    L.nwords = vf ? (S / 8 + 31) / 32 : (S + 31) / 32;
    L.mwords = vf ? (L.list_cap + 3) / 4 : 0;
    int off = NB * L.stage_bytes;
    auto take = [&](int bytes) {
        const int o = off;
        off = round_up(off + bytes, 16);
        return o;
    };
    L.off_meta = take(kMetaSlots * static_cast<int>(sizeof(RowMeta)));
    L.off_list_li = take(kMetaSlots * L.list_cap * 4);
    L.off_list_q = take(kMetaSlots * L.list_cap * 4);
    L.off_bitmap = take(kMetaSlots * L.nwords * 4);
    L.off_vpre = take(vf ? kMetaSlots * L.nwords * 2 : 0);
    L.off_vmask = take(kMetaSlots * L.mwords * 4);
    L.off_bars = take(num_bars(NB) * 8);
    L.off_wpart = take(kXBufs * C * (NC / 32) * static_cast<int>(sizeof(WarpPart)));
    L.off_rec = take(kXBufs * C * static_cast<int>(sizeof(CtaRec)));
    L.off_frs = take(kMaxCluster * 8);
    L.off_fixz = take(2 * L.list_cap * 4);
    L.off_fixv = take(2 * L.list_cap * 4);
    L.off_zav = take(2 * 4);
    L.off_rsw = take(2 * (NC / 32) * 4);
    L.off_scal = take(2 * 4 * 4);
    L.off_flag = take(8);
    L.off_grab = take(kGrab * 8);
    L.off_zq = take(kZq * 8);
    L.off_zqf = take(kZq * 4);
    L.off_ticket = take(kMetaSlots * 8);
    L.total = off;
    return L;
}

// A plan under one flag layout.  Automatic cluster size: the smallest cluster
// (up to 16 CTAs) whose CTAs fit two to an SM; one data stage that the write
// pass hands back chunk by chunk to the next row's copies; 256 streaming
// threads (128 for small slices).
int make_plan(int V, int K_max, int req_cluster, int req_threads, int req_stages, bool vf, Plan* out) {
    const int NB = req_stages > 0 ? req_stages : 1;
    int C = req_cluster;
    auto threads_for = [&](int S) {
        return req_threads > 0 ? req_threads : (S >= 8192 ? 256 : 128);
    };
    if (C <= 0) {
        // the smallest cluster whose CTAs fit two to an SM (the most bytes per
        // CTA that still leaves another CTA to cover each one's row exchange)
        C = kMaxCluster;
        for (int c = 1; c <= kMaxCluster; ++c) {
            const int Sc = round_up((V + c - 1) / c, 8);
            if (make_layout(Sc, K_max, threads_for(Sc), NB, c, vf).total <= kTwoPerSmBytes) {
                C = c;
                break;
            }
        }
        while (C > 1 && static_cast<long long>(C - 1) * round_up((V + C - 1) / C, 8) >= V) --C;
    }
    const int S = round_up((V + C - 1) / C, 8);
    const int NC = threads_for(S);
    const Layout L = make_layout(S, K_max, NC, NB, C, vf);
    if (L.total > kMaxSmem)
        return fail(SC_ERR_SHAPE,
                    "V = %d with cluster size %d and %d stages needs %d bytes of shared memory per CTA", V, C,
                    NB, L.total);
    const int nvb = S / 8;
    out->C = C;
    out->NC = NC;
    out->S = S;
    out->NB = NB;
    out->VF = vf;
    // chunks of a whole number of passes of the compute threads (every thread
    // has the same share of each chunk), at most kMaxChunks of them
    int ncv = NC * (kChunkVecTarget / NC > 1 ? kChunkVecTarget / NC : 1);
    if ((nvb + ncv - 1) / ncv > kMaxChunks) ncv = round_up((nvb + kMaxChunks - 1) / kMaxChunks, NC);
    out->ncv = ncv;
    out->L = L;
    return SC_OK;
}

using KernelFn = void (*)(KArgs);

KernelFn kernel_for(int NC, bool vf) {
    switch (NC) {
        case 128: return vf ? center_kernel<128, true> : center_kernel<128, false>;
        case 256: return vf ? center_kernel<256, true> : center_kernel<256, false>;
        case 384: return vf ? center_kernel<384, true> : center_kernel<384, false>;
        case 512: return vf ? center_kernel<512, true> : center_kernel<512, false>;
        default: return nullptr;
    }
}

std::mutex g_plan_mutex;
std::map<std::tuple<int, int, bool>, int> g_attr_set;                     // (device, NC, VF)
std::map<std::tuple<int, int, bool, int, int>, int> g_max_clusters;      // (device, NC, VF, C, smem)

// Sets the kernel's shared-memory and cluster attributes and returns the
// number of clusters that can be resident at once.
int prepare_kernel(int dev, const Plan& P, int* max_clusters) {
    KernelFn fn = kernel_for(P.NC, P.VF);
    if (!fn) return fail(SC_ERR_ARG, "threads = %d is not one of 128, 256, 384, 512", P.NC);
    std::lock_guard<std::mutex> lock(g_plan_mutex);
    cudaError_t e;
    auto key = std::make_tuple(dev, P.NC, P.VF);
    if (g_attr_set.find(key) == g_attr_set.end()) {
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic smem)");
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(non-portable cluster)");
        g_attr_set[key] = 1;
    }
    auto ckey = std::make_tuple(dev, P.NC, P.VF, P.C, P.L.total);
    auto cit = g_max_clusters.find(ckey);
    if (cit != g_max_clusters.end()) {
        *max_clusters = cit->second;
        return SC_OK;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(P.C, 1, 1);
    cfg.blockDim = dim3(P.NC + kAuxThreads, 1, 1);
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
    if (p->is_mode < SC_IS_NONE || p->is_mode > SC_IS_CLIP) return fail(SC_ERR_ARG, "is_mode = %d", p->is_mode);
    if (p->is_mode == SC_IS_CLIP) {
        if (p->centering) return fail(SC_ERR_ARG, "is_mode clip is defined with centering = 0");
        if (!(p->clip_low >= 0.0f && p->clip_low < 1.0f) || !(p->clip_high >= 0.0f) || !std::isfinite(p->clip_high))
            return fail(SC_ERR_ARG, "need 0 <= clip_low < 1 and finite clip_high >= 0");
    }
    if (p->is_mode == SC_IS_TIS && !(p->tis_max > 0.0f && std::isfinite(p->tis_max)))
        return fail(SC_ERR_ARG, "tis_max must be finite and > 0");
    if (p->is_mode == SC_IS_MIS &&
        !(p->mis_min >= 0.0f && p->mis_min <= p->mis_max && std::isfinite(p->mis_max)))
        return fail(SC_ERR_ARG, "need 0 <= mis_min <= mis_max < inf");
    if (p->centering != 0 && p->centering != 1) return fail(SC_ERR_ARG, "centering must be 0 or 1");
    if (p->cluster_size < 0 || p->cluster_size > kMaxCluster)
        return fail(SC_ERR_ARG, "cluster_size = %d outside 0..%d", p->cluster_size, kMaxCluster);
    if (p->threads != 0 && !kernel_for(p->threads, false))
        return fail(SC_ERR_ARG, "threads = %d is not 0, 128, 256, 384 or 512", p->threads);
    if (p->stages < 0 || p->stages > kMaxStages)
        return fail(SC_ERR_ARG, "stages = %d outside 0..%d", p->stages, kMaxStages);
    if (p->wait_limit_us < 0 || p->wait_limit_us > 60000000)
        return fail(SC_ERR_ARG, "wait_limit_us = %d outside 0..60000000", p->wait_limit_us);
    if (p->test_stall != 0 && p->test_stall != 1) return fail(SC_ERR_ARG, "test_stall must be 0 or 1");
    if (p->flag_layout < 0 || p->flag_layout > SC_FLAGS_VECTOR)
        return fail(SC_ERR_ARG, "flag_layout = %d is not 0, %d or %d", p->flag_layout, SC_FLAGS_ENTRY,
                    SC_FLAGS_VECTOR);
    return SC_OK;
}

// The plan for V and p on device dev, with its resident clusters.  A given
// flag layout, or a given cluster size, is kept (a given cluster size alone
// takes per-entry flags).  Otherwise each layout gets its smallest cluster
// that fits two CTAs to an SM, and the plan with more CTAs resident on the
// GPU wins, per-entry flags on a tie: per-vector flags free 15-20 KB of shared
// memory, which matters only where it lets a smaller cluster fill the SMs
// better (measured: 248320 entries, 5 CTAs x 58 clusters against 6 x 46, 6 %
// faster; at 151936 entries 3 x 97 against 4 x 74 was 13 % slower).
int plan_for(int dev, int V, const sc_params* p, Plan* P, int* mc) {
    if (p->flag_layout != 0 || p->cluster_size > 0) {
        int st = make_plan(V, p->K_max, p->cluster_size, p->threads, p->stages, p->flag_layout == SC_FLAGS_VECTOR, P);
        if (st != SC_OK) return st;
        return prepare_kernel(dev, *P, mc);
    }
    Plan pe, pv;
    int me = 0, mv = 0;
    int st = make_plan(V, p->K_max, 0, p->threads, p->stages, false, &pe);
    if (st != SC_OK) return st;
    st = prepare_kernel(dev, pe, &me);
    if (st != SC_OK) return st;
    *P = pe;
    *mc = me;
    if (make_plan(V, p->K_max, 0, p->threads, p->stages, true, &pv) == SC_OK && pv.C < pe.C &&
        prepare_kernel(dev, pv, &mv) == SC_OK && static_cast<long long>(mv) * pv.C > static_cast<long long>(me) * pe.C) {
        *P = pv;
        *mc = mv;
    }
    return ok();
}

}  // namespace
}  // namespace sc

extern "C" int sc_plan_query(int V, const sc_params* p, int* cluster_size, int* threads, int* slice,
                             int* smem_bytes, int* max_clusters, int* flag_layout) {
    using namespace sc;
    int st = check_params(V, p);
    if (st != SC_OK) return st;
    Plan P;
    // the shape checks of the requested (or per-entry automatic) plan need no device
    st = make_plan(V, p->K_max, p->cluster_size, p->threads, p->stages, p->flag_layout == SC_FLAGS_VECTOR, &P);
    if (st != SC_OK) return st;
    int dev = 0;
    st = check_device(&dev);
    if (st != SC_OK) return st;
    int mc = 0;
    st = plan_for(dev, V, p, &P, &mc);
    if (st != SC_OK) return st;
    if (cluster_size) *cluster_size = P.C;
    if (threads) *threads = P.NC;
    if (slice) *slice = P.S;
    if (smem_bytes) *smem_bytes = P.L.total;
    if (max_clusters) *max_clusters = mc;
    if (flag_layout) *flag_layout = P.VF ? SC_FLAGS_VECTOR : SC_FLAGS_ENTRY;
    return ok();
}

namespace sc {
namespace {

// A checked call of the fused kernel, ready to launch once it has a workspace.
struct CenterLaunch {
    KArgs ka;
    Plan P;
    long long G;  // clusters in the grid
};

// Every host-side check of sc_center_forward_backward (the workspace pointer
// only when `need_ws`) and the launch plan; writes nothing on the device.
int center_prepare(const uint16_t* logits, long long T, int V, long long logits_stride, const int32_t* rec_ids,
                   const float* rec_logprobs, const int32_t* rec_count, const int32_t* sampled_id,
                   const float* rollout_logprob, const int32_t* row_response, const float* adv, int n_resp,
                   const sc_params* p, uint16_t* grad_out, long long grad_stride, float* logp_out,
                   sc_row_diag* diag_out, uint32_t* status_dev, const void* workspace, bool need_ws,
                   CenterLaunch* out) {
    int st = check_params(V, p);
    if (st != SC_OK) return st;
    if (T < 0) return fail(SC_ERR_SHAPE, "T = %lld < 0", T);
    if (n_resp < 0) return fail(SC_ERR_SHAPE, "n_resp = %d < 0", n_resp);
    if (logits_stride < V || grad_stride < V)
        return fail(SC_ERR_SHAPE, "row strides (%lld, %lld) must be >= V = %d", logits_stride, grad_stride, V);
    if (p->is_mode != SC_IS_NONE && !rollout_logprob)
        return fail(SC_ERR_NULL, "is_mode tis/mis needs rollout_logprob");
    if (T == 0) return SC_OK;
    if (!logits || !sampled_id || !row_response || !grad_out || !logp_out || (need_ws && !workspace))
        return fail(SC_ERR_NULL, "logits, sampled_id, row_response, grad_out, logp_out and workspace are required");
    if (n_resp > 0 && !adv) return fail(SC_ERR_NULL, "adv is NULL with n_resp > 0");
    if (p->K_max > 0 && (!rec_ids || !rec_logprobs))
        return fail(SC_ERR_NULL, "rec_ids and rec_logprobs are required when K_max > 0");
    if (!aligned(logits, 16) || !aligned(grad_out, 16))
        return fail(SC_ERR_ALIGN, "logits and grad_out must be 16-byte aligned");
    if (logits_stride % 8 != 0 || grad_stride % 8 != 0)
        return fail(SC_ERR_ALIGN, "row strides must be multiples of 8 elements");
    if (!aligned(rec_ids, 4) || !aligned(rec_logprobs, 4) || !aligned(rec_count, 4) ||
        !aligned(sampled_id, 4) || !aligned(rollout_logprob, 4) || !aligned(row_response, 4) ||
        !aligned(adv, 4) || !aligned(logp_out, 4) || !aligned(diag_out, 16) || !aligned(status_dev, 4) ||
        !aligned(workspace, 16))
        return fail(SC_ERR_ALIGN, "metadata arrays must be 4-byte aligned, diag_out and workspace 16-byte aligned");
    {
        const char* l0 = reinterpret_cast<const char*>(logits);
        const char* g0 = reinterpret_cast<const char*>(grad_out);
        const long long lb = 2LL * ((T - 1) * logits_stride + V);
        const long long gb = 2LL * ((T - 1) * grad_stride + V);
        const bool same = (l0 == g0) && (logits_stride == grad_stride);
        if (!same && l0 < g0 + gb && g0 < l0 + lb)
            return fail(SC_ERR_ARG, "grad_out overlaps logits other than exactly (in place)");
    }
    Plan& P = out->P;
    // the shape checks of the requested (or per-entry automatic) plan need no device
    st = make_plan(V, p->K_max, p->cluster_size, p->threads, p->stages, p->flag_layout == SC_FLAGS_VECTOR, &P);
    if (st != SC_OK) return st;
    int dev = 0;
    st = check_device(&dev);
    if (st != SC_OK) return st;
    int mc = 0;
    st = plan_for(dev, V, p, &P, &mc);
    if (st != SC_OK) return st;
    const long long G = T < mc ? T : mc;
    out->G = G;
    // About the last eighth of the rows are handed out at run time (the rest,
    // rounded down to a multiple of the clusters, are dealt round robin).
    const long long T_static = (T - (T + kDynamicShare - 1) / kDynamicShare) / G * G;

    KArgs& ka = out->ka;
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
    ka.ws = nullptr;
    ka.T_static = T_static;
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
    ka.clip_lo = 1.0f - p->clip_low;
    ka.clip_hi = 1.0f + p->clip_high;
    ka.wait_ns = p->wait_limit_us > 0 ? 1000ull * static_cast<unsigned long long>(p->wait_limit_us) : kWaitLimitNs;
    ka.stall = p->test_stall;
    ka.C = P.C;
    ka.S = P.S;
    ka.ncv = P.ncv;
    ka.NB = P.NB;
    ka.L = P.L;
    return SC_OK;
}

int center_launch(CenterLaunch& cl, void* workspace, cudaStream_t stream) {
    const Plan& P = cl.P;
    cl.ka.ws = static_cast<unsigned long long*>(workspace);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cl.G * P.C), 1, 1);
    cfg.blockDim = dim3(P.NC + kAuxThreads, 1, 1);
    cfg.dynamicSmemBytes = P.L.total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = P.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // the kernel's shared-memory set-up may overlap the previous kernel's tail
    // (the kernel waits for it before reading any input)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel_for(P.NC, P.VF), cl.ka);
    if (e != cudaSuccess) return cuda_fail(e, "center_kernel launch");
    return ok();
}

}  // namespace
}  // namespace sc

extern "C" int sc_center_forward_backward(const uint16_t* logits, long long T, int V,
                                          long long logits_stride, const int32_t* rec_ids,
                                          const float* rec_logprobs, const int32_t* rec_count,
                                          const int32_t* sampled_id, const float* rollout_logprob,
                                          const int32_t* row_response, const float* adv, int n_resp,
                                          const sc_params* p, uint16_t* grad_out, long long grad_stride,
                                          float* logp_out, sc_row_diag* diag_out, uint32_t* status_dev,
                                          void* workspace, sc_stream_t stream) {
    using namespace sc;
    CenterLaunch cl;
    const int st = center_prepare(logits, T, V, logits_stride, rec_ids, rec_logprobs, rec_count, sampled_id,
                                  rollout_logprob, row_response, adv, n_resp, p, grad_out, grad_stride, logp_out,
                                  diag_out, status_dev, workspace, true, &cl);
    if (st != SC_OK) return st;
    if (T == 0) return ok();
    return center_launch(cl, workspace, reinterpret_cast<cudaStream_t>(stream));
}

// ---- the same call for callers that cannot allocate -----------------------
//
// Some callers are handed their input and output buffers and nothing else --
// for instance a plugin running inside another framework whose memory planner
// has already placed every buffer, or an embedded runtime that reserves all of
// its device memory at start-up -- and have no way to obtain the small
// workspace sc_center_forward_backward needs.  This variant keeps that
// workspace in the library itself: a fixed array in device memory, present on
// every GPU that loads the library until the process exits.

namespace {

// Room for the workspace of one call (SC_WORKSPACE_BYTES); every call shares it.
static __device__ __align__(256) unsigned char g_center_scratch[256];

}  // namespace

extern "C" int sc_center_forward_backward_noalloc(const uint16_t* logits, long long T, int V,
                                                  long long logits_stride, const int32_t* rec_ids,
                                                  const float* rec_logprobs, const int32_t* rec_count,
                                                  const int32_t* sampled_id, const float* rollout_logprob,
                                                  const int32_t* row_response, const float* adv, int n_resp,
                                                  const sc_params* p, uint16_t* grad_out, long long grad_stride,
                                                  float* logp_out, sc_row_diag* diag_out, uint32_t* status_dev,
                                                  sc_stream_t stream) {
    using namespace sc;
    // The scratch a call needs does not depend on T, V or K_max; the check
    // below refuses the call only if the workspace ever outgrew the array.
    if (SC_WORKSPACE_BYTES > static_cast<int>(sizeof(g_center_scratch)))
        return fail(SC_ERR_SHAPE, "the workspace (%d bytes) exceeds the library's scratch array (%d bytes)",
                    SC_WORKSPACE_BYTES, static_cast<int>(sizeof(g_center_scratch)));
    // every argument is checked before the array is touched
    CenterLaunch cl;
    const int st = center_prepare(logits, T, V, logits_stride, rec_ids, rec_logprobs, rec_count, sampled_id,
                                  rollout_logprob, row_response, adv, n_resp, p, grad_out, grad_stride, logp_out,
                                  diag_out, status_dev, nullptr, false, &cl);
    if (st != SC_OK) return st;
    if (T == 0) return ok();
    // The array's device address on the current device (the array's name in
    // host code is only a stand-in for it).  Looked up on every call: it is a
    // table lookup after the first, and stays right if the module was reloaded.
    void* scratch = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&scratch, g_center_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    // The row counter must start at zero: clear it in stream order (the array
    // keeps whatever the previous call, or a failed one, left in it).
    e = cudaMemsetAsync(scratch, 0, SC_WORKSPACE_BYTES, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(scratch)");
    return center_launch(cl, scratch, reinterpret_cast<cudaStream_t>(stream));
}
