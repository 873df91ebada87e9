// sc_topk.cu -- sampler-side capture of the top-K behaviour probabilities.
//
// What the sampler records per generated position (Agent Lightning docs page
// "Score Centering", section "Score Centering": the top K behaviour
// probabilities of the sampling call, with their original normalisation):
// mu = softmax(z * inv_t) over the V sampler logits, or with top_p < 1 that
// distribution restricted to its nucleus (the shortest prefix of the entries
// sorted by probability whose preceding mass is below top_p) and
// renormalised.  Entries are ordered by z, larger first, equal values by
// lower id.  Each row gets count = min(K, V, nucleus size) ids and log mu.
//
// GB300 design: a persistent grid of 512-thread CTAs, each split into two
// 256-thread groups that take rows independently (named barriers), so that one
// group's per-row sorting and reductions overlap the other's streaming.
// One-pass path (almost every row): a 1/16 sample sets the exponent offset and
// a candidate threshold; one pass over the row sums the softmax normaliser
// (compensated, fixed order) and collects the entries above the threshold;
// the candidates are sorted and give the top K and the nucleus (see fast_row).
// Exact path (rows the one-pass path cannot finish, taken by the whole CTA
// between rounds): radix selection on an order-preserving 32-bit key of z in
// digits of 12, 12 and 8 bits.
//   pass 1  row maximum and the 4096-bin histogram of the top digit;
//   pass 2  the softmax normaliser in 2^-40 fixed point (integer sums, so
//           the result does not depend on the order of the additions), the
//           per-bin mass histogram (top_p < 1), and the candidates: every
//           entry at or above the bin holding the K-th largest key, when
//           they fit the shared-memory buffer (a few hundred for real rows);
//   then    a block-wide bitonic sort of the candidates by (key, id).
// Crowded bins (many equal or nearly equal values) take further histogram
// passes on the next digits; a top-p crossing below the candidates takes one
// more pass (more when its bin is crowded).  Every pass reads the row with
// 16-byte loads; the row itself never needs to fit on chip.
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>

#include "sc_device.cuh"
#include "sc_internal.h"

namespace sc {
namespace {

constexpr int kNT = 512;           // threads per CTA
constexpr int kBins = 4096;        // bins of the 12-bit digits
constexpr int kCap = 2048;         // candidate buffer (entries)
constexpr int kMaxTopK = 1024;
constexpr double kFix = 1099511627776.0;  // 2^40: fixed-point unit of the probabilities
constexpr float kLog2e = 1.4426950408889634f;

struct TopkArgs {
    const float* logits;
    long long T, stride;
    int V, K;
    float inv_t, top_p;
    int32_t* ids;
    float* lps;
    int32_t* counts;
    unsigned long long* ws;  // run-time hand-out: [2] rows taken past T_static, [3] CTAs finished (or NULL)
    long long T_static;      // rows dealt round robin to the thread groups (all of them without ws)
};

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// read-only 16-byte global load with an L2 eviction hint
// 16 bytes global -> shared memory, asynchronous, under an L2 policy; the
// executing thread waits for its own copies (cp.async.wait_group)
__device__ __forceinline__ void cp_async16_hint(uint32_t dst, const void* src, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ float4 ldg_f4_hint(const float4* ptr, uint64_t policy) {
    float4 v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(ptr), "l"(policy));
    return v;
}

// Order-preserving key: a larger float gives a larger key (-0 counts as +0).
__device__ __forceinline__ uint32_t key_of(float z) {
    uint32_t b = __float_as_uint(z == 0.0f ? 0.0f : z);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float float_of(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// Digit `level` of a key (0: bits 31..20, 1: bits 19..8, 2: bits 7..0) and
// the bits above it.
__device__ __forceinline__ int digit_of(uint32_t k, int level) {
    return level == 0 ? static_cast<int>(k >> 20) : (level == 1 ? static_cast<int>((k >> 8) & 0xFFFu) : static_cast<int>(k & 0xFFu));
}
__device__ __forceinline__ uint32_t prefix_of(uint32_t k, int level) {
    return level == 0 ? 0u : (level == 1 ? (k >> 20) : (k >> 8));
}
__device__ __forceinline__ int digit_bins(int level) { return level == 2 ? 256 : kBins; }
// The smallest key whose digits down to `level` are (prefix, d).
__device__ __forceinline__ uint32_t lower_key(uint32_t prefix, int d, int level) {
    return level == 0 ? (static_cast<uint32_t>(d) << 20)
                      : (level == 1 ? ((prefix << 20) | (static_cast<uint32_t>(d) << 8)) : ((prefix << 8) | static_cast<uint32_t>(d)));
}

// Probability of logit z relative to the row maximum, and in fixed point.
__device__ __forceinline__ float rel_mass(float z, float mz, float kt) {
    const float y = (z - mz) * kt;
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(y));
    return e;
}
__device__ __forceinline__ unsigned long long to_fixed(float e) {
    return __float2ull_rz(e * 1099511627776.0f);  // exact scaling by 2^40 (e <= 1)
}
__device__ __forceinline__ unsigned long long fixed_q(float z, float mz, float kt) { return to_fixed(rel_mass(z, mz, kt)); }

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int mask) {
    const uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), mask);
    const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), mask);
    return (static_cast<unsigned long long>(hi) << 32) | lo;
}
__device__ __forceinline__ unsigned long long shfl_u64(unsigned long long v, int src) {
    const uint32_t lo = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), src);
    const uint32_t hi = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), src);
    return (static_cast<unsigned long long>(hi) << 32) | lo;
}
__device__ __forceinline__ unsigned long long shfl_up_u64(unsigned long long v, int d) {
    const uint32_t lo = __shfl_up_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), d);
    const uint32_t hi = __shfl_up_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), d);
    return (static_cast<unsigned long long>(hi) << 32) | lo;
}

struct Shared {
    uint32_t hist0[kBins];              // counts of the top digit (pass 1)
    float mhf[kBins];                   // masses of the top digit, FP32 (guides the top-p search)
    uint32_t hist[kBins];               // counts of a refining digit
    unsigned long long mhist[kBins];    // exact fixed-point masses of a refining digit
    unsigned long long cand[kCap];      // (key << 32) | ~id, sorted descending
    unsigned long long top[kMaxTopK];   // the selected entries, sorted
    unsigned long long scan[kNT / 32];  // block scan scratch
    unsigned long long s_fixed;         // the row's normaliser, fixed point
    uint32_t maxkey;
    int ncand;
    int found_bin;                      // result of find_from_top
    unsigned long long found_above;     // sum over the bins above it
    int tie_taken;
};

// Exclusive prefix sum over the threads of the block, in thread order.
__device__ unsigned long long block_exclusive_scan(Shared& sh, unsigned long long v, unsigned long long* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long y = shfl_up_u64(x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) sh.scan[warp] = x;
    __syncthreads();
    unsigned long long before = 0, all = 0;
    for (int w = 0; w < kNT / 32; ++w) {
        const unsigned long long t = sh.scan[w];
        if (w < warp) before += t;
        all += t;
    }
    __syncthreads();
    if (total) *total = all;
    return before + x - v;
}

// The bin b (of `nbins`, scanning from the top) where the running sum of
// `vals` reaches `target`: sum(bins above b) < target <= sum(bins above b) +
// vals[b].  Writes found_bin / found_above; -1 if the total is below target.
template <typename T>
__device__ void find_from_top(Shared& sh, const T* vals, int nbins, double target) {
    const int per = (nbins + kNT - 1) / kNT;
    // thread i owns bins nbins-1-i*per ... (descending)
    const int hi = nbins - 1 - static_cast<int>(threadIdx.x) * per;
    unsigned long long local = 0;
    for (int j = 0; j < per; ++j) {
        const int b = hi - j;
        if (b >= 0) local += static_cast<unsigned long long>(vals[b]);
    }
    if (threadIdx.x == 0) sh.found_bin = -1;
    unsigned long long total = 0;
    unsigned long long run = block_exclusive_scan(sh, local, &total);
    for (int j = 0; j < per; ++j) {
        const int b = hi - j;
        if (b < 0) break;
        const unsigned long long v = static_cast<unsigned long long>(vals[b]);
        if (static_cast<double>(run) < target && target <= static_cast<double>(run + v)) {
            sh.found_bin = b;
            sh.found_above = run;
        }
        run += v;
    }
    __syncthreads();
}

// Every entry of the row, f(z, id): 16-byte loads, kUnroll of them in flight
// per thread before any is used (every caller's f is order-independent).
constexpr int kUnroll = 4;
template <typename F>
__device__ __forceinline__ void for_each_entry(const float* row, int V, F&& f) {
    const int nv4 = V >> 2;
    const float4* r4 = reinterpret_cast<const float4*>(row);
    int i = threadIdx.x;
    for (; i + (kUnroll - 1) * kNT < nv4; i += kUnroll * kNT) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = __ldg(r4 + i + u * kNT);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int b = 4 * (i + u * kNT);
            f(v[u].x, b);
            f(v[u].y, b + 1);
            f(v[u].z, b + 2);
            f(v[u].w, b + 3);
        }
    }
    for (; i < nv4; i += kNT) {
        const float4 v = __ldg(r4 + i);
        f(v.x, 4 * i);
        f(v.y, 4 * i + 1);
        f(v.z, 4 * i + 2);
        f(v.w, 4 * i + 3);
    }
    for (int j = (nv4 << 2) + static_cast<int>(threadIdx.x); j < V; j += kNT) f(__ldg(row + j), j);
}

__device__ __forceinline__ unsigned long long pack_entry(uint32_t key, int id) {
    return (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(id));
}

// Appends every entry whose key is at least `lo` (and, if `hi_excl` is set,
// below it) to the candidate buffer; the count may exceed the buffer, which
// the caller checks.
__device__ void collect(Shared& sh, const float* row, int V, uint32_t lo, uint32_t hi, bool bounded) {
    for_each_entry(row, V, [&](float z, int id) {
        const uint32_t k = key_of(z);
        if (k >= lo && (!bounded || k < hi)) {
            const int pos = atomicAdd(&sh.ncand, 1);
            if (pos < kCap) sh.cand[pos] = pack_entry(k, id);
        }
    });
    __syncthreads();
}

// Bitonic sort of cand[0, n), larger first (n <= kCap).
__device__ void sort_desc(Shared& sh, int n) {
    int m = 1;
    while (m < n) m <<= 1;
    for (int i = n + static_cast<int>(threadIdx.x); i < m; i += kNT) sh.cand[i] = 0ull;
    __syncthreads();
    for (int k = 2; k <= m; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < m; i += kNT) {
                const int l = i ^ j;
                if (l > i) {
                    const unsigned long long x = sh.cand[i], y = sh.cand[l];
                    if (((i & k) == 0) ? (x < y) : (x > y)) {
                        sh.cand[i] = y;
                        sh.cand[l] = x;
                    }
                }
            }
            __syncthreads();
        }
}

// Histogram of digit `level` over the entries whose higher digits equal
// `pfx`: counts, and masses when `masses` is set.
__device__ void digit_hist(Shared& sh, const float* row, int V, int level, uint32_t pfx, bool masses, float mz,
                           float kt) {
    const int nb = digit_bins(level);
    for (int i = threadIdx.x; i < nb; i += kNT) {
        sh.hist[i] = 0u;
        if (masses) sh.mhist[i] = 0ull;
    }
    __syncthreads();
    for_each_entry(row, V, [&](float z, int id) {
        const uint32_t k = key_of(z);
        if (prefix_of(k, level) == pfx) {
            const int d = digit_of(k, level);
            atomicAdd(&sh.hist[d], 1u);
            if (masses) atomicAdd(&sh.mhist[d], fixed_q(z, mz, kt));
        }
    });
    __syncthreads();
}

// Appends, in id order, the first `need` entries whose key equals `key`
// (after `sh.ncand` entries already there).
__device__ void collect_ties_in_id_order(Shared& sh, const float* row, int V, uint32_t key, int need) {
    if (threadIdx.x == 0) sh.tie_taken = 0;
    __syncthreads();
    for (int base = 0; base < V; base += kNT * 4) {
        // thread i looks at ids base + 4i .. base + 4i + 3
        int my[4];
        int n = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int id = base + 4 * static_cast<int>(threadIdx.x) + c;
            if (id < V && key_of(__ldg(row + id)) == key) my[n++] = id;
        }
        unsigned long long total = 0;
        const int before = static_cast<int>(block_exclusive_scan(sh, static_cast<unsigned long long>(n), &total));
        const int taken = sh.tie_taken;
        for (int c = 0; c < n; ++c)
            if (taken + before + c < need) sh.cand[sh.ncand + taken + before + c] = pack_entry(key, my[c]);
        __syncthreads();
        if (threadIdx.x == 0) sh.tie_taken = taken + static_cast<int>(total);
        __syncthreads();
        if (sh.tie_taken >= need) break;
    }
    if (threadIdx.x == 0) sh.ncand += need;
    __syncthreads();
}

// Leaves in cand[0, n) -- sorted, larger first -- the entries of the row
// whose key is at least the `target`-th largest, ties at that key taken in
// id order so that exactly `target` ... n entries remain: n == target when the
// buffer had to be filled tie by tie, else every entry of the group that
// holds the target-th key (and more).  Uses hist / mhist as scratch.
// Returns n.
__device__ int select_top(Shared& sh, const float* row, int V, int target, int level0_bin,
                          unsigned long long level0_above, bool level0_collected, float mz, float kt) {
    if (!level0_collected) {
        uint32_t pfx = static_cast<uint32_t>(level0_bin);
        unsigned long long above = level0_above;
        for (int level = 1; level <= 2; ++level) {
            digit_hist(sh, row, V, level, pfx, false, mz, kt);
            find_from_top(sh, sh.hist, digit_bins(level), static_cast<double>(target) - static_cast<double>(above));
            const int b = sh.found_bin;
            above += sh.found_above;
            const unsigned long long group = sh.hist[b];
            __syncthreads();  // every thread has read this step's results
            if (threadIdx.x == 0) sh.ncand = 0;
            __syncthreads();
            if (above + group <= static_cast<unsigned long long>(kCap)) {
                collect(sh, row, V, lower_key(pfx, b, level), 0u, false);
                break;
            }
            if (level == 2) {  // one key value shared by too many entries
                const uint32_t key = lower_key(pfx, b, 2);
                if (key < 0xFFFFFFFFu) collect(sh, row, V, key + 1u, 0u, false);
                collect_ties_in_id_order(sh, row, V, key, target - static_cast<int>(above));
                break;
            }
            pfx = (pfx << 12) | static_cast<uint32_t>(b);
        }
    }
    const int n = min(sh.ncand, kCap);
    __syncthreads();
    sort_desc(sh, n);
    return n;
}

// The nucleus mass (fixed point) within the top-digit group b0 (exact mass of
// every entry above it: `above`), for a group too crowded to sort at once:
// narrowed digit by digit on exact fixed-point mass histograms.
__device__ unsigned long long refine_crossing(Shared& sh, const float* row, int V, int b0, unsigned long long above,
                                            double thr, float mz, float kt) {
    uint32_t pfx = static_cast<uint32_t>(b0);
    uint32_t lo = static_cast<uint32_t>(b0) << 20, span = 1u << 20;
    for (int level = 0;; ++level) {
        __syncthreads();  // every thread has read the caller's / last step's results
        if (threadIdx.x == 0) {
            sh.ncand = 0;
            sh.found_above = ~0ull;  // smallest running mass >= thr seen so far
        }
        __syncthreads();
        const bool bounded = lo + span != 0u;  // the group ends below the largest key
        collect(sh, row, V, lo, lo + span, bounded);
        const int n = sh.ncand;
        if (n <= kCap) {
            sort_desc(sh, n);
            const int per = (n + kNT - 1) / kNT;
            unsigned long long local = 0;
            for (int j = 0; j < per; ++j) {
                const int i = static_cast<int>(threadIdx.x) * per + j;
                if (i < n) local += fixed_q(float_of(static_cast<uint32_t>(sh.cand[i] >> 32)), mz, kt);
            }
            unsigned long long total = 0;
            unsigned long long run = above + block_exclusive_scan(sh, local, &total);
            for (int j = 0; j < per; ++j) {
                const int i = static_cast<int>(threadIdx.x) * per + j;
                if (i >= n) break;
                if (static_cast<double>(run) >= thr) atomicMin(&sh.found_above, run);
                run += fixed_q(float_of(static_cast<uint32_t>(sh.cand[i] >> 32)), mz, kt);
            }
            if (threadIdx.x == 0 && static_cast<double>(above + total) >= thr) atomicMin(&sh.found_above, above + total);
            __syncthreads();
            const unsigned long long P = sh.found_above;
            __syncthreads();
            return P == ~0ull ? above + total : P;
        }
        if (level == 2) {
            // one key value held by more entries than fit: all have the same mass q
            const unsigned long long q = fixed_q(float_of(lo), mz, kt);
            double need = q > 0 ? ceil((thr - static_cast<double>(above)) / static_cast<double>(q)) : 0.0;
            if (need > n) need = n;
            if (need < 0) need = 0;
            return above + static_cast<unsigned long long>(need) * q;
        }
        digit_hist(sh, row, V, level + 1, pfx, true, mz, kt);
        find_from_top(sh, sh.mhist, digit_bins(level + 1), thr - static_cast<double>(above));
        const int b = sh.found_bin;
        if (b < 0) return above;  // not reached: the group's mass crosses thr
        above += sh.found_above;
        if (level == 0) {
            lo = (pfx << 20) | (static_cast<uint32_t>(b) << 8);
            span = 1u << 8;
            pfx = (pfx << 12) | static_cast<uint32_t>(b);
        } else {
            lo = (pfx << 8) | static_cast<uint32_t>(b);
            span = 1u;
        }
    }
}

// The next top-digit bin above (dir = +1) or below (dir = -1) b that holds
// entries, -1 if none.
__device__ int next_bin(const Shared& sh, int b, int dir) {
    for (b += dir; b >= 0 && b < kBins; b += dir)
        if (sh.hist0[b]) return b;
    return -1;
}

// The nucleus mass (fixed point): the running mass of the sorted row before
// the first entry whose preceding mass reaches thr.  `bp` is the top-digit
// bin where the FP32 mass histogram puts the crossing; one pass collects that
// bin's entries and sums the exact mass above it, and the sorted walk finds
// the crossing, moving to the neighbouring bin when rounding of the FP32
// histogram pointed to the wrong one.
__device__ unsigned long long crossing_mass(Shared& sh, const float* row, int V, int bp, double thr, float mz,
                                            float kt, unsigned long long s_all) {
    for (int tries = 0; tries < kBins && bp >= 0; ++tries) {
        __syncthreads();
        if (threadIdx.x == 0) {
            sh.ncand = 0;
            sh.found_above = ~0ull;
        }
        __syncthreads();
        const uint32_t lo = static_cast<uint32_t>(bp) << 20;
        const bool top_group = bp == kBins - 1;
        const uint32_t hi = top_group ? 0u : static_cast<uint32_t>(bp + 1) << 20;
        unsigned long long local = 0ull;
        for_each_entry(row, V, [&](float z, int id) {
            const uint32_t k = key_of(z);
            if (!top_group && k >= hi) {
                local += fixed_q(z, mz, kt);
            } else if (k >= lo) {
                const int pos = atomicAdd(&sh.ncand, 1);
                if (pos < kCap) sh.cand[pos] = pack_entry(k, id);
            }
        });
        unsigned long long above = 0ull;
        (void)block_exclusive_scan(sh, local, &above);
        const int n = sh.ncand;
        if (static_cast<double>(above) >= thr) {  // the crossing lies above this bin
            bp = next_bin(sh, bp, +1);
            continue;
        }
        if (n > kCap) return refine_crossing(sh, row, V, bp, above, thr, mz, kt);
        sort_desc(sh, n);
        const int per = (n + kNT - 1) / kNT;
        unsigned long long lsum = 0;
        for (int j = 0; j < per; ++j) {
            const int i = static_cast<int>(threadIdx.x) * per + j;
            if (i < n) lsum += fixed_q(float_of(static_cast<uint32_t>(sh.cand[i] >> 32)), mz, kt);
        }
        unsigned long long total = 0;
        unsigned long long run = above + block_exclusive_scan(sh, lsum, &total);
        for (int j = 0; j < per; ++j) {
            const int i = static_cast<int>(threadIdx.x) * per + j;
            if (i >= n) break;
            if (static_cast<double>(run) >= thr) atomicMin(&sh.found_above, run);
            run += fixed_q(float_of(static_cast<uint32_t>(sh.cand[i] >> 32)), mz, kt);
        }
        if (threadIdx.x == 0 && static_cast<double>(above + total) >= thr) atomicMin(&sh.found_above, above + total);
        __syncthreads();
        const unsigned long long P = sh.found_above;
        if (P != ~0ull) return P;
        bp = next_bin(sh, bp, -1);  // the crossing lies below this bin
    }
    return s_all;
}

// The bin (scanning from the top) where the running FP32 mass reaches
// `target` (in 2^-40 units); found_bin, -1 if never.
__device__ void find_from_top_f(Shared& sh, const float* vals, double target) {
    constexpr int per = kBins / kNT;
    const int hi = kBins - 1 - static_cast<int>(threadIdx.x) * per;
    unsigned long long v[per];
    unsigned long long local = 0;
#pragma unroll
    for (int j = 0; j < per; ++j) {
        v[j] = static_cast<unsigned long long>(static_cast<double>(vals[hi - j]) * kFix);
        local += v[j];
    }
    if (threadIdx.x == 0) sh.found_bin = -1;
    unsigned long long total = 0;
    unsigned long long run = block_exclusive_scan(sh, local, &total);
#pragma unroll
    for (int j = 0; j < per; ++j) {
        if (static_cast<double>(run) < target && target <= static_cast<double>(run + v[j])) sh.found_bin = hi - j;
        run += v[j];
    }
    __syncthreads();
}

// The exact path for one row: radix selection over the whole row (two or more
// passes over it), for any row the one-pass path below cannot finish.
__device__ void exact_row(Shared& sh, const TopkArgs& a, long long t) {
    unsigned long long* top = sh.top;
    const int tid = threadIdx.x;
    const int V = a.V;
    const int Kp = min(a.K, V);
    const float kt = a.inv_t * kLog2e;
    const bool use_p = a.top_p < 1.0f;
    {
        const float* row = a.logits + t * a.stride;
        // ---- pass 1: the maximum and the top digit's histogram
        for (int i = tid; i < kBins; i += kNT) sh.hist0[i] = 0u;
        if (tid == 0) sh.maxkey = 0u;
        __syncthreads();
        uint32_t mk = 0u;
        for_each_entry(row, V, [&](float z, int) {
            const uint32_t k = key_of(z);
            mk = max(mk, k);
            atomicAdd(&sh.hist0[k >> 20], 1u);
        });
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mk = max(mk, __shfl_xor_sync(0xFFFFFFFFu, mk, o));
        if ((tid & 31) == 0) atomicMax(&sh.maxkey, mk);
        __syncthreads();
        const float mz = float_of(sh.maxkey);
        find_from_top(sh, sh.hist0, kBins, static_cast<double>(Kp));
        const int rbin = sh.found_bin;
        const unsigned long long rabove = sh.found_above;
        const bool coll0 = rabove + sh.hist0[rbin] <= static_cast<unsigned long long>(kCap);
        const uint32_t lowkey = static_cast<uint32_t>(rbin) << 20;

        // ---- pass 2: the normaliser and the candidates
        if (tid == 0) sh.ncand = 0;
        __syncthreads();
        unsigned long long s = 0ull;
        for_each_entry(row, V, [&](float z, int id) {
            const uint32_t k = key_of(z);
            s += fixed_q(z, mz, kt);
            if (coll0 && k >= lowkey) {
                const int pos = atomicAdd(&sh.ncand, 1);
                if (pos < kCap) sh.cand[pos] = pack_entry(k, id);
            }
        });
        unsigned long long s_all = 0ull;
        (void)block_exclusive_scan(sh, s, &s_all);  // deterministic: integer sum
        __syncthreads();
        const int n = select_top(sh, row, V, Kp, rbin, rabove, coll0, mz, kt);
        (void)n;
        for (int i = tid; i < Kp; i += kNT) top[i] = sh.cand[i];
        __syncthreads();

        // ---- the nucleus (top_p < 1)
        int count = Kp;
        double log_nuc = 0.0;
        if (use_p) {
            const double thr = static_cast<double>(a.top_p) * static_cast<double>(s_all);
            // running mass over the selected entries
            unsigned long long qk = 0ull;
            if (tid < Kp) qk = fixed_q(float_of(static_cast<uint32_t>(top[tid] >> 32)), mz, kt);
            // (Kp <= kMaxTopK <= 2 * kNT: a second entry per thread when Kp > kNT)
            unsigned long long qk2 = 0ull;
            if (tid + kNT < Kp) qk2 = fixed_q(float_of(static_cast<uint32_t>(top[tid + kNT] >> 32)), mz, kt);
            unsigned long long tot1 = 0ull, tot2 = 0ull;
            const unsigned long long b1 = block_exclusive_scan(sh, qk, &tot1);
            const unsigned long long b2 = block_exclusive_scan(sh, qk2, &tot2);
            if (tid == 0) sh.ncand = 0;  // kept entries among the selected ones
            __syncthreads();
            if (tid < Kp && static_cast<double>(b1) < thr) atomicAdd(&sh.ncand, 1);
            if (tid + kNT < Kp && static_cast<double>(tot1 + b2) < thr) atomicAdd(&sh.ncand, 1);
            __syncthreads();
            const int kept = sh.ncand;
            __syncthreads();
            unsigned long long P;
            if (kept < Kp) {
                count = kept;  // the nucleus ends inside the selection
                P = 0ull;
                if (tid == 0) sh.found_above = 0ull;
                __syncthreads();
                if (tid < kept) atomicAdd(&sh.found_above, qk);
                if (tid + kNT < kept) atomicAdd(&sh.found_above, qk2);
                __syncthreads();
                P = sh.found_above;
                __syncthreads();
            } else {
                // it ends further down (rows flatter than the selection): the FP32
                // mass histogram of the top digit, taken only now, points to the
                // bin, the exact search confirms it
                for (int i = tid; i < kBins; i += kNT) sh.mhf[i] = 0.0f;
                __syncthreads();
                for_each_entry(row, V, [&](float z, int) { atomicAdd(&sh.mhf[key_of(z) >> 20], rel_mass(z, mz, kt)); });
                __syncthreads();
                find_from_top_f(sh, sh.mhf, thr);
                int bp = sh.found_bin;
                if (bp < 0) bp = rbin;
                P = crossing_mass(sh, row, V, bp, thr, mz, kt, s_all);
            }
            log_nuc = log(static_cast<double>(P) / static_cast<double>(s_all));
        }

        // ---- outputs: ids and log mu, then the padding
        const double lse = static_cast<double>(mz) * a.inv_t + log(static_cast<double>(s_all) / kFix);
        int32_t* ids = a.ids + t * a.K;
        float* lps = a.lps + t * a.K;
        for (int i = tid; i < a.K; i += kNT) {
            if (i < count) {
                const uint32_t key = static_cast<uint32_t>(top[i] >> 32);
                const int id = static_cast<int>(~static_cast<uint32_t>(top[i]));
                ids[i] = id;
                lps[i] = static_cast<float>(static_cast<double>(float_of(key)) * a.inv_t - lse - log_nuc);
            } else {
                ids[i] = -1;
                lps[i] = 0.0f;
            }
        }
        if (tid == 0 && a.counts) a.counts[t] = count;
        __syncthreads();
    }
}

constexpr int kGroups = 2;            // independent thread groups of a CTA on the one-pass path (<= 4)
constexpr int kGT = kNT / kGroups;    // threads per group
constexpr int kGW = kGT / 32;         // warps per group
constexpr int kSampRun = 32;          // vectors per sampled run (one warp load)
constexpr int kSampEvery = 16;        // one run in kSampEvery is sampled
constexpr int kRound = 32;            // rows per group between the CTA's exact-path rounds
constexpr int kNucRes = 64;           // nucleus histogram: bins per binary order of magnitude of mass
constexpr int kNucBins = 40 * kNucRes;  // down to 2^-40 of the row maximum's mass (the fixed-point unit)

// A thread group's view: its threads, its named barrier, its shared state.
struct GroupShared {
    uint32_t keys[kGT];                 // the sample maxima, sorted
    unsigned long long cand[kCap];      // (key << 32) | ~id
    float mh[kNucBins];                 // wide nucleus: mass of the entries below tau per bin (FP32, a guide)
    unsigned long long u64red[kGW];     // group sums of 64-bit integers
    float fred[kGW], flo[kGW];          // group maximum / sums of pairs
    double dS, dlse;
    double pnuc, lnuc;  // the nucleus mass and log(nucleus mass / normaliser)
    unsigned long long above;           // wide nucleus: fixed-point mass before the crossing bin
    int ncand, cross, nbin, bstar;
};
constexpr int kRing = 6;  // 16-byte slots per thread: the one pass keeps kRing - 1 copies in flight
struct OnePass {
    GroupShared grp[kGroups];
    float4 ring[kGroups][kRing][kGT];  // slot j of thread i: ring[group][j][i]
};
struct KernelShared {
    union {
        Shared exact;                   // the exact path: the whole CTA, between rounds
        OnePass one;                    // the one-pass path: per group its state and copy ring
    } u;
    int ndefer;
    long long defer[kGroups * kRound];  // rows left to the exact path since it last ran
    long long take[kGroups];            // a group's row from the run-time hand-out
    int gdone[kGroups];                 // a group has no rows left
};

struct Group {
    int id, tid, lane, warp;
    // named barriers 1.. kGroups (0 is the CTA's), as immediates so that only
    // those are reserved
    __device__ void sync() const {
        switch (id) {
            case 0: asm volatile("bar.sync 1, %0;" ::"n"(kGT) : "memory"); break;
            case 1: asm volatile("bar.sync 2, %0;" ::"n"(kGT) : "memory"); break;
            case 2: asm volatile("bar.sync 3, %0;" ::"n"(kGT) : "memory"); break;
            default: asm volatile("bar.sync 4, %0;" ::"n"(kGT) : "memory"); break;
        }
    }
};

// A sum kept as an unevaluated FP32 pair hi + lo, added without error
// (two-sum): the same bits in every lane whatever the order of the operands.
struct Pair {
    float hi, lo;
};
__device__ __forceinline__ Pair pair_add(Pair a, Pair b) {
    float s, e;
    two_sum(a.hi, b.hi, s, e);
    return Pair{s, (a.lo + b.lo) + e};
}
__device__ __forceinline__ Pair pair_shfl_xor(Pair v, int o) {
    return Pair{__shfl_xor_sync(0xFFFFFFFFu, v.hi, o), __shfl_xor_sync(0xFFFFFFFFu, v.lo, o)};
}
// Sum of the group's pairs in a fixed order.
__device__ Pair group_sum_pair(GroupShared& gs, const Group& G, Pair v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = pair_add(v, pair_shfl_xor(v, o));
    if (G.lane == 0) {
        gs.fred[G.warp] = v.hi;
        gs.flo[G.warp] = v.lo;
    }
    G.sync();
    Pair r{0.0f, 0.0f};
    for (int w = 0; w < kGW; ++w) r = pair_add(r, Pair{gs.fred[w], gs.flo[w]});
    G.sync();
    return r;
}
__device__ float group_max_f(GroupShared& gs, const Group& G, float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    if (G.lane == 0) gs.fred[G.warp] = v;
    G.sync();
    float r = -INFINITY;
    for (int w = 0; w < kGW; ++w) r = fmaxf(r, gs.fred[w]);
    G.sync();
    return r;
}
// Bitonic sort of the group's kGT keys, larger first (one per thread): the
// steps within a warp by shuffles, the others through shared memory.
__device__ void group_sort_keys_desc(GroupShared& gs, const Group& G, uint32_t key) {
    const int i = G.tid;
    uint32_t x = key;
    for (int size = 2; size <= kGT; size <<= 1)
        for (int j = size >> 1; j > 0; j >>= 1) {
            const bool desc = (i & size) == 0;  // this pair's block sorts larger first
            uint32_t y;
            if (j < 32) {
                y = __shfl_xor_sync(0xFFFFFFFFu, x, j);
            } else {
                gs.keys[i] = x;
                G.sync();
                y = gs.keys[i ^ j];
                G.sync();
            }
            const bool lower = (i & j) == 0;  // i is the first of its pair
            const uint32_t hi = max(x, y), lo = min(x, y);
            x = (lower == desc) ? hi : lo;
        }
    gs.keys[i] = x;
    G.sync();
}
// Bitonic sort of c[0, m) (m = kGT E, a power of two), larger first, by the
// group: thread t holds entries [t E, t E + E) in registers; the stages whose
// partner lies in the same thread compare in registers, those within the warp
// exchange by shuffles, and only the stages across warps (six for any E) go
// through shared memory, each with two group barriers.  E <= 4 (up to 1024
// entries) keeps every entry in registers.
template <int E>
__device__ void group_bitonic_regs(unsigned long long* c, const Group& G) {
    constexpr int m = kGT * E;
    unsigned long long x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = c[G.tid * E + e];
    G.sync();  // every thread has its entries before any stage writes c
    for (int k = 2; k <= m; k <<= 1) {
        // the stages whose partner is in another thread (j >= E) ...
        for (int j = k >> 1; j >= E; j >>= 1) {
            if (j < 32 * E) {
                const int lj = j / E;  // partner lane
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int i = G.tid * E + e;
                    const unsigned long long y = shfl_xor_u64(x[e], lj);
                    const bool lower = (i & j) == 0, desc = (i & k) == 0;
                    x[e] = (lower == desc) ? (x[e] > y ? x[e] : y) : (x[e] < y ? x[e] : y);
                }
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) c[G.tid * E + e] = x[e];
                G.sync();
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int i = G.tid * E + e;
                    const unsigned long long y = c[i ^ j];
                    const bool lower = (i & j) == 0, desc = (i & k) == 0;
                    x[e] = (lower == desc) ? (x[e] > y ? x[e] : y) : (x[e] < y ? x[e] : y);
                }
                G.sync();
            }
        }
        // ... then those within the thread's own entries (compile-time indices)
#pragma unroll
        for (int jj = E / 2; jj > 0; jj >>= 1) {
            if (jj <= (k >> 1)) {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int f = e ^ jj;
                    if (f > e) {
                        const int i = G.tid * E + e;
                        const bool desc = (i & k) == 0;
                        const unsigned long long a0 = x[e], b0 = x[f];
                        if (desc ? (a0 < b0) : (a0 > b0)) {
                            x[e] = b0;
                            x[f] = a0;
                        }
                    }
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) c[G.tid * E + e] = x[e];
    G.sync();
}

// Bitonic sort of cand[off, off + n), larger first, by the group (off + the
// padded length must stay within kCap: the caller checks).  Padding entries
// are 0, below every real entry.
__device__ void group_sort_desc_at(GroupShared& gs, const Group& G, int off, int n) {
    int m = kGT;
    while (m < n) m <<= 1;
    unsigned long long* c = gs.cand + off;
    for (int i = n + G.tid; i < m; i += kGT) c[i] = 0ull;
    G.sync();
    switch (m / kGT) {
        case 1: group_bitonic_regs<1>(c, G); return;
        case 2: group_bitonic_regs<2>(c, G); return;
        case 4: group_bitonic_regs<4>(c, G); return;
        default: break;
    }
    // more than 1024 entries (rare): every stage through shared memory
    for (int k = 2; k <= m; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = G.tid; i < m; i += kGT) {
                const int l = i ^ j;
                if (l > i) {
                    const unsigned long long x = c[i], y = c[l];
                    if (((i & k) == 0) ? (x < y) : (x > y)) {
                        c[i] = y;
                        c[l] = x;
                    }
                }
            }
            G.sync();
        }
}
__device__ void group_sort_desc(GroupShared& gs, const Group& G, int n) { group_sort_desc_at(gs, G, 0, n); }

// Exclusive prefix sum of 64-bit integers over the group's threads, in
// thread order; *total gets the sum of all.
__device__ unsigned long long group_exclusive_scan_u64(GroupShared& gs, const Group& G, unsigned long long v,
                                                       unsigned long long* total) {
    unsigned long long x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long y = shfl_up_u64(x, d);
        if (G.lane >= d) x += y;
    }
    if (G.lane == 31) gs.u64red[G.warp] = x;
    G.sync();
    unsigned long long before = 0, all = 0;
    for (int w = 0; w < kGW; ++w) {
        const unsigned long long t = gs.u64red[w];
        if (w < G.warp) before += t;
        all += t;
    }
    G.sync();
    if (total) *total = all;
    return before + x - v;
}

// Every entry of the row, f(z, id), by the group's threads (16-byte loads,
// kUnroll of them in flight per thread).
template <typename F>
__device__ __forceinline__ void group_for_each_entry(const Group& G, const float* row, int V, F&& f) {
    const int nv4 = V >> 2;
    const float4* r4 = reinterpret_cast<const float4*>(row);
    int i = G.tid;
    for (; i + (kUnroll - 1) * kGT < nv4; i += kUnroll * kGT) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = __ldg(r4 + i + u * kGT);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int b = 4 * (i + u * kGT);
            f(v[u].x, b);
            f(v[u].y, b + 1);
            f(v[u].z, b + 2);
            f(v[u].w, b + 3);
        }
    }
    for (; i < nv4; i += kGT) {
        const float4 v = __ldg(r4 + i);
        f(v.x, 4 * i);
        f(v.y, 4 * i + 1);
        f(v.z, 4 * i + 2);
        f(v.w, 4 * i + 3);
    }
    for (int j = (nv4 << 2) + G.tid; j < V; j += kGT) f(__ldg(row + j), j);
}


// The nucleus bin of an entry below the candidate threshold: how many 1/64
// binary orders of magnitude its mass lies below the row maximum's (the same
// expression in both passes, so both put an entry in the same bin).
__device__ __forceinline__ int nucleus_bin(float z, float M, float kt64) {
    // floor of a nonnegative x < 2^23 by one add rounded toward zero: the
    // integer part lands in the low mantissa bits of 2^23 + x
    const float x = fminf((M - z) * kt64, 4194304.0f);
    return __float_as_int(__fadd_rz(x, 8388608.0f)) - 0x4B000000;
}

// The nucleus reaches below the candidates (the entries with z >= tau, sorted
// in cand[0, nc)): more passes over the row give its exact mass in 2^-40 fixed
// point (the normaliser S is the one-pass sum).  Pass 2: below tau, every
// entry's FP32 mass 2^((z - M) kt) goes into a histogram on bins of 1/64 of a
// binary order of magnitude, which only guides the search: the bin where the
// running mass
// (candidates first, then the bins from the top) reaches top_p S should hold
// the crossing.  Pass 3 sums the exact fixed-point mass of every entry above
// that bin and collects the bin's entries behind the candidates; one warp
// walks them, sorted, to the first entry whose preceding mass reaches top_p S,
// and the nucleus mass is the running sum there.  When the FP32 guide pointed
// one bin off (the exact mass above the bin already reaches the threshold, or
// the bin's entries do not), pass 3 repeats on the neighbouring bin.  Returns
// false (the row goes to the exact path) when a bin's entries do not fit the
// buffer, the crossing is not found in a few bins, or the fixed-point sums put
// it among the candidates after all (a near tie).
__device__ bool wide_nucleus(GroupShared& gs, const Group& G, const TopkArgs& a, const float* row, float M, float tau,
                             int nc, double S, double* log_nuc) {
    const int V = a.V;
    const float kt = a.inv_t * kLog2e;
    const float kt64 = kt * static_cast<float>(kNucRes);
    for (int b = G.tid; b < kNucBins; b += kGT) gs.mh[b] = 0.0f;
    G.sync();
    // ---- pass 2: the FP32 mass histogram below tau
    group_for_each_entry(G, row, V, [&](float z, int) {
        if (z < tau) {
            const int b = nucleus_bin(z, M, kt64);
            if (b < kNucBins) atomicAdd(&gs.mh[b], rel_mass(z, M, kt));
        }
    });
    G.sync();
    // the normaliser in fixed-point units (2^-40 of the row maximum's mass),
    // from the one-pass sum
    const double S_fix = S * kFix;
    // the candidates' fixed-point mass
    unsigned long long pc = 0ull;
    for (int i = G.tid; i < nc; i += kGT) pc += fixed_q(float_of(static_cast<uint32_t>(gs.cand[i] >> 32)), M, kt);
    unsigned long long P_cand = 0ull;
    (void)group_exclusive_scan_u64(gs, G, pc, &P_cand);
    const double thr = static_cast<double>(a.top_p) * S_fix;
    if (!(static_cast<double>(P_cand) < thr)) return false;  // a near tie at the end of the candidates
    // ---- the guide: the bin where the FP32 running mass crosses thr (thread i
    // owns bins [i per, (i + 1) per))
    constexpr int per = (kNucBins + kGT - 1) / kGT;
    const int b0 = G.tid * per;
    double local = 0.0;
    for (int j = 0; j < per; ++j)
        if (b0 + j < kNucBins) local += static_cast<double>(gs.mh[b0 + j]) * kFix;
    if (G.tid == 0) gs.bstar = kNucBins - 1;
    // (the FP32 masses only choose where to look: a plain double scan)
    double run = static_cast<double>(P_cand);
    {
        double x = local;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const double y = __shfl_up_sync(0xFFFFFFFFu, x, d);
            if (G.lane >= d) x += y;
        }
        if (G.lane == 31) gs.u64red[G.warp] = static_cast<unsigned long long>(__double_as_longlong(x));
        G.sync();
        double before = 0.0;
        for (int w = 0; w < G.warp; ++w) before += __longlong_as_double(static_cast<long long>(gs.u64red[w]));
        G.sync();
        run += before + x - local;
    }
    for (int j = 0; j < per; ++j) {
        const int b = b0 + j;
        if (b >= kNucBins) break;
        const double v = static_cast<double>(gs.mh[b]) * kFix;
        if (run < thr && thr <= run + v) gs.bstar = b;
        run += v;
    }
    G.sync();
    int bstar = gs.bstar;
    G.sync();
    for (int tries = 0; tries < 4; ++tries) {
        // ---- pass 3: the exact mass above bin bstar, and its entries
        if (G.tid == 0) gs.nbin = 0;
        G.sync();
        unsigned long long hi = 0ull;
        group_for_each_entry(G, row, V, [&](float z, int id) {
            if (z < tau) {
                const int b = nucleus_bin(z, M, kt64);
                if (b < bstar) {
                    hi += fixed_q(z, M, kt);
                } else if (b == bstar) {
                    const int pos = atomicAdd(&gs.nbin, 1);
                    if (nc + pos < kCap) gs.cand[nc + pos] = pack_entry(key_of(z), id);
                }
            }
        });
        unsigned long long above_hist = 0ull;
        (void)group_exclusive_scan_u64(gs, G, hi, &above_hist);
        const unsigned long long above = P_cand + above_hist;
        const int nb = gs.nbin;
        G.sync();
        if (static_cast<double>(above) >= thr) {  // the crossing lies in a bin above
            if (bstar == 0) return false;
            --bstar;
            continue;
        }
        int m = 1;
        while (m < nb) m <<= 1;
        if (nc + m > kCap) return false;
        if (nb > 0) group_sort_desc_at(gs, G, nc, nb);
        // ---- the walk: one warp, lane-contiguous chunks, running sums in fixed point
        if (G.warp == 0) {
            const int lane = G.lane;
            const int chunk = (nb + 31) / 32;
            const int i0 = nc + lane * chunk, i1 = min(nc + nb, i0 + chunk);
            auto q_of = [&](int i) { return fixed_q(float_of(static_cast<uint32_t>(gs.cand[i] >> 32)), M, kt); };
            unsigned long long loc = 0ull;
            for (int i = i0; i < i1; ++i) loc += q_of(i);
            unsigned long long inc = loc;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const unsigned long long y = shfl_up_u64(inc, d);
                if (lane >= d) inc += y;
            }
            unsigned long long r = above + inc - loc;  // mass before this lane's first entry
            unsigned long long P = ~0ull;
            for (int i = i0; i < i1; ++i) {
                if (static_cast<double>(r) >= thr) {
                    P = r;
                    break;
                }
                r += q_of(i);
            }
            // the first lane (in entry order) that found the crossing holds it;
            // if none did, the bin's entries end before it (total below thr)
            const unsigned found = __ballot_sync(0xFFFFFFFFu, P != ~0ull);
            const int src = found ? __ffs(found) - 1 : 31;
            const unsigned long long Pf = shfl_u64(found ? P : inc, src);
            if (lane == 0) {
                const unsigned long long end = above + Pf;  // (when not found: the bin's end)
                if (found) {
                    gs.pnuc = static_cast<double>(Pf);
                    gs.lnuc = log(static_cast<double>(Pf) / S_fix);
                } else if (static_cast<double>(end) >= thr) {
                    // the first entry of the next bin crosses: the nucleus ends with this bin
                    gs.pnuc = static_cast<double>(end);
                    gs.lnuc = log(static_cast<double>(end) / S_fix);
                } else {
                    gs.pnuc = -1.0;  // the crossing lies in a bin below
                }
            }
        }
        G.sync();
        const double P = gs.pnuc;
        *log_nuc = gs.lnuc;
        G.sync();
        if (P > 0.0) return true;
        if (bstar + 1 >= kNucBins) return false;
        ++bstar;
    }
    return false;
}

// One warp walks the sorted entries cand[beg, beg + n) with error-free FP32
// running sums that start at `base`, for the first entry whose preceding mass
// reaches thr = (t_hi + t_lo): 32 entries at a time (one per lane, an
// inclusive warp scan of their masses), stopping at the block that holds it.
// gs.cross gets its index relative to beg (n + 1 if none); gs.pnuc the
// nucleus mass: the running sum there, or the entries' total when it reaches
// thr only after the last of them, or -1 when the nucleus reaches past them.
__device__ void warp_walk(GroupShared& gs, int lane, int beg, int n, Pair base, float t_hi, float t_lo, float M,
                          float kt) {
    Pair run = base;
    int cross = n + 1;
    double P = -1.0;
    for (int b0 = 0; b0 < n; b0 += 32) {
        const int i = b0 + lane;
        const float q = i < n ? ex2((float_of(static_cast<uint32_t>(gs.cand[beg + i] >> 32)) - M) * kt) : 0.0f;
        Pair inc{q, 0.0f};
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const Pair y{__shfl_up_sync(0xFFFFFFFFu, inc.hi, d), __shfl_up_sync(0xFFFFFFFFu, inc.lo, d)};
            if (lane >= d) inc = pair_add(y, inc);
        }
        Pair ex{__shfl_up_sync(0xFFFFFFFFu, inc.hi, 1), __shfl_up_sync(0xFFFFFFFFu, inc.lo, 1)};
        if (lane == 0) ex = Pair{0.0f, 0.0f};
        const Pair pre = pair_add(run, ex);  // mass before entry i
        const bool hit = i < n && (pre.hi - t_hi) + (pre.lo - t_lo) >= 0.0f;
        const unsigned hits = __ballot_sync(0xFFFFFFFFu, hit);
        if (hits) {
            const int src = __ffs(hits) - 1;
            cross = b0 + src;
            P = __shfl_sync(0xFFFFFFFFu, (double)pre.hi + (double)pre.lo, src);
            break;
        }
        run = pair_add(run, Pair{__shfl_sync(0xFFFFFFFFu, inc.hi, 31), __shfl_sync(0xFFFFFFFFu, inc.lo, 31)});
    }
    if (cross > n && (run.hi - t_hi) + (run.lo - t_lo) >= 0.0f) P = (double)run.hi + (double)run.lo;
    if (lane == 0) {
        gs.cross = cross;
        gs.pnuc = P;
    }
    __syncwarp();
}

// ln x of a positive normal double: the binary exponent exactly, the
// mantissa's logarithm on the MUFU unit (absolute error under 2.5e-7, below
// the FP32 rounding of the log-probabilities written).  The row's two
// logarithms run in one thread while the group waits, and GB300's FP64 rate is
// a small fraction of its FP32 rate: against FP64 log, 0.419 -> 0.414 ms on
// 4096 x 151936 at top_p = 1.
__device__ __forceinline__ double ln_pos(double x) {
    const long long b = __double_as_longlong(x);
    const int e = static_cast<int>((b >> 52) & 0x7FF) - 1023;
    const double mant = __longlong_as_double((b & 0x000FFFFFFFFFFFFFLL) | 0x3FF0000000000000LL);  // [1, 2)
    return (static_cast<double>(__log2f(static_cast<float>(mant))) + static_cast<double>(e)) * 0.6931471805599453;
}

// The one-pass path for one row, run by one thread group.  A sample (every
// kSampEvery-th run of vectors) gives each thread a maximum; the largest of
// those maxima is the exponent offset, and the `rank`-th largest the candidate
// threshold, placed so that about 3 K entries of the row reach it.  One pass
// over the row then sums 2^((z - m) kt) per thread (compensated, in a fixed
// order; a thread that meets an entry above its offset m moves m up) and
// collects every entry at or above the threshold.  The candidates are
// sorted; the top K and, with top_p < 1, the nucleus come from them.  The
// pass reads the row through a ring of kRing 16-byte shared-memory slots per
// thread that asynchronous copies fill, so that kRing - 1 copies per thread
// stay in flight without holding registers, the loop unrolled over the ring so
// that every slot offset is a constant (4096 x 151936 FP32 at top_p = 1: 0.479
// ms with four 16-byte loads in flight per thread; 0.464 with the ring; 0.423
// unrolled, with one compensated addition per round; 0.410 with the offset's
// tests folded into the candidate test).  Returns
// false -- outputs untouched, the same decision in every thread of the group
// -- when the row needs the exact path: too few or too many candidates, a
// nucleus that reaches below them, entries that are not finite, or K above
// kCap / 4.
__device__ bool fast_row(GroupShared& gs, float4 (&ring)[kRing][kGT], const Group& G, const TopkArgs& a, long long t) {
    const float* row = a.logits + t * a.stride;
    const int V = a.V, tid = G.tid, lane = G.lane, warp = G.warp;
    const int Kp = min(a.K, V);
    const bool use_p = a.top_p < 1.0f;
    if ((use_p ? 6 : 4) * Kp > kCap) return false;
    const float kt = a.inv_t * kLog2e;
    const int nv4 = V >> 2;
    const float4* r4 = reinterpret_cast<const float4*>(row);

    // ---- this thread's vectors tid, tid + kGT, ... through its own ring of
    // kRing 16-byte slots; the first kRing - 1 copies start before the sample
    const uint64_t last = l2_policy_evict_first();  // the row's last read
    const int nmine = tid < nv4 ? (nv4 - 1 - tid) / kGT + 1 : 0;
    const uint32_t rs = smem_addr(&ring[0][tid]);
    constexpr uint32_t kSlot = 16u * kGT;  // bytes between a thread's slots
#pragma unroll
    for (int j = 0; j < kRing - 1; ++j) {
        if (j < nmine) cp_async16_hint(rs + j * kSlot, r4 + tid + j * kGT, last);
        cp_async_commit();
    }

    // ---- the threshold and the offset from the sample
    float tau = -INFINITY;  // candidates: z >= tau (-inf: every entry)
    float o = -INFINITY;    // exponent offset of the sums
    if (V > kCap) {
        const int nruns = nv4 / kSampRun;
        float smax = -INFINITY;
        // (kept in L2 until the pass below reads the same lines again)
        const uint64_t keep = l2_policy_evict_last();
        for (int r = warp * kSampEvery; r < nruns; r += kGW * kSampEvery) {
            const float4 v = ldg_f4_hint(r4 + r * kSampRun + lane, keep);
            smax = fmaxf(smax, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
        }
        group_sort_keys_desc(gs, G, key_of(smax));
        // about 3 K entries reach the threshold, 4 K with top_p < 1 (so that
        // most nuclei end among them at the usual temperatures)
        const int depth = use_p ? 4 : 3;
        const int rank = min(kGT, max(8, (depth * Kp + kSampEvery - 1) / kSampEvery));
        tau = float_of(gs.keys[rank - 1]);
        o = float_of(gs.keys[0]);
        G.sync();
        if (!isfinite(o)) {
            // the ring's first copies land before its slots are written again
            // (the next row's copies, or the exact path's shared memory)
            cp_async_wait<0>();
            return false;
        }
    }

    // ---- one pass: the sums and the candidates
    if (tid == 0) gs.ncand = 0;
    G.sync();
    // (z - m) is formed first and then scaled, so the terms nearest the
    // offset -- the ones that dominate the sum -- carry no rounding of the offset
    float m = o;                      // this thread's offset
    float s = 0.0f, c = 0.0f;         // compensated sum of 2^((z - m) kt)
    const f2_t KT2 = f2_pack(kt, kt);
    auto raise = [&](float m_new) {   // an entry above this thread's offset
        if (m > -INFINITY) {
            const float f = ex2((m - m_new) * kt);
            s *= f;
            c *= f;
        }
        m = m_new;
    };
    auto add = [&](float e) {
        const float y = e - c;
        const float u = s + y;
        c = (u - s) - y;
        s = u;
    };
    auto collect1 = [&](float z, int id) {
        if (z >= tau) {
            const int pos = atomicAdd(&gs.ncand, 1);
            if (pos < kCap) gs.cand[pos] = pack_entry(key_of(z), id);
        }
    };
    // The ring's rounds (kRing vectors, 4 kRing terms) are summed plainly and
    // each round's sum is Kahan-added once: at most a few FP32 roundings of a
    // round's own sum, under 1e-6 of the row's normaliser (the per-vector
    // compensated form: 0.436 ms against 0.423 on 4096 x 151936 at top_p = 1).
    float bsum = 0.0f;  // the current cycle's terms (relative to m)
    // Whole rounds need kRing vectors per thread, so V > 4 (kRing - 1) kGT >=
    // kCap there: the row had a sample, its offset o is finite, and so is m.
    // And tau <= o <= m, so an entry above m is also a candidate.
    static_assert(4 * (kRing - 1) * kGT >= kCap, "whole rounds only on sampled rows");
    auto take4b = [&](const float4& v, int id0) {
        const float m4 = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
        if (m4 >= tau && m4 > m) {
            add(bsum);
            bsum = 0.0f;
            raise(m4);
        }
        {
            const f2_t NM = f2_pack(-m, -m);
            const f2_t e01 = f2_ex2(f2_mul(f2_add(f2_pack(v.x, v.y), NM), KT2));
            const f2_t e23 = f2_ex2(f2_mul(f2_add(f2_pack(v.z, v.w), NM), KT2));
            const f2_t e = f2_add(e01, e23);
            bsum += f2_lo(e) + f2_hi(e);
        }
        if (m4 >= tau) {
            collect1(v.x, id0);
            collect1(v.y, id0 + 1);
            collect1(v.z, id0 + 2);
            collect1(v.w, id0 + 3);
        }
    };
    auto take4 = [&](const float4& v, int id0) {
        const float m4 = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
        if (m4 > m) raise(m4);
        if (m > -INFINITY) {
            const f2_t NM = f2_pack(-m, -m);
            const f2_t e01 = f2_ex2(f2_mul(f2_add(f2_pack(v.x, v.y), NM), KT2));
            const f2_t e23 = f2_ex2(f2_mul(f2_add(f2_pack(v.z, v.w), NM), KT2));
            const f2_t e = f2_add(e01, e23);
            add(f2_lo(e) + f2_hi(e));
        }
        if (m4 >= tau) {
            collect1(v.x, id0);
            collect1(v.y, id0 + 1);
            collect1(v.z, id0 + 2);
            collect1(v.w, id0 + 3);
        }
    };
    {
        // vector j sits in slot j mod kRing; the copy of vector j + kRing - 1
        // goes to the slot that vector j - 1 was read from
        int j = 0;
        for (; j + kRing <= nmine; j += kRing) {  // whole rounds: every slot offset a constant
#pragma unroll
            for (int u = 0; u < kRing; ++u) {
                if (j + u + kRing - 1 < nmine)
                    cp_async16_hint(rs + ((u + kRing - 1) % kRing) * kSlot, r4 + tid + (j + u + kRing - 1) * kGT, last);
                cp_async_commit();
                cp_async_wait<kRing - 1>();  // vector j + u's copy has landed
                const uint4 w = lds128(rs + u * kSlot);
                take4b(make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z), __uint_as_float(w.w)),
                       4 * (tid + (j + u) * kGT));
            }
            add(bsum);
            bsum = 0.0f;
        }
        cp_async_wait<0>();  // the rest (fewer than kRing vectors, slots 0..) has landed
        for (int u = 0; j < nmine; ++j, ++u) {
            const uint4 w = lds128(rs + u * kSlot);
            take4(make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z), __uint_as_float(w.w)),
                  4 * (tid + j * kGT));
        }
        for (int j = (nv4 << 2) + tid; j < V; j += kGT) {
            const float z = __ldg(row + j);
            if (z > m) raise(z);
            if (m > -INFINITY) add(ex2((z - m) * kt));
            collect1(z, j);
        }
    }
    // ---- the normaliser: every thread's sum moved to the row maximum M
    // (threads already there untouched), summed without error in a fixed order
    const float M = group_max_f(gs, G, m);
    float part = s - c;
    if (!(m > -INFINITY)) part = 0.0f;
    else if (m != M) part *= ex2((m - M) * kt);
    const Pair tot = group_sum_pair(gs, G, Pair{part, 0.0f});
    if (tid == 0) {
        const double S = (double)tot.hi + (double)tot.lo;
        gs.dS = S;
        gs.dlse = (double)M * a.inv_t + ln_pos(S);
    }
    G.sync();
    const double S = gs.dS, lse = gs.dlse;
    const int nc = gs.ncand;
    if (!isfinite(M) || !(S > 0.0) || !isfinite(S) || !isfinite(lse) || nc < Kp || nc > kCap) return false;
    group_sort_desc(gs, G, nc);

    // ---- the nucleus: one warp walks the sorted candidates with error-free
    // FP32 running sums; past them, the wide-nucleus passes
    int count = Kp;
    double log_nuc = 0.0;
    if (use_p) {
        const double thr = (double)a.top_p * S;
        const float t_hi = (float)thr, t_lo = (float)(thr - (double)t_hi);
        if (warp == 0) warp_walk(gs, lane, 0, nc, Pair{0.0f, 0.0f}, t_hi, t_lo, M, kt);
        G.sync();
        const int cross = gs.cross;
        const double P = gs.pnuc;
        G.sync();
        if (P > 0.0) count = min(Kp, cross <= nc ? cross : nc);
        if (P > 0.0) {
            // log(P / S), in one thread, without an FP64 division or logarithm
            if (tid == 0) gs.lnuc = ln_pos(P) - ln_pos(S);
            G.sync();
            log_nuc = gs.lnuc;
            G.sync();
        } else {
            // every candidate (and so the top K) is in the nucleus
            if (!wide_nucleus(gs, G, a, row, M, tau, nc, S, &log_nuc)) return false;
            count = Kp;
        }
    }

    // ---- outputs
    int32_t* ids = a.ids + t * a.K;
    float* lps = a.lps + t * a.K;
    for (int i = tid; i < a.K; i += kGT) {
        if (i < count) {
            const uint32_t key = static_cast<uint32_t>(gs.cand[i] >> 32);
            ids[i] = static_cast<int>(~static_cast<uint32_t>(gs.cand[i]));
            lps[i] = static_cast<float>(static_cast<double>(float_of(key)) * a.inv_t - lse - log_nuc);
        } else {
            ids[i] = -1;
            lps[i] = 0.0f;
        }
    }
    if (tid == 0 && a.counts) a.counts[t] = count;
    G.sync();
    return true;
}

// Without a workspace, rows are dealt to the thread groups round robin
// (group b * kGroups + g of the grid takes rows b * kGroups + g + k * groups).
// With one, each group takes its first row that way and every later row from
// a counter in the workspace, one row per take with the next take always in
// flight (its latency hides behind the row), so that the groups that drew
// costly rows (a nucleus far below the candidates) take fewer rows.  Each
// group takes its rows on the one-pass path; a row it cannot finish waits for
// the end of the round, when the whole CTA takes the deferred rows on the
// exact path.
__global__ void __launch_bounds__(kNT, 2) topk_capture_kernel(const __grid_constant__ TopkArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    KernelShared& ks = *reinterpret_cast<KernelShared*>(smem_raw);
    const Group G{static_cast<int>(threadIdx.x) / kGT, static_cast<int>(threadIdx.x) % kGT,
                  static_cast<int>(threadIdx.x) & 31, (static_cast<int>(threadIdx.x) % kGT) >> 5};
    const long long ngroups = static_cast<long long>(gridDim.x) * kGroups;
    const long long me = static_cast<long long>(blockIdx.x) * kGroups + G.id;  // this group's index
    if (threadIdx.x == 0) ks.ndefer = 0;
    if (G.tid == 0) ks.gdone[G.id] = 0;
    __syncthreads();
    long long k = 0;                  // rows this group has dealt itself
    unsigned long long pend = 0ull;   // group thread 0: the value of the take in flight
    if (a.ws && G.tid == 0 && me < a.T_static) pend = atomicAdd(a.ws + 2, 1ull);
    bool done = false;                // this group has no rows left
    for (;;) {
        for (int r = 0; r < kRound && !done; ++r) {
            long long t = me + k * ngroups;
            if (t < a.T_static) {
                ++k;
            } else if (a.ws && me < a.T_static) {
                // the take issued one row ago; issue the next
                if (G.tid == 0) {
                    ks.take[G.id] = static_cast<long long>(a.T_static + pend);
                    if (a.T_static + pend < static_cast<unsigned long long>(a.T)) pend = atomicAdd(a.ws + 2, 1ull);
                }
                G.sync();
                t = ks.take[G.id];
                G.sync();
            } else {
                t = a.T;  // (no more rows: dealt out, or this group started past them)
            }
            if (t >= a.T) {
                done = true;
                break;
            }
            if (!fast_row(ks.u.one.grp[G.id], ks.u.one.ring[G.id], G, a, t) && G.tid == 0) ks.defer[atomicAdd(&ks.ndefer, 1)] = t;
        }
        if (G.tid == 0) ks.gdone[G.id] = done ? 1 : 0;
        __syncthreads();
        const int nd = ks.ndefer;
        bool all_done = true;
        for (int g = 0; g < kGroups; ++g) all_done = all_done && ks.gdone[g];
        for (int q = 0; q < nd; ++q) exact_row(ks.u.exact, a, ks.defer[q]);
        __syncthreads();
        if (threadIdx.x == 0) ks.ndefer = 0;
        __syncthreads();
        if (all_done) break;
    }
    // The last CTA to finish leaves the workspace's words zero for the next
    // launch (every CTA is past its last take by now).
    if (a.ws && threadIdx.x == 0) {
        __threadfence();
        const unsigned long long fin = atomicAdd(a.ws + 3, 1ull);
        if (fin == static_cast<unsigned long long>(gridDim.x) - 1ull) {
            atomicExch(a.ws + 2, 0ull);
            atomicExch(a.ws + 3, 0ull);
        }
    }
}

}  // namespace
}  // namespace sc

extern "C" int sc_topk_capture(const float* logits, long long T, int V, long long logits_stride, float inv_temperature,
                               int K, float top_p, int32_t* ids_out, float* logprobs_out, int32_t* count_out,
                               void* workspace, sc_stream_t stream) {
    using namespace sc;
    if (T < 0) return fail(SC_ERR_SHAPE, "T = %lld < 0", T);
    if (V < 1 || V > (1 << 24)) return fail(SC_ERR_SHAPE, "V = %d outside 1..2^24", V);
    if (K < 1 || K > kMaxTopK) return fail(SC_ERR_SHAPE, "K = %d outside 1..%d", K, kMaxTopK);
    if (logits_stride < V) return fail(SC_ERR_SHAPE, "logits_stride %lld < V = %d", logits_stride, V);
    if (!(inv_temperature > 0.0f) || !std::isfinite(inv_temperature))
        return fail(SC_ERR_ARG, "inv_temperature must be finite and > 0");
    if (!(top_p > 0.0f && top_p <= 1.0f)) return fail(SC_ERR_ARG, "top_p must be in (0, 1]");
    if (T == 0) return ok();
    if (!logits || !ids_out || !logprobs_out) return fail(SC_ERR_NULL, "logits, ids_out and logprobs_out are required");
    if (!aligned(logits, 16) || logits_stride % 4 != 0)
        return fail(SC_ERR_ALIGN, "logits must be 16-byte aligned with a stride that is a multiple of 4");
    if (!aligned(ids_out, 4) || !aligned(logprobs_out, 4) || !aligned(count_out, 4))
        return fail(SC_ERR_ALIGN, "outputs must be 4-byte aligned");
    if (!aligned(workspace, 16)) return fail(SC_ERR_ALIGN, "workspace must be 16-byte aligned");
    int dev = 0;
    int st = check_device(&dev);
    if (st != SC_OK) return st;
    static std::mutex mu;
    static std::map<int, int> grid_for;
    int grid = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = grid_for.find(dev);
        if (it == grid_for.end()) {
            cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(topk_capture_kernel),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(sizeof(KernelShared)));
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(topk smem)");
            int per_sm = 0, sms = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_capture_kernel, kNT, sizeof(KernelShared));
            if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
            if (per_sm < 1) return fail(SC_ERR_UNSUPPORTED, "the top-K kernel does not fit an SM");
            it = grid_for.emplace(dev, per_sm * sms).first;
        }
        grid = it->second;
    }
    TopkArgs ka;
    std::memset(&ka, 0, sizeof ka);
    ka.logits = logits;
    ka.T = T;
    ka.stride = logits_stride;
    ka.V = V;
    ka.K = K;
    ka.inv_t = inv_temperature;
    ka.top_p = top_p;
    ka.ids = ids_out;
    ka.lps = logprobs_out;
    ka.counts = count_out;
    const long long g = T < grid ? T : grid;
    // with a workspace, each thread group's first row is dealt at launch and
    // the rest handed out at run time
    ka.ws = static_cast<unsigned long long*>(workspace);
    const long long ng = g * kGroups;
    ka.T_static = workspace ? (T < ng ? T : ng) : T;
    topk_capture_kernel<<<static_cast<unsigned>(g), kNT, sizeof(KernelShared), reinterpret_cast<cudaStream_t>(stream)>>>(ka);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "topk_capture_kernel launch");
    return ok();
}
