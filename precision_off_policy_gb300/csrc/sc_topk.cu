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
};

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

// A thread group's view: its threads, its named barrier, its shared state.
struct GroupShared {
    uint32_t keys[kGT];                 // the sample maxima, sorted
    unsigned long long cand[kCap];      // (key << 32) | ~id
    float fred[kGW], flo[kGW];          // group maximum / sums of pairs
    double dS, dlse;
    double pnuc, lnuc;  // the nucleus mass and log(nucleus mass / normaliser)
    int ncand, cross;
};
struct KernelShared {
    union {
        Shared exact;                   // the exact path: the whole CTA, between rounds
        GroupShared grp[kGroups];       // the one-pass path: one per group
    } u;
    int ndefer;
    long long defer[kGroups * kRound];  // rows of this round left to the exact path
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
// Bitonic sort of cand[0, n), larger first (n <= kCap), by the group.
__device__ void group_sort_desc(GroupShared& gs, const Group& G, int n) {
    int m = 1;
    while (m < n) m <<= 1;
    for (int i = n + G.tid; i < m; i += kGT) gs.cand[i] = 0ull;
    G.sync();
    for (int k = 2; k <= m; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = G.tid; i < m; i += kGT) {
                const int l = i ^ j;
                if (l > i) {
                    const unsigned long long x = gs.cand[i], y = gs.cand[l];
                    if (((i & k) == 0) ? (x < y) : (x > y)) {
                        gs.cand[i] = y;
                        gs.cand[l] = x;
                    }
                }
            }
            G.sync();
        }
}

// The one-pass path for one row, run by one thread group.  A sample (every
// kSampEvery-th run of vectors) gives each thread a maximum; the largest of
// those maxima is the exponent offset, and the `rank`-th largest the candidate
// threshold, placed so that about 3 K entries of the row reach it.  One pass
// over the row then sums 2^((z - m) kt) per thread (compensated, in a fixed
// order; a thread that meets an entry above its offset m moves m up) and
// collects every entry at or above the threshold.  The candidates are
// sorted; the top K and, with top_p < 1, the nucleus come from them.  Returns
// false -- outputs untouched, the same decision in every thread of the group
// -- when the row needs the exact path: too few or too many candidates, a
// nucleus that reaches below them, entries that are not finite, or K above
// kCap / 4.
__device__ bool fast_row(GroupShared& gs, const Group& G, const TopkArgs& a, long long t) {
    const float* row = a.logits + t * a.stride;
    const int V = a.V, tid = G.tid, lane = G.lane, warp = G.warp;
    const int Kp = min(a.K, V);
    if (4 * Kp > kCap) return false;
    const float kt = a.inv_t * kLog2e;
    const int nv4 = V >> 2;
    const float4* r4 = reinterpret_cast<const float4*>(row);

    // ---- the threshold and the offset from the sample
    float tau = -INFINITY;  // candidates: z >= tau (-inf: every entry)
    float o = -INFINITY;    // exponent offset of the sums
    if (V > kCap) {
        const int nruns = nv4 / kSampRun;
        float smax = -INFINITY;
        for (int r = warp * kSampEvery; r < nruns; r += kGW * kSampEvery) {
            const float4 v = __ldg(r4 + r * kSampRun + lane);
            smax = fmaxf(smax, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
        }
        group_sort_keys_desc(gs, G, key_of(smax));
        const int rank = min(kGT, max(8, (3 * Kp + kSampEvery - 1) / kSampEvery));
        tau = float_of(gs.keys[rank - 1]);
        o = float_of(gs.keys[0]);
        G.sync();
        if (!isfinite(o)) return false;
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
        int i = tid;
        for (; i + (kUnroll - 1) * kGT < nv4; i += kUnroll * kGT) {
            float4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) v[u] = __ldg(r4 + i + u * kGT);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) take4(v[u], 4 * (i + u * kGT));
        }
        for (; i < nv4; i += kGT) take4(__ldg(r4 + i), 4 * i);
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
        gs.dlse = (double)M * a.inv_t + log(S);
    }
    G.sync();
    const double S = gs.dS, lse = gs.dlse;
    const int nc = gs.ncand;
    if (!isfinite(M) || !(S > 0.0) || !isfinite(S) || !isfinite(lse) || nc < Kp || nc > kCap) return false;
    group_sort_desc(gs, G, nc);

    // ---- the nucleus: one warp walks the sorted candidates with error-free
    // FP32 running sums
    int count = Kp;
    double log_nuc = 0.0;
    if (a.top_p < 1.0f) {
        if (warp == 0) {
            const double thr = (double)a.top_p * S;
            const float t_hi = (float)thr, t_lo = (float)(thr - (double)t_hi);
            const int per = (nc + 31) / 32;
            const int i0 = lane * per, i1 = min(nc, i0 + per);
            auto mass = [&](int i) { return ex2((float_of(static_cast<uint32_t>(gs.cand[i] >> 32)) - M) * kt); };
            Pair loc{0.0f, 0.0f};
            for (int i = i0; i < i1; ++i) loc = pair_add(loc, Pair{mass(i), 0.0f});
            // exclusive scan of the lanes' pairs, in lane order
            Pair inc = loc;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const Pair y{__shfl_up_sync(0xFFFFFFFFu, inc.hi, d), __shfl_up_sync(0xFFFFFFFFu, inc.lo, d)};
                if (lane >= d) inc = pair_add(y, inc);
            }
            const Pair all{__shfl_sync(0xFFFFFFFFu, inc.hi, 31), __shfl_sync(0xFFFFFFFFu, inc.lo, 31)};
            Pair run{__shfl_up_sync(0xFFFFFFFFu, inc.hi, 1), __shfl_up_sync(0xFFFFFFFFu, inc.lo, 1)};
            if (lane == 0) run = Pair{0.0f, 0.0f};
            // first candidate whose preceding mass reaches thr
            int mine = nc + 1;
            for (int i = i0; i < i1; ++i) {
                if ((run.hi - t_hi) + (run.lo - t_lo) >= 0.0f) {
                    mine = i;
                    break;
                }
                run = pair_add(run, Pair{mass(i), 0.0f});
            }
            int cross = mine;
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) cross = min(cross, __shfl_xor_sync(0xFFFFFFFFu, cross, o2));
            if (lane == 0) {
                gs.cross = cross;
                if (cross > nc) gs.pnuc = (all.hi - t_hi) + (all.lo - t_lo) >= 0.0f ? (double)all.hi + (double)all.lo : -1.0;
            }
            if (mine == cross && cross <= nc) gs.pnuc = (double)run.hi + (double)run.lo;
            __syncwarp();
            // the one FP64 logarithm of the nucleus, in one thread (GB300's FP64
            // rate is a small fraction of its FP32 rate)
            if (lane == 0) gs.lnuc = gs.pnuc > 0.0 ? log(gs.pnuc / S) : 0.0;
        }
        G.sync();
        const int cross = gs.cross;
        const double P = gs.pnuc;
        log_nuc = gs.lnuc;
        G.sync();
        if (!(P > 0.0)) return false;  // the nucleus reaches below the candidates
        count = min(Kp, cross <= nc ? cross : nc);
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

// Rows are dealt to the thread groups round robin (group b * kGroups + g of
// the grid takes rows b * kGroups + g + k * groups).  Each group takes its
// rows on the one-pass path; a row it cannot finish waits for the end of the
// round, when the whole CTA takes the deferred rows on the exact path.
__global__ void __launch_bounds__(kNT, 2) topk_capture_kernel(const __grid_constant__ TopkArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    KernelShared& ks = *reinterpret_cast<KernelShared*>(smem_raw);
    const Group G{static_cast<int>(threadIdx.x) / kGT, static_cast<int>(threadIdx.x) % kGT,
                  static_cast<int>(threadIdx.x) & 31, (static_cast<int>(threadIdx.x) % kGT) >> 5};
    const long long ngroups = static_cast<long long>(gridDim.x) * kGroups;
    const long long first = static_cast<long long>(blockIdx.x) * kGroups;  // this CTA's first group
    // rounds: as many as the CTA's first group has rows (the others have at most as many)
    const long long rows0 = first < a.T ? (a.T - first + ngroups - 1) / ngroups : 0;
    if (threadIdx.x == 0) ks.ndefer = 0;
    __syncthreads();
    for (long long k0 = 0; k0 < rows0; k0 += kRound) {
        const long long k1 = min(rows0, k0 + kRound);
        for (long long k = k0; k < k1; ++k) {
            const long long t = first + G.id + k * ngroups;
            if (t >= a.T) break;
            if (!fast_row(ks.u.grp[G.id], G, a, t) && G.tid == 0) ks.defer[atomicAdd(&ks.ndefer, 1)] = t;
        }
        __syncthreads();
        const int nd = ks.ndefer;
        for (int q = 0; q < nd; ++q) exact_row(ks.u.exact, a, ks.defer[q]);
        __syncthreads();
        if (threadIdx.x == 0) ks.ndefer = 0;
        __syncthreads();
    }
}

}  // namespace
}  // namespace sc

extern "C" int sc_topk_capture(const float* logits, long long T, int V, long long logits_stride, float inv_temperature,
                               int K, float top_p, int32_t* ids_out, float* logprobs_out, int32_t* count_out,
                               sc_stream_t stream) {
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
    topk_capture_kernel<<<static_cast<unsigned>(g), kNT, sizeof(KernelShared), reinterpret_cast<cudaStream_t>(stream)>>>(ka);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "topk_capture_kernel launch");
    return ok();
}
