// sc_gemm.cu -- dense bf16 GEMM on the fifth-generation tensor cores (tcgen05),
// the building block of the LM head's three products (z = H W^T, dH = g W,
// dW = g^T H).
//
//   C[M, N] = A[M, K] . B[K, N]      (FP32 accumulation in tensor memory)
//
// A is stored either K-major ([M][K], K contiguous) or M-major ([K][M]); B
// either K-major ([N][K]) or N-major ([K][N]).  C is row-major [M][N] and is
// written as bf16 (round to nearest even), as FP32, or added in FP32 to what C
// already holds (vector reductions performed in L2).
//
// Design (one CTA per SM, persistent over 128 x 256 output tiles):
// * warp 0, one thread: the TMA producer.  For every K step of 64 it loads
//   the A tile (128 x 64) and the B tile (256 x 64) into one of four
//   shared-memory stages with 2-D tensor copies in the 128-byte swizzled
//   layout the tensor cores read, and signals the stage's mbarrier with the
//   bytes in flight.
// * warp 1: allocates the 512 tensor-memory columns (two 128 x 256 FP32
//   accumulators); one thread issues the tcgen05.mma instructions (four of
//   K = 16 per stage) and commits each stage back to the producer and each
//   finished accumulator to the epilogue.
// * warps 2-5: the epilogue.  Each warp owns 32 accumulator rows (the
//   tensor-memory lanes its warp index selects); it reads 32 or 64 columns at a time with tcgen05.ld, converts them, writes
//   them to a swizzled 4 KiB staging buffer and stores them: bf16 with a TMA
//   tensor store (double-buffered); FP32 read back transposed so that each
//   store instruction writes four whole 128-byte row segments (plain 16-byte
//   stores, or vector reductions for the reduce-add), which keeps the TMA unit
//   free for the operand loads where the products with a short K would
//   otherwise wait on it.  It hands the accumulator back as soon as it is read,
//   so the next tile's MMAs overlap this tile's stores.
// Every wait is bounded (about 1 s of %globaltimer); on expiry the kernel
// sets a status bit, stops issuing work, lets the copies and MMAs it started
// complete and frees its tensor memory before it returns.
#include <cuda.h>

#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "sc_device.cuh"
#include "sc_internal.h"

namespace sc {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr int kABytes = BM * BK * 2;             // 16 KiB
constexpr int kBBytes = BN * BK * 2;             // 32 KiB
constexpr int kStageBytes = kABytes + kBBytes;   // 48 KiB
constexpr int kEpiBuf = 32 * 128;                // one warp's staging buffer: 32 rows x 128 B
constexpr int kEpiWarps = 4;  // one per tensor-memory lane quadrant (measured: eight were slower)
constexpr int kThreads = 64 + 32 * kEpiWarps;    // producer, MMA, four epilogue warps
constexpr int kTmemCols = 512;                   // two accumulators of BN FP32 columns
constexpr int kSmemData = kStages * kStageBytes + kEpiWarps * 2 * kEpiBuf;
constexpr int kSmemBars = 256;
constexpr int kSmemTotal = kSmemData + kSmemBars + 1024;  // + alignment slack
constexpr unsigned long long kWaitNs = 1000000000ull;
constexpr uint32_t kStatusTimeout = 0x2u;         // SC_STATUS_TIMEOUT_LOAD

static_assert(kSmemTotal <= 232448, "shared memory per CTA");

struct GemmArgs {
    long long M, N, K;
    long long N_full;  // columns stored in whole 16-byte units: N rounded down to them
    void* C;           // C itself, for the columns past N_full (plain stores)
    long long ldc;
    int num_m, num_n, k_steps;
    int k_splits, kps;  // split-K: the K steps of a tile in k_splits ranges of kps
    long long c_split_rows;  // split s stores its rows at C row s * c_split_rows + m
    long long tiles;    // output tiles times k_splits
    int a_mn, b_mn;   // operand majorness: 0 K-major, 1 M- / N-major
    int c_mode;       // 0 bf16 store, 1 FP32 store, 2 FP32 reduce-add
    int m_fastest;    // tile order: consecutive tiles share their B tile (1) or their A tile (0)
    uint32_t idesc;   // tcgen05 instruction descriptor
    uint32_t* status;
};

// ---- tcgen05 / TMA tensor helpers -------------------------------------------

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// 16 bytes to global memory (16-byte aligned), and the FP32 vector reduction
__device__ __forceinline__ void st_v4(void* p, const uint4& w) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w)
                 : "memory");
}
__device__ __forceinline__ void red_add_v4f32(void* p, const uint4& w) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(__uint_as_float(w.x)),
                 "f"(__uint_as_float(w.y)), "f"(__uint_as_float(w.z)), "f"(__uint_as_float(w.w))
                 : "memory");
}
// A hint that brings the 128-byte line at p into L2 (nothing is returned).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}
// At most one committed store group may still be reading shared memory.
__device__ __forceinline__ void bulk_wait_read_le1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// D[tmem] (+)= A[smem] . B[smem], kind::f16 (bf16 inputs, FP32 accumulator).
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// 32 consecutive FP32 columns of this warp's 32 lanes: one row per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Shared-memory matrix descriptor of a tile in the 128-byte swizzled layout
// (start, leading and stride byte offsets in 16-byte units; version 1;
// layout type 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Descriptor of the K = 16 slice kk (0..3) of a stage's operand tile.
// K-major: rows of 64 elements (128 B), 8-row groups 1024 B apart; the slice
// starts 32 B further along the row.  M-/N-major: 64-element blocks of the
// M (N) extent 8 KiB apart (one TMA box of 64 K rows each), 8-row groups of K
// 1024 B apart; the slice starts 16 rows (2 KiB) further down.
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int mn_major, int kk) {
    return mn_major ? smem_desc(base + 2048u * kk, 8192u, 1024u) : smem_desc(base + 32u * kk, 16u, 1024u);
}

// CM: the output mode (0 bf16, 1 FP32, 2 FP32 reduce-add), one instance each,
// so that each carries only its own epilogue.
template <int CM>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ GemmArgs g, const __grid_constant__ CUtensorMap tmA,
                const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // the swizzled layouts repeat every 1024 B
    unsigned char* sbase = smem_raw + (base - raw);
    const uint32_t stage0 = base;
    const uint32_t epi0 = base + kStages * kStageBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sbase + kSmemData);
    // bars: full[kStages], empty[kStages], acc_full[2], acc_empty[2], drain
    auto full = [&](int s) { return smem_addr(&bars[s]); };
    auto empty = [&](int s) { return smem_addr(&bars[kStages + s]); };
    auto acc_full = [&](int a) { return smem_addr(&bars[2 * kStages + a]); };
    auto acc_empty = [&](int a) { return smem_addr(&bars[2 * kStages + 2 + a]); };
    const uint32_t drain = smem_addr(&bars[2 * kStages + 4]);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbase + kSmemData + 128);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + kSmemData + 136);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full(s), 1u);
            mbar_init(empty(s), 1u);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full(a), 1u);
            mbar_init(acc_empty(a), static_cast<uint32_t>(kEpiWarps));
        }
        mbar_init(drain, 1u);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto give_up = [&]() {
        if (g.status) atomicOr(g.status, kStatusTimeout);
        *abort_flag = 1;
    };
    // tile t: split t / (num_m num_n) (the slowest index, so that consecutive
    // tiles share operand tiles as within one split), then m and n in the
    // chosen order; its K steps [ks0, ks1)
    auto tile_coords = [&](long long t, int& mt, int& nt, int& ks0, int& ks1) {
        const long long t2 = static_cast<long long>(g.num_m) * g.num_n;
        const int split = static_cast<int>(t / t2);
        const long long r = t - split * t2;
        if (g.m_fastest) {
            mt = static_cast<int>(r % g.num_m);
            nt = static_cast<int>(r / g.num_m);
        } else {
            nt = static_cast<int>(r % g.num_n);
            mt = static_cast<int>(r / g.num_n);
        }
        ks0 = split * g.kps;
        ks1 = min(g.k_steps, ks0 + g.kps);
    };

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            uint32_t it = 0;  // stages issued
            for (long long t = blockIdx.x; t < g.tiles && !*abort_flag; t += gridDim.x) {
                int mt, nt, ks0, ks1;
                tile_coords(t, mt, nt, ks0, ks1);
                const int m0 = mt * BM, n0 = nt * BN;
                for (int ks = ks0; ks < ks1; ++ks, ++it) {
                    const int s = static_cast<int>(it % kStages);
                    if (it >= static_cast<uint32_t>(kStages) &&
                        !mbar_wait_bounded(empty(s), ((it / kStages) - 1u) & 1u, kWaitNs)) {
                        give_up();
                        break;
                    }
                    const uint32_t sa = stage0 + s * kStageBytes, sb = sa + kABytes;
                    mbar_expect_tx(full(s), static_cast<uint32_t>(kStageBytes));
                    const int k0 = ks * BK;
                    if (g.a_mn) {
                        tma_load_2d(sa, &tmA, m0, k0, full(s));
                        tma_load_2d(sa + 8192u, &tmA, m0 + 64, k0, full(s));
                    } else {
                        tma_load_2d(sa, &tmA, k0, m0, full(s));
                    }
                    if (g.b_mn) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) tma_load_2d(sb + 8192u * j, &tmB, n0 + 64 * j, k0, full(s));
                    } else {
                        tma_load_2d(sb, &tmB, k0, n0, full(s));
                    }
                }
            }
            // copies in flight land before the CTA can leave
            const uint32_t first = it > static_cast<uint32_t>(kStages) ? it - kStages : 0u;
            for (uint32_t j = first; j < it; ++j)
                (void)mbar_wait_bounded(full(static_cast<int>(j % kStages)), (j / kStages) & 1u, kWaitNs);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            uint32_t it = 0, lt = 0;  // stages consumed, local tiles
            bool ok = true;
            for (long long t = blockIdx.x; t < g.tiles && ok && !*abort_flag; t += gridDim.x, ++lt) {
                const int acc = static_cast<int>(lt & 1u);
                if (lt >= 2u && !mbar_wait_bounded(acc_empty(acc), ((lt >> 1) - 1u) & 1u, kWaitNs)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * BN);
                int mt, nt, ks0, ks1;
                tile_coords(t, mt, nt, ks0, ks1);
                for (int ks = ks0; ks < ks1; ++ks, ++it) {
                    const int s = static_cast<int>(it % kStages);
                    if (!mbar_wait_bounded(full(s), (it / kStages) & 1u, kWaitNs)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = stage0 + s * kStageBytes, sb = sa + kABytes;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma(d, operand_desc(sa, g.a_mn, kk), operand_desc(sb, g.b_mn, kk), g.idesc,
                               (ks != ks0 || kk != 0) ? 1u : 0u);
                    tc_commit(empty(s));  // the stage is free once these MMAs have read it
                }
                if (ok) tc_commit(acc_full(acc));
            }
            // every MMA issued has completed before the tensor memory is freed
            tc_commit(drain);
            (void)mbar_wait_bounded(drain, 0u, kWaitNs);
        }
    } else {
        // ================= epilogue: tensor memory -> global =================
        const int q = warp & 3;  // tensor-memory lanes 32q .. 32q + 31
        const uint32_t buf0 = epi0 + static_cast<uint32_t>((warp - 2) * 2 * kEpiBuf);
        const int cols = CM == 0 ? 64 : 32;  // columns per 128-byte staging row
        const int nchunks = BN / cols;
        uint32_t lt = 0, nst = 0;
        for (long long t = blockIdx.x; t < g.tiles; t += gridDim.x, ++lt) {
            const int acc = static_cast<int>(lt & 1u);
            // (the decision to leave is taken warp-wide: the loads below are .sync.aligned)
            const bool got = mbar_wait_bounded(acc_full(acc), (lt >> 1) & 1u, kWaitNs);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) give_up();
                break;
            }
            tc_fence_after();
            int mt, nt, ks0, ks1;
            tile_coords(t, mt, nt, ks0, ks1);
            const long long r0 = static_cast<long long>(mt) * BM + 32 * q;
            const long long roff = g.kps > 0 ? static_cast<long long>(ks0 / g.kps) * g.c_split_rows : 0;
            const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(acc * BN);
            if constexpr (CM == 2) {
                // The C rows that this lane's reductions will add to in the CTA's next
                // tile, brought into L2 one tile ahead, so that the reductions find
                // their lines there (blocked LM head, dW added to by blocks 1..:
                // 11.50-11.62 -> 11.25-11.33 ms; plain loads, an add and stores
                // instead of the reductions were slower, 11.93-12.18 ms).
                const long long tn = t + gridDim.x;
                if (tn < g.tiles) {
                    int mt2, nt2, ka, kb;
                    tile_coords(tn, mt2, nt2, ka, kb);
                    const long long prow = static_cast<long long>(mt2) * BM + 32 * q + lane;
                    const long long pcol = static_cast<long long>(nt2) * BN;
                    if (prow < g.M) {
                        const char* pr = static_cast<const char*>(g.C) + (prow * g.ldc + pcol) * 4;
#pragma unroll
                        for (int j = 0; j < BN / 32; ++j)
                            if (pcol + 32 * j < g.N) prefetch_l2(pr + 128 * j);
                    }
                }
            }
            for (int c = 0; c < nchunks; ++c) {
                const long long c0 = static_cast<long long>(nt) * BN + c * cols;
                if (r0 >= g.M || c0 >= g.N) break;  // (chunks are in column order)
                // The 16-byte units of a row before N_full are stored whole; the
                // few columns past it (N not a multiple of 16 bytes) one by one below.
                uint32_t v[64];
                uint32_t(&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
                uint32_t(&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
                tmem_ld32(tbase + static_cast<uint32_t>(c * cols), lo);
                if (cols == 64) tmem_ld32(tbase + static_cast<uint32_t>(c * cols + 32), hi);
                tmem_ld_wait();
                if (c0 + cols > g.N_full) {
                    // columns [max(c0, N_full), N) of this thread's row, one by one
                    const long long row = r0 + lane;
                    if (row < g.M) {
                        const long long crow = roff + row;
#pragma unroll
                        for (int j = 0; j < 64; ++j) {
                            const long long col = c0 + j;
                            if (j < cols && col >= g.N_full && col < g.N) {
                                if (CM == 0) {
                                    uint16_t* cp = static_cast<uint16_t*>(g.C) + crow * g.ldc + col;
                                    *cp = static_cast<uint16_t>(pack_bf16x2(__uint_as_float(v[j]), 0.0f) & 0xFFFFu);
                                } else if (CM == 1) {
                                    static_cast<float*>(g.C)[crow * g.ldc + col] = __uint_as_float(v[j]);
                                } else {
                                    atomicAdd(static_cast<float*>(g.C) + crow * g.ldc + col, __uint_as_float(v[j]));
                                }
                            }
                        }
                    }
                    if (c0 >= g.N_full) continue;  // nothing of this chunk in whole units
                }
                if constexpr (CM == 0) {
                    // bf16: a TMA tensor store per chunk, double-buffered (measured faster
                    // than plain stores on the long-K products that write bf16)
                    const uint32_t buf = buf0 + static_cast<uint32_t>((nst & 1u) * kEpiBuf);
                    if (lane == 0) bulk_wait_read_le1();  // the store that used this buffer has read it
                    __syncwarp();
                    const uint32_t row = buf + 128u * lane;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint32_t w0, w1, w2, w3;
                        if (cols == 64) {  // eight bf16 per 16-byte chunk, round to nearest even
                            w0 = pack_bf16x2(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1]));
                            w1 = pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3]));
                            w2 = pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5]));
                            w3 = pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]));
                        } else {
                            w0 = v[4 * j + 0];
                            w1 = v[4 * j + 1];
                            w2 = v[4 * j + 2];
                            w3 = v[4 * j + 3];
                        }
                        sts128(row + 16u * static_cast<uint32_t>(j ^ (lane & 7)), w0, w1, w2, w3);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, static_cast<int>(c0), static_cast<int>(roff + r0), buf);
                        bulk_commit_group();
                    }
                    ++nst;
                    continue;
                }
                // Staged through this warp's swizzled 4 KiB buffer and read back
                // transposed, so that each store instruction writes four whole
                // 128-byte row segments; plain stores (or vector reductions) keep
                // the epilogue out of the TMA unit, which the operand loads need.
                const uint32_t buf = buf0;
                __syncwarp();  // every lane has read the previous chunk back
                const uint32_t row = buf + 128u * lane;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint32_t w0, w1, w2, w3;
                    if (cols == 64) {  // eight bf16 per 16-byte chunk, round to nearest even
                        w0 = pack_bf16x2(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1]));
                        w1 = pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3]));
                        w2 = pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5]));
                        w3 = pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]));
                    } else {
                        w0 = v[4 * j + 0];
                        w1 = v[4 * j + 1];
                        w2 = v[4 * j + 2];
                        w3 = v[4 * j + 3];
                    }
                    sts128(row + 16u * static_cast<uint32_t>(j ^ (lane & 7)), w0, w1, w2, w3);
                }
                __syncwarp();
                {
                    const int seg = lane & 7;  // 16-byte segment of a row
                    const int esz = CM == 0 ? 2 : 4;
                    const long long col = c0 + seg * (16 / esz);
                    if (col < g.N_full) {  // (N_full counts whole 16-byte units)
#pragma unroll
                        for (int it = 0; it < 8; ++it) {
                            const int rr = 4 * it + (lane >> 3);
                            if (r0 + rr < g.M) {
                                const uint4 w = lds128(buf + 128u * static_cast<uint32_t>(rr) +
                                                       16u * static_cast<uint32_t>(seg ^ (rr & 7)));
                                char* dst = static_cast<char*>(g.C) + ((roff + r0 + rr) * g.ldc + col) * esz;
                                if (CM == 2)
                                    red_add_v4f32(dst, w);
                                else
                                    st_v4(dst, w);
                            }
                        }
                    }
                }
            }
            // the accumulator is read: the MMAs of a later tile may use it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(acc));
        }
        if (lane == 0) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---- host side ----------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_gemm_mutex;
EncodeTiledFn g_encode = nullptr;
std::map<int, int> g_gemm_attr;  // device -> attributes set
std::map<int, int> g_sm_count;   // device -> SMs

int encoder(EncodeTiledFn* out) {
    std::lock_guard<std::mutex> lock(g_gemm_mutex);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                               cudaEnableDefault, &q);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)");
        if (q != cudaDriverEntryPointSuccess || !fn)
            return fail(SC_ERR_UNSUPPORTED, "the driver has no cuTensorMapEncodeTiled");
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    *out = g_encode;
    return SC_OK;
}

// 2-D tensor map of a row-major matrix [rows][cols] (cols contiguous, row
// stride `ld` elements), boxes of box_cols x box_rows, 128-byte swizzle.
int make_map(EncodeTiledFn enc, CUtensorMap* map, const void* ptr, CUtensorMapDataType dt, int esize,
             long long rows, long long cols, long long ld, int box_cols, int box_rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * static_cast<cuuint64_t>(esize)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(SC_ERR_ARG, "cuTensorMapEncodeTiled failed (%d) for a %lld x %lld matrix, row stride %lld",
                    static_cast<int>(r), rows, cols, ld);
    return SC_OK;
}

// tcgen05 instruction descriptor, kind::f16: FP32 accumulator, bf16 A and B,
// operand majorness, N / 8 and M / 16.
uint32_t instr_desc(int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
           (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(BN >> 3) << 17) |
           (static_cast<uint32_t>(BM >> 4) << 24);
}

}  // namespace

int gemm_bf16(const uint16_t* A, long long lda, int a_mn, const uint16_t* B, long long ldb, int b_mn, void* C,
              long long ldc, int c_mode, long long M, long long N, long long K, int m_fastest, uint32_t* status,
              cudaStream_t stream, int k_splits) {
    if (M < 1 || N < 1 || K < 1) return fail(SC_ERR_SHAPE, "GEMM sizes M=%lld N=%lld K=%lld must be >= 1", M, N, K);
    if (M > (1LL << 31) || N > (1LL << 31) || K > (1LL << 31))
        return fail(SC_ERR_SHAPE, "GEMM sizes must be below 2^31");
    if (c_mode < 0 || c_mode > 2) return fail(SC_ERR_ARG, "c_mode = %d", c_mode);
    if (k_splits < 1 || (k_splits > 1 && c_mode != 1)) return fail(SC_ERR_ARG, "split K stores FP32 slices");
    if (!A || !B || !C) return fail(SC_ERR_NULL, "A, B and C are required");
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || !aligned(status, 4))
        return fail(SC_ERR_ALIGN, "A, B and C must be 16-byte aligned");
    const int cesize = c_mode == 0 ? 2 : 4;
    if (lda % 8 || ldb % 8 || (ldc * cesize) % 16)
        return fail(SC_ERR_ALIGN, "row strides must be multiples of 16 bytes");
    if (lda < (a_mn ? M : K) || ldb < (b_mn ? N : K) || ldc < N)
        return fail(SC_ERR_SHAPE, "a row stride is shorter than its row");
    EncodeTiledFn enc = nullptr;
    int st = encoder(&enc);
    if (st != SC_OK) return st;
    CUtensorMap ta, tb, tc;
    st = a_mn ? make_map(enc, &ta, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, M, lda, 64, 64)
              : make_map(enc, &ta, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, K, lda, 64, BM);
    if (st != SC_OK) return st;
    st = b_mn ? make_map(enc, &tb, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, N, ldb, 64, 64)
              : make_map(enc, &tb, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, N, K, ldb, 64, BN);
    if (st != SC_OK) return st;
    const long long per16 = 16 / cesize;              // elements in a 16-byte unit
    const long long n_full = N / per16 * per16;        // columns stored in whole 16-byte units
    // with split K, C holds one slice of round_up(M, BM) rows per split
    const long long ksteps = (K + BK - 1) / BK;
    const long long kps = (ksteps + k_splits - 1) / k_splits;
    const long long splits = (ksteps + kps - 1) / kps;  // (no empty ranges)
    const long long m_pad = (M + BM - 1) / BM * BM;
    const long long c_rows = splits > 1 ? splits * m_pad : M;
    const long long n_map = n_full > 0 ? n_full : per16;  // (a map needs a nonzero extent)
    // (the kernel's tensor stores use it for bf16 output; the FP32 modes store with
    // plain 16-byte stores and vector reductions)
    st = c_mode == 0 ? make_map(enc, &tc, C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c_rows, n_map, ldc, 64, 32)
                     : make_map(enc, &tc, C, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, c_rows, n_map, ldc, 32, 32);
    if (st != SC_OK) return st;
    int dev = 0;
    st = check_device(&dev);
    if (st != SC_OK) return st;
    int sms = 0;
    {
        std::lock_guard<std::mutex> lock(g_gemm_mutex);
        if (!g_gemm_attr.count(dev)) {
            for (const void* fn : {reinterpret_cast<const void*>(gemm_kernel<0>),
                                   reinterpret_cast<const void*>(gemm_kernel<1>),
                                   reinterpret_cast<const void*>(gemm_kernel<2>)}) {
                const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTotal);
                if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(gemm smem)");
            }
            int n = 0;
            const cudaError_t e2 = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
            if (e2 != cudaSuccess) return cuda_fail(e2, "cudaDeviceGetAttribute(SMs)");
            g_sm_count[dev] = n;
            g_gemm_attr[dev] = 1;
        }
        sms = g_sm_count[dev];
    }
    GemmArgs ga;
    std::memset(&ga, 0, sizeof ga);
    ga.M = M;
    ga.N = N;
    ga.K = K;
    ga.N_full = n_full;
    ga.C = C;
    ga.ldc = ldc;
    ga.num_m = static_cast<int>((M + BM - 1) / BM);
    ga.num_n = static_cast<int>((N + BN - 1) / BN);
    ga.k_steps = static_cast<int>(ksteps);
    ga.kps = static_cast<int>(kps);
    ga.k_splits = static_cast<int>(splits);
    ga.c_split_rows = splits > 1 ? m_pad : 0;
    ga.tiles = static_cast<long long>(ga.num_m) * ga.num_n * ga.k_splits;
    ga.a_mn = a_mn ? 1 : 0;
    ga.b_mn = b_mn ? 1 : 0;
    ga.c_mode = c_mode;
    ga.m_fastest = m_fastest ? 1 : 0;
    ga.idesc = instr_desc(ga.a_mn, ga.b_mn);
    ga.status = status;
    const long long grid = ga.tiles < sms ? ga.tiles : sms;
    const dim3 gdim(static_cast<unsigned>(grid));
    if (c_mode == 0)
        gemm_kernel<0><<<gdim, kThreads, kSmemTotal, stream>>>(ga, ta, tb, tc);
    else if (c_mode == 1)
        gemm_kernel<1><<<gdim, kThreads, kSmemTotal, stream>>>(ga, ta, tb, tc);
    else
        gemm_kernel<2><<<gdim, kThreads, kSmemTotal, stream>>>(ga, ta, tb, tc);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "gemm_kernel launch");
    return SC_OK;
}

namespace {

// The sum of `splits` FP32 slices [rows][cols] (row stride lds, slice s
// starting s * slice rows further) -> bf16 (row stride ldd), round to nearest
// even; the slices added in slice order.  Eight columns per thread.
__global__ void sum_slices_to_bf16_kernel(const float* src, long long lds, long long slice, int splits, uint16_t* dst,
                                          long long ldd, long long rows, long long cols) {
    const long long c8 = (cols + 7) / 8;
    const long long n = rows * c8;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long r = i / c8, c = (i - r * c8) * 8;
        uint16_t* dp = dst + r * ldd + c;
        if (c + 8 <= cols) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            for (int sp = 0; sp < splits; ++sp) {
                const float* p = src + (sp * slice + r) * lds + c;
                const float4 x = *reinterpret_cast<const float4*>(p);
                const float4 y = *reinterpret_cast<const float4*>(p + 4);
                a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
                b.x += y.x; b.y += y.y; b.z += y.z; b.w += y.w;
            }
            uint4 o;
            o.x = pack_bf16x2(a.x, a.y);
            o.y = pack_bf16x2(a.z, a.w);
            o.z = pack_bf16x2(b.x, b.y);
            o.w = pack_bf16x2(b.z, b.w);
            *reinterpret_cast<uint4*>(dp) = o;
        } else {
            for (long long j = 0; c + j < cols; ++j) {
                float v = 0.0f;
                for (int sp = 0; sp < splits; ++sp) v += src[(sp * slice + r) * lds + c + j];
                dp[j] = static_cast<uint16_t>(pack_bf16x2(v, 0.0f) & 0xFFFFu);
            }
        }
    }
}

}  // namespace

// Splits of K that fill the SMs best for an M x N output: the count in 1..8
// whose tiles come closest to whole waves (the smallest on a tie).
int best_k_splits(long long M, long long N, long long K, int sms) {
    const long long tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const long long ksteps = (K + BK - 1) / BK;
    int best = 1;
    double best_eff = 0.0;
    for (int s = 1; s <= 8 && s <= ksteps / 8 + 1; ++s) {
        const double waves = static_cast<double>(tiles * s) / sms;
        const double eff = waves / static_cast<double>((tiles * s + sms - 1) / sms);
        if (eff > best_eff + 1e-3) {
            best_eff = eff;
            best = s;
        }
    }
    return best;
}

int sm_count(int* out) {
    int dev = 0;
    int st = check_device(&dev);
    if (st != SC_OK) return st;
    std::lock_guard<std::mutex> lock(g_gemm_mutex);
    if (!g_sm_count.count(dev)) {
        int n = 0;
        const cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SMs)");
        g_sm_count[dev] = n;
    }
    *out = g_sm_count[dev];
    return SC_OK;
}

// Rows of the FP32 slices gemm_bf16_split needs for an M-row product.
long long split_slice_rows(long long M) { return (M + BM - 1) / BM * BM; }

// C (bf16) = A . B with K split `k_splits` ways: split s stores its FP32
// partial product in slice s of acc (split_slice_rows(M) rows each, row
// stride ldacc, a multiple of 4), and one kernel adds the slices in slice order
// and rounds the sum to C -- the same bits whatever order the tiles ran in.
int gemm_bf16_split(const uint16_t* A, long long lda, int a_mn, const uint16_t* B, long long ldb, int b_mn,
                    uint16_t* C, long long ldc, float* acc, long long ldacc, long long M, long long N, long long K,
                    int m_fastest, int k_splits, uint32_t* status, cudaStream_t stream) {
    if (k_splits <= 1)
        return gemm_bf16(A, lda, a_mn, B, ldb, b_mn, C, ldc, 0, M, N, K, m_fastest, status, stream, 1);
    int st = gemm_bf16(A, lda, a_mn, B, ldb, b_mn, acc, ldacc, 1, M, N, K, m_fastest, status, stream, k_splits);
    if (st != SC_OK) return st;
    const long long ksteps = (K + BK - 1) / BK, kps = (ksteps + k_splits - 1) / k_splits;
    const int splits = static_cast<int>((ksteps + kps - 1) / kps);
    const long long work = M * ((N + 7) / 8);
    const int blocks = static_cast<int>(work / 256 + 1 < 4096 ? work / 256 + 1 : 4096);
    sum_slices_to_bf16_kernel<<<blocks, 256, 0, stream>>>(acc, ldacc, split_slice_rows(M), splits, C, ldc, M, N);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "sum_slices_to_bf16_kernel launch");
    return SC_OK;
}

}  // namespace sc

extern "C" int sc_gemm_bf16(const uint16_t* A, long long lda, int a_layout, const uint16_t* B, long long ldb,
                            int b_layout, void* C, long long ldc, int c_mode, long long M, long long N, long long K,
                            uint32_t* status_dev, sc_stream_t stream) {
    using namespace sc;
    if (a_layout != 0 && a_layout != 1) return fail(SC_ERR_ARG, "a_layout = %d", a_layout);
    if (b_layout != 0 && b_layout != 1) return fail(SC_ERR_ARG, "b_layout = %d", b_layout);
    // consecutive output tiles share the larger operand's tile, so that it
    // streams from HBM once while the smaller one is re-read from L2
    const int m_fastest = M <= N ? 1 : 0;
    const int st = gemm_bf16(A, lda, a_layout, B, ldb, b_layout, C, ldc, c_mode, M, N, K, m_fastest, status_dev,
                             reinterpret_cast<cudaStream_t>(stream), 1);
    if (st != SC_OK) return st;
    return ok();
}
