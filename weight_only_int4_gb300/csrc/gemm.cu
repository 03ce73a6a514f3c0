// Prefill GEMM of the W4A16 layer on the 5th-generation tensor cores.
//
// Design: clusters of two CTAs (one per SM) form a CTA pair that owns 256 x 256
// output tiles, persistently. CTA r of the pair holds rows [128r, 128r + 128)
// of the tile's x block and dequantises columns [128r, 128r + 128) of its
// weight block; one thread of the even CTA issues tcgen05.mma.cta_group::2
// (M=256, N=256, K=16), which reads A and B from both CTAs' shared memory and
// leaves each CTA's 128 rows of the FP32 accumulator in its own tensor memory.
// Per 64-deep K step an SM therefore receives 16 KB of x and 4 KB of packed
// weights for 4.2 MFLOP, half the x bytes of a single-CTA 256 x 128 tile.
//
// Warp roles, in each CTA of the pair:
//   warp 0      producer: TMA brings the CTA's x block [128 x 64] (128-byte
//               swizzle) and packed weight tile [8 words x 128]; the warp's
//               lanes stage the step's scales and zero-point words with
//               cp.async (zero-filled outside N and K). All of it lands in
//               one stage of a load ring and completes one mbarrier.
//   warps 8-23  (two groups of eight, alternate K steps) dequantise the packed tile ONCE into a [128 x 64] fp16/bf16
//               operand tile in the canonical K-major 128-byte-swizzled layout
//               the MMA reads: w = (q - z) * s, with (q - z) exact in 16-bit
//               arithmetic and one rounding for the product. This is the
//               cooperative shared tile of "ROCm KQuantGemmKWmmaQ4K/Q6K:
//               redesign around a cooperative shared tile" (section "Confirmed
//               mechanism"): the weight tile is loaded and dequantised once and
//               every MMA of the tile consumes the same copy -- here all 256
//               rows of x of the pair. As on "Add BF16xFP4 MoE GEMM stage1
//               kernel" (section "Technical Details"), weights are decoded in
//               software before the MMA, which takes fp16/bf16 operands. The
//               even CTA's operand barrier completes when its own dequant
//               warps and one relay arrival for the odd CTA are in: both x
//               blocks have landed and both operand tiles are written.
//   warps 1-2   (odd CTA) relays: forward the odd CTA's tile completions to the
//               even CTA with one cluster-scope release per K step, in turns.
//   warp 1      (even CTA) one thread issues the MMAs into one of two
//               256-column accumulators, which alternate so the epilogue of
//               one tile overlaps the MMAs of the next; its commits free the
//               ring stages and publish accumulators in BOTH CTAs (multicast).
//   warps 4-7   epilogue: tcgen05.ld of the CTA's 128 accumulator rows, round
//               to the output dtype, predicated 16-byte stores (every store is
//               guarded on both M and N, the lesson of the col_n_valid guard on
//               the MoE page, section "Technical Details"); then arrive on the
//               even CTA's accumulator-free barrier.
//   warp 2      allocates (with its peer) and frees the tensor memory.
//
// Every mbarrier wait is bounded (about two seconds); on expiry the kernel
// records W4A16_ERR_TIMEOUT in a device word and raises the abort flag of both
// CTAs, every role stops, the producer and the MMA thread wait (bounded) for
// their own operations in flight, the pair synchronises, tensor memory is
// freed and the kernel returns.
#include "internal.h"
#include "mxfp4.cuh"
#include "ptx.cuh"

#include "tmap.h"

#include <algorithm>
#include <mutex>

namespace w4a16 {

__device__ unsigned int g_device_error = 0;

namespace {

constexpr int BM = 256, BN = 256, BK = 64;   // tile of a CTA pair
constexpr int CM = BM / 2, CN = BN / 2;      // x rows and weight columns held by each CTA
#ifndef W4A16_GEMM_LOAD_STAGES
#define W4A16_GEMM_LOAD_STAGES 7
#endif
#ifndef W4A16_GEMM_B_STAGES
#define W4A16_GEMM_B_STAGES 4
#endif
constexpr int kLoadStages = W4A16_GEMM_LOAD_STAGES;   // x tile + packed weights + scales + zero-points
constexpr int kBStages = W4A16_GEMM_B_STAGES;         // dequantised operand tiles
constexpr int kThreads = 768;
constexpr int kEpiWarp0 = 4;             // warps 4..7
constexpr int kDeqWarp0 = 8;             // warps 8..23: two groups taking alternate K steps
constexpr int kDeqWarps = 8;             // per group: two threads per column of the CTA's tile
constexpr int kDeqGroups = 2;
constexpr int kRelayWarps = 2;           // odd CTA: warps 1..kRelayWarps forward operand-tile completions
constexpr uint32_t kABytes = CM * BK * 2;            // 16 KB
constexpr uint32_t kWBytes = (BK / 8) * CN * 4;      //  4 KB
constexpr uint32_t kSBytes = 2 * CN * 2;             // 512 B: scales of the two 32-row halves of a step
constexpr uint32_t kZBytes = 2 * (CN / 8) * 4;       // 128 B: zero-point words of the two halves
constexpr uint32_t kLoadStageBytes = (kABytes + kWBytes + kSBytes + kZBytes + 1023) & ~1023u;
constexpr uint32_t kBBytes = CN * BK * 2;            // 16 KB
constexpr uint32_t kAccCols = BN;                    // one accumulator: 128 lanes x 256 FP32 columns
constexpr uint32_t kTmemCols = 2 * kAccCols;         // two accumulators
constexpr uint32_t kSuspendNs = 20000;
constexpr unsigned long long kWaitLimitCycles = 4000000000ull;   // ~2 s at 2 GHz
constexpr unsigned int kErrTimeout = 9u;
static_assert(kTmemCols == 512, "tensor memory budget");
// Parity waits are only sound if a waiter never reaches a barrier while a
// phase it skipped is still open (it would take that phase's parity for its
// own). Relays and dequant groups each own whole operand stages, so they
// consume those barriers' phases in order. A dequant group skips the other
// groups' load stages; when it waits for step j it has finished step j - G,
// whose operand stage was freed by MMA j - G - B, and the in-order MMAs have
// then consumed every load stage up to that step, which covers the skipped
// step j - L whenever L >= G + B.
static_assert(kBStages % kRelayWarps == 0, "each relay owns whole operand stages");
static_assert(kBStages % kDeqGroups == 0, "each dequant group owns whole operand stages");
static_assert(kLoadStages % kDeqGroups == 0 || kLoadStages >= kDeqGroups + kBStages,
              "a dequant group may skip a load-stage phase only if it is already complete");

struct __align__(8) Barriers {
    uint64_t lfull[kLoadStages];    // x + weights (TMA bytes) and scales/zero-points (cp.async) landed
    uint64_t lempty[kLoadStages];   // MMAs reading the x tile retired (tcgen05.commit)
    uint64_t bfull[kBStages];       // even CTA: both operand tiles written (its dequant warps + one relay arrival)
    uint64_t bempty[kBStages];      // MMAs reading the operand tile retired (tcgen05.commit)
    uint64_t bready[kBStages];      // odd CTA: its operand tile written (one arrival per dequant warp)
    uint64_t tfull[2];              // accumulator complete
    uint64_t tempty[2];             // even CTA: accumulator drained (one arrival per epilogue warp of the pair)
    uint64_t drain;                 // final commit of the MMA thread
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes =
    1024 /*align slack*/ + kLoadStages * kLoadStageBytes + kBStages * kBBytes + sizeof(Barriers);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// Abort flag of this CTA; on a timeout the flag of the peer CTA is raised too.
struct Abort {
    volatile int* flag;
    uint32_t addr;    // local shared address of the flag (same offset in the peer)
    uint32_t peer;    // cluster rank of the other CTA of the pair
};

// Bounded wait: false if the wait ran out (or another role of either CTA
// already gave up). The thread sleeps inside try_wait while the phase is
// incomplete. kCluster acquires at cluster scope: needed only where the phase
// publishes data written by the other CTA (the even CTA's operand barrier);
// every other wait either guards data of its own CTA or only orders a reuse
// after the reads that freed it, for which CTA scope suffices and costs far less.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Abort& ab) {
    const unsigned long long t0 = clock64();
    for (;;) {
        if (kCluster ? mbar_try_wait_cluster(bar, parity, kSuspendNs) : mbar_try_wait_suspend(bar, parity, kSuspendNs))
            return true;
        if (*ab.flag) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *ab.flag = 1;
            st_cluster_u32(ab.addr, ab.peer, 1u);
            atomicOr(&g_device_error, 1u << kErrTimeout);
            return false;
        }
    }
}

// As wait_bar, but polling without suspending: for the single threads whose
// wake-up latency sits on the critical path (relays and the MMA issuer).
template <bool kCluster = false>
__device__ __forceinline__ bool spin_bar(uint32_t bar, uint32_t parity, const Abort& ab) {
    const unsigned long long t0 = clock64();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (kCluster ? mbar_try_wait_cluster(bar, parity, 0) : mbar_try_wait(bar, parity)) return true;
        if (*ab.flag) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *ab.flag = 1;
            st_cluster_u32(ab.addr, ab.peer, 1u);
            atomicOr(&g_device_error, 1u << kErrTimeout);
            return false;
        }
    }
}

// Lane 0 waits (bounded) and acquires the completed phase; the warp-wide
// shuffle that broadcasts the verdict also orders the other lanes' later
// accesses after lane 0's acquire. (Letting all 32 lanes poll one mbarrier
// serialises their polls and costs hundreds of cycles per wait.)
__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity, const Abort& ab, int lane) {
    int ok = 1;
    if (lane == 0) ok = wait_bar(bar, parity, ab) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

template <bool kBf16>
struct Deq;
template <>
struct Deq<false> {
    static constexpr uint32_t kMagic = 0x64006400u;   // fp16 1024.0
    __device__ static uint32_t sub2(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
    __device__ static uint32_t mul2(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
    __device__ static uint32_t pack2(float lo, float hi) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
};
template <>
struct Deq<true> {
    static constexpr uint32_t kMagic = 0x43004300u;   // bf16 128.0
    __device__ static uint32_t sub2(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
    __device__ static uint32_t mul2(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
    __device__ static uint32_t pack2(float lo, float hi) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
};

// kMx: MXFP4 weights (bf16 only): `sc` holds the E8M0 bytes [K/32, N] and
// there are no zero-points; every 32-row half of a K step is one scale block.
template <bool kBf16, bool kSym, bool kMx = false>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
            const uint16_t* __restrict__ sc, const uint32_t* __restrict__ qz, uint16_t* __restrict__ y, int M,
            int N, int K, int g) {
    extern __shared__ uint8_t smem_raw[];
    // both CTAs of the pair compute the same layout: the MMA addresses the
    // peer's operand tiles at this CTA's offsets
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* bsmem = smem + kLoadStages * kLoadStageBytes;
    Barriers* bars = reinterpret_cast<Barriers*>(bsmem + kBStages * kBBytes);
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t bsmem_base = smem_u32(bsmem);
    // load stage s: [x block | packed weights | scales | zero-point words]
    auto ld_a = [&](int s) { return smem_base + s * kLoadStageBytes; };
    auto ld_w = [&](int s) { return smem + s * kLoadStageBytes + kABytes; };
    auto ld_s = [&](int s) { return smem + s * kLoadStageBytes + kABytes + kWBytes; };
    auto ld_z = [&](int s) { return smem + s * kLoadStageBytes + kABytes + kWBytes + kSBytes; };
    auto op_b = [&](int s) { return bsmem_base + s * kBBytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();          // 0: the CTA that issues the MMAs
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int num_m = (M + BM - 1) / BM, num_n = (N + BN - 1) / BN;
    const int tiles = num_m * num_n;
    const int kt_total = (K + BK - 1) / BK;
    const int groups = K / g;
    const Abort ab{&bars->abort, smem_u32(&bars->abort), rank ^ 1u};

    if (threadIdx.x == 0) {
        for (int s = 0; s < kLoadStages; ++s) {
            mbar_init(smem_u32(&bars->lfull[s]), 1);
            mbar_init(smem_u32(&bars->lempty[s]), 1);
        }
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(smem_u32(&bars->bfull[s]), kDeqWarps + 1);
            mbar_init(smem_u32(&bars->bempty[s]), 1);
            mbar_init(smem_u32(&bars->bready[s]), kDeqWarps);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&bars->tfull[a]), 1);
            mbar_init(smem_u32(&bars->tempty[a]), 2 * 4);
        }
        mbar_init(smem_u32(&bars->drain), 1);
        bars->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmap_x);
        tma_prefetch_desc(&tmap_w);
    }
    if (warp == 2) tmem_alloc_pair(smem_u32(&bars->tmem_base), kTmemCols);
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised, tensor memory allocated
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer warp
        // lane l stages, for 32-row half (l >> 4) of the step, the scales of the
        // 8 columns [8(l&15), 8(l&15)+8) of this CTA's 128 and their zero-point
        // word with cp.async (zero-filled outside N and K); lane 0 then issues the
        // TMA copies of the x block and the packed weight tile.
        const int half = lane >> 4, sub = lane & 15;
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_parity[kLoadStages];
        bool issued[kLoadStages];
        for (int s = 0; s < kLoadStages; ++s) issued[s] = false, issued_parity[s] = 0;
        bool ok = true;
        for (int t = pair; t < tiles && ok; t += npairs) {
            const int m_blk = t % num_m, n_blk = t / num_m;
            const int row0 = m_blk * BM + static_cast<int>(rank) * CM;
            const int col0 = n_blk * BN + static_cast<int>(rank) * CN;
            const int n = col0 + 8 * sub;
            for (int kt = 0; kt < kt_total; ++kt) {
                if (!warp_wait_bar(smem_u32(&bars->lempty[stage]), phase ^ 1u, ab, lane)) { ok = false; break; }
                const uint32_t fb = smem_u32(&bars->lfull[stage]);
                const int grp = (kt * BK + half * (BK / 2)) / g;
                const bool valid = n < N && grp < groups;
                const size_t so = valid ? static_cast<size_t>(grp) * N + n : 0;
                if constexpr (kMx) {
                    // 8 exponent bytes of the lane's columns for this 32-row block
                    cp_async_8(smem_u32(ld_s(stage)) + half * CN + 8 * sub,
                               reinterpret_cast<const uint8_t*>(sc) + so, valid ? 8u : 0u);
                } else {
                    cp_async_16(smem_u32(ld_s(stage)) + half * (CN * 2) + 16 * sub, sc + so, valid ? 16u : 0u);
                }
                if constexpr (!kSym) {
                    const size_t zo = valid ? static_cast<size_t>(grp) * (N >> 3) + (n >> 3) : 0;
                    cp_async_4(smem_u32(ld_z(stage)) + half * (CN / 8) * 4 + 4 * sub, qz + zo, valid ? 4u : 0u);
                }
                cp_async_mbar_arrive(fb);
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_expect_tx(fb, kABytes + kWBytes);
                    tma_load_2d(ld_a(stage), &tmap_x, kt * BK, row0, fb);
                    tma_load_2d(smem_u32(ld_w(stage)), &tmap_w, col0, kt * (BK / 8), fb);
                }
                issued[stage] = true;
                issued_parity[stage] = phase;
                if (++stage == kLoadStages) { stage = 0; phase ^= 1u; }
            }
        }
        // copies still in flight must land before this CTA's shared memory is released
        if (lane == 0) {
            for (int s = 0; s < kLoadStages; ++s) {
                if (!issued[s]) continue;
                const uint32_t fb = smem_u32(&bars->lfull[s]);
                const unsigned long long t0 = clock64();
                while (!mbar_try_wait(fb, issued_parity[s]) && clock64() - t0 < kWaitLimitCycles) {
                }
            }
        }
    } else if (rank == 1 && warp >= 1 && warp <= kRelayWarps) {
        // ------------------------------------------------------------ relays (odd CTA)
        // A release at cluster scope holds the issuing thread for about a
        // microsecond, too long for the dequant warps to pay every step. They
        // arrive at CTA scope on bready; relay r forwards steps j = r (mod
        // kRelayWarps), i.e. operand stages r, r + kRelayWarps, ..., to the even
        // CTA's bfull with one cluster-scope release, which also publishes the
        // dequant warps' tile writes it acquired.
        if (lane == 0) {
            const int r = warp - 1;
            bool ok = true;
            long long j = 0;
            for (int t = pair; t < tiles && ok; t += npairs) {
                for (int kt = 0; kt < kt_total; ++kt, ++j) {
                    if (j % kRelayWarps != r) continue;
                    const int bs = static_cast<int>(j % kBStages);
                    const uint32_t ph = static_cast<uint32_t>((j / kBStages) & 1);
                    if (!spin_bar(smem_u32(&bars->bready[bs]), ph, ab)) { ok = false; break; }
                    mbar_arrive_cluster(smem_u32(&bars->bfull[bs]), 0);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (even CTA)
        if (rank == 0 && lane == 0) {
            constexpr uint32_t kIdesc = umma_idesc_f16(BM, BN, kBf16);
            constexpr uint16_t kPair = 0x3;
            int ls = 0, bs = 0;
            uint32_t bph = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int t = pair; t < tiles && ok; t += npairs) {
                if (!wait_bar(smem_u32(&bars->tempty[acc]), acc_phase ^ 1u, ab)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
                for (int kt = 0; kt < kt_total; ++kt) {
                    // completes when both CTAs' x blocks landed and both operand tiles are written
                    // (the dequant warps wait for their CTA's x block before they arrive)
                    if (!spin_bar<true>(smem_u32(&bars->bfull[bs]), bph, ab)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t adesc = sw128_kmajor_desc(ld_a(ls));
                    const uint64_t bdesc = sw128_kmajor_desc(op_b(bs));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        // advance 16 elements (32 bytes) along K inside the swizzle atom
                        umma_f16_pair(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, kIdesc, (kt | kk) != 0);
                    }
                    umma_commit_pair_mc(smem_u32(&bars->lempty[ls]), kPair);
                    umma_commit_pair_mc(smem_u32(&bars->bempty[bs]), kPair);
                    if (++ls == kLoadStages) ls = 0;
                    if (++bs == kBStages) { bs = 0; bph ^= 1u; }
                }
                if (!ok) break;
                umma_commit_pair_mc(smem_u32(&bars->tfull[acc]), kPair);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            // every MMA issued by this thread retires before tensor memory is freed
            umma_commit_pair(smem_u32(&bars->drain));
            const unsigned long long t0 = clock64();
            while (!mbar_try_wait(smem_u32(&bars->drain), 0) && clock64() - t0 < kWaitLimitCycles) {
            }
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                 // tensor-memory lane quarter of this warp
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = pair; t < tiles; t += npairs) {
            const int m_blk = t % num_m, n_blk = t / num_m;
            if (!warp_wait_bar(smem_u32(&bars->tfull[acc]), acc_phase, ab, lane)) break;
            tc_fence_after();
            const int m = m_blk * BM + static_cast<int>(rank) * CM + q * 32 + lane;
            uint16_t* yrow = y + static_cast<size_t>(m) * N;
#pragma unroll 1
            for (int ch = 0; ch < BN / 32; ++ch) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(acc * kAccCols + ch * 32),
                                   r);
                tmem_wait_ld();
                const int n = n_blk * BN + ch * 32;
                if (m < M) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        if (n + 8 * v < N) {
                            uint4 o;
                            o.x = Deq<kBf16>::pack2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                            o.y = Deq<kBf16>::pack2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                            o.z = Deq<kBf16>::pack2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                            o.w = Deq<kBf16>::pack2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                            *reinterpret_cast<uint4*>(yrow + n + 8 * v) = o;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(smem_u32(&bars->tempty[acc]), 0);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    } else if (warp >= kDeqWarp0) {
        // ------------------------------------------------------------ dequantisers
        // A dequant warp's step is a chain of waits, shared-memory loads and
        // stores whose latency, not issue slots, bounds it: two groups of
        // warps take alternate K steps so that two steps are in flight.
        const int tg = threadIdx.x - kDeqWarp0 * 32;    // 0..511
        const int grp = tg >> 8;                         // group: steps j with j % kDeqGroups == grp
        const int td = tg & 255;
        const int d = td & (CN - 1);                     // column of this CTA's tile
        const int half = td >> 7;                        // 32-row half of the step: words 4*half .. 4*half+3
        int ls = 0, bs = 0;
        uint32_t lph = 0, bph = 0;
        bool ok = true;
        int j = 0;
        auto advance = [&]() {
            ++j;
            if (++ls == kLoadStages) { ls = 0; lph ^= 1u; }
            if (++bs == kBStages) { bs = 0; bph ^= 1u; }
        };
        for (int t = pair; t < tiles && ok; t += npairs) {
            for (int kt = 0; kt < kt_total; ++kt) {
                if (j % kDeqGroups != grp) {
                    advance();
                    continue;
                }
                if (!warp_wait_bar(smem_u32(&bars->lfull[ls]), lph, ab, lane) ||
                    !warp_wait_bar(smem_u32(&bars->bempty[bs]), bph ^ 1u, ab, lane)) {
                    ok = false;
                    break;
                }
                const uint32_t* wt = reinterpret_cast<const uint32_t*>(ld_w(ls));
                const uint16_t* st = reinterpret_cast<const uint16_t*>(ld_s(ls));
                const uint32_t* zt = reinterpret_cast<const uint32_t*>(ld_z(ls));
                const uint32_t b_row = op_b(bs) + static_cast<uint32_t>(d) * 128u;
                if constexpr (kMx) {
                    mx::operand_column<CN>(wt, b_row, d, half, reinterpret_cast<const uint8_t*>(st)[half * CN + d]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(rank == 0 ? &bars->bfull[bs] : &bars->bready[bs]));
                    advance();
                    continue;
                }
                const uint32_t s16 = st[half * CN + d];
                const uint32_t z4 = kSym ? 8u : ((zt[half * (CN / 8) + (d >> 3)] >> (4 * (d & 7))) & 0xFu);
                const uint32_t ss = s16 | (s16 << 16);
                const uint32_t zz = Deq<kBf16>::kMagic | z4 | (z4 << 16);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int c = half * 4 + cc;
                    const uint32_t w = wt[c * CN + d];
                    const uint32_t w4 = w >> 4;
                    uint32_t o[4];
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        // byte b of w -> low half, byte b of (w >> 4) -> high half:
                        // halves (magic + q[8c + 2b], magic + q[8c + 2b + 1])
                        const uint32_t h = and_or(prmt(w, w4, static_cast<uint32_t>(b | ((4 + b) << 8))),
                                                  0x000F000Fu, Deq<kBf16>::kMagic);
                        o[b] = Deq<kBf16>::mul2(Deq<kBf16>::sub2(h, zz), ss);
                    }
                    const uint32_t dst = b_row + (static_cast<uint32_t>(c ^ (d & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(o[0]), "r"(o[1]),
                                 "r"(o[2]), "r"(o[3])
                                 : "memory");
                }
                // the MMA (async proxy, issued from the even CTA) reads these writes
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(rank == 0 ? &bars->bfull[bs] : &bars->bready[bs]));
                advance();
            }
        }
    }

    __syncwarp();   // single-lane roles (MMA issuer) rejoin their warp
    tc_fence_before();
    // neither CTA leaves while the pair's MMAs, commits or remote arrivals may
    // still touch its shared or tensor memory
    cluster_sync();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Clusters of two CTAs that can be resident at once (one CTA per SM; a GPC
// with an odd number of free SMs leaves one idle), per device.
template <bool kBf16, bool kSym, bool kMx>
int resident_pairs(const DeviceProps& dp) {
    static std::mutex mu;
    static int cached[64] = {0};
    const int dev = (dp.device >= 0 && dp.device < 64) ? dp.device : 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (dp.sms / 2));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_kernel<kBf16, kSym, kMx>, &cfg) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            n = dp.sms / 2;
        }
        cached[dev] = n;
    }
    return cached[dev];
}

template <bool kBf16, bool kSym, bool kMx = false>
cudaError_t launch_typed(const void* x, const uint32_t* qw, const void* sc, const uint32_t* qz, void* y, int M,
                         int N, int K, int g, const DeviceProps& dp, cudaStream_t s) {
    auto kern = gemm_kernel<kBf16, kSym, kMx>;
    if (cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), dp.device, kSmemBytes);
        e != cudaSuccess)
        return e;
    CUtensorMap tx, tw;
    const CUtensorMapDataType adt = kBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (!encode_2d(&tx, adt, x, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, BK, CM,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_INT32, qw, (uint64_t)N, (uint64_t)(K / 8),
                   (uint64_t)N * 4, CN, BK / 8, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int pairs = std::max(1, std::min(tiles, resident_pairs<kBf16, kSym, kMx>(dp)));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tx, tw, static_cast<const uint16_t*>(sc), qz, static_cast<uint16_t*>(y), M,
                              N, K, g);
}

}  // namespace

cudaError_t launch_gemm(const void* x, const uint32_t* qw, const void* sc, const uint32_t* qz, void* y, int M, int N,
                        int K, int g, bool bf16, const DeviceProps& dp, cudaStream_t s) {
    if (bf16)
        return qz ? launch_typed<true, false>(x, qw, sc, qz, y, M, N, K, g, dp, s)
                  : launch_typed<true, true>(x, qw, sc, qz, y, M, N, K, g, dp, s);
    return qz ? launch_typed<false, false>(x, qw, sc, qz, y, M, N, K, g, dp, s)
              : launch_typed<false, true>(x, qw, sc, qz, y, M, N, K, g, dp, s);
}

cudaError_t launch_mx_gemm(const void* x, const uint32_t* qw, const uint8_t* es, void* y, int M, int N, int K,
                           const DeviceProps& dp, cudaStream_t s) {
    return launch_typed<true, true, true>(x, qw, es, nullptr, y, M, N, K, mx::kBlock, dp, s);
}

cudaError_t read_and_clear_device_error(uint32_t* out, cudaStream_t s) {
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    uint32_t v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    }
    *out = v;
    return e;
}

}  // namespace w4a16
