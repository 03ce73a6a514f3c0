// GEMM of the W4A16 layer for a few rows of x (M <= 128) on the
// 5th-generation tensor cores, with the operands swapped.
//
// For small M the weights dominate everything: the layer must stream and
// dequantise K*N weights whatever M is, while the MMA work shrinks with M.
// Here the unit of work is a 128-column block of weights with all M rows:
// the dequantised weight tile [128 x 128] is the MMA's A operand (M_mma =
// 128), the x tile [MP x 128] its B operand (N_mma = MP, M rounded up to a
// multiple of 32), and each CTA's tensor memory holds D[n][m] = y[m][n] for
// its columns. The weight tile is loaded and dequantised once per CTA and
// every row of x reuses it (the cooperative shared tile of "ROCm
// KQuantGemmKWmmaQ4K/Q6K: redesign around a cooperative shared tile",
// section "Confirmed mechanism"), but the shared tile lives in tensor memory:
// the dequantising threads write it there with tcgen05.st (thread = weight
// column = tensor-memory lane) and the MMA reads A from tensor memory. No
// shared-memory operand ring, no swizzled stores; tensor memory holds two
// accumulators and four to six operand stages, shared memory only the load
// ring. A tcgen05.mma with M = 128, K = 16 takes about 93 cycles for any N up
// to 128 (measured on GB300), so the MMA count per weight, not the rows of x,
// sets this kernel's floor: about 33 us at 43008 x 5376.
//
// Work is split stream-K: the (column block, K step) pairs, column block
// first, are cut into equal contiguous ranges, one per CTA (one CTA per SM),
// so every SM dequantises the same number of steps whatever the number of
// column blocks (336 blocks over 152 SMs would otherwise leave a third of the
// SMs idle in the last round). A column block whose steps are split between
// CTAs is finished per epilogue warp (32 columns) by the last contributor to
// arrive: each writes its FP32 partial (column-major, rows contiguous) to a
// workspace slot, takes the (block, warp) ticket, and the last one sums the
// partials in ascending CTA order (deterministic), stores y and resets the
// ticket.
//
// Warp roles, one CTA per SM, each walking the CTA's (column block, K range)
// segments in order:
//   warp 0      producer: per 128-deep K step, TMA brings the x tile [MP x 128] in 64-column
//               boxes (128-byte swizzle, rows >= M zero-filled) and the packed
//               weight tile [step/8 words x 128]; the lanes stage the step's
//               scales and zero-point words with cp.async. One mbarrier per stage.
//   warps 8-23  two groups of eight on alternate K steps dequantise the packed
//               tile into an operand stage of tensor memory: warp w writes
//               lanes 32 (w % 4) .. + 31 (its quarter), the two warps of a
//               quarter the two 64-deep halves of the step; w = (q - z) * s,
//               (q - z) exact in 16-bit arithmetic, one rounding.
//   warp 1      one thread issues 8 x tcgen05.mma (kind::f16, M=128, N=MP,
//               K=16, A from tensor memory) per step into one of two
//               MP-column FP32 accumulators.
//   warps 4-7   epilogue: tcgen05.ld of the accumulator (lane = column n,
//               column = row m of x), round, store y[m][n] (consecutive lanes
//               write consecutive columns), predicated on m < M and n < N.
//   warp 2      allocates and frees the tensor memory.
//
// Every mbarrier wait is bounded (about two seconds); on expiry the kernel
// records W4A16_ERR_TIMEOUT in its device word (read by w4a16_device_status),
// every role stops, the producer and the MMA thread wait (bounded) for their
// own operations in flight, tensor memory is freed and the kernel returns.
#include "internal.h"
#include "mxfp4.cuh"
#include "ptx.cuh"
#include "tmap.h"

#include <algorithm>
#include <cstring>

namespace w4a16 {

__device__ unsigned int g_skinny_error = 0;

namespace {

constexpr int BN = 128;                  // weight columns per tile (M of the MMA)
constexpr int kThreads = 768;
constexpr int kEpiWarp0 = 4;             // warps 4..7
constexpr int kDeqWarp0 = 8;             // warps 8..23: groups taking K steps in turn
#ifndef W4A16_SKINNY_DEQ_GROUPS
#define W4A16_SKINNY_DEQ_GROUPS 2
#endif
constexpr int kDeqGroups = W4A16_SKINNY_DEQ_GROUPS;   // 2 or 4
constexpr int kDeqWarps = 16 / kDeqGroups;            // warps per group: every quarter of the lanes, once or twice
constexpr int kDeqSplit = kDeqWarps / 4;              // threads per weight column in a group
constexpr uint32_t kTmemCols = 512;      // the whole tensor memory of the SM (one CTA per SM)
constexpr uint32_t kSuspendNs = 20000;
constexpr unsigned long long kWaitLimitCycles = 4000000000ull;   // ~2 s at 2 GHz
constexpr unsigned int kErrTimeout = 9u;
constexpr size_t kSmemBudget = 220 * 1024;

template <int MP>
struct Cfg {
    static_assert(MP % 32 == 0 && MP >= 32 && MP <= 128, "rows of x per tile");
    // K per step: 256 up to 64 padded rows of x (half the per-step pipeline
    // hand-offs: 68-75 us against 71-81 us with 128 at N = 43008, K = 5376);
    // 128 above, where a 256-deep step leaves room for only two load stages
    static constexpr int BK = MP <= 64 ? 256 : 128;
    static constexpr int kSub = BK / 64;            // 64-column boxes of x per step (one 128-byte swizzle row each)
    static constexpr int kQuarters = BK / 32;       // 32-row scale blocks per step
    static constexpr uint32_t kWBytes = (BK / 8) * BN * 4;          // packed weights
    static constexpr uint32_t kSBytes = kQuarters * BN * 2;         // scales of the step's 32-row blocks
    static constexpr uint32_t kZBytes = kQuarters * (BN / 8) * 4;   // zero-point words of the blocks
    static constexpr uint32_t kABytes = MP * BK * 2;                // x tile
    static constexpr uint32_t kLoadStageBytes = (kABytes + kWBytes + kSBytes + kZBytes + 1023) & ~1023u;
    // as many load stages as fit (at most 10), a multiple of the dequant groups
    // (each group then owns whole ring stages: no waiter skips a phase)
    static constexpr int kRaw = static_cast<int>((kSmemBudget - 2048) / kLoadStageBytes);
    static constexpr int kLoadStages = (kRaw > 10 ? 10 : kRaw) & ~(kDeqGroups - 1);
    // tensor memory: two accumulators of MP columns, then operand stages of
    // BK / 2 columns (two 16-bit values per 32-bit column), a multiple of the groups
    static constexpr uint32_t kAccCols = MP;
    static constexpr uint32_t kOpCol0 = 2 * MP;
    static constexpr uint32_t kOpCols = BK / 2;
    static constexpr int kOpStages = static_cast<int>((kTmemCols - kOpCol0) / kOpCols) & ~(kDeqGroups - 1);
    static_assert(kLoadStages >= 2 && kOpStages >= 2, "rings");
    static_assert(kLoadStages % 2 == 0, "two producer warps own alternate load stages");
    static_assert(kLoadStages % kDeqGroups == 0 && kOpStages % kDeqGroups == 0,
                  "each dequant group owns whole ring stages");
};

template <int MP>
struct __align__(8) Barriers {
    uint64_t lfull[Cfg<MP>::kLoadStages];
    uint64_t lempty[Cfg<MP>::kLoadStages];
    uint64_t afull[Cfg<MP>::kOpStages];    // operand stage written (tensor memory)
    uint64_t aempty[Cfg<MP>::kOpStages];   // operand stage read by the MMAs
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

template <int MP>
constexpr size_t smem_bytes() {
    return 1024 + Cfg<MP>::kLoadStages * Cfg<MP>::kLoadStageBytes + sizeof(Barriers<MP>);
}

// Launch with programmatic stream serialization (0: plain launches).
#ifndef W4A16_SKINNY_PDL
#define W4A16_SKINNY_PDL 1
#endif
constexpr bool kSkinnyPdl = W4A16_SKINNY_PDL != 0;

#ifndef W4A16_SKINNY_SPIN
#define W4A16_SKINNY_SPIN 64
#endif
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort) {
    // a completed or nearly completed phase is seen without the suspend path's cost
    for (int i = 0; i < W4A16_SKINNY_SPIN; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait_suspend(bar, parity, kSuspendNs)) return true;
        if (*abort) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort = 1;
            atomicOr(&g_skinny_error, 1u << kErrTimeout);
            return false;
        }
    }
}

// Lane 0 waits and acquires; the shuffle broadcasts the verdict and orders the
// other lanes' later accesses after lane 0's acquire.
__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity, volatile int* abort, int lane) {
    int ok = 1;
    if (lane == 0) ok = wait_bar(bar, parity, abort) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// The CTA's range of (column block, K step) units, column block first, walked
// as segments: column block t, K steps [k0, k1).
// Without stream-K the CTA takes whole column blocks blockIdx.x, + gridDim.x, ...
struct Segments {
    long long u, u_end;
    int kt_total;
    bool streamk;
    int tiles;
    __device__ bool next(int& t, int& k0, int& k1) {
        if (!streamk) {
            if (u >= tiles) return false;
            t = static_cast<int>(u);
            k0 = 0;
            k1 = kt_total;
            u += gridDim.x;
            return true;
        }
        if (u >= u_end) return false;
        t = static_cast<int>(u / kt_total);
        k0 = static_cast<int>(u - static_cast<long long>(t) * kt_total);
        k1 = static_cast<int>(u_end - u < kt_total - k0 ? k0 + (u_end - u) : kt_total);
        u += k1 - k0;
        return true;
    }
};
__device__ __forceinline__ long long unit_start(int b, long long U, int G) { return static_cast<long long>(b) * U / G; }
// the CTA whose range holds unit u
__device__ __forceinline__ int unit_owner(long long u, long long U, int G) { return static_cast<int>(((u + 1) * G - 1) / U); }
#ifndef W4A16_SKINNY_STREAMK_MAX_M
#define W4A16_SKINNY_STREAMK_MAX_M 128
#endif
constexpr int kStreamKMaxM = W4A16_SKINNY_STREAMK_MAX_M;   // larger M: whole column blocks per CTA
constexpr int kSlotFloats = BN * 128;   // one partial [BN columns][up to 128 rows], rows contiguous

template <bool kBf16>
struct Dq;
template <>
struct Dq<false> {
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
    __device__ static uint16_t out(float v) { return __half_as_ushort(__float2half_rn(v)); }
};
template <>
struct Dq<true> {
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
    __device__ static uint16_t out(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
};

// kMx: MXFP4 weights (bf16 only): `sc` holds the E8M0 bytes [K/32, N] and
// there are no zero-points; every 32-row half of a K step is one scale block.
template <bool kBf16, bool kSym, int MP, bool kMx = false>
__global__ void __launch_bounds__(kThreads, 1)
gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_s, const __grid_constant__ CUtensorMap tmap_z,
                   const uint32_t* __restrict__ qz, uint16_t* __restrict__ y, int M, int N, int K, int g,
                   float* __restrict__ partials, uint32_t* __restrict__ tickets, int streamk, int z_tma) {
    using C = Cfg<MP>;
    constexpr int L = C::kLoadStages;
    constexpr int BK = C::BK, kSub = C::kSub, kOpStages = C::kOpStages;
    constexpr uint32_t kWBytes = C::kWBytes, kSBytes = C::kSBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Barriers<MP>* bars = reinterpret_cast<Barriers<MP>*>(smem + L * C::kLoadStageBytes);
    const uint32_t smem_base = smem_u32(smem);
    // load stage s: [x tile | packed weights | scales | zero-point words]
    auto ld_a = [&](int s) { return smem_base + s * C::kLoadStageBytes; };
    auto ld_w = [&](int s) { return smem + s * C::kLoadStageBytes + C::kABytes; };
    auto ld_s = [&](int s) { return smem + s * C::kLoadStageBytes + C::kABytes + kWBytes; };
    auto ld_z = [&](int s) { return smem + s * C::kLoadStageBytes + C::kABytes + kWBytes + kSBytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = (N + BN - 1) / BN;
    const int kt_total = (K + BK - 1) / BK;
    const int groups = K / g;
    const int srows = g <= BK ? BK / g : 1;   // scale / zero-point rows per K step
    volatile int* abort_flag = &bars->abort;
    const long long U = static_cast<long long>(tiles) * kt_total;
    const int G = gridDim.x;
    const long long u_begin = streamk ? unit_start(blockIdx.x, U, G) : blockIdx.x;
    const long long u_end = streamk ? unit_start(blockIdx.x + 1, U, G) : tiles;

    // Programmatic launch: the next kernel of the stream may start its
    // prologue once every CTA of this grid is past this point. Before the
    // dependency wait below this grid touches no global memory: it only
    // initialises barriers, prefetches the tensor maps and allocates tensor
    // memory (one CTA per SM by shared memory, so it never waits there for a
    // CTA of the preceding grid).
    if (kSkinnyPdl) griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < L; ++s) {
            mbar_init(smem_u32(&bars->lfull[s]), 1);
            mbar_init(smem_u32(&bars->lempty[s]), 1);
        }
        for (int s = 0; s < kOpStages; ++s) {
            mbar_init(smem_u32(&bars->afull[s]), kDeqWarps);
            mbar_init(smem_u32(&bars->aempty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&bars->tfull[a]), 1);
            mbar_init(smem_u32(&bars->tempty[a]), 4);
        }
        mbar_init(smem_u32(&bars->drain), 1);
        bars->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmap_x);
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_s);
        if (z_tma) tma_prefetch_desc(&tmap_z);
    }
    if (warp == 2) tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    // every read of x, weights and workspace and every write comes after the
    // preceding kernel has completed and its writes are visible
    if (kSkinnyPdl) griddep_wait();

    if (warp == 0 || warp == 3) {
        // ------------------------------------------------------------ producer warps
        // warp 0 loads the even steps, warp 3 the odd ones (one thread issuing
        // every copy of every step could not keep up with the MMAs)
        const int pw = warp == 0 ? 0 : 1;
        const int half = lane >> 4, sub = lane & 15;
        (void)half;
        int stage = 0;
        uint32_t phase = 0;
        int pj = 0;
        uint32_t issued_parity[L];
        bool issued[L];
        for (int s = 0; s < L; ++s) issued[s] = false, issued_parity[s] = 0;
        bool ok = true;
        Segments seg{u_begin, u_end, kt_total, streamk != 0, tiles};
        int t, k0, k1;
        while (ok && seg.next(t, k0, k1)) {
            const int n0 = t * BN;
            const int n = n0 + 8 * sub;
            for (int kt = k0; kt < k1; ++kt) {
                if ((pj++ & 1) != pw) {   // the other producer's step
                    if (++stage == L) { stage = 0; phase ^= 1u; }
                    continue;
                }
                if (!warp_wait_bar(smem_u32(&bars->lempty[stage]), phase ^ 1u, abort_flag, lane)) { ok = false; break; }
                const uint32_t fb = smem_u32(&bars->lfull[stage]);
                const int row0 = (kt * BK) / g;             // first scale / zero-point row of the step
                if constexpr (!kSym) {
                    if (!z_tma) {
                        // zero-point rows of N / 8 words that are not a multiple of 16 bytes:
                        // 4-byte copies by the lanes (rows >= K / g and columns >= N read as 0)
                        for (int r = half; r < srows; r += 2) {
                            const int grp = row0 + r;
                            const bool valid = n < N && grp < groups;
                            const size_t zo = valid ? static_cast<size_t>(grp) * (N >> 3) + (n >> 3) : 0;
                            cp_async_4(smem_u32(ld_z(stage)) + r * (BN / 8) * 4 + 4 * sub, qz + zo, valid ? 4u : 0u);
                        }
                        cp_async_mbar_arrive(fb);
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    const uint32_t ztx = (!kSym && z_tma) ? srows * (BN / 8) * 4 : 0u;
                    mbar_arrive_expect_tx(fb, C::kABytes + kWBytes + srows * BN * (kMx ? 1 : 2) + ztx);
#pragma unroll
                    for (int p = 0; p < kSub; ++p)   // x in 64-column boxes (the 128-byte swizzle's width)
                        tma_load_2d(ld_a(stage) + p * (MP * 128), &tmap_x, kt * BK + 64 * p, 0, fb);
                    tma_load_2d(smem_u32(ld_w(stage)), &tmap_w, n0, kt * (BK / 8), fb);
                    // the step's scale rows (box of srows rows; rows past K / g and columns past N read as 0)
                    tma_load_2d(smem_u32(ld_s(stage)), &tmap_s, n0, row0, fb);
                    if (ztx) tma_load_2d(smem_u32(ld_z(stage)), &tmap_z, n0 / 8, row0, fb);
                }
                issued[stage] = true;
                issued_parity[stage] = phase;
                if (++stage == L) { stage = 0; phase ^= 1u; }
            }
        }
        // copies still in flight must land before this CTA's shared memory is released
        if (lane == 0) {
            for (int s = 0; s < L; ++s) {
                if (!issued[s]) continue;
                const uint32_t fb = smem_u32(&bars->lfull[s]);
                const unsigned long long t0 = clock64();
                while (!mbar_try_wait(fb, issued_parity[s]) && clock64() - t0 < kWaitLimitCycles) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdesc = umma_idesc_f16(BN, MP, kBf16);
            int ls = 0, as = 0;
            uint32_t aph = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            Segments seg{u_begin, u_end, kt_total, streamk != 0, tiles};
            int t, k0, k1;
            while (ok && seg.next(t, k0, k1)) {
                if (!wait_bar(smem_u32(&bars->tempty[acc]), acc_phase ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::kAccCols);
                for (int kt = k0; kt < k1; ++kt) {
                    // completes when the dequant group has written the operand stage,
                    // which it starts only after the step's x tile has landed
                    if (!wait_bar(smem_u32(&bars->afull[as]), aph, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_tmem = tmem_base + C::kOpCol0 + static_cast<uint32_t>(as) * C::kOpCols;
#pragma unroll
                    for (int p = 0; p < kSub; ++p) {
                        const uint64_t xdesc = sw128_kmajor_desc(ld_a(ls) + p * (MP * 128));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)   // 16 values of K = 8 columns of the operand
                            umma_f16_ta(d_tmem, a_tmem + 8u * (4 * p + kk), xdesc + 2u * kk, kIdesc,
                                        (kt - k0) + p + kk != 0);
                    }
                    umma_commit(smem_u32(&bars->lempty[ls]));
                    umma_commit(smem_u32(&bars->aempty[as]));
                    if (++ls == L) ls = 0;
                    if (++as == kOpStages) { as = 0; aph ^= 1u; }
                }
                if (!ok) break;
                umma_commit(smem_u32(&bars->tfull[acc]));
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            // every MMA issued by this thread retires before tensor memory is freed
            umma_commit(smem_u32(&bars->drain));
            const unsigned long long t0 = clock64();
            while (!mbar_try_wait(smem_u32(&bars->drain), 0) && clock64() - t0 < kWaitLimitCycles) {
            }
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                 // tensor-memory lane quarter: columns 32q .. 32q+31
        const int et = threadIdx.x - kEpiWarp0 * 32;   // 0..127: column of the block
        int acc = 0;
        uint32_t acc_phase = 0;
        Segments seg{u_begin, u_end, kt_total, streamk != 0, tiles};
        int t, k0, k1;
        while (seg.next(t, k0, k1)) {
            if (!warp_wait_bar(smem_u32(&bars->tfull[acc]), acc_phase, abort_flag, lane)) break;
            tc_fence_after();
            const int n = t * BN + q * 32 + lane;
            const bool whole = k0 == 0 && k1 == kt_total;
            // a split block: slot 1 for the segment that starts the block, 0 for the others
            float* part = partials + (static_cast<size_t>(blockIdx.x) * 2 + (k0 > 0 ? 0 : 1)) * kSlotFloats;
#pragma unroll 1
            for (int ch = 0; ch < MP / 32; ++ch) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(acc * C::kAccCols + ch * 32),
                                   r);
                tmem_wait_ld();
                if (whole) {
                    if (n < N) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int m = ch * 32 + i;
                            if (m < M) y[static_cast<size_t>(m) * N + n] = Dq<kBf16>::out(__uint_as_float(r[i]));
                        }
                    }
                } else if (ch * 32 < M) {
                    // this column's rows ch*32 .. ch*32+31, contiguous (rows >= M are never read)
                    float4* dst = reinterpret_cast<float4*>(part + et * 128 + ch * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                             __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->tempty[acc]));
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            if (whole) continue;
            // split block: each warp settles its 32 columns on its own (a ticket per
            // column block and warp, no barrier across warps): the last contributing
            // CTA to arrive sums every contributor's partial in ascending CTA order
            // and stores y
            const long long first = static_cast<long long>(t) * kt_total;
            const int b_lo = unit_owner(first, U, G), b_hi = unit_owner(first + kt_total - 1, U, G);
            __threadfence();
            __syncwarp();
            uint32_t last = 0;
            if (lane == 0) last = atomicAdd(tickets + 4 * t + q, 1u) == static_cast<unsigned>(b_hi - b_lo);
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence();
                if (n < N) {
                    // rows in batches of 16: four 16-byte loads per contributor in flight
                    for (int m0 = 0; m0 < M; m0 += 16) {
                        float4 acc4[4];
                        const float4* lo =
                            reinterpret_cast<const float4*>(partials + (static_cast<size_t>(b_lo) * 2 + 1) * kSlotFloats +
                                                            et * 128 + m0);
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc4[i] = __ldcg(lo + i);
                        for (int b0 = b_lo + 1; b0 <= b_hi; ++b0) {
                            const float4* src = reinterpret_cast<const float4*>(
                                partials + static_cast<size_t>(b0) * 2 * kSlotFloats + et * 128 + m0);
                            float4 v[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) v[i] = __ldcg(src + i);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                acc4[i].x += v[i].x;
                                acc4[i].y += v[i].y;
                                acc4[i].z += v[i].z;
                                acc4[i].w += v[i].w;
                            }
                        }
                        const float* f = reinterpret_cast<const float*>(acc4);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (m0 + i < M) y[static_cast<size_t>(m0 + i) * N + n] = Dq<kBf16>::out(f[i]);
                    }
                }
                if (lane == 0) tickets[4 * t + q] = 0u;
            }
        }
    } else if (warp >= kDeqWarp0) {
        // ------------------------------------------------------------ dequantisers
        const int tg = threadIdx.x - kDeqWarp0 * 32;    // 0..511
        const int grp = tg / (kDeqWarps * 32);           // group: steps j with j % kDeqGroups == grp
        const int td = tg % (kDeqWarps * 32);
        const int d = td & (BN - 1);                     // column of the tile = tensor-memory lane (warp's quarter)
        const int tq = td >> 7;                          // this thread's part of the step's K
        constexpr int kBlocks = C::kQuarters / kDeqSplit;   // 32-row blocks per thread
        const uint32_t lane_field = static_cast<uint32_t>((warp & 3) * 32) << 16;
        int ls = 0, as = 0;
        uint32_t lph = 0, aph = 0;
        bool ok = true;
        int j = 0;
        auto advance = [&]() {
            ++j;
            if (++ls == L) { ls = 0; lph ^= 1u; }
            if (++as == kOpStages) { as = 0; aph ^= 1u; }
        };
        Segments seg{u_begin, u_end, kt_total, streamk != 0, tiles};
        int t, k0, k1;
        while (ok && seg.next(t, k0, k1)) {
            for (int kt = k0; kt < k1; ++kt) {
                if (j % kDeqGroups != grp) {
                    advance();
                    continue;
                }
                if (!warp_wait_bar(smem_u32(&bars->lfull[ls]), lph, abort_flag, lane) ||
                    !warp_wait_bar(smem_u32(&bars->aempty[as]), aph ^ 1u, abort_flag, lane)) {
                    ok = false;
                    break;
                }
                tc_fence_after();   // the MMAs that read this operand stage have completed
                const uint32_t* wt = reinterpret_cast<const uint32_t*>(ld_w(ls));
                const uint16_t* st = reinterpret_cast<const uint16_t*>(ld_s(ls));
                const uint32_t* zt = reinterpret_cast<const uint32_t*>(ld_z(ls));
                const uint32_t op = tmem_base + lane_field + C::kOpCol0 + static_cast<uint32_t>(as) * C::kOpCols;
                // this column's values of K, two 32-row blocks (32 bf16/fp16 pairs, pair c
                // holding k = 2c, 2c + 1) per tensor-memory store
#pragma unroll
                for (int r2 = 0; r2 < kBlocks; r2 += 2) {
                    uint32_t o[32];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int qt = kBlocks * tq + r2 + r;        // 32-row block: word rows 4*qt .. 4*qt+3
                        const uint32_t* wp = wt + (qt >> 1) * 8 * BN;   // its 64-row half's 8 word rows
                        const int half = qt & 1;
                        const int srow = g <= BK ? (qt * 32) / g : 0;   // the block's scale row in the stage
                        if constexpr (kMx) {
                            uint32_t v[16];
                            mx::operand_column_regs<BN>(wp, d, half, reinterpret_cast<const uint8_t*>(st)[srow * BN + d], v);
#pragma unroll
                            for (int u = 0; u < 16; ++u) o[16 * r + u] = v[u];
                            continue;
                        }
                        const uint32_t s16 = st[srow * BN + d];
                        const uint32_t z4 = kSym ? 8u : ((zt[srow * (BN / 8) + (d >> 3)] >> (4 * (d & 7))) & 0xFu);
                        const uint32_t ss = s16 | (s16 << 16);
                        const uint32_t zz = Dq<kBf16>::kMagic | z4 | (z4 << 16);
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {
                            const uint32_t w = wp[(half * 4 + cc) * BN + d];
                            const uint32_t w4 = w >> 4;
#pragma unroll
                            for (int b = 0; b < 4; ++b) {
                                // byte b of w -> low half, byte b of (w >> 4) -> high half:
                                // halves (magic + q[8c + 2b], magic + q[8c + 2b + 1])
                                const uint32_t h = and_or(prmt(w, w4, static_cast<uint32_t>(b | ((4 + b) << 8))),
                                                          0x000F000Fu, Dq<kBf16>::kMagic);
                                o[16 * r + 4 * cc + b] = Dq<kBf16>::mul2(Dq<kBf16>::sub2(h, zz), ss);
                            }
                        }
                    }
                    tmem_st_32x32b_x32(op + static_cast<uint32_t>(kBlocks * tq + r2) * 16u, o);
                }
                tmem_wait_st();
                // the MMA (another thread) reads these tensor-memory writes
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->afull[as]));
                advance();
            }
        }
    }

    __syncwarp();   // single-lane roles (MMA issuer) rejoin their warp
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <bool kBf16, bool kSym, int MP, bool kMx = false>
cudaError_t launch_mp(const void* x, const uint32_t* qw, const void* sc, const uint32_t* qz, void* y, int M, int N,
                      int K, int g, float* partials, uint32_t* tickets, const DeviceProps& dp, cudaStream_t s) {
    auto kern = gemm_skinny_kernel<kBf16, kSym, MP, kMx>;
    constexpr size_t kSmem = smem_bytes<MP>();
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
    if (cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), dp.device, kSmem); e != cudaSuccess)
        return e;
    CUtensorMap tx, tw;
    const CUtensorMapDataType adt = kBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (!encode_2d(&tx, adt, x, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, 64, MP, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    constexpr int BK = Cfg<MP>::BK;
    if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_INT32, qw, (uint64_t)N, (uint64_t)(K / 8), (uint64_t)N * 4, BN,
                   BK / 8, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    // scales [K/g, N] (MXFP4: exponent bytes [K/32, N]) and packed zero-points [K/g, N/8]: boxes of
    // the rows one K step uses by 128 columns
    CUtensorMap ts, tz;
    const uint32_t srows = g <= BK ? BK / g : 1;
    const CUtensorMapDataType sdt = kMx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : adt;
    if (!encode_2d(&ts, sdt, sc, (uint64_t)N, (uint64_t)(K / g), (uint64_t)N * (kMx ? 1 : 2), BN, srows,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const bool z_tma = !kSym && N % 32 == 0;   // zero-point rows a multiple of 16 bytes
    if (z_tma) {
        if (!encode_2d(&tz, CU_TENSOR_MAP_DATA_TYPE_INT32, qz, (uint64_t)(N / 8), (uint64_t)(K / g),
                       (uint64_t)(N / 8) * 4, BN / 8, srows, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        memset(&tz, 0, sizeof(tz));
    }
    const int tiles = (N + BN - 1) / BN;
    const long long units = static_cast<long long>(tiles) * ((K + BK - 1) / BK);
    const bool streamk = M <= kStreamKMaxM;
    const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(streamk ? units : tiles, dp.sms)));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = kSkinnyPdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, tx, tw, ts, tz, qz, static_cast<uint16_t*>(y), M, N, K, g, partials, tickets,
                              streamk ? 1 : 0, z_tma ? 1 : 0);
}

template <bool kBf16, bool kSym, bool kMx = false>
cudaError_t launch_typed(const void* x, const uint32_t* qw, const void* sc, const uint32_t* qz, void* y, int M, int N,
                         int K, int g, float* pt, uint32_t* tk, const DeviceProps& dp, cudaStream_t s) {
    if (M <= 32) return launch_mp<kBf16, kSym, 32, kMx>(x, qw, sc, qz, y, M, N, K, g, pt, tk, dp, s);
    if (M <= 64) return launch_mp<kBf16, kSym, 64, kMx>(x, qw, sc, qz, y, M, N, K, g, pt, tk, dp, s);
    return launch_mp<kBf16, kSym, 128, kMx>(x, qw, sc, qz, y, M, N, K, g, pt, tk, dp, s);
}

}  // namespace

size_t skinny_partial_bytes(const DeviceProps& dp) {
    return static_cast<size_t>(dp.sms) * 2 * kSlotFloats * sizeof(float);
}

size_t skinny_ticket_bytes(int N) {
    // one ticket per column block and epilogue warp
    return (static_cast<size_t>((N + BN - 1) / BN) * 4 * sizeof(uint32_t) + 255) & ~size_t(255);
}

size_t skinny_workspace_bytes(int N, const DeviceProps& dp) { return skinny_partial_bytes(dp) + skinny_ticket_bytes(N); }

cudaError_t launch_gemm_skinny(const void* x, const uint32_t* qw, const void* sc, const uint32_t* qz, void* y, int M,
                               int N, int K, int g, bool bf16, float* pt, uint32_t* tk, const DeviceProps& dp,
                               cudaStream_t s) {
    if (M < 1 || M > kSkinnyMaxM || M > 128 || !pt || !tk) return cudaErrorInvalidValue;
    if (bf16)
        return qz ? launch_typed<true, false>(x, qw, sc, qz, y, M, N, K, g, pt, tk, dp, s)
                  : launch_typed<true, true>(x, qw, sc, qz, y, M, N, K, g, pt, tk, dp, s);
    return qz ? launch_typed<false, false>(x, qw, sc, qz, y, M, N, K, g, pt, tk, dp, s)
              : launch_typed<false, true>(x, qw, sc, qz, y, M, N, K, g, pt, tk, dp, s);
}

cudaError_t launch_mx_gemm_skinny(const void* x, const uint32_t* qw, const uint8_t* es, void* y, int M, int N, int K,
                                  float* pt, uint32_t* tk, const DeviceProps& dp, cudaStream_t s) {
    if (M < 1 || M > kSkinnyMaxM || M > 128 || !pt || !tk) return cudaErrorInvalidValue;
    return launch_typed<true, true, true>(x, qw, es, nullptr, y, M, N, K, mx::kBlock, pt, tk, dp, s);
}

}  // namespace w4a16

namespace w4a16 {
cudaError_t read_and_clear_skinny_error(uint32_t* out) {
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_skinny_error, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_skinny_error, &zero, sizeof(zero));
    }
    *out = v;
    return e;
}
}  // namespace w4a16
