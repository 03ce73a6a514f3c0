// Prefill GEMM of the W4A16 layer on the 5th-generation tensor cores.
//
// Design (one CTA per SM, persistent over 256 x 128 output tiles):
//
//   warp 0      producer: per 64-deep K step, TMA brings the x tile [256 x 64]
//               (128-byte swizzle) and the packed weight tile [8 words x 128];
//               the warp's lanes stage the step's scales and zero-point words
//               with cp.async (zero-filled outside N and K). All of it lands
//               in one stage of a 5-deep ring and completes one mbarrier; the
//               ring depth (bytes in flight per SM) is what bounds this kernel.
//   warps 8-15  dequantise the packed tile ONCE into a [128 x 64] fp16/bf16
//               operand tile in the canonical K-major 128-byte-swizzled layout
//               the MMA reads: w = (q - z) * s, with (q - z) exact in 16-bit
//               arithmetic and one rounding for the product. This is the
//               cooperative shared tile of "ROCm KQuantGemmKWmmaQ4K/Q6K:
//               redesign around a cooperative shared tile" (section "Confirmed
//               mechanism"): the weight tile is loaded and dequantised once per
//               CTA and every MMA of the tile consumes the same copy -- here
//               both 128-row halves of the x tile, so each dequantised weight
//               feeds 256 rows of x. As on "Add BF16xFP4 MoE GEMM stage1
//               kernel" (section "Technical Details"), weights are decoded in
//               software before the MMA, which takes fp16/bf16 operands.
//   warp 1      one thread issues tcgen05.mma (kind::f16, M=128, N=128, K=16,
//               twice per K slice: one per M half) into FP32 accumulators in
//               tensor memory; two 256-column accumulators alternate so the
//               epilogue of one tile overlaps the MMAs of the next.
//   warps 4-7   epilogue: tcgen05.ld from tensor memory, round to the output
//               dtype, predicated 16-byte stores (every store is guarded on
//               both M and N, the lesson of the col_n_valid guard on the MoE
//               page, section "Technical Details").
//
// Every mbarrier wait is bounded (about two seconds); on expiry the kernel
// records W4A16_ERR_TIMEOUT in a device word, every role stops, the producer
// and the MMA thread wait (bounded) for their own operations in flight, tensor
// memory is freed and the kernel returns.
#include "internal.h"
#include "ptx.cuh"

#include "tmap.h"

#include <algorithm>
#include <mutex>

namespace w4a16 {

__device__ unsigned int g_device_error = 0;

namespace {

constexpr int BM = 256, BN = 128, BK = 64;
constexpr int UM = 128;                  // rows per tcgen05.mma: a tile is two M halves
#ifndef W4A16_GEMM_LOAD_STAGES
#define W4A16_GEMM_LOAD_STAGES 5
#endif
#ifndef W4A16_GEMM_B_STAGES
#define W4A16_GEMM_B_STAGES 2
#endif
constexpr int kLoadStages = W4A16_GEMM_LOAD_STAGES;   // x tile + packed weights + scales + zero-points
constexpr int kBStages = W4A16_GEMM_B_STAGES;         // dequantised operand tiles
constexpr int kThreads = 512;
constexpr int kEpiWarp0 = 4;             // warps 4..7
constexpr int kDeqWarp0 = 8;             // warps 8..15: two threads per column of the tile
constexpr int kDeqWarps = 8;
constexpr uint32_t kABytes = BM * BK * 2;            // 32 KB
constexpr uint32_t kWBytes = (BK / 8) * BN * 4;      //  4 KB
constexpr uint32_t kSBytes = 2 * BN * 2;             // 512 B: scales of the two 32-row halves of a step
constexpr uint32_t kZBytes = 2 * (BN / 8) * 4;       // 128 B: zero-point words of the two halves
constexpr uint32_t kLoadStageBytes = (kABytes + kWBytes + kSBytes + kZBytes + 1023) & ~1023u;
constexpr uint32_t kBBytes = BN * BK * 2;            // 16 KB
constexpr uint32_t kAccCols = 2 * BN;                // one accumulator: two M halves side by side
constexpr uint32_t kTmemCols = 2 * kAccCols;         // two accumulators
constexpr uint32_t kSuspendNs = 20000;
constexpr unsigned long long kWaitLimitCycles = 4000000000ull;   // ~2 s at 2 GHz
constexpr unsigned int kErrTimeout = 9u;
static_assert(kTmemCols == 512, "tensor memory budget");

struct __align__(8) Barriers {
    uint64_t lfull[kLoadStages];    // x + weights (TMA bytes) and scales/zero-points (cp.async) landed
    uint64_t lempty[kLoadStages];   // MMAs reading the x tile retired (tcgen05.commit)
    uint64_t bfull[kBStages];       // dequantised operand tile written (one arrival per dequant warp)
    uint64_t bempty[kBStages];      // MMAs reading the operand tile retired (tcgen05.commit)
    uint64_t tfull[2];              // accumulator complete
    uint64_t tempty[2];             // accumulator drained by the epilogue (one arrival per epilogue warp)
    uint64_t drain;                 // final commit of the MMA thread
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes =
    1024 /*align slack*/ + kLoadStages * kLoadStageBytes + kBStages * kBBytes + sizeof(Barriers);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// Bounded wait: false if the wait ran out (or another role already gave up).
// The thread sleeps inside try_wait while the phase is incomplete.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait_suspend(bar, parity, kSuspendNs)) return true;
        if (*abort) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort = 1;
            atomicOr(&g_device_error, 1u << kErrTimeout);
            return false;
        }
    }
}

// Lane 0 waits (bounded) and acquires the completed phase; the warp-wide
// shuffle that broadcasts the verdict also orders the other lanes' later
// accesses after lane 0's acquire. (Letting all 32 lanes poll one mbarrier
// serialises their polls and costs hundreds of cycles per wait.)
__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity, volatile int* abort, int lane) {
    int ok = 1;
    if (lane == 0) ok = wait_bar(bar, parity, abort) ? 1 : 0;
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

template <bool kBf16, bool kSym>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
            const uint16_t* __restrict__ sc, const uint32_t* __restrict__ qz, uint16_t* __restrict__ y, int M,
            int N, int K, int g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* bsmem = smem + kLoadStages * kLoadStageBytes;
    Barriers* bars = reinterpret_cast<Barriers*>(bsmem + kBStages * kBBytes);
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t bsmem_base = smem_u32(bsmem);
    // load stage s: [x tile (two 128-row halves) | packed weights | scales | zero-point words]
    auto ld_a = [&](int s) { return smem_base + s * kLoadStageBytes; };
    auto ld_w = [&](int s) { return smem + s * kLoadStageBytes + kABytes; };
    auto ld_s = [&](int s) { return smem + s * kLoadStageBytes + kABytes + kWBytes; };
    auto ld_z = [&](int s) { return smem + s * kLoadStageBytes + kABytes + kWBytes + kSBytes; };
    auto op_b = [&](int s) { return bsmem_base + s * kBBytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_m = (M + BM - 1) / BM, num_n = (N + BN - 1) / BN;
    const int tiles = num_m * num_n;
    const int kt_total = (K + BK - 1) / BK;
    const int groups = K / g;
    volatile int* abort_flag = &bars->abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kLoadStages; ++s) {
            mbar_init(smem_u32(&bars->lfull[s]), 1);
            mbar_init(smem_u32(&bars->lempty[s]), 1);
        }
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(smem_u32(&bars->bfull[s]), kDeqWarps);
            mbar_init(smem_u32(&bars->bempty[s]), 1);
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
    }
    if (warp == 2) tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer warp
        // lane l stages, for 32-row half (l >> 4) of the step, the scales of the
        // 8 columns [8(l&15), 8(l&15)+8) and their zero-point word with cp.async
        // (zero-filled outside N and K); lane 0 then issues the TMA copies of the
        // x tile and the packed weight tile.
        const int half = lane >> 4, sub = lane & 15;
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_parity[kLoadStages];
        bool issued[kLoadStages];
        for (int s = 0; s < kLoadStages; ++s) issued[s] = false, issued_parity[s] = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
            const int m_blk = t % num_m, n_blk = t / num_m;
            const int n = n_blk * BN + 8 * sub;
            for (int kt = 0; kt < kt_total; ++kt) {
                if (!warp_wait_bar(smem_u32(&bars->lempty[stage]), phase ^ 1u, abort_flag, lane)) { ok = false; break; }
                const uint32_t fb = smem_u32(&bars->lfull[stage]);
                const int grp = (kt * BK + half * (BK / 2)) / g;
                const bool valid = n < N && grp < groups;
                const size_t so = valid ? static_cast<size_t>(grp) * N + n : 0;
                cp_async_16(smem_u32(ld_s(stage)) + half * (BN * 2) + 16 * sub, sc + so, valid ? 16u : 0u);
                if constexpr (!kSym) {
                    const size_t zo = valid ? static_cast<size_t>(grp) * (N >> 3) + (n >> 3) : 0;
                    cp_async_4(smem_u32(ld_z(stage)) + half * (BN / 8) * 4 + 4 * sub, qz + zo, valid ? 4u : 0u);
                }
                cp_async_mbar_arrive(fb);
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_expect_tx(fb, kABytes + kWBytes);
                    tma_load_2d(ld_a(stage), &tmap_x, kt * BK, m_blk * BM, fb);
                    tma_load_2d(smem_u32(ld_w(stage)), &tmap_w, n_blk * BN, kt * (BK / 8), fb);
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
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdesc = umma_idesc_f16(UM, BN, kBf16);
            int ls = 0, bs = 0;
            uint32_t lph = 0, bph = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                if (!wait_bar(smem_u32(&bars->tempty[acc]), acc_phase ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
                for (int kt = 0; kt < kt_total; ++kt) {
                    if (!wait_bar(smem_u32(&bars->lfull[ls]), lph, abort_flag) ||
                        !wait_bar(smem_u32(&bars->bfull[bs]), bph, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bdesc = sw128_kmajor_desc(op_b(bs));
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        // M half h: rows [128h, 128h + 128) of the x tile -> accumulator columns [128h, 128h + 128)
                        const uint64_t adesc = sw128_kmajor_desc(ld_a(ls) + h * (UM * BK * 2));
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            // advance 16 elements (32 bytes) along K inside the swizzle atom
                            umma_f16(d_tmem + h * BN, adesc + 2u * kk, bdesc + 2u * kk, kIdesc, (kt | kk) != 0);
                        }
                    }
                    umma_commit(smem_u32(&bars->lempty[ls]));
                    umma_commit(smem_u32(&bars->bempty[bs]));
                    if (++ls == kLoadStages) { ls = 0; lph ^= 1u; }
                    if (++bs == kBStages) { bs = 0; bph ^= 1u; }
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
        const int q = warp & 3;                 // tensor-memory lane quarter of this warp
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
            const int m_blk = t % num_m, n_blk = t / num_m;
            if (!warp_wait_bar(smem_u32(&bars->tfull[acc]), acc_phase, abort_flag, lane)) break;
            tc_fence_after();
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                const int m = m_blk * BM + h * UM + q * 32 + lane;
                uint16_t* yrow = y + static_cast<size_t>(m) * N;
#pragma unroll 1
                for (int ch = 0; ch < BN / 32; ++ch) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                           static_cast<uint32_t>(acc * kAccCols + h * BN + ch * 32),
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
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->tempty[acc]));
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    } else if (warp >= kDeqWarp0) {
        // ------------------------------------------------------------ dequantisers
        const int td = threadIdx.x - kDeqWarp0 * 32;   // 0..255
        const int d = td & (BN - 1);                     // column of the tile
        const int half = td >> 7;                        // 32-row half of the step: words 4*half .. 4*half+3
        int ls = 0, bs = 0;
        uint32_t lph = 0, bph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
            for (int kt = 0; kt < kt_total; ++kt) {
                if (!warp_wait_bar(smem_u32(&bars->lfull[ls]), lph, abort_flag, lane) ||
                    !warp_wait_bar(smem_u32(&bars->bempty[bs]), bph ^ 1u, abort_flag, lane)) {
                    ok = false;
                    break;
                }
                const uint32_t* wt = reinterpret_cast<const uint32_t*>(ld_w(ls));
                const uint16_t* st = reinterpret_cast<const uint16_t*>(ld_s(ls));
                const uint32_t* zt = reinterpret_cast<const uint32_t*>(ld_z(ls));
                const uint32_t b_row = op_b(bs) + static_cast<uint32_t>(d) * 128u;
                const uint32_t s16 = st[half * BN + d];
                const uint32_t z4 = kSym ? 8u : ((zt[half * (BN / 8) + (d >> 3)] >> (4 * (d & 7))) & 0xFu);
                const uint32_t ss = s16 | (s16 << 16);
                const uint32_t zz = Deq<kBf16>::kMagic | z4 | (z4 << 16);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int c = half * 4 + cc;
                    const uint32_t w = wt[c * BN + d];
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
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->bfull[bs]));
                if (++ls == kLoadStages) { ls = 0; lph ^= 1u; }
                if (++bs == kBStages) { bs = 0; bph ^= 1u; }
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

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <bool kBf16, bool kSym>
cudaError_t launch_typed(const void* x, const uint32_t* qw, const void* sc, const uint32_t* qz, void* y, int M,
                         int N, int K, int g, const DeviceProps& dp, cudaStream_t s) {
    auto kern = gemm_kernel<kBf16, kSym>;
    static int configured_device[64] = {0};
    if (dp.device >= 0 && dp.device < 64 && !configured_device[dp.device]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        configured_device[dp.device] = 1;
    }
    CUtensorMap tx, tw;
    const CUtensorMapDataType adt = kBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (!encode_2d(&tx, adt, x, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, BK, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (!encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_INT32, qw, (uint64_t)N, (uint64_t)(K / 8),
                   (uint64_t)N * 4, BN, BK / 8, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int grid = std::max(1, std::min(tiles, dp.sms));
    kern<<<grid, kThreads, kSmemBytes, s>>>(tx, tw, static_cast<const uint16_t*>(sc), qz, static_cast<uint16_t*>(y),
                                            M, N, K, g);
    return cudaGetLastError();
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
