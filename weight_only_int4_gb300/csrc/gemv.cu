// Decode GEMV of the W4A16 layer (and of MXFP4 weights), 1 <= M <= 16.
//
// The kernel is memory-bound: per call it must stream K*N/2 bytes of packed
// weights, (K/g)*N scales and (K/g)*N/2 bytes of packed zero-points, each once.
// "Keep W4A16 zero-points packed at 4 bits instead of expanding to 2 bytes"
// (sections "Problem" and "Known regression") shows both halves of the design
// problem: time tracks bytes, and at batch 4 the nibble extract costs time
// unless the loads of the next tile are in flight while the current one is
// converted. Here:
//
//   * Work items are (column block, 32-row chunk of K) pairs, ordered column
//     block first. A persistent grid of at most one CTA per SM takes equal
//     contiguous ranges of items ("stream-K"), so every SM streams the same
//     number of bytes whatever N and K are. When CTAs have few chunks per
//     warp, a grid of a whole number of CTAs per column block is taken
//     instead if it is cheaper: no range then crosses a block boundary. One
//     row takes 288-column blocks where that gives every CTA one whole block.
//   * Inside a CTA the warps take the chunks of the current column block in
//     turn. Each warp streams its chunks through its own kStages-deep ring in
//     shared memory: one lane issues bulk asynchronous copies (TMA, completion
//     counted in bytes on the stage's mbarrier) of the chunk's 4 packed word
//     rows, its scales, its packed zero-points and the x slice, kStages chunks
//     ahead of the one being converted, so memory and ALU overlap with about
//     kWarps * (kStages - 1) chunks in flight per CTA and no load instructions
//     on the lanes. A lane owns COLS columns in groups of adjacent columns,
//     32 groups apart, so its shared-memory reads are contiguous across the warp.
//   * Nibbles become 16-bit floats by the exponent-bias trick: OR a nibble into
//     the mantissa of 1024.0 (fp16) or 128.0 (bf16). One row (and two rows of
//     small layers) use FP32 FMAs with the zero-point applied once per chunk
//     through
//         sum_k (q - z) x = sum_k (magic + q) x - (magic + z) sum_k x,
//     with sum_k x of the chunk formed by a warp reduction over the chunk's x
//     slice (one value per lane) when the chunk is converted, or, when every
//     warp has many chunks to amortise it over, computed for all chunks once
//     per CTA after the dependency wait (kXPre); the products
//     (magic + q) * x are exact in an FP32 FMA with 16-bit inputs
//     (fma.rn.f32.f16 / .bf16). More rows go through warp-level m16n8k16
//     tensor-core MMAs (kMma): (q - z) exact in packed 16-bit arithmetic as
//     the A operand, x as B, FP32 accumulators. The scale is applied in FP32
//     once per chunk.
//   * Column blocks split between CTAs are summed deterministically in
//     ascending CTA order: within a thread-block cluster over distributed
//     shared memory when the grid is block-aligned and all clusters fit,
//     otherwise by the last CTA to take the block's atomic ticket, which
//     reads the others' partial vectors from the workspace and resets the
//     ticket to zero for the next call.
#include "internal.h"
#include "mxfp4.cuh"
#include "ptx.cuh"
#include "tmap.h"

#include <algorithm>
#include <cstring>
#include <array>
#include <map>
#include <mutex>
#include <tuple>

namespace w4a16 {

__device__ unsigned int g_gemv_error = 0;

namespace {

// Warps per CTA and depth of each warp's shared-memory ring.
#ifndef W4A16_GEMV_WARPS
#define W4A16_GEMV_WARPS 16
#endif
#ifndef W4A16_GEMV_STAGES
#define W4A16_GEMV_STAGES 2
#endif
// Chunks per warp whose weights are prefetched into L2 before the grid
// dependency wait (FMA and MMA conversions), and whether launches allow
// programmatic overlap with the preceding kernel of the stream. Measured (us,
// depth 0 / 1 / 2): 1x43008x5376 25.84 / 24.42 / 24.66, 1x5376x21504 15.03 /
// 14.40 / 14.71 on FMAs; 4x43008x5376 38.75 / 40.21 / 40.18, 4x4096x2048 4.90
// / 5.03 / 5.15 on MMAs.
#ifndef W4A16_GEMV_L2_PREFETCH
#define W4A16_GEMV_L2_PREFETCH 1
#endif
#ifndef W4A16_GEMV_L2_PREFETCH_MMA
#define W4A16_GEMV_L2_PREFETCH_MMA 0
#endif
#ifndef W4A16_GEMV_PDL
#define W4A16_GEMV_PDL 1
#endif
constexpr int kWarps = W4A16_GEMV_WARPS;
constexpr int kStages = W4A16_GEMV_STAGES;
// Ring depth of the MMA templates (8 rows x 128 columns, 16 rows x 64
// columns): their chunks convert several times faster, so more copies must be
// in flight to cover the load latency.
#ifndef W4A16_GEMV_MMA_STAGES8
#define W4A16_GEMV_MMA_STAGES8 2
#endif
#ifndef W4A16_GEMV_MMA_STAGES16
#define W4A16_GEMV_MMA_STAGES16 2
#endif
__host__ __device__ constexpr int ring_stages(bool mma, int mt) {
    return !mma ? kStages : mt == 8 ? W4A16_GEMV_MMA_STAGES8 : W4A16_GEMV_MMA_STAGES16;
}
constexpr int kL2Prefetch = W4A16_GEMV_L2_PREFETCH;
constexpr int kL2PrefetchMma = W4A16_GEMV_L2_PREFETCH_MMA;
constexpr int kThreads = kWarps * 32;
constexpr int kChunk = 32;            // rows of K per chunk
constexpr int kRowsPerChunk = 4;      // packed word rows per chunk
constexpr int kFactMaxM = 4;          // zero-point through the chunk's sum of x up to this M
// W4A16 rows from this M on go through the tensor-core MMA conversion (kMma)
#ifndef W4A16_GEMV_MMA_MIN_M
#define W4A16_GEMV_MMA_MIN_M 2
#endif
constexpr int kMmaMinM = W4A16_GEMV_MMA_MIN_M;
// ... except layers of at most kFmaSmallMaxWeights weights with at most
// kFmaSmallMaxM rows, which stay on FP32 FMAs (2048 x 2048, M = 2: 4.03 us
// against 4.24 with MMAs; from M = 3 the MMA conversion wins: 4.39 -> 4.32).
constexpr int kFmaSmallMaxM = 2;
constexpr long long kFmaSmallMaxWeights = 4ll << 20;

constexpr int kXPreMinChunksPerWarp = 8;
constexpr size_t kXsumSmemLimit = 32 * 1024;
constexpr unsigned long long kWaitLimitCycles = 4000000000ull;   // ~2 s at 2 GHz
constexpr unsigned int kErrTimeout = 9u;

template <bool kBf16>
struct Act;
template <>
struct Act<false> {
    static constexpr uint32_t kMagic = 0x64006400u;   // fp16 1024.0 in both halves
    static constexpr float kMagicF = 1024.f;
    __device__ static float to_float(uint16_t b) { return __half2float(__ushort_as_half(b)); }
    __device__ static uint16_t from_float(float v) { return __half_as_ushort(__float2half_rn(v)); }
    __device__ static uint32_t sub2(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
};
template <>
struct Act<true> {
    static constexpr uint32_t kMagic = 0x43004300u;   // bf16 128.0 in both halves
    static constexpr float kMagicF = 128.f;
    __device__ static float to_float(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
    __device__ static uint16_t from_float(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
    __device__ static uint32_t sub2(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
};

// One stage of a warp's ring holds, for one 32-row chunk of K and one column
// block of CB = 32 * COLS columns: the 4 packed word rows [4][CB], the scales
// [CB], the zero-point words [CB / 8] and the x slice [M][32]. A lane owns
// COLS columns in groups of W adjacent columns (W = 4, or 3 for 9 columns a
// lane), one group per 32*W columns, so every lane-wise shared-memory read of
// a warp covers contiguous bytes (3-column groups: three 4-byte reads, still
// conflict free; their 2-byte scale reads conflict a little). The MMA
// conversion reads the same layout with its own lane mapping.
__host__ __device__ constexpr int round128(int v) { return (v + 127) & ~127; }

__host__ __device__ constexpr int group_width(int cols) { return cols < 4 ? cols : cols % 4 == 0 ? 4 : 3; }
// A tensor copy moves at most 256 elements along a row: wider blocks arrive
// as one copy per lane group (32 * W columns each).
__host__ __device__ constexpr bool split_boxes(int cols) { return 32 * cols > 256; }
__host__ __device__ constexpr int box_cols(int cols) { return split_boxes(cols) ? 32 * group_width(cols) : 32 * cols; }
__host__ __device__ constexpr int scale_bytes(int cols) {
    return split_boxes(cols) ? (cols / group_width(cols)) * round128(box_cols(cols) * 2) : round128(32 * cols * 2);
}

template <int COLS, int MT>
struct Stage {
    static constexpr int CB = 32 * COLS;
    static constexpr int W = group_width(COLS);           // columns per group
    static constexpr int G = COLS / W;                    // groups per lane
    static_assert(COLS % W == 0, "whole groups");
    static constexpr bool kSplit = split_boxes(COLS);     // [G][4][32W] words, G scale rows
    static constexpr int kBox = box_cols(COLS);
    static constexpr int kSStride = kSplit ? round128(kBox * 2) : 0;   // bytes between the groups' scale rows
    // every block is a tensor-copy destination: 128-byte aligned
    static constexpr int kQ = 0;                                          // [4][CB] (or [G][4][kBox]) uint32
    static constexpr int kS = kQ + round128(kRowsPerChunk * CB * 4);      // [CB] 16-bit scales (or G rows)
    static constexpr int kZ = kS + scale_bytes(COLS);                     // [CB / 8] uint32
    static constexpr int kX = kZ + round128(CB / 2);                      // [MT][32] 16-bit x
    static constexpr int kBytes = kX + round128(MT * kChunk * 2);
    static_assert(kS % 128 == 0 && kZ % 128 == 0 && kX % 128 == 0 && kBytes % 128 == 0 &&
                      (kRowsPerChunk * kBox * 4) % 128 == 0,
                  "tensor-copy destinations must be 128-byte aligned");
    __device__ static int col(int lane, int gi, int u) { return gi * 32 * W + lane * W + u; }
    // byte offsets of the lane's group gi: word row i, and its scales
    __device__ static int q_off(int i, int lane, int gi) {
        return kSplit ? kQ + gi * (kRowsPerChunk * kBox * 4) + i * kBox * 4 + lane * W * 4
                      : kQ + i * CB * 4 + col(lane, gi, 0) * 4;
    }
    // `bytes`: 2 for 16-bit scales, 1 for MXFP4 exponent bytes (whose rows fit
    // the same slots)
    __device__ static int s_off(int lane, int gi, int bytes = 2) {
        return kSplit ? kS + gi * kSStride + lane * W * bytes : kS + col(lane, gi, 0) * bytes;
    }
};

__host__ __device__ constexpr int stage_bytes(int cols, int mt) {
    return round128(kRowsPerChunk * 32 * cols * 4) + scale_bytes(cols) + round128(32 * cols / 2) +
           round128(mt * kChunk * 2);
}

template <int BYTES>
__device__ __forceinline__ void lds(uint32_t addr, uint32_t (&v)[(BYTES + 3) / 4]) {
    if constexpr (BYTES == 12) {   // three words, 4-byte aligned
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v[0]) : "r"(addr));
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v[1]) : "r"(addr + 4));
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v[2]) : "r"(addr + 8));
    } else if constexpr (BYTES == 3) {   // three bytes: v[0] = b0 | b1 << 8 | b2 << 16
        uint16_t b0, b1, b2;
        asm volatile("ld.shared.u8 %0, [%1];" : "=h"(b0) : "r"(addr));
        asm volatile("ld.shared.u8 %0, [%1];" : "=h"(b1) : "r"(addr + 1));
        asm volatile("ld.shared.u8 %0, [%1];" : "=h"(b2) : "r"(addr + 2));
        v[0] = static_cast<uint32_t>(b0) | (static_cast<uint32_t>(b1) << 8) | (static_cast<uint32_t>(b2) << 16);
    } else if constexpr (BYTES == 6) {   // three halves, 2-byte aligned: v[0] = h0 | h1 << 16, v[1] = h2
        uint16_t h0, h1, h2;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h0) : "r"(addr));
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h1) : "r"(addr + 2));
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h2) : "r"(addr + 4));
        v[0] = static_cast<uint32_t>(h0) | (static_cast<uint32_t>(h1) << 16);
        v[1] = h2;
    } else if constexpr (BYTES == 16)
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]) : "r"(addr));
    else if constexpr (BYTES == 8)
        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v[0]), "=r"(v[1]) : "r"(addr));
    else if constexpr (BYTES == 4)
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v[0]) : "r"(addr));
    else if constexpr (BYTES == 1)
        asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v[0]) : "r"(addr));
    else {
        uint16_t h;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(addr));
        v[0] = h;
    }
}

// Lane 0 waits, bounded (about two seconds), sleeping in try_wait, and
// acquires the completed phase; the shuffle and warp barrier that follow order
// the other lanes' reads of the stage after that acquire. (Letting all 32 lanes
// poll one mbarrier serialises their polls and costs hundreds of cycles.)
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int lane) {
    int ok = 1;
    if (lane == 0 && !mbar_try_wait(bar, parity)) {
        const unsigned long long t0 = clock64();
        while (!mbar_try_wait_suspend(bar, parity, 20000)) {
            if (clock64() - t0 > kWaitLimitCycles) {
                atomicOr(&g_gemv_error, 1u << kErrTimeout);
                ok = 0;
                break;
            }
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

struct GemvArgs {
    CUtensorMap tq;       // qweight int32 [K/8, N], box [4 rows, CB]
    CUtensorMap ts;       // scales 16-bit [K/g, N] (MXFP4: exponent bytes [K/32, N]), box [1, CB]
    CUtensorMap tz;       // qzeros int32 [K/g, N/8], box [1, CB/8] (used when N % 32 == 0)
    CUtensorMap tx;       // x 16-bit [M, K], box [MT rows, 32]
    const uint32_t* qz;
    uint16_t* y;
    uint32_t* tickets;    // [n_cb], zero between calls
    float* partials;      // [grid][2][M * CB], at most kMaxLive floats per slot
    const uint16_t* x;
    int M, N, K, g_shift;
    int chunks;
    int cluster;          // > 1: the grid is clusters of this many CTAs, one column block each
    long long items;      // n_cb * chunks
};

__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(pred));
    return pred != 0;
}

// Byte offsets inside dynamic shared memory: warp partials | chunk sums of x (kXPre) | barriers | rings.
__host__ __device__ constexpr uint32_t xsum_offset(int live_per_warp) { return kWarps * live_per_warp * 4; }
__host__ __device__ constexpr uint32_t bar_offset(int live_per_warp, int xsum_entries) {
    return (xsum_offset(live_per_warp) + xsum_entries * 8 + 15) & ~15u;
}
__host__ __device__ constexpr uint32_t ring_offset(int live_per_warp, int xsum_entries, int stages) {
    return (bar_offset(live_per_warp, xsum_entries) + kWarps * stages * 8 + 127) & ~127u;
}

// First CTA whose item range contains item i (ranges are [b*T/G, (b+1)*T/G)).
__device__ __forceinline__ int owner_cta(long long i, long long T, int G) {
    return static_cast<int>(((i + 1) * G - 1) / T);
}
__device__ __forceinline__ long long range_start(int b, long long T, int G) { return (long long)b * T / G; }

// kMx: MXFP4 weights (bf16, with kSym and without kFact or kZBulk): each
// 32-row chunk is one E8M0 block. The warp first rewrites the chunk's bf16 x
// slice in place as fp16 scaled by a power of two per row (mx::x_to_f16);
// codes become fp16 pairs in one conversion instruction each, the products
// are exact in an FP32 FMA with fp16 inputs, and the power of two and the
// block scale 2^(e - 127) are applied in FP32 once per chunk.
// kXPre (with kFact): the chunk sums of x are computed for every chunk once per
// CTA, right after the dependency wait, instead of by a warp reduction in each
// chunk; worth it when every warp has many chunks to amortise it over.
// kMma: the products of a chunk go through warp-level m16n8k16 tensor-core
// MMAs instead of FP32 FMAs (rows 2..16): weights as A (16 columns x 16 k per
// MMA, (q - z) exact in 16 bits), x as B (8 rows per MMA, rows >= M zero),
// FP32 accumulators scaled once per chunk.
template <bool kBf16, int MT, int COLS, bool kSym, bool kFact, bool kZBulk, bool kMx = false, bool kXPre = false,
          bool kMma = false>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const __grid_constant__ GemvArgs a) {
    static_assert(!kXPre || kFact, "precomputed chunk sums serve the zero-point factorisation");
    static_assert(!kMma || (!kFact && ((MT == 8 && (COLS == 4 || COLS == 2)) || (MT == 16 && COLS == 2))),
                  "MMA conversion: 8 rows x 128 or 64 columns, 16 rows x 64 columns, zero-points per nibble pair");
    static_assert(!kMx || (kBf16 && kSym && !kFact && !kZBulk), "MXFP4: bf16, no zero-points");
    static_assert(!kMx || Stage<COLS, MT>::kX - Stage<COLS, MT>::kZ >= 4 * MT, "row factors fit the zero-point block");
    using A = Act<kBf16>;
    using St = Stage<COLS, MT>;
    constexpr int CB = St::CB;
    constexpr int E = MT * CB;
    constexpr int W = St::W, G = St::G;
    constexpr bool kTwoFamilies = kFact && !kBf16;   // fp16: nibbles at bits 0-3 and 4-7 of a half
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_last;

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);   // warp-uniform
    const int lane = threadIdx.x & 31;
    const int M = a.M, N = a.N, K = a.K, g_shift = a.g_shift, chunks = a.chunks;
    const long long T = a.items;
    const int Gd = gridDim.x, b = blockIdx.x;
    const long long i_begin = range_start(b, T, Gd), i_end = range_start(b + 1, T, Gd);
    float* red = reinterpret_cast<float*>(smem);                                   // [kWarps][E]
    const int xs_entries = kXPre ? M * chunks : 0;
    float2* xsum = reinterpret_cast<float2*>(smem + xsum_offset(E));               // [M][chunks] (kXPre)
    constexpr int kSt = ring_stages(kMma, MT);   // depth of each warp's ring
    const uint32_t bars = smem_u32(smem) + bar_offset(E, xs_entries) + warp * kSt * 8;
    // rings start on a 128-byte boundary of the shared window (128 bytes of slack are reserved)
    const uint32_t ring = ((smem_u32(smem) + ring_offset(E, xs_entries, kSt) + 127u) & ~127u) + warp * kSt * St::kBytes;

    // The next kernel of the stream may start its own prologue as this grid's
    // CTAs exit. Before the dependency wait below this grid touches no caller
    // data: it only initialises barriers and asks L2 for the weights of each
    // warp's first chunks.
    griddep_launch_dependents();
    if (lane == 0) {
        for (int st = 0; st < kSt; ++st) mbar_init(bars + 8 * st, 1);
        fence_mbar_init();
        if (warp == 0) {
            tma_prefetch_desc(&a.tq);
            tma_prefetch_desc(&a.ts);
            if constexpr (kZBulk) tma_prefetch_desc(&a.tz);
            tma_prefetch_desc(&a.tx);
        }
        if (i_begin < i_end) {
            const int cb = static_cast<int>(i_begin / chunks);
            const int c0 = static_cast<int>(i_begin - static_cast<long long>(cb) * chunks);
            const int c1 = static_cast<int>(std::min<long long>(chunks, c0 + (i_end - i_begin)));
            constexpr int kPf = kMma ? kL2PrefetchMma : kL2Prefetch;
            for (int j = 0, c = c0 + warp; j < kPf && c < c1; ++j, c += kWarps) {
                const int t = (c * kChunk) >> g_shift;
#pragma unroll
                for (int gi = 0; gi < (St::kSplit ? G : 1); ++gi) {
                    tma_prefetch_l2_2d(&a.tq, cb * CB + gi * St::kBox, c * kRowsPerChunk);
                    tma_prefetch_l2_2d(&a.ts, cb * CB + gi * St::kBox, t);
                }
                if constexpr (kZBulk) tma_prefetch_l2_2d(&a.tz, cb * (CB / 8), t);
            }
        }
    }
    __syncthreads();
    griddep_wait();

    // kXPre: per (row, chunk), the sum of x over the chunk and the offset the
    // magic bias adds, computed once while the first copies are in flight
    auto chunk_sums = [&]() {
        for (int p = threadIdx.x; p < M * chunks; p += kThreads) {
            const int m = p / chunks, c = p - m * chunks;
            const uint4* xp = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(m) * K + c * kChunk);
            float se = 0.f, so = 0.f;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 u = __ldg(xp + v);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    se += A::to_float(static_cast<uint16_t>(w[h]));
                    so += A::to_float(static_cast<uint16_t>(w[h] >> 16));
                }
            }
            const float off = kTwoFamilies ? (A::kMagicF * se + (A::kMagicF / 16.f) * so) : A::kMagicF * (se + so);
            xsum[p] = make_float2(off, se + so);
        }
    };
    bool sums_pending = kXPre;

    uint32_t phase_bits = 0;   // parity of the next completion of each stage's barrier
    bool ok = true;
    int drain_lo = 0, drain_hi = 0;   // after a timeout: this warp's chunks whose copies may be in flight

    for (long long it = i_begin; it < i_end;) {
        const int cb = static_cast<int>(it / chunks);
        const int c0 = static_cast<int>(it - static_cast<long long>(cb) * chunks);
        const int c1 = static_cast<int>(std::min<long long>(chunks, c0 + (i_end - it)));
        const int nj = ok ? (c1 - c0 - warp + kWarps - 1) / kWarps : 0;   // this warp's chunks

        float yacc[MT][COLS];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int j = 0; j < COLS; ++j) yacc[m][j] = 0.f;

        // one lane: bring chunk c of this column block into stage st (tensor TMA, 4 copies)
        auto issue = [&](int st, int c) {
            const uint32_t base = ring + st * St::kBytes, bar = bars + 8 * st;
            const int t = (c * kChunk) >> g_shift;
            constexpr uint32_t kBytes =
                kRowsPerChunk * CB * 4 + (kMx ? CB : CB * 2) + (kZBulk ? CB / 2 : 0) + MT * kChunk * 2;
            mbar_arrive_expect_tx(bar, kBytes);
            if constexpr (St::kSplit) {
#pragma unroll
                for (int gi = 0; gi < G; ++gi) {
                    tma_load_2d(base + St::kQ + gi * (kRowsPerChunk * St::kBox * 4), &a.tq, cb * CB + gi * St::kBox,
                                c * kRowsPerChunk, bar);
                    tma_load_2d(base + St::kS + gi * St::kSStride, &a.ts, cb * CB + gi * St::kBox, t, bar);
                }
            } else {
                tma_load_2d(base + St::kQ, &a.tq, cb * CB, c * kRowsPerChunk, bar);
                tma_load_2d(base + St::kS, &a.ts, cb * CB, t, bar);
            }
            if constexpr (kZBulk) tma_load_2d(base + St::kZ, &a.tz, cb * (CB / 8), t, bar);
            tma_load_2d(base + St::kX, &a.tx, c * kChunk, 0, bar);
        };

        // kMx: lane l rescales x[m][l] of every row m < M of the stage's x
        // slice to fp16 in place; the rows' factors 2^-c go to the stage's
        // zero-point block, unused without zero-points
        auto mx_rescale = [&](uint32_t base) {
            uint16_t xb[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                xb[m] = 0;
                if (m < M)
                    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(xb[m]) : "r"(base + St::kX + m * kChunk * 2 + lane * 2));
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < M) {   // warp-uniform
                    const uint32_t emax = __reduce_max_sync(0xffffffffu, (static_cast<uint32_t>(xb[m]) >> 7) & 0xFFu);
                    const int sh = mx::x_shift(emax);
                    const uint32_t addr = base + St::kX + m * kChunk * 2 + lane * 2;
                    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(mx::x_to_f16(xb[m], sh)) : "memory");
                    if (lane == 0)
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(base + St::kZ + 4 * m), "f"(mx::x_unshift(sh))
                                     : "memory");
                }
            }
            __syncwarp();
        };

        auto compute = [&](int st, int c) {
            const uint32_t base = ring + st * St::kBytes;
            if constexpr (kMx) mx_rescale(base);
            // scales and zero-points of the lane's columns
            // zw: the zero-point word of the group's first column; zw2: of its last
            // (a 3-column group can cross a word)
            uint32_t sw[G][(2 * W + 3) / 4], zw[G], zw2[G];
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
                const int c0l = St::col(lane, gi, 0);
                if constexpr (kMx) {
                    uint32_t e[1];   // the W exponent bytes of the group
                    lds<W>(base + St::s_off(lane, gi, 1), e);
                    sw[gi][0] = e[0];
                } else
                    lds<2 * W>(base + St::s_off(lane, gi), sw[gi]);
                if constexpr (!kSym) {
                    const int c1l = c0l + W - 1;
                    if constexpr (kZBulk) {
                        uint32_t v[1];
                        lds<4>(base + St::kZ + (c0l >> 3) * 4, v);
                        zw[gi] = v[0];
                        if constexpr (W == 3) {
                            lds<4>(base + St::kZ + (c1l >> 3) * 4, v);
                            zw2[gi] = v[0];
                        } else {
                            zw2[gi] = zw[gi];
                        }
                    } else {
                        const int t = (c * kChunk) >> g_shift;
                        const int n = cb * CB + c0l, n1 = cb * CB + c1l;
                        const uint32_t* zr = a.qz + static_cast<size_t>(t) * (N >> 3);
                        zw[gi] = n < N ? __ldg(zr + (n >> 3)) : 0u;
                        if constexpr (W == 3)
                            zw2[gi] = n1 < N ? __ldg(zr + (n1 >> 3)) : 0u;
                        else
                            zw2[gi] = zw[gi];
                    }
                } else {
                    zw[gi] = 0u;
                    zw2[gi] = 0u;
                }
            }
            auto zval = [&](int j) -> uint32_t {
                const int gi = j / W, u = j % W;
                if constexpr (kSym) return 8u;
                if constexpr (W == 3) {
                    const int cl = St::col(lane, gi, 0), cu = cl + u;
                    const uint32_t w = (cu >> 3) == (cl >> 3) ? zw[gi] : zw2[gi];
                    return (w >> (4 * (cu & 7))) & 0xFu;
                } else {
                    return (zw[gi] >> (4 * ((St::col(lane, gi, 0) & 7) + u))) & 0xFu;
                }
            };
            auto sval = [&](int j) -> float {
                const int gi = j / W, u = j % W;
                if constexpr (kMx) return mx::scale_f32((sw[gi][u / 4] >> (8 * (u & 3))) & 0xFFu);
                return A::to_float(static_cast<uint16_t>(sw[gi][u / 2] >> (16 * (u & 1))));
            };

            // kFact: the accumulators collect sum (magic + q) x; (magic + z) * sum x is
            // subtracted when the chunk is scaled, so the reduction that forms sum x
            // runs beside the FMAs instead of ahead of them (with kXPre it is the
            // accumulators' starting value)
            float acc[MT][COLS], acc2[kTwoFamilies ? MT : 1][kTwoFamilies ? COLS : 1];
            float2 os[kFact ? MT : 1];
            if constexpr (kXPre) {
#pragma unroll
                for (int m = 0; m < MT; ++m) os[m] = (m < M) ? xsum[m * chunks + c] : make_float2(0.f, 0.f);
            } else if constexpr (kFact) {
                // per row: sum of x over the chunk and the offset the magic bias adds,
                // from the stage's x slice (lane l holds x[m][l]; the butterfly leaves
                // the same sums in every lane)
                float v[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    uint16_t xb = 0;
                    if (m < M)
                        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(xb) : "r"(base + St::kX + m * kChunk * 2 + lane * 2));
                    v[m] = A::to_float(xb);
                }
                // the rows' butterflies interleaved, so their shuffle latencies overlap
#pragma unroll
                for (int k = 16; k >= 2; k >>= 1)
#pragma unroll
                    for (int m = 0; m < MT; ++m) v[m] += __shfl_xor_sync(0xffffffffu, v[m], k);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    // even lanes: sum of the low halves of x's words, odd lanes: of the high halves
                    const float other = __shfl_xor_sync(0xffffffffu, v[m], 1);
                    const float se = (lane & 1) ? other : v[m], so = (lane & 1) ? v[m] : other;
                    const float off = kTwoFamilies ? fmaf(A::kMagicF, se, (A::kMagicF / 16.f) * so)
                                                   : A::kMagicF * (se + so);
                    os[m] = make_float2(off, se + so);
                }
            }
            // precomputed sums are ready at once: start at -((magic + z) * sum x)
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int j = 0; j < COLS; ++j)
                    acc[m][j] = kXPre ? -fmaf(static_cast<float>(zval(j)), os[m].y, os[m].x) : 0.f;
            if constexpr (kTwoFamilies) {
#pragma unroll
                for (int m = 0; m < MT; ++m)
#pragma unroll
                    for (int j = 0; j < COLS; ++j) acc2[m][j] = 0.f;
            }
            uint32_t zz[COLS];
            if constexpr (!kFact && !kMx) {
#pragma unroll
                for (int j = 0; j < COLS; ++j) {
                    const uint32_t z = zval(j);
                    zz[j] = A::kMagic | z | (z << 16);
                }
            }
#pragma unroll
            for (int i = 0; i < kRowsPerChunk; ++i) {
                uint32_t q[COLS];
#pragma unroll
                for (int gi = 0; gi < G; ++gi) {
                    uint32_t v[W];
                    lds<4 * W>(base + St::q_off(i, lane, gi), v);
#pragma unroll
                    for (int u = 0; u < W; ++u) q[gi * W + u] = v[u];
                }
                // nibble pairs of this word row for every column, converted once ...
                uint32_t h[COLS][4];
#pragma unroll
                for (int j = 0; j < COLS; ++j) {
                    const uint32_t w = q[j];
                    if constexpr (kTwoFamilies) {
                        // (1024 + q[k], 1024 + q[k+4]), (1024 + 16 q[k+1], 1024 + 16 q[k+5]),
                        // (1024 + q[k+2], 1024 + q[k+6]), (1024 + 16 q[k+3], 1024 + 16 q[k+7])
                        const uint32_t w8 = w >> 8;
                        h[j][0] = and_or(w, 0x000F000Fu, A::kMagic);
                        h[j][1] = and_or(w, 0x00F000F0u, A::kMagic);
                        h[j][2] = and_or(w8, 0x000F000Fu, A::kMagic);
                        h[j][3] = and_or(w8, 0x00F000F0u, A::kMagic);
                    } else if constexpr (kMx) {
                        // (E2M1(q[k+2b]), E2M1(q[k+2b+1])) in fp16
                        mx::e2m1x8_to_f16x2(w, h[j]);
                    } else {
#pragma unroll
                        for (int bb = 0; bb < 4; ++bb) {
                            // (magic + q[k+bb], magic + q[k+bb+4]); minus (magic + z): exact (q - z)
                            h[j][bb] = and_or(w >> (4 * bb), 0x000F000Fu, A::kMagic);
                            if constexpr (!kFact) h[j][bb] = A::sub2(h[j][bb], zz[j]);
                        }
                    }
                }
                // ... then streamed against one row of x at a time
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    uint32_t xw[4] = {0u, 0u, 0u, 0u};
                    if (m < M) lds<16>(base + St::kX + m * kChunk * 2 + i * 16, xw);
#pragma unroll
                    for (int j = 0; j < COLS; ++j) {
                        if constexpr (kMx) {
                            // pair b holds x[k+2b], x[k+2b+1] (word b of the fp16 x row)
#pragma unroll
                            for (int b = 0; b < 4; ++b) {
                                acc[m][j] = fma_mixed<false, 0, 0>(h[j][b], xw[b], acc[m][j]);
                                acc[m][j] = fma_mixed<false, 1, 1>(h[j][b], xw[b], acc[m][j]);
                            }
                        } else if constexpr (kTwoFamilies) {
                            acc[m][j] = fma_mixed<false, 0, 0>(h[j][0], xw[0], acc[m][j]);
                            acc[m][j] = fma_mixed<false, 1, 0>(h[j][0], xw[2], acc[m][j]);
                            acc[m][j] = fma_mixed<false, 0, 0>(h[j][2], xw[1], acc[m][j]);
                            acc[m][j] = fma_mixed<false, 1, 0>(h[j][2], xw[3], acc[m][j]);
                            acc2[m][j] = fma_mixed<false, 0, 1>(h[j][1], xw[0], acc2[m][j]);
                            acc2[m][j] = fma_mixed<false, 1, 1>(h[j][1], xw[2], acc2[m][j]);
                            acc2[m][j] = fma_mixed<false, 0, 1>(h[j][3], xw[1], acc2[m][j]);
                            acc2[m][j] = fma_mixed<false, 1, 1>(h[j][3], xw[3], acc2[m][j]);
                        } else {
                            // pair bb holds x[k+bb] (word bb/2 of x, half bb&1) and x[k+bb+4]
                            acc[m][j] = fma_mixed<kBf16, 0, 0>(h[j][0], xw[0], acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 1, 0>(h[j][0], xw[2], acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 0, 1>(h[j][1], xw[0], acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 1, 1>(h[j][1], xw[2], acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 0, 0>(h[j][2], xw[1], acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 1, 0>(h[j][2], xw[3], acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 0, 1>(h[j][3], xw[1], acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 1, 1>(h[j][3], xw[3], acc[m][j]);
                        }
                    }
                }
            }
            // scale once per chunk, in FP32
#pragma unroll
            for (int j = 0; j < COLS; ++j) {
                const float s = sval(j);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float t = acc[m][j];
                    if constexpr (kTwoFamilies) t = fmaf(acc2[m][j], 0.0625f, t);
                    if constexpr (kFact && !kXPre) t -= fmaf(static_cast<float>(zval(j)), os[m].y, os[m].x);
                    if constexpr (kMx) {
                        if (m < M) {
                            float u;
                            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(u) : "r"(base + St::kZ + 4 * m));
                            t *= u;
                        }
                    }
                    yacc[m][j] = fmaf(s, t, yacc[m][j]);
                }
            }
        };

        // kMma: one chunk through tensor-core MMAs. Thread (r, c) = (lane / 4,
        // lane % 4) takes packed word row c (k = 8c .. 8c + 7) of its columns; a
        // super tile of 64 columns holds four MMA tiles, tile j mapping MMA row r
        // to column 4r + j and row r + 8 to column 32 + 4r + j. The nibble pairs
        // (k, k + 4), (k + 1, k + 5) feed the first MMA's k pairs and (k + 2,
        // k + 6), (k + 3, k + 7) the second's; x is permuted the same way, so
        // every product meets its own x. C fragment: column 4r + j (+ 32), rows
        // m = 8 nt + 2c, 2c + 1.
        auto compute_mma = [&](int st, int c) {
          if constexpr (kMma) {
            constexpr int NT = MT / 8, SU = CB / 64;
            const uint32_t base = ring + st * St::kBytes;
            const int r = lane >> 2, tg = lane & 3;
            if constexpr (kMx) mx_rescale(base);
            uint32_t bx[NT][4];
            float um[NT][2];   // kMx: the factors of the fragment's rows 8 nt + 2 tg (+1)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                uint32_t xw[4];
                lds<16>(base + St::kX + (8 * nt + r) * kChunk * 2 + tg * 16, xw);   // rows >= M: zero fill
                if constexpr (kMx) {
                    // E2M1 pairs are (k, k + 1): x in its own order
#pragma unroll
                    for (int i = 0; i < 4; ++i) bx[nt][i] = xw[i];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int m = 8 * nt + 2 * tg + e;
                        um[nt][e] = 0.f;   // rows >= M: no factor written (and the fragment is zero)
                        if (m < M)
                            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(um[nt][e]) : "r"(base + St::kZ + 4 * m));
                    }
                } else {
                    bx[nt][0] = __byte_perm(xw[0], xw[2], 0x5410);   // x[k], x[k + 4]
                    bx[nt][1] = __byte_perm(xw[0], xw[2], 0x7632);   // x[k + 1], x[k + 5]
                    bx[nt][2] = __byte_perm(xw[1], xw[3], 0x5410);   // x[k + 2], x[k + 6]
                    bx[nt][3] = __byte_perm(xw[1], xw[3], 0x7632);   // x[k + 3], x[k + 7]
                }
            }
#pragma unroll
            for (int u = 0; u < SU; ++u) {
                const int c_lo = 64 * u + 4 * r, c_hi = c_lo + 32;   // first of 4 adjacent columns
                uint32_t q_lo[4], q_hi[4], s_lo[2], s_hi[2];
                lds<16>(base + St::kQ + (tg * CB + c_lo) * 4, q_lo);
                lds<16>(base + St::kQ + (tg * CB + c_hi) * 4, q_hi);
                if constexpr (kMx) {   // 4 exponent bytes each
                    uint32_t e[1];
                    lds<4>(base + St::kS + c_lo, e);
                    s_lo[0] = e[0];
                    lds<4>(base + St::kS + c_hi, e);
                    s_hi[0] = e[0];
                    s_lo[1] = s_hi[1] = 0u;
                } else {
                    lds<8>(base + St::kS + c_lo * 2, s_lo);
                    lds<8>(base + St::kS + c_hi * 2, s_hi);
                }
                uint32_t z_lo = 0u, z_hi = 0u;   // the 4 columns' zero-points: nibbles 0..3
                if constexpr (!kSym && !kMx) {
                    if constexpr (kZBulk) {
                        uint32_t v[1];
                        lds<4>(base + St::kZ + (c_lo >> 3) * 4, v);
                        z_lo = v[0] >> (4 * (c_lo & 7));
                        lds<4>(base + St::kZ + (c_hi >> 3) * 4, v);
                        z_hi = v[0] >> (4 * (c_hi & 7));
                    } else {
                        const size_t row = static_cast<size_t>((c * kChunk) >> g_shift) * (N >> 3);
                        const int n_lo = cb * CB + c_lo, n_hi = cb * CB + c_hi;
                        z_lo = n_lo < N ? __ldg(a.qz + row + (n_lo >> 3)) >> (4 * (n_lo & 7)) : 0u;
                        z_hi = n_hi < N ? __ldg(a.qz + row + (n_hi >> 3)) >> (4 * (n_hi & 7)) : 0u;
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // (magic + z) in both halves; the difference with (magic + q) is exact
                    const uint32_t zl = kSym ? 8u : ((z_lo >> (4 * j)) & 0xFu);
                    const uint32_t zh = kSym ? 8u : ((z_hi >> (4 * j)) & 0xFu);
                    const uint32_t zzl = A::kMagic + zl * 0x10001u, zzh = A::kMagic + zh * 0x10001u;
                    uint32_t hl[4], hh[4];
                    float sl, sh;
                    if constexpr (kMx) {
                        // codes -> fp16 pairs (k, k + 1); block scales 2^(e - 127)
                        mx::e2m1x8_to_f16x2(q_lo[j], hl);
                        mx::e2m1x8_to_f16x2(q_hi[j], hh);
                        sl = mx::scale_f32((s_lo[0] >> (8 * j)) & 0xFFu);
                        sh = mx::scale_f32((s_hi[0] >> (8 * j)) & 0xFFu);
                    } else {
#pragma unroll
                        for (int bb = 0; bb < 4; ++bb) {
                            hl[bb] = A::sub2(and_or(q_lo[j] >> (4 * bb), 0x000F000Fu, A::kMagic), zzl);
                            hh[bb] = A::sub2(and_or(q_hi[j] >> (4 * bb), 0x000F000Fu, A::kMagic), zzh);
                        }
                        sl = A::to_float(static_cast<uint16_t>(s_lo[j >> 1] >> (16 * (j & 1))));
                        sh = A::to_float(static_cast<uint16_t>(s_hi[j >> 1] >> (16 * (j & 1))));
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        float d[4] = {0.f, 0.f, 0.f, 0.f};
                        // MXFP4: fp16 x fp16 (x rescaled); int4: the activation dtype
                        constexpr bool kMmaBf16 = kBf16 && !kMx;
                        mma_m16n8k16<kMmaBf16>(d, hl[0], hh[0], hl[1], hh[1], bx[nt][0], bx[nt][1]);
                        mma_m16n8k16<kMmaBf16>(d, hl[2], hh[2], hl[3], hh[3], bx[nt][2], bx[nt][3]);
                        if constexpr (kMx) {
                            d[0] *= um[nt][0];
                            d[1] *= um[nt][1];
                            d[2] *= um[nt][0];
                            d[3] *= um[nt][1];
                        }
                        float* y = &yacc[0][0] + ((nt * SU + u) * 4 + j) * 4;
                        y[0] = fmaf(sl, d[0], y[0]);
                        y[1] = fmaf(sl, d[1], y[1]);
                        y[2] = fmaf(sh, d[2], y[2]);
                        y[3] = fmaf(sh, d[3], y[3]);
                    }
                }
            }
          }
        };

        // this warp's chunks c0 + warp + kWarps * j, through its kStages-deep ring
        if (elect_one())
            for (int j = 0; j < kSt && j < nj; ++j) issue(j, c0 + warp + kWarps * j);
        __syncwarp();
        if constexpr (kXPre) {
            if (sums_pending) {   // CTA-uniform: every thread runs the same segments
                chunk_sums();
                __syncthreads();
                sums_pending = false;
            }
        }
        for (int j = 0; j < nj; ++j) {
            const int st = j % kSt;
            if (!warp_wait(bars + 8 * st, (phase_bits >> st) & 1u, lane)) {
                ok = false;
                drain_lo = j;
                drain_hi = std::min(nj, j + kSt);
                break;
            }
            phase_bits ^= 1u << st;
            if constexpr (kMma)
                compute_mma(st, c0 + warp + kWarps * j);
            else
                compute(st, c0 + warp + kWarps * j);
            // every lane's reads of the stage precede the copy that refills it
            fence_proxy_async_smem();
            __syncwarp();
            if (j + kSt < nj && elect_one()) issue(st, c0 + warp + kWarps * (j + kSt));
        }
        // partial sums of the warps -> shared memory, reduced in warp order
        if constexpr (kMma) {
            constexpr int SU = CB / 64;
            const int r = lane >> 2, tg = lane & 3;
#pragma unroll
            for (int i = 0; i < MT * COLS; ++i) {
                const int e = i & 3, j = (i >> 2) & 3, u = (i >> 4) % SU, nt = (i >> 4) / SU;
                const int m = 8 * nt + 2 * tg + (e & 1), col = 64 * u + (e >> 1) * 32 + 4 * r + j;
                red[warp * E + m * CB + col] = (&yacc[0][0])[i];
            }
        } else {
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int j = 0; j < COLS; ++j) red[warp * E + m * CB + St::col(lane, j / W, j % W)] = yacc[m][j];
        }
        __syncthreads();
        const int EM = M * CB;                       // live entries: rows m < M
        for (int e = threadIdx.x; e < EM; e += kThreads) {
            float sum = red[e];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) sum += red[w * E + e];
            red[e] = sum;
        }

        auto store_y = [&](int e, float v) {
            const int m = e / CB, n = cb * CB + (e - m * CB);
            if (n < N) a.y[static_cast<size_t>(m) * N + n] = A::from_float(v);
        };

        if (c0 == 0 && c1 == chunks) {
            // this CTA owns the whole column block
            for (int e = threadIdx.x; e < EM; e += kThreads) store_y(e, red[e]);
        } else if (a.cluster > 1) {
            // The block's CTAs form this cluster, in K order by rank. Once every
            // CTA's partial is in its red[], rank 0 sums them in rank order (the
            // ticket path's order, so both give the same bits) through
            // distributed shared memory; the second barrier keeps the others'
            // shared memory alive until it has read it.
            cluster_sync();
            if (cluster_ctarank() == 0) {
                const int nc = a.cluster;
                for (int e = threadIdx.x; e < EM; e += kThreads) {
                    const uint32_t addr = smem_u32(red + e);
                    float v[8];
#pragma unroll
                    for (int r = 1; r < 8; ++r) v[r] = r < nc ? ld_cluster_f32(addr, r) : 0.f;
                    float sum = red[e];
#pragma unroll
                    for (int r = 1; r < 8; ++r)
                        if (r < nc) sum += v[r];
                    store_y(e, sum);
                }
            }
            cluster_sync();
        } else {
            const int slot = c0 > 0 ? 0 : 1;
            float* part = a.partials + (static_cast<size_t>(b) * 2 + slot) * EM;
            for (int e = threadIdx.x; e < EM; e += kThreads) part[e] = red[e];
            __syncthreads();
            const long long first = static_cast<long long>(cb) * chunks, last = first + chunks - 1;
            const int b_lo = owner_cta(first, T, Gd), b_hi = owner_cta(last, T, Gd);
            // One acquire-release increment publishes every thread's partial (the
            // CTA barrier above orders them before it) and, for the last
            // contributor, makes the others' partials visible to the loads below.
            if (threadIdx.x == 0) {
                unsigned old;
                asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.tickets + cb) : "memory");
                s_last = (old == static_cast<unsigned>(b_hi - b_lo));
            }
            __syncthreads();
            if (s_last) {
                // Contributor b_lo covers the block's first chunks, so its segment
                // starts at chunk 0 and it wrote slot 1; every later contributor
                // starts inside the block and wrote slot 0 (no CTA has an empty
                // range). Sums run in ascending CTA order, 8 loads in flight.
                for (int e = threadIdx.x; e < EM; e += kThreads) {
                    float sum = __ldcg(a.partials + (static_cast<size_t>(b_lo) * 2 + 1) * EM + e);
                    for (int b0 = b_lo + 1; b0 <= b_hi; b0 += 8) {
                        float v[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            v[u] = b0 + u <= b_hi ? __ldcg(a.partials + static_cast<size_t>(b0 + u) * 2 * EM + e) : 0.f;
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            if (b0 + u <= b_hi) sum += v[u];
                    }
                    store_y(e, sum);
                }
                if (threadIdx.x == 0) a.tickets[cb] = 0u;
            }
        }
        __syncthreads();   // red[] is reused by the next segment
        it += c1 - c0;
    }
    // only after a timeout: wait (bounded) for this warp's copies still in
    // flight, so none lands in shared memory after the CTA has exited
    if (lane == 0) {
        for (int j = drain_lo; j < drain_hi; ++j) {
            const int st = j % kSt;
            const uint32_t par = (phase_bits >> st) & 1u;
            const unsigned long long t0 = clock64();
            while (!mbar_try_wait(bars + 8 * st, par) && clock64() - t0 < kWaitLimitCycles) {
            }
            phase_bits ^= 1u << st;
        }
    }
}

// Whether `clusters` clusters of this launch can all be resident at once
// (asked once per kernel, cluster size and shared-memory size).
bool clusters_fit(const void* kern, const cudaLaunchConfig_t& cfg, int clusters) {
    static std::mutex mu;
    static std::map<std::tuple<const void*, unsigned, size_t>, int> cache;
    const auto key = std::make_tuple(kern, cfg.attrs[cfg.numAttrs - 1].val.clusterDim.x, cfg.dynamicSmemBytes);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it == cache.end()) {
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            active = 0;
        }
        it = cache.emplace(key, active).first;
    }
    return it->second >= clusters;
}

template <bool kBf16, int MT, int COLS, bool kSym, bool kFact, bool kZBulk, bool kMx = false, bool kXPre = false,
          bool kMma = false>
cudaError_t launch_one(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
    static_assert(Stage<COLS, MT>::kBytes == stage_bytes(COLS, MT), "stage layout");
    auto kern = gemv_kernel<kBf16, MT, COLS, kSym, kFact, kZBulk, kMx, kXPre, kMma>;
    const size_t smem = p.smem_bytes;
    if (smem > 48 * 1024) {
        if (cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), p.device, smem); e != cudaSuccess)
            return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (W4A16_GEMV_PDL) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    GemvArgs args = a;
    if (a.cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(a.cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = n + 1;
        // clusters only when all of them are resident at once; else tickets
        if (!clusters_fit(reinterpret_cast<const void*>(kern), cfg, p.grid / a.cluster)) args.cluster = 0;
        else ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

template <bool kBf16, int MT, int COLS, bool kFact, bool kXPre = false, bool kMma = false>
cudaError_t launch_sym(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
    const bool zb = (a.N % 32) == 0;
    if (!a.qz) return launch_one<kBf16, MT, COLS, true, kFact, false, false, kXPre, kMma>(a, p, s);
    return zb ? launch_one<kBf16, MT, COLS, false, kFact, true, false, kXPre, kMma>(a, p, s)
              : launch_one<kBf16, MT, COLS, false, kFact, false, false, kXPre, kMma>(a, p, s);
}

template <bool kBf16>
cudaError_t launch_dtype(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
    if (p.mma) {
        switch (p.mt) {
            case 8:
                return p.cols == 2 ? launch_sym<kBf16, 8, 2, false, false, true>(a, p, s)
                                   : launch_sym<kBf16, 8, 4, false, false, true>(a, p, s);
            case 16: return launch_sym<kBf16, 16, 2, false, false, true>(a, p, s);
            default: return cudaErrorInvalidValue;
        }
    }
    if (p.fact && p.xpre) {
        switch (p.mt) {
            case 1:
                return p.cols == 9 ? launch_sym<kBf16, 1, 9, true, true>(a, p, s)
                                   : launch_sym<kBf16, 1, 8, true, true>(a, p, s);
            case 2: return launch_sym<kBf16, 2, 4, true, true>(a, p, s);
            case 3: return launch_sym<kBf16, 3, 4, true, true>(a, p, s);
            case 4: return launch_sym<kBf16, 4, 4, true, true>(a, p, s);
            default: break;
        }
    }
    if (p.fact) {
        switch (p.mt) {
            case 1:
                return p.cols == 9 ? launch_sym<kBf16, 1, 9, true>(a, p, s) : launch_sym<kBf16, 1, 8, true>(a, p, s);
            case 2: return launch_sym<kBf16, 2, 4, true>(a, p, s);
            case 3: return launch_sym<kBf16, 3, 4, true>(a, p, s);
            case 4: return launch_sym<kBf16, 4, 4, true>(a, p, s);
            default: break;
        }
    }
    switch (p.mt) {
        case 1: return launch_sym<kBf16, 1, 8, false>(a, p, s);
        case 2: return launch_sym<kBf16, 2, 4, false>(a, p, s);
        case 3: return launch_sym<kBf16, 3, 4, false>(a, p, s);
        case 4: return launch_sym<kBf16, 4, 4, false>(a, p, s);
        case 6: return launch_sym<kBf16, 6, 2, false>(a, p, s);
        case 8: return launch_sym<kBf16, 8, 2, false>(a, p, s);
        case 12: return launch_sym<kBf16, 12, 1, false>(a, p, s);
        case 16: return launch_sym<kBf16, 16, 1, false>(a, p, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_mx_rows(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
    if (p.mma) {
        switch (p.mt) {
            case 8:
                return p.cols == 2 ? launch_one<true, 8, 2, true, false, false, true, false, true>(a, p, s)
                                   : launch_one<true, 8, 4, true, false, false, true, false, true>(a, p, s);
            case 16: return launch_one<true, 16, 2, true, false, false, true, false, true>(a, p, s);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (p.mt) {
        case 1:
            return p.cols == 9 ? launch_one<true, 1, 9, true, false, false, true>(a, p, s)
                               : launch_one<true, 1, 8, true, false, false, true>(a, p, s);
        case 2: return launch_one<true, 2, 4, true, false, false, true>(a, p, s);
        case 3: return launch_one<true, 3, 4, true, false, false, true>(a, p, s);
        case 4: return launch_one<true, 4, 4, true, false, false, true>(a, p, s);
        case 6: return launch_one<true, 6, 2, true, false, false, true>(a, p, s);
        case 8: return launch_one<true, 8, 2, true, false, false, true>(a, p, s);
        case 12: return launch_one<true, 12, 1, true, false, false, true>(a, p, s);
        case 16: return launch_one<true, 16, 1, true, false, false, true>(a, p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

constexpr int kMaxLive = 1024;        // max over row templates of M * columns per block
// Chunks per warp that crossing a column block boundary costs a CTA (fitted to
// timings: 2 x 16384 x 5376 says more than 1.7, 3 x 5376 x 21504 less than 2.4).
constexpr double kStraddleCost = 2.0;
// Fewest chunks a CTA is given (of kWarps = 16 streaming warps). Measured
// against 16, 4 and 2 (us): 4x2048x2048 6.00 / 5.23 / 5.30 / 5.30 at 16 / 8 /
// 4 / 2, 1x2048x2048 5.11 / 4.50 / 5.08 / 5.38, 4x1024x4096 6.17 / 5.91 /
// 6.44 / 6.44.
constexpr int kMinChunksPerCta = 8;
// Largest cluster (portable size) whose CTAs sum a column block through
// distributed shared memory instead of workspace slots and a ticket.
#ifndef W4A16_GEMV_MAX_CLUSTER
#define W4A16_GEMV_MAX_CLUSTER 8
#endif
constexpr int kMaxCluster = W4A16_GEMV_MAX_CLUSTER;

// two partial slots (head and tail segment) per CTA, at most one CTA per SM
size_t partial_region_bytes(const DeviceProps& dp) {
    return static_cast<size_t>(dp.sms) * 2 * kMaxLive * sizeof(float);
}

namespace {

// Never launched: a stand-in for the GEMV kernels (512 threads, one CTA per
// SM) in the occupancy query below.
__global__ void __launch_bounds__(kThreads, 1) cluster_probe_kernel() {}

// How many clusters of `size` CTAs (one CTA per SM) the device holds at once;
// asked once per device. It depends on how the SMs are grouped (a cluster
// lives in one GPC): on a 152-SM GB300, 76 of 2, 46 of 3, 36 of 4, 23 of 6,
// 15 of 7 or 8.
int cluster_capacity(const DeviceProps& dp, int size) {
    static std::mutex mu;
    static std::map<int, std::array<int, kMaxCluster + 1>> cache;
    if (size < 1 || size > kMaxCluster) return 0;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dp.device);
    if (it == cache.end()) {
        std::array<int, kMaxCluster + 1> cap{};
        const void* k = reinterpret_cast<const void*>(cluster_probe_kernel);
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dp.smem_optin)) ==
            cudaSuccess) {
            for (int c = 1; c <= kMaxCluster; ++c) {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(c);
                cfg.blockDim = dim3(kThreads);
                cfg.dynamicSmemBytes = dp.smem_optin;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = static_cast<unsigned>(c);
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                int n = 0;
                if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) n = 0;
                cap[c] = n;
            }
        }
        (void)cudaGetLastError();
        it = cache.emplace(dp.device, cap).first;
    }
    return it->second[size];
}

// `fact`: whether the kernel may apply zero-points through chunk sums of x
// (the W4A16 layer for M <= 4; never for MXFP4 weights, which have none).
// `narrow`: the 8-row MMA template with 64-column blocks instead of 128.
GemvPlan plan_cols(int M, int N, int K, bool fact, const DeviceProps& dp, bool narrow) {
    GemvPlan p;
    // `fact` marks the int4 layer; MXFP4 weights take the same conversion choice
    p.mma = M >= kMmaMinM && (M > kFmaSmallMaxM || static_cast<long long>(N) * K > kFmaSmallMaxWeights);
    if (p.mma) {
        p.mt = M <= 8 ? 8 : 16;
        p.cols = M <= 8 && !narrow ? 4 : 2;
    } else {
        p.mt = M <= 1 ? 1 : M <= 2 ? 2 : M <= 3 ? 3 : M <= 4 ? 4 : M <= 6 ? 6 : M <= 8 ? 8 : M <= 12 ? 12 : 16;
        p.cols = p.mt == 1 ? 8 : p.mt <= 4 ? 4 : p.mt <= 8 ? 2 : 1;
        // One row: when 256-column blocks outnumber the SMs but 288-column
        // blocks do not (43008 columns: 168 against 150 blocks on 152 SMs),
        // 9 columns a lane let every CTA own one whole block: no split-K fix-up
        // and no block boundary inside a CTA's range.
        if (p.mt == 1 && (N + 255) / 256 > dp.sms && (N + 287) / 288 <= dp.sms) p.cols = 9;
    }
    p.cb = 32 * p.cols;
    p.box_cols = box_cols(p.cols);
    p.n_cb = (N + p.cb - 1) / p.cb;
    p.warps = kWarps;
    const int chunks = K / kChunk;
    const long long items = static_cast<long long>(p.n_cb) * chunks;
    p.items = items;
    p.fact = fact && M <= kFactMaxM && !p.mma;
    const int live = p.mt * p.cb;
    auto size_grid = [&](int xsum_entries) {
        const int stages = ring_stages(p.mma, p.mt);
        p.smem_bytes = ring_offset(live, xsum_entries, stages) + 128 +
                       static_cast<size_t>(kWarps) * stages * stage_bytes(p.cols, p.mt);
        // One CTA per SM: every row template needs more than 64 registers a
        // thread, so two 512-thread CTAs never fit on one SM together, and a
        // larger grid runs as a second, partial wave. At least
        // kMinChunksPerCta chunks per CTA: on a small layer, half the warps of
        // a CTA busy on twice as many SMs beat every warp busy on half of them
        // (the conversion of a chunk is issue-bound on the SM's schedulers).
        const long long want = dp.sms;
        p.grid = static_cast<int>(std::max<long long>(1, std::min<long long>(want, items / kMinChunksPerCta)));
        // A CTA whose range crosses a column block boundary runs the two
        // segments one after the other (second pipeline fill, second reduction
        // and fix-up): about kStraddleCost chunks per warp, measured. A grid of
        // `sp` CTAs per column block never crosses one; take it when its chunks
        // per warp are fewer than the stream-K grid's plus that cost.
        const long long sp = std::min<long long>(want / p.n_cb, chunks / kMinChunksPerCta);
        if (sp >= 1 && p.n_cb * sp != p.grid) {
            const long long aligned = p.n_cb * sp;
            // compare items / (grid * kWarps) + kStraddleCost with items / (aligned * kWarps)
            const double cost_sk = static_cast<double>(items) / (static_cast<double>(p.grid) * kWarps) + kStraddleCost;
            const double cost_al = static_cast<double>(items) / (static_cast<double>(aligned) * kWarps);
            if (cost_al < cost_sk) p.grid = static_cast<int>(aligned);
        }
        // A block-aligned grid of 2..8 CTAs per block sums each block in a
        // cluster, if all its clusters can be resident at once. On a small
        // layer (at most two chunks per warp) a grid of clusters that fit is
        // taken even with fewer CTAs per block, down to half the grid: the
        // cluster sum saves about 0.7 us (4x2048x2048: 5.23 -> 4.95 us with 96
        // CTAs in clusters of 6 against 128 CTAs with tickets; 1x5376x21504
        // with ~100 chunks a CTA: 14.56 -> 15.09 us with 126 CTAs, so not there).
        p.cluster = 0;
        if (sp >= 2 && sp <= kMaxCluster && p.grid == p.n_cb * sp && p.n_cb <= cluster_capacity(dp, sp))
            p.cluster = static_cast<int>(sp);
        if (!p.cluster) {
            long long sc = std::min<long long>(std::min<long long>(want / p.n_cb, chunks / kMinChunksPerCta),
                                               kMaxCluster);
            while (sc >= 2 && p.n_cb > cluster_capacity(dp, static_cast<int>(sc))) --sc;
            const long long gc = p.n_cb * sc;
            if (sc >= 2 && 2 * gc >= p.grid && items <= gc * 2 * kWarps) {
                p.grid = static_cast<int>(gc);
                p.cluster = static_cast<int>(sc);
            }
        }
    };
    size_grid(0);
    // Precomputed chunk sums: a prologue over all chunks, against a warp
    // reduction per chunk. Measured at N = 43008, K = 5376 (12 chunks per warp)
    // the prologue wins by 0.3 us; at 4-6 chunks per warp and below the
    // per-chunk reduction wins by 3-11 %.
    const size_t xsum_bytes = static_cast<size_t>(M) * chunks * sizeof(float2);
    p.xpre = p.fact && items >= static_cast<long long>(kXPreMinChunksPerWarp) * kWarps * p.grid &&
             xsum_bytes <= kXsumSmemLimit;
    if (p.xpre) size_grid(M * chunks);
    p.ticket_bytes = (static_cast<size_t>(p.n_cb) * sizeof(uint32_t) + 255) & ~size_t(255);
    // Partial slots first, in a region whose size depends only on the device
    // (M * columns-per-block <= kMaxLive for every row template), tickets after
    // it: calls of different shapes sharing one workspace never write partial
    // sums over one another's tickets.
    p.partial_bytes = partial_region_bytes(dp);
    p.device = dp.device;
    return p;
}

// The 8-row MMA template takes 64-column blocks when they give a
// block-aligned grid (whole blocks or a whole number of CTAs per block), else
// 128-column blocks. Narrow blocks double the blocks, so more warps of more
// CTAs get chunks (aligned, us, 64 vs 128 columns: 4x2048x2048 4.37 / 5.12,
// 4x6144x2048 5.75 / 6.72, 8x2048x8192 6.92 / 8.64, 8x8192x4096 8.23 / 9.79);
// a stream-K grid of narrow blocks loses (3x5376x5376 11.5 / 8.9, 4x14336x2048
// 12.8 / 8.1), and more narrow blocks than SMs never align.
GemvPlan plan(int M, int N, int K, bool fact, const DeviceProps& dp) {
    GemvPlan p = plan_cols(M, N, K, fact, dp, true);
    if (p.mma && p.mt == 8 && p.grid % p.n_cb != 0) p = plan_cols(M, N, K, fact, dp, false);
    return p;
}

}  // namespace

GemvPlan plan_gemv(int M, int N, int K, int g, const DeviceProps& dp) {
    (void)g;
    return plan(M, N, K, true, dp);
}

size_t gemv_workspace_bytes(const GemvPlan& p) { return p.ticket_bytes + p.partial_bytes; }

GemvPlan plan_mx_gemv(int M, int N, int K, const DeviceProps& dp) { return plan(M, N, K, false, dp); }

cudaError_t launch_gemv(const void* x, const uint32_t* qw, const void* sc, const uint32_t* qz, void* y, int M,
                        int N, int K, int g, bool bf16, const GemvPlan& plan, float* partials, uint32_t* tickets,
                        cudaStream_t s) {
    GemvArgs a;
    const CUtensorMapDataType act = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const uint32_t cb = static_cast<uint32_t>(plan.cb);
    const uint32_t box = static_cast<uint32_t>(plan.box_cols);   // cb, or one lane group's columns
    if (!encode_2d(&a.tq, CU_TENSOR_MAP_DATA_TYPE_INT32, qw, (uint64_t)N, (uint64_t)(K / 8), (uint64_t)N * 4, box,
                   kRowsPerChunk, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&a.ts, act, sc, (uint64_t)N, (uint64_t)(K / g), (uint64_t)N * 2, box, 1,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&a.tx, act, x, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, kChunk, plan.mt,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    if (qz && N % 32 == 0) {
        if (!encode_2d(&a.tz, CU_TENSOR_MAP_DATA_TYPE_INT32, qz, (uint64_t)(N / 8), (uint64_t)(K / g),
                       (uint64_t)(N / 8) * 4, cb / 8, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        memset(&a.tz, 0, sizeof(a.tz));
    }
    a.x = static_cast<const uint16_t*>(x);
    a.qz = qz;
    a.y = static_cast<uint16_t*>(y);
    a.partials = partials;
    a.tickets = tickets;
    a.M = M;
    a.N = N;
    a.K = K;
    a.g_shift = __builtin_ctz(static_cast<unsigned>(g));
    a.chunks = K / kChunk;
    a.items = plan.items;
    a.cluster = plan.cluster;
    return bf16 ? launch_dtype<true>(a, plan, s) : launch_dtype<false>(a, plan, s);
}

cudaError_t launch_mx_gemv(const void* x, const uint32_t* qw, const uint8_t* es, void* y, int M, int N, int K,
                           const GemvPlan& plan, float* partials, uint32_t* tickets, cudaStream_t s) {
    if (plan.fact) return cudaErrorInvalidValue;   // the plan must come from plan_mx_gemv
    GemvArgs a;
    const uint32_t box = static_cast<uint32_t>(plan.box_cols);   // cb, or one lane group's columns
    if (!encode_2d(&a.tq, CU_TENSOR_MAP_DATA_TYPE_INT32, qw, (uint64_t)N, (uint64_t)(K / 8), (uint64_t)N * 4, box,
                   kRowsPerChunk, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&a.ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, es, (uint64_t)N, (uint64_t)(K / mx::kBlock), (uint64_t)N,
                   box, 1, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&a.tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, kChunk,
                   plan.mt, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    memset(&a.tz, 0, sizeof(a.tz));
    a.x = static_cast<const uint16_t*>(x);
    a.qz = nullptr;
    a.y = static_cast<uint16_t*>(y);
    a.partials = partials;
    a.tickets = tickets;
    a.M = M;
    a.N = N;
    a.K = K;
    a.g_shift = __builtin_ctz(static_cast<unsigned>(mx::kBlock));
    a.chunks = K / kChunk;
    a.items = plan.items;
    a.cluster = plan.cluster;
    return launch_mx_rows(a, plan, s);
}

// ---------------------------------------------------------------------------
// Built-in scratch for callers that cannot allocate device memory
// ---------------------------------------------------------------------------
// The GEMV's scratch (partial sums of column blocks shared by several CTAs,
// then one ticket word per column block) normally comes from the caller's
// workspace. This fixed array serves w4a16_gemv_noalloc instead. It is zero
// when the module loads; every GEMV call leaves its ticket words at zero, and
// w4a16_gemv_noalloc clears them before each launch as well.
static __device__ __align__(256) uint8_t g_gemv_noalloc_scratch[kGemvNoAllocScratchBytes];

cudaError_t gemv_noalloc_scratch(int device, bool may_look_up, void** ptr) {
    static std::mutex mu;
    static void* cache[64] = {nullptr};
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[device]) {
        if (!may_look_up) return cudaErrorStreamCaptureUnsupported;
        // host code may not use the array's name as an address: ask the runtime,
        // with `device` current (the caller's current device)
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_gemv_noalloc_scratch);
        if (e != cudaSuccess) return e;
        cache[device] = p;
    }
    *ptr = cache[device];
    return cudaSuccess;
}

// ---------------------------------------------------------------------------
// Self-test of the bounded wait
// ---------------------------------------------------------------------------
namespace {
// One warp waits, with the kernels' own bounded wait, on an mbarrier that
// nothing will complete: after about two seconds the wait gives up, records
// W4A16_ERR_TIMEOUT in the GEMV error word and the kernel returns normally.
__global__ void wait_selftest_kernel() {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
    }
    __syncwarp();
    (void)warp_wait(b, 0, lane);
}
}  // namespace

cudaError_t launch_wait_selftest(cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>();
    return cudaGetLastError();
}

cudaError_t read_and_clear_gemv_error(uint32_t* out) {
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(zero));
    }
    *out = v;
    return e;
}

}  // namespace w4a16
