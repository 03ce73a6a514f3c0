// Decode GEMV of the W4A16 layer, 1 <= M <= 16, on CUDA cores.
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
//     block first. A persistent grid of exactly two CTAs per SM takes equal
//     contiguous ranges of items ("stream-K"), so every SM streams the same
//     number of bytes whatever N and K are.
//   * Inside a CTA the 8 warps take the chunks of the current column block in
//     turn. A lane owns COLS adjacent columns and loads, per chunk, 4 rows x
//     COLS packed words with 128-bit non-allocating loads plus its scales and
//     zero-point word; the next chunk's loads are issued before the current
//     chunk is converted (register double buffer), so memory and ALU overlap.
//   * Nibbles become 16-bit floats by the exponent-bias trick: OR a nibble into
//     the mantissa of 1024.0 (fp16) or 128.0 (bf16). For M <= 4 the zero-point
//     is applied once per chunk through
//         sum_k (q - z) x = sum_k (magic + q) x - (magic + z) sum_k x,
//     with sum_k x of every chunk precomputed in shared memory; the products
//     (magic + q) * x are exact in an FP32 FMA with 16-bit inputs
//     (fma.rn.f32.f16 / .bf16). For M > 4 the zero-point is subtracted from
//     each nibble pair in packed 16-bit arithmetic (exact) before the FMA. The
//     scale is applied in FP32 once per chunk.
//   * Column blocks split between CTAs are finished by the last CTA to arrive
//     (an atomic ticket per column block): it sums the partial vectors of all
//     contributing CTAs in ascending CTA order, so the result is deterministic,
//     and resets the ticket to zero for the next call.
#include "internal.h"
#include "ptx.cuh"

#include <algorithm>

namespace w4a16 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kChunk = 32;            // rows of K per chunk
constexpr int kRowsPerChunk = 4;      // packed word rows per chunk
constexpr int kFactMaxM = 4;          // zero-point by chunk sums up to this M
constexpr size_t kXsumSmemLimit = 32 * 1024;

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

__device__ __forceinline__ uint4 ld_stream_v4(const uint32_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream_v2(const uint32_t* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_stream_v1(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

template <int COLS>
__device__ __forceinline__ void load_words(const uint32_t* p, uint32_t (&v)[COLS]) {
    if constexpr (COLS == 8) {
        const uint4 a = ld_stream_v4(p), b = ld_stream_v4(p + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else if constexpr (COLS == 4) {
        const uint4 a = ld_stream_v4(p);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else if constexpr (COLS == 2) {
        const uint2 a = ld_stream_v2(p);
        v[0] = a.x; v[1] = a.y;
    } else {
        v[0] = ld_stream_v1(p);
    }
}

// COLS 16-bit scales packed two per word (SW words; the last half unused when COLS == 1).
template <int COLS>
struct ScaleWords {
    static constexpr int SW = (COLS + 1) / 2;
};
template <int COLS>
__device__ __forceinline__ void load_scales(const uint16_t* p, uint32_t (&v)[ScaleWords<COLS>::SW]) {
    if constexpr (COLS == 8) {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else if constexpr (COLS == 4) {
        const uint2 a = __ldg(reinterpret_cast<const uint2*>(p));
        v[0] = a.x; v[1] = a.y;
    } else if constexpr (COLS == 2) {
        v[0] = __ldg(reinterpret_cast<const uint32_t*>(p));
    } else {
        v[0] = __ldg(p);
    }
}

template <int COLS>
struct ChunkRegs {
    uint32_t q[kRowsPerChunk][COLS];
    uint32_t s[ScaleWords<COLS>::SW];
    uint32_t z;
};

struct GemvArgs {
    const uint16_t* x;
    const uint32_t* qw;
    const uint16_t* sc;
    const uint32_t* qz;
    uint16_t* y;
    uint32_t* tickets;    // [n_cb], zero between calls
    float* partials;      // [grid][2][M * CB], at most kMaxLive floats per slot
    int M, N, K, g;
    int chunks;
    long long items;      // n_cb * chunks
};

// First CTA whose item range contains item i (ranges are [b*T/G, (b+1)*T/G)).
__device__ __forceinline__ int owner_cta(long long i, long long T, int G) {
    return static_cast<int>(((i + 1) * G - 1) / T);
}
__device__ __forceinline__ long long range_start(int b, long long T, int G) { return (long long)b * T / G; }

template <bool kBf16, int MT, int COLS, bool kSym, bool kFact>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const GemvArgs a) {
    using A = Act<kBf16>;
    constexpr int CB = 32 * COLS;
    constexpr int E = MT * CB;
    constexpr bool kTwoFamilies = kFact && !kBf16;   // fp16: nibbles at bits 0-3 and 4-7 of a half
    extern __shared__ float smem[];
    float* red = smem;                          // [kWarps][E]
    float2* xsum = reinterpret_cast<float2*>(smem + kWarps * E);   // [M][chunks]: (offset, sum x)
    __shared__ int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = a.M, N = a.N, K = a.K, g = a.g, chunks = a.chunks;
    const long long T = a.items;
    const int G = gridDim.x, b = blockIdx.x;
    const long long i_begin = range_start(b, T, G), i_end = range_start(b + 1, T, G);

    if constexpr (kFact) {
        // per (row, chunk): sum of x over the chunk, and the offset the magic bias adds
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
        __syncthreads();
    }

    for (long long it = i_begin; it < i_end;) {
        const int cb = static_cast<int>(it / chunks);
        const int c0 = static_cast<int>(it - static_cast<long long>(cb) * chunks);
        const int c1 = static_cast<int>(std::min<long long>(chunks, c0 + (i_end - it)));
        const int n0 = cb * CB + lane * COLS;
        const bool col_ok = n0 < N;               // N % 8 == 0 and COLS | 8: all COLS columns valid
        const int zshift = 4 * (n0 & 7);

        float yacc[MT][COLS];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int j = 0; j < COLS; ++j) yacc[m][j] = 0.f;

        auto load = [&](ChunkRegs<COLS>& r, int c) {
            const uint32_t* p = a.qw + static_cast<size_t>(c) * kRowsPerChunk * N + n0;
#pragma unroll
            for (int i = 0; i < kRowsPerChunk; ++i) load_words<COLS>(p + static_cast<size_t>(i) * N, r.q[i]);
            const int t = (c * kChunk) / g;
            load_scales<COLS>(a.sc + static_cast<size_t>(t) * N + n0, r.s);
            if constexpr (!kSym) r.z = __ldg(a.qz + static_cast<size_t>(t) * (N >> 3) + (n0 >> 3));
        };

        auto compute = [&](const ChunkRegs<COLS>& r, int c) {
            float acc[MT][COLS], acc2[kTwoFamilies ? MT : 1][kTwoFamilies ? COLS : 1];
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int j = 0; j < COLS; ++j) acc[m][j] = 0.f;
            if constexpr (kTwoFamilies) {
#pragma unroll
                for (int m = 0; m < MT; ++m)
#pragma unroll
                    for (int j = 0; j < COLS; ++j) acc2[m][j] = 0.f;
            }
            uint32_t zz[COLS];
            if constexpr (!kFact) {
#pragma unroll
                for (int j = 0; j < COLS; ++j) {
                    const uint32_t z = kSym ? 8u : ((r.z >> (zshift + 4 * j)) & 0xFu);
                    zz[j] = A::kMagic | z | (z << 16);
                }
            }
#pragma unroll
            for (int i = 0; i < kRowsPerChunk; ++i) {
                // nibble pairs of this word row for every column, converted once ...
                uint32_t h[COLS][4];
#pragma unroll
                for (int j = 0; j < COLS; ++j) {
                    const uint32_t w = r.q[i][j];
                    if constexpr (kTwoFamilies) {
                        // (1024 + q[k], 1024 + q[k+4]), (1024 + 16 q[k+1], 1024 + 16 q[k+5]),
                        // (1024 + q[k+2], 1024 + q[k+6]), (1024 + 16 q[k+3], 1024 + 16 q[k+7])
                        const uint32_t w8 = w >> 8;
                        h[j][0] = and_or(w, 0x000F000Fu, A::kMagic);
                        h[j][1] = and_or(w, 0x00F000F0u, A::kMagic);
                        h[j][2] = and_or(w8, 0x000F000Fu, A::kMagic);
                        h[j][3] = and_or(w8, 0x00F000F0u, A::kMagic);
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
                const int k = c * kChunk + i * 8;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint4 xv = (m < M) ? __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(m) * K + k))
                                             : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int j = 0; j < COLS; ++j) {
                        if constexpr (kTwoFamilies) {
                            acc[m][j] = fma_mixed<false, 0, 0>(h[j][0], xv.x, acc[m][j]);
                            acc[m][j] = fma_mixed<false, 1, 0>(h[j][0], xv.z, acc[m][j]);
                            acc[m][j] = fma_mixed<false, 0, 0>(h[j][2], xv.y, acc[m][j]);
                            acc[m][j] = fma_mixed<false, 1, 0>(h[j][2], xv.w, acc[m][j]);
                            acc2[m][j] = fma_mixed<false, 0, 1>(h[j][1], xv.x, acc2[m][j]);
                            acc2[m][j] = fma_mixed<false, 1, 1>(h[j][1], xv.z, acc2[m][j]);
                            acc2[m][j] = fma_mixed<false, 0, 1>(h[j][3], xv.y, acc2[m][j]);
                            acc2[m][j] = fma_mixed<false, 1, 1>(h[j][3], xv.w, acc2[m][j]);
                        } else {
                            // pair bb holds x[k+bb] (word bb/2 of x, half bb&1) and x[k+bb+4]
                            acc[m][j] = fma_mixed<kBf16, 0, 0>(h[j][0], xv.x, acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 1, 0>(h[j][0], xv.z, acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 0, 1>(h[j][1], xv.x, acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 1, 1>(h[j][1], xv.z, acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 0, 0>(h[j][2], xv.y, acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 1, 0>(h[j][2], xv.w, acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 0, 1>(h[j][3], xv.y, acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 1, 1>(h[j][3], xv.w, acc[m][j]);
                        }
                    }
                }
            }
            // scale (and, for kFact, zero-point) once per chunk, in FP32
#pragma unroll
            for (int j = 0; j < COLS; ++j) {
                const float s = A::to_float(static_cast<uint16_t>(r.s[j / 2] >> (16 * (j & 1))));
                if constexpr (kFact) {
                    const float zf = kSym ? 8.f : static_cast<float>((r.z >> (zshift + 4 * j)) & 0xFu);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const float2 os = (m < M) ? xsum[m * chunks + c] : make_float2(0.f, 0.f);
                        float t = acc[m][j];
                        if constexpr (kTwoFamilies) t = fmaf(acc2[m][j], 0.0625f, t);
                        yacc[m][j] = fmaf(s, t - fmaf(zf, os.y, os.x), yacc[m][j]);
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < MT; ++m) yacc[m][j] = fmaf(s, acc[m][j], yacc[m][j]);
                }
            }
        };

        if (col_ok) {
            ChunkRegs<COLS> b0, b1;
            int c = c0 + warp;
            if (c < c1) load(b0, c);
            for (; c < c1; c += 2 * kWarps) {
                const int cn = c + kWarps;
                if (cn < c1) load(b1, cn);
                compute(b0, c);
                const int cnn = cn + kWarps;
                if (cnn < c1) load(b0, cnn);
                if (cn < c1) compute(b1, cn);
            }
        }

        // partial sums of the 8 warps -> shared memory, reduced in warp order
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int j = 0; j < COLS; ++j) red[warp * E + m * CB + lane * COLS + j] = yacc[m][j];
        __syncthreads();
        const int EM = M * CB;                       // live entries: rows m < M
        for (int e = threadIdx.x; e < EM; e += kThreads) {
            float s = red[e];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) s += red[w * E + e];
            red[e] = s;
        }

        auto store_y = [&](int e, float v) {
            const int m = e / CB, n = cb * CB + (e - m * CB);
            if (n < N) a.y[static_cast<size_t>(m) * N + n] = A::from_float(v);
        };

        if (c0 == 0 && c1 == chunks) {
            // this CTA owns the whole column block
            for (int e = threadIdx.x; e < EM; e += kThreads) store_y(e, red[e]);
        } else {
            const int slot = c0 > 0 ? 0 : 1;
            float* part = a.partials + (static_cast<size_t>(b) * 2 + slot) * EM;
            for (int e = threadIdx.x; e < EM; e += kThreads) part[e] = red[e];
            __threadfence();
            __syncthreads();
            const long long first = static_cast<long long>(cb) * chunks, last = first + chunks - 1;
            const int b_lo = owner_cta(first, T, G), b_hi = owner_cta(last, T, G);
            if (threadIdx.x == 0) {
                const unsigned old = atomicAdd(a.tickets + cb, 1u);
                s_last = (old == static_cast<unsigned>(b_hi - b_lo));
            }
            __syncthreads();
            if (s_last) {
                __threadfence();
                for (int e = threadIdx.x; e < EM; e += kThreads) {
                    float s = 0.f;
                    for (int bb = b_lo; bb <= b_hi; ++bb) {
                        const long long st = std::max(range_start(bb, T, G), first);
                        const int sl = (st > first) ? 0 : 1;
                        s += __ldcg(a.partials + (static_cast<size_t>(bb) * 2 + sl) * EM + e);
                    }
                    store_y(e, s);
                }
                if (threadIdx.x == 0) a.tickets[cb] = 0u;
            }
        }
        __syncthreads();   // red[] is reused by the next segment
        it += c1 - c0;
    }
}

template <bool kBf16, int MT, int COLS, bool kSym, bool kFact>
cudaError_t launch_one(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
    auto kern = gemv_kernel<kBf16, MT, COLS, kSym, kFact>;
    const size_t smem = p.smem_bytes;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kern<<<p.grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <bool kBf16, int MT, int COLS, bool kFact>
cudaError_t launch_sym(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
    return a.qz ? launch_one<kBf16, MT, COLS, false, kFact>(a, p, s) : launch_one<kBf16, MT, COLS, true, kFact>(a, p, s);
}

template <bool kBf16>
cudaError_t launch_dtype(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
    if (p.fact) {
        switch (p.mt) {
            case 1: return launch_sym<kBf16, 1, 8, true>(a, p, s);
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

}  // namespace

constexpr int kMaxLive = 512;         // max over row templates of M * columns per block

size_t partial_region_bytes(const DeviceProps& dp) {
    return static_cast<size_t>(2) * dp.sms * 2 * kMaxLive * sizeof(float);
}

GemvPlan plan_gemv(int M, int N, int K, int g, const DeviceProps& dp) {
    (void)g;
    GemvPlan p;
    p.mt = M <= 1 ? 1 : M <= 2 ? 2 : M <= 3 ? 3 : M <= 4 ? 4 : M <= 6 ? 6 : M <= 8 ? 8 : M <= 12 ? 12 : 16;
    p.cols = p.mt == 1 ? 8 : p.mt <= 4 ? 4 : p.mt <= 8 ? 2 : 1;
    p.cb = 32 * p.cols;
    p.n_cb = (N + p.cb - 1) / p.cb;
    p.warps = kWarps;
    const int chunks = K / kChunk;
    const long long items = static_cast<long long>(p.n_cb) * chunks;
    p.items = items;
    // two resident CTAs per SM, each with at least one chunk per warp
    const long long want = 2LL * dp.sms;
    p.grid = static_cast<int>(std::max<long long>(1, std::min<long long>(want, items / kWarps)));
    const size_t xsum_bytes = static_cast<size_t>(M) * chunks * sizeof(float2);
    p.fact = M <= kFactMaxM && xsum_bytes <= kXsumSmemLimit;
    p.smem_bytes = static_cast<size_t>(kWarps) * p.mt * p.cb * sizeof(float) + (p.fact ? xsum_bytes : 0);
    p.ticket_bytes = (static_cast<size_t>(p.n_cb) * sizeof(uint32_t) + 255) & ~size_t(255);
    // Partial slots first, in a region whose size depends only on the device
    // (M * columns-per-block <= kMaxLive for every row template), tickets after
    // it: calls of different shapes sharing one workspace never write partial
    // sums over one another's tickets.
    p.partial_bytes = partial_region_bytes(dp);
    return p;
}

size_t gemv_workspace_bytes(const GemvPlan& p) { return p.ticket_bytes + p.partial_bytes; }

cudaError_t launch_gemv(const void* x, const uint32_t* qw, const void* sc, const uint32_t* qz, void* y, int M,
                        int N, int K, int g, bool bf16, const GemvPlan& plan, void* workspace, cudaStream_t s) {
    GemvArgs a;
    a.x = static_cast<const uint16_t*>(x);
    a.qw = qw;
    a.sc = static_cast<const uint16_t*>(sc);
    a.qz = qz;
    a.y = static_cast<uint16_t*>(y);
    a.partials = static_cast<float*>(workspace);
    a.tickets = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + plan.partial_bytes);
    a.M = M;
    a.N = N;
    a.K = K;
    a.g = g;
    a.chunks = K / kChunk;
    a.items = plan.items;
    return bf16 ? launch_dtype<true>(a, plan, s) : launch_dtype<false>(a, plan, s);
}

}  // namespace w4a16
