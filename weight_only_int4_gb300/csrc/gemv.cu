// Decode GEMV of the W4A16 layer, 1 <= M <= 16, on CUDA cores.
//
// The kernel is memory-bound: each weight nibble is read once, and per call
// it must stream K*N/2 bytes of packed weights, (K/g)*N scales and (K/g)*N/2
// bytes of packed zero-points. "Keep W4A16 zero-points packed at 4 bits
// instead of expanding to 2 bytes" (sections "Problem" and "Known regression")
// shows both halves of the design problem: time tracks bytes, and at batch 4
// the nibble extract costs time unless the loads of the next tile are in
// flight while the current one is converted. Here:
//
//   * a lane owns COLS adjacent columns and streams, per 32-row chunk of K,
//     4 rows x COLS packed words with 128-bit non-allocating loads, its scales
//     and its packed zero-point word;
//   * the next chunk's loads are issued before the current chunk is
//     converted (register double buffering), so memory and ALU overlap;
//   * nibbles become fp16/bf16 by the exponent-bias trick (OR the nibble into
//     the mantissa of 1024.0 / 128.0), the zero-point is subtracted in packed
//     16-bit arithmetic (exact: |q - z| <= 15), and (q - z) * x is accumulated
//     by a mixed-precision FMA with an FP32 accumulator (exact product, one
//     rounding); the group scale is applied once per chunk in FP32;
//   * K is split over the 8 warps of a CTA and over the CTAs of a thread-block
//     cluster; partial sums are reduced in shared memory, then across the
//     cluster through distributed shared memory, always in the same order, so
//     results are deterministic and no global workspace is needed.
#include "internal.h"
#include "ptx.cuh"

#include <cooperative_groups.h>

#include <algorithm>

namespace cg = cooperative_groups;

namespace w4a16 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kChunk = 32;            // rows of K per chunk
constexpr int kRowsPerChunk = 4;      // packed word rows per chunk

template <bool kBf16>
struct Act;
template <>
struct Act<false> {
    using T = __half;
    static constexpr uint32_t kMagic = 0x64006400u;   // fp16 1024.0 in both halves
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
    using T = __nv_bfloat16;
    static constexpr uint32_t kMagic = 0x43004300u;   // bf16 128.0 in both halves
    __device__ static float to_float(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
    __device__ static uint16_t from_float(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
    __device__ static uint32_t sub2(uint32_t a, uint32_t b) {
        uint32_t d;
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
};

// Streaming load: read once, do not allocate in L1.
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

// COLS consecutive 32-bit words.
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

// COLS consecutive 16-bit scales, returned as 16-bit patterns.
template <int COLS>
__device__ __forceinline__ void load_scales(const uint16_t* p, uint16_t (&v)[COLS]) {
    if constexpr (COLS == 8) {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = static_cast<uint16_t>(w[j / 2] >> (16 * (j & 1)));
    } else if constexpr (COLS == 4) {
        const uint2 a = __ldg(reinterpret_cast<const uint2*>(p));
        const uint32_t w[2] = {a.x, a.y};
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = static_cast<uint16_t>(w[j / 2] >> (16 * (j & 1)));
    } else if constexpr (COLS == 2) {
        const uint32_t a = __ldg(reinterpret_cast<const uint32_t*>(p));
        v[0] = static_cast<uint16_t>(a);
        v[1] = static_cast<uint16_t>(a >> 16);
    } else {
        v[0] = __ldg(p);
    }
}

template <int COLS>
struct ChunkRegs {
    uint32_t q[kRowsPerChunk][COLS];
    uint16_t s[COLS];
    uint32_t z;
};

template <bool kBf16, int MT, int COLS, bool kSym>
__global__ void __launch_bounds__(kThreads, 2)
gemv_kernel(const uint16_t* __restrict__ x, const uint32_t* __restrict__ qw, const uint16_t* __restrict__ sc,
            const uint32_t* __restrict__ qz, uint16_t* __restrict__ y, int M, int N, int K, int g, int cs) {
    using A = Act<kBf16>;
    constexpr int CB = 32 * COLS;
    constexpr int E = MT * CB;
    __shared__ float red[kWarps * E];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = static_cast<int>(blockIdx.x % cs);
    const int cb = static_cast<int>(blockIdx.x / cs);
    const int n0 = cb * CB + lane * COLS;
    const bool col_ok = n0 < N;                 // N % 8 == 0 and COLS | 8: all COLS columns valid
    const int chunks = K / kChunk;
    const int slice = rank * kWarps + warp;
    const int nslices = cs * kWarps;
    const int zshift = 4 * (n0 & 7);

    float yacc[MT][COLS];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int j = 0; j < COLS; ++j) yacc[m][j] = 0.f;

    auto load = [&](ChunkRegs<COLS>& r, int c) {
        const uint32_t* p = qw + static_cast<size_t>(c) * kRowsPerChunk * N + n0;
#pragma unroll
        for (int i = 0; i < kRowsPerChunk; ++i) load_words<COLS>(p + static_cast<size_t>(i) * N, r.q[i]);
        const int t = (c * kChunk) / g;
        load_scales<COLS>(sc + static_cast<size_t>(t) * N + n0, r.s);
        if constexpr (!kSym) r.z = __ldg(qz + static_cast<size_t>(t) * (N >> 3) + (n0 >> 3));
    };

    auto compute = [&](const ChunkRegs<COLS>& r, int c) {
        uint32_t zz[COLS];
#pragma unroll
        for (int j = 0; j < COLS; ++j) {
            const uint32_t z = kSym ? 8u : ((r.z >> (zshift + 4 * j)) & 0xFu);
            zz[j] = A::kMagic | z | (z << 16);          // (magic + z) in both halves, exact
        }
        float acc[MT][COLS];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int j = 0; j < COLS; ++j) acc[m][j] = 0.f;
#pragma unroll
        for (int i = 0; i < kRowsPerChunk; ++i) {
            uint4 xv[MT];
            const int k = c * kChunk + i * 8;
#pragma unroll
            for (int m = 0; m < MT; ++m)
                xv[m] = (m < M) ? __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(m) * K + k))
                                : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int j = 0; j < COLS; ++j) {
                const uint32_t w = r.q[i][j];
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    // halves: (magic + q[k + b], magic + q[k + b + 4]) -> (q - z) exactly
                    const uint32_t d = A::sub2(and_or(w >> (4 * b), 0x000F000Fu, A::kMagic), zz[j]);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const uint32_t xlo = (b < 2) ? xv[m].x : xv[m].y;   // x[k + b]
                        const uint32_t xhi = (b < 2) ? xv[m].z : xv[m].w;   // x[k + b + 4]
                        if (b & 1) {
                            acc[m][j] = fma_mixed<kBf16, 0, 1>(d, xlo, acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 1, 1>(d, xhi, acc[m][j]);
                        } else {
                            acc[m][j] = fma_mixed<kBf16, 0, 0>(d, xlo, acc[m][j]);
                            acc[m][j] = fma_mixed<kBf16, 1, 0>(d, xhi, acc[m][j]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < COLS; ++j) {
            const float s = A::to_float(r.s[j]);
#pragma unroll
            for (int m = 0; m < MT; ++m) yacc[m][j] = fmaf(s, acc[m][j], yacc[m][j]);
        }
    };

    if (col_ok) {
        ChunkRegs<COLS> b0, b1;
        int c = slice;
        if (c < chunks) load(b0, c);
        for (; c < chunks; c += 2 * nslices) {
            const int c1 = c + nslices;
            if (c1 < chunks) load(b1, c1);
            compute(b0, c);
            const int c2 = c1 + nslices;
            if (c2 < chunks) load(b0, c2);
            if (c1 < chunks) compute(b1, c1);
        }
    }

    // partial sums of the 8 warps -> shared memory, reduced in warp order
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int j = 0; j < COLS; ++j) red[warp * E + m * CB + lane * COLS + j] = yacc[m][j];
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads) {
        float s = red[e];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) s += red[w * E + e];
        red[e] = s;
    }

    auto store = [&](int e, float v) {
        const int m = e / CB, n = cb * CB + (e - m * CB);
        if (m < M && n < N) y[static_cast<size_t>(m) * N + n] = A::from_float(v);
    };

    if (cs == 1) {
        for (int e = threadIdx.x; e < E; e += kThreads) store(e, red[e]);
        return;
    }
    // cluster: CTA `rank` finishes entries [rank*E/cs, (rank+1)*E/cs), summing ranks in order
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int e0 = rank * E / cs, e1 = (rank + 1) * E / cs;
    for (int e = e0 + threadIdx.x; e < e1; e += kThreads) {
        float s = 0.f;
        for (int q = 0; q < cs; ++q) s += cluster.map_shared_rank(red, q)[e];
        store(e, s);
    }
    cluster.sync();   // keep this CTA's shared memory alive until every peer has read it
}

template <bool kBf16, int MT, int COLS, bool kSym>
cudaError_t launch_one(const void* x, const uint32_t* qw, const void* sc, const uint32_t* qz, void* y, int M,
                       int N, int K, int g, const GemvPlan& p, cudaStream_t s) {
    auto kern = gemv_kernel<kBf16, MT, COLS, kSym>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.n_cb * p.cluster), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<const uint16_t*>(x), qw, static_cast<const uint16_t*>(sc), qz,
                              static_cast<uint16_t*>(y), M, N, K, g, p.cluster);
}

template <bool kBf16, int MT, int COLS>
cudaError_t launch_sym(const void* x, const uint32_t* qw, const void* sc, const uint32_t* qz, void* y, int M, int N,
                       int K, int g, const GemvPlan& p, cudaStream_t s) {
    return qz ? launch_one<kBf16, MT, COLS, false>(x, qw, sc, qz, y, M, N, K, g, p, s)
              : launch_one<kBf16, MT, COLS, true>(x, qw, sc, qz, y, M, N, K, g, p, s);
}

template <bool kBf16>
cudaError_t launch_dtype(const void* x, const uint32_t* qw, const void* sc, const uint32_t* qz, void* y, int M,
                         int N, int K, int g, const GemvPlan& p, cudaStream_t s) {
    switch (p.mt) {
        case 1: return launch_sym<kBf16, 1, 8>(x, qw, sc, qz, y, M, N, K, g, p, s);
        case 2: return launch_sym<kBf16, 2, 8>(x, qw, sc, qz, y, M, N, K, g, p, s);
        case 3: return launch_sym<kBf16, 3, 4>(x, qw, sc, qz, y, M, N, K, g, p, s);
        case 4: return launch_sym<kBf16, 4, 4>(x, qw, sc, qz, y, M, N, K, g, p, s);
        case 6: return launch_sym<kBf16, 6, 2>(x, qw, sc, qz, y, M, N, K, g, p, s);
        case 8: return launch_sym<kBf16, 8, 2>(x, qw, sc, qz, y, M, N, K, g, p, s);
        case 12: return launch_sym<kBf16, 12, 1>(x, qw, sc, qz, y, M, N, K, g, p, s);
        case 16: return launch_sym<kBf16, 16, 1>(x, qw, sc, qz, y, M, N, K, g, p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

GemvPlan plan_gemv(int M, int N, int K, int g, const DeviceProps& dp) {
    (void)g;
    GemvPlan p;
    p.mt = M <= 1 ? 1 : M <= 2 ? 2 : M <= 3 ? 3 : M <= 4 ? 4 : M <= 6 ? 6 : M <= 8 ? 8 : M <= 12 ? 12 : 16;
    p.cols = p.mt <= 2 ? 8 : p.mt <= 4 ? 4 : p.mt <= 8 ? 2 : 1;
    p.cb = 32 * p.cols;
    p.n_cb = (N + p.cb - 1) / p.cb;
    p.warps = kWarps;
    // Fill the machine in one wave (2 CTAs per SM), splitting K over a cluster
    // only while every warp keeps at least one chunk of K.
    const int slots = 2 * dp.sms;
    const int chunks = K / kChunk;
    int cs = slots / std::max(1, p.n_cb);
    cs = std::min(cs, 8);
    cs = std::min(cs, std::max(1, chunks / kWarps));
    p.cluster = std::max(1, cs);
    return p;
}

cudaError_t launch_gemv(const void* x, const uint32_t* qw, const void* sc, const uint32_t* qz, void* y, int M,
                        int N, int K, int g, bool bf16, const GemvPlan& plan, cudaStream_t s) {
    return bf16 ? launch_dtype<true>(x, qw, sc, qz, y, M, N, K, g, plan, s)
                : launch_dtype<false>(x, qw, sc, qz, y, M, N, K, g, plan, s);
}

}  // namespace w4a16
