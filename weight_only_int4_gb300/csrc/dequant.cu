// Dense dequantised copy of the packed weights,
//
//     W[k, n] = RN((q[k, n] - z[k / g, n]) * s[k / g, n])   in the activation dtype, row-major [K, N],
//
// the dense dequantised weight copy that "Keep W4A16 zero-points packed at 4
// bits instead of expanding to 2 bytes" (section "Change") builds at load time
// beside the skinny GEMM. A pure streaming kernel: per element it reads 0.5 byte of
// packed code (plus 2.5/g of scale and zero-point) and writes 2 bytes, so it
// is bound by HBM bandwidth.
//
// A thread owns four packed word rows (32 rows of K, within one group) of 8
// adjacent columns: eight 16-byte loads of qweight, one of the 8 scales and
// one packed zero-point word shared by the four; consecutive threads take
// consecutive column groups, so loads and the 16-byte stores of each output
// row are coalesced. (One word row per thread, which loads each group's scales
// four times, was 7 % slower.) Per row and
// column pair: a byte permute puts nibble j of both columns' words into the
// low bits of two 16-bit halves, an OR with the exponent of 1024 (fp16) or
// 128 (bf16) turns them into magic + q, one packed subtract of magic + z gives
// the exact (q - z), one packed multiply by s rounds once.
#include "internal.h"
#include "mxfp4.cuh"
#include "ptx.cuh"

#include <algorithm>

namespace w4a16 {
namespace {

template <bool kBf16>
struct Dq;
template <>
struct Dq<false> {
    static constexpr uint32_t kMagic = 0x64006400u;   // fp16 1024.0 in both halves
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
};
template <>
struct Dq<true> {
    static constexpr uint32_t kMagic = 0x43004300u;   // bf16 128.0 in both halves
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
};

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ void st_stream(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

constexpr int kThreads = 256;
// Packed word rows (8 rows of K each) per thread: 4 share one load of their
// 32-row group's scales and zero-points (every group size is a multiple of 32).
#ifndef W4A16_DEQUANT_WORD_ROWS
#define W4A16_DEQUANT_WORD_ROWS 4
#endif
constexpr int kWordRows = W4A16_DEQUANT_WORD_ROWS;
static_assert(kWordRows == 1 || kWordRows == 2 || kWordRows == 4, "word rows per thread");

template <bool kBf16, bool kSym>
__global__ void __launch_bounds__(kThreads) dequant_kernel(const uint32_t* __restrict__ qw,
                                                          const uint16_t* __restrict__ sc,
                                                          const uint32_t* __restrict__ qz, uint16_t* __restrict__ out,
                                                          int N, long long items, int g_shift) {
    using D = Dq<kBf16>;
    const int ng = N >> 3;   // column groups of 8
    for (long long i = blockIdx.x * static_cast<long long>(kThreads) + threadIdx.x; i < items;
         i += static_cast<long long>(gridDim.x) * kThreads) {
        const long long wb = i / ng;
        const int c = static_cast<int>(i - wb * ng);
        const long long w0 = wb * kWordRows;
        const int t = static_cast<int>((w0 * 8) >> g_shift);    // the rows lie in one group (8 * kWordRows | g)
        uint4 q[kWordRows][2];
#pragma unroll
        for (int r = 0; r < kWordRows; ++r) {
            q[r][0] = ld_stream(qw + (w0 + r) * N + 8 * c);
            q[r][1] = ld_stream(qw + (w0 + r) * N + 8 * c + 4);
        }
        const uint4 s8 = ld_stream(sc + static_cast<long long>(t) * N + 8 * c);
        const uint32_t zw = kSym ? 0x88888888u : __ldg(qz + static_cast<long long>(t) * ng + c);
        const uint32_t ss[4] = {s8.x, s8.y, s8.z, s8.w};
        uint32_t zz[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            // (magic + z of column 2p, magic + z of column 2p+1)
            zz[p] = D::kMagic | ((zw >> (8 * p)) & 0xFu) | (((zw >> (8 * p + 4)) & 0xFu) << 16);
        }
#pragma unroll
        for (int r = 0; r < kWordRows; ++r) {
            uint32_t wd[8] = {q[r][0].x, q[r][0].y, q[r][0].z, q[r][0].w, q[r][1].x, q[r][1].y, q[r][1].z, q[r][1].w};
            uint16_t* orow = out + ((w0 + r) * 8) * static_cast<long long>(N) + 8 * c;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t o[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    // low 16 bits of each column's word -> the two halves; keep nibble j (now in bits 0-3)
                    const uint32_t h = and_or(prmt(wd[2 * p], wd[2 * p + 1], 0x5410u), 0x000F000Fu, D::kMagic);
                    o[p] = D::mul2(D::sub2(h, zz[p]), ss[p]);
                }
                st_stream(orow + static_cast<long long>(j) * N, o[0], o[1], o[2], o[3]);
#pragma unroll
                for (int u = 0; u < 8; ++u) wd[u] >>= 4;
            }
        }
    }
}

template <bool kBf16, bool kSym>
cudaError_t launch_typed(const uint32_t* qw, const void* sc, const uint32_t* qz, void* out, int N, int K, int g,
                         const DeviceProps& dp, cudaStream_t s) {
    const long long items = static_cast<long long>(K / 8 / kWordRows) * (N / 8);
    const long long want = (items + kThreads - 1) / kThreads;
    const int grid = static_cast<int>(std::min<long long>(want, static_cast<long long>(dp.sms) * 8));
    dequant_kernel<kBf16, kSym><<<grid, kThreads, 0, s>>>(qw, static_cast<const uint16_t*>(sc), qz,
                                                          static_cast<uint16_t*>(out), N, items,
                                                          __builtin_ctz(static_cast<unsigned>(g)));
    return cudaGetLastError();
}

// MXFP4 weights to a dense bf16 copy, W[k, n] = RN(E2M1(q[k, n]) * 2^(e[k / 32, n] - 127)).
// Same thread layout as above: kWordRows packed word rows of 8 adjacent
// columns, within one 32-row block, with the block's 8 exponent bytes in one
// 8-byte load.
__global__ void __launch_bounds__(kThreads) mx_dequant_kernel(const uint32_t* __restrict__ qw,
                                                             const uint8_t* __restrict__ es,
                                                             uint16_t* __restrict__ out, int N, long long items) {
    const int ng = N >> 3;
    for (long long i = blockIdx.x * static_cast<long long>(kThreads) + threadIdx.x; i < items;
         i += static_cast<long long>(gridDim.x) * kThreads) {
        const long long wb = i / ng;
        const int c = static_cast<int>(i - wb * ng);
        const long long w0 = wb * kWordRows;
        const long long blk = (w0 * 8) / mx::kBlock;
        uint4 q[kWordRows][2];
#pragma unroll
        for (int r = 0; r < kWordRows; ++r) {
            q[r][0] = ld_stream(qw + (w0 + r) * N + 8 * c);
            q[r][1] = ld_stream(qw + (w0 + r) * N + 8 * c + 4);
        }
        const uint2 e8 = __ldg(reinterpret_cast<const uint2*>(es + blk * N + 8 * c));
        uint32_t fa[4], fb[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint32_t ew = p < 2 ? e8.x : e8.y;
            const int sh = 16 * (p & 1);
            mx::pair_factors((ew >> sh) & 0xFFu, (ew >> (sh + 8)) & 0xFFu, fa[p], fb[p]);
        }
#pragma unroll
        for (int r = 0; r < kWordRows; ++r) {
            uint32_t wd[8] = {q[r][0].x, q[r][0].y, q[r][0].z, q[r][0].w, q[r][1].x, q[r][1].y, q[r][1].z, q[r][1].w};
            uint16_t* orow = out + ((w0 + r) * 8) * static_cast<long long>(N) + 8 * c;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t o[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    // code j of columns 2p and 2p+1 in bits 0-3 of the two halves
                    const uint32_t h = prmt(wd[2 * p], wd[2 * p + 1], 0x5410u) & 0x000F000Fu;
                    o[p] = mx::mul_bf16x2(mx::mul_bf16x2(mx::e2m1x2_scaled(h), fa[p]), fb[p]);
                }
                st_stream(orow + static_cast<long long>(j) * N, o[0], o[1], o[2], o[3]);
#pragma unroll
                for (int u = 0; u < 8; ++u) wd[u] >>= 4;
            }
        }
    }
}

}  // namespace

cudaError_t launch_mx_dequant(const uint32_t* qw, const uint8_t* es, void* out, int N, int K, const DeviceProps& dp,
                              cudaStream_t s) {
    const long long items = static_cast<long long>(K / 8 / kWordRows) * (N / 8);
    const long long want = (items + kThreads - 1) / kThreads;
    const int grid = static_cast<int>(std::min<long long>(want, static_cast<long long>(dp.sms) * 8));
    mx_dequant_kernel<<<grid, kThreads, 0, s>>>(qw, es, static_cast<uint16_t*>(out), N, items);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const uint32_t* qw, const void* sc, const uint32_t* qz, void* out, int N, int K, int g,
                           bool bf16, const DeviceProps& dp, cudaStream_t s) {
    if (bf16)
        return qz ? launch_typed<true, false>(qw, sc, qz, out, N, K, g, dp, s)
                  : launch_typed<true, true>(qw, sc, qz, out, N, K, g, dp, s);
    return qz ? launch_typed<false, false>(qw, sc, qz, out, N, K, g, dp, s)
              : launch_typed<false, true>(qw, sc, qz, out, N, K, g, dp, s);
}

}  // namespace w4a16
