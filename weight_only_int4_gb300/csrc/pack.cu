// Packing of 4-bit codes eight to a 32-bit word, and its inverse.
//
// Along rows (dim 0, the weight layout): nibble j of word [w, c] holds code
// [8w + j, c]. Along columns (dim 1, the zero-point layout of "Keep W4A16
// zero-points packed at 4 bits instead of expanding to 2 bytes", section
// "Change"): code [r, c] sits in word [r, c/8] at bits 4*(c%8).
//
// Load-time work, bandwidth-bound: each thread produces whole 16-byte output
// vectors where the shape allows it, with coalesced loads along the
// contiguous dimension.
#include "internal.h"

#include <algorithm>

namespace w4a16 {
namespace {

constexpr int kThreads = 256;

// dim 0, cols % 4 == 0: thread -> (word row w, 4 consecutive columns).
__global__ void pack_rows_x4(const uint8_t* __restrict__ src, uint32_t* __restrict__ dst, int64_t words,
                             int64_t cols) {
    const int64_t c4n = cols / 4;
    const int64_t total = words * c4n;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t w = i / c4n, c4 = i - w * c4n;
        uint32_t out[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(src + (8 * w + j) * cols) + c4);
#pragma unroll
            for (int b = 0; b < 4; ++b) out[b] |= ((v >> (8 * b)) & 0xFu) << (4 * j);
        }
        reinterpret_cast<uint4*>(dst + w * cols)[c4] = make_uint4(out[0], out[1], out[2], out[3]);
    }
}

__global__ void pack_rows_x1(const uint8_t* __restrict__ src, uint32_t* __restrict__ dst, int64_t words,
                             int64_t cols) {
    const int64_t total = words * cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t w = i / cols, c = i - w * cols;
        uint32_t out = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) out |= (static_cast<uint32_t>(src[(8 * w + j) * cols + c]) & 0xFu) << (4 * j);
        dst[i] = out;
    }
}

// dim 1: thread -> one word from 8 consecutive bytes of a row.
__global__ void pack_cols(const uint8_t* __restrict__ src, uint32_t* __restrict__ dst, int64_t nwords) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nwords;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(src) + i);
        uint32_t out = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            out |= ((v.x >> (8 * j)) & 0xFu) << (4 * j);
            out |= ((v.y >> (8 * j)) & 0xFu) << (4 * (j + 4));
        }
        dst[i] = out;
    }
}

__global__ void unpack_rows_x4(const uint32_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t words,
                               int64_t cols) {
    const int64_t c4n = cols / 4;
    const int64_t total = words * c4n;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t w = i / c4n, c4 = i - w * c4n;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + w * cols) + c4);
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t o = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) o |= ((in[b] >> (4 * j)) & 0xFu) << (8 * b);
            reinterpret_cast<uint32_t*>(dst + (8 * w + j) * cols)[c4] = o;
        }
    }
}

__global__ void unpack_rows_x1(const uint32_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t words,
                               int64_t cols) {
    const int64_t total = words * cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t w = i / cols, c = i - w * cols;
        const uint32_t v = __ldg(src + i);
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[(8 * w + j) * cols + c] = static_cast<uint8_t>((v >> (4 * j)) & 0xFu);
    }
}

__global__ void unpack_cols(const uint32_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t nwords) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nwords;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t v = __ldg(src + i);
        uint2 o = make_uint2(0u, 0u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            o.x |= ((v >> (4 * j)) & 0xFu) << (8 * j);
            o.y |= ((v >> (4 * (j + 4))) & 0xFu) << (8 * j);
        }
        reinterpret_cast<uint2*>(dst)[i] = o;
    }
}

int grid_for(int64_t work, const DeviceProps& dp) {
    const int64_t want = (work + kThreads - 1) / kThreads;
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)dp.sms * 16)));
}

}  // namespace

cudaError_t launch_pack(const uint8_t* src, uint32_t* dst, int64_t rows, int64_t cols, int dim,
                        const DeviceProps& dp, cudaStream_t s) {
    if (dim == 0) {
        const int64_t words = rows / 8;
        if (cols % 4 == 0)
            pack_rows_x4<<<grid_for(words * cols / 4, dp), kThreads, 0, s>>>(src, dst, words, cols);
        else
            pack_rows_x1<<<grid_for(words * cols, dp), kThreads, 0, s>>>(src, dst, words, cols);
    } else {
        const int64_t nwords = rows * (cols / 8);
        pack_cols<<<grid_for(nwords, dp), kThreads, 0, s>>>(src, dst, nwords);
    }
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t* src, uint8_t* dst, int64_t rows, int64_t cols, int dim,
                          const DeviceProps& dp, cudaStream_t s) {
    if (dim == 0) {
        const int64_t words = rows / 8;
        if (cols % 4 == 0)
            unpack_rows_x4<<<grid_for(words * cols / 4, dp), kThreads, 0, s>>>(src, dst, words, cols);
        else
            unpack_rows_x1<<<grid_for(words * cols, dp), kThreads, 0, s>>>(src, dst, words, cols);
    } else {
        const int64_t nwords = rows * (cols / 8);
        unpack_cols<<<grid_for(nwords, dp), kThreads, 0, s>>>(src, dst, nwords);
    }
    return cudaGetLastError();
}

}  // namespace w4a16
