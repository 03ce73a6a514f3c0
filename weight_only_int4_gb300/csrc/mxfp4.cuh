// MXFP4 weight decoding shared by the kernels: 4-bit E2M1 codes with one E8M0
// exponent byte per 32 K rows of a column, as on "Add BF16xFP4 MoE GEMM stage1
// kernel" (section "Technical Details"). The weight is
//
//     W = E2M1(c) * 2^(e - 127),   rounded to bf16 (exact unless it overflows),
//
// where code c has the sign in bit 3, a 2-bit exponent field E (bias 1) in
// bits 2..1 and a mantissa bit m in bit 0; E = 0 gives m / 2 (no implicit
// one). Byte e = 255 decodes to NaN, e = 0 to 2^-127.
//
// Decoding without a table: the code's bits moved into a bf16 pattern --
// sign to bit 15, E to the two low exponent bits 8..7, m to the top mantissa
// bit 6 -- read as bf16 is E2M1(c) * 2^-126 for every code. For E >= 1 the
// pattern is the normal number 2^(E - 127) (1 + m/2); for E = 0 it is the
// subnormal (m/2) 2^-126. Both follow from the bf16 encoding (bias 127,
// subnormals at exponent field 0 with weight 2^-126). One packed bf16
// multiply by 2^(e - 1) then yields W exactly whenever e <= 128 (2^(e - 1)
// is then a normal bf16 and every product has at most two significant bits
// and lies in [2^-128, 12]). For e >= 129 a first multiply by 2^126 gives
// E2M1(c) itself and a second by 2^(e - 127) gives W, or +-inf where W
// exceeds the bf16 range, exactly as a single rounding of the product.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

namespace w4a16 {
namespace mx {

constexpr int kBlock = 32;                      // K rows per E8M0 byte
constexpr uint32_t kTwoPow126x2 = 0x7E807E80u;  // bf16 2^126 in both halves

// Two codes, in bits 0..3 of each 16-bit half (all other bits zero), to the
// bf16 patterns of E2M1(c) * 2^-126: (c << 6) places m, E at bits 6..8 and
// (c << 12) the sign at bit 15; the two shifted copies occupy disjoint bit
// ranges, so one multiply by 0x1040 forms their sum without carries.
__device__ __forceinline__ uint32_t e2m1x2_scaled(uint32_t codes) { return (codes * 0x1040u) & 0x81C081C0u; }

// Whether one bf16 multiply by fast_scale(e) decodes the block exactly.
__device__ __forceinline__ bool fast(uint32_t e) { return e <= 128u; }

// bf16 2^(e - 1), for e <= 128.
__device__ __forceinline__ uint32_t fast_scale(uint32_t e) { return (e + 126u) << 7; }

// bf16 2^(e - 127) for e >= 1; NaN for 255; 2^-127 (a subnormal) for 0.
__device__ __forceinline__ uint32_t exact_scale(uint32_t e) {
    return e == 255u ? 0x7FC0u : e == 0u ? 0x0040u : (e << 7);
}

// FP32 2^(e - 127): the byte moved into the FP32 exponent field; 0 gives the
// subnormal 2^-127 and 255 NaN.
__device__ __forceinline__ float scale_f32(uint32_t e) {
    return __uint_as_float(e == 255u ? 0x7FC00000u : e == 0u ? 0x00400000u : (e << 23));
}

// Per 16-bit half h of a packed pair of scale bytes (e_lo, e_hi): the factors
// (a, b) with W = (pattern * a) * b exact for both halves: (2^(e - 1), 1) when
// e <= 128, else (2^126, 2^(e - 127)).
__device__ __forceinline__ void pair_factors(uint32_t e_lo, uint32_t e_hi, uint32_t& a, uint32_t& b) {
    const uint32_t a_lo = fast(e_lo) ? fast_scale(e_lo) : 0x7E80u;
    const uint32_t a_hi = fast(e_hi) ? fast_scale(e_hi) : 0x7E80u;
    const uint32_t b_lo = fast(e_lo) ? 0x3F80u : exact_scale(e_lo);
    const uint32_t b_hi = fast(e_hi) ? 0x3F80u : exact_scale(e_hi);
    a = a_lo | (a_hi << 16);
    b = b_lo | (b_hi << 16);
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// The 8 codes of a packed word (code j in bits 4j..4j+3) to four fp16 pairs:
// v[b] = (E2M1(code 2b), E2M1(code 2b + 1)). Every E2M1 value is an fp16
// number, so the hardware conversion is exact.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&v)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
        : "r"(w));
}

// Activations for an fp16 dot product against E2M1 codes. A run of bf16
// values whose largest biased exponent field is emax is multiplied by 2^c,
// c = min(141 - emax, 127), and rounded to fp16: the largest magnitude lands
// below 2^15 (fp16 stays finite) and every value whose magnitude is at least
// 2^-29 of the largest stays an fp16 normal number, so it converts exactly
// (bf16 has 8 significant bits, fp16 11). Smaller values round to the fp16
// subnormal grid, an absolute error of at most 2^-39 of the run's largest
// magnitude. inf and NaN stay inf and NaN. The clamp keeps 2^c a normal FP32
// number; it only acts when every value is below 2^-112, where multiplying
// by 2^127 still leaves each nonzero value at least 2^-6.
__device__ __forceinline__ int x_shift(uint32_t emax) { return min(141 - static_cast<int>(emax), 127); }
__device__ __forceinline__ uint16_t x_to_f16(uint16_t bits, int c) {
    const float v = __uint_as_float(static_cast<uint32_t>(bits) << 16) * __uint_as_float(static_cast<uint32_t>(c + 127) << 23);
    return __half_as_ushort(__float2half_rn(v));
}
// FP32 2^-c for c in [-114, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float x_unshift(int c) {
    return __uint_as_float(c == 127 ? 0x00400000u : static_cast<uint32_t>(127 - c) << 23);
}

// One thread's share of a GEMM operand tile: the 32 codes of column d in
// the 32-row half `half` of a 64-deep K step, read from the packed tile
// wt [8 words][kCols] and written as 32 bf16 weights to the column's 128-byte
// row at b_row of the K-major, 128-byte-swizzled operand tile (16-byte chunk
// c of the row lands at chunk c ^ (d & 7)). e is the block's exponent byte.
template <int kCols>
__device__ __forceinline__ void operand_column(const uint32_t* wt, uint32_t b_row, int d, int half, uint32_t e) {
    auto emit = [&](auto fast_path) {
        constexpr bool kFast = decltype(fast_path)::value;
        const uint32_t fa = kFast ? fast_scale(e) * 0x10001u : kTwoPow126x2;
        const uint32_t fb = exact_scale(e) * 0x10001u;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const int c = half * 4 + cc;
            const uint32_t w = wt[c * kCols + d];
            const uint32_t w4 = w >> 4;
            uint32_t o[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                // byte b of w -> low half, byte b of (w >> 4) -> high half: codes
                // 8c + 2b and 8c + 2b + 1 in bits 0-3 of the two halves
                uint32_t h;
                asm("prmt.b32 %0, %1, %2, %3;" : "=r"(h) : "r"(w), "r"(w4), "r"(static_cast<uint32_t>(b | ((4 + b) << 8))));
                o[b] = mul_bf16x2(e2m1x2_scaled(h & 0x000F000Fu), fa);
                if constexpr (!kFast) o[b] = mul_bf16x2(o[b], fb);
            }
            const uint32_t dst = b_row + (static_cast<uint32_t>(c ^ (d & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(o[0]), "r"(o[1]), "r"(o[2]),
                         "r"(o[3])
                         : "memory");
        }
    };
    // one multiply per pair when the block allows it; the branch is per thread
    if (fast(e))
        emit(std::true_type{});
    else
        emit(std::false_type{});
}

// The same 32 codes as 16 bf16 pairs in registers (pair 4cc + b holds codes
// 8cc + 2b and 8cc + 2b + 1 of the half), for an operand kept in tensor memory.
template <int kCols>
__device__ __forceinline__ void operand_column_regs(const uint32_t* wt, int d, int half, uint32_t e,
                                                    uint32_t (&o)[16]) {
    auto emit = [&](auto fast_path) {
        constexpr bool kFast = decltype(fast_path)::value;
        const uint32_t fa = kFast ? fast_scale(e) * 0x10001u : kTwoPow126x2;
        const uint32_t fb = exact_scale(e) * 0x10001u;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const uint32_t w = wt[(half * 4 + cc) * kCols + d];
            const uint32_t w4 = w >> 4;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                uint32_t h;
                asm("prmt.b32 %0, %1, %2, %3;" : "=r"(h) : "r"(w), "r"(w4), "r"(static_cast<uint32_t>(b | ((4 + b) << 8))));
                uint32_t v = mul_bf16x2(e2m1x2_scaled(h & 0x000F000Fu), fa);
                if constexpr (!kFast) v = mul_bf16x2(v, fb);
                o[4 * cc + b] = v;
            }
        }
    };
    if (fast(e))
        emit(std::true_type{});
    else
        emit(std::false_type{});
}

}  // namespace mx
}  // namespace w4a16
