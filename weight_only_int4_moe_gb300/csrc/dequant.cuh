// Weight dequantisation and the SwiGLU activation, shared by the tensor-core
// GEMM kernels and the small-batch matrix-vector kernels, so both form exactly
// the same fp16 weights and intermediates.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "kernels.cuh"

namespace moe {

__device__ __forceinline__ __half2 as_h2(uint32_t v) {
    return *reinterpret_cast<const __half2 *>(&v);
}
__device__ __forceinline__ uint32_t as_u32(__half2 h) {
    return *reinterpret_cast<const uint32_t *>(&h);
}

// One slab row of a sub-stage: 64 weights (k = 0..63 of the slab's k block) as
// 32 fp16 pairs (q - 8) * s, out[c] holding k = 2c (low half) and 2c + 1 (high).
// Word v holds k = 8v..8v+7: bits 4s and 16+4s are k = 8v+2s and 8v+2s+1.
// Shifted so that the pair's nibbles sit at bits 6..9 of each half, masked and
// ORed with the exponent of 16, the word is the fp16 pair (16 + q): a mantissa
// bit 6 of an fp16 in [16, 32) weighs 1.  One FMA then gives
// (16 + q) * s - 24 * s = (q - 8) * s with a single rounding of the exact
// result, so the weight is exact: 24 * s is exact in fp16 (24 has two
// significant bits, s at most eight, from bf16) for |s| in [2^-14, 2729], and
// (q - 8) * s needs at most 8 + 3 significant bits.  Four shifts, four
// logic operations and four FMAs per eight weights; one FMA-pipe instruction
// per two weights where a subtraction and a multiply took two (measured 3.5 %
// faster at decode).
__device__ __forceinline__ void dequant_row(const uint4 lo, const uint4 hi, uint32_t sc,
                                            const DequantConsts &k, uint32_t (&out)[32]) {
    const __half2 s0 = as_h2(__byte_perm(sc, 0, 0x1010));  // group 0 scale, both halves
    const __half2 s1 = as_h2(__byte_perm(sc, 0, 0x3232));  // group 1 scale
    const __half2 cm24 = as_h2(k.cm24);
    const __half2 b0 = __hmul2(s0, cm24), b1 = __hmul2(s1, cm24);  // -24 * s, exact
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        const __half2 s2 = (v < 4) ? s0 : s1;
        const __half2 b2 = (v < 4) ? b0 : b1;
        const uint32_t t[4] = {w[v] << 6, w[v] << 2, w[v] >> 2, w[v] >> 6};
#pragma unroll
        for (int s = 0; s < 4; ++s)
            out[4 * v + s] = as_u32(__hfma2(as_h2((t[s] & k.nib_mask) | k.magic16), s2, b2));
    }
}

// MXFP4: the same 32 pairs from FP4 E2M1 codes, e2m1(q) * 2^(e - 127).  The
// MXFP4 pack keeps each word's bytes in canonical order (byte c of word v holds
// k = 8v + 2c in its low nibble and 8v + 2c + 1 in its high one), so one
// cvt.rn.f16x2.e2m1x2 turns a byte into the exact fp16 pair (low nibble in the
// low half) and one multiply by the packed scale 2^(e - 127) finishes it: two
// instructions per two weights.
__device__ __forceinline__ void dequant_row_fp4(const uint4 lo, const uint4 hi, uint32_t sc,
                                                uint32_t out[32]) {
    const __half2 s0 = as_h2(__byte_perm(sc, 0, 0x1010));
    const __half2 s1 = as_h2(__byte_perm(sc, 0, 0x3232));
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        const __half2 s2 = (v < 4) ? s0 : s1;
        uint32_t c[4];
        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
            "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
            "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
            : "=r"(c[0]), "=r"(c[1]), "=r"(c[2]), "=r"(c[3])
            : "r"(w[v]));
#pragma unroll
        for (int b = 0; b < 4; ++b) out[4 * v + b] = as_u32(__hmul2(as_h2(c[b]), s2));
    }
}

// fp32 -> fp16, saturating at the largest finite fp16 value; `bad` records a
// value outside [-65504, 65504] (NaN included).
__device__ __forceinline__ uint16_t f16_sat(float v, bool &bad) {
    bad |= !(fabsf(v) <= 65504.0f);
    v = fminf(fmaxf(v, -65504.0f), 65504.0f);
    return __half_as_ushort(__float2half_rn(v));
}

// SiLU(g) * u = g / (1 + e^-g) * u.  The fast divide is within a few ulp of
// the IEEE one (its result is rounded to fp16 next) and gives g * 0 = -0 when
// e^-g overflows for very negative g.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

}  // namespace moe
