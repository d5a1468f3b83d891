// Weight packing: canonical INT4 nibbles and bf16 scales -> the stage layout
// the GEMM kernels stream with one bulk copy per stage (layout documented in
// include/moe_int4.h, moe_int4_pack).  The pages repack GPTQ-format INT4 into
// their kernel's own layout before use ("The Throughput Lever", section
// "Building the Benchmark"); this layout is designed for the sm_103a kernels:
// each stage is contiguous, each dequantising thread reads its row's 32 bytes
// as two conflict-free 16-byte shared-memory loads, and the nibble order lets
// one mask/OR produce two fp16 values at once.  MXFP4 weights use the same
// nibble layout (their codes are E2M1, not integers) with E8M0 scales converted
// to the fp16 factor their dequant multiplies by.
#include <cuda_fp16.h>

#include "kernels.cuh"

namespace moe {

// shuffle = 1 (INT4): within a 32-bit word, the nibbles of elements 2s and
// 2s + 1 go to bits 4s and 16 + 4s, so that one mask gives two fp16 operands;
// shuffle = 0 (MXFP4): the word keeps the canonical byte order (byte c holds
// elements 2c and 2c + 1), which the FP4 -> fp16x2 conversion reads directly.
__global__ void pack_weights_kernel(const uint8_t *__restrict__ q, uint32_t *__restrict__ out,
                                    int N, int K, int is_w13, size_t n_words, int shuffle) {
    const int KS = is_w13 ? K / kSlabK : K / (2 * kSlabK);
    const int RT = is_w13 ? (N / 2) / kSlabRows : N / kSlabRows;
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n_words;
         idx += (size_t)gridDim.x * blockDim.x) {
        const size_t stage = idx / (kStageWBytes / 4);
        const int within = (int)(idx % (kStageWBytes / 4));
        const int slab = within / (kSlabBytes / 4);
        const int rem = within % (kSlabBytes / 4);
        const int half = rem / 512;
        const int row = (rem % 512) / 4;
        const int w = rem % 4;
        const int v = 4 * half + w;
        const int kk = (int)(stage % KS);
        const int r = (int)((stage / KS) % RT);
        const size_t e = stage / ((size_t)KS * RT);
        int n, kb;
        if (is_w13) {
            n = (slab ? N / 2 : 0) + kSlabRows * r + row;
            kb = kk;
        } else {
            n = kSlabRows * r + row;
            kb = 2 * kk + slab;
        }
        const uint32_t src = *reinterpret_cast<const uint32_t *>(
            q + (e * N + n) * (size_t)(K / 2) + (size_t)kb * (kSlabK / 2) + 4 * v);
        uint32_t word = src;
        if (shuffle) {
            word = 0;
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint32_t b = (src >> (8 * s)) & 0xFFu;
                word |= (b & 0xFu) << (4 * s);
                word |= (b >> 4) << (16 + 4 * s);
            }
        }
        out[idx] = word;
    }
}

// bf16 scale -> fp16 (exact for magnitudes in [2^-14, 65504]; saturating above,
// fp16 subnormals below).  A non-zero scale outside [2^-14, 2729] in magnitude
// (or not finite) is counted in *inexact: there, the GEMMs' dequantised weight
// (16 + q) * s - 24 * s = (q - 8) * s is not exact in fp16 (the addend 24 * s
// needs 24 * 2729 < 65504; from 2^-14 up, it and the product keep a bf16
// scale's 8 significant bits plus at most 3).
__device__ __forceinline__ uint16_t bf16_bits_to_f16_sat(uint16_t b, uint32_t *inexact) {
    float v = __uint_as_float((uint32_t)b << 16);
    const float m = fabsf(v);
    if (inexact && v != 0.0f && !(m >= 0x1p-14f && m <= 2729.0f)) atomicAdd(inexact, 1u);
    v = fminf(fmaxf(v, -65504.0f), 65504.0f);
    return __half_as_ushort(__float2half_rn(v));
}

// E8M0 scale byte -> the fp16 factor of the MXFP4 dequant, the scale itself
// 2^(e - 127) (the dequant converts each E2M1 code to its exact fp16 value and
// multiplies).  Supported: e in [103, 140], where the factor is an fp16 power
// of two (normal or subnormal) and no weight overflows (6 * 2^13 < 65504);
// other codes, 255 (NaN) included, are clamped to that range and counted in
// *bad.  The weights are exact from e = 104 up (0.5 * 2^(e - 127) >= 2^-24).
__device__ __forceinline__ uint16_t e8m0_to_f16_factor(uint8_t e, uint32_t *bad) {
    int x = (int)e - 127;
    if (x < -24 || x > 13) {
        if (bad) atomicAdd(bad, 1u);
        x = x < -24 ? -24 : 13;
    }
    return x >= -14 ? (uint16_t)((x + 15) << 10) : (uint16_t)(1u << (x + 24));
}

struct Bf16Scale {
    using T = uint16_t;
    uint32_t *inexact;
    __device__ uint16_t operator()(uint16_t b) const { return bf16_bits_to_f16_sat(b, inexact); }
};
struct E8m0Scale {
    using T = uint8_t;
    uint32_t *bad;
    __device__ uint16_t operator()(uint8_t e) const { return e8m0_to_f16_factor(e, bad); }
};

// Scales [E][N][K/32] (bf16 bits or E8M0 bytes) -> per stage [slab][row][2] fp16.
template <class Conv>
__global__ void pack_scales_kernel(const typename Conv::T *__restrict__ s,
                                   uint32_t *__restrict__ out, int N, int K, int is_w13,
                                   size_t n_words, Conv conv) {
    const int KS = is_w13 ? K / kSlabK : K / (2 * kSlabK);
    const int RT = is_w13 ? (N / 2) / kSlabRows : N / kSlabRows;
    const int G = K / 32;
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n_words;
         idx += (size_t)gridDim.x * blockDim.x) {
        const size_t stage = idx / (kStageSBytes / 4);
        const int within = (int)(idx % (kStageSBytes / 4));
        const int slab = within / kSlabRows;
        const int row = within % kSlabRows;
        const int kk = (int)(stage % KS);
        const int r = (int)((stage / KS) % RT);
        const size_t e = stage / ((size_t)KS * RT);
        int n, kb;
        if (is_w13) {
            n = (slab ? N / 2 : 0) + kSlabRows * r + row;
            kb = kk;
        } else {
            n = kSlabRows * r + row;
            kb = 2 * kk + slab;
        }
        const typename Conv::T *src = s + (e * N + n) * (size_t)G + 2 * kb;
        out[idx] = (uint32_t)conv(src[0]) | ((uint32_t)conv(src[1]) << 16);
    }
}

template <class Conv>
cudaError_t launch_pack_impl(const uint8_t *q, const typename Conv::T *scales, Conv conv, int E,
                             int N, int K, int is_w13, void *packed, void *packed_scales,
                             int shuffle, cudaStream_t s) {
    const size_t n_words = (size_t)E * N * (K / 2) / 4;
    const size_t n_swords = (size_t)E * N * (K / 32) / 2;
    const int threads = 256;
    size_t blocks = (n_words + threads - 1) / threads;
    if (blocks > 65535 * 8) blocks = 65535 * 8;
    pack_weights_kernel<<<(unsigned)blocks, threads, 0, s>>>(
        q, reinterpret_cast<uint32_t *>(packed), N, K, is_w13, n_words, shuffle);
    size_t sblocks = (n_swords + threads - 1) / threads;
    if (sblocks > 65535 * 8) sblocks = 65535 * 8;
    pack_scales_kernel<Conv><<<(unsigned)sblocks, threads, 0, s>>>(
        scales, reinterpret_cast<uint32_t *>(packed_scales), N, K, is_w13, n_swords, conv);
    return cudaGetLastError();
}

cudaError_t launch_pack(const uint8_t *q, const uint16_t *scales, int E, int N, int K,
                        int is_w13, void *packed, void *packed_scales, uint32_t *inexact,
                        cudaStream_t s) {
    return launch_pack_impl(q, scales, Bf16Scale{inexact}, E, N, K, is_w13, packed,
                            packed_scales, 1, s);
}

cudaError_t launch_pack_mxfp4(const uint8_t *q, const uint8_t *scales, int E, int N, int K,
                              int is_w13, void *packed, void *packed_scales, uint32_t *bad,
                              cudaStream_t s) {
    return launch_pack_impl(q, scales, E8m0Scale{bad}, E, N, K, is_w13, packed, packed_scales,
                            0, s);
}

}  // namespace moe
