// Weight packing: canonical INT4 nibbles and bf16 scales -> the stage layout
// the GEMM kernels stream with one bulk copy per stage (layout documented in
// include/moe_int4.h, moe_int4_pack).  The pages repack GPTQ-format INT4 into
// their kernel's own layout before use ("The Throughput Lever", section
// "Building the Benchmark"); this layout is designed for the sm_103a kernels:
// each stage is contiguous, each dequantising thread reads its row's 32 bytes
// as two conflict-free 16-byte shared-memory loads, and the nibble order lets
// one mask/OR produce two bf16 values at once.
#include <cuda_fp16.h>

#include "kernels.cuh"

namespace moe {

__global__ void pack_weights_kernel(const uint8_t *__restrict__ q, uint32_t *__restrict__ out,
                                    int N, int K, int is_w13, size_t n_words) {
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
        uint32_t word = 0;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const uint32_t b = (src >> (8 * s)) & 0xFFu;
            word |= (b & 0xFu) << (4 * s);
            word |= (b >> 4) << (16 + 4 * s);
        }
        out[idx] = word;
    }
}

// bf16 scale -> fp16 (exact for magnitudes in [2^-14, 65504]; saturating above,
// fp16 subnormals below).
__device__ __forceinline__ uint16_t bf16_bits_to_f16_sat(uint16_t b) {
    float v = __uint_as_float((uint32_t)b << 16);
    v = fminf(fmaxf(v, -65504.0f), 65504.0f);
    return __half_as_ushort(__float2half_rn(v));
}

__global__ void pack_scales_kernel(const uint16_t *__restrict__ s, uint32_t *__restrict__ out,
                                   int N, int K, int is_w13, size_t n_words) {
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
        const uint16_t *src = s + (e * N + n) * (size_t)G + 2 * kb;
        out[idx] = (uint32_t)bf16_bits_to_f16_sat(src[0]) |
                   ((uint32_t)bf16_bits_to_f16_sat(src[1]) << 16);
    }
}

cudaError_t launch_pack(const uint8_t *q, const uint16_t *scales, int E, int N, int K,
                        int is_w13, void *packed, void *packed_scales, cudaStream_t s) {
    const size_t n_words = (size_t)E * N * (K / 2) / 4;
    const size_t n_swords = (size_t)E * N * (K / 32) / 2;
    const int threads = 256;
    size_t blocks = (n_words + threads - 1) / threads;
    if (blocks > 65535 * 8) blocks = 65535 * 8;
    pack_weights_kernel<<<(unsigned)blocks, threads, 0, s>>>(
        q, reinterpret_cast<uint32_t *>(packed), N, K, is_w13, n_words);
    size_t sblocks = (n_swords + threads - 1) / threads;
    if (sblocks > 65535 * 8) sblocks = 65535 * 8;
    pack_scales_kernel<<<(unsigned)sblocks, threads, 0, s>>>(
        scales, reinterpret_cast<uint32_t *>(packed_scales), N, K, is_w13, n_swords);
    return cudaGetLastError();
}

}  // namespace moe
