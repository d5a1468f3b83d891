// The small-batch path (gemv.cu): the expert MLP as matrix-vector products,
// one routed pair at a time, without align or gather.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.cuh"

namespace moe {

struct GemvArgs {
    const uint16_t *x;          // [M][H] bf16 bits
    const int32_t *ids;         // [P] expert of each (token, slot) pair
    const float *topk_weights;  // [P]
    const uint8_t *w13, *s13, *w2, *s2;  // packed weights and scales
    float *gu;                  // [SA][P][2][I] gate / up partial sums per k split
    float *out;                 // [M][H] fp32 accumulator, zeroed by the gate/up kernel
    size_t out_n16;             // its size in float4s
    uint32_t *err;              // error words (flags, dropped pairs)
    int M, top_k, P, E, H, I;
    int RT1, KB, SA, KBs;       // gate/up: row tiles (I / 128), 64-k blocks, k splits, per split
    int RT2, KB2, SB, KB2s;     // down: row tiles (H / 128), 64-k blocks, k splits, per split
    int fmt;                    // 0 INT4, 1 MXFP4
    DequantConsts dq;
};
// step 1: the gate/up kernel; step 2: the down kernel (programmatic dependent launch)
cudaError_t launch_gemv(const GemvArgs &a, int step, cudaStream_t s, int *launches);

}  // namespace moe
