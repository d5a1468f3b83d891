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

// The down step of the separate plan at short routing blocks, in the same
// style: per align block, the expert's down rows are streamed once and reduced
// against the block's real rows of the gate/up intermediate, two rows per MMA.
struct BlockDownArgs {
    const int32_t *sorted_ids;   // [cap] pair of each bucketed row (>= P: padding)
    const int32_t *expert_ids;   // [blocks] expert of each block
    const int32_t *num_post_pad; // [1] rows in use (a multiple of block_m)
    const uint16_t *a_out;       // [cap][I] fp16 intermediate, bucketed order
    const float *topk_weights;   // [P]
    const uint8_t *w2, *s2;      // packed down weights and scales
    float *out;                  // [M][H] fp32 accumulator (zeroed by the gate/up GEMM)
    uint32_t *err;
    int P, E, H, I, top_k, block_m, blocks_cap;
    int cap;                     // rows of sorted_ids and a_out
    int RT2, KB2, SB, KB2s;      // row tiles (H / 128), 64-k blocks, k splits, per split
    int fmt;
    DequantConsts dq;
};
// Programmatic dependent launch after the gate/up GEMM.
cudaError_t launch_block_down(const BlockDownArgs &a, cudaStream_t s, int *launches);

}  // namespace moe
