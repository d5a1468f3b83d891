// Internal interface between the kernel translation units and the C ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// Launch configuration with programmatic stream serialization: the kernel may
// start before the previous kernel of the stream has finished (it waits with
// griddepcontrol.wait before using that kernel's results).
inline cudaLaunchConfig_t pdl_config(unsigned grid, unsigned block, size_t smem, cudaStream_t s) {
    cudaLaunchConfig_t c{};
    c.gridDim = dim3(grid);
    c.blockDim = dim3(block);
    c.dynamicSmemBytes = smem;
    c.stream = s;
    return c;
}
inline unsigned pdl_attr(cudaLaunchAttribute &a) {
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return 1;
}

struct AlignArgs {
    const int32_t *ids;    // [P]
    int P, E, block_m;
    int32_t *sorted_ids;   // [capacity]
    int32_t *expert_ids;   // [capacity / block_m]
    int32_t *num_post_pad; // [1]
    uint32_t *err;         // [2] or null
    int32_t *chunk_tab;    // [n_chunks][E] (multi-block path)
    int n_chunks;          // 0: single-block path
    int32_t *pos_of;       // [P] or null: each pair's position in sorted_ids (-1: dropped)
};

// Router: per token, the top_k experts by logit (ties: lower index first) and
// their renormalised softmax weights.
struct RouteArgs {
    const float *logits;  // [M][E]
    int M, E, top_k;
    int32_t *ids;         // [M][top_k]
    float *weights;       // [M][top_k]
};

// Per-call zeroing done by the align launch's spare blocks.
struct ZeroArgs {
    void *ptr[2];
    size_t n16[2];  // 16-byte units
};

// Router alone (one warp per token).
cudaError_t launch_route(const RouteArgs &r, int sms, cudaStream_t s, int *launches);
// Router fused with the align (one kernel when the routing is small, else the
// router kernel then the align launch); a.ids must be r.ids.
cudaError_t launch_route_align(const RouteArgs &r, const AlignArgs &a, const ZeroArgs &z,
                               int zero_ctas, int sms, cudaStream_t s, int *launches);
cudaError_t launch_align(const AlignArgs &a, const ZeroArgs &z, int zero_ctas, cudaStream_t s,
                         int *launches);
cudaError_t launch_gather_rows(const uint16_t *x, const int32_t *sorted, const int32_t *npp, int P,
                               int top_k, int H, uint16_t *xs, size_t cap_rows, uint32_t *err,
                               int sms, cudaStream_t s, int *launches);
cudaError_t launch_finalize(const float *acc, uint16_t *out, size_t n, int sms, cudaStream_t s,
                            int *launches);
cudaError_t launch_pack(const uint8_t *q, const uint16_t *scales, int E, int N, int K,
                        int is_w13, void *packed, void *packed_scales, uint32_t *inexact,
                        cudaStream_t s);
cudaError_t launch_pack_mxfp4(const uint8_t *q, const uint8_t *scales, int E, int N, int K,
                              int is_w13, void *packed, void *packed_scales, uint32_t *bad,
                              cudaStream_t s);

// Packed weight geometry shared by the pack kernel and the GEMMs.
constexpr int kSlabRows = 128;
constexpr int kSlabK = 64;
constexpr int kSlabBytes = kSlabRows * kSlabK / 2;      // 4096
constexpr int kStageWBytes = 2 * kSlabBytes;            // 8192
constexpr int kStageSBytes = 2 * kSlabRows * 2 * 2;     // 1024
constexpr int kStageBytes = kStageWBytes + kStageSBytes;  // 9216

// Dequantisation constants (fp16 pairs and nibble masks), passed as kernel
// parameters so that they stay constant-bank operands instead of immediates
// the compiler re-materialises in registers for every use.
struct DequantConsts {
    uint32_t nib_mask;  // 0x03C003C0: a nibble at bits 6..9 of each half
    uint32_t magic16;   // fp16 pair (16, 16): with the nibble, the pair (16 + q)
    uint32_t cm24;      // fp16 pair (-24, -24): times the scale, the FMA's addend
};

// One of the two grouped GEMMs: g[0] the gate/up GEMM, g[1] the down GEMM.
struct GemmPhase {
    const uint8_t *wq;         // packed INT4 stages
    const uint8_t *wsc;        // packed scales
    int RT;                    // row tiles per expert
    int KSS, KS;               // k sub-stages per tile (one 8 KB packed stage each) and
                               // pipeline stages per tile (two sub-stages, the last maybe one)
};

struct GemmParams {
    GemmPhase g[2];            // the kernel runs g[kind - 1] (the fused kernel both, in turn)
    const int32_t *sorted_ids; // align output
    const int32_t *expert_ids;
    const int32_t *num_post_pad;
    const float *topk_weights; // down: [P]
    uint16_t *a_out;           // gate/up output, fp16 intermediate [rows][I]
    float *partial;            // gate/up split slots [G][2][2][BM][128]
    int32_t *tile_cnt;         // gate/up split counters [tiles]
    float *out_acc;            // down: fp32 accumulator [M][H]
    float4 *zero_out;          // gate/up: zeroes these zero_n16 16-byte units (the down
    size_t zero_n16;           // GEMM's accumulator) on the side; null: nothing
    uint32_t *err;             // [2]
    // fused kernel only: the gather of x and the hand-offs between CTAs
    const uint16_t *x;         // bf16 [M][H]
    uint16_t *x16;             // fp16 rows of x in bucketed order [cap][H]
    const int32_t *pos_of;     // [P]: each pair's row in x16 (-1: dropped), from the align
    int32_t *blk_done;         // [blocks]: gate/up tiles finished, per expert block
    int32_t *prep_done;        // [1]: CTAs done with their share of the gather and zeroing
    int M, top_k, H, I, P, E;
    int cap;                   // rows of sorted_ids, of the gathered x and of a_out
    int block_m;               // BM: routing block height (multiple of 16, <= 192)
    int n_w, n_b, n_a;         // ring depths: weight stages, B stages, A (TMEM) stages
    int ni;                    // MMA-issuing warps (= accumulators per buffer): 4 or 2
    int nbuf;                  // accumulator buffers (pieces alternate between them)
    int np;                    // A-slot release parts per stage: 1, or 2 (per sub-stage)
    int b_sub;                 // 1: B ring slots hold one sub-stage (wide blocks)
    int epi_f4;                // down: combine through shared memory as float4 adds
    int fmt;                   // weight format: MOE_W_INT4 or MOE_W_MXFP4 (picks the kernel)
    int round_robin;           // 1: whole waves of tiles round-robin, the rest split by stages
                               // (0: all split by stages)
    int skip_stage;            // debug-bounds builds: CTA 0 never issues the weight copy of
                               // its stage with this index (-1: none), so the wait for it
                               // runs out (the timeout test); ignored by other builds
    uint32_t b_stage_bytes;
    uint32_t smem_b_off, smem_misc_off, smem_bytes;
    DequantConsts dq;
};

// The INT4 dequantisation constants (see dequant_row).
inline DequantConsts int4_dequant_consts() {
    DequantConsts d;
    d.nib_mask = 0x03C003C0u;  // bits 6..9 of each half
    d.magic16 = 0x4C004C00u;   // fp16 16 in both halves
    d.cm24 = 0xCE00CE00u;      // fp16 -24 in both halves
    return d;
}

// kind 1: gate/up GEMM + SwiGLU; kind 2: down GEMM + weighted combine; kind 3:
// both in one persistent launch (the fused decode kernel: gather, gate/up, then
// down, blocks of at most 128 rows).  The tensor maps cover the B operand rows in
// bucketed order, 64-column x block_m-row boxes, 128-byte swizzle: tmap_x the fp16
// x rows (gate/up), tmap_a the fp16 intermediate (down); a kind uses its own.
cudaError_t launch_gemm(int kind, const GemmParams &p, const CUtensorMap *tmap_x,
                        const CUtensorMap *tmap_a, int grid, cudaStream_t s, int *launches);
// Fills the ring depths and shared-memory layout of p for the given kind.
bool plan_gemm_smem(int kind, GemmParams &p);

}  // namespace moe
