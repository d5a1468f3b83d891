// Expert-parallel data movement ("From PCIe to NVLink", section "Part I: Laying
// the Foundation": the experts sharded over the GPUs, EP8 / EP4).  Around the
// all-to-all exchanges of an expert-parallel layer, a rank gathers the x rows it
// sends (one per routed pair, in send order) and, once the expert outputs come
// back, adds each returned row into its token's output row.  Both are plain
// row copies / row reductions over global memory: one warp per row, 16-byte
// accesses, a grid of a few waves over the SMs.
#include "kernels.cuh"
#include "moe_int4.h"

namespace moe {

namespace {

// dst[i] = src[rows[i]] for 2-byte rows of H elements (H a multiple of 8).
__global__ void ep_gather_kernel(const uint16_t *__restrict__ src, const int32_t *__restrict__ rows,
                                 int n, int H, int src_rows, uint16_t *__restrict__ dst,
                                 uint32_t *bad) {
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    const int n8 = H / 8;
    for (int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < n; i += warps) {
        const int r = rows[i];
        uint4 *d = reinterpret_cast<uint4 *>(dst + (size_t)i * H);
        if (r < 0 || r >= src_rows) {  // an index outside the source: the row is zeroed
            if (lane == 0 && bad) atomicOr(bad, 1u);
            for (int c = lane; c < n8; c += 32) d[c] = make_uint4(0, 0, 0, 0);
            continue;
        }
        const uint4 *s = reinterpret_cast<const uint4 *>(src + (size_t)r * H);
        for (int c = lane; c < n8; c += 32) d[c] = __ldg(s + c);
    }
}

// out[rows[i]] += src[i] for fp32 rows of H elements (H a multiple of 4); rows
// may repeat, so the adds are atomic (float4 reductions).
__global__ void ep_combine_kernel(const float *__restrict__ src, const int32_t *__restrict__ rows,
                                  int n, int H, int out_rows, float *__restrict__ out,
                                  uint32_t *bad) {
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    const int n4 = H / 4;
    for (int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < n; i += warps) {
        const int r = rows[i];
        if (r < 0 || r >= out_rows) {  // dropped, and reported
            if (lane == 0 && bad) atomicOr(bad, 1u);
            continue;
        }
        const float4 *s = reinterpret_cast<const float4 *>(src + (size_t)i * H);
        float4 *o = reinterpret_cast<float4 *>(out + (size_t)r * H);
        for (int c = lane; c < n4; c += 32) atomicAdd(o + c, __ldg(s + c));
    }
}

int grid_for(int n, cudaStream_t) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int per_block = 8;  // warps (rows) per 256-thread block
    int blocks = (n + per_block - 1) / per_block;
    if (blocks > sms * 8) blocks = sms * 8;
    return blocks < 1 ? 1 : blocks;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

}  // namespace moe

extern "C" {

int moe_ep_gather(const uint16_t *src, int src_rows, const int32_t *rows, int n, int H,
                  uint16_t *dst, uint32_t *bad, moe_stream_t stream) {
    if (n < 0 || H <= 0 || src_rows < 0) return MOE_ERR_SHAPE;
    if (n == 0) return MOE_OK;
    if (!src || !rows || !dst) return MOE_ERR_NULL;
    if (H % 8) return MOE_ERR_SHAPE;
    if (!moe::aligned16(src) || !moe::aligned16(dst)) return MOE_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    moe::ep_gather_kernel<<<moe::grid_for(n, s), 256, 0, s>>>(src, rows, n, H, src_rows, dst, bad);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_ep_combine(const float *src, const int32_t *rows, int n, int H, float *out, int out_rows,
                   uint32_t *bad, moe_stream_t stream) {
    if (n < 0 || H <= 0 || out_rows < 0) return MOE_ERR_SHAPE;
    if (n == 0) return MOE_OK;
    if (!src || !rows || !out) return MOE_ERR_NULL;
    if (H % 4) return MOE_ERR_SHAPE;
    if (!moe::aligned16(src) || !moe::aligned16(out)) return MOE_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    moe::ep_combine_kernel<<<moe::grid_for(n, s), 256, 0, s>>>(src, rows, n, H, out_rows, out, bad);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
