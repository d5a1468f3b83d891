// Align (bucket routing pairs by expert, pad buckets to the block height), the
// per-call zeroing of accumulators, and the final fp32 -> bf16 conversion.
//
// The align step turns the routed token batch into per-expert groups for the
// grouped GEMMs ("The Throughput Lever", section "The Result: Two Regimes": each
// token activates top-8 of the experts and the kernel works expert by expert).
// Output contract: for each expert in ascending order, the flat pair indices
// t*top_k+j routed to it in ascending order, then pad entries (value P) up to a
// multiple of block_m; one expert id per block; the total count.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "kernels.cuh"

namespace moe {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;

// Exclusive prefix sum over one value per thread of a 1024-thread block.
// `warp_tot` is shared scratch of 32 ints.  Returns the exclusive prefix and
// writes the block total to *total (all threads).
__device__ int block_exclusive_scan(int v, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += n;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int t = warp_tot[lane];
        int ti = t;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, ti, d);
            if (lane >= d) ti += n;
        }
        warp_tot[lane] = ti - t;  // exclusive prefix of warp totals
        if (lane == 31) warp_tot[32] = ti;
    }
    __syncthreads();
    int res = warp_tot[wid] + incl - v;
    *total = warp_tot[32];
    __syncthreads();
    return res;
}

// Given per-expert counts cnt[0..E) (shared), compute padded bucket offsets
// into off[0..E) (shared), write expert_ids, pad entries and num_post_pad, and
// add the dropped pairs to the error words (which accumulate until the caller
// clears them).  One 1024-thread block; E <= 1024.
__device__ void align_layout(const AlignArgs &a, const int *cnt, int *off, int *scan_tmp) {
    const int e = threadIdx.x;
    const int c = (e < a.E) ? cnt[e] : 0;
    const int pc = ((c + a.block_m - 1) / a.block_m) * a.block_m;
    int total = 0;
    const int o = block_exclusive_scan(pc, scan_tmp, &total);
    int valid_total = 0;
    block_exclusive_scan(c, scan_tmp, &valid_total);
    if (e < a.E) {
        off[e] = o;
        for (int b = o / a.block_m; b < (o + pc) / a.block_m; ++b) a.expert_ids[b] = e;
        for (int p = o + c; p < o + pc; ++p) a.sorted_ids[p] = a.P;
    }
    if (threadIdx.x == 0) {
        *a.num_post_pad = total;
        if (a.err) {
            const uint32_t dropped = (uint32_t)(a.P - valid_total);
            if (dropped) {
                atomicOr(&a.err[0], kErrBadExpert);
                atomicAdd(&a.err[1], dropped);
            }
        }
    }
}

// Place the pairs of items [i0, i0 + 1024) using per-expert running bases
// base[e] (shared, advanced on return).  wtab: shared [32][E] ints.  e_pre >= -1:
// this thread's item's id, already read (-2: read it here).  Only the warps
// that hold items take part in the per-expert running sums (one warp at a
// handful of pairs, where walking all 32 was most of the round).
__device__ void align_place_round(const AlignArgs &a, int i0, int *base, int *wtab,
                                  int e_pre = -2) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int items = (a.P - i0 < kAlignThreads) ? a.P - i0 : kAlignThreads;
    const int nw = (items + 31) / 32;  // warps with items
    for (int idx = threadIdx.x; idx < nw * a.E; idx += kAlignThreads) wtab[idx] = 0;
    __syncthreads();
    const int i = i0 + threadIdx.x;
    const int e = (e_pre >= -1) ? e_pre : (i < a.P) ? a.ids[i] : -1;
    const bool valid = (e >= 0) && (e < a.E);
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (valid && rank == 0) wtab[wid * a.E + e] = __popc(peers);
    __syncthreads();
    for (int ee = threadIdx.x; ee < a.E; ee += kAlignThreads) {
        int acc = base[ee];
        for (int w = 0; w < nw; ++w) {
            const int t = wtab[w * a.E + ee];
            wtab[w * a.E + ee] = acc;
            acc += t;
        }
        base[ee] = acc;
    }
    __syncthreads();
    if (valid) a.sorted_ids[wtab[wid * a.E + e] + rank] = i;
    if (a.pos_of && i < a.P) a.pos_of[i] = valid ? wtab[wid * a.E + e] + rank : -1;
    __syncthreads();
}

__device__ void zero_regions(const ZeroArgs &z, int cta, int nctas) {
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    const size_t stride = (size_t)nctas * blockDim.x;
    const size_t first = (size_t)cta * blockDim.x + threadIdx.x;
    for (int r = 0; r < 2; ++r) {
        float4 *p = reinterpret_cast<float4 *>(z.ptr[r]);
        const size_t n = z.n16[r];
        for (size_t idx = first; idx < n; idx += stride) p[idx] = zero;
    }
}

// Rows of x in bucketed order, as the fp16 tensor-core operand of the gate/up
// GEMM: xs[pos] = fp16(x[sorted_ids[pos] / top_k]) for every real entry (pad
// rows are left as they are; the GEMM ignores their results).  One warp per row.
// U: 16-byte loads in flight per lane.  A warp copies a row in ceil(H / (256 U))
// dependent memory round trips; where the rows are few (decode) that latency is
// the kernel's duration, so U = 16 (2 round trips at H = 7168); where there are
// many, U = 4 keeps the registers low enough for every block to be resident.
template <int U>
__global__ void gather_rows_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ sorted,
                                   const int32_t *__restrict__ num_post_pad, int P, int top_k, int H,
                                   uint16_t *__restrict__ xs, int cap, uint32_t *err) {
    pdl_wait();  // sorted_ids and num_post_pad come from the align launch
    // Only now may the gate/up GEMM start: its weight stream reads the align's
    // outputs without waiting for this kernel (it waits only before it reads
    // the gathered rows).
    pdl_launch_dependents();
    int npp = *num_post_pad;
    if (!bounds_ok(npp >= 0 && npp <= cap, err)) npp = 0;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    bool bad = false;
    for (int pos = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; pos < npp; pos += warps) {
        const int pair = sorted[pos];
        if (pair >= P) continue;  // a pad
        if (!bounds_ok(pair >= 0, err)) continue;
        gather_row<U>(x + (size_t)(pair / top_k) * H, xs + (size_t)pos * H, H, bad);
    }
    report_range(bad, err);
}

cudaError_t launch_gather_rows(const uint16_t *x, const int32_t *sorted, const int32_t *npp, int P,
                               int top_k, int H, uint16_t *xs, size_t cap_rows, uint32_t *err,
                               int sms, cudaStream_t s, int *launches) {
    size_t blocks = (cap_rows + 7) / 8;  // 8 warps (rows) per block
    if (blocks > (size_t)sms * 8) blocks = (size_t)sms * 8;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = pdl_config((unsigned)blocks, 256, 0, s);
    cudaLaunchAttribute attr;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl_attr(attr);
    const int cap = cap_rows > (size_t)INT32_MAX ? INT32_MAX : (int)cap_rows;
    // the U = 16 kernel keeps two 256-thread blocks per SM resident: use it
    // where the whole grid fits in that
    if (blocks <= (size_t)sms * 2)
        cudaLaunchKernelEx(&cfg, gather_rows_kernel<16>, x, sorted, npp, P, top_k, H, xs, cap, err);
    else
        cudaLaunchKernelEx(&cfg, gather_rows_kernel<4>, x, sorted, npp, P, top_k, H, xs, cap, err);
    if (launches) *launches += 1;
    return cudaGetLastError();
}

// Whole align in one block (P small).
__device__ void align_one_block(const AlignArgs &a, int *sm) {
    int *cnt = sm;                    // [E]
    int *base = cnt + a.E;            // [E]
    int *scan_tmp = base + a.E;       // [33]
    int *wtab = scan_tmp + 64;        // [32][E]
    for (int e = threadIdx.x; e < a.E; e += kAlignThreads) cnt[e] = 0;
    __syncthreads();
    int e_first = -1;  // this thread's id in the first round, kept for the placement
    for (int i = threadIdx.x; i < a.P; i += kAlignThreads) {
        const int e = a.ids[i];
        if (i == (int)threadIdx.x) e_first = e;
        if (e >= 0 && e < a.E) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    align_layout(a, cnt, base, scan_tmp);
    __syncthreads();
    for (int i0 = 0; i0 < a.P; i0 += kAlignThreads)
        align_place_round(a, i0, base, wtab, i0 == 0 ? e_first : -2);
}

// Whole align in one block (P small); blocks 1.. zero the accumulators.
__global__ void __launch_bounds__(kAlignThreads)
    align_fused_kernel(const AlignArgs a, const ZeroArgs z) {
    extern __shared__ int sm[];
    pdl_launch_dependents();  // the gather may set up; it waits for this grid
    if (blockIdx.x > 0) {
        zero_regions(z, blockIdx.x - 1, gridDim.x - 1);
        return;
    }
    align_one_block(a, sm);
}

// ------------------------------------------------------------------ router --
// "The Throughput Lever", section "The Result: Two Regimes": each token picks 8
// of 384 experts by top-8 routing.  One warp per token: lane l holds logits
// l, l + 32, ... (up to 32 of them, E <= 1024).  Each of the top_k rounds takes
// the warp's largest remaining logit (ties: the lower expert index), so the
// selection is decided by exact fp32 comparisons.  The weights are the softmax
// over the chosen logits, which equals the softmax over all E renormalised over
// the chosen k.  NaN logits rank as -inf.
__device__ void route_token(const RouteArgs &r, int t, int lane) {
    const float *lg = r.logits + (size_t)t * r.E;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int e = lane + 32 * i;
        const float x = (e < r.E) ? lg[e] : -INFINITY;
        v[i] = isnan(x) ? -INFINITY : x;
    }
    uint32_t taken = 0;
    float my_sel = 0.f, mx = 0.f;
    for (int j = 0; j < r.top_k; ++j) {
        float bv = -INFINITY;
        int be = 0x7fffffff;  // no candidate
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int e = lane + 32 * i;
            if (e < r.E && !((taken >> i) & 1u) && (be == 0x7fffffff || v[i] > bv)) {
                bv = v[i];
                be = e;
            }
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == j) my_sel = bv;
        if (j == 0) mx = bv;
        if (lane == 0) r.ids[(size_t)t * r.top_k + j] = be;
    }
    const float ex = (lane < r.top_k) ? expf(my_sel - mx) : 0.f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane < r.top_k) r.weights[(size_t)t * r.top_k + lane] = ex / sum;
}

__global__ void route_kernel(const RouteArgs r) {
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < r.M; t += warps)
        route_token(r, t, lane);
}

// Router and align in one launch (small routings): block 0 routes every token,
// then aligns its own output; blocks 1.. zero the accumulators.
__global__ void __launch_bounds__(kAlignThreads)
    route_align_fused_kernel(const RouteArgs r, const AlignArgs a, const ZeroArgs z) {
    extern __shared__ int sm[];
    pdl_launch_dependents();  // the gather may set up; it waits for this grid
    if (blockIdx.x > 0) {
        zero_regions(z, blockIdx.x - 1, gridDim.x - 1);
        return;
    }
    const int lane = threadIdx.x & 31;
    for (int t = threadIdx.x >> 5; t < r.M; t += kAlignWarps) route_token(r, t, lane);
    __syncthreads();  // the block's routed ids are visible to the whole block
    align_one_block(a, sm);
}

// Multi-block align, step 1: per-chunk histograms; extra blocks zero.
__global__ void __launch_bounds__(kAlignThreads)
    align_hist_kernel(const AlignArgs a, const ZeroArgs z) {
    extern __shared__ int sm[];
    if ((int)blockIdx.x < a.n_chunks) {
        int *cnt = sm;
        for (int e = threadIdx.x; e < a.E; e += kAlignThreads) cnt[e] = 0;
        __syncthreads();
        const int i = blockIdx.x * kAlignThreads + threadIdx.x;
        if (i < a.P) {
            const int e = a.ids[i];
            if (e >= 0 && e < a.E) atomicAdd(&cnt[e], 1);
        }
        __syncthreads();
        for (int e = threadIdx.x; e < a.E; e += kAlignThreads)
            a.chunk_tab[(size_t)blockIdx.x * a.E + e] = cnt[e];
    }
    zero_regions(z, blockIdx.x, gridDim.x);
}

// Step 2 (one block): bucket offsets, expert ids, pads; turns chunk_tab into
// per-chunk starting positions.
__global__ void __launch_bounds__(kAlignThreads) align_scan_kernel(const AlignArgs a) {
    extern __shared__ int sm[];
    int *cnt = sm;
    int *off = cnt + a.E;
    int *scan_tmp = off + a.E;
    for (int e = threadIdx.x; e < a.E; e += kAlignThreads) {
        int s = 0;
        for (int c = 0; c < a.n_chunks; ++c) s += a.chunk_tab[(size_t)c * a.E + e];
        cnt[e] = s;
    }
    __syncthreads();
    align_layout(a, cnt, off, scan_tmp);
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += kAlignThreads) {
        int run = off[e];
        for (int c = 0; c < a.n_chunks; ++c) {
            const int t = a.chunk_tab[(size_t)c * a.E + e];
            a.chunk_tab[(size_t)c * a.E + e] = run;
            run += t;
        }
    }
}

// Step 3: each block places its chunk.
__global__ void __launch_bounds__(kAlignThreads) align_scatter_kernel(const AlignArgs a) {
    extern __shared__ int sm[];
    pdl_launch_dependents();  // the gather may set up; it waits for this grid
    int *base = sm;            // [E]
    int *wtab = base + a.E;    // [32][E]
    for (int e = threadIdx.x; e < a.E; e += kAlignThreads)
        base[e] = a.chunk_tab[(size_t)blockIdx.x * a.E + e];
    __syncthreads();
    align_place_round(a, blockIdx.x * kAlignThreads, base, wtab);
}

// out[i] = bf16(acc[i]) (round to nearest even), 8 elements per step.
__global__ void finalize_kernel(const float *__restrict__ acc, uint16_t *__restrict__ out,
                                size_t n8) {
    pdl_wait();  // acc is the down GEMM's output
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
         i += (size_t)gridDim.x * blockDim.x) {
        const float4 a0 = reinterpret_cast<const float4 *>(acc)[2 * i];
        const float4 a1 = reinterpret_cast<const float4 *>(acc)[2 * i + 1];
        __nv_bfloat162 b0 = __floats2bfloat162_rn(a0.x, a0.y);
        __nv_bfloat162 b1 = __floats2bfloat162_rn(a0.z, a0.w);
        __nv_bfloat162 b2 = __floats2bfloat162_rn(a1.x, a1.y);
        __nv_bfloat162 b3 = __floats2bfloat162_rn(a1.z, a1.w);
        uint4 v;
        v.x = *reinterpret_cast<uint32_t *>(&b0);
        v.y = *reinterpret_cast<uint32_t *>(&b1);
        v.z = *reinterpret_cast<uint32_t *>(&b2);
        v.w = *reinterpret_cast<uint32_t *>(&b3);
        reinterpret_cast<uint4 *>(out)[i] = v;
    }
}

size_t align_smem_fused(int E) { return (size_t)(2 * E + 64 + kAlignWarps * E) * sizeof(int); }
size_t align_smem_scan(int E) { return (size_t)(2 * E + 64) * sizeof(int); }
size_t align_smem_scatter(int E) { return (size_t)(E + kAlignWarps * E) * sizeof(int); }

// Raises the dynamic shared-memory limit of the align kernels, once per device
// (under a lock: concurrent first calls from several host threads); a failure
// is returned, and not recorded as done.
static cudaError_t launch_align_attrs() {
    static std::mutex mu;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (attr_done[dev]) return cudaSuccess;
    const int maxs = (int)align_smem_fused(1024);
    const void *fns[] = {(const void *)align_fused_kernel, (const void *)align_hist_kernel,
                         (const void *)align_scan_kernel, (const void *)align_scatter_kernel,
                         (const void *)route_align_fused_kernel};
    for (const void *f : fns) {
        e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, maxs);
        if (e != cudaSuccess) return e;
    }
    attr_done[dev] = true;
    return cudaSuccess;
}

cudaError_t launch_align(const AlignArgs &a, const ZeroArgs &z, int zero_ctas,
                         cudaStream_t s, int *launches) {
    cudaError_t ea = launch_align_attrs();
    if (ea != cudaSuccess) return ea;
    if (a.n_chunks <= 0) {
        align_fused_kernel<<<1 + zero_ctas, kAlignThreads, align_smem_fused(a.E), s>>>(a, z);
        if (launches) *launches += 1;
    } else {
        align_hist_kernel<<<a.n_chunks + zero_ctas, kAlignThreads, (size_t)a.E * sizeof(int), s>>>(a, z);
        align_scan_kernel<<<1, kAlignThreads, align_smem_scan(a.E), s>>>(a);
        align_scatter_kernel<<<a.n_chunks, kAlignThreads, align_smem_scatter(a.E), s>>>(a);
        if (launches) *launches += 3;
    }
    return cudaGetLastError();
}

cudaError_t launch_route(const RouteArgs &r, int sms, cudaStream_t s, int *launches) {
    size_t blocks = ((size_t)r.M + 3) / 4;  // 4 warps (tokens) per block
    if (blocks > (size_t)sms * 16) blocks = (size_t)sms * 16;
    if (blocks < 1) blocks = 1;
    route_kernel<<<(unsigned)blocks, 128, 0, s>>>(r);
    if (launches) *launches += 1;
    return cudaGetLastError();
}

// Largest routing done by one block of the fused kernel (tokens): beyond one
// token per warp, spreading the router over many SMs is faster.
constexpr int kFusedRouteMaxTokens = kAlignWarps;  // one token per warp of the block

cudaError_t launch_route_align(const RouteArgs &r, const AlignArgs &a, const ZeroArgs &z,
                               int zero_ctas, int sms, cudaStream_t s, int *launches) {
    if (a.n_chunks <= 0 && r.M <= kFusedRouteMaxTokens) {
        cudaError_t e = launch_align_attrs();
        if (e != cudaSuccess) return e;
        route_align_fused_kernel<<<1 + zero_ctas, kAlignThreads, align_smem_fused(a.E), s>>>(r, a, z);
        if (launches) *launches += 1;
        return cudaGetLastError();
    }
    cudaError_t e = launch_route(r, sms, s, launches);
    if (e != cudaSuccess) return e;
    return launch_align(a, z, zero_ctas, s, launches);
}

cudaError_t launch_finalize(const float *acc, uint16_t *out, size_t n, int sms, cudaStream_t s,
                            int *launches) {
    const size_t n8 = n / 8;
    size_t blocks = (n8 + 255) / 256;
    if (blocks > (size_t)sms * 8) blocks = (size_t)sms * 8;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = pdl_config((unsigned)blocks, 256, 0, s);
    cudaLaunchAttribute attr;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl_attr(attr);
    cudaLaunchKernelEx(&cfg, finalize_kernel, acc, out, n8);
    if (launches) *launches += 1;
    return cudaGetLastError();
}

}  // namespace moe
