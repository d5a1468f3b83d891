// Small-batch decode on the CUDA cores: the expert MLP as matrix-vector
// products, one routed pair at a time.
//
// "The Throughput Lever" (section "The Result: Two Regimes"): below a few hundred
// tokens per call the layer streams the touched experts' weights from memory.
// At a handful of pairs the tensor-core GEMMs run one 16-column MMA per 128
// weight rows, and their time is the per-stage latency of the dequant -> MMA ->
// release loop, not memory.  Here every lane owns one weight row and streams it:
// 32 lanes read 32 consecutive rows' 16-byte pieces of the packed layout, one
// coalesced 512-byte read per warp, dequantise them in registers with the same
// fp16 arithmetic as the GEMM kernels (so the weights are bit-identical), and
// accumulate fp16 weight x fp16 activation products in fp32 (exact products, as
// on the tensor cores).  No align and no gather: a pair's token row is read
// directly.
//
//  * Gate/up kernel: CTA (pair, k split, group of 4 row tiles), 16 warps = 4
//    tiles x 4 lane quadrants of 32 rows.  A lane computes the gate and the up
//    dot products of one intermediate feature over the split's k range and
//    writes them to a per-split partial buffer (no atomics: every (split, pair,
//    feature) has one writer).  It also zeroes the fp32 output accumulator.
//  * Down kernel (programmatic dependent launch): CTA (pair, k split, group of
//    4 output row tiles).  It sums the gate/up partials of its k range, forms
//    the fp16 intermediate SiLU(g) * u (saturating, as the GEMM epilogue does),
//    then a lane computes one output feature's dot product over the range and
//    adds routing weight x result into the token's fp32 output row.
// The k splits give every SM tens of warps with loads in flight; their count
// is chosen per call (moe_int4_forward) so the grid covers the SMs.
#include <cuda_fp16.h>

#include "dequant.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kGvThreads = 512;  // 16 warps: 4 row tiles x 4 lane quadrants

// 16 bytes of a weight stream, read once: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const uint8_t *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// One lane's row of one packed stage: two 64-k slab rows (32 bytes each, in two
// 16-byte halves 2048 bytes apart) and their two scale words.
struct RowLoad {
    uint4 a_lo, a_hi, b_lo, b_hi;
    uint32_t sa, sb;
};

__device__ __forceinline__ RowLoad load_row(const uint8_t *w, const uint8_t *sc) {
    RowLoad r;
    r.a_lo = ld_stream(w);
    r.a_hi = ld_stream(w + 2048);
    r.b_lo = ld_stream(w + kSlabBytes);
    r.b_hi = ld_stream(w + kSlabBytes + 2048);
    r.sa = __ldg(reinterpret_cast<const uint32_t *>(sc));
    r.sb = __ldg(reinterpret_cast<const uint32_t *>(sc + kStageSBytes / 2));
    return r;
}

template <int FMT>
__device__ __forceinline__ void dequant(const uint4 lo, const uint4 hi, uint32_t sc,
                                        const DequantConsts &k, uint32_t (&v)[32]) {
    if (FMT == 1)
        dequant_row_fp4(lo, hi, sc, v);
    else
        dequant_row(lo, hi, sc, k, v);
}

// acc += sum over 64 k of w[k] * x[k]: v holds the 64 fp16 weights as pairs
// (k = 2c low, 2c + 1 high), xs the 64 activations.
__device__ __forceinline__ float dot64(const uint32_t (&v)[32], const float *xs, float acc) {
    const float4 *x4 = reinterpret_cast<const float4 *>(xs);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const float4 xv = x4[c];
        const float2 w0 = __half22float2(as_h2(v[2 * c]));
        const float2 w1 = __half22float2(as_h2(v[2 * c + 1]));
        acc = fmaf(w0.x, xv.x, acc);
        acc = fmaf(w0.y, xv.y, acc);
        acc = fmaf(w1.x, xv.z, acc);
        acc = fmaf(w1.y, xv.w, acc);
    }
    return acc;
}

template <int FMT>
__global__ void __launch_bounds__(kGvThreads) gemv_gate_up_kernel(const GemvArgs a) {
    extern __shared__ float xs[];  // the split's k range of x: fp32 of the fp16 operand
    // the fp32 output accumulator, zeroed before the down kernel adds into it
    {
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        const size_t stride = (size_t)gridDim.x * blockDim.x;
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.out_n16; i += stride)
            reinterpret_cast<float4 *>(a.out)[i] = z;
    }
    pdl_launch_dependents();  // the down kernel may set up; it waits for this grid
    const int tgroups = (a.RT1 + 3) / 4;
    const int per_pair = a.SA * tgroups;
    const int p = blockIdx.x / per_pair;
    const int s = (blockIdx.x % per_pair) / tgroups, tg = blockIdx.x % tgroups;
    const int kb0 = s * a.KBs;
    const int kb1 = (kb0 + a.KBs < a.KB) ? kb0 + a.KBs : a.KB;
    if (p >= a.P || kb0 >= kb1) return;
    const int e = a.ids[p];
    if (e < 0 || e >= a.E) {  // dropped pair: counted once, as the align counts it
        if (s == 0 && tg == 0 && threadIdx.x == 0 && a.err) {
            atomicOr(&a.err[0], kErrBadExpert);
            atomicAdd(&a.err[1], 1u);
        }
        return;
    }
    const int t = p / a.top_k;
    bool bad = false;
    const uint32_t *xr = reinterpret_cast<const uint32_t *>(a.x + (size_t)t * a.H + kb0 * 64);
    const int n2 = (kb1 - kb0) * 32;  // bf16 pairs of the range
    for (int c = threadIdx.x; c < n2; c += blockDim.x) {
        const float2 f = __half22float2(as_h2(bf16x2_to_f16x2_sat(__ldg(xr + c), bad)));
        xs[2 * c] = f.x;
        xs[2 * c + 1] = f.y;
    }
    report_range(bad, a.err);
    __syncthreads();
    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = tg * 4 + (wid >> 2);
    if (r >= a.RT1) return;
    const int row = (wid & 3) * 32 + lane;
    const size_t st0 = ((size_t)e * a.RT1 + r) * a.KB;
    const uint8_t *wrow = a.w13 + st0 * kStageWBytes + row * 16;
    const uint8_t *srow = a.s13 + st0 * kStageSBytes + row * 4;
    float g = 0.f, u = 0.f;
    // two k blocks of loads in flight while one is computed
    RowLoad cur = load_row(wrow + (size_t)kb0 * kStageWBytes, srow + (size_t)kb0 * kStageSBytes);
    RowLoad nxt = cur;
    if (kb0 + 1 < kb1)
        nxt = load_row(wrow + (size_t)(kb0 + 1) * kStageWBytes,
                       srow + (size_t)(kb0 + 1) * kStageSBytes);
#pragma unroll 1
    for (int kb = kb0; kb < kb1; ++kb) {
        RowLoad nn = nxt;
        if (kb + 2 < kb1)
            nn = load_row(wrow + (size_t)(kb + 2) * kStageWBytes,
                          srow + (size_t)(kb + 2) * kStageSBytes);
        const float *x = xs + (kb - kb0) * 64;
        uint32_t v[32];
        dequant<FMT>(cur.a_lo, cur.a_hi, cur.sa, a.dq, v);  // gate row
        g = dot64(v, x, g);
        dequant<FMT>(cur.b_lo, cur.b_hi, cur.sb, a.dq, v);  // up row
        u = dot64(v, x, u);
        cur = nxt;
        nxt = nn;
    }
    float *gu = a.gu + ((size_t)s * a.P + p) * 2 * a.I;
    const int feat = r * kSlabRows + row;
    gu[feat] = g;
    gu[a.I + feat] = u;
}

template <int FMT>
__global__ void __launch_bounds__(kGvThreads) gemv_down_kernel(const GemvArgs a) {
    extern __shared__ float av[];  // the split's k range of the intermediate (fp16 values)
    const int tgroups = (a.RT2 + 3) / 4;
    const int per_pair = a.SB * tgroups;
    const int p = blockIdx.x / per_pair;
    const int s = (blockIdx.x % per_pair) / tgroups, tg = blockIdx.x % tgroups;
    const int ks0 = s * a.KS2s;
    const int ks1 = (ks0 + a.KS2s < a.KS2) ? ks0 + a.KS2s : a.KS2;
    if (p >= a.P || ks0 >= ks1) return;
    const int e = a.ids[p];  // a call input: readable before the wait
    if (e < 0 || e >= a.E) return;
    pdl_wait();  // the gate/up partials and the zeroed output
    bool bad = false;
    const int n = (ks1 - ks0) * 2 * kSlabK;
    for (int c = threadIdx.x; c < n; c += blockDim.x) {
        const int i = ks0 * 2 * kSlabK + c;
        const float *gp = a.gu + (size_t)p * 2 * a.I + i;
        const size_t split = (size_t)a.P * 2 * a.I;
        float gs = 0.f, us = 0.f;
        for (int sa0 = 0; sa0 < a.SA; sa0 += 8) {  // eight splits' loads at a time
            float gv[8], uv[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const bool in = sa0 + q < a.SA;
                gv[q] = in ? __ldcg(gp + (sa0 + q) * split) : 0.f;
                uv[q] = in ? __ldcg(gp + (sa0 + q) * split + a.I) : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                gs += gv[q];
                us += uv[q];
            }
        }
        av[c] = __half2float(__ushort_as_half(f16_sat(silu_mul(gs, us), bad)));
    }
    report_range(bad, a.err);
    __syncthreads();
    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = tg * 4 + (wid >> 2);
    if (r >= a.RT2) return;
    const int row = (wid & 3) * 32 + lane;
    const size_t st0 = ((size_t)e * a.RT2 + r) * a.KS2;
    const uint8_t *wrow = a.w2 + st0 * kStageWBytes + row * 16;
    const uint8_t *srow = a.s2 + st0 * kStageSBytes + row * 4;
    float y = 0.f;
    RowLoad cur = load_row(wrow + (size_t)ks0 * kStageWBytes, srow + (size_t)ks0 * kStageSBytes);
    RowLoad nxt = cur;
    if (ks0 + 1 < ks1)
        nxt = load_row(wrow + (size_t)(ks0 + 1) * kStageWBytes,
                       srow + (size_t)(ks0 + 1) * kStageSBytes);
#pragma unroll 1
    for (int ks = ks0; ks < ks1; ++ks) {
        RowLoad nn = nxt;
        if (ks + 2 < ks1)
            nn = load_row(wrow + (size_t)(ks + 2) * kStageWBytes,
                          srow + (size_t)(ks + 2) * kStageSBytes);
        const float *x = av + (ks - ks0) * 2 * kSlabK;
        uint32_t v[32];
        dequant<FMT>(cur.a_lo, cur.a_hi, cur.sa, a.dq, v);  // k block 2 ks
        y = dot64(v, x, y);
        dequant<FMT>(cur.b_lo, cur.b_hi, cur.sb, a.dq, v);  // k block 2 ks + 1
        y = dot64(v, x + kSlabK, y);
        cur = nxt;
        nxt = nn;
    }
    const int t = p / a.top_k;
    atomicAdd(a.out + (size_t)t * a.H + r * kSlabRows + row, a.topk_weights[p] * y);
}

}  // namespace

cudaError_t launch_gemv(const GemvArgs &a, int step, cudaStream_t s, int *launches) {
    if (step == 1) {  // gate/up: a plain launch (it overwrites the workspace partials)
        const int ga = a.P * a.SA * ((a.RT1 + 3) / 4);
        const size_t sma = (size_t)a.KBs * 64 * sizeof(float);
        if (sma > 48 * 1024) return cudaErrorInvalidValue;
        if (a.fmt == 1)
            gemv_gate_up_kernel<1><<<ga, kGvThreads, sma, s>>>(a);
        else
            gemv_gate_up_kernel<0><<<ga, kGvThreads, sma, s>>>(a);
        const cudaError_t e = cudaGetLastError();
        if (e == cudaSuccess && launches) *launches += 1;
        return e;
    }
    const int gb = a.P * a.SB * ((a.RT2 + 3) / 4);
    const size_t smb = (size_t)a.KS2s * 2 * kSlabK * sizeof(float);
    if (smb > 48 * 1024) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = pdl_config((unsigned)gb, kGvThreads, smb, s);
    cudaLaunchAttribute attr;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl_attr(attr);
    const cudaError_t e = (a.fmt == 1) ? cudaLaunchKernelEx(&cfg, gemv_down_kernel<1>, a)
                                       : cudaLaunchKernelEx(&cfg, gemv_down_kernel<0>, a);
    if (e != cudaSuccess) return e;
    if (launches) *launches += 1;
    return cudaGetLastError();
}

}  // namespace moe
