// Small-batch decode: the expert MLP as matrix-vector products, one routed pair
// at a time.
//
// "The Throughput Lever" (section "The Result: Two Regimes"): below a few hundred
// tokens per call the layer streams the touched experts' weights from memory.
// At a handful of pairs the tcgen05 GEMMs run one 16-column MMA per 128 weight
// rows, and their time is the per-stage latency of the dequant -> MMA -> release
// hand-off between warps, not memory.  Here every warp is on its own: it
// streams weight rows, dequantises them in registers with the GEMM kernels' fp16
// arithmetic (so the weights are bit-identical) and reduces them against the
// activation with register-operand MMAs (mma.sync m16n8k16, fp16 operands,
// fp32 accumulators: exact products, as on the tcgen05 path).  No align, no
// gather and no shared-memory weight tiles.
//
// A lane owns two weight rows (gate/up: the gate and the up row of one
// intermediate feature; down: two output rows 64 apart) and, per MMA, four
// consecutive k of each.  Its rows fill the A operand's rows g and g + 8 of the
// MMA (g = lane / 4); the B operand is block-diagonal: B[k'][n] holds the
// activation only where n = (k' mod 8) / 2, so column n of the result gathers
// the lanes 4g + n alone, and D[g][n], D[g + 8][n] are lane 4g + n's two dot
// products.  Only lanes with g == lane % 4 supply the activation; the others
// point at zeros.  One MMA covers 8 weights per lane, against 4 fp32 FMAs and
// 4 conversions per 4 weights on the plain CUDA-core dot product: about 1.7
// instructions per weight with the dequantisation, where that took 3.75.
//
//  * Gate/up kernel: CTA (k split, 128-feature tile, pair), pair fastest so the
//    pairs of one expert read the same weights close together in time; 4 warps
//    of 32 features.  Per-split partial sums go to a workspace buffer (one
//    writer each, no atomics).  It also zeroes the fp32 output accumulator.
//  * Down kernel (programmatic dependent launch): CTA (k split, 256 output
//    rows, pair); 4 warps of 64 rows.  It sums the gate/up partials of its k
//    range, forms the fp16 intermediate SiLU(g) * u (saturating, as the GEMM
//    epilogue does), and adds routing weight x result into the token's fp32
//    output row with float2 atomics.
//  * Per-block down kernel (the separate plan's down step at routing blocks of
//    at most 16 rows): CTA (k split, 256 output rows, align block); the block's
//    real rows of the gate/up intermediate take the activation's place, two rows
//    per MMA (columns 0..3 and 4..7).
// The k splits are chosen per call (moe_int4_forward): the grid of the small-
// batch kernels is about one wave of small CTAs over the SMs.
#include <cuda_fp16.h>

#include "dequant.cuh"
#include "kernels.cuh"
#include "gemv.cuh"

namespace moe {

namespace {

constexpr int kGvWarps = 4;
constexpr int kGvThreads = 32 * kGvWarps;
// One slab of loads in flight per warp ahead of the one being reduced, and six
// resident CTAs per SM (80 registers per thread): two slabs at five CTAs, or
// rings of 2-4 slabs in shared memory, measured slower.
constexpr int kGvAhead = 1;
constexpr int kGvMinCtas = 6;
// Shared memory of both kernels: 128 bytes of zeros (the B operand of the
// off-diagonal lanes), 64 bytes of padding so that the zeros and the
// activation rows sit in different banks, then the split's activation in fp16.
constexpr int kGvZeroBytes = 128;
constexpr int kGvActOffset = 192;

// 16 bytes of a weight stream, read once: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const uint8_t *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// A lane's two rows of one 64-k slab: 32 bytes each (two 16-byte halves 2048
// bytes apart) and each row's scale word (two fp16 group scales).
struct RowPair {
    uint4 lo0, hi0, lo1, hi1;
    uint32_t s0, s1;
};

__device__ __forceinline__ RowPair load_pair(const uint8_t *w0, const uint8_t *w1,
                                             const uint8_t *sc0, const uint8_t *sc1) {
    RowPair r;
    r.lo0 = ld_stream(w0);
    r.hi0 = ld_stream(w0 + kSlabBytes / 2);
    r.lo1 = ld_stream(w1);
    r.hi1 = ld_stream(w1 + kSlabBytes / 2);
    r.s0 = __ldg(reinterpret_cast<const uint32_t *>(sc0));
    r.s1 = __ldg(reinterpret_cast<const uint32_t *>(sc1));
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

// d += A * B for one m16n8k16 tile: fp16 A (four registers), fp16 B (two), fp32 d.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 64-k slab of the lane's two rows against 64 activations.  v0 / v1 hold
// the rows' fp16 pairs (v[c]: k = 2c, 2c + 1); xk points at the 64 fp16
// activations (diagonal lanes) or at 128 bytes of zeros (the others).  Each
// 16-byte activation load feeds two MMAs of four k each.
__device__ __forceinline__ void slab_mma(float (&d)[4], const uint32_t (&v0)[32],
                                         const uint32_t (&v1)[32], const uint8_t *xk) {
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint4 xb = *reinterpret_cast<const uint4 *>(xk + 16 * w);
        mma_f16_16816(d, v0[4 * w], v1[4 * w], v0[4 * w + 1], v1[4 * w + 1], xb.x, xb.y);
        mma_f16_16816(d, v0[4 * w + 2], v1[4 * w + 2], v0[4 * w + 3], v1[4 * w + 3], xb.z, xb.w);
    }
}

// Where a lane's two rows live: slab(kb) is the byte offset of 64-k slab kb
// from the rows' first slab, scale(kb) the same for the scale words.
template <class SlabOff, class ScaleOff>
struct RowPairSrc {
    const uint8_t *w0, *w1, *sc0, *sc1;
    SlabOff slab;
    ScaleOff scale;
    __device__ __forceinline__ RowPair load(int kb) const {
        return load_pair(w0 + slab(kb), w1 + slab(kb), sc0 + scale(kb), sc1 + scale(kb));
    }
};
template <class SlabOff, class ScaleOff>
__device__ __forceinline__ RowPairSrc<SlabOff, ScaleOff> row_pair_src(
    const uint8_t *w0, const uint8_t *w1, const uint8_t *sc0, const uint8_t *sc1, SlabOff slab,
    ScaleOff scale) {
    return {w0, w1, sc0, sc1, slab, scale};
}

// The first kGvAhead slabs' loads, issued before the activation is staged
// (the weights are call inputs, independent of it).
template <class Src>
__device__ __forceinline__ void prefetch_slabs(RowPair (&ring)[kGvAhead + 1], const Src &src,
                                               int kb0, int kb1) {
#pragma unroll
    for (int i = 0; i < kGvAhead; ++i)
        if (kb0 + i < kb1) ring[i] = src.load(kb0 + i);
}

// The k loop of one warp: slabs kb0 .. kb1 - 1 of the lane's two rows, with
// kGvAhead slabs of loads in flight ahead of the one being reduced (the first
// ones issued by prefetch_slabs).  act is the split's activation (kb0 first)
// or the zeros.
template <int FMT, class Src>
__device__ __forceinline__ void reduce_slabs(float (&d)[4], RowPair (&ring)[kGvAhead + 1],
                                             const Src &src, int kb0, int kb1,
                                             const uint8_t *act, bool diag,
                                             const DequantConsts &dq) {
#pragma unroll 1
    for (int kb = kb0; kb < kb1; ++kb) {
        if (kb + kGvAhead < kb1) ring[kGvAhead] = src.load(kb + kGvAhead);
        uint32_t v0[32], v1[32];
        dequant<FMT>(ring[0].lo0, ring[0].hi0, ring[0].s0, dq, v0);
        dequant<FMT>(ring[0].lo1, ring[0].hi1, ring[0].s1, dq, v1);
        slab_mma(d, v0, v1, diag ? act + (size_t)(kb - kb0) * 128 : act);
#pragma unroll
        for (int i = 0; i < kGvAhead; ++i) ring[i] = ring[i + 1];
    }
}

// Zeroes the 128 bytes at smem (threads 0..7).
__device__ __forceinline__ void zero_b_operand(uint8_t *smem) {
    if (threadIdx.x < kGvZeroBytes / 16)
        reinterpret_cast<uint4 *>(smem)[threadIdx.x] = make_uint4(0, 0, 0, 0);
}

template <int FMT>
__global__ void __launch_bounds__(kGvThreads, kGvMinCtas) gemv_gate_up_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    // the fp32 output accumulator, zeroed before the down kernel adds into it
    {
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        const size_t stride = (size_t)gridDim.x * blockDim.x;
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.out_n16; i += stride)
            reinterpret_cast<float4 *>(a.out)[i] = z;
    }
    pdl_launch_dependents();  // the down kernel may set up; it waits for this grid
    const int p = blockIdx.x % a.P;
    const int r = (blockIdx.x / a.P) % a.RT1;
    const int s = blockIdx.x / (a.P * a.RT1);
    const int kb0 = s * a.KBs;
    const int kb1 = (kb0 + a.KBs < a.KB) ? kb0 + a.KBs : a.KB;
    if (s >= a.SA || kb0 >= kb1) return;
    const int e = a.ids[p];
    if (e < 0 || e >= a.E) {  // dropped pair: counted once, as the align counts it
        if (s == 0 && r == 0 && threadIdx.x == 0 && a.err) {
            atomicOr(&a.err[0], kErrBadExpert);
            atomicAdd(&a.err[1], 1u);
        }
        return;
    }
    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = wid * 32 + lane;  // the feature's row in its 128-row slabs
    const size_t st0 = ((size_t)e * a.RT1 + r) * a.KB;
    const uint8_t *wg = a.w13 + st0 * kStageWBytes + row * 16;  // gate: slab 0 of each stage
    const uint8_t *sg = a.s13 + st0 * kStageSBytes + row * 4;
    const auto src = row_pair_src(
        wg, wg + kSlabBytes, sg, sg + kStageSBytes / 2,
        [](int kb) { return (size_t)kb * kStageWBytes; },
        [](int kb) { return (size_t)kb * kStageSBytes; });
    RowPair ring[kGvAhead + 1];
    prefetch_slabs(ring, src, kb0, kb1);
    // the split's k range of the token's x row as the fp16 operand
    const int t = p / a.top_k;
    bool bad = false;
    const uint32_t *xr = reinterpret_cast<const uint32_t *>(a.x + (size_t)t * a.H + kb0 * 64);
    uint32_t *xs = reinterpret_cast<uint32_t *>(smem + kGvActOffset);
    const int n2 = (kb1 - kb0) * 32;  // bf16 pairs of the range
    for (int c = threadIdx.x; c < n2; c += blockDim.x)
        xs[c] = bf16x2_to_f16x2_sat(__ldg(xr + c), bad);
    zero_b_operand(smem);
    report_range(bad, a.err);
    __syncthreads();
    const bool diag = (lane >> 2) == (lane & 3);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    reduce_slabs<FMT>(d, ring, src, kb0, kb1, diag ? smem + kGvActOffset : smem, diag, a.dq);
    // D[g][n] / D[g + 8][n] are lane 4g + n's gate / up sums: lanes with
    // lane % 4 < 2 hold n = 2 (lane % 4) and the next one
    if ((lane & 3) < 2) {
        const int src = (lane >> 2) * 4 + (lane & 3) * 2;  // the first of the two lanes
        const int feat = r * kSlabRows + wid * 32 + src;
        float *gu = a.gu + ((size_t)s * a.P + p) * 2 * a.I;
        *reinterpret_cast<float2 *>(gu + feat) = make_float2(d[0], d[1]);
        *reinterpret_cast<float2 *>(gu + a.I + feat) = make_float2(d[2], d[3]);
    }
}

template <int FMT>
__global__ void __launch_bounds__(kGvThreads, kGvMinCtas) gemv_down_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int tiles2 = (a.RT2 + 1) / 2;  // 256-row CTA tiles
    const int p = blockIdx.x % a.P;
    const int q = (blockIdx.x / a.P) % tiles2;
    const int s = blockIdx.x / (a.P * tiles2);
    const int kb0 = s * a.KB2s;
    const int kb1 = (kb0 + a.KB2s < a.KB2) ? kb0 + a.KB2s : a.KB2;
    if (s >= a.SB || kb0 >= kb1) return;
    const int e = a.ids[p];  // a call input: readable before the wait
    if (e < 0 || e >= a.E) return;
    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = 2 * q + (wid >> 1);  // the warp's 128-row tile
    const bool rows_in = r < a.RT2;
    const int row = (wid & 1) * 32 + lane;  // rows row and row + 64 of the tile's slabs
    const size_t st0 = ((size_t)e * a.RT2 + (rows_in ? r : 0)) * (a.KB2 / 2);
    const uint8_t *w = a.w2 + st0 * kStageWBytes + row * 16;
    const uint8_t *sc = a.s2 + st0 * kStageSBytes + row * 4;
    // 64-k block kb is slab kb % 2 of stage kb / 2
    const auto src = row_pair_src(
        w, w + 64 * 16, sc, sc + 64 * 4,
        [](int kb) { return (size_t)(kb >> 1) * kStageWBytes + (kb & 1) * kSlabBytes; },
        [](int kb) { return (size_t)(kb >> 1) * kStageSBytes + (kb & 1) * (kStageSBytes / 2); });
    RowPair ring[kGvAhead + 1];
    if (rows_in) prefetch_slabs(ring, src, kb0, kb1);  // weights: call inputs, before the wait
    pdl_wait();  // the gate/up partials and the zeroed output
    // the split's k range of the intermediate: fp16 SiLU(g) * u of the summed partials
    bool bad = false;
    uint32_t *as = reinterpret_cast<uint32_t *>(smem + kGvActOffset);
    const int n2 = (kb1 - kb0) * 32;  // fp16 pairs of the range
    const size_t split = (size_t)a.P * 2 * a.I;
    for (int c = threadIdx.x; c < n2; c += blockDim.x) {
        const float *gp = a.gu + (size_t)p * 2 * a.I + kb0 * 64 + 2 * c;
        float2 gs = make_float2(0.f, 0.f), us = make_float2(0.f, 0.f);
        for (int sa0 = 0; sa0 < a.SA; sa0 += 4) {  // four splits' loads at a time
            float2 gv[4], uv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool in = sa0 + j < a.SA;
                const float *g = gp + (size_t)(in ? sa0 + j : 0) * split;
                gv[j] = in ? __ldcg(reinterpret_cast<const float2 *>(g)) : make_float2(0.f, 0.f);
                uv[j] = in ? __ldcg(reinterpret_cast<const float2 *>(g + a.I))
                           : make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                gs.x += gv[j].x;
                gs.y += gv[j].y;
                us.x += uv[j].x;
                us.y += uv[j].y;
            }
        }
        const uint32_t lo = f16_sat(silu_mul(gs.x, us.x), bad);
        const uint32_t hi = f16_sat(silu_mul(gs.y, us.y), bad);
        as[c] = lo | (hi << 16);
    }
    zero_b_operand(smem);
    report_range(bad, a.err);
    __syncthreads();
    if (!rows_in) return;
    const bool diag = (lane >> 2) == (lane & 3);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    reduce_slabs<FMT>(d, ring, src, kb0, kb1, diag ? smem + kGvActOffset : smem, diag, a.dq);
    if ((lane & 3) < 2) {
        const int src = (lane >> 2) * 4 + (lane & 3) * 2;
        const int o = r * kSlabRows + (wid & 1) * 32 + src;  // output rows o, o + 1 (+ 64)
        const float tw = a.topk_weights[p];
        float *y = a.out + (size_t)(p / a.top_k) * a.H;
        atomicAdd(reinterpret_cast<float2 *>(y + o), make_float2(tw * d[0], tw * d[1]));
        atomicAdd(reinterpret_cast<float2 *>(y + o + 64), make_float2(tw * d[2], tw * d[3]));
    }
}

// ---------------------------------------------------------------- block down --
// The separate plan's down step at short routing blocks (up to 32 rows; the plan
// uses it at 16, where it measured faster than the down GEMM): per
// align block, a CTA streams 256 of the expert's down rows over its k split once
// and reduces them against the block's real rows of the gate/up intermediate,
// up to kBdRows at a time: MMA q takes rows 2q (result columns 0..3) and 2q + 1
// (columns 4..7) of the pass, through the same block-diagonal operand as above.
// Block rows per pass (two per MMA) and resident CTAs per SM (111 registers
// per thread); four rows at five CTAs ran alike, two at six were slower.
constexpr int kBdRows = 8;
constexpr int kBdMinCtas = 4;

// One slab against NQ row pairs of a pass.
template <int NQ>
__device__ __forceinline__ void slab_mma_rows(float (&d)[NQ][4], const uint32_t (&v0)[32],
                                              const uint32_t (&v1)[32],
                                              const uint8_t *const (&xk)[NQ]) {
#pragma unroll
    for (int w = 0; w < 8; ++w) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const uint4 xb = *reinterpret_cast<const uint4 *>(xk[q] + 16 * w);
            mma_f16_16816(d[q], v0[4 * w], v1[4 * w], v0[4 * w + 1], v1[4 * w + 1], xb.x, xb.y);
            mma_f16_16816(d[q], v0[4 * w + 2], v1[4 * w + 2], v0[4 * w + 3], v1[4 * w + 3], xb.z,
                          xb.w);
        }
    }
}

// The k loop of one warp against a pass's rows (act[q]: this lane's source for
// MMA q, slab kb0 first, or null for the zeros).
template <int FMT, int NQ, class Src>
__device__ __forceinline__ void reduce_rows(float (&d)[NQ][4], RowPair (&ring)[kGvAhead + 1],
                                            const Src &src, int kb0, int kb1,
                                            const uint8_t *const (&act)[NQ],
                                            const uint8_t *zeros, const DequantConsts &dq) {
#pragma unroll 1
    for (int kb = kb0; kb < kb1; ++kb) {
        if (kb + kGvAhead < kb1) ring[kGvAhead] = src.load(kb + kGvAhead);
        uint32_t v0[32], v1[32];
        dequant<FMT>(ring[0].lo0, ring[0].hi0, ring[0].s0, dq, v0);
        dequant<FMT>(ring[0].lo1, ring[0].hi1, ring[0].s1, dq, v1);
        const uint8_t *xk[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) xk[q] = act[q] ? act[q] + (size_t)(kb - kb0) * 128 : zeros;
        slab_mma_rows<NQ>(d, v0, v1, xk);
#pragma unroll
        for (int i = 0; i < kGvAhead; ++i) ring[i] = ring[i + 1];
    }
}

// One pass over nr <= 2 NQ rows of a block: the k loop, then routing weight x
// result into each row's token.  o is the lane's first output row.
template <int FMT, int NQ, class Src>
__device__ __forceinline__ void block_pass(const BlockDownArgs &a, RowPair (&ring)[kGvAhead + 1],
                                           const Src &src, int kb0, int kb1, uint8_t *smem,
                                           int span, const int *row_p, int nr, int o, int lane) {
    const int g = lane >> 2, j4 = lane & 3;
    const int slot = (g == j4) ? 0 : (g == j4 + 4) ? 1 : -1;
    const uint8_t *act[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        const int m = 2 * q + slot;
        act[q] = (slot >= 0 && m < nr) ? smem + kGvActOffset + (size_t)m * span : nullptr;
    }
    float d[NQ][4] = {};
    reduce_rows<FMT, NQ>(d, ring, src, kb0, kb1, act, smem, a.dq);
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        const int m = 2 * q + (j4 >> 1);
        if (m >= nr) continue;
        const int pm = row_p[m];
        const float tw = a.topk_weights[pm];
        float *y = a.out + (size_t)(pm / a.top_k) * a.H;  // output rows o, o + 1 (and + 64)
        atomicAdd(reinterpret_cast<float2 *>(y + o), make_float2(tw * d[q][0], tw * d[q][1]));
        atomicAdd(reinterpret_cast<float2 *>(y + o + 64), make_float2(tw * d[q][2], tw * d[q][3]));
    }
}

template <int FMT>
__global__ void __launch_bounds__(kGvThreads, kBdMinCtas) block_down_kernel(const BlockDownArgs a) {
    constexpr int NQ = kBdRows / 2;
    extern __shared__ __align__(16) uint8_t smem[];
    const int tiles2 = (a.RT2 + 1) / 2;  // 256-row CTA tiles
    const int b = blockIdx.x % a.blocks_cap;
    const int tq = (blockIdx.x / a.blocks_cap) % tiles2;
    const int s = blockIdx.x / (a.blocks_cap * tiles2);
    const int kb0 = s * a.KB2s;
    const int kb1 = (kb0 + a.KB2s < a.KB2) ? kb0 + a.KB2s : a.KB2;
    if (s >= a.SB || kb0 >= kb1) return;
    // The routing buffers: the align kernel has completed before any CTA of
    // this grid starts (the gate/up GEMM's predecessors wait for it before they
    // launch their dependents), so they are read before the wait, through L2.
    // (Debug-bounds builds record an out-of-range value and skip the block.)
    int npp = __ldcg(a.num_post_pad);
    if (!bounds_ok(npp >= 0 && npp <= a.cap && npp % a.block_m == 0, a.err)) npp = 0;
    if (b * a.block_m >= npp) return;
    const int e = __ldcg(a.expert_ids + b);
    if (!bounds_ok(e >= 0 && e < a.E, a.err) || e < 0 || e >= a.E) return;
    const int span = a.KB2s * 128;
    int *row_j = reinterpret_cast<int *>(smem + kGvActOffset + kBdRows * span);  // bucketed row
    int *row_p = row_j + 32;                                                       // its pair
    int *row_n = row_p + 32;
    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (wid == 0) {  // the block's real rows (block_m <= 32), in bucketed order
        const int j = b * a.block_m + lane;
        const int p = lane < a.block_m ? __ldcg(a.sorted_ids + j) : a.P;
        const bool real = bounds_ok(p >= 0, a.err) && p >= 0 && p < a.P;  // >= P: padding
        const uint32_t m = __ballot_sync(0xffffffffu, real);
        if (real) {
            const int pos = __popc(m & ((1u << lane) - 1u));
            row_j[pos] = j;
            row_p[pos] = p;
        }
        if (lane == 0) *row_n = __popc(m);
    }
    const int r = 2 * tq + (wid >> 1);  // the warp's 128-row tile
    const bool rows_in = r < a.RT2;
    const int row = (wid & 1) * 32 + lane;  // rows row and row + 64 of the tile's slabs
    const size_t st0 = ((size_t)e * a.RT2 + (rows_in ? r : 0)) * (a.KB2 / 2);
    const uint8_t *w = a.w2 + st0 * kStageWBytes + row * 16;
    const uint8_t *sc = a.s2 + st0 * kStageSBytes + row * 4;
    const auto src = row_pair_src(
        w, w + 64 * 16, sc, sc + 64 * 4,
        [](int kb) { return (size_t)(kb >> 1) * kStageWBytes + (kb & 1) * kSlabBytes; },
        [](int kb) { return (size_t)(kb >> 1) * kStageSBytes + (kb & 1) * (kStageSBytes / 2); });
    RowPair ring[kGvAhead + 1];
    if (rows_in) prefetch_slabs(ring, src, kb0, kb1);  // weights: call inputs, before the wait
    zero_b_operand(smem);
    pdl_wait();  // the intermediate and the zeroed accumulator
    __syncthreads();
    const int n = *row_n;
    const int o = r * kSlabRows + (wid & 1) * 32 + (lane >> 2) * 4 + (lane & 1) * 2;
    for (int c0 = 0; c0 < n; c0 += kBdRows) {
        const int nr = (n - c0 < kBdRows) ? n - c0 : kBdRows;
        // the pass's intermediate rows over the split's k range
        const int n16 = (kb1 - kb0) * 8;  // 16-byte pieces per row
        for (int c = threadIdx.x; c < nr * n16; c += blockDim.x) {
            const int m = c / n16, k16 = c - m * n16;
            const uint4 *ar = reinterpret_cast<const uint4 *>(
                a.a_out + (size_t)row_j[c0 + m] * a.I + kb0 * 64);
            reinterpret_cast<uint4 *>(smem + kGvActOffset + (size_t)m * span)[k16] =
                __ldcg(ar + k16);
        }
        __syncthreads();
        if (rows_in) {
            if (c0 > 0) prefetch_slabs(ring, src, kb0, kb1);  // a further pass re-streams
            // one variant per row-pair count: the MMAs stay unconditional
            const int nq = (nr + 1) / 2;
            if (nq == 1 || kBdRows <= 2)
                block_pass<FMT, 1>(a, ring, src, kb0, kb1, smem, span, row_p + c0, nr, o, lane);
            else if (nq == 2 || kBdRows <= 4)
                block_pass<FMT, (kBdRows >= 4 ? 2 : 1)>(a, ring, src, kb0, kb1, smem, span,
                                                        row_p + c0, nr, o, lane);
            else if (nq == 3 || kBdRows <= 6)
                block_pass<FMT, (kBdRows >= 6 ? 3 : 1)>(a, ring, src, kb0, kb1, smem, span,
                                                        row_p + c0, nr, o, lane);
            else
                block_pass<FMT, (kBdRows >= 8 ? 4 : 1)>(a, ring, src, kb0, kb1, smem, span,
                                                        row_p + c0, nr, o, lane);
        }
        __syncthreads();  // the staged rows are read before the next pass overwrites them
    }
}

}  // namespace

cudaError_t launch_gemv(const GemvArgs &a, int step, cudaStream_t s, int *launches) {
    if (step == 1) {  // gate/up: a plain launch (it overwrites the workspace partials)
        const int ga = a.P * a.RT1 * a.SA;
        const size_t sma = kGvActOffset + (size_t)a.KBs * 64 * 2;
        if (sma > 48 * 1024) return cudaErrorInvalidValue;
        if (a.fmt == 1)
            gemv_gate_up_kernel<1><<<ga, kGvThreads, sma, s>>>(a);
        else
            gemv_gate_up_kernel<0><<<ga, kGvThreads, sma, s>>>(a);
        const cudaError_t e = cudaGetLastError();
        if (e == cudaSuccess && launches) *launches += 1;
        return e;
    }
    const int gb = a.P * ((a.RT2 + 1) / 2) * a.SB;
    const size_t smb = kGvActOffset + (size_t)a.KB2s * 64 * 2;
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

cudaError_t launch_block_down(const BlockDownArgs &a, cudaStream_t s, int *launches) {
    static_assert(kBdRows == 2 || kBdRows == 4 || kBdRows == 6 || kBdRows == 8, "rows per pass");
    if (a.block_m > 32 || a.blocks_cap <= 0) return cudaErrorInvalidValue;
    const int grid = a.blocks_cap * ((a.RT2 + 1) / 2) * a.SB;
    const size_t smem = kGvActOffset + (size_t)kBdRows * a.KB2s * 128 + 96 * sizeof(int);
    if (smem > 48 * 1024) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = pdl_config((unsigned)grid, kGvThreads, smem, s);
    cudaLaunchAttribute attr;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl_attr(attr);
    const cudaError_t e = (a.fmt == 1) ? cudaLaunchKernelEx(&cfg, block_down_kernel<1>, a)
                                       : cudaLaunchKernelEx(&cfg, block_down_kernel<0>, a);
    if (e != cudaSuccess) return e;
    if (launches) *launches += 1;
    return cudaGetLastError();
}

}  // namespace moe
