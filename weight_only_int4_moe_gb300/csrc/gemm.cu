// Grouped INT4 GEMMs of the MoE expert MLP on tcgen05 tensor cores (sm_103a).
//
// "The Throughput Lever" (sections "Phase 3: The INT4 Marlin MoE Throughput
// Lever" and "The Result: Two Regimes") measures the grouped INT4 MoE GEMM: below
// a few hundred tokens per call it streams the touched experts' weights from
// memory and its time grows with the number of active experts; above, every
// expert is streamed once and extra tokens ride along.  One kernel design serves
// both regimes:
//
//  * Swap-AB: the MMA's M side (128 lanes of tensor memory) is 128 weight rows,
//    its N side is the tokens routed to one expert block (16..192, the block's
//    real row count rounded up to 16), so a decode call with one token per expert
//    streams each touched weight once and wastes no weight traffic.
//  * A pipeline stage is two k sub-stages of two 128x64 INT4 slabs each (16 KB,
//    plus 2 KB of fp16 scales), stored contiguously by the pack step.  Two
//    producer threads fetch a stage with one bulk TMA copy each (weights and
//    scales), so the weight stream reaches HBM speed with few, large requests.
//  * Three teams of four dequant warps take stages in turn; each warp covers
//    its 32-row lane quadrant of both slabs and both sub-stages, turning the
//    packed words into fp16 weights (q-8)*s -- a shift and a mask/OR that put
//    the nibble into the mantissa of fp16 16, then one FMA (v*s - 24s, exact),
//    two weights per instruction -- and storing them into tensor memory, which
//    tcgen05.mma reads as its A operand.
//  * The B operand (fp16 activations) sits in shared memory in the 128-byte-
//    swizzled K-major layout, fetched by 2-D TMA tensor copies of rows in
//    bucketed order: x gathered once per call into that order (gate/up), the
//    intermediate (down).
//  * Accumulators live in tensor memory, in two alternating buffers where it
//    has room, so the MMAs of the next piece run while dedicated epilogue warps
//    read the previous one.  gate/up keeps the gate and up rows of the same
//    128 intermediate features in the same lanes, so the epilogue forms
//    SiLU(g)*u in registers and writes the fp16 intermediate.  The down
//    epilogue scales by the routing weight and adds into the fp32 [M][H]
//    output (the top-k combine), through shared memory as float4 adds (four
//    features of one token per lane) where there is room: a lane holds one
//    feature of many tokens, and scalar adds would cost one reduction request
//    per token.  Wide gate/up (one accumulator buffer) has the idle issuing
//    warps take half of each full piece's SwiGLU columns.
//  * Work = (expert block, 128-row tile) x stages on a persistent grid of one
//    CTA per SM.  Whole waves of tiles go round-robin (CTA c takes tiles c,
//    c + G, ...), so the CTAs running at one time share a few expert blocks and
//    re-read each block's B operand from L2 rather than from memory; the last
//    one to two waves' worth of tiles is split evenly over the CTAs by stages
//    (a CTA's range may cut a tile).  A gate/up tile cut between CTAs is
//    finished by whichever piece arrives last (partial sums in per-CTA slots +
//    a counter); no CTA ever waits for another.
//
// Warp roles (768 threads): 0 weight producer, 1 TMEM owner (in gate/up it
// also zeroes the down GEMM's fp32 accumulator; with blocks of up to 128 rows
// it then waits for each stage's B slot on the issuers' behalf), 2 B loader,
// 3 scale producer, 4-15 dequant (three teams), 16-19 MMA issue, 20-23
// epilogue.  Each (slab, sub-stage) has its own issuing warp and accumulator
// (the epilogue sums them): one thread issuing tcgen05.mma waits tens of
// cycles per instruction while MMAs from several warps overlap.  At decode
// sizes the issuers' per-stage path (barrier, MMAs, commits) sets the stage
// rate, so it is kept short.  Every mbarrier wait is bounded
// (MOE_DEVERR_TIMEOUT).
#include <cuda_fp16.h>

#include <mutex>

#include "dequant.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kThreads = 768;
constexpr int kTmemCols = 512;
constexpr int kTeams = 3;                        // dequant teams, taking stages in turn
constexpr int kTeamWarps = 4;                    // dequant warps per team (one per lane quadrant)
constexpr int kDequantWarps = kTeams * kTeamWarps;
constexpr int kFirstDequantWarp = 4;
constexpr int kFirstIssuerWarp = kFirstDequantWarp + kDequantWarps;  // 16..19: MMA issue
constexpr int kFirstEpilogueWarp = kFirstIssuerWarp + 4;             // 20..23: epilogue
static_assert(kFirstEpilogueWarp + 4 == kThreads / 32, "warp roles fill the block");
constexpr uint32_t kStageW = 2 * kStageWBytes;  // 16 KB of INT4 per stage
constexpr uint32_t kStageS = 2 * kStageSBytes;  // 2 KB of scales per stage
constexpr uint32_t kStage = kStageW + kStageS;  // 18 KB
constexpr uint32_t kACols = 128;                // TMEM columns per A stage
// Hardware named barriers (0 is __syncthreads).  A hardware barrier cannot give
// up, so each is used only where every participant is certain to arrive (see
// the dequant role for the A-slot hand-off).
constexpr uint32_t kBarEpi = 1;     // the four epilogue warps
constexpr uint32_t kBarSlot0 = 2;   // A stage s written: its team arrives; the issuers and
                                    // (narrow blocks) warp 1 wait (ids 2..4: one per A
                                    // stage or stage half)
constexpr uint32_t kBarPrep = 5;    // fused kernel: the gather and zeroing warps (1, 4..23)
constexpr uint32_t kGatherWarps = 20;  // fused kernel: warps 4..23 gather before their roles
constexpr uint32_t kPrepThreads = (1 + kGatherWarps) * 32;
// The dequant teams' wait for a free A slot gives up only after this many
// cycles, far longer than any other wait (see the dequant role).
constexpr long long kSlotWaitCycles = 16 * kWaitTimeoutCycles;

// The schedule: tiles [0, rr) round-robin (whole tiles, CTA c takes c, c + G,
// ...), then tiles [rr, tiles) split evenly by stages.  Stage indices of the
// split part count from its first tile.  rr is a whole number of waves, one
// fewer than fit, so the split part holds between G and 2G - 1 tiles and
// balances the end; with fewer than 2G tiles everything is split.
struct Sched {
    long long start, end;  // this CTA's stage range within the split part
    long long T;           // stages of the split part
    int tiles, rr, KS, G, cta;
};

__device__ __forceinline__ Sched make_sched(const GemmParams &p, const GemmPhase &g) {
    Sched s;
    int npp = __ldcg(p.num_post_pad);
    if (!bounds_ok(npp >= 0 && npp <= p.cap && npp % p.block_m == 0, p.err)) npp = 0;
    s.tiles = (npp / p.block_m) * g.RT;
    s.KS = g.KS;
    s.G = gridDim.x;
    s.cta = blockIdx.x;
    const int waves = s.tiles / s.G;
    s.rr = (p.round_robin && waves >= 2) ? (waves - 1) * s.G : 0;
    s.T = (long long)(s.tiles - s.rr) * s.KS;
    s.start = (s.T * s.cta) / s.G;
    s.end = (s.T * (s.cta + 1)) / s.G;
    return s;
}

struct PieceIter {
    long long it;
    int next_tile;
    __device__ void init(const Sched &s) {
        it = s.start;
        next_tile = s.cta;
    }
    __device__ bool next(const Sched &s, int &tile, int &kb0, int &kb1) {
        if (next_tile < s.rr) {
            tile = next_tile;
            kb0 = 0;
            kb1 = s.KS;
            next_tile += s.G;
            return true;
        }
        if (it >= s.end) return false;
        tile = s.rr + (int)(it / s.KS);
        kb0 = (int)(it % s.KS);
        const long long rem = s.end - it;
        kb1 = (s.KS - kb0 <= rem) ? s.KS : kb0 + (int)rem;
        it += kb1 - kb0;
        return true;
    }
};

// First stage index of CTA c and the CTA owning stage `it` (split part).
__device__ __forceinline__ long long range_start(long long T, int G, int c) {
    return (T * c) / G;
}
__device__ __forceinline__ int range_owner(long long T, int G, long long it) {
    return (int)(((it + 1) * G - 1) / T);
}

// Number of real (non-pad) rows of a block: pads are at the end of a block.
__device__ __forceinline__ int block_rows(const int32_t *sorted, int pos0, int BM, int P) {
    const int lane = threadIdx.x & 31;
    int cnt = 0;
    for (int j = lane; j < BM; j += 32) cnt += (__ldcg(sorted + pos0 + j) < P) ? 1 : 0;
    return __reduce_add_sync(0xffffffffu, cnt);
}

// block_rows in two halves, so that the issuing warps can load a block's
// entries one piece ahead: each lane's entries (up to 6, blocks of <= 192
// rows), then their count of real rows.
struct RowsAhead {
    int v[6];
};
__device__ __forceinline__ void rows_load(RowsAhead &r, const int32_t *sorted, int pos0, int BM) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < 6; ++k) {
        const int j = lane + 32 * k;
        r.v[k] = (j < BM) ? __ldcg(sorted + pos0 + j) : 0x7FFFFFFF;
    }
}
__device__ __forceinline__ int rows_count(const RowsAhead &r, int P) {
    int cnt = 0;
#pragma unroll
    for (int k = 0; k < 6; ++k) cnt += (r.v[k] < P) ? 1 : 0;
    return __reduce_add_sync(0xffffffffu, cnt);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          uint32_t *err, uint32_t backoff_ns = 0) {
    bool ok = mbar_wait(bar, parity, abort, err, backoff_ns);
    return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ bool warp_wait_limit(uint32_t bar, uint32_t parity, volatile int *abort,
                                                uint32_t *err, long long limit) {
    bool ok = mbar_wait(bar, parity, abort, err, 0, limit);
    return __all_sync(0xffffffffu, ok);
}

// Whole-warp wait for CTA stage `stage` in a weight-ring slot.  A team sees
// only every fourth stage, so it does not follow every phase of a slot; a
// parity match could be the phase two laps back if copies landed out of order.
// The producer writes the stage index into the slot's tag before issuing its
// copy, and it issues stage i only after stage i - n_w was consumed, so a
// parity match together with a matching tag is the right phase.  The common
// case (copy landed) takes one tag read, then one barrier test and one vote:
// a tag read first that matches means every earlier phase of the slot is
// complete, so the parity test that follows sees stage i's own phase (this
// test is the team's per-stage overhead, measured 4 % of the decode time).
__device__ __forceinline__ bool wait_stage(uint32_t bar, uint32_t parity,
                                           const volatile uint32_t *tag, uint32_t stage,
                                           volatile int *abort, uint32_t *err) {
    {
        const bool tag_ok = (*tag == stage);
        if (__all_sync(0xffffffffu, tag_ok && mbar_try_wait_nohint(bar, parity))) return true;
    }
    const long long t0 = clock64();
#pragma unroll 1
    while (true) {
        if (!warp_wait(bar, parity, abort, err)) return false;
        if (__all_sync(0xffffffffu, *tag == stage)) return true;
        if (*abort) return false;
        if (clock64() - t0 > kWaitTimeoutCycles) {
            *abort = 1;
            if (err) atomicOr(err, kErrTimeout);
            return false;
        }
    }
}

// Bounded wait (one thread) until the counter *ctr, which other CTAs increment
// with a release, reaches `target`: an acquire load, then polls with a short
// sleep.  Gives up (false: the CTA's abort flag and MOE_DEVERR_TIMEOUT) after
// kWaitTimeoutCycles or when another role of the CTA has aborted.
__device__ bool wait_counter(const int32_t *ctr, int target, volatile int *abort, uint32_t *err) {
    if (ld_acquire_gpu(ctr) >= target) return true;
    const long long t0 = clock64();
#pragma unroll 1
    while (true) {
        __nanosleep(128);
        if (ld_acquire_gpu(ctr) >= target) return true;
        if (*abort) return false;
        if (clock64() - t0 > kWaitTimeoutCycles) {
            *abort = 1;
            if (err) atomicOr(err, kErrTimeout);
            return false;
        }
    }
}

// A GEMM kind as a type: the fused kernel runs each role's phase loop once per
// kind through a generic lambda, so that `kind` is a compile-time constant in
// both phases as it is in the separate kernels.
template <int K>
struct KindC {
    static constexpr int value = K;
};

// The fused kernel's gather: fp16 rows of x in bucketed order (the gate/up
// GEMM's B operand).  The work is cut into pieces of 256 elements of one pair's
// row (one 16-byte load per lane), dealt out over the gathering warps of the
// whole grid (`gw` of `nw`) in contiguous runs, so that even a handful of rows
// (decode) is copied in about one memory round trip: a lane keeps up to 4 loads
// in flight.  `pos_of` (from the align) gives each pair's row.
__device__ __forceinline__ void fused_gather(const GemmParams &p, int gw, int nw, bool &bad) {
    const int lane = threadIdx.x & 31;
    const int pieces = (p.H + 255) / 256;  // H % 256 == 128: a half last piece
    const long long total = (long long)p.P * pieces;
    const long long lo = total * gw / nw, hi = total * (gw + 1) / nw;
    for (long long i0 = lo; i0 < hi; i0 += 4) {
        uint4 v[4];
        int dst_row[4], col[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const long long it = i0 + u;
            dst_row[u] = -1;
            if (it < hi) {
                const int pair = (int)(it / pieces);
                col[u] = (int)(it % pieces) * 256 + lane * 8;
                if (col[u] < p.H) {
                    v[u] = *reinterpret_cast<const uint4 *>(p.x + (size_t)(pair / p.top_k) * p.H +
                                                            col[u]);
                    dst_row[u] = __ldcg(p.pos_of + pair);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (dst_row[u] >= 0 && bounds_ok(dst_row[u] < p.cap, p.err))
                *reinterpret_cast<uint4 *>(p.x16 + (size_t)dst_row[u] * p.H + col[u]) =
                    bf16x8_to_f16x8_sat(v[u], bad);
    }
}

// Sub-stages of stage j of a tile with `kss` sub-stages (the last may hold one).
__device__ __forceinline__ int stage_subs(int j, int kss) {
    return (2 * j + 2 <= kss) ? 2 : 1;
}

// Issuing warps that take part in (and release) one A part of a stage: with
// four issuers (one per slab x sub-stage) a sub-stage part has two of them.
__host__ __device__ __forceinline__ int part_issuers(int ni, int np) {
    return (ni == 4) ? 4 / np : ni;
}

// Gate/up epilogue of a full piece with one accumulator per slab (gate at
// column tl, up at tl + BM): SiLU(g) * u of accumulator columns [j_lo, j_hi)
// of this warp's lane quadrant, written as the fp16 intermediate rows
// a_row0 + column * I (columns >= nr are not stored).
__device__ __forceinline__ void swiglu_store(uint32_t tl, int BM, int j_lo, int j_hi, int nr,
                                             uint16_t *a_row0, int I, bool &bad) {
    for (int j0 = j_lo; j0 < j_hi; j0 += 16) {
        float gv[16], uv[16];
        tmem_ld2_32x32b_x16_wait(tl + j0, tl + BM + j0, gv, uv);
        // all 16 SwiGLU values first (independent exp and reciprocal chains
        // overlap; columns past nr hold finite or garbage values that are
        // never stored), then the stores of the real columns
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) gv[jj] = silu_mul(gv[jj], uv[jj]);
        uint16_t *dst = a_row0 + (size_t)j0 * I;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj, dst += I)
            if (j0 + jj < nr) *dst = f16_sat(gv[jj], bad);
    }
}

}  // namespace

// WIDE: the wide-block configuration (blocks of 144..192 tokens): A released
// per sub-stage half (np = 2); down has one issuer and B slots of one
// sub-stage.  Separate instantiations keep the common path's registers.
// KIND 3 is the fused decode kernel: every role runs the gate/up GEMM's pieces,
// then the down GEMM's, through the same rings (the down weights stream while
// the gate/up epilogues finish); it also gathers the x rows and zeroes the
// output accumulator, each CTA its share, and it waits on counters instead of
// on a kernel boundary: the gate/up B loads wait until every CTA has finished
// its gather share, and a block's down B loads until its gate/up tiles are all
// written.  Every such wait is bounded.  Blocks of up to 128 rows only.
// FMT: the weight format (0 INT4, 1 MXFP4); it changes only the dequant.
template <int KIND, int WIDE, int FMT>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const GemmParams p, const __grid_constant__ CUtensorMap tmap_x,
                    const __grid_constant__ CUtensorMap tmap_a) {
    constexpr bool kFused = (KIND == 3);
    static_assert(!(kFused && WIDE), "the fused kernel runs narrow blocks");
    constexpr int kKind0 = kFused ? 1 : KIND;  // the GEMMs this kernel runs, in order
    constexpr int kKind1 = kFused ? 2 : KIND;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw_addr);

    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BM = p.block_m;
    const int n_w = p.n_w, n_b = p.n_b, n_a = p.n_a;
    // Narrow blocks (one part, one B slot per stage, two or four issuers):
    // warp 1 waits for each stage's B slot and then joins the stage's A-slot
    // barrier, so no MMA issuer waits for B (the issuers' per-stage path
    // bounds the stage rate at decode sizes).
    const bool b_waiter = !WIDE && p.ni != 1;
    const int ni = p.ni;    // MMA issuers (4: one per dequant group, 2: one per slab)

    // shared-memory map
    const uint32_t w_ring = base;
    const uint32_t b_ring = base + p.smem_b_off;
    const uint32_t misc = base + p.smem_misc_off;
    const uint32_t bar_w_full = misc;
    const uint32_t bar_w_empty = bar_w_full + 8 * n_w;
    const uint32_t bar_b_full = bar_w_empty + 8 * n_w;
    const uint32_t bar_b_empty = bar_b_full + 8 * n_b;
    // a_free[t][part]: part `part` of the A slot of team t's next stage is free
    // (the MMAs of the stage n_a earlier on it are done); np = 2 releases each
    // sub-stage half of a slot on its own
    constexpr int np = WIDE ? 2 : 1;
    constexpr bool b_sub = (WIDE && KIND == 2);
    // Wide gate/up has one accumulator buffer, so its MMAs wait for every
    // piece's epilogue; the four issuing warps (one per lane quadrant, idle then)
    // take the upper half of a full piece's columns.
    constexpr bool kHelp = (WIDE && KIND == 1);
    const uint32_t bar_a_free = bar_b_empty + 8 * n_b;
    // acc_full[b] / acc_empty[b]: accumulator buffer b holds a finished piece /
    // has been read by the epilogue (buffers alternate between pieces)
    const uint32_t bar_acc_full = bar_a_free + 8 * kTeams * np;
    const uint32_t bar_acc_empty = bar_acc_full + 16;
    const uint32_t bar_drain = bar_acc_empty + 16;
    const uint32_t misc_words = bar_drain + 8;  // tmem slot, abort flag, bcast
    uint8_t *misc_ptr = smem + (misc_words - base);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(misc_ptr);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc_ptr + 4);
    volatile int *bcast = reinterpret_cast<volatile int *>(misc_ptr + 8);
    // stage tags of the weight ring: the CTA stage index last issued into each slot
    volatile uint32_t *w_tag = reinterpret_cast<volatile uint32_t *>(smem + (misc - base) + 512);
    // down epilogue: (token, routing weight) of each column of the current block
    int2 *col_tab = reinterpret_cast<int2 *>(smem + (misc - base) + 1024);
    // down epilogue (epi_f4): per epilogue warp, 8 columns x 32 rows of fp32
    // to turn into float4s of 4 rows of one column (after the column table)
    float *epi_stage = reinterpret_cast<float *>(smem + (misc - base) + 1024 + 256 * 8);

    if (threadIdx.x == 0) {
        for (int i = 0; i < n_w; ++i) {
            mbar_init(bar_w_full + 8 * i, 2);  // weight + scale producers
            mbar_init(bar_w_empty + 8 * i, kTeamWarps);
        }
        for (int i = 0; i < n_b; ++i) {
            mbar_init(bar_b_full + 8 * i, 1);
            mbar_init(bar_b_empty + 8 * i, ni);
        }
        for (int i = 0; i < kTeams * np; ++i) mbar_init(bar_a_free + 8 * i, part_issuers(ni, np));
        for (int i = 0; i < n_w; ++i) w_tag[i] = 0xFFFFFFFFu;
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_acc_full + 8 * i, ni);
            mbar_init(bar_acc_empty + 8 * i, kHelp ? 8 : 4);
        }
        mbar_init(bar_drain, ni);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (wid == 1) {
        tmem_alloc(misc_words, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Programmatic dependent launch.  In the separate GEMM kernels, the align
    // kernel has completed before any CTA of this grid starts: the gather
    // launches its dependents only after its own wait for the align, and the
    // down GEMM's only predecessor is the gate/up GEMM.  So the routing buffers
    // (align outputs) are read without waiting, through L2 (ld.global.cg: no
    // stale L1 lines), and the weight stream, its dequant and the issue loop
    // start while the previous kernel still runs.  Only the roles that read what
    // the previous kernel wrote wait for it: the B loader (gathered x rows, or
    // the intermediate) and the epilogue (split counters and partial slots, the
    // accumulator that the gate/up GEMM zeroes).  The fused kernel follows the
    // align kernel itself, so all of it waits.
    if (kFused) pdl_wait();
    pdl_launch_dependents();

    // Tensor-memory column map: nbuf accumulator buffers of ni accumulators
    // (BM columns each), then the A ring of n_a stages x 128 columns.
    // Accumulator of (slab g, sub-stage u): (ni == 4 ? 2g + u : g) within its
    // buffer; gate/up: slab 0 feeds the gate accumulator(s), slab 1 the up ones.
    const int nbuf = p.nbuf;
    const uint32_t acc_buf_cols = (uint32_t)(ni * BM);
    const uint32_t col_a = (uint32_t)nbuf * acc_buf_cols;

    int tile, kb0, kb1;

    if (kFused && wid >= kFirstDequantWarp) {
        // The fused kernel's warps 4..23 gather x first (each CTA its share), an
        // idle time for them anyway: the weight stream waits for the gather.  The
        // tensor-memory owner warp then publishes the share with its zeroing.
        bool bad = false;
        fused_gather(p, blockIdx.x * kGatherWarps + (wid - kFirstDequantWarp),
                     gridDim.x * kGatherWarps, bad);
        report_range(bad, p.err);
        __threadfence();
        fence_proxy_async_global();
        named_bar_sync(kBarPrep, kPrepThreads);
    }

    if (wid == 0 || wid == 3) {
        // --------------------------- weight (warp 0) / scale (warp 3) producer --
        if (lane == 0) {
            const bool scales = (wid == 3);
            const uint32_t sub_bytes = scales ? kStageSBytes : kStageWBytes;
            const uint32_t dst_off = scales ? kStageW : 0u;
            const uint64_t pol = l2_policy_evict_first();
            uint32_t i = 0;
            Ring w(n_w);
            bool ok = true;
            // Fused kernel: the weight stream starts once every CTA has published
            // its gather share.  Started earlier, its burst of requests (about
            // 150 KB per SM) queues ahead of the gather's few row loads in the
            // memory system and delays them several times over (measured at
            // decode sizes: the gather then took 10 us instead of about 2).
            if (kFused) ok = wait_counter(p.prep_done, (int)gridDim.x, abort_flag, p.err);
            auto phase = [&](auto kc) {
                constexpr int kind = decltype(kc)::value;
                const GemmPhase &G = p.g[kind - 1];
                const Sched sched = make_sched(p, G);
                PieceIter pi;
                pi.init(sched);
                const uint8_t *src = scales ? G.wsc : G.wq;
                while (ok && pi.next(sched, tile, kb0, kb1)) {
                    const int b = tile / G.RT, r = tile % G.RT;
                    int e = __ldcg(p.expert_ids + b);
                    if (!bounds_ok(e >= 0 && e < p.E, p.err)) e = 0;
                    const size_t sub0 = ((size_t)e * G.RT + r) * G.KSS;  // first sub-stage of the tile
                    for (int j = kb0; j < kb1; ++j, ++i, w.next()) {
                        if (!mbar_wait(bar_w_empty + 8 * w.idx, w.ph ^ 1, abort_flag, p.err, 128)) {
                            ok = false;
                            break;
                        }
                        const uint32_t bytes = stage_subs(j, G.KSS) * sub_bytes;
                        if (kDebugBounds && !scales && (int)i == p.skip_stage && blockIdx.x == 0)
                            continue;  // the timeout test: this stage never lands
                        if (!scales) w_tag[w.idx] = i;
                        mbar_arrive_expect_tx(bar_w_full + 8 * w.idx, bytes);
                        bulk_g2s(w_ring + w.idx * kStage + dst_off, src + (sub0 + 2 * j) * sub_bytes,
                                 bytes, bar_w_full + 8 * w.idx, pol);
                    }
                }
            };
            if (kKind0 == 1) phase(KindC<1>{});
            if (kKind1 == 2 && ok) phase(KindC<2>{});
            if (!ok) {  // let copies in flight land before the CTA exits
                volatile int never = 0;
                const uint32_t first = (i > (uint32_t)n_w) ? i - n_w : 0;
                for (uint32_t j = first; j < i; ++j)
                    mbar_wait(bar_w_full + 8 * (j % n_w), (j / n_w) & 1, &never, nullptr);
            }
        }
    } else if (wid == 1) {
        // ------------------------------------------------- output zeroing --
        // The tensor-memory owner has nothing to do until the end, so it clears
        // the down GEMM's fp32 accumulator, a grid-strided share per CTA, while
        // the weights stream (gate/up and fused kernels).  Streaming stores: the
        // zero lines should not push the B rows that other row tiles re-read out
        // of L2.  The separate down GEMM reads the accumulator only after this
        // grid has completed; in the fused kernel the share is published below.
        if (p.zero_out) {
            const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
            const size_t stride = (size_t)gridDim.x * 32;
            for (size_t i = (size_t)blockIdx.x * 32 + lane; i < p.zero_n16; i += stride)
                __stcs(p.zero_out + i, z4);
        }
        if (kFused) {
            // publish this CTA's share of the gather (warps 4..23) and of the
            // zeroing: each thread's writes, then one release of the count
            __threadfence();
            fence_proxy_async_global();
            named_bar_sync(kBarPrep, kPrepThreads);
            if (lane == 0) red_release_gpu(p.prep_done, 1);
        }
        if (b_waiter) {
            // ------------------------------------------------ B waiter --
            // Every stage in order, as the issuers take them: B slot landed,
            // then the stage's A-slot barrier (a bar.sync like the issuers',
            // so this warp never arrives twice on one barrier instance).
            // After an error it still visits every barrier, without waiting.
            const uint32_t slot_cnt = (uint32_t)(kTeamWarps + part_issuers(ni, np) + 1) * 32u;
            Ring a(n_a), bq(n_b);
            bool ok = true;
            auto phase = [&](auto kc) {
                constexpr int kind = decltype(kc)::value;
                const GemmPhase &G = p.g[kind - 1];
                const Sched sched = make_sched(p, G);
                PieceIter pi;
                pi.init(sched);
                while (pi.next(sched, tile, kb0, kb1)) {
#pragma unroll 1
                    for (int j = kb0; j < kb1; ++j, a.next(), bq.next()) {
                        if (ok) ok = warp_wait(bar_b_full + 8 * bq.idx, bq.ph, abort_flag, p.err);
                        named_bar_sync(kBarSlot0 + a.idx, slot_cnt);
                    }
                }
            };
            if (kKind0 == 1) phase(KindC<1>{});
            if (kKind1 == 2) phase(KindC<2>{});
        }
    } else if (wid == 2) {
        // ------------------------------------------------------ B loader --
        // B rows of the block (bucketed order) by 2-D TMA tensor copies: one
        // 64-column k block per copy, gate/up one per sub-stage, down two.
        if (!kFused) pdl_wait();  // B rows are the previous kernel's output
        if (lane == 0) {
            uint32_t i = 0;
            bool ok = true;
            Ring bq(n_b);
            auto phase = [&](auto kc) {
                constexpr int kind = decltype(kc)::value;
                const GemmPhase &G = p.g[kind - 1];
                const CUtensorMap *tm = (kind == 1) ? &tmap_x : &tmap_a;
                const int kb_per_sub = (kind == 1) ? 1 : 2;
                const int kss = G.KSS;
                const Sched sched = make_sched(p, G);
                PieceIter pi;
                pi.init(sched);
                int ready_b = -1;  // fused: the block whose B rows are known written
                if (kFused && kind == 1) {
                    // every CTA's share of the gathered x rows is written
                    ok = wait_counter(p.prep_done, (int)gridDim.x, abort_flag, p.err);
                    fence_proxy_async_global();
                }
                while (ok && pi.next(sched, tile, kb0, kb1)) {
                    const int b = tile / G.RT;
                    if (kFused && kind == 2 && b != ready_b) {
                        // every gate/up tile of block b (its whole intermediate rows)
                        ok = wait_counter(p.blk_done + b, p.g[0].RT, abort_flag, p.err);
                        fence_proxy_async_global();
                        ready_b = b;
                    }
                    for (int j = kb0; j < kb1 && ok; ++j) {
                        // one slot per stage, or (wide blocks) one per sub-stage
                        const int nsub = stage_subs(j, kss);
                        const int nslots = b_sub ? nsub : 1;
                        const int nblk = b_sub ? kb_per_sub : nsub * kb_per_sub;
                        for (int sl = 0; sl < nslots; ++sl, ++i, bq.next()) {
                            const uint32_t s = bq.idx;
                            if (!mbar_wait(bar_b_empty + 8 * s, bq.ph ^ 1, abort_flag, p.err, 128)) {
                                ok = false;
                                break;
                            }
                            const uint32_t dst = b_ring + s * p.b_stage_bytes;
                            const int kb_first = 2 * kb_per_sub * j + sl * kb_per_sub;
                            mbar_arrive_expect_tx(bar_b_full + 8 * s, (uint32_t)nblk * BM * 128u);
                            for (int qb = 0; qb < nblk; ++qb)
                                tma_load_2d(dst + qb * BM * 128, tm, (kb_first + qb) * 64, b * BM,
                                            bar_b_full + 8 * s);
                        }
                    }
                }
            };
            if (kKind0 == 1) phase(KindC<1>{});
            if (kKind1 == 2 && ok) phase(KindC<2>{});
            if (!ok) {
                volatile int never = 0;
                const uint32_t first = (i > (uint32_t)n_b) ? i - n_b : 0;
                for (uint32_t jj = first; jj < i; ++jj)
                    mbar_wait(bar_b_full + 8 * (jj % n_b), (jj / n_b) & 1, &never, nullptr, 64);
            }
        }
    } else if (wid >= kFirstDequantWarp && wid < kFirstIssuerWarp) {
        // ------------------------------------------------------- dequant --
        // Three teams of four warps take stages in turn (stage i: team i % 3),
        // so a team's waits overlap the other teams' arithmetic.  Warp
        // 4 + 4t + q of team t dequantises rows 32q..32q+31 (its tensor-memory
        // lane quadrant) of both slabs and both sub-stages.  A team visits
        // every one of its stages even after an error (no work, but every
        // barrier arrival still happens), so no named barrier can be left
        // waiting.
        const int team = (wid - kFirstDequantWarp) >> 2;
        const int q = wid & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const uint32_t my_w = w_ring + (uint32_t)row * 16u;  // shared addresses
        const uint32_t my_s = w_ring + kStageW + (uint32_t)row * 4u;
        const uint32_t my_t = tmem + lane_off + col_a;
        const uint32_t slot_cnt =
            (uint32_t)(kTeamWarps + part_issuers(ni, np) + (b_waiter ? 1 : 0)) * 32u;
        const DequantConsts dqc = p.dq;
        volatile int no_abort = 0;
        Ring w(n_w), a(n_a);  // a: the A slot only (its phase is not used)
        w.advance(team);
        a.advance(team);
        uint32_t a_ph = 0;    // parity bits (per part) of this team's next a_free phases
        long long s0 = 0;           // CTA stage index of the current piece's first stage
        long long own = team;       // next stage of this team
        bool ok = true;
        auto phase = [&](auto kc) {
            constexpr int kind = decltype(kc)::value;
            const GemmPhase &G = p.g[kind - 1];
            const int kss = G.KSS;
            const Sched sched = make_sched(p, G);
            PieceIter pi;
            pi.init(sched);
            while (pi.next(sched, tile, kb0, kb1)) {
                const long long s1 = s0 + (kb1 - kb0);
                for (; own < s1; own += kTeams, w.advance(kTeams), a.advance(kTeams)) {
                    const int j = kb0 + (int)(own - s0);
                    if (ok)
                        ok = wait_stage(bar_w_full + 8 * w.idx, w.ph, w_tag + w.idx,
                                        (uint32_t)own, abort_flag, p.err);
                    const int nsub = ok ? stage_subs(j, kss) : 0;
                    const uint32_t sw = my_w + w.idx * kStage;
                    const uint32_t ss = my_s + w.idx * kStage;
                    const uint32_t st = my_t + a.idx * kACols;
                    for (int part = 0; part < np; ++part) {
                        // Part `part` of the A slot is reused only once the MMAs
                        // of the stage n_a earlier on it are done; the issuers
                        // signal that on this team's own barrier for the part,
                        // whose phases follow the team's stages in order, so a
                        // parity wait is never more than one phase behind.
                        //
                        // The hand-off to the issuers is a hardware named barrier
                        // (a bar.arrive here, a bar.sync there; measured 5 %
                        // faster than an mbarrier at decode), which cannot give up.
                        // So this team must never arrive on the part's barrier
                        // again before the issuers have consumed its previous
                        // arrival, even after an error: this wait ignores the abort
                        // flag and its limit is 16 times every other wait's.  The
                        // issuers release the slot as soon as they have passed
                        // the (at most three) stages before it, and each of those
                        // stalls them only for other waits, every one bounded by
                        // the normal limit and ended early by the abort flag, so
                        // this wait runs out only if the tensor cores stop
                        // completing MMAs.
                        if (own >= n_a) {
                            const bool freed =
                                warp_wait_limit(bar_a_free + 8 * (team * np + part),
                                                (a_ph >> part) & 1u, &no_abort, p.err,
                                                kSlotWaitCycles);
                            a_ph ^= 1u << part;
                            if (!freed) ok = false;
                        }
                        const int u_lo = (np == 2) ? part : 0, u_hi = (np == 2) ? part + 1 : 2;
                        for (int uu = u_lo; uu < u_hi && uu < nsub && ok; ++uu) {
#pragma unroll
                            for (int g = 0; g < 2; ++g) {
                                const uint32_t src = sw + uu * kStageWBytes + g * kSlabBytes;
                                const uint4 lo = lds128(src);
                                const uint4 hi = lds128(src + 2048);
                                const uint32_t sc = lds32(ss + uu * kStageSBytes + g * 512);
                                if (g == 1 && uu == nsub - 1) {  // every load of this stage is done
                                    __syncwarp();
                                    if (lane == 0) mbar_arrive(bar_w_empty + 8 * w.idx);
                                }
                                uint32_t v[32];
                                if (FMT == 1)
                                    dequant_row_fp4(lo, hi, sc, v);
                                else
                                    dequant_row(lo, hi, sc, dqc, v);
                                tc_fence_after();
                                // wide blocks: one wait per part (measured 1-2 % faster
                                // there); narrow: a wait per store (faster at decode)
                                if (WIDE)
                                    tmem_st_32x32b_x32(st + uu * 64 + g * 32, v);
                                else
                                    tmem_st_32x32b_x32_wait(st + uu * 64 + g * 32, v);
                            }
                        }
                        if (WIDE) tmem_wait_st();
                        tc_fence_before();
                        named_bar_arrive(kBarSlot0 + a.idx * np + part, slot_cnt);  // part written
                    }
                }
                s0 = s1;
            }
        };
        if (kKind0 == 1) phase(KindC<1>{});
        if (kKind1 == 2) phase(KindC<2>{});
    } else if (wid >= kFirstIssuerWarp && wid < kFirstEpilogueWarp) {
        // ------------------------------------------------------- MMA issue --
        // Warp 16 + qe issues the MMAs of sub-tile qe (slab qe & 1,
        // sub-stage qe >> 1) into its own accumulator; with two issuers, warps
        // 16 and 17 each cover both sub-stages of slab 0 / 1.  A piece goes to
        // accumulator buffer c % nbuf, so with two buffers the next piece's
        // MMAs run while the epilogue warps read the previous one.
        const int qe = wid - kFirstIssuerWarp;
        const bool issuer = qe < ni;
        // units (slab, sub-stage) of this issuer: ni = 4 one, ni = 2 a slab's
        // two, ni = 1 all four (slab loop inside)
        const int ig = (ni == 1) ? 0 : (qe & 1);
        const int g_hi = (ni == 1) ? 2 : ig + 1;
        const int iu_lo = (ni == 4) ? (qe >> 1) : 0;
        const int iu_hi = (ni == 4) ? (qe >> 1) + 1 : 2;
        const uint32_t acc_off = (uint32_t)((ni == 4 ? 2 * ig + (qe >> 1) : ig) * BM);
        const uint32_t slot_cnt =
            (uint32_t)(kTeamWarps + part_issuers(ni, np) + (b_waiter ? 1 : 0)) * 32u;
        Ring a(n_a), bq(n_b);
        Ring acc((uint32_t)nbuf);  // accumulator buffer and its lap parity, per piece
        uint32_t next_team = (uint32_t)(n_a % kTeams);  // team of stage (CTA stage + n_a)
        bool ok = true;
        bool range_bad = false;  // a SwiGLU value saturated (helping issuers)
        auto phase = [&](auto kc) {
            constexpr int kind = decltype(kc)::value;
            const GemmPhase &G = p.g[kind - 1];
            const int kss = G.KSS;
            const int kb_per_sub = (kind == 1) ? 1 : 2;
            const Sched sched = make_sched(p, G);
            PieceIter pi;
            pi.init(sched);
            // Wide blocks: the next piece's block entries are loaded while this
            // piece is issued, so no piece starts with a dependent global load
            // (measured faster for wide blocks only).
            PieceIter pa = pi;
            int tile_a, kb0_a, kb1_a;
            RowsAhead ahead;
            if (WIDE && pa.next(sched, tile_a, kb0_a, kb1_a))
                rows_load(ahead, p.sorted_ids, (tile_a / G.RT) * BM, BM);
            while (pi.next(sched, tile, kb0, kb1)) {
                const int b = tile / G.RT;
                const int pos0 = b * BM;
                int nr;
                if (WIDE) {
                    nr = rows_count(ahead, p.P);
                    if (pa.next(sched, tile_a, kb0_a, kb1_a))
                        rows_load(ahead, p.sorted_ids, (tile_a / G.RT) * BM, BM);
                } else {
                    // 16-row blocks issue 16-column MMAs whatever their row count,
                    // so they skip the dependent load of the block's entries
                    // (measured 2 % faster for the down GEMM at decode)
                    nr = (BM == 16) ? 16 : block_rows(p.sorted_ids, pos0, BM, p.P);
                }
                // ---- issue (every stage is visited, see the dequant role)
                if (issuer) {
                    const uint32_t idesc =
                        idesc_f16_m128(nr <= 16 ? 16u : (uint32_t)((nr + 15) & ~15));
                    const uint32_t buf = acc.idx;
                    const uint32_t acc_col = tmem + buf * acc_buf_cols + acc_off;
                    bool fresh = true;
                    if (ok)
                        ok = warp_wait(bar_acc_empty + 8 * buf, acc.ph ^ 1, abort_flag, p.err, 32);
                    if (b_waiter) {
                        // Narrow blocks: one part and this issuer's unit(s) of slab
                        // ig, in straight-line code; warp 1 has seen the B slot
                        // land when the barrier completes.
#pragma unroll 1
                        for (int j = kb0; j < kb1; ++j, a.next(), bq.next(),
                                 next_team = (next_team + 1 == (uint32_t)kTeams) ? 0u
                                                                                : next_team + 1) {
                            const int nsub = stage_subs(j, kss);
                            const uint32_t a_st = tmem + col_a + a.idx * kACols + ig * 32;
                            const uint32_t bsm = b_ring + bq.idx * p.b_stage_bytes;
                            const uint32_t rel_a = bar_a_free + 8 * next_team;  // np = 1
                            const uint32_t rel_b = bar_b_empty + 8 * bq.idx;
                            named_bar_sync(kBarSlot0 + a.idx, slot_cnt);  // A written, B landed
                            tc_fence_after();
                            for (int uu = iu_lo; uu < iu_hi; ++uu) {
                                const bool last_u = (uu == iu_hi - 1);
                                const uint32_t sub = (kind == 1) ? (uint32_t)uu
                                                                 : (uint32_t)(kb_per_sub * uu + ig);
                                const uint32_t r1 = last_u ? rel_a : 0u, r2 = last_u ? rel_b : 0u;
                                if (ok && uu < nsub) {
                                    mma_ts_f16_k64_commit(
                                        acc_col, a_st + uu * 64,
                                        smem_desc_sw128(bsm + sub * (uint32_t)(BM * 128)), idesc,
                                        fresh ? 0u : 1u, r1, r2);
                                    fresh = false;
                                } else {
                                    tc_commit2_elect(r1, r2);
                                }
                            }
                        }
                    } else
                    for (int j = kb0; j < kb1; ++j, a.next(),
                             next_team = (next_team + 1 == (uint32_t)kTeams) ? 0u : next_team + 1) {
                        const int nsub = stage_subs(j, kss);
                        const uint32_t a_st = tmem + col_a + a.idx * kACols;
                        if (!b_sub && ok)
                            ok = warp_wait(bar_b_full + 8 * bq.idx, bq.ph, abort_flag, p.err);
                        for (int part = 0; part < np; ++part) {
                            const int u_lo = (np == 2) ? (part > iu_lo ? part : iu_lo) : iu_lo;
                            const int u_hi =
                                (np == 2) ? (part + 1 < iu_hi ? part + 1 : iu_hi) : iu_hi;
                            // this issuer takes part in the part's barrier if it has
                            // a unit there (always with np = 1)
                            if (u_lo >= u_hi) continue;
                            named_bar_sync(kBarSlot0 + a.idx * np + part, slot_cnt);  // part in TMEM
                            for (int uu = u_lo; uu < u_hi; ++uu) {
                                // with one B slot per sub-stage, a missing tail
                                // sub-stage has no B slot (the loader skips it too)
                                const bool has_b = !b_sub || uu < nsub;
                                if (b_sub && has_b && ok)
                                    ok = warp_wait(bar_b_full + 8 * bq.idx, bq.ph, abort_flag,
                                                   p.err);
                                const uint32_t bsm = b_ring + bq.idx * p.b_stage_bytes;
                                // release the part after its last block (to the team
                                // that uses the slot next) and the B slot after its
                                // last use
                                const bool last_u = (uu == u_hi - 1);
                                const uint32_t rel_a =
                                    last_u ? bar_a_free + 8 * (next_team * np + part) : 0u;
                                const bool last_b = b_sub || (part == np - 1 && uu == u_hi - 1);
                                for (int g = ig; g < g_hi; ++g) {
                                    const bool last_g = (g == g_hi - 1);
                                    const uint32_t sub = b_sub ? (uint32_t)g
                                                       : (kind == 1) ? (uint32_t)uu
                                                                     : (uint32_t)(kb_per_sub * uu + g);
                                    const uint32_t r1 = last_g ? rel_a : 0u;
                                    const uint32_t r2 =
                                        (last_g && last_b && has_b) ? bar_b_empty + 8 * bq.idx : 0u;
                                    if (ok && uu < nsub) {
                                        const uint64_t bd =
                                            smem_desc_sw128(bsm + sub * (uint32_t)(BM * 128));
                                        tc_fence_after();
                                        mma_ts_f16_k64_commit(acc_col, a_st + uu * 64 + g * 32, bd,
                                                              idesc, fresh ? 0u : 1u, r1, r2);
                                        fresh = false;
                                    } else {
                                        tc_commit2_elect(r1, r2);
                                    }
                                }
                                if (b_sub && has_b) bq.next();
                            }
                        }
                        if (!b_sub) bq.next();
                    }
                    tc_commit_elect(bar_acc_full + 8 * buf);
                }
                if (kHelp) {
                    // the upper half of a full piece's columns; every issuing warp
                    // arrives on acc_empty once per piece (full or not)
                    const uint32_t buf = acc.idx;
                    const bool got = warp_wait(bar_acc_full + 8 * buf, acc.ph, abort_flag, p.err, 32);
                    if (got) {
                        tc_fence_after();
                        if (kb0 == 0 && kb1 == G.KS) {
                            const int hq = wid & 3;
                            const int half = ((nr + 31) / 32) * 16;
                            swiglu_store(tmem + ((uint32_t)(hq * 32) << 16) + buf * acc_buf_cols,
                                         BM, half, nr, nr,
                                         p.a_out + (size_t)pos0 * p.I + (tile % G.RT) * kSlabRows +
                                             hq * 32 + lane,
                                         p.I, range_bad);
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar_acc_empty + 8 * buf);
                    }
                }
                acc.next();
            }
        };
        if (kKind0 == 1) phase(KindC<1>{});
        if (kKind1 == 2) phase(KindC<2>{});
        if (kHelp) report_range(range_bad, p.err);
        if (issuer) {  // every MMA of this CTA must finish before TMEM is released
            volatile int never = 0;
            tc_commit_elect(bar_drain);
            warp_wait(bar_drain, 0, &never, nullptr, 32);
        }
    } else if (wid >= kFirstEpilogueWarp) {
        // -------------------------------------------------------- epilogue --
        // At the end of each piece the four warps (lane quadrants 0..3) read the
        // accumulators of its buffer for their 32 TMEM lanes.
        const int q = wid & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        Ring acc((uint32_t)nbuf);  // accumulator buffer and its lap parity, per piece
        bool ok = true;
        bool range_bad = false;  // a SwiGLU value saturated
        if (!kFused) pdl_wait();  // counters, partial slots and the accumulator (see above)
        bool zero_seen = !kFused;  // fused: every CTA's zeroing share is published
        auto phase = [&](auto kc) {
            constexpr int kind = decltype(kc)::value;
            const GemmPhase &G = p.g[kind - 1];
            const Sched sched = make_sched(p, G);
            PieceIter pi;
            pi.init(sched);
            const long long T = sched.T;
            while (pi.next(sched, tile, kb0, kb1)) {
                const int b = tile / G.RT, r = tile % G.RT;
                const int pos0 = b * BM;
                const int nr = block_rows(p.sorted_ids, pos0, BM, p.P);
                const uint32_t buf = acc.idx;
                if (kind == 2) {
                    // The combine needs each column's token and routing weight: look
                    // them up once per block (these loads overlap the wait for the
                    // piece's MMAs) instead of as a dependent chain of global loads
                    // per column.  The barrier below orders these writes before the
                    // reads.
                    for (int col = row; col < nr; col += 128) {  // nr may exceed the 128 threads
                        int pair = __ldcg(p.sorted_ids + pos0 + col);
                        if (!bounds_ok(pair >= 0 && pair < p.P, p.err)) pair = 0;
                        col_tab[col] =
                            make_int2(pair / p.top_k, __float_as_int(p.topk_weights[pair]));
                    }
                }
                const bool u1 = !(kb1 - kb0 == 1 && stage_subs(kb0, G.KSS) == 1);
                bool got =
                    ok && warp_wait(bar_acc_full + 8 * buf, acc.ph, abort_flag, p.err, 32);
                if (kind == 2 && !zero_seen && got) {
                    // the combine adds into rows that every CTA zeroed its share of
                    got = wait_counter(p.prep_done, (int)gridDim.x, abort_flag, p.err);
                    zero_seen = got;
                }
                // the four warps decide together (they share named barrier 1)
                if (named_bar_or(kBarEpi, 128, !got)) ok = false;
                if (ok) {
                    tc_fence_after();
                    const int feat = r * kSlabRows + row;
                    const uint32_t tl = tmem + lane_off + buf * acc_buf_cols;
                    if (kind == 1) {
                        const bool full = (kb0 == 0 && kb1 == G.KS);
                        bool tile_done = full;  // this piece completes the tile's rows
                        float *sl = nullptr;
                        if (!full) {
                            const long long piece_start = (long long)(tile - sched.rr) * G.KS + kb0;
                            const int slot = (piece_start == sched.start) ? 0 : 1;
                            sl = p.partial + ((size_t)(sched.cta * 2 + slot) * 2) * BM * 128;
                        }
                        // wide: the issuing warps take columns [half, nr) of a full piece
                        const int j_end = (kHelp && full) ? ((nr + 31) / 32) * 16 : nr;
                        for (int j0 = 0; j0 < j_end; j0 += 16) {
                            float gv[16], uv[16];
                            if (ni == 4) {
                                // accumulator of (slab g, sub-stage u) is column (2g + u) * BM
                                tmem_ld2_32x32b_x16_wait(tl + 0 * BM + j0, tl + 2 * BM + j0, gv, uv);
                                if (u1) {
                                    float g1[16], u1v[16];
                                    tmem_ld2_32x32b_x16_wait(tl + 1 * BM + j0, tl + 3 * BM + j0, g1,
                                                             u1v);
#pragma unroll
                                    for (int jj = 0; jj < 16; ++jj) {
                                        gv[jj] += g1[jj];
                                        uv[jj] += u1v[jj];
                                    }
                                }
                            } else {
                                tmem_ld2_32x32b_x16_wait(tl + j0, tl + BM + j0, gv, uv);
                            }
                            if (full) {
                                // all 16 SwiGLU values first (independent exp and
                                // reciprocal chains overlap; columns past nr hold
                                // finite or garbage values that are never stored),
                                // then the stores of the real columns
#pragma unroll
                                for (int jj = 0; jj < 16; ++jj) gv[jj] = silu_mul(gv[jj], uv[jj]);
                                uint16_t *dst = p.a_out + (size_t)(pos0 + j0) * p.I + feat;
#pragma unroll
                                for (int jj = 0; jj < 16; ++jj, dst += p.I)
                                    if (j0 + jj < nr) *dst = f16_sat(gv[jj], range_bad);
                            } else {
#pragma unroll
                                for (int jj = 0; jj < 16; ++jj) {
                                    const int jr = j0 + jj;
                                    if (jr < nr) {
                                        sl[(size_t)jr * 128 + row] = gv[jj];
                                        sl[(size_t)(BM + jr) * 128 + row] = uv[jj];
                                    }
                                }
                            }
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar_acc_empty + 8 * buf);
                        if (!full) {
                            __threadfence();
                            named_bar_sync(kBarEpi, 128);
                            if (row == 0) {
                                const int len = kb1 - kb0;
                                const int old = atomicAdd(&p.tile_cnt[tile], len);
                                *bcast = (old + len == G.KS) ? 1 : 0;
                            }
                            named_bar_sync(kBarEpi, 128);
                            const bool last = *bcast != 0;
                            named_bar_sync(kBarEpi, 128);
                            tile_done = last;
                            if (last) {
                                __threadfence();
                                const long long ts = (long long)(tile - sched.rr) * G.KS,
                                                te = ts + G.KS;
                                const int c_first = range_owner(T, sched.G, ts);
                                const int c_last = range_owner(T, sched.G, te - 1);
                                for (int jr = 0; jr < nr; ++jr) {
                                    float gs = 0.f, us = 0.f;
                                    for (int cc = c_first; cc <= c_last; ++cc) {
                                        const long long cs = range_start(T, sched.G, cc);
                                        if (range_start(T, sched.G, cc + 1) == cs) continue;  // empty
                                        const int sslot = (cs >= ts) ? 0 : 1;
                                        const float *ps =
                                            p.partial + ((size_t)(cc * 2 + sslot) * 2) * BM * 128;
                                        gs += __ldcg(ps + (size_t)jr * 128 + row);
                                        us += __ldcg(ps + (size_t)(BM + jr) * 128 + row);
                                    }
                                    p.a_out[(size_t)(pos0 + jr) * p.I + feat] =
                                        f16_sat(silu_mul(gs, us), range_bad);
                                }
                            }
                        }
                        if (kFused && tile_done) {
                            // the tile's intermediate rows are written: publish them to
                            // the down B loads of block b (every thread's stores, then
                            // one release of the block's count)
                            __threadfence();
                            fence_proxy_async_global();
                            named_bar_sync(kBarEpi, 128);
                            if (row == 0) red_release_gpu(p.blk_done + b, 1);
                        }
                    } else {
                        for (int j0 = 0; j0 < nr; j0 += 16) {
                            float dv[16];
                            if (ni == 1) {
                                tmem_ld_32x32b_x16_wait(tl + j0, dv);
                            } else if (ni == 4) {
                                float d1[16];
                                tmem_ld2_32x32b_x16_wait(tl + 0 * BM + j0, tl + 2 * BM + j0, dv, d1);
#pragma unroll
                                for (int jj = 0; jj < 16; ++jj) dv[jj] += d1[jj];
                                if (u1) {
                                    float d2[16], d3[16];
                                    tmem_ld2_32x32b_x16_wait(tl + 1 * BM + j0, tl + 3 * BM + j0, d2,
                                                             d3);
#pragma unroll
                                    for (int jj = 0; jj < 16; ++jj) dv[jj] += d2[jj] + d3[jj];
                                }
                            } else {
                                float d1[16];
                                tmem_ld2_32x32b_x16_wait(tl + j0, tl + BM + j0, dv, d1);
#pragma unroll
                                for (int jj = 0; jj < 16; ++jj) dv[jj] += d1[jj];
                            }
                            if (b_sub || p.epi_f4) {
                                // A lane's 16 values are one row (output feature) of 16
                                // columns (tokens), and a scalar add per value is one
                                // reduction request per column per warp.  Through shared
                                // memory, each lane instead adds a float4: 4 consecutive
                                // features of one token, a quarter of the requests.  8
                                // columns at a time (1 KB per warp).
                                float *stg = epi_stage + q * 256;
#pragma unroll
                                for (int jj = 0; jj < 16; ++jj)
                                    dv[jj] *= __int_as_float(col_tab[j0 + jj].y);
#pragma unroll
                                for (int h = 0; h < 16; h += 8) {
                                    if (j0 + h >= nr) break;  // no real column left (decode)
#pragma unroll
                                    for (int jj = 0; jj < 8; ++jj) stg[jj * 32 + lane] = dv[h + jj];
                                    __syncwarp();
#pragma unroll
                                    for (int rr = 0; rr < 2; ++rr) {
                                        const int idx = rr * 32 + lane;  // (column, 4-row group)
                                        const int jt = idx >> 3, f4 = idx & 7;
                                        const int jr = j0 + h + jt;
                                        const float4 v4 =
                                            *reinterpret_cast<const float4 *>(stg + jt * 32 + 4 * f4);
                                        if (jr < nr)
                                            atomicAdd(reinterpret_cast<float4 *>(
                                                          p.out_acc + (size_t)col_tab[jr].x * p.H +
                                                          r * kSlabRows + q * 32 + 4 * f4),
                                                      v4);
                                    }
                                    __syncwarp();
                                }
                            } else {
                                // the 16 columns' (token, weight) entries and products
                                // first, then the reductions of the real columns (the
                                // table has 256 entries, so j0 + 15 is in bounds)
                                int tok[16];
#pragma unroll
                                for (int jj = 0; jj < 16; ++jj) {
                                    const int2 tw = col_tab[j0 + jj];
                                    tok[jj] = tw.x;
                                    dv[jj] *= __int_as_float(tw.y);
                                }
#pragma unroll
                                for (int jj = 0; jj < 16; ++jj)
                                    if (j0 + jj < nr)
                                        atomicAdd(p.out_acc + (size_t)tok[jj] * p.H + feat, dv[jj]);
                            }
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar_acc_empty + 8 * buf);
                        // every warp is done with the column table before any warp
                        // writes the next block's
                        named_bar_sync(kBarEpi, 128);
                    }
                }
                acc.next();
            }
        };
        if (kKind0 == 1) phase(KindC<1>{});
        if (kKind1 == 2) phase(KindC<2>{});
        report_range(range_bad, p.err);
    }

    __syncthreads();
    if (wid == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

bool plan_gemm_smem(int kind, GemmParams &p) {
    p.dq = int4_dequant_consts();
    const int BM = p.block_m;
    if (BM < 16 || BM % 16 != 0 || BM > 192) return false;
    if (kind == 3 && BM > 128) return false;  // the fused kernel runs narrow blocks
    p.np = 1;
    p.b_sub = 0;
    int n_b;
    if (BM <= 128) {
        // k blocks per B stage: gate/up two 64-wide blocks, down four (the fused
        // kernel's slots are sized for down)
        p.b_stage_bytes = (uint32_t)((kind == 1 ? 2 : 4) * BM * 128);
        // MMA issuers (one accumulator each), accumulator buffers and the A
        // stages that tensor memory then leaves, in order of preference: more A
        // stages first, then more issuers, then more buffers -- four issuers
        // with three A stages (two buffers, else one: measured faster at 32-row
        // blocks than two buffers with two A stages), then two A stages (four
        // issuers with one buffer measured faster at 64-row gate/up blocks than
        // two with two), then two issuers.  With one buffer the issuers wait for
        // the epilogue at every piece end, which the down GEMM's short pieces
        // (eight stages, an epilogue of atomics) feel most: there two issuers
        // with two buffers come first (2 % faster at 64-row blocks).
        p.ni = 0;
        int opts[6][3] = {{4, 2, 3}, {4, 1, 3}, {4, 2, 2}, {4, 1, 2}, {2, 2, 2}, {2, 1, 2}};
        if (kind == 2) {
            opts[3][0] = 2;  // {2, 2, 2} before {4, 1, 2}
            opts[3][1] = 2;
            opts[4][0] = 4;
            opts[4][1] = 1;
        }
        for (int o = 0; o < 6 && !p.ni; ++o)
            if (opts[o][0] * opts[o][1] * BM + opts[o][2] * (int)kACols <= kTmemCols) {
                p.ni = opts[o][0];
                p.nbuf = opts[o][1];
            }
        if (!p.ni) return false;
        p.n_a = (kTmemCols - p.nbuf * p.ni * BM) / (int)kACols;
        if (p.n_a > 3) p.n_a = 3;            // one named barrier per A stage (ids 2..4)
        if (p.n_a > kTeams) p.n_a = kTeams;  // a team's A-slot barrier stays within one phase
        if (p.n_a < 2) return false;
        n_b = (BM <= 32) ? 8 : (BM <= 64) ? 4 : 3;
        if (kind != 1 && BM > 32) n_b = (BM <= 64) ? 3 : 2;  // down stages carry four k blocks
    } else {
        // Wide blocks (up to 192 tokens: one pass over an expert's weights where
        // 128-token blocks would need two).  One A stage, released per sub-stage
        // half (np = 2) so the next stage's first half is written while this
        // stage's second half is multiplied.  gate/up: gate and up accumulators of
        // BM columns.  down: one issuer, two buffers of one accumulator, and B
        // slots of one sub-stage (a whole 192-row stage of four k blocks would not
        // fit in shared memory).
        p.n_a = 1;
        p.np = 2;
        p.b_stage_bytes = (uint32_t)(2 * BM * 128);
        if (kind == 1) {
            p.ni = 2;
            p.nbuf = 1;
        } else {
            // one accumulator, so two buffers fit: the epilogue of one piece
            // overlaps the MMAs of the next
            p.ni = 1;
            p.nbuf = 2;
            p.b_sub = 1;
        }
        if (p.nbuf * p.ni * BM + p.n_a * (int)kACols > kTmemCols) return false;
        n_b = 3;
    }
    const uint32_t limit = 227 * 1024 - 1024;  // opt-in maximum minus alignment slack
    p.n_b = n_b;
    const uint32_t b_bytes = (uint32_t)n_b * p.b_stage_bytes;
    // barriers + words + column table, and for the down GEMM the epilogue's
    // float4 staging (4 KB) wherever it costs no weight-ring stage (always
    // with wide blocks, whose epilogue has no other path)
    const uint32_t misc0 = 1024 + 256 * 8 + 16, stage_bytes = 4 * 1024;
    auto ring = [&](uint32_t misc_bytes) {
        const int n = (int)((limit - b_bytes - misc_bytes) / kStage);
        return n > 10 ? 10 : n;
    };
    p.epi_f4 = (kind != 1 && (p.b_sub || ring(misc0 + stage_bytes) == ring(misc0))) ? 1 : 0;
    const uint32_t misc = misc0 + (p.epi_f4 ? stage_bytes : 0u);
    const int n_w = ring(misc);
    if (n_w < 3) return false;
    p.n_w = n_w;
    const uint32_t w_bytes = (uint32_t)n_w * kStage;
    p.smem_b_off = (w_bytes + 1023u) & ~1023u;
    p.smem_misc_off = p.smem_b_off + b_bytes;
    p.smem_bytes = p.smem_misc_off + misc + 1024;  // + slack for the 1 KB alignment
    return p.smem_bytes <= 227u * 1024u;
}

cudaError_t launch_gemm(int kind, const GemmParams &p, const CUtensorMap *tmap_x,
                        const CUtensorMap *tmap_a, int grid, cudaStream_t s, int *launches) {
    const int wide = (p.np == 2 || p.b_sub) ? 1 : 0;
    const int fmt = (p.fmt == 1) ? 1 : 0;  // MOE_W_MXFP4
    if (kind < 1 || kind > 3 || (kind == 3 && wide)) return cudaErrorInvalidValue;
    const int v = (fmt * 3 + (kind - 1)) * 2 + wide;  // instantiation index
    static std::mutex mu;
    static bool attr_done[64][12] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    typedef void (*KernelFn)(const GemmParams, const CUtensorMap, const CUtensorMap);
    const KernelFn fns[12] = {moe_gemm_kernel<1, 0, 0>, moe_gemm_kernel<1, 1, 0>,
                              moe_gemm_kernel<2, 0, 0>, moe_gemm_kernel<2, 1, 0>,
                              moe_gemm_kernel<3, 0, 0>, nullptr,
                              moe_gemm_kernel<1, 0, 1>, moe_gemm_kernel<1, 1, 1>,
                              moe_gemm_kernel<2, 0, 1>, moe_gemm_kernel<2, 1, 1>,
                              moe_gemm_kernel<3, 0, 1>, nullptr};
    {
        // once per device and instantiation, under a lock (concurrent first
        // calls); a failure is returned and not recorded as done
        std::lock_guard<std::mutex> lk(mu);
        if (!attr_done[dev][v]) {
            e = cudaFuncSetAttribute(fns[v], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     227 * 1024);
            if (e != cudaSuccess) return e;
            attr_done[dev][v] = true;
        }
    }
    cudaLaunchConfig_t cfg = pdl_config((unsigned)grid, kThreads, p.smem_bytes, s);
    cudaLaunchAttribute attr;
    cfg.attrs = &attr;
    cfg.numAttrs = pdl_attr(attr);
    cudaLaunchKernelEx(&cfg, fns[v], p, *tmap_x, *tmap_a);
    if (launches) *launches += 1;
    return cudaGetLastError();
}

}  // namespace moe
