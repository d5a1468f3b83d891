// Grouped INT4 GEMMs of the MoE expert MLP on tcgen05 tensor cores (sm_103a).
//
// "The Throughput Lever" (sections "Phase 3: The INT4 Marlin MoE Throughput
// Lever" and "The Result: Two Regimes") measures the grouped INT4 MoE GEMM: below
// a few hundred tokens per call it streams the touched experts' weights from
// memory and its time grows with the number of active experts; above, every
// expert is streamed once and extra tokens ride along.  The kernel here is built
// for both regimes on one design:
//
//  * Swap-AB: the MMA's M side (128 lanes of tensor memory) is 128 weight rows,
//    its N side is the tokens routed to one expert block (16..192, the block's
//    real row count rounded up to 16), so a decode call with one token per expert
//    wastes no weight traffic.
//  * One 8 KB stage = two 128x64 INT4 slabs (+1 KB of bf16 scales), stored
//    contiguously by the pack step and fetched with one bulk TMA copy into a deep
//    shared-memory ring (the weight stream is the HBM-bound part).
//  * Eight dequant warps turn a slab row into 64 bf16 weights with the scale
//    applied ((q-8)*s: mask/OR into a bf16 with exponent 2^7, subtract 136,
//    multiply by the scale; two weights per instruction) and store them straight
//    into tensor memory, which tcgen05.mma reads as its A operand.  Shared-memory
//    bandwidth is left to the TMA writes.
//  * The B operand (activations) sits in shared memory in the 128-byte-swizzled
//    K-major layout: gathered rows of x via cp.async for gate/up, contiguous rows
//    of the intermediate via a 2-D TMA tensor copy for down.
//  * Accumulators live in tensor memory.  gate/up keeps gate and up rows of the
//    same intermediate features in the same lanes (two accumulators), so the
//    epilogue forms SiLU(g)*u in registers and writes the bf16 intermediate.  The
//    down epilogue scales by the routing weight and adds into an fp32 [M][H]
//    accumulator (the top-k combine).
//  * Work = (expert block, 128-row tile) x k iterations, split evenly over a
//    persistent grid of one CTA per SM (a k range may cut a tile).  A gate/up tile
//    cut between CTAs is finished by whichever piece arrives last (partial sums
//    in per-CTA slots + a counter; nothing spins on another CTA).
//
// Warp roles (512 threads): 0 weight producer (TMA), 1 MMA issuer + TMEM owner,
// 2 B loader, 3 idle, 4-11 dequant (4-7 slab 0, 8-11 slab 1), 12-15 epilogue.
#include <cuda_bf16.h>

#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kThreads = 512;
constexpr int kTmemCols = 512;

struct Sched {
    long long start, end;  // k-iteration range of this CTA (split mode)
    int tiles, KS, G, cta, split;
};

__device__ __forceinline__ Sched make_sched(const GemmParams &p) {
    Sched s;
    const int npp = *p.num_post_pad;
    s.tiles = (npp / p.block_m) * p.RT;
    s.KS = p.KS;
    s.G = gridDim.x;
    s.cta = blockIdx.x;
    s.split = p.split;
    const long long T = (long long)s.tiles * s.KS;
    s.start = (T * s.cta) / s.G;
    s.end = (T * (s.cta + 1)) / s.G;
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
        if (s.split) {
            if (it >= s.end) return false;
            tile = (int)(it / s.KS);
            kb0 = (int)(it % s.KS);
            const long long rem = s.end - it;
            kb1 = (s.KS - kb0 <= rem) ? s.KS : kb0 + (int)rem;
            it += kb1 - kb0;
            return true;
        }
        if (next_tile >= s.tiles) return false;
        tile = next_tile;
        kb0 = 0;
        kb1 = s.KS;
        next_tile += s.G;
        return true;
    }
};

// First iteration index of CTA c and the CTA owning iteration `it` (split mode).
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
    for (int j = lane; j < BM; j += 32) cnt += (sorted[pos0 + j] < P) ? 1 : 0;
    return __reduce_add_sync(0xffffffffu, cnt);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          uint32_t *err) {
    bool ok = mbar_wait(bar, parity, abort, err);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t dq_pair(uint32_t w, __nv_bfloat162 s2) {
    const uint32_t v = (w & 0x000F000Fu) | 0x43004300u;  // bf16 pair 128+q
    const __nv_bfloat162 c136 = __halves2bfloat162(__ushort_as_bfloat16(0x4308),
                                                   __ushort_as_bfloat16(0x4308));
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&v);
    b = __hmul2(__hsub2(b, c136), s2);
    return *reinterpret_cast<uint32_t *>(&b);
}

__device__ __forceinline__ void dequant_row(const uint4 lo, const uint4 hi, uint32_t sc,
                                            uint32_t (&out)[32]) {
    const __nv_bfloat16 s_lo = __ushort_as_bfloat16((unsigned short)(sc & 0xFFFFu));
    const __nv_bfloat16 s_hi = __ushort_as_bfloat16((unsigned short)(sc >> 16));
    const __nv_bfloat162 s0 = __halves2bfloat162(s_lo, s_lo);
    const __nv_bfloat162 s1 = __halves2bfloat162(s_hi, s_hi);
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        const __nv_bfloat162 s2 = (v < 4) ? s0 : s1;
#pragma unroll
        for (int s = 0; s < 4; ++s) out[4 * v + s] = dq_pair(w[v] >> (4 * s), s2);
    }
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    return g / (1.0f + __expf(-g)) * u;
}

}  // namespace

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const GemmParams p, const __grid_constant__ CUtensorMap tmap_a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw_addr);

    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BM = p.block_m;
    const int n_w = p.n_w, n_b = p.n_b, n_a = p.n_a;

    // shared-memory map
    const uint32_t w_ring = base;
    const uint32_t b_ring = base + p.smem_b_off;
    const uint32_t misc = base + p.smem_misc_off;
    const uint32_t bar_w_full = misc;
    const uint32_t bar_w_empty = bar_w_full + 8 * n_w;
    const uint32_t bar_b_full = bar_w_empty + 8 * n_w;
    const uint32_t bar_b_empty = bar_b_full + 8 * n_b;
    const uint32_t bar_a_full = bar_b_empty + 8 * n_b;
    const uint32_t bar_a_empty = bar_a_full + 8 * n_a;
    const uint32_t bar_acc_full = bar_a_empty + 8 * n_a;
    const uint32_t bar_acc_empty = bar_acc_full + 8;
    const uint32_t bar_drain = bar_acc_empty + 8;
    const uint32_t misc_words = bar_drain + 8;  // tmem slot, abort flag, bcast
    uint8_t *misc_ptr = smem + (misc_words - base);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(misc_ptr);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc_ptr + 4);
    volatile int *bcast = reinterpret_cast<volatile int *>(misc_ptr + 8);
    int32_t *tok_off = reinterpret_cast<int32_t *>(misc_ptr + 16);  // [BM] B-loader table

    if (threadIdx.x == 0) {
        for (int i = 0; i < n_w; ++i) {
            mbar_init(bar_w_full + 8 * i, 1);
            mbar_init(bar_w_empty + 8 * i, 8);
        }
        for (int i = 0; i < n_b; ++i) {
            mbar_init(bar_b_full + 8 * i, 1);
            mbar_init(bar_b_empty + 8 * i, 1);
        }
        for (int i = 0; i < n_a; ++i) {
            mbar_init(bar_a_full + 8 * i, 8);
            mbar_init(bar_a_empty + 8 * i, 1);
        }
        mbar_init(bar_acc_full, 1);
        mbar_init(bar_acc_empty, 4);
        mbar_init(bar_drain, 1);
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

    // tensor-memory column map
    const uint32_t col_d0 = 0;                          // gate acc (kind 1) / acc (kind 2)
    const uint32_t col_d1 = (KIND == 1) ? BM : 0;       // up acc (kind 1)
    const uint32_t col_a = (KIND == 1) ? 2 * BM : BM;   // A ring: n_a stages x 64 columns

    const Sched sched = make_sched(p);
    PieceIter pi;
    pi.init(sched);
    int tile, kb0, kb1;

    if (wid == 0) {
        // ------------------------------------------------ weight producer --
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            uint32_t i = 0;
            bool ok = true;
            while (ok && pi.next(sched, tile, kb0, kb1)) {
                const int b = tile / p.RT, r = tile % p.RT;
                const int e = p.expert_ids[b];
                const size_t st0 = ((size_t)e * p.RT + r) * p.KS;
                for (int kb = kb0; kb < kb1; ++kb, ++i) {
                    const uint32_t s = i % n_w;
                    if (!mbar_wait(bar_w_empty + 8 * s, ((i / n_w) & 1) ^ 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = w_ring + s * kStageBytes;
                    mbar_arrive_expect_tx(bar_w_full + 8 * s, kStageBytes);
                    bulk_g2s(dst, p.wq + (st0 + kb) * kStageWBytes, kStageWBytes,
                             bar_w_full + 8 * s, pol);
                    bulk_g2s(dst + kStageWBytes, p.wsc + (st0 + kb) * kStageSBytes,
                             kStageSBytes, bar_w_full + 8 * s, pol);
                }
            }
            if (!ok) {  // let copies in flight land before the CTA exits
                volatile int never = 0;
                const uint32_t first = (i > (uint32_t)n_w) ? i - n_w : 0;
                for (uint32_t j = first; j < i; ++j)
                    mbar_wait(bar_w_full + 8 * (j % n_w), (j / n_w) & 1, &never, nullptr);
            }
        }
    } else if (wid == 1) {
        // ---------------------------------------------------- MMA issuer --
        uint32_t i = 0, c = 0;
        bool ok = true;
        while (ok && pi.next(sched, tile, kb0, kb1)) {
            const int b = tile / p.RT;
            const int nr = block_rows(p.sorted_ids, b * BM, BM, p.P);
            const uint32_t n_mma = nr <= 16 ? 16u : (uint32_t)((nr + 15) & ~15);
            const uint32_t idesc = idesc_bf16_m128(n_mma);
            if (!warp_wait(bar_acc_empty, (c & 1) ^ 1, abort_flag, p.err)) { ok = false; break; }
            tc_fence_after();
            for (int kb = kb0; kb < kb1; ++kb, ++i) {
                const uint32_t as = i % n_a, bs = i % n_b;
                if (!warp_wait(bar_a_full + 8 * as, (i / n_a) & 1, abort_flag, p.err) ||
                    !warp_wait(bar_b_full + 8 * bs, (i / n_b) & 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t a0 = tmem + col_a + as * 64;
                    const uint32_t bsm = b_ring + bs * p.b_stage_bytes;
                    const uint64_t bd0 = smem_desc_sw128(bsm);
                    const uint32_t first = (kb == kb0) ? 0u : 1u;
                    if (KIND == 1) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_ts_bf16(tmem + col_d0, a0 + 8 * k, bd0 + 2 * k, idesc,
                                        (k > 0) | first);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_ts_bf16(tmem + col_d1, a0 + 32 + 8 * k, bd0 + 2 * k, idesc,
                                        (k > 0) | first);
                    } else {
                        const uint64_t bd1 = smem_desc_sw128(bsm + (uint32_t)BM * 128u);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_ts_bf16(tmem + col_d0, a0 + 8 * k, bd0 + 2 * k, idesc,
                                        (k > 0) | first);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_ts_bf16(tmem + col_d0, a0 + 32 + 8 * k, bd1 + 2 * k, idesc, 1u);
                    }
                    tc_commit(bar_a_empty + 8 * as);
                    tc_commit(bar_b_empty + 8 * bs);
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) tc_commit(bar_acc_full);
            __syncwarp();
            ++c;
        }
        // wait for every MMA issued by this warp before the CTA releases TMEM
        if (lane == 0) {
            volatile int never = 0;
            tc_commit(bar_drain);
            mbar_wait(bar_drain, 0, &never, nullptr);
        }
        __syncwarp();
    } else if (wid == 2) {
        // ------------------------------------------------------ B loader --
        uint32_t i = 0;
        bool ok = true;
        if (KIND == 1) {
            const uint32_t tile_bytes = p.b_stage_bytes;
            while (ok && pi.next(sched, tile, kb0, kb1)) {
                const int b = tile / p.RT;
                const int pos0 = b * BM;
                const int nr = block_rows(p.sorted_ids, pos0, BM, p.P);
                __syncwarp();
                for (int j = lane; j < nr; j += 32)
                    tok_off[j] = (p.sorted_ids[pos0 + j] / p.top_k) * p.H;
                __syncwarp();
                for (int kb = kb0; kb < kb1; ++kb, ++i) {
                    const uint32_t s = i % n_b;
                    if (!warp_wait(bar_b_empty + 8 * s, ((i / n_b) & 1) ^ 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst0 = b_ring + s * tile_bytes;
                    const uint16_t *src0 = p.x + kb * 64;
                    for (int idx = lane; idx < nr * 8; idx += 32) {
                        const int j = idx >> 3, ch = idx & 7;
                        cp_async_16(dst0 + j * 128 + ((ch ^ (j & 7)) << 4),
                                    src0 + tok_off[j] + ch * 8);
                    }
                    cp_async_commit();
                    if (i > 0) {
                        cp_async_wait_1();
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar_b_full + 8 * ((i - 1) % n_b));
                    }
                }
            }
            cp_async_wait_0();
            fence_proxy_async_smem();
            __syncwarp();
            if (ok && i > 0 && lane == 0) mbar_arrive(bar_b_full + 8 * ((i - 1) % n_b));
        } else {
            if (lane == 0) {
                const uint32_t bytes = 2u * BM * 128u;
                while (ok && pi.next(sched, tile, kb0, kb1)) {
                    const int b = tile / p.RT;
                    for (int kb = kb0; kb < kb1; ++kb, ++i) {
                        const uint32_t s = i % n_b;
                        if (!mbar_wait(bar_b_empty + 8 * s, ((i / n_b) & 1) ^ 1, abort_flag,
                                       p.err)) {
                            ok = false;
                            break;
                        }
                        const uint32_t dst = b_ring + s * p.b_stage_bytes;
                        mbar_arrive_expect_tx(bar_b_full + 8 * s, bytes);
                        tma_load_2d(dst, &tmap_a, (2 * kb) * 64, b * BM, bar_b_full + 8 * s);
                        tma_load_2d(dst + BM * 128, &tmap_a, (2 * kb + 1) * 64, b * BM,
                                    bar_b_full + 8 * s);
                    }
                }
                if (!ok) {
                    volatile int never = 0;
                    const uint32_t first = (i > (uint32_t)n_b) ? i - n_b : 0;
                    for (uint32_t j = first; j < i; ++j)
                        mbar_wait(bar_b_full + 8 * (j % n_b), (j / n_b) & 1, &never, nullptr);
                }
            }
        }
    } else if (wid >= 4 && wid < 12) {
        // ------------------------------------------------------- dequant --
        const int g = (wid - 4) >> 2;
        const int q = wid & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        uint32_t i = 0;
        bool ok = true;
        while (ok && pi.next(sched, tile, kb0, kb1)) {
            for (int kb = kb0; kb < kb1; ++kb, ++i) {
                const uint32_t ws = i % n_w;
                if (!warp_wait(bar_w_full + 8 * ws, (i / n_w) & 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                const uint8_t *st = smem + (size_t)ws * kStageBytes;
                const uint4 lo = *reinterpret_cast<const uint4 *>(st + g * kSlabBytes + row * 16);
                const uint4 hi =
                    *reinterpret_cast<const uint4 *>(st + g * kSlabBytes + 2048 + row * 16);
                const uint32_t sc =
                    *reinterpret_cast<const uint32_t *>(st + kStageWBytes + g * 512 + row * 4);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_w_empty + 8 * ws);
                uint32_t v[32];
                dequant_row(lo, hi, sc, v);
                const uint32_t as = i % n_a;
                if (!warp_wait(bar_a_empty + 8 * as, ((i / n_a) & 1) ^ 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_st_32x32b_x32_wait(tmem + lane_off + col_a + as * 64 + g * 32, v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_a_full + 8 * as);
            }
        }
    } else if (wid >= 12) {
        // ------------------------------------------------------ epilogue --
        const int q = wid & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const long long T = (long long)sched.tiles * sched.KS;
        uint32_t c = 0;
        bool ok = true;
        while (ok && pi.next(sched, tile, kb0, kb1)) {
            const int b = tile / p.RT, r = tile % p.RT;
            const int pos0 = b * BM;
            const int nr = block_rows(p.sorted_ids, pos0, BM, p.P);
            const bool got = warp_wait(bar_acc_full, c & 1, abort_flag, p.err);
            // the four epilogue warps leave together (they share named barrier 1)
            if (named_bar_or(1, 128, !got)) { ok = false; break; }
            tc_fence_after();
            if (KIND == 1) {
                const bool full = (kb0 == 0 && kb1 == p.KS);
                const int feat = r * kSlabRows + row;
                if (full) {
                    for (int j0 = 0; j0 < nr; j0 += 16) {
                        float gv[16], uv[16];
                        tmem_ld2_32x32b_x16_wait(tmem + lane_off + col_d0 + j0,
                                                 tmem + lane_off + col_d1 + j0, gv, uv);
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int j = j0 + jj;
                            if (j < nr)
                                p.a_out[(size_t)(pos0 + j) * p.I + feat] =
                                    __bfloat16_as_ushort(__float2bfloat16_rn(silu_mul(gv[jj], uv[jj])));
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_acc_empty);
                } else {
                    const long long piece_start = (long long)tile * p.KS + kb0;
                    const int slot = (piece_start == sched.start) ? 0 : 1;
                    float *sl = p.partial + ((size_t)(sched.cta * 2 + slot) * 2) * BM * 128;
                    for (int j0 = 0; j0 < nr; j0 += 16) {
                        float gv[16], uv[16];
                        tmem_ld2_32x32b_x16_wait(tmem + lane_off + col_d0 + j0,
                                                 tmem + lane_off + col_d1 + j0, gv, uv);
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int j = j0 + jj;
                            if (j < nr) {
                                sl[(size_t)j * 128 + row] = gv[jj];
                                sl[(size_t)(BM + j) * 128 + row] = uv[jj];
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_acc_empty);
                    __threadfence();
                    named_bar_sync(1, 128);
                    if (row == 0) {
                        const int len = kb1 - kb0;
                        const int old = atomicAdd(&p.tile_cnt[tile], len);
                        *bcast = (old + len == p.KS) ? 1 : 0;
                    }
                    named_bar_sync(1, 128);
                    const bool last = *bcast != 0;
                    named_bar_sync(1, 128);
                    if (last) {
                        __threadfence();
                        const long long ts = (long long)tile * p.KS, te = ts + p.KS;
                        const int c_first = range_owner(T, sched.G, ts);
                        const int c_last = range_owner(T, sched.G, te - 1);
                        for (int j = 0; j < nr; ++j) {
                            float gs = 0.f, us = 0.f;
                            for (int cc = c_first; cc <= c_last; ++cc) {
                                const long long cs = range_start(T, sched.G, cc);
                                if (range_start(T, sched.G, cc + 1) == cs) continue;  // empty range
                                const int sslot = (cs >= ts) ? 0 : 1;
                                const float *ps =
                                    p.partial + ((size_t)(cc * 2 + sslot) * 2) * BM * 128;
                                gs += __ldcg(ps + (size_t)j * 128 + row);
                                us += __ldcg(ps + (size_t)(BM + j) * 128 + row);
                            }
                            p.a_out[(size_t)(pos0 + j) * p.I + feat] =
                                __bfloat16_as_ushort(__float2bfloat16_rn(silu_mul(gs, us)));
                        }
                    }
                }
            } else {
                const int feat = r * kSlabRows + row;
                for (int j0 = 0; j0 < nr; j0 += 16) {
                    float dv[16];
                    tmem_ld_32x32b_x16_wait(tmem + lane_off + col_d0 + j0, dv);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = j0 + jj;
                        if (j < nr) {
                            const int pair = p.sorted_ids[pos0 + j];
                            const int t = pair / p.top_k;
                            atomicAdd(p.out_acc + (size_t)t * p.H + feat,
                                      p.topk_weights[pair] * dv[jj]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_acc_empty);
            }
            ++c;
        }
    }

    __syncthreads();
    if (wid == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

bool plan_gemm_smem(int kind, GemmParams &p) {
    const int BM = p.block_m;
    if (BM < 16 || BM % 16 != 0 || BM > 192) return false;
    p.b_stage_bytes = (uint32_t)((kind == 1 ? 1 : 2) * BM * 128);
    const int a_cols = (kind == 1) ? 2 * BM : BM;
    p.n_a = (kTmemCols - a_cols) / 64;
    if (p.n_a > 4) p.n_a = 4;
    if (p.n_a < 2) return false;
    const uint32_t limit = 227 * 1024 - 1024;  // opt-in maximum minus alignment slack
    const uint32_t misc = 1024 + 16 + 4 * 192;  // barriers + words + loader table
    int n_b = (BM <= 64) ? 4 : 3;
    if (kind == 2 && BM > 128) n_b = 2;
    p.n_b = n_b;
    const uint32_t b_bytes = (uint32_t)n_b * p.b_stage_bytes;
    int n_w = (int)((limit - b_bytes - misc) / kStageBytes);
    if (n_w > 16) n_w = 16;
    if (n_w < 4) return false;
    p.n_w = n_w;
    const uint32_t w_bytes = (uint32_t)n_w * kStageBytes;
    p.smem_b_off = (w_bytes + 1023u) & ~1023u;
    p.smem_misc_off = p.smem_b_off + b_bytes;
    p.smem_bytes = p.smem_misc_off + misc + 1024;  // + slack for the 1 KB alignment
    return p.smem_bytes <= 227u * 1024u;
}

cudaError_t launch_gemm(int kind, const GemmParams &p, const CUtensorMap *tmap_a, int grid,
                        cudaStream_t s, int *launches) {
    static bool attr_done[64][2] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev][kind - 1]) {
        cudaError_t e = (kind == 1)
            ? cudaFuncSetAttribute(moe_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   227 * 1024)
            : cudaFuncSetAttribute(moe_gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   227 * 1024);
        if (e != cudaSuccess) return e;
        attr_done[dev][kind - 1] = true;
    }
    if (kind == 1)
        moe_gemm_kernel<1><<<grid, kThreads, p.smem_bytes, s>>>(p, *tmap_a);
    else
        moe_gemm_kernel<2><<<grid, kThreads, p.smem_bytes, s>>>(p, *tmap_a);
    if (launches) *launches += 1;
    return cudaGetLastError();
}

}  // namespace moe
