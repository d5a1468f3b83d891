// Host side of the C ABI declared in include/moe_int4.h: argument checks,
// workspace planning, the launch sequence of a forward (align -> gate/up GEMM ->
// down GEMM -> finalize), tensor-map encoding, error read-back and stage timing.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <cmath>
#include <cstdlib>
#include <mutex>
#include <utility>

#include "moe_int4.h"
#include "kernels.cuh"
#include "gemv.cuh"

using namespace moe;

namespace {

constexpr int kMaxGrid = 160;          // persistent GEMM grid cap (GB300: 152 SMs)
constexpr int kSingleBlockAlignMax = 4096;
// Largest routing (pairs) that runs the fused decode kernel.  Same-box A/B
// against the separate kernels: faster at K2.6 M = 1 and 9 (8, 72 pairs) and
// mid-size M = 1 and 32 (6, 192), slower by 0.6-1 % from about 700 pairs up
// (K2.6 M = 90, verify M = 256 and 512, mid-size M = 128), where the separate
// gather kernel copies the rows faster than the fused kernel's gather share.
constexpr int kFusedMaxPairs = 512;
// The small-batch matrix-vector kernels stream each routed pair's expert on its
// own, so they run where that re-reads little: at most 128 pairs and at most
// 1.2 pairs per expert the routing is expected to touch (uniform routing), or
// at most 256 pairs when all experts together fit in half the L2, where a
// re-read is an L2 hit.  Same-box A/B against the tensor-core plans (us):
// K2.6 M = 1 47.7 / 69.3, M = 8 285 / 313, M = 9 312 / 357, M = 16 521 / 569;
// mid-size M = 1 24.2 / 34.4, M = 4 54.9 / 74.4, but M = 16 (1.8 pairs per
// touched expert) 179 / 133 and K2.6 M = 32 (1.35) 1078 / 933; the tiny shape
// M = 128 12.9 / 106.  Grouping an expert's pairs so that they share the
// weight loads (up to four per CTA, a leader CTA per group found by a search
// over the routing) measured slower at every size: 377 / 324 us at K2.6
// M = 9, 208 / 157 at mid-size M = 32; most groups hold one pair there, and the
// search and the second MMA set cost more than the re-reads.
constexpr int kGemvMaxPairs = 128;
constexpr double kGemvMaxRereads = 1.2;
constexpr int kGemvMaxPairsL2 = 256;
constexpr double kGemvL2Bytes = 64.0 * (1 << 20);
// Their k splits: slots for one wave of 4-warp CTAs over a GB300's 152 SMs at
// six resident CTAs per SM, and a CTA's fixed cost (staging, first loads) in
// units of one 64-k block of its loop.
constexpr int kGemvSlots = 152 * 6;
constexpr int kGemvCtaCost = 2;
// The separate plan's down step runs as per-block matrix-vector work (one pass
// over the expert's down rows per routing block) at blocks of up to this many
// rows.  Same-box A/B against the down GEMM (us per call): K2.6 M = 65 1 372 /
// 1 431, M = 90 1 548 / 1 593; at 32-row blocks verify M = 256 2 149 / 1 885,
// so not there.  Its CTAs (4 warps, 8 block rows per pass) run 4 per SM.
constexpr int kBlockDownMaxRows = 16;
constexpr int kBlockDownSlots = 152 * 4;
// Below kFusedMaxPairs the separate plan with this down step replaces the
// fused decode kernel at up to this many pairs per expected touched expert
// (same-box A/B, us: K2.6 M = 17 571 / 598, M = 32 894 / 956, M = 64 1 345 /
// 1 435; mid-size M = 8 94 / 102, M = 16 132 / 134; but mid-size M = 32, 3.1
// rows per expert, 166 / 157).
constexpr double kBlockDownMaxRowsPerExpert = 2.5;
constexpr int kAlignChunk = 1024;

thread_local int g_last_launches = 0;

inline size_t rup(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

int check_shape(const moe_int4_shape *sh) {
    if (!sh) return MOE_ERR_NULL;
    if (sh->E < 1 || sh->E > 1024) return MOE_ERR_SHAPE;
    if (sh->top_k < 1 || sh->top_k > sh->E || sh->top_k > 32) return MOE_ERR_SHAPE;
    if (sh->hidden < 128 || sh->hidden % 128) return MOE_ERR_SHAPE;
    if (sh->inter < 128 || sh->inter % 128) return MOE_ERR_SHAPE;
    if (sh->group != 32) return MOE_ERR_SHAPE;
    if (sh->out_dtype != MOE_OUT_BF16 && sh->out_dtype != MOE_OUT_F32) return MOE_ERR_SHAPE;
    if (sh->weight_format != MOE_W_INT4 && sh->weight_format != MOE_W_MXFP4) return MOE_ERR_SHAPE;
    if (sh->flags & ~(MOE_FLAG_UNFUSED | MOE_FLAG_NO_GEMV)) return MOE_ERR_SHAPE;
    return MOE_OK;
}

int choose_block_m(long long P, int E) {
    const long long touched = P < E ? P : E;
    const double avg = touched > 0 ? (double)P / (double)touched : 1.0;
    // Room for the busier experts: with skewed routing (a fifth of the experts
    // taking half of the assignments) those hold about 2.5x the mean, and one
    // block per expert saves a pass over its weights.  A block taller than its
    // rows costs little, since the MMA width follows the real row count.  The
    // margin 2 x mean + 8 was the faster choice for both skewed (M = 256, 1024)
    // and uniform routings.
    int bm = (int)(avg * 2.0 + 8.0);
    bm = (bm + 15) / 16 * 16;
    if (bm < 16) bm = 16;
    if (bm > 192) bm = 192;
    if (bm > 128) {
        // A wide block (144..192 rows) pays off only where it saves a pass over
        // an expert's weights: where a typical expert (its mean count plus a
        // little) needs fewer 192-row blocks than 128-row ones.  Otherwise the
        // extra blocks are short tails either way and the 128-row kernel, with
        // its deeper A ring, is faster.
        const double n = avg * 1.05;
        if (std::ceil(n / 192.0) >= std::ceil(n / 128.0)) bm = 128;
    }
    return bm;
}

struct Plan {
    int M, E, k, H, I, P, BM, RT1, RT2, n_chunks, out_f32;
    bool fused;  // the fused decode kernel (gather + gate/up + down in one launch)
    bool gemv;   // the small-batch matrix-vector kernels
    int SA, KBs, SB, KB2s;  // their k splits in 64-k blocks (gate/up over H, down over I)
    bool block_down;        // the separate plan's down step as per-block matrix-vector work
    int bd_SB, bd_KB2s;     // its k splits
    size_t cap, blocks_cap, tiles1_cap;
    size_t off_err, off_npp, off_sorted, off_expert, off_chunk, off_pos, off_cnt, off_partial, off_a,
        off_x16, off_acc, off_gu, off_io_x, off_io_ids, off_io_w, off_io_out, total, total_io;
};

Plan make_plan(int M, const moe_int4_shape *sh) {
    Plan p{};
    p.M = M;
    p.E = sh->E;
    p.k = sh->top_k;
    p.H = sh->hidden;
    p.I = sh->inter;
    p.P = M * sh->top_k;
    p.out_f32 = sh->out_dtype == MOE_OUT_F32;
    p.BM = choose_block_m(p.P, p.E);
    p.RT1 = p.I / 128;
    p.RT2 = p.H / 128;
    p.n_chunks = p.P > kSingleBlockAlignMax ? (p.P + kAlignChunk - 1) / kAlignChunk : 0;
    const size_t touched = (size_t)(p.P < p.E ? p.P : p.E);
    p.cap = (size_t)p.P + touched * (size_t)(p.BM - 1);
    p.blocks_cap = p.cap / p.BM + 1;
    p.tiles1_cap = p.blocks_cap * p.RT1;
    // expected touched experts: each token picks top_k distinct of E
    const double exp_touched = p.E * (1.0 - std::pow(1.0 - (double)p.k / p.E, (double)p.M));
    {
        const double expert_bytes = 3.0 * p.H * p.I * (0.5 + 2.0 / 32);  // weights + scales
        const bool in_l2 = p.E * expert_bytes <= kGemvL2Bytes;
        p.gemv = !(sh->flags & (MOE_FLAG_UNFUSED | MOE_FLAG_NO_GEMV)) &&
                 (in_l2 ? p.P <= kGemvMaxPairsL2
                        : p.P <= kGemvMaxPairs && p.P <= kGemvMaxRereads * exp_touched);
    }
    // The per-block down kernel where blocks are short; below the fused kernel's
    // pair limit only where they hold few rows, since with fuller blocks the
    // fused kernel's single launch wins.
    const bool block_down_ok = !p.gemv && !(sh->flags & (MOE_FLAG_UNFUSED | MOE_FLAG_NO_GEMV)) &&
                               p.BM <= kBlockDownMaxRows;
    const bool few_rows = p.P <= kBlockDownMaxRowsPerExpert * exp_touched;
    p.fused = !p.gemv && !(sh->flags & MOE_FLAG_UNFUSED) && p.P <= kFusedMaxPairs &&
              p.BM <= 128 && !(block_down_ok && few_rows);
    p.block_down = block_down_ok && !p.fused;
    if (p.gemv || p.block_down) {
        // (splits, 64-k blocks per split) of n blocks over `base` CTAs per split:
        // the fewest waves x (blocks per CTA + fixed cost), fewer splits on ties
        auto splits = [&](int base, int n, int max_per, int slots) {
            int best_sp = 1, best_per = n;
            long long best = -1;
            for (int sp = 1; sp <= n && sp <= 64; ++sp) {
                const int per = (n + sp - 1) / sp;
                if (per > max_per) continue;
                const int used = (n + per - 1) / per;
                const long long waves = ((long long)base * used + slots - 1) / slots;
                const long long cost = waves * (per + kGemvCtaCost);
                if (best < 0 || cost < best) best = cost, best_sp = used, best_per = per;
            }
            return std::make_pair(best_sp, best_per);
        };
        if (p.gemv) {
            // at most 256 blocks per split (32 KB of fp16 activations)
            const auto a = splits(p.P * p.RT1, p.H / 64, 256, kGemvSlots);
            const auto b = splits(p.P * ((p.RT2 + 1) / 2), p.I / 64, 256, kGemvSlots);
            p.SA = a.first;
            p.KBs = a.second;
            p.SB = b.first;
            p.KB2s = b.second;
        } else {
            // about one routing block per touched expert; at most 32 blocks per
            // split (eight intermediate rows of 4 KB)
            const int blocks = (int)std::ceil(exp_touched);
            const auto b = splits(blocks * ((p.RT2 + 1) / 2), p.I / 64, 32, kBlockDownSlots);
            p.bd_SB = b.first;
            p.bd_KB2s = b.second;
        }
    }
    size_t o = 0;
    p.off_err = o; o += 256;
    p.off_npp = o; o += 256;
    p.off_sorted = o; o = rup(o + p.cap * 4, 256);
    p.off_expert = o; o = rup(o + p.blocks_cap * 4, 256);
    p.off_chunk = o; o = rup(o + (size_t)p.n_chunks * p.E * 4, 256);
    p.off_pos = o; o = rup(o + (p.fused ? (size_t)p.P * 4 : 0), 256);  // pair -> position
    // counters zeroed by the align launch: gate/up split counters, then (fused
    // kernel) per-block finished gate/up tiles and the CTAs done with their
    // gather and zeroing share
    p.off_cnt = o; o = rup(o + (p.tiles1_cap + p.blocks_cap + 1) * 4, 256);
    p.off_partial = o; o = rup(o + (size_t)kMaxGrid * 4 * p.BM * 128 * 4, 256);
    p.off_a = o; o = rup(o + p.cap * (size_t)p.I * 2, 256);
    p.off_x16 = o; o = rup(o + p.cap * (size_t)p.H * 2, 256);  // x rows, bucketed, fp16
    p.off_acc = o; o = rup(o + (p.out_f32 ? 0 : (size_t)p.M * p.H * 4), 256);
    p.off_gu = o; o = rup(o + (p.gemv ? (size_t)p.SA * p.P * 2 * p.I * 4 : 0), 256);
    p.total = o;
    p.off_io_x = o; o = rup(o + (size_t)p.M * p.H * 2, 256);
    p.off_io_ids = o; o = rup(o + (size_t)p.P * 4, 256);
    p.off_io_w = o; o = rup(o + (size_t)p.P * 4, 256);
    p.off_io_out = o; o = rup(o + (size_t)p.M * p.H * (p.out_f32 ? 4 : 2), 256);
    p.total_io = o;
    return p;
}

struct DeviceInfo {
    int sms = 0;
    int ok = -1;  // -1 unknown, 0 unsupported, 1 sm_103
};
std::mutex g_mu;
DeviceInfo g_dev[64];

int device_info(int *sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (d.ok < 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_ERR_CUDA;
        d.ok = (major == 10 && minor == 3) ? 1 : 0;
    }
    if (!d.ok) return MOE_ERR_UNSUPPORTED;
    *sms = d.sms;
    return MOE_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Tensor map over fp16 rows [rows][cols] (bucketed x or the intermediate), box
// = 64 columns x BM rows, 128-byte swizzle (the MMA's K-major B layout).
bool encode_rows_map(CUtensorMap *m, void *a, size_t rows, int I, int BM) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)I, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)I * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)BM};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// ---------------------------------------------------------------- profiling --
struct Profiler {
    bool on = false;
    bool recorded = false;
    int dev = -1;
    cudaEvent_t ev[5] = {};
};
Profiler g_prof;

void prof_record(int i, cudaStream_t s) {
    if (g_prof.on && g_prof.ev[i]) cudaEventRecord(g_prof.ev[i], s);
}

}  // namespace

extern "C" {

size_t moe_int4_packed_bytes(int E, int N, int K) {
    if (E <= 0 || N <= 0 || K <= 0) return 0;
    return (size_t)E * N * (size_t)(K / 2);
}

size_t moe_int4_packed_scale_bytes(int E, int N, int K) {
    if (E <= 0 || N <= 0 || K <= 0) return 0;
    return (size_t)E * N * (size_t)(K / 32) * 2;
}

int moe_int4_pack(const uint8_t *q, const uint16_t *scales, int E, int N, int K, int is_w13,
                  void *packed, void *packed_scales, uint32_t *inexact_scales,
                  moe_stream_t stream) {
    if (!q || !scales || !packed || !packed_scales) return MOE_ERR_NULL;
    if (E < 1 || N < 1 || K < 1) return MOE_ERR_SHAPE;
    if (is_w13) {
        if (N % 256 || K % 64) return MOE_ERR_SHAPE;
    } else {
        if (N % 128 || K % 128) return MOE_ERR_SHAPE;
    }
    if (!aligned16(q) || !aligned16(scales) || !aligned16(packed) || !aligned16(packed_scales))
        return MOE_ERR_ALIGN;
    cudaError_t e = launch_pack(q, scales, E, N, K, is_w13, packed, packed_scales,
                                inexact_scales, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_mxfp4_pack(const uint8_t *q, const uint8_t *scales, int E, int N, int K, int is_w13,
                   void *packed, void *packed_scales, uint32_t *bad_scales,
                   moe_stream_t stream) {
    if (!q || !scales || !packed || !packed_scales) return MOE_ERR_NULL;
    if (E < 1 || N < 1 || K < 1) return MOE_ERR_SHAPE;
    if (is_w13) {
        if (N % 256 || K % 64) return MOE_ERR_SHAPE;
    } else {
        if (N % 128 || K % 128) return MOE_ERR_SHAPE;
    }
    if (!aligned16(q) || !aligned16(scales) || !aligned16(packed) || !aligned16(packed_scales))
        return MOE_ERR_ALIGN;
    cudaError_t e = launch_pack_mxfp4(q, scales, E, N, K, is_w13, packed, packed_scales,
                                      bad_scales, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

size_t moe_align_capacity(int M, int top_k, int E, int block_m) {
    if (M < 0 || top_k < 1 || E < 1 || block_m < 1) return 0;
    const long long P = (long long)M * top_k;
    const long long touched = P < E ? P : E;
    return (size_t)(P + touched * (block_m - 1));
}

size_t moe_align_scratch_bytes(int M, int top_k, int E) {
    if (M < 0 || top_k < 1 || E < 1) return 0;
    const long long P = (long long)M * top_k;
    if (P <= kSingleBlockAlignMax) return 0;
    return (size_t)((P + kAlignChunk - 1) / kAlignChunk) * E * 4;
}

int moe_align(const int32_t *topk_ids, int M, int top_k, int E, int block_m,
              int32_t *sorted_ids, int32_t *expert_ids, int32_t *num_post_pad,
              uint32_t *err_flags, void *scratch, size_t scratch_bytes, moe_stream_t stream) {
    if (M < 0 || top_k < 1 || top_k > 32 || E < 1 || E > 1024 || block_m < 1 || block_m > 256)
        return MOE_ERR_SHAPE;
    if ((long long)M * top_k > (1LL << 30)) return MOE_ERR_SHAPE;
    if (!num_post_pad || (M > 0 && (!topk_ids || !sorted_ids || !expert_ids)))
        return MOE_ERR_NULL;
    const size_t need = moe_align_scratch_bytes(M, top_k, E);
    if (need && (!scratch || scratch_bytes < need)) return MOE_ERR_WORKSPACE;
    AlignArgs a{};
    a.ids = topk_ids;
    a.P = M * top_k;
    a.E = E;
    a.block_m = block_m;
    a.sorted_ids = sorted_ids;
    a.expert_ids = expert_ids;
    a.num_post_pad = num_post_pad;
    a.err = err_flags;
    a.chunk_tab = reinterpret_cast<int32_t *>(scratch);
    a.n_chunks = need ? (a.P + kAlignChunk - 1) / kAlignChunk : 0;
    ZeroArgs z{};
    cudaError_t e = launch_align(a, z, 0, reinterpret_cast<cudaStream_t>(stream), nullptr);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

size_t moe_int4_workspace_bytes(int M, const moe_int4_shape *shape, int flags) {
    if (check_shape(shape) != MOE_OK || M < 0 || M > (1 << 20)) return 0;
    if (M == 0) return 256;
    Plan p = make_plan(M, shape);
    return (flags & MOE_WS_HOST_IO) ? p.total_io : p.total;
}

int moe_int4_fused(int M, const moe_int4_shape *shape) {
    if (check_shape(shape) != MOE_OK || M < 1 || M > (1 << 20)) return 0;
    return make_plan(M, shape).fused ? 1 : 0;
}

int moe_int4_block_down(int M, const moe_int4_shape *shape) {
    if (check_shape(shape) != MOE_OK || M < 1 || M > (1 << 20)) return 0;
    return make_plan(M, shape).block_down ? 1 : 0;
}

int moe_int4_gemv(int M, const moe_int4_shape *shape) {
    if (check_shape(shape) != MOE_OK || M < 1 || M > (1 << 20)) return 0;
    return make_plan(M, shape).gemv ? 1 : 0;
}

int moe_int4_block_m(int M, const moe_int4_shape *shape) {
    if (check_shape(shape) != MOE_OK || M < 0) return 0;
    return choose_block_m((long long)M * shape->top_k, shape->E);
}

int moe_int4_workspace_layout(int M, const moe_int4_shape *shape, size_t *offsets) {
    if (!offsets) return MOE_ERR_NULL;
    const int rc = check_shape(shape);
    if (rc != MOE_OK) return rc;
    if (M < 1 || M > (1 << 20)) return MOE_ERR_SHAPE;
    const Plan p = make_plan(M, shape);
    offsets[0] = p.off_err;
    offsets[1] = p.off_npp;
    offsets[2] = p.off_sorted;
    offsets[3] = p.off_expert;
    offsets[4] = p.off_a;
    offsets[5] = p.off_acc;
    return MOE_OK;
}

}  // extern "C"

namespace {

// The forward; with router_logits set, the routing (topk_ids / topk_weights,
// written) is computed in the align launch, else it is read from them.
int forward_impl(const uint16_t *x, const void *w13_packed, const void *w13_scales,
                 const void *w2_packed, const void *w2_scales, const float *router_logits,
                 const int32_t *topk_ids, const float *topk_weights, void *out, int M,
                 const moe_int4_shape *shape, void *workspace, size_t workspace_bytes,
                 moe_stream_t stream) {
    g_last_launches = 0;
    int rc = check_shape(shape);
    if (rc != MOE_OK) return rc;
    if (M < 0 || M > (1 << 20)) return MOE_ERR_SHAPE;
    if (M == 0) return MOE_OK;
    if (!x || !w13_packed || !w13_scales || !w2_packed || !w2_scales || !topk_ids ||
        !topk_weights || !out || !workspace)
        return MOE_ERR_NULL;
    const void *ptrs[] = {x, w13_packed, w13_scales, w2_packed, w2_scales, topk_ids,
                          topk_weights, out, workspace, router_logits};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_ALIGN;
    const Plan pl = make_plan(M, shape);
    if (workspace_bytes < pl.total) return MOE_ERR_WORKSPACE;
    int sms = 0;
    rc = device_info(&sms);
    if (rc != MOE_OK) return rc;
    const int grid = sms < kMaxGrid ? sms : kMaxGrid;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
    int launches = 0;

    uint32_t *err = reinterpret_cast<uint32_t *>(ws + pl.off_err);
    int32_t *npp = reinterpret_cast<int32_t *>(ws + pl.off_npp);
    int32_t *sorted = reinterpret_cast<int32_t *>(ws + pl.off_sorted);
    int32_t *expert = reinterpret_cast<int32_t *>(ws + pl.off_expert);
    uint16_t *a_buf = reinterpret_cast<uint16_t *>(ws + pl.off_a);
    // fp32 output: the down GEMM accumulates straight into `out`
    float *acc = pl.out_f32 ? reinterpret_cast<float *>(out)
                            : reinterpret_cast<float *>(ws + pl.off_acc);

    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_prof.on) {
            int dev = 0;
            cudaGetDevice(&dev);
            if (g_prof.dev != dev) {
                for (auto &e : g_prof.ev)
                    if (e) cudaEventDestroy(e), e = nullptr;
                for (auto &e : g_prof.ev) cudaEventCreate(&e);
                g_prof.dev = dev;
            }
            g_prof.recorded = true;
        }
    }
    prof_record(0, s);

    if (pl.gemv) {
        // a few tokens: matrix-vector kernels on the CUDA cores, no align
        if (router_logits) {
            RouteArgs ra{};
            ra.logits = router_logits;
            ra.M = pl.M;
            ra.E = pl.E;
            ra.top_k = pl.k;
            ra.ids = const_cast<int32_t *>(topk_ids);
            ra.weights = const_cast<float *>(topk_weights);
            if (launch_route(ra, sms, s, &launches) != cudaSuccess) return MOE_ERR_CUDA;
        }
        prof_record(1, s);
        GemvArgs ga{};
        ga.x = x;
        ga.ids = topk_ids;
        ga.topk_weights = topk_weights;
        ga.w13 = reinterpret_cast<const uint8_t *>(w13_packed);
        ga.s13 = reinterpret_cast<const uint8_t *>(w13_scales);
        ga.w2 = reinterpret_cast<const uint8_t *>(w2_packed);
        ga.s2 = reinterpret_cast<const uint8_t *>(w2_scales);
        ga.gu = reinterpret_cast<float *>(ws + pl.off_gu);
        ga.out = acc;
        ga.out_n16 = (size_t)pl.M * pl.H / 4;
        ga.err = err;
        ga.M = pl.M;
        ga.top_k = pl.k;
        ga.P = pl.P;
        ga.E = pl.E;
        ga.H = pl.H;
        ga.I = pl.I;
        ga.RT1 = pl.RT1;
        ga.KB = pl.H / 64;
        ga.SA = pl.SA;
        ga.KBs = pl.KBs;
        ga.RT2 = pl.RT2;
        ga.KB2 = pl.I / 64;
        ga.SB = pl.SB;
        ga.KB2s = pl.KB2s;
        ga.fmt = shape->weight_format;
        ga.dq = int4_dequant_consts();
        if (launch_gemv(ga, 1, s, &launches) != cudaSuccess) return MOE_ERR_CUDA;
        prof_record(2, s);
        if (launch_gemv(ga, 2, s, &launches) != cudaSuccess) return MOE_ERR_CUDA;
        prof_record(3, s);
        if (!pl.out_f32 && launch_finalize(acc, reinterpret_cast<uint16_t *>(out),
                                           (size_t)pl.M * pl.H, sms, s, &launches) != cudaSuccess)
            return MOE_ERR_CUDA;
        prof_record(4, s);
        g_last_launches = launches;
        return MOE_OK;
    }

    AlignArgs al{};
    al.ids = topk_ids;
    al.P = pl.P;
    al.E = pl.E;
    al.block_m = pl.BM;
    al.sorted_ids = sorted;
    al.expert_ids = expert;
    al.num_post_pad = npp;
    al.err = err;
    al.chunk_tab = reinterpret_cast<int32_t *>(ws + pl.off_chunk);
    al.n_chunks = pl.n_chunks;
    al.pos_of = pl.fused ? reinterpret_cast<int32_t *>(ws + pl.off_pos) : nullptr;
    // the align launch zeroes the counters; the gate/up GEMM (or the fused
    // kernel) zeroes the down accumulator (off the align's critical path)
    ZeroArgs z{};
    z.ptr[0] = ws + pl.off_cnt;
    z.n16[0] = ((pl.tiles1_cap + pl.blocks_cap + 1) * 4 + 15) / 16;
    uint16_t *x16 = reinterpret_cast<uint16_t *>(ws + pl.off_x16);
    const size_t zero_bytes = (z.n16[0] + z.n16[1]) * 16;
    int zero_ctas = (int)(zero_bytes / (64 * 1024));
    if (zero_ctas < 1) zero_ctas = 1;
    if (zero_ctas > 2 * sms) zero_ctas = 2 * sms;
    if (router_logits) {
        RouteArgs ra{};
        ra.logits = router_logits;
        ra.M = pl.M;
        ra.E = pl.E;
        ra.top_k = pl.k;
        ra.ids = const_cast<int32_t *>(topk_ids);
        ra.weights = const_cast<float *>(topk_weights);
        if (launch_route_align(ra, al, z, zero_ctas, sms, s, &launches) != cudaSuccess)
            return MOE_ERR_CUDA;
    } else if (launch_align(al, z, zero_ctas, s, &launches) != cudaSuccess) {
        return MOE_ERR_CUDA;
    }
    if (!pl.fused && launch_gather_rows(x, sorted, npp, pl.P, pl.k, pl.H, x16, pl.cap, err, sms,
                                        s, &launches) != cudaSuccess)
        return MOE_ERR_CUDA;
    prof_record(1, s);

    GemmParams g{};
    g.sorted_ids = sorted;
    g.expert_ids = expert;
    g.num_post_pad = npp;
    g.topk_weights = topk_weights;
    g.err = err;
    g.M = pl.M;
    g.top_k = pl.k;
    g.H = pl.H;
    g.I = pl.I;
    g.P = pl.P;
    g.E = pl.E;
    g.cap = pl.cap > (size_t)INT32_MAX ? INT32_MAX : (int)pl.cap;
    g.block_m = pl.BM;
    g.round_robin = 1;
    g.fmt = shape->weight_format;
    g.skip_stage = -1;
#ifdef MOE_DEBUG_BOUNDS
    // the debug build's timeout test: MOE_INT4_DEBUG_SKIP_STAGE=i makes CTA 0
    // of the first GEMM kernel leave its weight stage i out (see GemmParams)
    if (const char *v = getenv("MOE_INT4_DEBUG_SKIP_STAGE")) g.skip_stage = atoi(v);
#endif

    int32_t *cnt = reinterpret_cast<int32_t *>(ws + pl.off_cnt);
    g.g[0].wq = reinterpret_cast<const uint8_t *>(w13_packed);
    g.g[0].wsc = reinterpret_cast<const uint8_t *>(w13_scales);
    g.g[0].RT = pl.RT1;
    g.g[0].KSS = pl.H / 64;
    g.g[0].KS = (g.g[0].KSS + 1) / 2;
    g.g[1].wq = reinterpret_cast<const uint8_t *>(w2_packed);
    g.g[1].wsc = reinterpret_cast<const uint8_t *>(w2_scales);
    g.g[1].RT = pl.RT2;
    g.g[1].KSS = pl.I / 128;
    g.g[1].KS = (g.g[1].KSS + 1) / 2;
    g.a_out = a_buf;
    g.partial = reinterpret_cast<float *>(ws + pl.off_partial);
    g.tile_cnt = cnt;
    g.out_acc = acc;
    CUtensorMap tmap_x, tmap_a;
    if (!encode_rows_map(&tmap_x, x16, pl.cap, pl.H, pl.BM) ||
        !encode_rows_map(&tmap_a, a_buf, pl.cap, pl.I, pl.BM))
        return MOE_ERR_CUDA;

    if (pl.fused) {
        // one persistent kernel: gather, gate/up + SwiGLU, down + combine
        GemmParams gf = g;
        gf.zero_out = reinterpret_cast<float4 *>(acc);
        gf.zero_n16 = (size_t)pl.M * pl.H * 4 / 16;
        gf.x = x;
        gf.x16 = x16;
        gf.pos_of = al.pos_of;
        gf.blk_done = cnt + pl.tiles1_cap;
        gf.prep_done = cnt + pl.tiles1_cap + pl.blocks_cap;
        if (!plan_gemm_smem(3, gf)) return MOE_ERR_SHAPE;
        if (launch_gemm(3, gf, &tmap_x, &tmap_a, grid, s, &launches) != cudaSuccess)
            return MOE_ERR_CUDA;
        prof_record(2, s);
        prof_record(3, s);
    } else {
        GemmParams g1 = g;
        g1.zero_out = reinterpret_cast<float4 *>(acc);
        g1.zero_n16 = (size_t)pl.M * pl.H * 4 / 16;
        if (!plan_gemm_smem(1, g1)) return MOE_ERR_SHAPE;
        if (launch_gemm(1, g1, &tmap_x, &tmap_a, grid, s, &launches) != cudaSuccess)
            return MOE_ERR_CUDA;
        prof_record(2, s);
        if (pl.block_down) {
            BlockDownArgs bd{};
            bd.sorted_ids = sorted;
            bd.expert_ids = expert;
            bd.num_post_pad = npp;
            bd.a_out = a_buf;
            bd.topk_weights = topk_weights;
            bd.w2 = reinterpret_cast<const uint8_t *>(w2_packed);
            bd.s2 = reinterpret_cast<const uint8_t *>(w2_scales);
            bd.out = acc;
            bd.err = err;
            bd.P = pl.P;
            bd.E = pl.E;
            bd.H = pl.H;
            bd.I = pl.I;
            bd.top_k = pl.k;
            bd.block_m = pl.BM;
            bd.blocks_cap = (int)pl.blocks_cap;
            bd.cap = g.cap;
            bd.RT2 = pl.RT2;
            bd.KB2 = pl.I / 64;
            bd.SB = pl.bd_SB;
            bd.KB2s = pl.bd_KB2s;
            bd.fmt = shape->weight_format;
            bd.dq = int4_dequant_consts();
            if (launch_block_down(bd, s, &launches) != cudaSuccess) return MOE_ERR_CUDA;
        } else {
            GemmParams g2 = g;
            g2.skip_stage = -1;
            if (!plan_gemm_smem(2, g2)) return MOE_ERR_SHAPE;
            if (launch_gemm(2, g2, &tmap_x, &tmap_a, grid, s, &launches) != cudaSuccess)
                return MOE_ERR_CUDA;
        }
        prof_record(3, s);
    }

    if (!pl.out_f32 && launch_finalize(acc, reinterpret_cast<uint16_t *>(out),
                                       (size_t)pl.M * pl.H, sms, s, &launches) != cudaSuccess)
        return MOE_ERR_CUDA;
    prof_record(4, s);
    g_last_launches = launches;
    return MOE_OK;
}

}  // namespace

extern "C" {

int moe_int4_forward(const uint16_t *x, const void *w13_packed, const void *w13_scales,
                     const void *w2_packed, const void *w2_scales, const int32_t *topk_ids,
                     const float *topk_weights, void *out, int M,
                     const moe_int4_shape *shape, void *workspace, size_t workspace_bytes,
                     moe_stream_t stream) {
    return forward_impl(x, w13_packed, w13_scales, w2_packed, w2_scales, nullptr, topk_ids,
                        topk_weights, out, M, shape, workspace, workspace_bytes, stream);
}

int moe_int4_forward_routed(const uint16_t *x, const void *w13_packed, const void *w13_scales,
                            const void *w2_packed, const void *w2_scales,
                            const float *router_logits, int32_t *topk_ids, float *topk_weights,
                            void *out, int M, const moe_int4_shape *shape, void *workspace,
                            size_t workspace_bytes, moe_stream_t stream) {
    if (M > 0 && !router_logits) return MOE_ERR_NULL;
    return forward_impl(x, w13_packed, w13_scales, w2_packed, w2_scales, router_logits,
                        topk_ids, topk_weights, out, M, shape, workspace, workspace_bytes,
                        stream);
}

int moe_route(const float *router_logits, int M, int E, int top_k, int32_t *topk_ids,
              float *topk_weights, moe_stream_t stream) {
    if (M < 0 || M > (1 << 20) || E < 1 || E > 1024 || top_k < 1 || top_k > 32 || top_k > E)
        return MOE_ERR_SHAPE;
    if (M == 0) return MOE_OK;
    if (!router_logits || !topk_ids || !topk_weights) return MOE_ERR_NULL;
    int sms = 0;
    const int rc = device_info(&sms);
    if (rc != MOE_OK) return rc;
    RouteArgs ra{};
    ra.logits = router_logits;
    ra.M = M;
    ra.E = E;
    ra.top_k = top_k;
    ra.ids = topk_ids;
    ra.weights = topk_weights;
    return launch_route(ra, sms, reinterpret_cast<cudaStream_t>(stream), nullptr) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

int moe_int4_forward_host(const uint16_t *x_host, const void *w13_packed,
                          const void *w13_scales, const void *w2_packed, const void *w2_scales,
                          const int32_t *topk_ids_host, const float *topk_weights_host,
                          void *out_host, int M, const moe_int4_shape *shape,
                          void *workspace, size_t workspace_bytes, moe_stream_t stream) {
    int rc = check_shape(shape);
    if (rc != MOE_OK) return rc;
    if (M < 0 || M > (1 << 20)) return MOE_ERR_SHAPE;
    if (M == 0) return MOE_OK;
    if (!x_host || !topk_ids_host || !topk_weights_host || !out_host || !workspace)
        return MOE_ERR_NULL;
    const Plan pl = make_plan(M, shape);
    if (workspace_bytes < pl.total_io) return MOE_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MOE_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
    uint16_t *dx = reinterpret_cast<uint16_t *>(ws + pl.off_io_x);
    int32_t *dids = reinterpret_cast<int32_t *>(ws + pl.off_io_ids);
    float *dw = reinterpret_cast<float *>(ws + pl.off_io_w);
    void *dout = ws + pl.off_io_out;
    const size_t out_bytes = (size_t)M * pl.H * (pl.out_f32 ? 4 : 2);
    if (cudaMemcpyAsync(dx, x_host, (size_t)M * pl.H * 2, cudaMemcpyHostToDevice, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(dids, topk_ids_host, (size_t)pl.P * 4, cudaMemcpyHostToDevice, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(dw, topk_weights_host, (size_t)pl.P * 4, cudaMemcpyHostToDevice, s) !=
            cudaSuccess)
        return MOE_ERR_CUDA;
    rc = moe_int4_forward(dx, w13_packed, w13_scales, w2_packed, w2_scales, dids, dw, dout, M,
                          shape, workspace, pl.total, stream);
    if (rc != MOE_OK) return rc;
    if (cudaMemcpyAsync(out_host, dout, out_bytes, cudaMemcpyDeviceToHost, s) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_int4_get_errors(const void *workspace, uint32_t *flags, uint32_t *count,
                        moe_stream_t stream) {
    if (!workspace) return MOE_ERR_NULL;
    uint32_t h[2] = {0, 0};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(h, workspace, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (flags) *flags = h[0];
    if (count) *count = h[1];
    return MOE_OK;
}

int moe_int4_clear_errors(void *workspace, moe_stream_t stream) {
    if (!workspace) return MOE_ERR_NULL;
    return cudaMemsetAsync(workspace, 0, 8, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

const char *moe_int4_strerror(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_NULL: return "a required pointer is NULL";
        case MOE_ERR_SHAPE: return "unsupported or inconsistent sizes";
        case MOE_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "a CUDA runtime call failed";
        case MOE_ERR_UNSUPPORTED: return "device is not compute capability 10.3 (sm_103a)";
        case MOE_ERR_NOALLOC_LIMIT: return "routing too large for moe_align_noalloc's 1 MiB scratch";
        default: return "unknown error code";
    }
}

int moe_int4_profile_enable(int on) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_prof.on = on != 0;
    g_prof.recorded = false;
    return MOE_OK;
}

int moe_int4_profile_read(float *ms) {
    if (!ms) return MOE_ERR_NULL;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_prof.recorded || !g_prof.ev[4]) return MOE_ERR_CUDA;
    if (cudaEventSynchronize(g_prof.ev[4]) != cudaSuccess) return MOE_ERR_CUDA;
    for (int i = 0; i < 4; ++i)
        if (cudaEventElapsedTime(&ms[i], g_prof.ev[i], g_prof.ev[i + 1]) != cudaSuccess)
            return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_int4_last_launch_count(void) { return g_last_launches; }

}  // extern "C"
