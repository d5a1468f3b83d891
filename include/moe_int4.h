/*
 * moe_int4.h -- C ABI of the weight-only INT4 MoE expert-MLP library for one
 * NVIDIA GB300 (sm_103a).
 *
 * The layer (pages: "The Throughput Lever: Quantifying the MoE GEMM and Mapping
 * the Road to B300", sections "Phase 3: The INT4 Marlin MoE Throughput Lever",
 * "Building the Benchmark" and "The Result: Two Regimes"):
 *
 *   for every token t and routing slot j with expert e = topk_ids[t, j]:
 *     g = W_gate[e] x_t,  u = W_up[e] x_t          (gate/up grouped GEMM)
 *     a = SiLU(g) * u                              (SwiGLU, fused in the epilogue)
 *     y = W_down[e] a                              (down grouped GEMM)
 *     out[t] = sum_j topk_weights[t, j] * y        (top-k weighted combine)
 *
 * with INT4 weights in groups of 32 along the reduction axis, each weight
 * value = (q - 8) * scale, q in {0..15}, scale bf16 ("Building the Benchmark":
 * INT4, group size 32).  Activations are bf16 and the output bf16 or fp32.  The
 * tensor cores multiply fp16 operands with fp32 accumulation: each dequantised
 * weight (q - 8) * scale is formed in fp16 with one rounding (11 significant
 * bits, where bf16 would keep 8; it is exact for scales in [2^-14, 2729], since
 * a bf16 scale's 8 significant bits times |q - 8| <= 8 fit in 11 and the
 * kernels' addend -24 * scale stays in range, and moe_int4_pack counts the
 * scales outside that range), x is converted to fp16
 * (exact for |x| in [2^-14, 65504]; below, fp16 subnormals are within 2^-25 of
 * x), and the SwiGLU intermediate is stored as fp16.  An x element or an
 * intermediate beyond +-65504 (or not finite) is saturated to +-65504 and
 * raises the device flag MOE_DEVERR_RANGE: such a call's output is not valid.
 *
 * Conventions for every entry point:
 *  - All array pointers are DEVICE pointers owned by the caller, except those of
 *    moe_int4_forward_host (host pointers, documented there).  The library never
 *    frees or keeps caller memory past the call's stream work.
 *  - Every call is stream-ordered and asynchronous on `stream` (a cudaStream_t;
 *    NULL is the legacy default stream); none synchronises the host, except
 *    moe_int4_get_errors, which reads back a few bytes, and moe_int4_forward_host,
 *    which waits for its result.  No call allocates device memory.
 *  - bf16 values are passed as their 16-bit patterns (uint16_t).
 *  - Return value: MOE_OK (0) or a negative MOE_ERR_* code detected on the host
 *    before anything is launched.  Bad data found on the device (an expert id
 *    outside [0, E)) does not trap: the routing pair is dropped, and a flag and
 *    a count are recorded in the workspace (moe_int4_get_errors).
 */
#ifndef MOE_INT4_H
#define MOE_INT4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* same type as cudaStream_t */

enum {
    MOE_OK = 0,
    MOE_ERR_NULL = -1,        /* a required pointer is NULL */
    MOE_ERR_SHAPE = -2,       /* unsupported or inconsistent sizes */
    MOE_ERR_ALIGN = -3,       /* a pointer is not 16-byte aligned */
    MOE_ERR_WORKSPACE = -4,   /* workspace too small */
    MOE_ERR_CUDA = -5,        /* a CUDA runtime call failed (launch, copy) */
    MOE_ERR_UNSUPPORTED = -6, /* current device is not compute capability 10.3 */
    MOE_ERR_NOALLOC_LIMIT = -7 /* too large for moe_align_noalloc's fixed scratch */
};

/* Device-side error flags (bit set), read with moe_int4_get_errors. */
#define MOE_DEVERR_BAD_EXPERT_ID 0x1u /* a topk_ids entry outside [0, E) was dropped */
#define MOE_DEVERR_TIMEOUT 0x2u       /* a pipeline wait gave up (kernel bug guard) */
#define MOE_DEVERR_BOUNDS 0x4u        /* debug-bounds builds only (-DMOE_DEBUG_BOUNDS): an index
                                         read back from a routing buffer was out of range; the
                                         access was kept in bounds and the result is invalid */
#define MOE_DEVERR_RANGE 0x8u         /* a value outside fp16's finite range reached an fp16
                                         tensor-core operand and was saturated to +-65504: an x
                                         element or a SwiGLU intermediate beyond +-65504,
                                         infinite or NaN; the output is not valid */

/* Output element types (moe_int4_shape.out_dtype). */
#define MOE_OUT_BF16 0 /* bf16, rounded to nearest even from the fp32 combine */
#define MOE_OUT_F32 1  /* the fp32 combine itself */

/* Expert weight formats (moe_int4_shape.weight_format), both with one scale per
 * 32 consecutive elements along the reduction axis:
 *   MOE_W_INT4   value = (q - 8) * scale, q in 0..15, scale bf16 (moe_int4_pack).
 *   MOE_W_MXFP4  value = e2m1(q) * 2^(e - 127): q an FP4 E2M1 code (bit 3 sign,
 *                bits 2..1 exponent with bias 1, bit 0 mantissa, exponent 0
 *                subnormal: 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives), e an
 *                E8M0 scale byte (OCP Microscaling v1.0; "From 1,060 to 4,016
 *                tok/s on one B300": MXFP4 experts) -- moe_mxfp4_pack. */
#define MOE_W_INT4 0
#define MOE_W_MXFP4 1

/* Forward flags (moe_int4_shape.flags). */
#define MOE_FLAG_UNFUSED 0x1 /* run the gather, gate/up and down steps as separate
                                tensor-core kernels even where the fused decode kernel or
                                the small-batch path applies (same results) */
#define MOE_FLAG_NO_GEMV 0x2 /* keep to the tensor-core kernels (fused where it applies)
                                where the matrix-vector kernels would run */

/* Layer shape.  Supported: 1 <= E <= 1024, 1 <= top_k <= min(E, 32),
 * hidden % 128 == 0, inter % 128 == 0, group == 32, weight_format one of
 * MOE_W_*, flags a combination of MOE_FLAG_*.  Zero-initialised weight_format and
 * flags mean INT4 and the default launch plan. */
typedef struct {
    int32_t E;             /* number of experts */
    int32_t top_k;         /* routing slots per token */
    int32_t hidden;        /* H: model width (K of the gate/up GEMM, N of the down GEMM) */
    int32_t inter;         /* I: expert intermediate width */
    int32_t group;         /* quantisation group along K; must be 32 */
    int32_t out_dtype;     /* MOE_OUT_BF16 or MOE_OUT_F32 */
    int32_t weight_format; /* MOE_W_INT4 or MOE_W_MXFP4 (how the weights were packed) */
    int32_t flags;         /* MOE_FLAG_* */
} moe_int4_shape;

/* ------------------------------------------------------------------------- */
/* Weight packing (offline, once per weight set; "Building the Benchmark":     */
/* the pages repack GPTQ-format INT4 into the kernel's layout before timing)   */
/* ------------------------------------------------------------------------- */

/* Bytes of the packed INT4 buffer for E matrices of N rows x K columns:
 * E*N*K/2 (same size as the canonical input). */
size_t moe_int4_packed_bytes(int E, int N, int K);
/* Bytes of the packed scale buffer: E*N*(K/32)*2. */
size_t moe_int4_packed_scale_bytes(int E, int N, int K);

/*
 * moe_int4_pack: canonical INT4 weights -> device layout of the GEMM kernels.
 *
 * In:  q       uint8 [E][N][K/2]; element k of a row is in byte k/2, low nibble
 *              for even k, high nibble for odd k; value = (q - 8) * scale.
 *      scales  bf16 bits [E][N][K/32]; one scale per 32 consecutive k.
 *      is_w13  1: the gate/up matrix, N = 2*inter (rows [0,inter) gate,
 *              [inter, 2*inter) up), K = hidden.  0: the down matrix, N = hidden,
 *              K = inter.
 * Out: packed (moe_int4_packed_bytes) and packed_scales
 *      (moe_int4_packed_scale_bytes), caller-allocated, 16-byte aligned.
 *
 * Packed layout (a "slab" is 128 rows x 64 k; a "stage" is two slabs):
 *   w13: stage (e, r, kb) for row tile r in [0, inter/128) and k block kb in
 *        [0, hidden/64): slab 0 = gate rows 128r..128r+127, slab 1 = up rows
 *        inter+128r.., both for k in [64kb, 64kb+64).
 *   w2:  stage (e, r, ks) for r in [0, hidden/128), ks in [0, inter/128):
 *        slab 0 = rows 128r.. for k block 2ks, slab 1 = same rows, k block 2ks+1.
 *   Stages are stored in order e, r, then k (8192 bytes each).  Inside a slab,
 *   byte offset h*2048 + row*16 + w*4 holds word v = 4h + w of the row; bits
 *   4s..4s+3 of word v hold q at k = 8v + 2s and bits 16+4s..16+4s+3 hold q at
 *   k = 8v + 2s + 1 (s = 0..3), k relative to the slab's k block.
 *   Scales: per stage 1024 bytes, [slab][row][2] fp16, groups 2kb and 2kb+1 of
 *   the slab's k block; each bf16 scale is converted to fp16 (exact for
 *   magnitudes in [2^-14, 65504], saturating above, fp16 subnormal below).
 * inexact_scales  optional (NULL: not counted): device uint32, incremented
 *   (atomically, on the stream) once per non-zero scale whose magnitude lies
 *   outside [2^-14, 2729] or that is not finite.  When it stays 0, every
 *   dequantised weight (q - 8) * scale the kernels form is exact in fp16.  The
 *   caller zeroes it first.
 * Errors: MOE_ERR_NULL, MOE_ERR_SHAPE (N or K not multiples as above),
 *   MOE_ERR_ALIGN, MOE_ERR_CUDA.
 */
int moe_int4_pack(const uint8_t *q, const uint16_t *scales, int E, int N, int K,
                  int is_w13, void *packed, void *packed_scales, uint32_t *inexact_scales,
                  moe_stream_t stream);

/*
 * moe_mxfp4_pack: canonical MXFP4 weights -> the same device layout (forward
 * with shape.weight_format = MOE_W_MXFP4).
 *
 * In:  q       uint8 [E][N][K/2], FP4 E2M1 codes in the nibble order of
 *              moe_int4_pack.
 *      scales  uint8 E8M0 [E][N][K/32] (2^(e - 127)); one per 32 consecutive k.
 *      is_w13  as for moe_int4_pack.
 * Out: packed (moe_int4_packed_bytes) and packed_scales
 *      (moe_int4_packed_scale_bytes), caller-allocated, 16-byte aligned.  Stages,
 *      slabs, rows and words are laid out as for moe_int4_pack, but inside word v
 *      of a row the bytes keep their canonical order: byte c holds the codes of
 *      k = 8v + 2c (low nibble) and 8v + 2c + 1 (high nibble).  Each scale is
 *      stored as the fp16 factor the kernels multiply by, the scale 2^(e - 127)
 *      itself, supported for e in [103, 140] (scales 2^-24 .. 2^13: an fp16
 *      power of two, and no weight beyond 65504); codes outside that range (and
 *      255, NaN) are clamped to its ends and counted.  The dequantised fp16
 *      weights are exact for e in [104, 140].
 *      bad_scales  optional (NULL: not counted): device uint32, incremented
 *              (atomically, on the stream) once per clamped scale; the caller
 *              zeroes it first.
 * Errors: as moe_int4_pack.
 */
int moe_mxfp4_pack(const uint8_t *q, const uint8_t *scales, int E, int N, int K, int is_w13,
                   void *packed, void *packed_scales, uint32_t *bad_scales,
                   moe_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Align: bucket routing pairs by expert and pad each bucket to block_m       */
/* ("The Result: Two Regimes": each token's top-8 experts are gathered into    */
/* per-expert groups for the grouped GEMM)                                     */
/* ------------------------------------------------------------------------- */

/* Capacity (entries) that sorted_ids needs: M*top_k + min(E, M*top_k)*(block_m-1).
 * expert_ids needs capacity/block_m entries. */
size_t moe_align_capacity(int M, int top_k, int E, int block_m);
/* Device scratch bytes moe_align needs (0 when M*top_k <= 4096). */
size_t moe_align_scratch_bytes(int M, int top_k, int E);

/*
 * moe_align: stable counting sort of the P = M*top_k routing pairs by expert.
 * In:  topk_ids int32 [M][top_k].
 * Out: sorted_ids int32: for each expert e = 0..E-1 in order, the flat pair
 *        indices t*top_k+j routed to e in ascending order, then pad entries equal
 *        to P up to the next multiple of block_m (experts with no pair take no
 *        space).  Entries past num_post_pad are not written.
 *      expert_ids int32: the expert of each block of block_m entries.
 *      num_post_pad int32 [1]: total entries written.
 *      Pairs whose id is outside [0, E) are dropped and reported in
 *      err_flags (uint32 [2] = flags, count; NULL: not reported): the call ORs
 *      MOE_DEVERR_BAD_EXPERT_ID into the flags and adds the number dropped to
 *      the count, so the caller zeroes both words first (a clean call leaves
 *      them as they were).
 * block_m: 1..256.  scratch: moe_align_scratch_bytes bytes (NULL if 0).
 * Errors: MOE_ERR_NULL, MOE_ERR_SHAPE, MOE_ERR_WORKSPACE, MOE_ERR_CUDA.
 */
int moe_align(const int32_t *topk_ids, int M, int top_k, int E, int block_m,
              int32_t *sorted_ids, int32_t *expert_ids, int32_t *num_post_pad,
              uint32_t *err_flags, void *scratch, size_t scratch_bytes,
              moe_stream_t stream);

/*
 * moe_align_noalloc: moe_align for callers that cannot allocate device memory.
 * (The pages have no counterpart: this entry point serves callers of this
 * library, such as a plugin that a host runtime hands only its input and
 * output buffers, or a latency-critical path where cudaMalloc/cudaFree may
 * block or synchronise the device.)
 * Same inputs, outputs and results as moe_align; the per-chunk scratch table
 * comes from a fixed 1 MiB device array inside the library instead of the
 * caller, held on every GPU that loads the library until the process exits.
 * Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 * Limit: moe_align_scratch_bytes(M, top_k, E) <= 1 MiB (E = 384: up to
 * 698,368 pairs; E = 1024: 262,144), else MOE_ERR_NOALLOC_LIMIT and nothing
 * is launched.
 * Routings of up to 4096 pairs need no table and touch neither the array nor
 * any set-up.  The first larger call on each device looks up the array's
 * device address on the current device (cudaGetSymbolAddress); make that
 * first call before any stream capture.  The address is cached per device and
 * does not survive cudaDeviceReset: after a reset, do not call this entry
 * point again in the same process.  Nothing in the array needs to start at zero (each call
 * writes every entry it reads), but all calls share it: calls whose kernels
 * overlap on the GPU (different streams, or host threads) race and give wrong
 * results; serialise them, e.g. on one stream.
 * Errors: those of moe_align (MOE_ERR_WORKSPACE excepted), MOE_ERR_NOALLOC_LIMIT,
 * MOE_ERR_UNSUPPORTED (device ordinal >= 64).
 */
int moe_align_noalloc(const int32_t *topk_ids, int M, int top_k, int E, int block_m,
                      int32_t *sorted_ids, int32_t *expert_ids, int32_t *num_post_pad,
                      uint32_t *err_flags, moe_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Forward                                                                    */
/* ------------------------------------------------------------------------- */

/* Workspace flag: also reserve room for the host-IO staging of
 * moe_int4_forward_host. */
#define MOE_WS_HOST_IO 0x1

/* Workspace bytes for a forward of M tokens (0 < M <= 1<<20). */
size_t moe_int4_workspace_bytes(int M, const moe_int4_shape *shape, int flags);

/* The routing block height the forward uses for M tokens (16..192). */
int moe_int4_block_m(int M, const moe_int4_shape *shape);

/* 1 if a forward of M tokens runs the fused decode kernel (gather, gate/up and
 * down GEMMs in one launch; see moe_int4_forward), 0 if it runs them as separate
 * kernels (or M or the shape is invalid). */
int moe_int4_fused(int M, const moe_int4_shape *shape);

/* 1 if a forward of M tokens runs the small-batch path (the expert MLP as
 * per-pair matrix-vector products; see moe_int4_forward), 0 otherwise. */
int moe_int4_gemv(int M, const moe_int4_shape *shape);

/* 1 if a forward of M tokens runs the separate plan with its down step as
 * per-block matrix-vector work (routing blocks of at most 16 rows; see
 * moe_int4_forward), 0 otherwise. */
int moe_int4_block_down(int M, const moe_int4_shape *shape);

/*
 * moe_int4_workspace_layout: byte offsets inside the workspace of a forward of
 * M tokens, for inspecting a finished call: offsets[0] error words (uint32 flags,
 * uint32 dropped count), [1] num_post_pad (int32), [2] sorted_ids (int32,
 * moe_align contract with block_m = moe_int4_block_m), [3] expert_ids (int32),
 * [4] the fp16 SwiGLU intermediate [row][inter] indexed by position in
 * sorted_ids (rows of pad entries are undefined), [5] the fp32 [M][hidden]
 * combine accumulator of a bf16-output forward (unused for fp32 output).
 * Returns MOE_OK or MOE_ERR_SHAPE / MOE_ERR_NULL.
 */
int moe_int4_workspace_layout(int M, const moe_int4_shape *shape, size_t *offsets);

/*
 * moe_int4_forward: out = the MoE expert MLP of x (see the top of this file).
 * In:  x             bf16 [M][hidden]
 *      w13_packed    moe_int4_pack(is_w13=1) output, w13_scales its scales
 *      w2_packed     moe_int4_pack(is_w13=0) output, w2_scales its scales
 *      topk_ids      int32 [M][top_k]
 *      topk_weights  fp32 [M][top_k], used as given
 * Out: out           [M][hidden] of shape->out_dtype (bf16 bits or fp32),
 *                    overwritten (tokens whose pairs were all dropped get 0).
 * workspace: >= moe_int4_workspace_bytes(M, shape, 0) bytes of device memory,
 *   16-byte aligned.  It holds the align buffers, the gathered fp16 x rows, the
 *   fp16 intermediate, fp32 accumulators and the error words; two calls in
 *   flight at once must not share it.  No initial contents are required except
 *   for the error words (its first 8 bytes), which accumulate over calls: clear
 *   them (moe_int4_clear_errors) once after allocating the workspace.
 * M == 0 returns MOE_OK without touching out.  Every pointer must be 16-byte
 * aligned.  The call launches only kernels (no host sync, no allocation).
 * Launch plan: where the pairs seldom share an expert (at most 64 pairs and at
 * most 1.2 pairs per expert that a uniform routing of M tokens is expected to
 * touch), or where all experts together fit in 64 MiB (at most 256 pairs), two
 * matrix-vector kernels, gate/up + SwiGLU and then down + combine, each routed
 * pair reading its token's row and its expert's packed weights directly (no
 * align; a shared expert is read once per pair).  Otherwise the align kernel,
 * then either a gather kernel and one kernel per GEMM, where at routing blocks
 * of at most 16 rows the down step streams each block's expert once and reduces
 * it against the block's rows as matrix-vector work; or, for routings of at
 * most 512 pairs whose blocks hold more than about 2.5 rows per expert (or with
 * MOE_FLAG_NO_GEMV), one persistent tensor-core kernel that gathers x, runs the
 * gate/up GEMM and then the down GEMM (its CTAs hand work to each other through
 * counters in the workspace, with bounded waits; it expects to get every SM
 * within about two seconds).  All plans form the same fp16 weights and intermediates and
 * accumulate in fp32; they differ only in summation order.  bf16 output adds a
 * conversion kernel.
 * Errors: MOE_ERR_NULL, MOE_ERR_SHAPE, MOE_ERR_ALIGN, MOE_ERR_WORKSPACE,
 *   MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA.
 */
int moe_int4_forward(const uint16_t *x, const void *w13_packed, const void *w13_scales,
                     const void *w2_packed, const void *w2_scales,
                     const int32_t *topk_ids, const float *topk_weights,
                     void *out, int M, const moe_int4_shape *shape,
                     void *workspace, size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Router ("The Throughput Lever", "The Result: Two Regimes": each token      */
/* activates top_k of E experts through top-k routing)                        */
/* ------------------------------------------------------------------------- */

/*
 * moe_route: per token, the top_k experts by router logit and their weights.
 * In:  router_logits fp32 [M][E] (finite).
 * Out: topk_ids int32 [M][top_k]: experts in descending logit order; equal
 *        logits are taken in ascending expert index (exact fp32 comparisons,
 *        so the ids are reproducible bit for bit).
 *      topk_weights fp32 [M][top_k]: the softmax over all E logits renormalised
 *        over the chosen top_k, i.e. the softmax over the chosen logits.
 * Sizes: 1 <= E <= 1024, 1 <= top_k <= min(E, 32), 0 <= M <= 1<<20.
 * Errors: MOE_ERR_SHAPE, MOE_ERR_NULL, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA.
 */
int moe_route(const float *router_logits, int M, int E, int top_k, int32_t *topk_ids,
              float *topk_weights, moe_stream_t stream);

/*
 * moe_int4_forward_routed: moe_int4_forward with the routing computed from
 * router logits: the router (as moe_route) runs in the same launch as the
 * align for routings up to 32 tokens, writes topk_ids and topk_weights (device
 * buffers [M][top_k] owned by the caller, also returned), and the layer then
 * runs exactly as moe_int4_forward on them.  router_logits: fp32 [M][E].
 * Workspace, layout, errors and output: as moe_int4_forward.
 */
int moe_int4_forward_routed(const uint16_t *x, const void *w13_packed, const void *w13_scales,
                            const void *w2_packed, const void *w2_scales,
                            const float *router_logits, int32_t *topk_ids, float *topk_weights,
                            void *out, int M, const moe_int4_shape *shape, void *workspace,
                            size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_int4_forward_host: the same layer with x, topk_ids, topk_weights and out
 * in HOST memory (pinned memory makes the copies asynchronous).  The inputs are
 * copied into the workspace's staging area, the forward runs on `stream`, the
 * output is copied back, and the call waits for the stream before returning.
 * Weights and workspace are device memory as for moe_int4_forward; the
 * workspace must be >= moe_int4_workspace_bytes(M, shape, MOE_WS_HOST_IO).
 */
int moe_int4_forward_host(const uint16_t *x_host, const void *w13_packed,
                          const void *w13_scales, const void *w2_packed,
                          const void *w2_scales, const int32_t *topk_ids_host,
                          const float *topk_weights_host, void *out_host, int M,
                          const moe_int4_shape *shape, void *workspace,
                          size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_int4_get_errors: read (synchronously on `stream`) the device error flags
 * (MOE_DEVERR_*) and the count of dropped routing pairs accumulated in the
 * workspace since the last moe_int4_clear_errors.  Every forward on the
 * workspace ORs its flags into the first word and adds its dropped pairs to
 * the second; nothing resets them but moe_int4_clear_errors, so a flag raised
 * by one call (a timeout, a bad id) is still there after later clean calls.
 * Either output may be NULL.
 */
int moe_int4_get_errors(const void *workspace, uint32_t *flags, uint32_t *count,
                        moe_stream_t stream);
/* moe_int4_clear_errors: zero the error words (stream-ordered). */
int moe_int4_clear_errors(void *workspace, moe_stream_t stream);

/* Human-readable text for a MOE_ERR_* code (static storage). */
const char *moe_int4_strerror(int code);

/*
 * Stage timing for measurement: while enabled (on != 0), every forward records
 * CUDA events around its align, gate/up GEMM, down GEMM and finalize launches on
 * its stream.  moe_int4_profile_read waits for the last forward's events and
 * writes the four stage durations in milliseconds to ms[0..3]; returns
 * MOE_ERR_CUDA if no profiled forward has run.  Not for use during stream
 * capture.
 */
int moe_int4_profile_enable(int on);
int moe_int4_profile_read(float *ms);

/* Number of kernel launches the last moe_int4_forward made on this thread. */
int moe_int4_last_launch_count(void);

/*
 * Expert-parallel row movement ("From PCIe to NVLink", section "Part I: Laying
 * the Foundation": the experts sharded over the GPUs).  Around the all-to-all
 * exchanges of an expert-parallel layer, a rank gathers the x rows of the pairs
 * it sends, and adds the expert outputs that come back into its tokens' rows.
 * Both are stream-ordered, allocate nothing and do not synchronise.
 *
 * moe_ep_gather: dst[i][:] = src[rows[i]][:] for i < n, rows of H 2-byte
 *   elements (bf16 bits; H a multiple of 8).  src is [src_rows][H]; a row index
 *   outside [0, src_rows) zeroes dst[i] and sets bit 0 of *bad (device uint32;
 *   may be NULL).  src and dst 16-byte aligned.
 * moe_ep_combine: out[rows[i]][:] += src[i][:] for i < n, fp32 rows of H
 *   elements (H a multiple of 4); out is [out_rows][H], rows may repeat (the adds
 *   are atomic, so their order, and the last bits of a sum, may vary).  A row
 *   index outside [0, out_rows) is dropped and sets bit 0 of *bad.  src and out
 *   16-byte aligned.
 * Errors: MOE_ERR_NULL, MOE_ERR_SHAPE, MOE_ERR_ALIGN, MOE_ERR_CUDA.  n = 0 is a
 * no-op.
 */
int moe_ep_gather(const uint16_t *src, int src_rows, const int32_t *rows, int n, int H,
                  uint16_t *dst, uint32_t *bad, moe_stream_t stream);
int moe_ep_combine(const float *src, const int32_t *rows, int n, int H, float *out,
                   int out_rows, uint32_t *bad, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_INT4_H */
