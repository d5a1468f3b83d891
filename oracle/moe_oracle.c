/*
 * Oracle for the weight-only INT4 MoE expert MLP.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: it exists so that tests, the smoke check and the CPU-baseline leg of
 * the benchmark can check the CUDA kernels against a plain, slow, obviously
 * correct fp64 computation.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes, and where the pages say so:
 *
 *  - Weights are INT4 with one scale per group of 32 along the reduction axis
 *    ("The Throughput Lever", section "Building the Benchmark": INT4 with group
 *    size 32).  A weight is value = (q - 8) * scale, q in {0..15}, scale bf16
 *    (the workload definition of the tiny configuration).  The product is formed
 *    exactly in fp64.
 *  - The layer is a grouped MoE GEMM over a routed token batch ("The Throughput
 *    Lever", section "Phase 3: The INT4 Marlin MoE Throughput Lever", and the
 *    two-regime discussion in "The Result: Two Regimes"): for every token t and
 *    routing slot j with expert e = ids[t, j]
 *        g_i = sum_h W13[e, i, h]     x[t, h]          (gate rows 0..I-1)
 *        u_i = sum_h W13[e, I + i, h] x[t, h]          (up rows I..2I-1)
 *        a_i = g_i / (1 + exp(-g_i)) * u_i             (SwiGLU)
 *        y_h = sum_i W2[e, h, i] a_i
 *        out[t, h] += w[t, j] * y_h                     (top-k weighted combine)
 *  - Routing pairs whose expert id is outside [0, E) are dropped and counted.
 *  - The MXFP4 variant ("From 1,060 to 4,016 tok/s on one B300", whose model
 *    has MXFP4 experts, and its section "Finding 2: the MoE autotuner only saw
 *    decode shapes") changes only the weight: value = e2m1(q) * 2^(e - 127),
 *    the OCP Microscaling v1.0 FP4 element (sign, 2-bit exponent with bias 1, one
 *    mantissa bit; exponent 0 subnormal) with one E8M0 power-of-two scale per 32
 *    along the reduction axis.  The pages name the format without defining it;
 *    this is the published definition.  Exact in fp64.
 *
 * Canonical storage read here (not a device layout):
 *  - q bytes [E][N][K/2]: logical element k of a row sits in byte k/2, in the
 *    low nibble when k is even and in the high nibble when k is odd.
 *  - scales: bf16 bit patterns [E][N][K/32].
 *  - x: bf16 bit patterns [M][H].  topk_weights: fp32 [M][k].
 *
 * The align step (bucketing routing pairs by expert, padding each bucket to a
 * multiple of block_m) is written out as the definition: for each expert in
 * ascending order, the flat pair indices t*k+j routed to it in ascending order,
 * then pad entries holding the value P = M*k up to the next multiple of block_m.
 * One expert id is written for every block of block_m entries.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_double(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Canonical nibble k of a row of packed bytes. */
int oracle_nibble(const uint8_t *row, int64_t k) {
    uint8_t b = row[k / 2];
    return (k % 2 == 0) ? (b & 0x0F) : (b >> 4);
}

/* Weight formats. */
enum { ORACLE_INT4 = 0, ORACLE_MXFP4 = 1 };

/* FP4 E2M1 element: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa;
 * exponent 0 is subnormal (0 or 0.5). */
double oracle_e2m1(int code) {
    int sign = (code >> 3) & 1, ex = (code >> 1) & 3, man = code & 1;
    double mag = (ex == 0) ? 0.5 * man : ldexp(1.0 + 0.5 * man, ex - 1);
    return sign ? -mag : mag;
}

/* E8M0 scale: 2^(bits - 127); the code 255 is NaN. */
double oracle_e8m0(uint8_t bits) {
    return bits == 255 ? NAN : ldexp(1.0, (int)bits - 127);
}

/* Dequantised weight W[e, n, k] of a matrix of N rows and K columns per expert,
 * exact in fp64.  INT4: (q - 8) * s[e, n, k / 32] with s bf16 (uint16 bit
 * patterns).  MXFP4: e2m1(q) * e8m0(s[e, n, k / 32]) with s one byte. */
double oracle_weight_fmt(int fmt, const uint8_t *q, const void *s, int64_t N, int64_t K,
                         int64_t e, int64_t n, int64_t k) {
    const uint8_t *row = q + (e * N + n) * (K / 2);
    int nib = oracle_nibble(row, k);
    int64_t g = (e * N + n) * (K / 32) + k / 32;
    if (fmt == ORACLE_MXFP4) return oracle_e2m1(nib) * oracle_e8m0(((const uint8_t *)s)[g]);
    return (double)(nib - 8) * oracle_bf16_to_double(((const uint16_t *)s)[g]);
}

double oracle_weight(const uint8_t *q, const uint16_t *s, int64_t N, int64_t K,
                     int64_t e, int64_t n, int64_t k) {
    return oracle_weight_fmt(ORACLE_INT4, q, s, N, K, e, n, k);
}

/* SwiGLU intermediate a[0..I) of one (token, expert) pair. */
void oracle_pair_intermediate_fmt(int fmt, const uint16_t *x_row, const uint8_t *q13,
                                  const void *s13, int64_t e, int64_t H, int64_t I,
                                  double *a) {
    for (int64_t i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            double xv = oracle_bf16_to_double(x_row[h]);
            g += oracle_weight_fmt(fmt, q13, s13, 2 * I, H, e, i, h) * xv;
            u += oracle_weight_fmt(fmt, q13, s13, 2 * I, H, e, I + i, h) * xv;
        }
        a[i] = g / (1.0 + exp(-g)) * u;
    }
}

void oracle_pair_intermediate(const uint16_t *x_row, const uint8_t *q13,
                              const uint16_t *s13, int64_t e, int64_t H,
                              int64_t I, double *a) {
    oracle_pair_intermediate_fmt(ORACLE_INT4, x_row, q13, s13, e, H, I, a);
}

/* Expert output y[0..H) = W2[e] a for one pair. */
void oracle_pair_down_fmt(int fmt, const double *a, const uint8_t *q2, const void *s2,
                          int64_t e, int64_t H, int64_t I, double *y) {
    for (int64_t h = 0; h < H; ++h) {
        double acc = 0.0;
        for (int64_t i = 0; i < I; ++i)
            acc += oracle_weight_fmt(fmt, q2, s2, H, I, e, h, i) * a[i];
        y[h] = acc;
    }
}

void oracle_pair_down(const double *a, const uint8_t *q2, const uint16_t *s2,
                      int64_t e, int64_t H, int64_t I, double *y) {
    oracle_pair_down_fmt(ORACLE_INT4, a, q2, s2, e, H, I, y);
}

/*
 * Full layer output for a list of tokens: out[r, h] for token tokens[r],
 * r in [0, n_tokens).  scratch must hold I + H doubles.  Returns the number of
 * routing pairs of those tokens that were dropped (expert id outside [0, E)).
 */
int64_t oracle_moe_forward_tokens_fmt(int fmt, const uint16_t *x, const uint8_t *q13,
                                      const void *s13, const uint8_t *q2, const void *s2,
                                      const int32_t *topk_ids, const float *topk_weights,
                                      int64_t M, int64_t E, int64_t top_k, int64_t H,
                                      int64_t I, const int64_t *tokens, int64_t n_tokens,
                                      double *scratch, double *out) {
    int64_t dropped = 0;
    double *a = scratch;
    double *y = scratch + I;
    for (int64_t r = 0; r < n_tokens; ++r) {
        int64_t t = tokens[r];
        double *o = out + r * H;
        for (int64_t h = 0; h < H; ++h) o[h] = 0.0;
        if (t < 0 || t >= M) continue;
        for (int64_t j = 0; j < top_k; ++j) {
            int64_t e = topk_ids[t * top_k + j];
            if (e < 0 || e >= E) {
                ++dropped;
                continue;
            }
            double w = (double)topk_weights[t * top_k + j];
            oracle_pair_intermediate_fmt(fmt, x + t * H, q13, s13, e, H, I, a);
            oracle_pair_down_fmt(fmt, a, q2, s2, e, H, I, y);
            for (int64_t h = 0; h < H; ++h) o[h] += w * y[h];
        }
    }
    return dropped;
}

int64_t oracle_moe_forward_tokens(const uint16_t *x, const uint8_t *q13,
                                  const uint16_t *s13, const uint8_t *q2,
                                  const uint16_t *s2, const int32_t *topk_ids,
                                  const float *topk_weights, int64_t M, int64_t E,
                                  int64_t top_k, int64_t H, int64_t I,
                                  const int64_t *tokens, int64_t n_tokens,
                                  double *scratch, double *out) {
    return oracle_moe_forward_tokens_fmt(ORACLE_INT4, x, q13, s13, q2, s2, topk_ids,
                                         topk_weights, M, E, top_k, H, I, tokens, n_tokens,
                                         scratch, out);
}

/*
 * Intermediate a for a list of routing pairs (flat index t*k+j): out[r, i].
 * Pairs with an out-of-range expert give a row of zeros.
 */
void oracle_moe_intermediate_pairs_fmt(int fmt, const uint16_t *x, const uint8_t *q13,
                                       const void *s13, const int32_t *topk_ids, int64_t M,
                                       int64_t E, int64_t top_k, int64_t H, int64_t I,
                                       const int64_t *pairs, int64_t n_pairs, double *out) {
    for (int64_t r = 0; r < n_pairs; ++r) {
        int64_t p = pairs[r];
        double *o = out + r * I;
        int64_t e = (p >= 0 && p < M * top_k) ? topk_ids[p] : -1;
        if (e < 0 || e >= E) {
            for (int64_t i = 0; i < I; ++i) o[i] = 0.0;
            continue;
        }
        oracle_pair_intermediate_fmt(fmt, x + (p / top_k) * H, q13, s13, e, H, I, o);
    }
}

void oracle_moe_intermediate_pairs(const uint16_t *x, const uint8_t *q13,
                                   const uint16_t *s13, const int32_t *topk_ids,
                                   int64_t M, int64_t E, int64_t top_k, int64_t H,
                                   int64_t I, const int64_t *pairs, int64_t n_pairs,
                                   double *out) {
    oracle_moe_intermediate_pairs_fmt(ORACLE_INT4, x, q13, s13, topk_ids, M, E, top_k, H, I,
                                      pairs, n_pairs, out);
}

/*
 * Align: the bucketed, padded index buffers.
 * Returns num_post_pad, or -1 if a capacity is too small.  *n_dropped receives
 * the number of pairs whose expert id is outside [0, E).
 */
int64_t oracle_align(const int32_t *topk_ids, int64_t M, int64_t top_k, int64_t E,
                     int64_t block_m, int32_t *sorted_ids, int64_t sorted_cap,
                     int32_t *expert_ids, int64_t blocks_cap, int64_t *n_dropped) {
    int64_t P = M * top_k;
    int64_t pos = 0;
    int64_t dropped = 0;
    for (int64_t i = 0; i < P; ++i)
        if (topk_ids[i] < 0 || topk_ids[i] >= E) ++dropped;
    for (int64_t e = 0; e < E; ++e) {
        int64_t start = pos;
        for (int64_t i = 0; i < P; ++i) {
            if (topk_ids[i] == e) {
                if (pos >= sorted_cap) return -1;
                sorted_ids[pos++] = (int32_t)i;
            }
        }
        int64_t count = pos - start;
        int64_t padded = ((count + block_m - 1) / block_m) * block_m;
        while (pos < start + padded) {
            if (pos >= sorted_cap) return -1;
            sorted_ids[pos++] = (int32_t)P;
        }
        for (int64_t b = start / block_m; b < (start + padded) / block_m; ++b) {
            if (b >= blocks_cap) return -1;
            expert_ids[b] = (int32_t)e;
        }
    }
    *n_dropped = dropped;
    return pos;
}

/*
 * Router: for each token, the top_k experts by router logit (larger first;
 * equal logits: the lower expert index first) and their renormalised softmax
 * weights.  A softmax over all E experts renormalised over the k selected ones
 * equals the softmax over the k selected logits alone (the common denominator
 * cancels), so the weights are computed that way, in fp64 from the fp32
 * logits.  Logits must be finite.
 * Source: "The Throughput Lever", section "The Result: Two Regimes" (each
 * token activates 8 of 384 experts through top-8 routing); the softmax /
 * top-k / renormalise recipe is that of the routed workloads.
 */
void oracle_route(const float *logits, int64_t M, int64_t E, int64_t top_k, int32_t *ids,
                  double *weights) {
    for (int64_t t = 0; t < M; ++t) {
        const float *l = logits + t * E;
        int32_t *id = ids + t * top_k;
        double *w = weights + t * top_k;
        for (int64_t j = 0; j < top_k; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                int taken = 0;
                for (int64_t i = 0; i < j; ++i)
                    if (id[i] == e) taken = 1;
                if (taken) continue;
                if (best < 0 || l[e] > l[best]) best = e;  /* strict: ties keep the lower index */
            }
            id[j] = (int32_t)best;
        }
        const double mx = (double)l[id[0]];
        double sum = 0.0;
        for (int64_t j = 0; j < top_k; ++j) {
            w[j] = exp((double)l[id[j]] - mx);
            sum += w[j];
        }
        for (int64_t j = 0; j < top_k; ++j) w[j] /= sum;
    }
}

