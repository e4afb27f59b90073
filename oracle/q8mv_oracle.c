/*
 * Q8_0 decode matvec: CPU oracle in fp64.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline / reference legs load this file's
 * library.  The GPU library never includes, links or calls it, and this file
 * includes nothing from the GPU library.
 *
 * What it computes (Phobos docs, "Q8_0 matvec" example page):
 *   - "The tensors": A is [1, K] f32 (one activation row), W is [K, N] signed
 *     bytes (one column per output), S is [KB, N] f32 where row b of S scales
 *     rows 32*b up to 32*b + 32 of W, and C is [1, N] f32.  The value a weight
 *     stands for is W[k, n] * S[k / 32, n], so
 *         C[0, n] = sum over k of A[0, k] * W[k, n] * S[k / 32, n].
 *   - "Factoring out the scale": inside a block every weight of a column shares
 *     one scale, so the block sum is taken on the raw bytes and scaled once:
 *         sum_{k in b} A[k] W[k,n] S[b,n] = S[b,n] * sum_{k in b} A[k] W[k,n].
 *   - "Bounds": K need not be a multiple of 32; the loop over K is whole blocks
 *     plus one masked remainder, so the last block may hold fewer than 32 rows
 *     and KB = ceil(K / 32).  Rows at or past K are never read.
 *   - "Line by line": acc starts at 0 and C is assigned acc after the last
 *     block, so C is overwritten (not accumulated into) and K = 0 gives C = 0.
 *
 * Readings where the pages are silent:
 *   - Layout: every tensor is contiguous row-major, W[k, n] at k*N + n and
 *     S[b, n] at b*N + n (the slices W[k :+ BLK, pn*TILE_N :+ TILE_N] of the
 *     kernel listing index rows by k and columns by n).
 *   - Precision: the pages fix f32 tiles for the GPU kernel but nothing for a
 *     checker, so every product and sum here is taken in fp64.  Each product
 *     A*W is exact in fp64 (24-bit by 8-bit significands); A*W*S rounds once.
 *   - Signed bytes cover -128 .. 127; -128 is a legal weight.
 *
 * Both forms are pinned by CPU tests against exact rational brute force,
 * closed forms, one-hot special cases, linearity and exact-integer inputs.
 */
#include <stdint.h>
#include <stdlib.h>
#include <math.h>

#define Q8MV_ORACLE_BLK 32

static int64_t oracle_num_blocks(int64_t K) {
    return (K + Q8MV_ORACLE_BLK - 1) / Q8MV_ORACLE_BLK;
}

/* Return codes: 0 ok, -1 bad argument, -2 out of host memory. */

/*
 * Per-weight form ("The tensors"): C[n] = sum_k A[k] * W[k,n] * S[k/32, n],
 * each term formed and added in fp64, k ascending.
 */
int q8mv_oracle_unfactored(int64_t K, int64_t N, const float *A, const int8_t *W,
                           const float *S, double *C) {
    if (K < 0 || N < 0) return -1;
    if (N > 0 && C == NULL) return -1;
    if (K > 0 && N > 0 && (A == NULL || W == NULL || S == NULL)) return -1;
    for (int64_t n = 0; n < N; ++n) C[n] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double a = (double)A[k];
        const int8_t *w_row = W + k * N;
        const float *s_row = S + (k / Q8MV_ORACLE_BLK) * N;
        for (int64_t n = 0; n < N; ++n)
            C[n] += a * (double)w_row[n] * (double)s_row[n];
    }
    return 0;
}

/*
 * Block-factored form ("Factoring out the scale", "Line by line"): for each
 * block b, part[n] = sum_{k in b, k < K} A[k] * W[k,n] on the raw bytes, then
 * acc[n] += part[n] * S[b,n], one multiply per block and column.
 *
 * bound (nullable) receives sum_k |A[k] * W[k,n] * S[k/32,n]|, the magnitude
 * against which a rounded result's error is judged.
 */
int q8mv_oracle_factored(int64_t K, int64_t N, const float *A, const int8_t *W,
                         const float *S, double *C, double *bound) {
    if (K < 0 || N < 0) return -1;
    if (N > 0 && C == NULL) return -1;
    if (K > 0 && N > 0 && (A == NULL || W == NULL || S == NULL)) return -1;
    for (int64_t n = 0; n < N; ++n) {
        C[n] = 0.0;
        if (bound) bound[n] = 0.0;
    }
    if (K == 0 || N == 0) return 0;

    double *part = (double *)malloc((size_t)N * sizeof(double));
    double *mag = (double *)malloc((size_t)N * sizeof(double));
    if (part == NULL || mag == NULL) {
        free(part);
        free(mag);
        return -2;
    }
    const int64_t KB = oracle_num_blocks(K);
    for (int64_t b = 0; b < KB; ++b) {
        const int64_t k_begin = b * Q8MV_ORACLE_BLK;
        int64_t k_end = k_begin + Q8MV_ORACLE_BLK;
        if (k_end > K) k_end = K; /* masked remainder of the last block */
        for (int64_t n = 0; n < N; ++n) {
            part[n] = 0.0;
            mag[n] = 0.0;
        }
        /* the block's dot product on the unscaled bytes */
        for (int64_t k = k_begin; k < k_end; ++k) {
            const double a = (double)A[k];
            const int8_t *w_row = W + k * N;
            for (int64_t n = 0; n < N; ++n) {
                const double aw = a * (double)w_row[n];
                part[n] += aw;
                mag[n] += fabs(aw);
            }
        }
        /* the block's scale, applied once per column */
        const float *s_row = S + b * N;
        for (int64_t n = 0; n < N; ++n) {
            const double s = (double)s_row[n];
            C[n] += part[n] * s;
            if (bound) bound[n] += mag[n] * fabs(s);
        }
    }
    free(part);
    free(mag);
    return 0;
}

/*
 * The unscaled block sums themselves, part[b, n] = sum_{k in b, k < K}
 * A[k] * W[k, n], as a [KB, N] fp64 array.  With integer-valued A these are
 * integers, which is what a bit-exact check of a kernel's block sums needs.
 */
int q8mv_oracle_block_sums(int64_t K, int64_t N, const float *A, const int8_t *W,
                           double *part) {
    if (K < 0 || N < 0) return -1;
    const int64_t KB = oracle_num_blocks(K);
    if (KB > 0 && N > 0 && (A == NULL || W == NULL || part == NULL)) return -1;
    for (int64_t b = 0; b < KB; ++b) {
        double *p_row = part + b * N;
        for (int64_t n = 0; n < N; ++n) p_row[n] = 0.0;
        const int64_t k_begin = b * Q8MV_ORACLE_BLK;
        int64_t k_end = k_begin + Q8MV_ORACLE_BLK;
        if (k_end > K) k_end = K;
        for (int64_t k = k_begin; k < k_end; ++k) {
            const double a = (double)A[k];
            const int8_t *w_row = W + k * N;
            for (int64_t n = 0; n < N; ++n) p_row[n] += a * (double)w_row[n];
        }
    }
    return 0;
}

/*
 * Several activation rows against the same weights: A is [M, K] and C, bound
 * are [M, N], all row-major.  Row m of C is the block-factored matvec above of
 * row m of A; rows never mix.  The Q8_0 matvec example page ("The tensors")
 * defines one activation row; a decode step of M sequences applies it to each.
 */
int q8mv_oracle_batched(int64_t M, int64_t K, int64_t N, const float *A, const int8_t *W,
                        const float *S, double *C, double *bound) {
    if (M < 0 || K < 0 || N < 0) return -1;
    if (M > 0 && N > 0 && C == NULL) return -1;
    if (M > 0 && K > 0 && A == NULL) return -1;
    for (int64_t m = 0; m < M; ++m) {
        const int rc = q8mv_oracle_factored(K, N, A + m * K, W, S, C + m * N, bound ? bound + m * N : NULL);
        if (rc != 0) return rc;
    }
    return 0;
}

/*
 * Fused epilogue ("dot and tensor cores" page, "The fused epilogue"): an
 * elementwise statement right after the product is applied to each output as
 * it is written, instead of storing the product and sweeping it again.  The
 * page's two forms are a scale of the product (s = s * scale) and an update
 * of the target that reads its previous value (acc = acc * corr + dot(p, v)).
 * The statement here covers both, plus the bias, activation and residual of a
 * decode layer, in this order, for output (m, n) of an [M, N] result:
 *
 *     y = alpha * x[m,n] + beta * c_old[m,n] + bias[n]
 *     y = act(y)                       (0 none, 1 relu, 2 silu, 3 gelu tanh)
 *     out[m,n] = y + residual[m,n]
 *
 * with x the fp64 product, c_old (read only when beta != 0), bias and residual
 * optional f32 arrays.  silu(y) = y / (1 + exp(-y)); the tanh form of gelu is
 * 0.5 y (1 + tanh(sqrt(2/pi) (y + 0.044715 y^3))) (Hendrycks and Gimpel).
 * mag (nullable) receives |alpha x| + |beta c_old| + |bias| + |act(y)| +
 * |residual|, the magnitude a rounded result's error is judged against.
 */
int q8mv_oracle_epilogue(int64_t M, int64_t N, const double *x, const float *c_old, const float *bias,
                         const float *residual, double alpha, double beta, int act, double *out,
                         double *mag) {
    if (M < 0 || N < 0 || act < 0 || act > 3) return -1;
    if (M > 0 && N > 0 && (x == NULL || out == NULL)) return -1;
    if (M > 0 && N > 0 && beta != 0.0 && c_old == NULL) return -1;
    const double k_gelu = 0.79788456080286535588; /* sqrt(2 / pi) */
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            const int64_t i = m * N + n;
            const double ax = alpha * x[i];
            const double bc = beta != 0.0 ? beta * (double)c_old[i] : 0.0;
            const double b = bias ? (double)bias[n] : 0.0;
            double y = ax + bc + b;
            if (act == 1) {
                y = y > 0.0 ? y : 0.0;
            } else if (act == 2) {
                y = y / (1.0 + exp(-y));
            } else if (act == 3) {
                y = 0.5 * y * (1.0 + tanh(k_gelu * (y + 0.044715 * y * y * y)));
            }
            const double r = residual ? (double)residual[i] : 0.0;
            out[i] = y + r;
            if (mag) mag[i] = fabs(ax) + fabs(bc) + fabs(b) + fabs(y) + fabs(r);
        }
    }
    return 0;
}

/*
 * Weights stored one output row per row ("dot and tensor cores" page: dot_t
 * contracts the last axis of both operands, the layout of a linear layer's
 * weights).  Wt is [N, K] with Wt[n, k] at n*K + k, and St is [N, KB] with
 * St[n, b] at n*KB + b: row n holds output n's bytes and its block scales.
 * The product is the Q8_0 matvec of the "Q8_0 matvec" page with W = Wt^T and
 * S = St^T:
 *     C[n] = sum_b St[n, b] * ( sum_{k in b, k < K} A[k] * Wt[n, k] )
 * written directly over the transposed indexing, blocks in order, fp64.
 * bound (nullable) receives sum_k |A[k] Wt[n,k] St[n, k/32]|.
 */
int q8mv_oracle_transposed(int64_t K, int64_t N, const float *A, const int8_t *Wt, const float *St,
                           double *C, double *bound) {
    if (K < 0 || N < 0) return -1;
    if (N > 0 && C == NULL) return -1;
    if (K > 0 && N > 0 && (A == NULL || Wt == NULL || St == NULL)) return -1;
    const int64_t KB = oracle_num_blocks(K);
    for (int64_t n = 0; n < N; ++n) {
        const int8_t *w_row = Wt + n * K;
        const float *s_row = St + n * KB;
        double acc = 0.0, mag = 0.0;
        for (int64_t b = 0; b < KB; ++b) {
            const int64_t k_begin = b * Q8MV_ORACLE_BLK;
            int64_t k_end = k_begin + Q8MV_ORACLE_BLK;
            if (k_end > K) k_end = K;
            double part = 0.0, part_mag = 0.0;
            for (int64_t k = k_begin; k < k_end; ++k) {
                const double aw = (double)A[k] * (double)w_row[k];
                part += aw;
                part_mag += fabs(aw);
            }
            const double s = (double)s_row[b];
            acc += part * s;
            mag += part_mag * fabs(s);
        }
        C[n] = acc;
        if (bound) bound[n] = mag;
    }
    return 0;
}

/*
 * Int8 activations ("dot and tensor cores" page, "Hardware paths": an i8
 * dot_t accumulates in i32, and a single row takes dp4a).  The pages do not
 * say how an f32 activation row becomes i8; the reading used here quantizes
 * each 32-element block b of A on its own, in f32 arithmetic:
 *     amax_b = max_{k in b} |A[k]|
 *     d_b    = amax_b / 127                    (f32 division)
 *     q[k]   = rint(A[k] * (127 / amax_b))     (f32 division once, f32 product,
 *                                               round half to even, clamped to
 *                                               -127 .. 127; q = 0 if amax_b = 0)
 * so that A[k] is approximately q[k] * d_b.  Every operation is a single IEEE
 * f32 operation (no contraction), so any IEEE implementation gets the same q.
 */
int q8mv_oracle_quantize(int64_t K, const float *A, int8_t *q, float *d) {
    if (K < 0) return -1;
    if (K > 0 && (A == NULL || q == NULL || d == NULL)) return -1;
    const int64_t KB = oracle_num_blocks(K);
    for (int64_t b = 0; b < KB; ++b) {
        const int64_t k_begin = b * Q8MV_ORACLE_BLK;
        int64_t k_end = k_begin + Q8MV_ORACLE_BLK;
        if (k_end > K) k_end = K;
        float amax = 0.0f;
        for (int64_t k = k_begin; k < k_end; ++k) {
            const float a = fabsf(A[k]);
            if (a > amax) amax = a;
        }
        const float db = amax / 127.0f;
        const float id = amax > 0.0f ? 127.0f / amax : 0.0f;
        d[b] = db;
        for (int64_t k = k_begin; k < k_end; ++k) {
            const float x = A[k] * id;
            float r = rintf(x);
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            q[k] = (int8_t)r;
        }
    }
    return 0;
}

/*
 * The Q8_0 product with int8 activations, weights stored one output row per
 * row (Wt [N, K], St [N, KB]): each block's dot product of codes is an exact
 * integer, scaled once by the activation block's d_b and the weight block's
 * scale:
 *     C[n] = sum_b (d_b * St[n, b]) * ( sum_{k in b} q[k] * Wt[n, k] )
 * in fp64.  bound (nullable) receives sum_b |d_b St[n, b]| * sum_k |q[k] Wt[n, k]|.
 */
int q8mv_oracle_i8(int64_t K, int64_t N, const int8_t *q, const float *d, const int8_t *Wt, const float *St,
                   double *C, double *bound) {
    if (K < 0 || N < 0) return -1;
    if (N > 0 && C == NULL) return -1;
    if (K > 0 && N > 0 && (q == NULL || d == NULL || Wt == NULL || St == NULL)) return -1;
    const int64_t KB = oracle_num_blocks(K);
    for (int64_t n = 0; n < N; ++n) {
        double acc = 0.0, mag = 0.0;
        for (int64_t b = 0; b < KB; ++b) {
            const int64_t k_begin = b * Q8MV_ORACLE_BLK;
            int64_t k_end = k_begin + Q8MV_ORACLE_BLK;
            if (k_end > K) k_end = K;
            int64_t isum = 0, iabs = 0;
            for (int64_t k = k_begin; k < k_end; ++k) {
                const int64_t p = (int64_t)q[k] * (int64_t)Wt[n * K + k];
                isum += p;
                iabs += p < 0 ? -p : p;
            }
            const double scale = (double)d[b] * (double)St[n * KB + b];
            acc += scale * (double)isum;
            mag += fabs(scale) * (double)iabs;
        }
        C[n] = acc;
        if (bound) bound[n] = mag;
    }
    return 0;
}
