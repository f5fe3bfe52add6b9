/*
 * CPU oracle for the fused attention + post-attention Ulysses re-shard.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * definition that the CUDA path is checked against.  It shares no code with the
 * CUDA path; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark may build, load or call it.
 *
 * What it computes (X-Stage paper, abstract: "tile-granular fusion of the
 * post-attention All-to-All with FlashAttention"; gist.science technical
 * summary, "Key Contributions" item 3, FlashAttention-A2A piggybacking):
 *
 *   1. Exact bidirectional softmax attention, fp64, one query row at a time:
 *        x_j   = scale * sum_d Q[b,i,h,d] * K[b,j,h,d]        (j < S)
 *        m     = max_j x_j
 *        w_j   = exp(x_j - m)
 *        l     = sum_j w_j
 *        O[b,i,h,d] = (sum_j w_j * V[b,j,h,d]) / l
 *      FlashAttention computes exactly this (up to rounding order), so the
 *      oracle is the definition itself: no tiling, no online rescaling.
 *
 *   2. The Ulysses sequence re-shard, done explicitly in its two steps.
 *      Virtual rank r holds heads [r*H/P, (r+1)*H/P) for the full sequence
 *      (the head shard a Ulysses rank owns after the pre-attention
 *      All-to-All):  L_r[b,s,j,d] = O[b,s,r*H/P + j,d].
 *      The post-attention All-to-All sends, from every rank r to every rank p,
 *      the rows of p's contiguous sequence block:
 *        out_p[b,s',r*H/P + j,d] = L_r[b, p*S/P + s', j, d],   s' < S/P.
 *
 *   3. Causal variant (not on the pages, which treat bidirectional DiT
 *      attention; it is the masked self-attention of autoregressive models):
 *      query row i attends to keys j <= i only, i.e. definition 1 with every
 *      sum and the max running over j = 0 .. i.  Row i of the causal result is
 *      therefore row i of plain attention over the first i + 1 keys and values,
 *      which is how it is computed below (the same row routine, n_keys = i + 1).
 *
 * Inputs are bf16 bit patterns (uint16) in [B,S,H,D] layout, D fastest; they
 * are widened to double exactly.  Outputs are double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static size_t idx4(int64_t b, int64_t s, int64_t h, int64_t d, int64_t S, int64_t H, int64_t D) {
    return (size_t)(((b * S + s) * H + h) * D + d);
}

/* Widen one (b, h) slice of a [B,S,H,D] bf16 tensor to a dense [S][D] double matrix. */
static void widen_head(const uint16_t* t, double* dst, int64_t b, int64_t h,
                       int64_t S, int64_t H, int64_t D) {
    for (int64_t s = 0; s < S; ++s)
        for (int64_t d = 0; d < D; ++d)
            dst[s * D + d] = bf16_to_double(t[idx4(b, s, h, d, S, H, D)]);
}

/*
 * One query row of exact softmax attention over keys 0 .. S-1.
 *   qrow [D], kd/vd [S][D] (double), x: scratch [S] (receives the normalised
 *   weights w_j / l on return), orow [D] output.
 */
static void attention_row(const double* qrow, const double* kd, const double* vd,
                          int64_t S, int64_t D, double scale, double* x, double* orow) {
    double m = -INFINITY;
    for (int64_t j = 0; j < S; ++j) {
        const double* kj = kd + j * D;
        double dot = 0.0;
#pragma omp simd reduction(+ : dot)
        for (int64_t d = 0; d < D; ++d) dot += qrow[d] * kj[d];
        x[j] = scale * dot;
        if (x[j] > m) m = x[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < S; ++j) {
        x[j] = exp(x[j] - m);
        l += x[j];
    }
    for (int64_t d = 0; d < D; ++d) orow[d] = 0.0;
    for (int64_t j = 0; j < S; ++j) {
        const double wj = x[j];
        const double* vj = vd + j * D;
#pragma omp simd
        for (int64_t d = 0; d < D; ++d) orow[d] += wj * vj[d];
    }
    for (int64_t d = 0; d < D; ++d) orow[d] /= l;
    for (int64_t j = 0; j < S; ++j) x[j] /= l;
}

static int set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Number of threads the OpenMP runtime will use for the next parallel region. */
int oracle_max_threads(int nthreads) { return set_threads(nthreads); }

/* Keys that query row i attends to: all S, or (causal) keys 0 .. i. */
static int64_t keys_of_row(int64_t i, int64_t S, int causal) { return causal ? i + 1 : S; }

static int attention_rows_impl(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               int64_t B, int64_t S, int64_t H, int64_t D, double scale,
                               const int64_t* rows_b, const int64_t* rows_s, int64_t n_rows,
                               double* o_rows, int nthreads, int causal) {
    if (B < 1 || S < 1 || H < 1 || D < 1 || n_rows < 0) return -1;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows_b[r] < 0 || rows_b[r] >= B || rows_s[r] < 0 || rows_s[r] >= S) return -1;
    set_threads(nthreads);
    double* kd = (double*)malloc(sizeof(double) * (size_t)(S * D));
    double* vd = (double*)malloc(sizeof(double) * (size_t)(S * D));
    if (!kd || !vd) { free(kd); free(vd); return -1; }
    int status = 0;
    for (int64_t b = 0; b < B; ++b) {
        /* skip batch entries with no requested row */
        int64_t any = 0;
        for (int64_t r = 0; r < n_rows; ++r) any |= (rows_b[r] == b);
        if (!any) continue;
        for (int64_t h = 0; h < H; ++h) {
            widen_head(k, kd, b, h, S, H, D);
            widen_head(v, vd, b, h, S, H, D);
#pragma omp parallel
            {
                double* x = (double*)calloc((size_t)S, sizeof(double));
                double* qrow = (double*)calloc((size_t)D, sizeof(double));
                if (!x || !qrow) {
#pragma omp atomic write
                    status = -1;
                } else {
#pragma omp for schedule(dynamic, 4)
                    for (int64_t r = 0; r < n_rows; ++r) {
                        if (rows_b[r] != b) continue;
                        for (int64_t d = 0; d < D; ++d)
                            qrow[d] = bf16_to_double(q[idx4(b, rows_s[r], h, d, S, H, D)]);
                        attention_row(qrow, kd, vd, keys_of_row(rows_s[r], S, causal), D, scale, x,
                                      o_rows + (size_t)((r * H + h) * D));
                    }
                }
                free(x);
                free(qrow);
            }
        }
    }
    free(kd);
    free(vd);
    return status;
}

/*
 * Selected query rows of exact attention.
 *   q, k, v : bf16 bits [B,S,H,D]
 *   rows_b, rows_s : n_rows query positions (b, s)
 *   o_rows  : double [n_rows, H, D] output (row r, head h at (r*H + h)*D)
 * Returns 0, or -1 on allocation failure / bad arguments.
 */
int oracle_attention_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          int64_t B, int64_t S, int64_t H, int64_t D, double scale,
                          const int64_t* rows_b, const int64_t* rows_s, int64_t n_rows,
                          double* o_rows, int nthreads) {
    return attention_rows_impl(q, k, v, B, S, H, D, scale, rows_b, rows_s, n_rows, o_rows, nthreads, 0);
}

/* The same rows of causal attention (row s attends to keys 0 .. s). */
int oracle_attention_rows_causal(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 int64_t B, int64_t S, int64_t H, int64_t D, double scale,
                                 const int64_t* rows_b, const int64_t* rows_s, int64_t n_rows,
                                 double* o_rows, int nthreads) {
    return attention_rows_impl(q, k, v, B, S, H, D, scale, rows_b, rows_s, n_rows, o_rows, nthreads, 1);
}

static int attention_impl(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          int64_t B, int64_t S, int64_t H, int64_t D, double scale,
                          double* o, int nthreads, int causal) {
    if (B < 1 || S < 1 || H < 1 || D < 1) return -1;
    set_threads(nthreads);
    double* kd = (double*)malloc(sizeof(double) * (size_t)(S * D));
    double* vd = (double*)malloc(sizeof(double) * (size_t)(S * D));
    if (!kd || !vd) { free(kd); free(vd); return -1; }
    int status = 0;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t h = 0; h < H; ++h) {
            widen_head(k, kd, b, h, S, H, D);
            widen_head(v, vd, b, h, S, H, D);
#pragma omp parallel
            {
                double* x = (double*)calloc((size_t)S, sizeof(double));
                double* qrow = (double*)calloc((size_t)D, sizeof(double));
                double* orow = (double*)calloc((size_t)D, sizeof(double));
                if (!x || !qrow || !orow) {
#pragma omp atomic write
                    status = -1;
                } else {
#pragma omp for schedule(static)
                    for (int64_t i = 0; i < S; ++i) {
                        for (int64_t d = 0; d < D; ++d) qrow[d] = bf16_to_double(q[idx4(b, i, h, d, S, H, D)]);
                        attention_row(qrow, kd, vd, keys_of_row(i, S, causal), D, scale, x, orow);
                        for (int64_t d = 0; d < D; ++d) o[idx4(b, i, h, d, S, H, D)] = orow[d];
                    }
                }
                free(x);
                free(qrow);
                free(orow);
            }
        }
    }
    free(kd);
    free(vd);
    return status;
}

/*
 * Full exact attention: o is double [B,S,H,D].
 */
int oracle_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     int64_t B, int64_t S, int64_t H, int64_t D, double scale,
                     double* o, int nthreads) {
    return attention_impl(q, k, v, B, S, H, D, scale, o, nthreads, 0);
}

/* Full exact causal attention: o is double [B,S,H,D]. */
int oracle_attention_causal(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            int64_t B, int64_t S, int64_t H, int64_t D, double scale,
                            double* o, int nthreads) {
    return attention_impl(q, k, v, B, S, H, D, scale, o, nthreads, 1);
}

static int attention_weights_impl(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                  int64_t B, int64_t S, int64_t H, int64_t D, double scale,
                                  int64_t b, int64_t i, int64_t h, double* w, double* orow, int causal) {
    if (b < 0 || b >= B || i < 0 || i >= S || h < 0 || h >= H) return -1;
    double* kd = (double*)malloc(sizeof(double) * (size_t)(S * D));
    double* vd = (double*)malloc(sizeof(double) * (size_t)(S * D));
    double* qrow = (double*)malloc(sizeof(double) * (size_t)D);
    if (!kd || !vd || !qrow) { free(kd); free(vd); free(qrow); return -1; }
    widen_head(k, kd, b, h, S, H, D);
    widen_head(v, vd, b, h, S, H, D);
    for (int64_t d = 0; d < D; ++d) qrow[d] = bf16_to_double(q[idx4(b, i, h, d, S, H, D)]);
    const int64_t n = keys_of_row(i, S, causal);
    attention_row(qrow, kd, vd, n, D, scale, w, orow);
    for (int64_t j = n; j < S; ++j) w[j] = 0.0;   /* keys the row does not attend to */
    free(kd);
    free(vd);
    free(qrow);
    return 0;
}

/*
 * The normalised softmax weights of one query row (b, i, h): w[S], sum 1.
 * Exposed so that the row-sum and non-negativity of the weights can be checked.
 */
int oracle_attention_weights(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                             int64_t B, int64_t S, int64_t H, int64_t D, double scale,
                             int64_t b, int64_t i, int64_t h, double* w, double* orow) {
    return attention_weights_impl(q, k, v, B, S, H, D, scale, b, i, h, w, orow, 0);
}

/* The same for causal attention: w[j] = 0 for j > i, sum over j <= i is 1. */
int oracle_attention_weights_causal(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                    int64_t B, int64_t S, int64_t H, int64_t D, double scale,
                                    int64_t b, int64_t i, int64_t h, double* w, double* orow) {
    return attention_weights_impl(q, k, v, B, S, H, D, scale, b, i, h, w, orow, 1);
}

/*
 * Step 2a of the re-shard: split O [B,S,H,D] into the P head shards a Ulysses
 * rank holds, L[r] = [B,S,H/P,D], stored back to back (r outermost).
 */
int oracle_head_shards(const double* o, double* L, int64_t B, int64_t S, int64_t H,
                       int64_t D, int64_t P) {
    if (P < 1 || H % P != 0) return -1;
    const int64_t Hl = H / P;
    for (int64_t r = 0; r < P; ++r)
        for (int64_t b = 0; b < B; ++b)
            for (int64_t s = 0; s < S; ++s)
                for (int64_t j = 0; j < Hl; ++j)
                    for (int64_t d = 0; d < D; ++d)
                        L[(size_t)(r * B * S * Hl * D) + idx4(b, s, j, d, S, Hl, D)] =
                            o[idx4(b, s, r * Hl + j, d, S, H, D)];
    return 0;
}

/*
 * Step 2b: the post-attention All-to-All.  Rank r sends to rank p the rows of
 * p's sequence block [p*S/P, (p+1)*S/P) for its heads; p places them at the
 * global head index r*H/P + j.  out[p] = [B,S/P,H,D], stored back to back.
 */
int oracle_a2a(const double* L, double* out, int64_t B, int64_t S, int64_t H,
               int64_t D, int64_t P) {
    if (P < 1 || H % P != 0 || S % P != 0) return -1;
    const int64_t Hl = H / P, Sl = S / P;
    for (int64_t r = 0; r < P; ++r)          /* source rank */
        for (int64_t p = 0; p < P; ++p)      /* destination rank */
            for (int64_t b = 0; b < B; ++b)
                for (int64_t s2 = 0; s2 < Sl; ++s2)
                    for (int64_t j = 0; j < Hl; ++j)
                        for (int64_t d = 0; d < D; ++d)
                            out[(size_t)(p * B * Sl * H * D) + idx4(b, s2, r * Hl + j, d, Sl, H, D)] =
                                L[(size_t)(r * B * S * Hl * D) + idx4(b, p * Sl + s2, j, d, S, Hl, D)];
    return 0;
}

/*
 * The inverse All-to-All (sequence shards back to head shards), used only to
 * check that the forward exchange is a permutation (round trip).
 */
int oracle_a2a_inverse(const double* out, double* L, int64_t B, int64_t S, int64_t H,
                       int64_t D, int64_t P) {
    if (P < 1 || H % P != 0 || S % P != 0) return -1;
    const int64_t Hl = H / P, Sl = S / P;
    for (int64_t p = 0; p < P; ++p)
        for (int64_t r = 0; r < P; ++r)
            for (int64_t b = 0; b < B; ++b)
                for (int64_t s2 = 0; s2 < Sl; ++s2)
                    for (int64_t j = 0; j < Hl; ++j)
                        for (int64_t d = 0; d < D; ++d)
                            L[(size_t)(r * B * S * Hl * D) + idx4(b, p * Sl + s2, j, d, S, Hl, D)] =
                                out[(size_t)(p * B * Sl * H * D) + idx4(b, s2, r * Hl + j, d, Sl, H, D)];
    return 0;
}
