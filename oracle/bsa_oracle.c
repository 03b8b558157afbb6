/*
 * bsa_oracle.c -- plain, slow, fp64 CPU oracle for content-dependent
 * block-sparse attention (forward).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library: it re-derives every step
 * from the pages' text, one obvious loop at a time, in double precision.
 *
 * Pages followed (cited by page title and section):
 *   [P1] "sparse-attention-triton-bench" (nishantmodi.me), section
 *        "Two-stage block indexer": Stage 1 coarse scoring (mean-pool each
 *        B-token key block, score every query against every block
 *        representative), Stage 2 fine attention (take the top-k blocks,
 *        run dense attention over the k*B selected tokens).
 *   [P2] "yayme/CUDA-kernel" README, sparsity-pattern definition: query i
 *        attends key j iff |i-j| <= w (local window) or j % s == 0 (global
 *        stride); a tile is skipped iff it holds no active pair.
 *   [P3] "Block-Sparse & Linear Attention Kernels", section 2, "Sliding
 *        Window Attention (Mistral)": softmax(q_i K_win^T / sqrt(d_k)) V_win;
 *        section 1, "Common Sparse Patterns": the causal (lower-triangle)
 *        pattern.
 *   [P1] section "What's next", per-head sparsity budgets: top_k chosen per
 *        head instead of one global value, on the same per-head stage-1
 *        scores.
 *
 * Readings where the pages are silent:
 *   - softmax scale 1/sqrt(d) comes from [P3]; the caller passes it;
 *   - stage-1 scores are unscaled dot products (a positive scale cannot
 *     change the ranking);
 *   - ties in the top-k go to the lower block index; the selected set is
 *     reported in ascending block order, padded with -1 when k > nb;
 *   - a ragged last block is pooled over its valid tokens only;
 *   - the sliding window is causal and holds W tokens including the query
 *     itself: i-W < j <= i;
 *   - the softmax is a plain two-pass softmax (max, then exponentials), NOT
 *     an online one, so it shares no structure with the GPU path;
 *   - a row with no selected token yields O = 0, lse = -inf, psum = 0;
 *   - causal dynamic selection: query i may select only the blocks that hold
 *     a key j <= i, i.e. b <= floor(i / B), and attends only keys j <= i
 *     inside them (the causal pattern of [P3] section 1 applied at both
 *     stages);
 *   - the always-include-local-block variant: the query's own block
 *     floor(i / B) is selected first and the other k - 1 blocks by score;
 *     a budget of 0 selects nothing;
 *   - a per-head budget k_h lies in [0, k]; k is the list width.
 *
 * Layout: Q, K, V are [BH][N][d] row-major, element type bf16 (raw bit
 * patterns, widened exactly) or fp32.  All outputs are double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_BF16 0
#define ORC_FP32 1

#define ORC_MASK_LOCAL_GLOBAL 1
#define ORC_MASK_SLIDING 2
#define ORC_MASK_CAUSAL 3

/* Exact widening of one input element to double. */
static double widen(const void *base, int dtype, int64_t i) {
    if (dtype == ORC_BF16) {
        uint32_t u = (uint32_t)((const uint16_t *)base)[i] << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    return (double)((const float *)base)[i];
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * [P1] Stage 1, first half: the representative of key block b is the mean
 * of the keys in it.  Kbar is [BH][nb][d], nb = ceil(N/B).
 */
void orc_pool(const void *K, int dtype, int64_t BH, int64_t N, int64_t d,
              int64_t B, double *Kbar) {
    int64_t nb = (N + B - 1) / B;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t bh = 0; bh < BH; ++bh) {
        for (int64_t b = 0; b < nb; ++b) {
            int64_t j0 = b * B;
            int64_t j1 = j0 + B < N ? j0 + B : N;
            double count = (double)(j1 - j0);
            for (int64_t c = 0; c < d; ++c) {
                double sum = 0.0;
                for (int64_t j = j0; j < j1; ++j)
                    sum += widen(K, dtype, (bh * N + j) * d + c);
                Kbar[(bh * nb + b) * d + c] = sum / count;
            }
        }
    }
}

/*
 * [P1] Stage 1, second half: score each query against every block
 * representative, S[r][b] = q_i . Kbar_b, for the requested rows only
 * (rows[r] = bh*N + i).  S is [nrows][nb].
 */
void orc_scores(const void *Q, int dtype, int64_t BH, int64_t N, int64_t d,
                const double *Kbar, int64_t nb, const int64_t *rows,
                int64_t nrows, double *S) {
    (void)BH;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t bh = rows[r] / N;
        int64_t i = rows[r] % N;
        for (int64_t b = 0; b < nb; ++b) {
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += widen(Q, dtype, (bh * N + i) * d + c) *
                       Kbar[(bh * nb + b) * d + c];
            S[r * nb + b] = dot;
        }
    }
}

typedef struct {
    double score;
    int32_t block;
} scored_block;

/* Order: higher score first; equal scores -> lower block index first. */
static int by_score_then_block(const void *pa, const void *pb) {
    const scored_block *a = (const scored_block *)pa;
    const scored_block *b = (const scored_block *)pb;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->block > b->block) - (a->block < b->block);
}

static int ascending_int(const void *pa, const void *pb) {
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/*
 * [P1] Stage 2, selection: "take the top-k highest-scoring blocks".  Each
 * row's blocks are fully sorted by (score desc, block asc) and the first
 * min(k, nb) kept; they are written in ascending block order, the rest of
 * the row padded with -1.  kth[r] receives the score of the last block kept
 * (the k-th best), used by the tests' tie band.
 */
void orc_topk(const double *S, int64_t nrows, int64_t nb, int64_t k,
              int32_t *idx, double *kth) {
    int64_t kk = k < nb ? k : nb;
#pragma omp parallel
    {
        scored_block *tmp = (scored_block *)malloc(sizeof(scored_block) * (size_t)nb);
#pragma omp for schedule(static)
        for (int64_t r = 0; r < nrows; ++r) {
            for (int64_t b = 0; b < nb; ++b) {
                tmp[b].score = S[r * nb + b];
                tmp[b].block = (int32_t)b;
            }
            qsort(tmp, (size_t)nb, sizeof(scored_block), by_score_then_block);
            int32_t *out = idx + r * k;
            for (int64_t t = 0; t < kk; ++t) out[t] = tmp[t].block;
            qsort(out, (size_t)kk, sizeof(int32_t), ascending_int);
            for (int64_t t = kk; t < k; ++t) out[t] = -1;
            if (kth) kth[r] = kk > 0 ? tmp[kk - 1].score : -INFINITY;
        }
        free(tmp);
    }
}

/*
 * Stage 2 selection with the options ([P1] "What's next" per-head budgets;
 * [P3] section 1 causal pattern; the local-block variant).  Row r is query
 * i of (batch*head) row bh, rows[r] = bh*N + i.  Its budget is
 * k_r = head_k[bh] (or k when head_k is NULL); its eligible blocks are all
 * nb blocks, or b <= floor(i/B) when causal.  With `local`, block
 * floor(i/B) is taken first (if k_r >= 1) and the other k_r - 1 are the
 * best-scoring eligible blocks except it; without, the k_r best eligible
 * blocks.  Best = (score desc, block asc).  Output as orc_topk: ascending
 * ids, -1 padded to width k.
 */
void orc_select(const double *S, const int64_t *rows, int64_t nrows,
                int64_t nb, int64_t N, int64_t B, int64_t k,
                const int32_t *head_k, int causal, int local, int32_t *idx) {
#pragma omp parallel
    {
        scored_block *tmp = (scored_block *)malloc(sizeof(scored_block) * (size_t)nb);
#pragma omp for schedule(static)
        for (int64_t r = 0; r < nrows; ++r) {
            int64_t bh = rows[r] / N;
            int64_t i = rows[r] % N;
            int64_t own = i / B;
            int64_t kr = head_k ? head_k[bh] : k;
            if (kr < 0) kr = 0;
            if (kr > k) kr = k;
            int64_t last = causal ? own : nb - 1;   /* eligible: b <= last */
            int32_t *out = idx + r * k;
            int64_t taken = 0;
            if (local && kr >= 1) out[taken++] = (int32_t)own;
            int64_t ne = 0;
            for (int64_t b = 0; b <= last; ++b) {
                if (local && b == own) continue;
                tmp[ne].score = S[r * nb + b];
                tmp[ne].block = (int32_t)b;
                ++ne;
            }
            qsort(tmp, (size_t)ne, sizeof(scored_block), by_score_then_block);
            for (int64_t t = 0; t < ne && taken < kr; ++t) out[taken++] = tmp[t].block;
            qsort(out, (size_t)taken, sizeof(int32_t), ascending_int);
            for (int64_t t = taken; t < k; ++t) out[t] = -1;
        }
        free(tmp);
    }
}

/*
 * Softmax attention of one query over an explicit token list, two passes:
 * s_j = scale * q.k_j ; m = max s_j ; p_j = exp(s_j - m) ; l = sum p_j ;
 * o = sum p_j v_j / l.  Also returns lse = m + log l and the row sum of the
 * normalised weights (1 up to rounding).
 */
static void attend_tokens(const void *Q, const void *K, const void *V,
                          int dtype, int64_t N, int64_t d, int64_t bh,
                          int64_t i, const int64_t *tok, int64_t ntok,
                          double scale, double *s_buf, double *o,
                          double *lse, double *psum) {
    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    if (ntok == 0) {
        *lse = -INFINITY;
        *psum = 0.0;
        return;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < ntok; ++t) {
        int64_t j = tok[t];
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c)
            dot += widen(Q, dtype, (bh * N + i) * d + c) *
                   widen(K, dtype, (bh * N + j) * d + c);
        s_buf[t] = scale * dot;
        if (s_buf[t] > m) m = s_buf[t];
    }
    double l = 0.0;
    for (int64_t t = 0; t < ntok; ++t) {
        double p = exp(s_buf[t] - m);
        s_buf[t] = p;
        l += p;
    }
    double total = 0.0;
    for (int64_t t = 0; t < ntok; ++t) {
        double w = s_buf[t] / l;
        total += w;
        int64_t j = tok[t];
        for (int64_t c = 0; c < d; ++c)
            o[c] += w * widen(V, dtype, (bh * N + j) * d + c);
    }
    *lse = m + log(l);
    *psum = total;
}

/*
 * [P1] Stage 2, fine attention: for row r (rows[r] = bh*N + i) the token set
 * is the union of the B tokens of each listed block idx[r][0..k) (entries
 * < 0 are padding; a ragged last block contributes its valid tokens only),
 * and the output is dense softmax attention over that set.  With `causal`
 * only the keys j <= i of those blocks are in the set ([P3] section 1).
 * O is [nrows][d]; lse and psum are [nrows].
 */
void orc_fine(const void *Q, const void *K, const void *V, int dtype,
              int64_t BH, int64_t N, int64_t d, int64_t B,
              const int32_t *idx, int64_t k, const int64_t *rows,
              int64_t nrows, int causal, double scale, double *O, double *lse,
              double *psum) {
    (void)BH;
#pragma omp parallel
    {
        int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)(k * B + 1));
        double *sb = (double *)malloc(sizeof(double) * (size_t)(k * B + 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < nrows; ++r) {
            int64_t bh = rows[r] / N;
            int64_t i = rows[r] % N;
            int64_t ntok = 0;
            for (int64_t t = 0; t < k; ++t) {
                int32_t b = idx[r * k + t];
                if (b < 0) continue;
                for (int64_t j = (int64_t)b * B; j < ((int64_t)b + 1) * B && j < N; ++j)
                    if (!causal || j <= i) tok[ntok++] = j;
            }
            attend_tokens(Q, K, V, dtype, N, d, bh, i, tok, ntok, scale, sb,
                          O + r * d, lse + r, psum + r);
        }
        free(tok);
        free(sb);
    }
}

/*
 * Token-level masks of the static patterns.
 *  [P2] local + global: |i-j| <= w  or  j % s == 0  (w < 0 disables the
 *       local band, s <= 0 disables the global columns);
 *  [P3] sliding window, causal, W tokens including i:  i-W < j <= i.
 *  [P3] section 1, causal (lower triangle):  j <= i.
 */
/*
 * [P1] What's next, backward pass: gradients of the fine stage through the
 * sparse softmax-weighted sum, with the selection held fixed (it is a
 * discrete choice).  For row i of head bh with token set T_i (the listed
 * blocks' keys; only j <= i when causal), s_ij = scale q_i.k_j,
 * p_ij = softmax over T_i, o_i = sum_j p_ij v_j, and a given dO:
 *   dv_j += p_ij do_i
 *   dp_ij = do_i . v_j
 *   ds_ij = p_ij (dp_ij - sum_t p_it dp_it)
 *   dq_i  = scale sum_j ds_ij k_j
 *   dk_j += scale ds_ij q_i
 * idx holds the lists of every row [BH*N][k]; every row is processed, one
 * head per thread (dK, dV gather over a head's rows).  dQ, dK, dV are
 * [BH][N][d] doubles.  A row with no token contributes nothing.
 */
void orc_fine_backward(const void *Q, const void *K, const void *V, const void *dO,
                       int dtype, int64_t BH, int64_t N, int64_t d, int64_t B,
                       const int32_t *idx, int64_t k, int causal, double scale,
                       double *dQ, double *dK, double *dV) {
    memset(dQ, 0, sizeof(double) * (size_t)(BH * N * d));
    memset(dK, 0, sizeof(double) * (size_t)(BH * N * d));
    memset(dV, 0, sizeof(double) * (size_t)(BH * N * d));
#pragma omp parallel
    {
        int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)(k * B + 1));
        double *p = (double *)malloc(sizeof(double) * (size_t)(k * B + 1));
        double *dp = (double *)malloc(sizeof(double) * (size_t)(k * B + 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < BH; ++bh) {
            for (int64_t i = 0; i < N; ++i) {
                const int64_t r = bh * N + i;
                int64_t nt = 0;
                for (int64_t t = 0; t < k; ++t) {
                    int32_t b = idx[r * k + t];
                    if (b < 0) continue;
                    for (int64_t j = (int64_t)b * B; j < ((int64_t)b + 1) * B && j < N; ++j)
                        if (!causal || j <= i) tok[nt++] = j;
                }
                if (nt == 0) continue;
                double m = -INFINITY;
                for (int64_t t = 0; t < nt; ++t) {
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c)
                        dot += widen(Q, dtype, r * d + c) * widen(K, dtype, (bh * N + tok[t]) * d + c);
                    p[t] = scale * dot;
                    if (p[t] > m) m = p[t];
                }
                double l = 0.0;
                for (int64_t t = 0; t < nt; ++t) {
                    p[t] = exp(p[t] - m);
                    l += p[t];
                }
                double rowsum = 0.0;                 /* sum_t p_it dp_it */
                for (int64_t t = 0; t < nt; ++t) {
                    p[t] /= l;
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c)
                        dot += widen(dO, dtype, r * d + c) * widen(V, dtype, (bh * N + tok[t]) * d + c);
                    dp[t] = dot;
                    rowsum += p[t] * dot;
                }
                for (int64_t t = 0; t < nt; ++t) {
                    const int64_t jr = bh * N + tok[t];
                    const double ds = p[t] * (dp[t] - rowsum);
                    for (int64_t c = 0; c < d; ++c) {
                        dV[jr * d + c] += p[t] * widen(dO, dtype, r * d + c);
                        dQ[r * d + c] += scale * ds * widen(K, dtype, jr * d + c);
                        dK[jr * d + c] += scale * ds * widen(Q, dtype, r * d + c);
                    }
                }
            }
        }
        free(tok);
        free(p);
        free(dp);
    }
}

int orc_mask(int kind, int64_t w, int64_t s, int64_t W, int64_t i, int64_t j) {
    if (kind == ORC_MASK_LOCAL_GLOBAL) {
        int64_t dist = i > j ? i - j : j - i;
        int local = (w >= 0) && (dist <= w);
        int global = (s > 0) && (j % s == 0);
        return local || global;
    }
    if (kind == ORC_MASK_SLIDING) return (j > i - W) && (j <= i);
    if (kind == ORC_MASK_CAUSAL) return j <= i;
    return 1;
}

/*
 * Static patterns by their plain definition: dense softmax attention over
 * {j in [0,N) : mask(i, j)} -- skipping inactive tiles is only a speed-up
 * ([P2] tile skipping; [P3] section 2 block-sparse loop), so the oracle
 * visits every key.
 */
void orc_masked(const void *Q, const void *K, const void *V, int dtype,
                int64_t BH, int64_t N, int64_t d, int kind, int64_t w,
                int64_t s, int64_t W, const int64_t *rows, int64_t nrows,
                double scale, double *O, double *lse, double *psum) {
    (void)BH;
#pragma omp parallel
    {
        int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)N);
        double *sb = (double *)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < nrows; ++r) {
            int64_t bh = rows[r] / N;
            int64_t i = rows[r] % N;
            int64_t ntok = 0;
            for (int64_t j = 0; j < N; ++j)
                if (orc_mask(kind, w, s, W, i, j)) tok[ntok++] = j;
            attend_tokens(Q, K, V, dtype, N, d, bh, i, tok, ntok, scale, sb,
                          O + r * d, lse + r, psum + r);
        }
        free(tok);
        free(sb);
    }
}

/*
 * [P2] active tiles by brute force: tile (I, J) of size tq x tk is active iff
 * some in-range pair (i, j) inside it is active.  Only tile rows
 * [row_begin, row_end) are evaluated; act is [row_end-row_begin][ceil(N/tk)].
 * Returns the number of active (i, j) pairs seen in those tile rows.
 */
int64_t orc_active_tiles(int64_t N, int64_t tq, int64_t tk, int kind,
                         int64_t w, int64_t s, int64_t W, int64_t row_begin,
                         int64_t row_end, uint8_t *act) {
    int64_t nkt = (N + tk - 1) / tk;
    int64_t pairs = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : pairs)
    for (int64_t I = row_begin; I < row_end; ++I) {
        for (int64_t J = 0; J < nkt; ++J) {
            int any = 0;
            for (int64_t i = I * tq; i < (I + 1) * tq && i < N; ++i)
                for (int64_t j = J * tk; j < (J + 1) * tk && j < N; ++j)
                    if (orc_mask(kind, w, s, W, i, j)) {
                        any = 1;
                        ++pairs;
                    }
            act[(I - row_begin) * nkt + J] = (uint8_t)any;
        }
    }
    return pairs;
}
