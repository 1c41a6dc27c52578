/*
 * CPU oracle for the block-sparse attention forward and backward passes, the
 * tile layout, the coarse key-tile selection that produces the block-sparse
 * selection, and the output un-tiling with the gate.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * FP64 statement of what the GPU library computes.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or helper with the CUDA library, and the library never calls it.
 *
 * Source of the definition: the FastVideo kernel page (hao-ai-lab/FastVideo
 * commit 8503617, fastvideo-kernel/python).
 *   - Commit adding the sm_121a tile-128 block-sparse forward: the operation
 *     takes q, k, v, q2k_idx, q2k_num and variable_block_sizes and returns the
 *     attention output; each query tile attends to the key tiles its
 *     selection lists; tiles are 64 or 128 tokens.
 *   - sm_121a hardening commit, "Kernel" items: a NaN softmax sum yields a NaN
 *     output row (the test is l != 0, not l > 0); rows without keys stay 0;
 *     keys past a tile's valid count are masked, so NaN/Inf stored in padding
 *     rows of K or V cannot reach the output.
 *   - Attn-QAT SM100 commit: "softmax statistics" are an output of the forward
 *     pass (here: the natural-log log-sum-exp per query row).
 *
 * Readings where the page is silent (stated once here, used below):
 *   - q2k_idx is [B,H,NT,max_kv], q2k_num is [B,H,NT], block_sizes is [NT];
 *     the selection is per (batch, head, query tile).
 *   - Selected key tiles must be distinct and in [0, NT); anything else is an
 *     input error (return code), never silently accepted.
 *   - A query row r of tile t with r >= block_sizes[t] is padding: output +0,
 *     lse = -inf.  An empty key list gives output +0 and lse = -inf.
 *   - m is the maximum score with NaN propagating; l = sum exp(s - m);
 *     out = (sum exp(s - m) v) / l when l != 0, else 0; lse = m + log(l).
 *   - Padding rows of Q, K and V are never read.
 *
 * The definition is computed literally: all scores of a row first, then the
 * maximum, then the weights; no online softmax, no tiling, FP64 throughout,
 * sums in index order.  Build with -ffp-contract=off so no multiply-add is
 * fused and results are identical on every host.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_INDEX -7
#define ORACLE_ERR_NOMEM -8

/* bf16 is the top half of an IEEE binary32, so the widening is exact. */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *k, *v;     /* bf16 bits, tile-major [B,H,NT*T,D] */
    const int32_t *q2k_idx, *q2k_num, *block_sizes;
    int B, H, NT, T, D, max_kv;
    double scale;
    const int64_t *units;          /* flat (b*H + h)*NT + t */
    int64_t n_units;
    double *out;                   /* [n_units, T, D] */
    double *lse;                   /* [n_units, T] or NULL */
    int64_t next;                  /* shared work cursor */
    pthread_mutex_t lock;
    int status;
} job_t;

/* One query tile: every valid row r < n_t gets the softmax over the valid rows
 * of its selected key tiles. */
static int one_query_tile(job_t *J, int64_t unit, int64_t slot, double *scores, double *qrow,
                          double *acc) {
    const int T = J->T, D = J->D, NT = J->NT;
    const int64_t Sp = (int64_t)NT * T;
    const int t = (int)(unit % NT);
    const int64_t bh = unit / NT;
    const int n_t = J->block_sizes[t];
    const int K = J->q2k_num[unit];
    const int32_t *sel = J->q2k_idx + unit * J->max_kv;
    const uint16_t *Qp = J->q + bh * Sp * D;
    const uint16_t *Kp = J->k + bh * Sp * D;
    const uint16_t *Vp = J->v + bh * Sp * D;
    double *O = J->out + slot * (int64_t)T * D;
    double *L = J->lse ? J->lse + slot * (int64_t)T : NULL;

    for (int r = 0; r < T; ++r) {
        for (int d = 0; d < D; ++d) O[(int64_t)r * D + d] = 0.0;
        if (L) L[r] = -INFINITY;
        if (r >= n_t) continue;                       /* padding query row */

        for (int d = 0; d < D; ++d) qrow[d] = bf16_to_double(Qp[((int64_t)t * T + r) * D + d]);

        /* 1. scores over the key list, in list order */
        int64_t n = 0;
        for (int i = 0; i < K; ++i) {
            const int j = sel[i];
            for (int c = 0; c < J->block_sizes[j]; ++c) {
                const uint16_t *krow = Kp + ((int64_t)j * T + c) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += qrow[d] * bf16_to_double(krow[d]);
                scores[n++] = J->scale * dot;
            }
        }
        if (n == 0) continue;                         /* no keys: row stays 0 */

        /* 2. maximum, NaN propagating */
        double m = -INFINITY;
        for (int64_t e = 0; e < n; ++e) {
            if (isnan(scores[e]) || isnan(m)) m = NAN;
            else if (scores[e] > m) m = scores[e];
        }

        /* 3. weights, their sum, and the weighted sum of values */
        double l = 0.0;
        for (int d = 0; d < D; ++d) acc[d] = 0.0;
        int64_t e = 0;
        for (int i = 0; i < K; ++i) {
            const int j = sel[i];
            for (int c = 0; c < J->block_sizes[j]; ++c, ++e) {
                const double w = exp(scores[e] - m);
                const uint16_t *vrow = Vp + ((int64_t)j * T + c) * D;
                l += w;
                for (int d = 0; d < D; ++d) acc[d] += w * bf16_to_double(vrow[d]);
            }
        }
        for (int d = 0; d < D; ++d) O[(int64_t)r * D + d] = (l != 0.0) ? acc[d] / l : 0.0;
        if (L) L[r] = m + log(l);
    }
    return ORACLE_OK;
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    int64_t max_keys = (int64_t)J->max_kv * J->T;
    double *scores = (double *)malloc(sizeof(double) * (size_t)(max_keys > 0 ? max_keys : 1));
    double *qrow = (double *)malloc(sizeof(double) * (size_t)J->D);
    double *acc = (double *)malloc(sizeof(double) * (size_t)J->D);
    if (!scores || !qrow || !acc) {
        pthread_mutex_lock(&J->lock);
        J->status = ORACLE_ERR_NOMEM;
        pthread_mutex_unlock(&J->lock);
    } else {
        for (;;) {
            pthread_mutex_lock(&J->lock);
            int64_t slot = J->next++;
            pthread_mutex_unlock(&J->lock);
            if (slot >= J->n_units) break;
            one_query_tile(J, J->units[slot], slot, scores, qrow, acc);
        }
    }
    free(scores);
    free(qrow);
    free(acc);
    return NULL;
}

/* Checks the selection of every requested unit: counts in [0, max_kv], indices
 * in [0, NT) and pairwise distinct. */
static int check_units(const job_t *J) {
    const int64_t total = (int64_t)J->B * J->H * J->NT;
    for (int t = 0; t < J->NT; ++t)
        if (J->block_sizes[t] < 0 || J->block_sizes[t] > J->T) return ORACLE_ERR_ARG;
    for (int64_t s = 0; s < J->n_units; ++s) {
        const int64_t u = J->units[s];
        if (u < 0 || u >= total) return ORACLE_ERR_ARG;
        const int K = J->q2k_num[u];
        if (K < 0 || K > J->max_kv) return ORACLE_ERR_INDEX;
        const int32_t *sel = J->q2k_idx + u * J->max_kv;
        for (int i = 0; i < K; ++i) {
            if (sel[i] < 0 || sel[i] >= J->NT) return ORACLE_ERR_INDEX;
            for (int i2 = 0; i2 < i; ++i2)
                if (sel[i2] == sel[i]) return ORACLE_ERR_INDEX;
        }
    }
    return ORACLE_OK;
}

/* Block-sparse attention forward, FP64, for the listed query tiles.
 *   q, k, v     bf16 bit patterns, tile-major [B, H, NT*T, D]
 *   units       flat query-tile ids (b*H + h)*NT + t, n_units of them
 *   out         [n_units, T, D] doubles; lse [n_units, T] doubles or NULL
 * Returns 0, or a negative error for bad arguments / bad selections. */
int oracle_block_sparse_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const int32_t *q2k_idx, const int32_t *q2k_num,
                            const int32_t *block_sizes, int B, int H, int NT, int T, int D,
                            int max_kv, double scale, const int64_t *units, int64_t n_units,
                            double *out, double *lse, int nthreads) {
    if (!q || !k || !v || !q2k_idx || !q2k_num || !block_sizes || !units || !out) return ORACLE_ERR_ARG;
    if (B <= 0 || H <= 0 || NT <= 0 || T <= 0 || D <= 0 || max_kv < 0 || n_units < 0) return ORACLE_ERR_ARG;
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v;
    J.q2k_idx = q2k_idx; J.q2k_num = q2k_num; J.block_sizes = block_sizes;
    J.B = B; J.H = H; J.NT = NT; J.T = T; J.D = D; J.max_kv = max_kv;
    J.scale = scale; J.units = units; J.n_units = n_units; J.out = out; J.lse = lse;
    int rc = check_units(&J);
    if (rc != ORACLE_OK) return rc;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_mutex_init(&J.lock, NULL);
    pthread_t th[256];
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    pthread_mutex_destroy(&J.lock);
    return J.status;
}

/* Tile layout: dst[b, h, row, :] = src[b, row_to_token[row], h, :] for every
 * tile-major row; a row whose map entry is -1 is padding and is written as +0.
 *   src bf16 bits [B, S, H, D]; dst bf16 bits [B, H, NT*T, D].
 * Source: the fused tile_to_bhsd commit on the same page (one pass that
 * scatters token-major Q/K/V into tile-major BHSD). */
int oracle_tile_layout(const uint16_t *src, const int32_t *row_to_token, uint16_t *dst, int B, int S,
                       int H, int D, int NT, int T) {
    if (!src || !row_to_token || !dst || B <= 0 || S < 0 || H <= 0 || D <= 0 || NT <= 0 || T <= 0)
        return ORACLE_ERR_ARG;
    const int64_t Sp = (int64_t)NT * T;
    for (int64_t row = 0; row < Sp; ++row) {
        const int32_t s = row_to_token[row];
        if (s < -1 || s >= S) return ORACLE_ERR_INDEX;
    }
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int64_t row = 0; row < Sp; ++row) {
                const int32_t s = row_to_token[row];
                uint16_t *o = dst + (((int64_t)b * H + h) * Sp + row) * D;
                for (int d = 0; d < D; ++d)
                    o[d] = (s < 0) ? (uint16_t)0 : src[(((int64_t)b * S + s) * H + h) * D + d];
            }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------
 * Coarse key-tile selection of video sparse attention: the step that produces
 * q2k_idx / q2k_num for the block-sparse forward.
 *
 * The page names video sparse attention (VSA) and its block-sparse fine stage
 * (commit adding the sm_121a tile-128 forward; fused tile_to_bhsd commit:
 * "Wan VSA inference"), but not the coarse stage's arithmetic.  Plain reading,
 * stated here and used below:
 *   1. every non-empty tile t (n_t = block_sizes[t] > 0) is pooled to the mean
 *      of its valid rows: qm[t] = (sum_{r < n_t} q[t*T + r]) / n_t, and km[t]
 *      likewise from k; padding rows are never read;
 *   2. the tile-level score is the dot product score[t][j] = sum_d qm[t][d] *
 *      km[j][d], each term added with one fused multiply-add (a positive
 *      softmax scale would not change the ranking);
 *   3. query tile t keeps the topk key tiles j with the largest score among
 *      the candidates (n_j > 0 and the score is not NaN), ties going to the
 *      smaller j; with fewer candidates it keeps all of them; an empty query
 *      tile keeps none;
 *   4. the kept tiles are written in ascending order to q2k_idx[b,h,t,0:kk],
 *      the rest of the row is -1, and q2k_num[b,h,t] = kk.
 * The selection is an integer result decided by floating point, so this
 * oracle takes the decision in the precision of the GPU kernel (fp32), with
 * every sum in index order: the means by plain adds, the scores by fmaf
 * (-ffp-contract=off keeps every other operation unfused).
 * scores (nullable) receives the fp32 score matrix [B,H,NT,NT] (NaN for a
 * non-candidate pair) so that tests can tell exact ties from clear gaps.
 * ------------------------------------------------------------------------ */
int oracle_coarse_select(const uint16_t *q, const uint16_t *k, const int32_t *block_sizes, int B, int H,
                         int NT, int T, int D, int topk, int32_t *q2k_idx, int32_t *q2k_num, float *scores) {
    if (!q || !k || !block_sizes || !q2k_idx || !q2k_num || B <= 0 || H <= 0 || NT <= 0 || T <= 0 ||
        D <= 0 || topk < 0)
        return ORACLE_ERR_ARG;
    for (int t = 0; t < NT; ++t)
        if (block_sizes[t] < 0 || block_sizes[t] > T) return ORACLE_ERR_ARG;
    const int64_t Sp = (int64_t)NT * T;
    float *qm = (float *)malloc(sizeof(float) * (size_t)NT * D);
    float *km = (float *)malloc(sizeof(float) * (size_t)NT * D);
    float *row = (float *)malloc(sizeof(float) * (size_t)NT);
    unsigned char *taken = (unsigned char *)malloc((size_t)NT);
    if (!qm || !km || !row || !taken) {
        free(qm);
        free(km);
        free(row);
        free(taken);
        return ORACLE_ERR_NOMEM;
    }
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            const int64_t bh = (int64_t)b * H + h;
            /* 1. tile means, fp32, rows in order */
            for (int t = 0; t < NT; ++t) {
                const int n = block_sizes[t];
                for (int d = 0; d < D; ++d) {
                    float sq = 0.f, sk = 0.f;
                    for (int r = 0; r < n; ++r) {
                        const int64_t at = (bh * Sp + (int64_t)t * T + r) * D + d;
                        sq += (float)bf16_to_double(q[at]);
                        sk += (float)bf16_to_double(k[at]);
                    }
                    qm[(int64_t)t * D + d] = n > 0 ? sq / (float)n : 0.f;
                    km[(int64_t)t * D + d] = n > 0 ? sk / (float)n : 0.f;
                }
            }
            for (int t = 0; t < NT; ++t) {
                /* 2. scores of query tile t against every candidate key tile */
                int n_cand = 0;
                for (int j = 0; j < NT; ++j) {
                    float s = 0.f;
                    for (int d = 0; d < D; ++d) s = fmaf(qm[(int64_t)t * D + d], km[(int64_t)j * D + d], s);
                    const int cand = block_sizes[j] > 0 && !isnan(s);
                    row[j] = cand ? s : NAN;
                    taken[j] = 0;
                    n_cand += cand;
                }
                if (scores) memcpy(scores + (bh * NT + t) * NT, row, sizeof(float) * (size_t)NT);
                /* 3. the kk best candidates: repeatedly the largest score not yet
                 *    taken, the smaller index on a tie */
                int kk = block_sizes[t] > 0 ? (topk < n_cand ? topk : n_cand) : 0;
                for (int i = 0; i < kk; ++i) {
                    int best = -1;
                    for (int j = 0; j < NT; ++j) {
                        if (taken[j] || isnan(row[j])) continue;
                        if (best < 0 || row[j] > row[best]) best = j;
                    }
                    taken[best] = 1;
                }
                /* 4. ascending order, -1 after */
                int32_t *out = q2k_idx + (bh * NT + t) * (int64_t)topk;
                int o = 0;
                for (int j = 0; j < NT; ++j)
                    if (taken[j]) out[o++] = j;
                for (; o < topk; ++o) out[o] = -1;
                q2k_num[bh * NT + t] = kk;
            }
        }
    free(qm);
    free(km);
    free(row);
    free(taken);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------
 * Output un-tiling with the gate: the step after the block-sparse forward.
 * The fused tile_to_bhsd commit on the page describes the layer's tiled path
 * (Q, K, V and the gate scattered into a tile buffer); reading of the step
 * back: every tile-major output row r that holds a token (s = row_to_token[r]
 * >= 0) goes back to token-major order, multiplied element-wise by that
 * token's gate when a gate is given:
 *   out_tok[b, s, h, :] = bf16( float(O[b, h, r, :]) * float(gate[b, s, h, :]) )
 * The product of two bf16 values is exact in fp32, so the only rounding is
 * the final round-to-nearest-even to bf16 (NaN stays NaN).  Padding rows are
 * not read; tokens that no row maps to are left as they are.
 *   o_tile bf16 bits [B, H, NT*T, D]; gate NULL or bf16 bits [B, S, H, D];
 *   out bf16 bits [B, S, H, D].
 * ------------------------------------------------------------------------ */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7fffu + ((u >> 16) & 1u);  /* ties to the even upper half */
    return (uint16_t)(u >> 16);
}

int oracle_untile(const uint16_t *o_tile, const uint16_t *gate, const int32_t *row_to_token, uint16_t *out,
                  int B, int S, int H, int D, int NT, int T) {
    if (!o_tile || !row_to_token || !out || B <= 0 || S < 0 || H <= 0 || D <= 0 || NT <= 0 || T <= 0)
        return ORACLE_ERR_ARG;
    const int64_t Sp = (int64_t)NT * T;
    for (int64_t row = 0; row < Sp; ++row)
        if (row_to_token[row] < -1 || row_to_token[row] >= S) return ORACLE_ERR_INDEX;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int64_t row = 0; row < Sp; ++row) {
                const int32_t s = row_to_token[row];
                if (s < 0) continue;
                const uint16_t *o = o_tile + (((int64_t)b * H + h) * Sp + row) * D;
                uint16_t *dst = out + (((int64_t)b * S + s) * H + h) * D;
                const uint16_t *gt = gate ? gate + (((int64_t)b * S + s) * H + h) * D : NULL;
                for (int d = 0; d < D; ++d)
                    dst[d] = gt ? f32_to_bf16_rne((float)(bf16_to_double(o[d]) * bf16_to_double(gt[d]))) : o[d];
            }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------
 * Block-sparse attention backward (the Attn-QAT SM100 commit on the page
 * names the backward pass and its 64x128 dQ / dK-dV tiles; the gradients are
 * those of the forward defined above).  For every valid query row with key
 * list L (the valid rows of its selected key tiles), in FP64:
 *   s_e = scale * q.k_e,  p = softmax(s) over L,
 *   dp_e = do.v_e,  delta = sum_e p_e dp_e,  ds_e = p_e (dp_e - delta),
 *   dq = scale * sum_e ds_e k_e,  dk_e += scale * ds_e q,  dv_e += p_e do.
 * A row with no keys contributes nothing and gets dq = 0; keys no row selects
 * get dk = dv = 0; padding rows of dq, dk, dv are 0.  Computed per
 * (batch, head) in index order, one thread per (batch, head).
 *   q, k, v, dout: bf16 bits [B,H,NT*T,D]; dq, dk, dv: double [B,H,NT*T,D].
 * ------------------------------------------------------------------------ */
typedef struct {
    const uint16_t *q, *k, *v, *dout;
    const int32_t *q2k_idx, *q2k_num, *block_sizes;
    int B, H, NT, T, D, max_kv;
    double scale;
    double *dq, *dk, *dv;
    int64_t next;
    pthread_mutex_t lock;
    int status;
} bwd_job_t;

static void bwd_one_head(bwd_job_t *J, int64_t bh, double *s, double *p, double *dp, double *qrow,
                         double *drow) {
    const int T = J->T, D = J->D, NT = J->NT;
    const int64_t Sp = (int64_t)NT * T;
    const uint16_t *Qp = J->q + bh * Sp * D, *Kp = J->k + bh * Sp * D, *Vp = J->v + bh * Sp * D;
    const uint16_t *dOp = J->dout + bh * Sp * D;
    double *dQ = J->dq + bh * Sp * D, *dK = J->dk + bh * Sp * D, *dV = J->dv + bh * Sp * D;
    for (int64_t i = 0; i < Sp * D; ++i) dQ[i] = dK[i] = dV[i] = 0.0;
    for (int t = 0; t < NT; ++t) {
        const int64_t unit = bh * NT + t;
        const int K = J->q2k_num[unit];
        const int32_t *sel = J->q2k_idx + unit * J->max_kv;
        for (int r = 0; r < J->block_sizes[t]; ++r) {
            const int64_t qi = (int64_t)t * T + r;
            for (int d = 0; d < D; ++d) {
                qrow[d] = bf16_to_double(Qp[qi * D + d]);
                drow[d] = bf16_to_double(dOp[qi * D + d]);
            }
            int64_t n = 0;
            for (int i = 0; i < K; ++i) {
                const int j = sel[i];
                for (int c = 0; c < J->block_sizes[j]; ++c) {
                    const int64_t kr = (int64_t)j * T + c;
                    double dot = 0.0, dv = 0.0;
                    for (int d = 0; d < D; ++d) {
                        dot += qrow[d] * bf16_to_double(Kp[kr * D + d]);
                        dv += drow[d] * bf16_to_double(Vp[kr * D + d]);
                    }
                    s[n] = J->scale * dot;
                    dp[n] = dv;
                    ++n;
                }
            }
            if (n == 0) continue;
            double m = -INFINITY;
            for (int64_t e = 0; e < n; ++e) {
                if (isnan(s[e]) || isnan(m)) m = NAN;
                else if (s[e] > m) m = s[e];
            }
            double l = 0.0;
            for (int64_t e = 0; e < n; ++e) l += (p[e] = exp(s[e] - m));
            double delta = 0.0;
            for (int64_t e = 0; e < n; ++e) {
                p[e] /= l;
                delta += p[e] * dp[e];
            }
            int64_t e = 0;
            for (int i = 0; i < K; ++i) {
                const int j = sel[i];
                for (int c = 0; c < J->block_sizes[j]; ++c, ++e) {
                    const int64_t kr = (int64_t)j * T + c;
                    const double ds = p[e] * (dp[e] - delta);
                    for (int d = 0; d < D; ++d) {
                        dQ[qi * D + d] += J->scale * ds * bf16_to_double(Kp[kr * D + d]);
                        dK[kr * D + d] += J->scale * ds * qrow[d];
                        dV[kr * D + d] += p[e] * drow[d];
                    }
                }
            }
        }
    }
}

static void *bwd_worker(void *arg) {
    bwd_job_t *J = (bwd_job_t *)arg;
    const int64_t max_keys = (int64_t)(J->max_kv > 0 ? J->max_kv : 1) * J->T;
    double *s = (double *)malloc(sizeof(double) * (size_t)max_keys);
    double *p = (double *)malloc(sizeof(double) * (size_t)max_keys);
    double *dp = (double *)malloc(sizeof(double) * (size_t)max_keys);
    double *qrow = (double *)malloc(sizeof(double) * (size_t)J->D);
    double *drow = (double *)malloc(sizeof(double) * (size_t)J->D);
    if (!s || !p || !dp || !qrow || !drow) {
        pthread_mutex_lock(&J->lock);
        J->status = ORACLE_ERR_NOMEM;
        pthread_mutex_unlock(&J->lock);
    } else {
        for (;;) {
            pthread_mutex_lock(&J->lock);
            const int64_t bh = J->next++;
            pthread_mutex_unlock(&J->lock);
            if (bh >= (int64_t)J->B * J->H) break;
            bwd_one_head(J, bh, s, p, dp, qrow, drow);
        }
    }
    free(s);
    free(p);
    free(dp);
    free(qrow);
    free(drow);
    return NULL;
}

int oracle_block_sparse_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                            const int32_t *q2k_idx, const int32_t *q2k_num, const int32_t *block_sizes, int B,
                            int H, int NT, int T, int D, int max_kv, double scale, double *dq, double *dk,
                            double *dv, int nthreads) {
    if (!q || !k || !v || !dout || !q2k_num || !block_sizes || !dq || !dk || !dv || B <= 0 || H <= 0 ||
        NT <= 0 || T <= 0 || D <= 0 || max_kv < 0 || (!q2k_idx && max_kv > 0))
        return ORACLE_ERR_ARG;
    bwd_job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.dout = dout;
    J.q2k_idx = q2k_idx; J.q2k_num = q2k_num; J.block_sizes = block_sizes;
    J.B = B; J.H = H; J.NT = NT; J.T = T; J.D = D; J.max_kv = max_kv; J.scale = scale;
    J.dq = dq; J.dk = dk; J.dv = dv;
    /* the same selection checks as the forward */
    job_t C;
    memset(&C, 0, sizeof C);
    C.q2k_idx = q2k_idx; C.q2k_num = q2k_num; C.block_sizes = block_sizes;
    C.B = B; C.H = H; C.NT = NT; C.T = T; C.max_kv = max_kv;
    C.n_units = (int64_t)B * H * NT;
    int64_t *all = (int64_t *)malloc(sizeof(int64_t) * (size_t)C.n_units);
    if (!all) return ORACLE_ERR_NOMEM;
    for (int64_t u = 0; u < C.n_units; ++u) all[u] = u;
    C.units = all;
    const int rc = check_units(&C);
    free(all);
    if (rc != ORACLE_OK) return rc;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    int started = 0;
    for (int i = 0; i < nthreads; ++i)
        if (pthread_create(&th[i], NULL, bwd_worker, &J) == 0) ++started;
    if (started == 0) bwd_worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    pthread_mutex_destroy(&J.lock);
    return J.status;
}
