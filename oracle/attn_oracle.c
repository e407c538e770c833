/*
 * attn_oracle.c -- TEST INFRASTRUCTURE, not part of the product path.
 *
 * A plain, slow, fp64 CPU statement of what the fused attention forward pass
 * computes.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load this library.  It shares no code, header, table or constant
 * with the CUDA path.
 *
 * Sources (the pages this restates):
 *  - "Fused attention kernel" (wikillm concept card), section Overview: exact
 *    attention is softmax of the score matrix times V; the fused kernel only
 *    reorganises that computation, so the result it must reach is the plain
 *    definition below.
 *  - same card, section Implementation sketch: the outputs are O and the
 *    row log-sum-exp  lse = m + log(l)  (natural log).
 *  - same card, section "8-bit forward pass (FP8, Hopper)": e4m3 format,
 *    one scale per block of Q, K and V, and incoherent processing, i.e. Q and
 *    K multiplied by an orthogonal matrix built from a random sign diagonal
 *    and a Hadamard matrix.
 *
 * Readings where the pages leave a step open (each also listed in the design
 * notes):
 *  - scores are scale * q.k (the sketch omits the scale; the problem statement
 *    carries it); lse is in natural-log units of the scaled scores;
 *  - causal masking is top-left aligned: query i sees keys j <= i of its own
 *    sequence;
 *  - the orthogonal matrix is M = D * H_d / sqrt(d) with H_d the Sylvester
 *    Hadamard matrix, H[i][j] = (-1)^popcount(i & j), and D = diag(signs);
 *  - a block scale is amax(|x|)/448 (448 = largest finite e4m3 value), an
 *    all-zero block takes scale 1, and codes are round-to-nearest-even with
 *    saturation to +-448.
 *
 * Every function returns 0 on success and a negative value on bad arguments.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Exact attention for a list of query rows.                                 */
/* ------------------------------------------------------------------------ */

typedef struct {
    const double *q, *k, *v;
    const double *bias;              /* additive score bias, or NULL */
    int64_t bias_sb, bias_sh, bias_sr;
    const int32_t *cu, *cuk;
    int32_t nseq, H, Hkv, d, causal;
    double scale;
    const int64_t *row_tok;
    const int32_t *row_head;
    int64_t r0, r1;
    double *o, *lse;
    int status;
} rows_job;

/* Sequence index s with cu[s] <= t < cu[s+1], or -1. */
static int32_t seq_of(const int32_t *cu, int32_t nseq, int64_t t)
{
    int32_t lo = 0, hi = nseq - 1;
    if (nseq <= 0 || t < cu[0] || t >= cu[nseq]) return -1;
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) / 2;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

static void *rows_worker(void *arg)
{
    rows_job *jb = (rows_job *)arg;
    const int32_t H = jb->H, Hkv = jb->Hkv, d = jb->d;
    const int64_t tok_stride = (int64_t)H * d;       /* q rows */
    const int64_t kv_stride = (int64_t)Hkv * d;      /* k, v rows */
    int64_t maxlen = 0;
    for (int32_t s = 0; s < jb->nseq; ++s) {
        int64_t L = (int64_t)jb->cuk[s + 1] - jb->cuk[s];
        if (L > maxlen) maxlen = L;
    }
    double *sc = (double *)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
    if (!sc) { jb->status = -2; return NULL; }

    for (int64_t r = jb->r0; r < jb->r1; ++r) {
        const int64_t t = jb->row_tok[r];
        const int32_t h = jb->row_head[r];
        double *orow = jb->o + r * d;
        const int32_t s = seq_of(jb->cu, jb->nseq, t);
        if (s < 0 || h < 0 || h >= H) { jb->status = -1; break; }
        const int64_t i = t - jb->cu[s];             /* position among its queries */
        const int64_t Lq = (int64_t)jb->cu[s + 1] - jb->cu[s];
        const int64_t kstart = jb->cuk[s];
        const int64_t Lk = (int64_t)jb->cuk[s + 1] - kstart;
        /* allowed keys j < nkeys: all of them, or (causal) those at or before
           the query's position when the queries are the last Lq of the Lk
           positions -- j <= i + Lk - Lq, which is j <= i when Lq = Lk */
        int64_t nkeys = jb->causal ? i + 1 + (Lk - Lq) : Lk;
        if (nkeys > Lk) nkeys = Lk;
        if (nkeys < 0) nkeys = 0;
        const int32_t hk = h / (H / Hkv);           /* the K/V head of query head h */

        const double *qrow = jb->q + t * tok_stride + (int64_t)h * d;
        /* scores s_j = scale * sum_c q_c k_jc, and their maximum */
        double mx = -INFINITY;
        for (int64_t j = 0; j < nkeys; ++j) {
            const double *krow = jb->k + (kstart + j) * kv_stride + (int64_t)hk * d;
            double acc = 0.0;
            for (int32_t c = 0; c < d; ++c) acc += qrow[c] * krow[c];
            sc[j] = jb->scale * acc;
            if (jb->bias)
                sc[j] += jb->bias[s * jb->bias_sb + (int64_t)h * jb->bias_sh + i * jb->bias_sr + j];
            if (sc[j] > mx) mx = sc[j];
        }
        if (mx == -INFINITY) {       /* every allowed key biased to -inf: no key */
            for (int32_t c = 0; c < d; ++c) orow[c] = 0.0;
            jb->lse[r] = -INFINITY;
            continue;
        }
        if (nkeys == 0) {            /* no allowed key: O = 0, lse = -inf */
            for (int32_t c = 0; c < d; ++c) orow[c] = 0.0;
            jb->lse[r] = -INFINITY;
            continue;
        }
        /* Z = sum_j exp(s_j - M);  O = sum_j exp(s_j - M) v_j / Z */
        double z = 0.0;
        for (int32_t c = 0; c < d; ++c) orow[c] = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) {
            const double w = exp(sc[j] - mx);
            const double *vrow = jb->v + (kstart + j) * kv_stride + (int64_t)hk * d;
            z += w;
            for (int32_t c = 0; c < d; ++c) orow[c] += w * vrow[c];
        }
        for (int32_t c = 0; c < d; ++c) orow[c] /= z;
        jb->lse[r] = mx + log(z);
    }
    free(sc);
    return NULL;
}

/*
 * O and LSE for the query rows (row_tok[r], row_head[r]), r < nrows, with
 * separate query and key sequences and grouped K/V heads.
 * q: packed [Tq, H, d]; k, v: packed [Tk, Hkv, d] (token-major).  Sequence s
 * holds queries cu_q[s] .. cu_q[s+1]-1 and keys cu_k[s] .. cu_k[s+1]-1.
 * Query head h uses K/V head h / (H / Hkv) (Hkv divides H).  Causal: the
 * queries of a sequence are its last Lq positions, so query i sees keys
 * j <= i + Lk - Lq (top-left j <= i when Lq = Lk); a query with no allowed
 * key gets O = 0, lse = -inf.
 * o: [nrows, d]; lse: [nrows].
 */
static int attention_rows_general(const double *q, const double *k, const double *v,
                                  const double *bias, int64_t bias_sb, int64_t bias_sh,
                                  int64_t bias_sr, const int32_t *cu_q, const int32_t *cu_k,
                                  int32_t nseq, int32_t H, int32_t Hkv, int32_t d, double scale,
                                  int32_t causal, const int64_t *row_tok,
                                  const int32_t *row_head, int64_t nrows, double *o, double *lse,
                                  int32_t nthreads)
{
    if (!q || !k || !v || !cu_q || !cu_k || !row_tok || !row_head || !o || !lse) return -1;
    if (nseq < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || d < 1 || nrows < 0) return -1;
    for (int32_t s = 0; s < nseq; ++s)
        if (cu_q[s + 1] < cu_q[s] || cu_k[s + 1] < cu_k[s]) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > nrows) nthreads = nrows > 0 ? (int32_t)nrows : 1;

    rows_job jobs[256];
    pthread_t th[256];
    for (int32_t w = 0; w < nthreads; ++w) {
        rows_job *jb = &jobs[w];
        jb->q = q; jb->k = k; jb->v = v; jb->cu = cu_q; jb->cuk = cu_k; jb->nseq = nseq;
        jb->bias = bias; jb->bias_sb = bias_sb; jb->bias_sh = bias_sh; jb->bias_sr = bias_sr;
        jb->H = H; jb->Hkv = Hkv; jb->d = d; jb->causal = causal; jb->scale = scale;
        jb->row_tok = row_tok; jb->row_head = row_head;
        jb->r0 = nrows * w / nthreads; jb->r1 = nrows * (w + 1) / nthreads;
        jb->o = o; jb->lse = lse; jb->status = 0;
    }
    for (int32_t w = 1; w < nthreads; ++w)
        if (pthread_create(&th[w], NULL, rows_worker, &jobs[w]) != 0)
            jobs[w].status = -3;                   /* not started: run it inline below */
    rows_worker(&jobs[0]);
    int status = jobs[0].status;
    for (int32_t w = 1; w < nthreads; ++w) {
        if (jobs[w].status == -3) { jobs[w].status = 0; rows_worker(&jobs[w]); }
        else pthread_join(th[w], NULL);
        if (jobs[w].status < 0) status = jobs[w].status;
    }
    return status;
}

int oracle_attention_rows_gqa(const double *q, const double *k, const double *v,
                              const int32_t *cu_q, const int32_t *cu_k, int32_t nseq,
                              int32_t H, int32_t Hkv, int32_t d, double scale, int32_t causal,
                              const int64_t *row_tok, const int32_t *row_head, int64_t nrows,
                              double *o, double *lse, int32_t nthreads)
{
    return attention_rows_general(q, k, v, NULL, 0, 0, 0, cu_q, cu_k, nseq, H, Hkv, d, scale,
                                  causal, row_tok, row_head, nrows, o, lse, nthreads);
}

/*
 * As oracle_attention_rows_gqa with an additive bias on the scores:
 * s_ij = scale * q_i . k_j + bias[s * sb + h * sh + i * sr + j], s the
 * sequence, i and j the query and key positions in it (strides in
 * elements; 0 broadcasts).  A bias of -inf removes a key; a row whose every
 * allowed key is removed gets O = 0, lse = -inf.
 */
int oracle_attention_rows_bias(const double *q, const double *k, const double *v,
                               const double *bias, int64_t bias_sb, int64_t bias_sh,
                               int64_t bias_sr, const int32_t *cu_q, const int32_t *cu_k,
                               int32_t nseq, int32_t H, int32_t Hkv, int32_t d, double scale,
                               int32_t causal, const int64_t *row_tok, const int32_t *row_head,
                               int64_t nrows, double *o, double *lse, int32_t nthreads)
{
    if (!bias) return -1;
    return attention_rows_general(q, k, v, bias, bias_sb, bias_sh, bias_sr, cu_q, cu_k, nseq, H,
                                  Hkv, d, scale, causal, row_tok, row_head, nrows, o, lse,
                                  nthreads);
}

/*
 * O and LSE for the query rows (row_tok[r], row_head[r]), r < nrows.
 * q, k, v: packed [T, H, d] (token-major); sequence s holds tokens
 * cu_seqlens[s] .. cu_seqlens[s+1]-1 (as queries and as keys).  A dense
 * [B, N, H, d] batch is the same bytes with cu_seqlens = 0, N, 2N, ...
 * o: [nrows, d]; lse: [nrows].
 */
int oracle_attention_rows(const double *q, const double *k, const double *v,
                          const int32_t *cu_seqlens, int32_t nseq,
                          int32_t H, int32_t d, double scale, int32_t causal,
                          const int64_t *row_tok, const int32_t *row_head, int64_t nrows,
                          double *o, double *lse, int32_t nthreads)
{
    return oracle_attention_rows_gqa(q, k, v, cu_seqlens, cu_seqlens, nseq, H, H, d, scale,
                                     causal, row_tok, row_head, nrows, o, lse, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Backward pass: gradients of O with respect to Q, K and V.                  */
/* ------------------------------------------------------------------------ */
/*
 * For one sequence and head, with S = scale * Q K^T over the allowed keys and
 * P = softmax(S) row by row (the forward definition above), O = P V and an
 * upstream gradient dO:
 *   dV = P^T dO,   dP = dO V^T,   dS = P * (dP - rowsum(dO * O)),
 *   dQ = scale * dS K,   dK = scale * dS^T Q
 * (rowsum(dO * O) = sum_j P_ij dP_ij, the softmax Jacobian's diagonal term).
 * Grouped K/V heads: dK and dV of a K/V head sum over its query heads.
 */
typedef struct {
    const double *q, *k, *v, *dout;
    const int32_t *cu;
    int32_t nseq, H, Hkv, d, causal;
    double scale;
    int64_t u0, u1;                 /* (sequence, K/V head) units */
    double *dq, *dk, *dv;
    int status;
} bwd_job;

static void *bwd_worker(void *arg)
{
    bwd_job *jb = (bwd_job *)arg;
    const int32_t H = jb->H, Hkv = jb->Hkv, d = jb->d, g = H / Hkv;
    const int64_t qs = (int64_t)H * d, ks = (int64_t)Hkv * d;
    int64_t maxlen = 0;
    for (int32_t s = 0; s < jb->nseq; ++s) {
        int64_t L = (int64_t)jb->cu[s + 1] - jb->cu[s];
        if (L > maxlen) maxlen = L;
    }
    const size_t LL = (size_t)(maxlen > 0 ? maxlen : 1);
    double *P = (double *)malloc(sizeof(double) * LL * LL);
    double *dP = (double *)malloc(sizeof(double) * LL * LL);
    double *orow = (double *)malloc(sizeof(double) * (size_t)d);
    if (!P || !dP || !orow) { free(P); free(dP); free(orow); jb->status = -2; return NULL; }
    for (int64_t u = jb->u0; u < jb->u1; ++u) {
        const int32_t s = (int32_t)(u / Hkv), hk = (int32_t)(u % Hkv);
        const int64_t st = jb->cu[s], L = (int64_t)jb->cu[s + 1] - st;
        for (int32_t gh = 0; gh < g; ++gh) {
            const int32_t h = hk * g + gh;
            for (int64_t i = 0; i < L; ++i) {
                const double *qi = jb->q + (st + i) * qs + (int64_t)h * d;
                const double *doi = jb->dout + (st + i) * qs + (int64_t)h * d;
                const int64_t nk = jb->causal ? i + 1 : L;
                double mx = -INFINITY;
                for (int64_t j = 0; j < nk; ++j) {
                    const double *kj = jb->k + (st + j) * ks + (int64_t)hk * d;
                    double acc = 0.0;
                    for (int32_t c = 0; c < d; ++c) acc += qi[c] * kj[c];
                    P[i * L + j] = jb->scale * acc;
                    if (P[i * L + j] > mx) mx = P[i * L + j];
                }
                double z = 0.0;
                for (int64_t j = 0; j < nk; ++j) { P[i * L + j] = exp(P[i * L + j] - mx); z += P[i * L + j]; }
                for (int64_t j = 0; j < nk; ++j) P[i * L + j] /= z;
                for (int64_t j = nk; j < L; ++j) P[i * L + j] = 0.0;
                /* O_i = sum_j P_ij v_j;  dP_ij = dO_i . v_j;  D_i = dO_i . O_i */
                for (int32_t c = 0; c < d; ++c) orow[c] = 0.0;
                for (int64_t j = 0; j < nk; ++j) {
                    const double *vj = jb->v + (st + j) * ks + (int64_t)hk * d;
                    double acc = 0.0;
                    for (int32_t c = 0; c < d; ++c) { orow[c] += P[i * L + j] * vj[c]; acc += doi[c] * vj[c]; }
                    dP[i * L + j] = acc;
                }
                double Di = 0.0;
                for (int32_t c = 0; c < d; ++c) Di += doi[c] * orow[c];
                /* dS_ij = P_ij (dP_ij - D_i), kept in dP */
                for (int64_t j = 0; j < nk; ++j) dP[i * L + j] = P[i * L + j] * (dP[i * L + j] - Di);
                for (int64_t j = nk; j < L; ++j) dP[i * L + j] = 0.0;
                /* dQ_i = scale * sum_j dS_ij k_j */
                double *dqi = jb->dq + (st + i) * qs + (int64_t)h * d;
                for (int32_t c = 0; c < d; ++c) dqi[c] = 0.0;
                for (int64_t j = 0; j < nk; ++j) {
                    const double *kj = jb->k + (st + j) * ks + (int64_t)hk * d;
                    for (int32_t c = 0; c < d; ++c) dqi[c] += jb->scale * dP[i * L + j] * kj[c];
                }
            }
            /* dV_j += sum_i P_ij dO_i;  dK_j += scale * sum_i dS_ij q_i */
            for (int64_t j = 0; j < L; ++j) {
                double *dvj = jb->dv + (st + j) * ks + (int64_t)hk * d;
                double *dkj = jb->dk + (st + j) * ks + (int64_t)hk * d;
                for (int64_t i = 0; i < L; ++i) {
                    const double pij = P[i * L + j], dsij = dP[i * L + j];
                    if (pij == 0.0 && dsij == 0.0) continue;
                    const double *doi = jb->dout + (st + i) * qs + (int64_t)h * d;
                    const double *qi = jb->q + (st + i) * qs + (int64_t)h * d;
                    for (int32_t c = 0; c < d; ++c) {
                        dvj[c] += pij * doi[c];
                        dkj[c] += jb->scale * dsij * qi[c];
                    }
                }
            }
        }
    }
    free(P); free(dP); free(orow);
    return NULL;
}

/*
 * Gradients for packed sequences: q, dout, dq [T, H, d]; k, v, dk, dv
 * [T, Hkv, d]; sequence s holds tokens cu_seqlens[s] .. cu_seqlens[s+1]-1.
 * dk and dv are zeroed here and accumulated over each group's query heads.
 */
int oracle_attention_backward(const double *q, const double *k, const double *v,
                              const double *dout, const int32_t *cu_seqlens, int32_t nseq,
                              int32_t H, int32_t Hkv, int32_t d, double scale, int32_t causal,
                              double *dq, double *dk, double *dv, int32_t nthreads)
{
    if (!q || !k || !v || !dout || !cu_seqlens || !dq || !dk || !dv) return -1;
    if (nseq < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || d < 1) return -1;
    for (int32_t s = 0; s < nseq; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;
    const int64_t T = cu_seqlens[nseq];
    memset(dk, 0, sizeof(double) * (size_t)T * Hkv * d);
    memset(dv, 0, sizeof(double) * (size_t)T * Hkv * d);
    const int64_t units = (int64_t)nseq * Hkv;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > units) nthreads = (int32_t)units;
    bwd_job jobs[256];
    pthread_t th[256];
    for (int32_t w = 0; w < nthreads; ++w) {
        bwd_job *jb = &jobs[w];
        jb->q = q; jb->k = k; jb->v = v; jb->dout = dout; jb->cu = cu_seqlens; jb->nseq = nseq;
        jb->H = H; jb->Hkv = Hkv; jb->d = d; jb->causal = causal; jb->scale = scale;
        jb->u0 = units * w / nthreads; jb->u1 = units * (w + 1) / nthreads;
        jb->dq = dq; jb->dk = dk; jb->dv = dv; jb->status = 0;
    }
    for (int32_t w = 1; w < nthreads; ++w)
        if (pthread_create(&th[w], NULL, bwd_worker, &jobs[w]) != 0) jobs[w].status = -3;
    bwd_worker(&jobs[0]);
    int status = jobs[0].status;
    for (int32_t w = 1; w < nthreads; ++w) {
        if (jobs[w].status == -3) { jobs[w].status = 0; bwd_worker(&jobs[w]); }
        else pthread_join(th[w], NULL);
        if (jobs[w].status < 0) status = jobs[w].status;
    }
    return status;
}

/*
 * Selected rows of the same gradients for ONE sequence and ONE K/V head, at
 * any length: q, dout [L, H, d]; k, v [L, Hkv, d] (one sequence's tokens).
 * For each query head h of K/V head hk's group (g = H / Hkv heads):
 *   lse_i and O_i over all queries i (the forward, as above), D_i = dO_i . O_i,
 *   dQ rows:  dq_rows[h - hk g][r] = scale sum_j P_ij (dO_i . v_j - D_i) k_j,
 *             i = qrows[r];
 * and over the group, for j = krows[r]:
 *   dv_rows[r] = sum_h sum_i P_ij dO_i,
 *   dk_rows[r] = sum_h sum_i scale P_ij (dO_i . v_j - D_i) q_i.
 * The first pass (lse, O, D of every query) runs on nthreads threads over
 * query rows; the selected rows are then summed directly.
 * dq_rows: [g, nq, d]; dk_rows, dv_rows: [nk, d].
 */
typedef struct {
    const double *q, *k, *v, *dout;
    int64_t L, i0, i1;
    int32_t H, Hkv, d, h, hk, causal;
    double scale;
    double *lse, *D;
} grad_rows_job;

static void *grad_rows_worker(void *arg)
{
    grad_rows_job *jb = (grad_rows_job *)arg;
    const int32_t d = jb->d;
    const int64_t qs = (int64_t)jb->H * d, ks = (int64_t)jb->Hkv * d;
    double *s = (double *)malloc(sizeof(double) * (size_t)(jb->L > 0 ? jb->L : 1));
    double *orow = (double *)malloc(sizeof(double) * (size_t)d);
    if (!s || !orow) { free(s); free(orow); return (void *)1; }
    for (int64_t i = jb->i0; i < jb->i1; ++i) {
        const double *qi = jb->q + i * qs + (int64_t)jb->h * d;
        const double *doi = jb->dout + i * qs + (int64_t)jb->h * d;
        const int64_t nk = jb->causal ? i + 1 : jb->L;
        double mx = -INFINITY;
        for (int64_t j = 0; j < nk; ++j) {
            const double *kj = jb->k + j * ks + (int64_t)jb->hk * d;
            double acc = 0.0;
            for (int32_t c = 0; c < d; ++c) acc += qi[c] * kj[c];
            s[j] = jb->scale * acc;
            if (s[j] > mx) mx = s[j];
        }
        double z = 0.0;
        for (int64_t j = 0; j < nk; ++j) { s[j] = exp(s[j] - mx); z += s[j]; }
        for (int32_t c = 0; c < d; ++c) orow[c] = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
            const double *vj = jb->v + j * ks + (int64_t)jb->hk * d;
            for (int32_t c = 0; c < d; ++c) orow[c] += (s[j] / z) * vj[c];
        }
        double Di = 0.0;
        for (int32_t c = 0; c < d; ++c) Di += doi[c] * orow[c];
        jb->lse[i] = mx + log(z);
        jb->D[i] = Di;
    }
    free(s); free(orow);
    return NULL;
}

int oracle_attention_backward_rows(const double *q, const double *k, const double *v,
                                   const double *dout, int64_t L, int32_t H, int32_t Hkv,
                                   int32_t d, double scale, int32_t causal, int32_t hk,
                                   const int64_t *qrows, int32_t nq, const int64_t *krows,
                                   int32_t nk, double *dq_rows, double *dk_rows,
                                   double *dv_rows, int32_t nthreads)
{
    if (!q || !k || !v || !dout || L < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || d < 1) return -1;
    if (hk < 0 || hk >= Hkv || nq < 0 || nk < 0) return -1;
    if ((nq > 0 && (!qrows || !dq_rows)) || (nk > 0 && (!krows || !dk_rows || !dv_rows))) return -1;
    for (int32_t r = 0; r < nq; ++r) if (qrows[r] < 0 || qrows[r] >= L) return -1;
    for (int32_t r = 0; r < nk; ++r) if (krows[r] < 0 || krows[r] >= L) return -1;
    const int32_t g = H / Hkv;
    const int64_t qs = (int64_t)H * d, ks = (int64_t)Hkv * d;
    double *lse = (double *)malloc(sizeof(double) * (size_t)L);
    double *D = (double *)malloc(sizeof(double) * (size_t)L);
    if (!lse || !D) { free(lse); free(D); return -2; }
    if (nk > 0) {
        memset(dk_rows, 0, sizeof(double) * (size_t)nk * d);
        memset(dv_rows, 0, sizeof(double) * (size_t)nk * d);
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > L) nthreads = (int32_t)L;
    int status = 0;
    for (int32_t gh = 0; gh < g && status == 0; ++gh) {
        const int32_t h = hk * g + gh;
        grad_rows_job jobs[256];
        pthread_t th[256];
        int started[256] = {0};
        for (int32_t w = 0; w < nthreads; ++w) {
            grad_rows_job *jb = &jobs[w];
            jb->q = q; jb->k = k; jb->v = v; jb->dout = dout; jb->L = L;
            jb->i0 = L * w / nthreads; jb->i1 = L * (w + 1) / nthreads;
            jb->H = H; jb->Hkv = Hkv; jb->d = d; jb->h = h; jb->hk = hk; jb->causal = causal;
            jb->scale = scale; jb->lse = lse; jb->D = D;
        }
        for (int32_t w = 1; w < nthreads; ++w)
            started[w] = pthread_create(&th[w], NULL, grad_rows_worker, &jobs[w]) == 0;
        if (grad_rows_worker(&jobs[0]) != NULL) status = -2;
        for (int32_t w = 1; w < nthreads; ++w) {
            void *ret = NULL;
            if (started[w]) pthread_join(th[w], &ret);
            else ret = grad_rows_worker(&jobs[w]);
            if (ret != NULL) status = -2;
        }
        if (status != 0) break;
        /* dQ rows of head h */
        for (int32_t r = 0; r < nq; ++r) {
            const int64_t i = qrows[r];
            const double *qi = q + i * qs + (int64_t)h * d;
            const double *doi = dout + i * qs + (int64_t)h * d;
            double *out = dq_rows + ((int64_t)gh * nq + r) * d;
            for (int32_t c = 0; c < d; ++c) out[c] = 0.0;
            const int64_t nkeys = causal ? i + 1 : L;
            for (int64_t j = 0; j < nkeys; ++j) {
                const double *kj = k + j * ks + (int64_t)hk * d;
                const double *vj = v + j * ks + (int64_t)hk * d;
                double sij = 0.0, dpij = 0.0;
                for (int32_t c = 0; c < d; ++c) { sij += qi[c] * kj[c]; dpij += doi[c] * vj[c]; }
                const double pij = exp(scale * sij - lse[i]);
                const double dsij = pij * (dpij - D[i]);
                for (int32_t c = 0; c < d; ++c) out[c] += scale * dsij * kj[c];
            }
        }
        /* dK, dV rows, this head's share */
        for (int32_t r = 0; r < nk; ++r) {
            const int64_t j = krows[r];
            const double *kj = k + j * ks + (int64_t)hk * d;
            const double *vj = v + j * ks + (int64_t)hk * d;
            for (int64_t i = causal ? j : 0; i < L; ++i) {
                const double *qi = q + i * qs + (int64_t)h * d;
                const double *doi = dout + i * qs + (int64_t)h * d;
                double sij = 0.0, dpij = 0.0;
                for (int32_t c = 0; c < d; ++c) { sij += qi[c] * kj[c]; dpij += doi[c] * vj[c]; }
                const double pij = exp(scale * sij - lse[i]);
                const double dsij = pij * (dpij - D[i]);
                for (int32_t c = 0; c < d; ++c) {
                    dv_rows[(int64_t)r * d + c] += pij * doi[c];
                    dk_rows[(int64_t)r * d + c] += scale * dsij * qi[c];
                }
            }
        }
    }
    free(lse); free(D);
    return status;
}

/*
 * Merge of partial results over disjoint key sets of the same query rows
 * (the combine step of attention split over key ranges): with lse_s and
 * O_s the results over part s,
 *   lse = log sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) O_s.
 * A part with no keys (lse_s = -inf) contributes nothing.
 * o_parts: [nparts, nrows, d]; lse_parts: [nparts, nrows]; o: [nrows, d];
 * lse: [nrows].
 */
int oracle_merge_partials(const double *o_parts, const double *lse_parts, int32_t nparts,
                          int64_t nrows, int32_t d, double *o, double *lse)
{
    if (!o_parts || !lse_parts || !o || !lse || nparts < 1 || nrows < 0 || d < 1) return -1;
    for (int64_t r = 0; r < nrows; ++r) {
        double mx = -INFINITY;
        for (int32_t s = 0; s < nparts; ++s)
            if (lse_parts[(int64_t)s * nrows + r] > mx) mx = lse_parts[(int64_t)s * nrows + r];
        double *orow = o + r * d;
        for (int32_t c = 0; c < d; ++c) orow[c] = 0.0;
        if (mx == -INFINITY) { lse[r] = -INFINITY; continue; }
        double z = 0.0;
        for (int32_t s = 0; s < nparts; ++s) {
            const double w = exp(lse_parts[(int64_t)s * nrows + r] - mx);
            const double *op = o_parts + ((int64_t)s * nrows + r) * d;
            z += w;
            for (int32_t c = 0; c < d; ++c) orow[c] += w * op[c];
        }
        for (int32_t c = 0; c < d; ++c) orow[c] /= z;
        lse[r] = mx + log(z);
    }
    return 0;
}

/*
 * Probability matrix of one sequence, for small checks: P[h][i][j] =
 * exp(s_ij - M_i) / Z_i over the allowed keys, 0 elsewhere.
 * q, k: [N, H, d]; p: [H, N, N].
 */
int oracle_attention_probs(const double *q, const double *k, int32_t N, int32_t H, int32_t d,
                           double scale, int32_t causal, double *p)
{
    if (!q || !k || !p || N < 1 || H < 1 || d < 1) return -1;
    const int64_t ts = (int64_t)H * d;
    for (int32_t h = 0; h < H; ++h) {
        for (int32_t i = 0; i < N; ++i) {
            double *prow = p + ((int64_t)h * N + i) * N;
            const int32_t nk = causal ? i + 1 : N;
            double mx = -INFINITY;
            for (int32_t j = 0; j < N; ++j) prow[j] = 0.0;
            for (int32_t j = 0; j < nk; ++j) {
                double acc = 0.0;
                for (int32_t c = 0; c < d; ++c)
                    acc += q[i * ts + (int64_t)h * d + c] * k[j * ts + (int64_t)h * d + c];
                prow[j] = scale * acc;
                if (prow[j] > mx) mx = prow[j];
            }
            double z = 0.0;
            for (int32_t j = 0; j < nk; ++j) { prow[j] = exp(prow[j] - mx); z += prow[j]; }
            for (int32_t j = 0; j < nk; ++j) prow[j] /= z;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Incoherent processing: random-sign diagonal times Hadamard matrix.        */
/* ------------------------------------------------------------------------ */

static int is_pow2(int32_t d) { return d > 0 && (d & (d - 1)) == 0; }

static int popcount32(uint32_t x)
{
    int n = 0;
    while (x) { n += (int)(x & 1u); x >>= 1; }
    return n;
}

/* Sylvester Hadamard matrix H_d (entries +-1), row-major d x d. */
int oracle_hadamard_matrix(int32_t d, double *hm)
{
    if (!hm || !is_pow2(d)) return -1;
    for (int32_t i = 0; i < d; ++i)
        for (int32_t j = 0; j < d; ++j)
            hm[(int64_t)i * d + j] = (popcount32((uint32_t)(i & j)) & 1) ? -1.0 : 1.0;
    return 0;
}

/*
 * out_row = x_row * M with M = diag(signs) * H_d / sqrt(d), i.e.
 * out[j] = sum_i x[i] * signs[i] * H[i][j] / sqrt(d), for every row of a
 * row-major [nrows, d] array.  signs == NULL means D = I.
 */
int oracle_rotate(const double *x, int64_t nrows, int32_t d, const int8_t *signs, double *out)
{
    if (!x || !out || nrows < 0 || !is_pow2(d)) return -1;
    double *hm = (double *)malloc(sizeof(double) * (size_t)d * (size_t)d);
    double *tmp = (double *)malloc(sizeof(double) * (size_t)d);
    if (!hm || !tmp) { free(hm); free(tmp); return -2; }
    oracle_hadamard_matrix(d, hm);
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    for (int64_t r = 0; r < nrows; ++r) {
        const double *xr = x + r * d;
        for (int32_t i = 0; i < d; ++i) tmp[i] = xr[i] * (signs ? (double)signs[i] : 1.0);
        for (int32_t j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int32_t i = 0; i < d; ++i) acc += tmp[i] * hm[(int64_t)i * d + j];
            out[r * d + j] = acc * inv_sqrt_d;
        }
    }
    free(hm);
    free(tmp);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* e4m3 (OCP 8-bit floating point, E4M3 "FN": bias 7, no infinities,         */
/* S.1111.111 is NaN, largest finite 448).                                   */
/* ------------------------------------------------------------------------ */

double oracle_e4m3_decode(uint8_t c)
{
    const int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m, -9);                 /* m/8 * 2^(1-7) */
    else mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Nearest e4m3 value, ties to the even code, saturating to +-448. */
uint8_t oracle_e4m3_encode(double x)
{
    if (isnan(x)) return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs(x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    /* codes 0..126 are the non-negative finite values in increasing order:
       find the largest code whose value does not exceed a. */
    int lo = 0, hi = 126;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (oracle_e4m3_decode((uint8_t)mid) <= a) lo = mid; else hi = mid - 1;
    }
    int c = lo;
    const double below = oracle_e4m3_decode((uint8_t)c);
    if (below != a) {
        const double above = oracle_e4m3_decode((uint8_t)(c + 1));
        const double dlo = a - below, dhi = above - a;
        if (dhi < dlo || (dhi == dlo && (c & 1))) c = c + 1;
    }
    return (uint8_t)(sign | c);
}

int oracle_e4m3_encode_array(const double *x, int64_t n, uint8_t *out)
{
    if (!x || !out || n < 0) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
    return 0;
}

int oracle_e4m3_decode_array(const uint8_t *c, int64_t n, double *out)
{
    if (!c || !out || n < 0) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
    return 0;
}

/*
 * Block quantisation of x [B, N, H, d] (already rotated for Q and K).
 * Blocks are `block` consecutive tokens of one (b, h) over all d channels
 * (the last block of a sequence may be partial); with per_tensor != 0 a
 * single scale covers the whole tensor.  scale = amax(|x|)/448 (1 when the
 * block is all zero); codes[i] = e4m3(x[i] / scale); descale[b][h][blk] =
 * scale, so x ~ decode(code) * descale.
 */
int oracle_block_quant(const double *x, int32_t B, int32_t N, int32_t H, int32_t d,
                       int32_t block, int32_t per_tensor, uint8_t *codes, double *descale)
{
    if (!x || !codes || !descale || B < 1 || N < 1 || H < 1 || d < 1 || block < 1) return -1;
    const int32_t nblk = (N + block - 1) / block;
    const int64_t ts = (int64_t)H * d;
    double tensor_amax = 0.0;
    if (per_tensor) {
        const int64_t n = (int64_t)B * N * H * d;
        for (int64_t i = 0; i < n; ++i) if (fabs(x[i]) > tensor_amax) tensor_amax = fabs(x[i]);
    }
    for (int32_t b = 0; b < B; ++b)
        for (int32_t h = 0; h < H; ++h)
            for (int32_t blk = 0; blk < nblk; ++blk) {
                const int32_t t0 = blk * block;
                const int32_t t1 = (t0 + block < N) ? t0 + block : N;
                double amax = tensor_amax;
                if (!per_tensor) {
                    amax = 0.0;
                    for (int32_t t = t0; t < t1; ++t)
                        for (int32_t c = 0; c < d; ++c) {
                            const double a = fabs(x[((int64_t)b * N + t) * ts + (int64_t)h * d + c]);
                            if (a > amax) amax = a;
                        }
                }
                const double scale = amax > 0.0 ? amax / 448.0 : 1.0;
                descale[((int64_t)b * H + h) * nblk + blk] = scale;
                for (int32_t t = t0; t < t1; ++t)
                    for (int32_t c = 0; c < d; ++c) {
                        const int64_t i = ((int64_t)b * N + t) * ts + (int64_t)h * d + c;
                        codes[i] = oracle_e4m3_encode(x[i] / scale);
                    }
            }
    return 0;
}
