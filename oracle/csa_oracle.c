/*
 * csa_oracle.c -- the oracle: a plain, slow, float64 CPU restatement of the CSA
 * Lightning-Indexer training step.
 *
 * TEST INFRASTRUCTURE ONLY.  The GPU library never includes, links, loads or calls
 * anything in this directory; only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no header, helper, table or
 * constant with the CUDA path: its parameter block below is its own.
 *
 * Sources (web pages; cited by title and section):
 *   [BUG]  "[Bug] DSV4 unfused CSA indexer loss uses a compressed-only teacher instead
 *          of the full CSA attention distribution" (Megatron-LM issue #5776), incl.
 *          its code excerpts and the follow-up comments (the proposal and review).
 *   [PR]   "Megatron-LM PR #8539" (cuDNN frontend 1.26 default changes).
 *
 * Every number is float64.  Inputs arrive as float64 copies of the exact values the
 * GPU reads (bf16 or fp32 widened exactly).  No blocking, fusion or reordering beyond
 * the definitions: each step is written out as the pages state it.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - indexer score I[t,s] = sum_j w[t,j] * max(0, q_idx[t,j] . k_idx[s]); the indexer
 *     softmax scale is already folded into w ([BUG] sec. 1 excerpt, weights_for_unfused);
 *   - output slot order of the selection: ascending key id, -1 pads last;
 *   - the window is the W original positions ending at (and including) the query,
 *     truncated at the start of the segment;
 *   - the sink enters Z_h as exp(a_h), unscaled.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int layout;                 /* 0 SBHD [S,B,...], 1 BSHD [B,S,...], 2 THD [T,...] */
    int batch;                  /* SBHD/BSHD: sequences B.  THD: number of segments */
    int seqlen;                 /* SBHD/BSHD: sequence length S.  THD: physical rows T */
    const int32_t *cu_q;        /* THD: [nseg+1] physical segment offsets */
    const int32_t *cu_q_real;   /* THD: [nseg+1] unpadded offsets, or NULL (= cu_q) */
    int max_seqlen;             /* THD: longest unpadded segment (sets the dense key width) */
    int ratio, window, topk;
    int heads, head_dim, idx_heads, idx_dim;
    double scale;               /* main-attention softmax scale sigma */
    int sparse;                 /* 1: C = selected keys.  0: C = every visible key */
    int reduction;              /* 0: mean over physical rows.  1: sum */
    double coeff;
} orc_params;

#define ORC_EPS 1e-10           /* [BUG] sec. 2 excerpt: clamp(min=1e-10) and log(x + 1e-10) */

/* ---------------------------------------------------------------- geometry */

typedef struct {
    int b;          /* segment / sequence */
    int s;          /* 0-based position in the segment; 1-based position i = s + 1 */
    int len;        /* real (unpadded) length of the segment */
    int pad;        /* 1 if the row is padding ([BUG] fused-path excerpt, padding_row_mask) */
    int v;          /* visible compressed keys: j visible iff j < i // ratio ([BUG] sec. 1 excerpt) */
    long c_base;    /* THD: first compressed row of the segment, packed by real length // ratio */
} orc_row;

static int orc_ncomp(const orc_params *P) { return P->seqlen / P->ratio; }

/* Width of the dense key axis: n_c (SBHD/BSHD) or the longest segment's n_c (THD). */
int orc_key_width(const orc_params *P)
{
    return P->layout == 2 ? P->max_seqlen / P->ratio : orc_ncomp(P);
}

/* K = min(topk, n_c) ([BUG] sec. 1 excerpts: min(index_topk, n_compressed) / max_seqlen_compressed). */
int orc_topk_width(const orc_params *P)
{
    int nc = orc_key_width(P);
    return P->topk < nc ? P->topk : nc;
}

int orc_rows(const orc_params *P)
{
    return P->layout == 2 ? P->seqlen : P->batch * P->seqlen;
}

static long orc_thd_cbase(const orc_params *P, int b)
{
    const int32_t *cr = P->cu_q_real ? P->cu_q_real : P->cu_q;
    long base = 0;
    for (int i = 0; i < b; i++) base += (cr[i + 1] - cr[i]) / P->ratio;
    return base;
}

static orc_row orc_decode(const orc_params *P, long r)
{
    orc_row R;
    memset(&R, 0, sizeof R);
    if (P->layout == 0) {               /* SBHD: row = s * B + b */
        R.s = (int)(r / P->batch);
        R.b = (int)(r % P->batch);
        R.len = P->seqlen;
    } else if (P->layout == 1) {        /* BSHD: row = b * S + s */
        R.b = (int)(r / P->seqlen);
        R.s = (int)(r % P->seqlen);
        R.len = P->seqlen;
    } else {                            /* THD: rows packed by cu_q */
        int b = 0;
        while (b + 1 < P->batch && P->cu_q[b + 1] <= r) b++;
        R.b = b;
        R.s = (int)(r - P->cu_q[b]);
        const int32_t *cr = P->cu_q_real ? P->cu_q_real : P->cu_q;
        R.len = cr[b + 1] - cr[b];
        R.c_base = orc_thd_cbase(P, b);
    }
    R.pad = R.s >= R.len;
    R.v = R.pad ? 0 : (R.s + 1) / P->ratio;
    return R;
}

/* memory row of original position p of the row's segment (query, kv) */
static long orc_qrow(const orc_params *P, const orc_row *R, int p)
{
    if (P->layout == 0) return (long)p * P->batch + R->b;
    if (P->layout == 1) return (long)R->b * P->seqlen + p;
    return (long)P->cu_q[R->b] + p;
}

/* global id of compressed key j of the row's segment: b * n_c + j, or the packed THD offset
 * ([PR] item 1: global ids b * S_k + local; [BUG] fused-path excerpt, local_to_global_flat) */
static long orc_gid(const orc_params *P, const orc_row *R, int j)
{
    if (P->layout == 2) return R->c_base + j;
    return (long)R->b * orc_ncomp(P) + j;
}

/* memory row of the compressed key with global id g */
static long orc_crow(const orc_params *P, long g)
{
    if (P->layout == 0) {
        long nc = orc_ncomp(P);
        return (g % nc) * P->batch + g / nc;
    }
    return g;
}

static double orc_dot(const double *a, const double *b, int n)
{
    double s = 0.0;
    for (int i = 0; i < n; i++) s += a[i] * b[i];
    return s;
}

/* ---------------------------------------------------------------- step 1: scores */

/* I[t,s] for one row and compressed key with global id g; r indexes the row's q_idx and w. */
static double orc_score(const orc_params *P, const double *q_idx, const double *w, const double *k_idx,
                        long r, long g)
{
    const int HI = P->idx_heads, DI = P->idx_dim;
    const double *kk = k_idx + orc_crow(P, g) * DI;
    double I = 0.0;
    for (int j = 0; j < HI; j++) {
        double x = orc_dot(q_idx + (r * HI + j) * DI, kk, DI);
        I += w[r * HI + j] * (x > 0.0 ? x : 0.0);
    }
    return I;
}

/* Row-dependent inputs (q_idx, w, q) hold either every row (compact = 0, indexed by memory row) or
 * only the listed rows in list order (compact = 1).  This is storage only; the arithmetic is the same. */
#define ORC_SRC(i, r) (compact ? (long)(i) : (long)(r))

/* Dense indexer scores of the listed rows: out[i][j] = I[row_i, j] for visible local keys j,
 * -inf elsewhere.  out is [nrows][orc_key_width]. */
void orc_scores(const orc_params *P, const double *q_idx, const double *w, const double *k_idx,
                const int32_t *rows, int nrows, int compact, double *out)
{
    const int NC = orc_key_width(P);
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nrows; i++) {
        orc_row R = orc_decode(P, rows[i]);
        for (int j = 0; j < NC; j++)
            out[(long)i * NC + j] = j < R.v ? orc_score(P, q_idx, w, k_idx, ORC_SRC(i, rows[i]), orc_gid(P, &R, j))
                                            : -INFINITY;
    }
}

/* ---------------------------------------------------------------- step 2: top-k */

typedef struct { double score; int j; } orc_cand;

static int orc_by_score(const void *a, const void *b)
{
    const orc_cand *x = a, *y = b;
    if (x->score > y->score) return -1;          /* larger score first */
    if (x->score < y->score) return 1;
    return x->j - y->j;                           /* equal scores: lower index first */
}

static int orc_by_index(const void *a, const void *b)
{
    return ((const orc_cand *)a)->j - ((const orc_cand *)b)->j;
}

/* Top-k selection from given scores (float64, or float32 widened exactly).
 * Row i keeps the k_t = min(K, v) keys with the largest score among its v visible keys, ties to
 * the lower index; slots hold their global ids in ascending order, then -1 pads
 * ([BUG] sec. 3 excerpt: valid = topk < positions // ratio, else -1).  ids is [nrows][K]. */
void orc_topk(const orc_params *P, const double *scores, const int32_t *rows, int nrows, int32_t *ids)
{
    const int NC = orc_key_width(P), K = orc_topk_width(P);
#pragma omp parallel for schedule(dynamic, 4)
    for (int i = 0; i < nrows; i++) {
        orc_row R = orc_decode(P, rows[i]);
        int32_t *out = ids + (long)i * K;
        for (int k = 0; k < K; k++) out[k] = -1;
        if (R.v == 0) continue;
        orc_cand *c = malloc(sizeof(orc_cand) * (size_t)R.v);
        for (int j = 0; j < R.v; j++) {
            c[j].score = scores[(long)i * NC + j];
            c[j].j = j;
        }
        qsort(c, (size_t)R.v, sizeof(orc_cand), orc_by_score);
        int kt = R.v < K ? R.v : K;
        qsort(c, (size_t)kt, sizeof(orc_cand), orc_by_index);
        for (int k = 0; k < kt; k++) out[k] = (int32_t)orc_gid(P, &R, c[k].j);
        free(c);
    }
}

/* The support C of a row, as (slot, global id) pairs.  Sparse: the selected, valid ids of the row
 * (the slots of ids); dense: every visible key, slot = local index.  Returns |C|. */
static int orc_support(const orc_params *P, const orc_row *R, const int32_t *row_ids, int *slot, long *gid)
{
    int n = 0;
    if (P->sparse) {
        const int K = orc_topk_width(P);
        for (int k = 0; k < K; k++)
            if (row_ids[k] >= 0) { slot[n] = k; gid[n] = row_ids[k]; n++; }
    } else {
        for (int j = 0; j < R->v; j++) { slot[n] = j; gid[n] = orc_gid(P, R, j); n++; }
    }
    return n;
}

/* Width of the teacher output: K slots aligned to ids (sparse) or the dense key axis. */
int orc_teacher_width(const orc_params *P)
{
    return P->sparse ? orc_topk_width(P) : orc_key_width(P);
}

/* ---------------------------------------------------------------- step 3: teacher */

/* Full-CSA teacher of the listed rows, by the display equations of [BUG] "Paper reference":
 *   Z_h = exp(a_h) + sum_{j in C} exp(c_hj) + sum_{r in W} exp(w_hr)
 *   t_j = sum_h exp(c_hj)/Z_h  /  max(sum_{k in C} sum_h exp(c_hk)/Z_h, 1e-10)
 * with c_hj = sigma q[t,h].kv_c[j], w_hr = sigma q[t,h].kv[r] ([BUG] sec. 3: the real attention
 * call shares one denominator over window, compressed keys and sink).  The clamp is the L1
 * normalisation of [BUG] sec. 2 excerpt.  Each exp is taken relative to the head's largest term,
 * which changes no ratio.  ids is [nrows][K] for the listed rows; out is [nrows][teacher width]. */
void orc_teacher(const orc_params *P, const double *q, const double *kv, const double *kv_c,
                 const double *sink, const int32_t *ids, const int32_t *rows, int nrows, int compact, double *out)
{
    const int H = P->heads, D = P->head_dim, K = orc_topk_width(P), NC = orc_key_width(P);
    const int TW = orc_teacher_width(P);
    const int cap = K > NC ? K : NC;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nrows; i++) {
        const long r = rows[i];
        double *t = out + (long)i * TW;
        for (int k = 0; k < TW; k++) t[k] = 0.0;
        orc_row R = orc_decode(P, r);
        if (R.v == 0) continue;
        int *slot = malloc(sizeof(int) * (size_t)cap);
        long *gid = malloc(sizeof(long) * (size_t)cap);
        int nC = orc_support(P, &R, ids + (long)i * K, slot, gid);
        if (nC == 0) { free(slot); free(gid); continue; }
        int p0 = R.s - P->window + 1;
        if (p0 < 0) p0 = 0;
        int nW = P->window > 0 ? R.s - p0 + 1 : 0;
        double *c = malloc(sizeof(double) * (size_t)nC);
        double *wl = malloc(sizeof(double) * (size_t)(nW > 0 ? nW : 1));
        double *T = calloc((size_t)nC, sizeof(double));
        for (int h = 0; h < H; h++) {
            const double *qh = q + (ORC_SRC(i, r) * H + h) * D;
            double m = sink[h];
            for (int k = 0; k < nC; k++) {
                c[k] = P->scale * orc_dot(qh, kv_c + orc_crow(P, gid[k]) * D, D);
                if (c[k] > m) m = c[k];
            }
            for (int k = 0; k < nW; k++) {
                wl[k] = P->scale * orc_dot(qh, kv + orc_qrow(P, &R, p0 + k) * D, D);
                if (wl[k] > m) m = wl[k];
            }
            if (m == -INFINITY) m = 0.0;         /* every term is exp(-inf) = 0 */
            double Z = exp(sink[h] - m);
            for (int k = 0; k < nC; k++) Z += exp(c[k] - m);
            for (int k = 0; k < nW; k++) Z += exp(wl[k] - m);
            for (int k = 0; k < nC; k++) T[k] += exp(c[k] - m) / Z;
        }
        double S = 0.0;
        for (int k = 0; k < nC; k++) S += T[k];
        if (S < ORC_EPS) S = ORC_EPS;
        for (int k = 0; k < nC; k++) t[slot[k]] = T[k] / S;
        free(c); free(wl); free(T); free(slot); free(gid);
    }
}

/* The non-compressed log-sum-exp of the listed rows: for each head,
 *   u_h = log( exp(a_h) + sum_{r in W} exp(w_hr) ),   w_hr = sigma q[t,h].kv[r]
 * the sink and window part of the denominator, which [BUG]'s proposal suggests taking from the attention
 * forward (non_compressed_lse) instead of recomputing it.  -inf when there is neither sink nor window.
 * out is [nrows][heads]. */
void orc_noncompressed_lse(const orc_params *P, const double *q, const double *kv, const double *sink,
                           const int32_t *rows, int nrows, int compact, double *out)
{
    const int H = P->heads, D = P->head_dim;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nrows; i++) {
        const long r = rows[i];
        orc_row R = orc_decode(P, r);
        int p0 = R.s - P->window + 1;
        if (p0 < 0) p0 = 0;
        const int nW = (P->window > 0 && !R.pad) ? R.s - p0 + 1 : 0;
        double *wl = malloc(sizeof(double) * (size_t)(nW > 0 ? nW : 1));
        for (int h = 0; h < H; h++) {
            const double *qh = q + (ORC_SRC(i, r) * H + h) * D;
            double m = sink[h];
            for (int k = 0; k < nW; k++) {
                wl[k] = P->scale * orc_dot(qh, kv + orc_qrow(P, &R, p0 + k) * D, D);
                if (wl[k] > m) m = wl[k];
            }
            if (m == -INFINITY) { out[(long)i * H + h] = -INFINITY; continue; }
            double Z = exp(sink[h] - m);
            for (int k = 0; k < nW; k++) Z += exp(wl[k] - m);
            out[(long)i * H + h] = m + log(Z);
        }
        free(wl);
    }
}

/* The teacher from a given non-compressed log-sum-exp u[nrows][heads] (orc_noncompressed_lse, or the
 * attention forward's): Z_h = exp(u_h) + sum_{j in C} exp(c_hj), the rest as orc_teacher.  Equal to the
 * full-CSA teacher when u is the sink-and-window log-sum-exp of the same inputs. */
void orc_teacher_lse(const orc_params *P, const double *q, const double *kv_c, const double *lse,
                     const int32_t *ids, const int32_t *rows, int nrows, int compact, double *out)
{
    const int H = P->heads, D = P->head_dim, K = orc_topk_width(P), NC = orc_key_width(P);
    const int TW = orc_teacher_width(P);
    const int cap = K > NC ? K : NC;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nrows; i++) {
        const long r = rows[i];
        double *t = out + (long)i * TW;
        for (int k = 0; k < TW; k++) t[k] = 0.0;
        orc_row R = orc_decode(P, r);
        if (R.v == 0) continue;
        int *slot = malloc(sizeof(int) * (size_t)cap);
        long *gid = malloc(sizeof(long) * (size_t)cap);
        int nC = orc_support(P, &R, ids + (long)i * K, slot, gid);
        if (nC == 0) { free(slot); free(gid); continue; }
        double *c = malloc(sizeof(double) * (size_t)nC);
        double *T = calloc((size_t)nC, sizeof(double));
        for (int h = 0; h < H; h++) {
            const double *qh = q + (ORC_SRC(i, r) * H + h) * D;
            const double u = lse[(long)i * H + h];
            double m = u;
            for (int k = 0; k < nC; k++) {
                c[k] = P->scale * orc_dot(qh, kv_c + orc_crow(P, gid[k]) * D, D);
                if (c[k] > m) m = c[k];
            }
            if (m == -INFINITY) m = 0.0;
            double Z = exp(u - m);
            for (int k = 0; k < nC; k++) Z += exp(c[k] - m);
            for (int k = 0; k < nC; k++) T[k] += exp(c[k] - m) / Z;
        }
        double S = 0.0;
        for (int k = 0; k < nC; k++) S += T[k];
        if (S < ORC_EPS) S = ORC_EPS;
        for (int k = 0; k < nC; k++) t[slot[k]] = T[k] / S;
        free(c); free(T); free(slot); free(gid);
    }
}

/* The CSA sparse attention forward of the listed rows, the step right after the path ([BUG] sec. 3: the
 * attention call takes the query, the window rows and the selected compressed rows as one key/value set
 * (kv_full) with the sink; reading: the same rows are keys and values, the sink enters the denominator
 * only):
 *   l_h    = log(exp(a_h) + sum_{j in C} exp(c_hj) + sum_{r in W} exp(w_hr))
 *   O[t,h] = sum_{j in C} exp(c_hj - l_h) kv_c[j] + sum_{r in W} exp(w_hr - l_h) kv[r]
 * out [nrows][heads][head_dim]; lse [nrows][heads] (natural log; -inf with no term at all).  Rows with no
 * visible compressed key keep their window and sink terms. */
void orc_attention(const orc_params *P, const double *q, const double *kv, const double *kv_c, const double *sink,
                   const int32_t *ids, const int32_t *rows, int nrows, int compact, double *out, double *lse)
{
    const int H = P->heads, D = P->head_dim, K = orc_topk_width(P), NC = orc_key_width(P);
    const int cap = K > NC ? K : NC;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nrows; i++) {
        const long r = rows[i];
        orc_row R = orc_decode(P, r);
        int *slot = malloc(sizeof(int) * (size_t)cap);
        long *gid = malloc(sizeof(long) * (size_t)cap);
        const int nC = R.v > 0 ? orc_support(P, &R, ids + (long)i * K, slot, gid) : 0;
        int p0 = R.s - P->window + 1;
        if (p0 < 0) p0 = 0;
        const int nW = (P->window > 0 && !R.pad) ? R.s - p0 + 1 : 0;
        double *c = malloc(sizeof(double) * (size_t)(nC > 0 ? nC : 1));
        double *wl = malloc(sizeof(double) * (size_t)(nW > 0 ? nW : 1));
        for (int h = 0; h < H; h++) {
            const double *qh = q + (ORC_SRC(i, r) * H + h) * D;
            double *o = out + ((long)i * H + h) * D;
            for (int d = 0; d < D; d++) o[d] = 0.0;
            double m = sink[h];
            for (int k = 0; k < nC; k++) {
                c[k] = P->scale * orc_dot(qh, kv_c + orc_crow(P, gid[k]) * D, D);
                if (c[k] > m) m = c[k];
            }
            for (int k = 0; k < nW; k++) {
                wl[k] = P->scale * orc_dot(qh, kv + orc_qrow(P, &R, p0 + k) * D, D);
                if (wl[k] > m) m = wl[k];
            }
            if (m == -INFINITY) { lse[(long)i * H + h] = -INFINITY; continue; }
            double Z = exp(sink[h] - m);
            for (int k = 0; k < nC; k++) Z += exp(c[k] - m);
            for (int k = 0; k < nW; k++) Z += exp(wl[k] - m);
            const double l = m + log(Z);
            lse[(long)i * H + h] = l;
            for (int k = 0; k < nC; k++) {
                const double p = exp(c[k] - l);
                const double *v = kv_c + orc_crow(P, gid[k]) * D;
                for (int d = 0; d < D; d++) o[d] += p * v[d];
            }
            for (int k = 0; k < nW; k++) {
                const double p = exp(wl[k] - l);
                const double *v = kv + orc_qrow(P, &R, p0 + k) * D;
                for (int d = 0; d < D; d++) o[d] += p * v[d];
            }
        }
        free(c); free(wl); free(slot); free(gid);
    }
}

/* ---------------------------------------------------------------- step 4: KL */

/* KL(t || p) of one row with p = softmax(I) over the n support entries:
 *   L = sum_s t_s (log(t_s + 1e-10) - log(p_s + 1e-10))       ([BUG] sec. 2 excerpt)
 * and, if g != NULL, its exact derivative with respect to each I_s:
 *   dL/dI_s = p_s (A - t_s / (p_s + 1e-10)),  A = sum_k t_k p_k / (p_k + 1e-10).
 * p is returned in p (n entries) when non-NULL. */
double orc_kl_row(const double *t, const double *I, int n, double *g, double *p_out)
{
    if (n <= 0) return 0.0;
    double m = -INFINITY;
    for (int k = 0; k < n; k++) if (I[k] > m) m = I[k];
    double *p = malloc(sizeof(double) * (size_t)n);
    double z = 0.0;
    for (int k = 0; k < n; k++) { p[k] = exp(I[k] - m); z += p[k]; }
    for (int k = 0; k < n; k++) p[k] /= z;
    double L = 0.0, A = 0.0;
    for (int k = 0; k < n; k++) {
        L += t[k] * (log(t[k] + ORC_EPS) - log(p[k] + ORC_EPS));
        A += t[k] * p[k] / (p[k] + ORC_EPS);
    }
    if (g)
        for (int k = 0; k < n; k++) g[k] = p[k] * (A - t[k] / (p[k] + ORC_EPS));
    if (p_out) memcpy(p_out, p, sizeof(double) * (size_t)n);
    free(p);
    return L;
}

/* Loss factor: coeff / (physical rows) in mean mode, coeff in sum mode
 * (the follow-up review on [BUG]: padding rows add 0 to the numerator but count in the divisor). */
double orc_loss_factor(const orc_params *P)
{
    return P->reduction == 0 ? P->coeff / (double)orc_rows(P) : P->coeff;
}

/* ---------------------------------------------------------------- step 5: backward */

/* Loss and indexer gradients of the listed rows, holding ids and teacher fixed.
 *   loss     = factor * sum_rows L_t
 *   dW[t,j]  = sum_{s in C} g_ts * max(0, x_tjs)
 *   dQ[t,j]  = sum_{s in C} g_ts * w[t,j] * 1[x_tjs > 0] * k_idx[s]
 *   dK[s]   += sum_t sum_j g_ts * w[t,j] * 1[x_tjs > 0] * q_idx[t,j]
 * with x_tjs = q_idx[t,j].k_idx[s] and g_ts = factor * dL_t/dI_ts (ReLU'(0) = 0).  No gradient
 * reaches q, kv, kv_c or the sink: the teacher is a constant here ([BUG] follow-up proposal:
 * teacher-side inputs stay detached; gradients only for indexer Q, weights and K).
 * dq: [nrows][HI][DI], dw: [nrows][HI] (rows in list order); dk: [compressed rows][DI], accumulated
 * (the caller zeroes it); loss_rows (optional): [nrows] unscaled L_t. */
double orc_loss_grads(const orc_params *P, const double *q_idx, const double *w, const double *k_idx,
                      const int32_t *ids, const double *teacher, const int32_t *rows, int nrows, int compact,
                      long n_key_rows, double *loss_rows, double *dq, double *dw, double *dk)
{
    const int HI = P->idx_heads, DI = P->idx_dim, K = orc_topk_width(P), NC = orc_key_width(P);
    const int TW = orc_teacher_width(P);
    const int cap = K > NC ? K : NC;
    const double f = orc_loss_factor(P);
    double total = 0.0;
    int nthreads = 1;
#ifdef _OPENMP
    nthreads = omp_get_max_threads();
#endif
    double *dk_local = dk ? calloc((size_t)nthreads * (size_t)n_key_rows * DI, sizeof(double)) : NULL;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : total)
    for (int i = 0; i < nrows; i++) {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        const long r = rows[i];
        if (dq) memset(dq + (long)i * HI * DI, 0, sizeof(double) * (size_t)HI * DI);
        if (dw) memset(dw + (long)i * HI, 0, sizeof(double) * (size_t)HI);
        if (loss_rows) loss_rows[i] = 0.0;
        orc_row R = orc_decode(P, r);
        if (R.v == 0) continue;
        int *slot = malloc(sizeof(int) * (size_t)cap);
        long *gid = malloc(sizeof(long) * (size_t)cap);
        int n = orc_support(P, &R, ids + (long)i * K, slot, gid);
        if (n == 0) { free(slot); free(gid); continue; }
        double *I = malloc(sizeof(double) * (size_t)n);
        double *t = malloc(sizeof(double) * (size_t)n);
        double *g = malloc(sizeof(double) * (size_t)n);
        for (int k = 0; k < n; k++) {
            I[k] = orc_score(P, q_idx, w, k_idx, ORC_SRC(i, r), gid[k]);
            t[k] = teacher[(long)i * TW + slot[k]];
        }
        double L = orc_kl_row(t, I, n, g, NULL);
        if (loss_rows) loss_rows[i] = L;
        total += L;
        for (int k = 0; k < n; k++) {
            const double gs = f * g[k];
            const long kr = orc_crow(P, gid[k]);
            const double *kk = k_idx + kr * DI;
            const long src = ORC_SRC(i, r);
            for (int j = 0; j < HI; j++) {
                const double *qj = q_idx + (src * HI + j) * DI;
                double x = orc_dot(qj, kk, DI);
                if (x <= 0.0) continue;
                if (dw) dw[(long)i * HI + j] += gs * x;
                const double a = gs * w[src * HI + j];
                if (dq) for (int d = 0; d < DI; d++) dq[((long)i * HI + j) * DI + d] += a * kk[d];
                if (dk_local) {
                    double *dkr = dk_local + ((long)tid * n_key_rows + kr) * DI;
                    for (int d = 0; d < DI; d++) dkr[d] += a * qj[d];
                }
            }
        }
        free(I); free(t); free(g); free(slot); free(gid);
    }
    if (dk_local) {
        for (int tid = 0; tid < nthreads; tid++)
            for (long e = 0; e < n_key_rows * DI; e++) dk[e] += dk_local[(long)tid * n_key_rows * DI + e];
        free(dk_local);
    }
    return f * total;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
