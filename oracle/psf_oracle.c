/*
 * psf_oracle.c -- plain fp64 CPU oracle for packed-sequence softmax attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library. The product path never calls
 * it, and it shares no code, header or constant with the CUDA library.
 *
 * Every function below is the plain definition written out, in double
 * precision, with no blocking, fusion or reordering:
 *
 *  - attention forward: out_i = sum_j softmax_j(scale * q_i . k_j) v_j over the
 *    keys j visible to query i, and lse_i = log sum_j exp(scale * q_i . k_j)
 *    (natural log of the scaled logits). A query with no visible key gives
 *    out = 0 and lse = -inf.
 *      [nemo_automodel.components.attention.ffpa_attention, `_ffpa_varlen_fwd`,
 *       `_ffpa_dense_fwd`: the return value, out [T, Hq, D] and an fp32 lse [Hq, T]]
 *  - visibility, "segments" mode: query row i and key row j of one segment
 *    (local indices, m queries and n keys, delta = n - m) see each other when
 *    (not causal or j <= i + delta) and (no window or j >= i + delta - W + 1):
 *    the causal mask sits at the segment's bottom-right corner and a positive
 *    left window W counts the current token.
 *      [nemo_automodel.components.attention.fa4, module docstring bullet 2;
 *       nemo_automodel.components.attention.utils,
 *       `preprocess_args_and_kwargs_for_attn`, **kwargs: window_size]
 *  - visibility, "document" mode: the mask is materialised from document ids
 *    and global positions, never from segment arrays: the query at global
 *    position p of batch row b sees key j of the same row when j lies in the
 *    same maximal run of equal id as p, j <= p, and p - j < W if a window is
 *    set. Padding queries (id 0) give zero output and lse = -inf.
 *      [nemo_automodel.components.attention.fa4, `document_causal_fa4_attention`
 *       (padding queries give zero output) and module docstring bullet 2 (a
 *       query at global position p sees the keys of its own document up to p)]
 *  - softcap c > 0 (off by default): each logit z = scale * q . k becomes
 *    c * tanh(z / c) before the mask and the softmax, and the backward carries
 *    the factor 1 - tanh(z / c)^2 into dS.
 *      [ffpa_attention page, `ffpa_attention_forward` softcap argument]
 *  - attention backward from the caller-supplied out and lse:
 *      Delta_i = dO_i . out_i,  P_ij = exp(scale q_i.k_j - lse_i) (0 when
 *      lse_i = -inf), dP_ij = dO_i . v_j, dS_ij = P_ij (dP_ij - Delta_i),
 *      dQ_i = scale sum_j dS_ij k_j, dK_j = scale sum_i dS_ij q_i,
 *      dV_j = sum_i P_ij dO_i, with dK/dV summed over the query heads that
 *      share a KV head (query head h uses KV head h / (Hq/Hkv)).
 *      [nemo_automodel.components.attention.ffpa_attention, `_ffpa_varlen_bwd`,
 *       `_ffpa_dense_bwd`: gradients from the out and lse the caller passes in,
 *       dK/dV summed over the query heads of each KV head]
 *    dQ is computed row by row (per query) and dK/dV column by column (per key),
 *    so either can be evaluated on a sample of rows.
 *  - segment builder: every document run of a batch row (padding runs too) is
 *    split at the end of the query shard; each piece contributes its overlap
 *    with the shard as queries and all of its tokens as keys; pieces without
 *    queries become zero-query segments; segments are listed row-major.
 *      [nemo_automodel.components.attention.fa4, module docstring bullets 1-3,
 *       `_varlen_segments`, `_varlen_layout`]
 *  - lse merge: l = logaddexp(l1, l2), o = o1 exp(l1 - l) + o2 exp(l2 - l);
 *    a row with both inputs -inf stays 0 with lse -inf.
 *      [nemo_automodel.components.models.gemma4_moe.cp_attention, the
 *       docstring of its online-softmax merge, which handles -inf]
 *  - cross-chunk segment builder: a query shard [q0, q0 + Lq) and an earlier
 *    key chunk [k0, k0 + Lk) (k0 + Lk <= q0) of every batch row; a document
 *    (a maximal run of one nonzero id) present in both pairs its shard queries
 *    with its chunk keys as one segment, which the chunk runs without a causal
 *    mask (every chunk key precedes every shard query). Since runs are
 *    contiguous, only the run holding position q0 can reach back into the chunk.
 *    Each row gives three segments in the packed shard / chunk rows:
 *    (no queries x the chunk keys before that run), (the run's shard queries x
 *    its chunk keys), (the other shard queries x no keys); the middle one is
 *    empty when no document is shared.
 *      [nemo_automodel.components.models.gemma4_moe.cp_attention,
 *       `_build_packed_ring_segments`: documents present in both the shard and
 *       the chunk, their query and key tokens paired, cu_q[i] with cu_k[i]]
 *
 * Layouts: q [Tq, Hq, Dqk], k [Tk, Hkv, Dqk], v [Tk, Hkv, Dv], out [Tq, Hq, Dv],
 * lse [Hq, Tq], all row-major and contiguous, double precision.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { MODE_SEGMENTS = 0, MODE_DOCUMENT = 1 };

typedef struct {
    int mode;
    int causal;  /* segments mode only; document mode is causal by definition */
    int window;  /* > 0: left window counting the current token; <= 0: none */
    /* segments mode */
    const int32_t *cu_q, *cu_k;
    int nseg;
    int32_t *seg_of_q; /* [Tq], -1 when the row lies in no segment */
    int32_t *seg_of_k; /* [Tk] */
    /* document mode */
    const int32_t *doc_ids; /* [B, Sk] */
    int B, Sk, Lq, q0;
    int32_t *run_of; /* [B, Sk]: index of the maximal run of equal id */
} visibility;

typedef struct {
    const double *q, *k, *v, *dout, *out, *lse;
    double *o_out, *lse_out, *dq, *dk, *dv, *delta;
    int Tq, Tk, Hq, Hkv, Dqk, Dv;
    double scale;
    double softcap; /* > 0: logits capped as softcap * tanh(z / softcap); 0: off */
    const visibility *vis;
    const int32_t *rows; /* rows (or key rows) to evaluate */
    int nrows;
} problem;

static double dot(const double *a, const double *b, int n) {
    double s = 0.0;
    for (int d = 0; d < n; ++d) s += a[d] * b[d];
    return s;
}

/* ---- visibility ------------------------------------------------------- */

static int segments_pair_visible(const visibility *vz, int s, int i, int j) {
    int m = vz->cu_q[s + 1] - vz->cu_q[s];
    int n = vz->cu_k[s + 1] - vz->cu_k[s];
    int delta = n - m;
    if (vz->causal && j > i + delta) return 0;
    if (vz->window > 0 && j < i + delta - vz->window + 1) return 0;
    return 1;
}

static int document_pair_visible(const visibility *vz, int b, int p, int j) {
    const int32_t *run = vz->run_of + (size_t)b * vz->Sk;
    if (run[j] != run[p]) return 0;
    if (j > p) return 0;
    if (vz->window > 0 && p - j >= vz->window) return 0;
    return 1;
}

/* Keys visible to query row r, written to idx. Returns their number, or -1
 * when the row's output is forced to zero (a padding query in document mode). */
static int visible_keys(const visibility *vz, int r, int32_t *idx) {
    int c = 0;
    if (vz->mode == MODE_SEGMENTS) {
        int s = vz->seg_of_q[r];
        if (s < 0) return 0;
        int i = r - vz->cu_q[s];
        int n = vz->cu_k[s + 1] - vz->cu_k[s];
        for (int j = 0; j < n; ++j)
            if (segments_pair_visible(vz, s, i, j)) idx[c++] = vz->cu_k[s] + j;
        return c;
    }
    int b = r / vz->Lq, i = r % vz->Lq, p = vz->q0 + i;
    if (vz->doc_ids[(size_t)b * vz->Sk + p] == 0) return -1;
    for (int j = 0; j < vz->Sk; ++j)
        if (document_pair_visible(vz, b, p, j)) idx[c++] = b * vz->Sk + j;
    return c;
}

/* Query rows that see key row kr (padding queries excluded in document mode). */
static int visible_queries(const visibility *vz, int kr, int32_t *idx) {
    int c = 0;
    if (vz->mode == MODE_SEGMENTS) {
        int s = vz->seg_of_k[kr];
        if (s < 0) return 0;
        int j = kr - vz->cu_k[s];
        int m = vz->cu_q[s + 1] - vz->cu_q[s];
        for (int i = 0; i < m; ++i)
            if (segments_pair_visible(vz, s, i, j)) idx[c++] = vz->cu_q[s] + i;
        return c;
    }
    int b = kr / vz->Sk, j = kr % vz->Sk;
    for (int i = 0; i < vz->Lq; ++i) {
        int p = vz->q0 + i;
        if (vz->doc_ids[(size_t)b * vz->Sk + p] == 0) continue;
        if (document_pair_visible(vz, b, p, j)) idx[c++] = b * vz->Lq + i;
    }
    return c;
}

static int setup_visibility(visibility *vz, int Tq, int Tk) {
    vz->seg_of_q = vz->seg_of_k = vz->run_of = NULL;
    if (vz->mode == MODE_SEGMENTS) {
        vz->seg_of_q = (int32_t *)malloc(sizeof(int32_t) * (size_t)(Tq > 0 ? Tq : 1));
        vz->seg_of_k = (int32_t *)malloc(sizeof(int32_t) * (size_t)(Tk > 0 ? Tk : 1));
        if (!vz->seg_of_q || !vz->seg_of_k) return -1;
        for (int r = 0; r < Tq; ++r) vz->seg_of_q[r] = -1;
        for (int r = 0; r < Tk; ++r) vz->seg_of_k[r] = -1;
        for (int s = 0; s < vz->nseg; ++s) {
            for (int r = vz->cu_q[s]; r < vz->cu_q[s + 1] && r < Tq; ++r) vz->seg_of_q[r] = s;
            for (int r = vz->cu_k[s]; r < vz->cu_k[s + 1] && r < Tk; ++r) vz->seg_of_k[r] = s;
        }
        return 0;
    }
    vz->run_of = (int32_t *)malloc(sizeof(int32_t) * (size_t)vz->B * (size_t)(vz->Sk > 0 ? vz->Sk : 1));
    if (!vz->run_of) return -1;
    for (int b = 0; b < vz->B; ++b) {
        const int32_t *ids = vz->doc_ids + (size_t)b * vz->Sk;
        int32_t *run = vz->run_of + (size_t)b * vz->Sk;
        int r = 0;
        for (int j = 0; j < vz->Sk; ++j) {
            if (j > 0 && ids[j] != ids[j - 1]) ++r;
            run[j] = r;
        }
    }
    return 0;
}

static void free_visibility(visibility *vz) {
    free(vz->seg_of_q);
    free(vz->seg_of_k);
    free(vz->run_of);
}

/* ---- thread pool over a row list --------------------------------------- */

typedef struct {
    const problem *pb;
    int begin, end;
    void (*fn)(const problem *, int, int);
} work_slice;

static void *run_slice(void *arg) {
    work_slice *w = (work_slice *)arg;
    w->fn(w->pb, w->begin, w->end);
    return NULL;
}

static void parallel_rows(const problem *pb, int nthreads, void (*fn)(const problem *, int, int)) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > pb->nrows) nthreads = pb->nrows > 0 ? pb->nrows : 1;
    if (nthreads == 1) {
        fn(pb, 0, pb->nrows);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    work_slice *ws = (work_slice *)malloc(sizeof(work_slice) * (size_t)nthreads);
    int per = (pb->nrows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        ws[t].pb = pb;
        ws[t].fn = fn;
        ws[t].begin = t * per < pb->nrows ? t * per : pb->nrows;
        ws[t].end = (t + 1) * per < pb->nrows ? (t + 1) * per : pb->nrows;
        pthread_create(&th[t], NULL, run_slice, &ws[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    free(ws);
}

/* ---- logits ------------------------------------------------------------- */

/*
 * The logit of a (query, key) pair from q . k: z = scale * q . k, or with a
 * softcap c > 0, c * tanh(z / c), applied before the mask and the softmax.
 *   [ffpa_attention page, `ffpa_attention_forward` (softcap argument; the
 *    eager attention it falls back to for softcap caps the scaled scores as
 *    softcap * tanh(scores / softcap))]
 */
static double logit(const problem *pb, double qk) {
    double z = pb->scale * qk;
    return pb->softcap > 0.0 ? pb->softcap * tanh(z / pb->softcap) : z;
}

/* d logit / dz: 1 - tanh(z / c)^2 with a softcap, else 1. */
static double logit_slope(const problem *pb, double qk) {
    if (!(pb->softcap > 0.0)) return 1.0;
    double t = tanh(pb->scale * qk / pb->softcap);
    return 1.0 - t * t;
}

/* ---- forward ------------------------------------------------------------ */

static void fwd_rows(const problem *pb, int begin, int end) {
    int Tk = pb->Tk > 0 ? pb->Tk : 1;
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)Tk);
    double *z = (double *)malloc(sizeof(double) * (size_t)Tk);
    int G = pb->Hq / pb->Hkv;
    for (int t = begin; t < end; ++t) {
        int r = pb->rows[t];
        int nvis = visible_keys(pb->vis, r, idx);
        for (int h = 0; h < pb->Hq; ++h) {
            int hk = h / G;
            double *o = pb->o_out + ((size_t)r * pb->Hq + h) * pb->Dv;
            double *l = pb->lse_out + (size_t)h * pb->Tq + r;
            for (int d = 0; d < pb->Dv; ++d) o[d] = 0.0;
            if (nvis <= 0) {
                *l = -INFINITY;
                continue;
            }
            const double *qi = pb->q + ((size_t)r * pb->Hq + h) * pb->Dqk;
            double zmax = -INFINITY;
            for (int c = 0; c < nvis; ++c) {
                const double *kj = pb->k + ((size_t)idx[c] * pb->Hkv + hk) * pb->Dqk;
                z[c] = logit(pb, dot(qi, kj, pb->Dqk));
                if (z[c] > zmax) zmax = z[c];
            }
            double sum = 0.0;
            for (int c = 0; c < nvis; ++c) sum += exp(z[c] - zmax);
            double lse = zmax + log(sum);
            for (int c = 0; c < nvis; ++c) {
                double p = exp(z[c] - lse);
                const double *vj = pb->v + ((size_t)idx[c] * pb->Hkv + hk) * pb->Dv;
                for (int d = 0; d < pb->Dv; ++d) o[d] += p * vj[d];
            }
            *l = lse;
        }
    }
    free(idx);
    free(z);
}

/* ---- backward ----------------------------------------------------------- */

static void delta_rows(const problem *pb, int begin, int end) {
    for (int t = begin; t < end; ++t) {
        int r = pb->rows[t];
        for (int h = 0; h < pb->Hq; ++h) {
            const double *g = pb->dout + ((size_t)r * pb->Hq + h) * pb->Dv;
            const double *o = pb->out + ((size_t)r * pb->Hq + h) * pb->Dv;
            pb->delta[(size_t)h * pb->Tq + r] = dot(g, o, pb->Dv);
        }
    }
}

static void dq_rows(const problem *pb, int begin, int end) {
    int Tk = pb->Tk > 0 ? pb->Tk : 1;
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)Tk);
    int G = pb->Hq / pb->Hkv;
    for (int t = begin; t < end; ++t) {
        int r = pb->rows[t];
        int nvis = visible_keys(pb->vis, r, idx);
        for (int h = 0; h < pb->Hq; ++h) {
            int hk = h / G;
            double *dq = pb->dq + ((size_t)r * pb->Hq + h) * pb->Dqk;
            for (int d = 0; d < pb->Dqk; ++d) dq[d] = 0.0;
            double lse = pb->lse[(size_t)h * pb->Tq + r];
            if (nvis <= 0 || lse == -INFINITY) continue;
            const double *qi = pb->q + ((size_t)r * pb->Hq + h) * pb->Dqk;
            const double *gi = pb->dout + ((size_t)r * pb->Hq + h) * pb->Dv;
            double delta = pb->delta[(size_t)h * pb->Tq + r];
            for (int c = 0; c < nvis; ++c) {
                const double *kj = pb->k + ((size_t)idx[c] * pb->Hkv + hk) * pb->Dqk;
                const double *vj = pb->v + ((size_t)idx[c] * pb->Hkv + hk) * pb->Dv;
                double qk = dot(qi, kj, pb->Dqk);
                double p = exp(logit(pb, qk) - lse);
                double ds = p * (dot(gi, vj, pb->Dv) - delta) * logit_slope(pb, qk);
                for (int d = 0; d < pb->Dqk; ++d) dq[d] += pb->scale * ds * kj[d];
            }
        }
    }
    free(idx);
}

static void dkdv_rows(const problem *pb, int begin, int end) {
    int Tq = pb->Tq > 0 ? pb->Tq : 1;
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)Tq);
    int G = pb->Hq / pb->Hkv;
    for (int t = begin; t < end; ++t) {
        int kr = pb->rows[t];
        int nq = visible_queries(pb->vis, kr, idx);
        for (int hk = 0; hk < pb->Hkv; ++hk) {
            double *dk = pb->dk + ((size_t)kr * pb->Hkv + hk) * pb->Dqk;
            double *dv = pb->dv + ((size_t)kr * pb->Hkv + hk) * pb->Dv;
            for (int d = 0; d < pb->Dqk; ++d) dk[d] = 0.0;
            for (int d = 0; d < pb->Dv; ++d) dv[d] = 0.0;
            const double *kj = pb->k + ((size_t)kr * pb->Hkv + hk) * pb->Dqk;
            const double *vj = pb->v + ((size_t)kr * pb->Hkv + hk) * pb->Dv;
            for (int h = hk * G; h < (hk + 1) * G; ++h) {
                for (int c = 0; c < nq; ++c) {
                    int r = idx[c];
                    double lse = pb->lse[(size_t)h * pb->Tq + r];
                    if (lse == -INFINITY) continue;
                    const double *qi = pb->q + ((size_t)r * pb->Hq + h) * pb->Dqk;
                    const double *gi = pb->dout + ((size_t)r * pb->Hq + h) * pb->Dv;
                    double qk = dot(qi, kj, pb->Dqk);
                    double p = exp(logit(pb, qk) - lse);
                    double ds = p * (dot(gi, vj, pb->Dv) - pb->delta[(size_t)h * pb->Tq + r]) * logit_slope(pb, qk);
                    for (int d = 0; d < pb->Dv; ++d) dv[d] += p * gi[d];
                    for (int d = 0; d < pb->Dqk; ++d) dk[d] += pb->scale * ds * qi[d];
                }
            }
        }
    }
    free(idx);
}

/* ---- exported entry points --------------------------------------------- */

static int32_t *all_rows(int n) {
    int32_t *r = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    for (int i = 0; i < n; ++i) r[i] = i;
    return r;
}

static visibility make_visibility(int mode, int causal, int window, const int32_t *cu_q,
                                  const int32_t *cu_k, int nseg, const int32_t *doc_ids, int B,
                                  int Sk, int Lq, int q0) {
    visibility vz;
    memset(&vz, 0, sizeof(vz));
    vz.mode = mode;
    vz.causal = causal;
    vz.window = window;
    vz.cu_q = cu_q;
    vz.cu_k = cu_k;
    vz.nseg = nseg;
    vz.doc_ids = doc_ids;
    vz.B = B;
    vz.Sk = Sk;
    vz.Lq = Lq;
    vz.q0 = q0;
    return vz;
}

/*
 * Forward. mode 0 ("segments"): cu_q/cu_k/nseg/causal/window describe the
 * mask. mode 1 ("document"): doc_ids [B, Sk], the query shard [q0, q0 + Lq) of
 * every row, and window describe it; Tq must be B * Lq and Tk must be B * Sk.
 * rows (nullable) selects the query rows to evaluate; other rows are untouched.
 */
int oracle_attn_fwd(int mode, int causal, int window, const int32_t *cu_q, const int32_t *cu_k,
                    int nseg, const int32_t *doc_ids, int B, int Sk, int Lq, int q0,
                    const double *q, const double *k, const double *v, int Tq, int Tk, int Hq,
                    int Hkv, int Dqk, int Dv, double scale, double softcap, const int32_t *rows, int nrows,
                    double *out, double *lse, int nthreads) {
    if (Hkv <= 0 || Hq % Hkv != 0) return -1;
    visibility vz = make_visibility(mode, causal, window, cu_q, cu_k, nseg, doc_ids, B, Sk, Lq, q0);
    if (setup_visibility(&vz, Tq, Tk) != 0) return -2;
    int32_t *own = NULL;
    if (!rows) {
        own = all_rows(Tq);
        rows = own;
        nrows = Tq;
    }
    problem pb;
    memset(&pb, 0, sizeof(pb));
    pb.q = q;
    pb.k = k;
    pb.v = v;
    pb.o_out = out;
    pb.lse_out = lse;
    pb.Tq = Tq;
    pb.Tk = Tk;
    pb.Hq = Hq;
    pb.Hkv = Hkv;
    pb.Dqk = Dqk;
    pb.Dv = Dv;
    pb.scale = scale;
    pb.softcap = softcap;
    pb.vis = &vz;
    pb.rows = rows;
    pb.nrows = nrows;
    parallel_rows(&pb, nthreads, fwd_rows);
    free(own);
    free_visibility(&vz);
    return 0;
}

/*
 * Backward from caller-supplied out [Tq,Hq,Dv] and lse [Hq,Tq]. dq is written
 * for q_rows (nullable = all), dk/dv for k_rows (nullable = all); either output
 * pointer may be NULL to skip that part.
 */
int oracle_attn_bwd(int mode, int causal, int window, const int32_t *cu_q, const int32_t *cu_k,
                    int nseg, const int32_t *doc_ids, int B, int Sk, int Lq, int q0,
                    const double *dout, const double *q, const double *k, const double *v,
                    const double *out, const double *lse, int Tq, int Tk, int Hq, int Hkv, int Dqk,
                    int Dv, double scale, double softcap, const int32_t *q_rows, int nq_rows, const int32_t *k_rows,
                    int nk_rows, double *dq, double *dk, double *dv, int nthreads) {
    if (Hkv <= 0 || Hq % Hkv != 0) return -1;
    visibility vz = make_visibility(mode, causal, window, cu_q, cu_k, nseg, doc_ids, B, Sk, Lq, q0);
    if (setup_visibility(&vz, Tq, Tk) != 0) return -2;
    problem pb;
    memset(&pb, 0, sizeof(pb));
    pb.q = q;
    pb.k = k;
    pb.v = v;
    pb.dout = dout;
    pb.out = out;
    pb.lse = lse;
    pb.Tq = Tq;
    pb.Tk = Tk;
    pb.Hq = Hq;
    pb.Hkv = Hkv;
    pb.Dqk = Dqk;
    pb.Dv = Dv;
    pb.scale = scale;
    pb.softcap = softcap;
    pb.vis = &vz;
    pb.delta = (double *)malloc(sizeof(double) * (size_t)Hq * (size_t)(Tq > 0 ? Tq : 1));
    int32_t *every_q = all_rows(Tq);
    pb.rows = every_q;
    pb.nrows = Tq;
    parallel_rows(&pb, nthreads, delta_rows);
    if (dq) {
        int32_t *own = NULL;
        if (!q_rows) {
            own = all_rows(Tq);
            q_rows = own;
            nq_rows = Tq;
        }
        pb.dq = dq;
        pb.rows = q_rows;
        pb.nrows = nq_rows;
        parallel_rows(&pb, nthreads, dq_rows);
        free(own);
    }
    if (dk && dv) {
        int32_t *own = NULL;
        if (!k_rows) {
            own = all_rows(Tk);
            k_rows = own;
            nk_rows = Tk;
        }
        pb.dk = dk;
        pb.dv = dv;
        pb.rows = k_rows;
        pb.nrows = nk_rows;
        parallel_rows(&pb, nthreads, dkdv_rows);
        free(own);
    }
    free(every_q);
    free(pb.delta);
    free_visibility(&vz);
    return 0;
}

/*
 * Segment builder. doc_ids [B, Sk]; the query shard is [q0, q0 + Lq) of every
 * row. Writes cu_q/cu_k (capacity + 1 entries each) and returns the number of
 * segments, or -1 when capacity is too small.
 * skip_pad != 0: a piece of a padding run (id 0) becomes two segments, its
 * queries with no keys and then its keys with no queries, so no padding query
 * attends anything (out 0, lse -inf, the value padding queries must get) and
 * the key segments still tile the keys.
 *   [fa4 page, `document_causal_fa4_attention`: padding queries are zero;
 *    cp_attention page, `_build_packed_ring_segments`: pad query rows zeroed]
 */
int oracle_build_segments(const int32_t *doc_ids, int B, int Sk, int Lq, int q0, int32_t *cu_q,
                          int32_t *cu_k, int capacity, int32_t *max_q, int32_t *max_k, int skip_pad) {
    int q_end = q0 + Lq;
    int nseg = 0;
    int mq = 0, mk = 0;
    cu_q[0] = 0;
    cu_k[0] = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t *ids = doc_ids + (size_t)b * Sk;
        int a = 0;
        while (a < Sk) {
            int e = a + 1;
            while (e < Sk && ids[e] == ids[a]) ++e; /* maximal run [a, e) */
            int cuts[3] = {a, e, e};
            int npieces = 1;
            if (a < q_end && q_end < e) {
                cuts[1] = q_end;
                npieces = 2;
            }
            for (int pc = 0; pc < npieces; ++pc) {
                int pa = cuts[pc], pe = cuts[pc + 1];
                int lo = pa > q0 ? pa : q0;
                int hi = pe < q_end ? pe : q_end;
                int nq = hi > lo ? hi - lo : 0;
                int nk = pe - pa;
                if (nq > mq) mq = nq;
                if (nk > mk) mk = nk;
                if (skip_pad && ids[a] == 0) {
                    if (nseg + 2 > capacity) return -1;
                    cu_q[nseg + 1] = cu_q[nseg] + nq; /* the queries, no keys */
                    cu_k[nseg + 1] = cu_k[nseg];
                    ++nseg;
                    cu_q[nseg + 1] = cu_q[nseg]; /* the keys, no queries */
                    cu_k[nseg + 1] = cu_k[nseg] + nk;
                    ++nseg;
                    continue;
                }
                if (nseg >= capacity) return -1;
                cu_q[nseg + 1] = cu_q[nseg] + nq;
                cu_k[nseg + 1] = cu_k[nseg] + nk;
                ++nseg;
            }
            a = e;
        }
    }
    *max_q = mq;
    *max_k = mk;
    return nseg;
}

/* lse merge of two partial results over disjoint key sets: o/l [T, H, D] / [H, T]. */
void oracle_lse_merge(const double *o1, const double *l1, const double *o2, const double *l2,
                      double *o, double *l, int T, int H, int D) {
    for (int h = 0; h < H; ++h) {
        for (int t = 0; t < T; ++t) {
            double a = l1[(size_t)h * T + t], b = l2[(size_t)h * T + t];
            double m = a > b ? a : b;
            double lm = (m == -INFINITY) ? -INFINITY : m + log(exp(a - m) + exp(b - m));
            l[(size_t)h * T + t] = lm;
            double *od = o + ((size_t)t * H + h) * D;
            const double *x = o1 + ((size_t)t * H + h) * D;
            const double *y = o2 + ((size_t)t * H + h) * D;
            if (lm == -INFINITY) {
                for (int d = 0; d < D; ++d) od[d] = 0.0;
                continue;
            }
            double wa = exp(a - lm), wb = exp(b - lm);
            for (int d = 0; d < D; ++d) od[d] = wa * x[d] + wb * y[d];
        }
    }
}

/*
 * Cross-chunk segments of a query shard against an earlier key chunk (see the
 * header). Writes cu_q / cu_k (3 B + 1 entries each) over the packed shard rows
 * (b * Lq + p - q0) and chunk rows (b * Lk + j - k0); returns 3 B, or -1 when
 * the chunk does not lie before the shard.
 */
int oracle_build_cross_segments(const int32_t *doc_ids, int B, int S, int q0, int Lq, int k0, int Lk,
                                int32_t *cu_q, int32_t *cu_k, int32_t *max_q, int32_t *max_k) {
    if (q0 < 0 || Lq < 0 || k0 < 0 || Lk < 0 || k0 + Lk > q0 || q0 + Lq > S) return -1;
    int mq = 0, mk = 0, n = 0;
    cu_q[0] = 0;
    cu_k[0] = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t *ids = doc_ids + (size_t)b * S;
        int nq = 0, ks = k0 + Lk; /* shared run: queries [q0, q0 + nq), keys [ks, k0 + Lk) */
        if (Lq > 0 && Lk > 0 && ids[q0] != 0) {
            int d = ids[q0];
            int s0 = q0;
            while (s0 > 0 && ids[s0 - 1] == d) --s0;
            int e = q0;
            while (e < S && ids[e] == d) ++e;
            if (s0 < k0 + Lk) {
                ks = s0 > k0 ? s0 : k0;
                nq = (e < q0 + Lq ? e : q0 + Lq) - q0;
            }
        }
        const int qn[3] = {0, nq, Lq - nq};
        const int kn[3] = {ks - k0, k0 + Lk - ks, 0};
        for (int i = 0; i < 3; ++i) {
            cu_q[n + 1] = cu_q[n] + qn[i];
            cu_k[n + 1] = cu_k[n] + kn[i];
            if (qn[i] > mq) mq = qn[i];
            if (kn[i] > mk) mk = kn[i];
            ++n;
        }
    }
    *max_q = mq;
    *max_k = mk;
    return n;
}
