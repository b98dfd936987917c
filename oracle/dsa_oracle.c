/*
 * dsa_oracle.c -- CPU reference of the DeepSeek Sparse Attention hot path.
 *
 * TEST INFRASTRUCTURE, not the product.  Plain loops in double precision,
 * written from the pages' description of the method:
 *
 *  - ik_llama_opt commit log, "Add GLM-5.2/DeepSeek-V3.2 DSA lightning
 *    indexer" (the indexer formula: ReLU of the key.query dot, scaled per-head
 *    weights, sum over heads, causal mask, top-k of min(top_k, n) keys) and
 *    "GLM-5.2 DSA indexer: decode-correct via persistent indexer-K cache"
 *    (single-head fp16 indexer-key cache written at the token's own slot
 *    before scoring; Walsh-Hadamard rotation of q and k before the fp16 store,
 *    score preserving because (Hq).(Hk) = q.k).
 *  - ds4 PR #523 "hy3: Metal decode path + shared gate/up fusion", milestone
 *    M3 bullets on glm_mla_attention_one (576-wide cached rows = 512 latent +
 *    64 rotated rope tail; per-row expansion through kv_b into 192 nope-key
 *    and 256 value dims per head; one softmax over the candidate rows).
 *  - ik_llama_opt commit log, "MLA tensor parallelism under -sm graph"
 *    (wk_b / wv_b absorbed weights derived from wkv_b): the absorbed form in
 *    which queries are pre-multiplied by W_UK and attention runs on the
 *    512-d latent.
 *
 * Readings where the pages are silent are listed in the design notes; the
 * ones that shape this file: no extra indexer scale constant (the caller
 * folds it into w), causal bound inclusive, ties to the lower position,
 * output positions ascending, softmax scale passed in.
 */
#include "dsa_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define D_I 128
#define D_L 512
#define D_R 64
#define D_ROW 576

/* ---------------------------------------------------------------- storage */

double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1, e = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

uint16_t oracle_f64_to_f16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return 0x7E00;
    if (a >= 65520.0) return sign | 0x7C00;           /* rounds to infinity */
    if (a < ldexp(1.0, -14)) {                         /* subnormal range: step 2^-24 */
        double q = rint(ldexp(a, 24));                 /* exact scaling; ties to even */
        return sign | (uint16_t)q;                     /* q == 1024 is the smallest normal */
    }
    int e2;
    frexp(a, &e2);                                     /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;                                    /* a in [2^E, 2^(E+1)) */
    double q = rint(ldexp(a, 10 - E));                 /* in [1024, 2048] */
    if (q >= 2048.0) { q = 1024.0; E += 1; }
    if (E + 15 >= 31) return sign | 0x7C00;
    return sign | (uint16_t)(((E + 15) << 10) | ((int)q - 1024));
}

/* ---------------------------------------------------------------- Hadamard */

void oracle_fwht128(const double *x, double *y)
{
    double v[D_I];
    for (int i = 0; i < D_I; i++) v[i] = x[i];
    /* Sylvester recursion H_2n = [[H_n, H_n], [H_n, -H_n]] as butterflies. */
    for (int len = 1; len < D_I; len <<= 1)
        for (int i = 0; i < D_I; i += 2 * len)
            for (int j = i; j < i + len; j++) {
                double a = v[j], b = v[j + len];
                v[j] = a + b;
                v[j + len] = a - b;
            }
    double s = 1.0 / sqrt((double)D_I);
    for (int i = 0; i < D_I; i++) y[i] = v[i] * s;
}

/* ---------------------------------------------------------------- helpers */

static int seq_of(int t, int B, const int32_t *cu_q)
{
    for (int b = 0; b < B; b++)
        if (t >= cu_q[b] && t < cu_q[b + 1]) return b;
    return -1;
}

static int check_batch(int B, int T, const int32_t *cu_q, const int32_t *q_pos)
{
    if (B < 1 || T < 0 || cu_q[0] != 0 || cu_q[B] != T) return -1;
    for (int b = 0; b < B; b++)
        if (cu_q[b + 1] < cu_q[b]) return -1;
    for (int t = 0; t < T; t++)
        if (q_pos[t] < 0) return -1;
    return 0;
}

int oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* ---------------------------------------------------------------- append */

int oracle_k_append(const void *k_new, int k_dtype, int B, int T,
                    const int32_t *cu_q, const int32_t *q_pos, const int64_t *kv_off,
                    uint16_t *k_cache, int hadamard)
{
    if (check_batch(B, T, cu_q, q_pos) || (k_dtype != 0 && k_dtype != 1)) return -1;
    for (int t = 0; t < T; t++) {
        int b = seq_of(t, B, cu_q);
        double k[D_I], kr[D_I];
        for (int d = 0; d < D_I; d++)
            k[d] = k_dtype == 0 ? (double)((const float *)k_new)[(int64_t)t * D_I + d]
                                : oracle_f16_to_f64(((const uint16_t *)k_new)[(int64_t)t * D_I + d]);
        if (hadamard) oracle_fwht128(k, kr);
        else memcpy(kr, k, sizeof kr);
        uint16_t *row = k_cache + (kv_off[b] + q_pos[t]) * (int64_t)D_I;
        for (int d = 0; d < D_I; d++) row[d] = oracle_f64_to_f16(kr[d]);
    }
    return 0;
}

/* ---------------------------------------------------------------- score */

int oracle_indexer_score(const uint16_t *q_idx, const float *w, const uint16_t *k_cache,
                         int B, int T, const int32_t *cu_q, const int32_t *q_pos,
                         const int64_t *kv_off, int H_I, int hadamard_q,
                         double *scores, int64_t ld)
{
    if (check_batch(B, T, cu_q, q_pos) || H_I < 1) return -1;
    for (int t = 0; t < T; t++)
        if (q_pos[t] + 1 > ld) return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; t++) {
        int b = seq_of(t, B, cu_q);
        double *q = malloc(sizeof(double) * (size_t)H_I * D_I);
        if (!q) { bad = 1; continue; }
        for (int h = 0; h < H_I; h++) {
            double raw[D_I];
            for (int d = 0; d < D_I; d++)
                raw[d] = oracle_f16_to_f64(q_idx[((int64_t)t * H_I + h) * D_I + d]);
            if (hadamard_q) oracle_fwht128(raw, q + (size_t)h * D_I);
            else memcpy(q + (size_t)h * D_I, raw, sizeof raw);
        }
        double *row = scores + (int64_t)t * ld;
        for (int64_t s = 0; s < ld; s++) {
            if (s > q_pos[t]) { row[s] = -INFINITY; continue; }
            const uint16_t *kr = k_cache + (kv_off[b] + s) * (int64_t)D_I;
            double k[D_I];
            for (int d = 0; d < D_I; d++) k[d] = oracle_f16_to_f64(kr[d]);
            double I = 0.0;
            for (int h = 0; h < H_I; h++) {
                double dot = 0.0;
                for (int d = 0; d < D_I; d++) dot += q[(size_t)h * D_I + d] * k[d];
                double r = dot > 0.0 ? dot : 0.0;            /* ReLU on the dot ... */
                I += (double)w[(int64_t)t * H_I + h] * r;     /* ... then the head weight */
            }
            row[s] = I;
        }
        free(q);
    }
    return bad ? -1 : 0;
}

/* ---------------------------------------------------------------- top-k */

typedef struct { double v; int32_t s; } cand_t;

static int by_score_desc_pos_asc(const void *pa, const void *pb)
{
    const cand_t *a = pa, *b = pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->s > b->s) - (a->s < b->s);
}

static int by_pos(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

int oracle_topk(const double *scores, int64_t ld, int T, const int32_t *q_pos,
                int k, int32_t *idx)
{
    if (k < 1 || T < 0) return -1;
    for (int t = 0; t < T; t++)
        if (q_pos[t] < 0 || q_pos[t] + 1 > ld) return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; t++) {
        int n = q_pos[t] + 1;
        int32_t *out = idx + (int64_t)t * k;
        cand_t *c = malloc(sizeof(cand_t) * (size_t)n);
        if (!c) { bad = 1; continue; }
        for (int s = 0; s < n; s++) {
            c[s].v = scores[(int64_t)t * ld + s];
            c[s].s = s;
        }
        /* -0.0 == +0.0 under this comparison, so signed zeros tie by position. */
        qsort(c, (size_t)n, sizeof(cand_t), by_score_desc_pos_asc);
        int m = n < k ? n : k;
        for (int i = 0; i < m; i++) out[i] = c[i].s;
        qsort(out, (size_t)m, sizeof(int32_t), by_pos);
        for (int i = m; i < k; i++) out[i] = -1;
        free(c);
    }
    return bad ? -1 : 0;
}

/* ---------------------------------------------------------------- attention */

/* One (token, head): softmax over the listed cache rows, in double. */
int oracle_topk_sink(const double *scores, int64_t ld, int T, const int32_t *q_pos,
                     int k, int n_sink, const int32_t *anchor, int32_t *idx)
{
    if (n_sink < 0 || T < 0 || ld < 1) return -1;
    double *boosted = malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * (size_t)ld);
    if (!boosted) return -1;
    memcpy(boosted, scores, sizeof(double) * (size_t)T * (size_t)ld);
    for (int t = 0; t < T; t++) {
        int64_t lo = anchor ? anchor[t] : 0;
        if (lo < 0) lo = 0;
        int64_t hi = lo + n_sink;
        if (hi > (int64_t)q_pos[t] + 1) hi = (int64_t)q_pos[t] + 1;
        if (hi > ld) hi = ld;
        for (int64_t s = lo; s < hi; s++) boosted[(int64_t)t * ld + s] = INFINITY;
    }
    int rc = oracle_topk(boosted, ld, T, q_pos, k, idx);
    free(boosted);
    return rc;
}

static void attend_rows(const double *ql, const double *qr, const uint16_t *kv_cache,
                        int64_t base, const int32_t *pos, int n, double sm_scale,
                        double *o, double *lse)
{
    for (int d = 0; d < D_L; d++) o[d] = 0.0;
    if (n == 0) { if (lse) *lse = -INFINITY; return; }
    double *z = malloc(sizeof(double) * (size_t)n);
    double m = -INFINITY;
    for (int j = 0; j < n; j++) {
        const uint16_t *c = kv_cache + (base + pos[j]) * (int64_t)D_ROW;
        double acc = 0.0;
        for (int d = 0; d < D_L; d++) acc += ql[d] * oracle_bf16_to_f64(c[d]);
        for (int d = 0; d < D_R; d++) acc += qr[d] * oracle_bf16_to_f64(c[D_L + d]);
        z[j] = sm_scale * acc;
        if (z[j] > m) m = z[j];
    }
    double l = 0.0;
    for (int j = 0; j < n; j++) {
        double p = exp(z[j] - m);
        l += p;
        const uint16_t *c = kv_cache + (base + pos[j]) * (int64_t)D_ROW;
        for (int d = 0; d < D_L; d++) o[d] += p * oracle_bf16_to_f64(c[d]);
    }
    for (int d = 0; d < D_L; d++) o[d] /= l;
    if (lse) *lse = m + log(l);
    free(z);
}

int oracle_sparse_attn_f64(const double *q_lat, const double *q_rope, const uint16_t *kv_cache,
                           int B, int T, const int32_t *cu_q, const int32_t *q_pos,
                           const int64_t *kv_off, const int32_t *idx, int k, int H,
                           double sm_scale, double *out, double *lse)
{
    if (check_batch(B, T, cu_q, q_pos) || k < 1 || H < 1) return -1;
    for (int t = 0; t < T; t++)
        for (int i = 0; i < k; i++) {
            int32_t j = idx[(int64_t)t * k + i];
            if (j != -1 && (j < 0 || j > q_pos[t])) return -2;
        }
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int t = 0; t < T; t++)
        for (int h = 0; h < H; h++) {
            int b = seq_of(t, B, cu_q);
            int32_t *pos = malloc(sizeof(int32_t) * (size_t)k);
            int n = 0;
            for (int i = 0; i < k; i++) {
                int32_t j = idx[(int64_t)t * k + i];
                if (j >= 0) pos[n++] = j;
            }
            attend_rows(q_lat + ((int64_t)t * H + h) * D_L, q_rope + ((int64_t)t * H + h) * D_R,
                        kv_cache, kv_off[b], pos, n, sm_scale,
                        out + ((int64_t)t * H + h) * D_L, lse ? lse + (int64_t)t * H + h : NULL);
            free(pos);
        }
    return 0;
}

static double *bf16_array_to_f64(const uint16_t *x, int64_t n)
{
    double *y = malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!y) return NULL;
    for (int64_t i = 0; i < n; i++) y[i] = oracle_bf16_to_f64(x[i]);
    return y;
}

int oracle_sparse_attn(const uint16_t *q_lat, const uint16_t *q_rope, const uint16_t *kv_cache,
                       int B, int T, const int32_t *cu_q, const int32_t *q_pos,
                       const int64_t *kv_off, const int32_t *idx, int k, int H,
                       double sm_scale, double *out, double *lse)
{
    double *ql = bf16_array_to_f64(q_lat, (int64_t)T * H * D_L);
    double *qr = bf16_array_to_f64(q_rope, (int64_t)T * H * D_R);
    int rc = (ql && qr) ? oracle_sparse_attn_f64(ql, qr, kv_cache, B, T, cu_q, q_pos, kv_off,
                                                 idx, k, H, sm_scale, out, lse)
                        : -1;
    free(ql);
    free(qr);
    return rc;
}

/* One (token, head) of the NoPE form: rows of D_L latent values only. */
static void attend_rows_nope(const double *ql, const uint16_t *kv_latent, int64_t base,
                             const int32_t *pos, int n, double sm_scale, double *o, double *lse)
{
    for (int d = 0; d < D_L; d++) o[d] = 0.0;
    if (n == 0) { if (lse) *lse = -INFINITY; return; }
    double *z = malloc(sizeof(double) * (size_t)n);
    double m = -INFINITY;
    for (int j = 0; j < n; j++) {
        const uint16_t *c = kv_latent + (base + pos[j]) * (int64_t)D_L;
        double acc = 0.0;
        for (int d = 0; d < D_L; d++) acc += ql[d] * oracle_bf16_to_f64(c[d]);
        z[j] = sm_scale * acc;
        if (z[j] > m) m = z[j];
    }
    double l = 0.0;
    for (int j = 0; j < n; j++) {
        double p = exp(z[j] - m);
        l += p;
        const uint16_t *c = kv_latent + (base + pos[j]) * (int64_t)D_L;
        for (int d = 0; d < D_L; d++) o[d] += p * oracle_bf16_to_f64(c[d]);
    }
    for (int d = 0; d < D_L; d++) o[d] /= l;
    if (lse) *lse = m + log(l);
    free(z);
}

int oracle_sparse_attn_nope_f64(const double *q_lat, const uint16_t *kv_latent,
                                int B, int T, const int32_t *cu_q, const int32_t *q_pos,
                                const int64_t *kv_off, const int32_t *idx, int k, int H,
                                double sm_scale, double *out, double *lse)
{
    if (check_batch(B, T, cu_q, q_pos) || k < 1 || H < 1) return -1;
    for (int t = 0; t < T; t++)
        for (int i = 0; i < k; i++) {
            int32_t j = idx[(int64_t)t * k + i];
            if (j != -1 && (j < 0 || j > q_pos[t])) return -2;
        }
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int t = 0; t < T; t++)
        for (int h = 0; h < H; h++) {
            int b = seq_of(t, B, cu_q);
            int32_t *pos = malloc(sizeof(int32_t) * (size_t)k);
            int n = 0;
            for (int i = 0; i < k; i++) {
                int32_t j = idx[(int64_t)t * k + i];
                if (j >= 0) pos[n++] = j;
            }
            attend_rows_nope(q_lat + ((int64_t)t * H + h) * D_L, kv_latent, kv_off[b], pos, n, sm_scale,
                             out + ((int64_t)t * H + h) * D_L, lse ? lse + (int64_t)t * H + h : NULL);
            free(pos);
        }
    return 0;
}

int oracle_sparse_attn_nope(const uint16_t *q_lat, const uint16_t *kv_latent,
                            int B, int T, const int32_t *cu_q, const int32_t *q_pos,
                            const int64_t *kv_off, const int32_t *idx, int k, int H,
                            double sm_scale, double *out, double *lse)
{
    double *ql = bf16_array_to_f64(q_lat, (int64_t)T * H * D_L);
    int rc = ql ? oracle_sparse_attn_nope_f64(ql, kv_latent, B, T, cu_q, q_pos, kv_off, idx, k, H,
                                              sm_scale, out, lse)
                : -1;
    free(ql);
    return rc;
}

int oracle_dense_attn_f64(const double *q_lat, const double *q_rope, const uint16_t *kv_cache,
                          int B, int T, const int32_t *cu_q, const int32_t *q_pos,
                          const int64_t *kv_off, int H, double sm_scale,
                          double *out, double *lse)
{
    if (check_batch(B, T, cu_q, q_pos) || H < 1) return -1;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int t = 0; t < T; t++)
        for (int h = 0; h < H; h++) {
            int b = seq_of(t, B, cu_q);
            int n = q_pos[t] + 1;
            int32_t *pos = malloc(sizeof(int32_t) * (size_t)n);
            for (int s = 0; s < n; s++) pos[s] = s;
            attend_rows(q_lat + ((int64_t)t * H + h) * D_L, q_rope + ((int64_t)t * H + h) * D_R,
                        kv_cache, kv_off[b], pos, n, sm_scale,
                        out + ((int64_t)t * H + h) * D_L, lse ? lse + (int64_t)t * H + h : NULL);
            free(pos);
        }
    return 0;
}

int oracle_unabsorbed_attn(const double *q_nope, const double *q_rope, const uint16_t *kv_cache,
                           int B, int T, const int32_t *cu_q, const int32_t *q_pos,
                           const int64_t *kv_off, const double *W_UK, const double *W_UV,
                           const int32_t *idx, int k, int H, double sm_scale, double *out)
{
    enum { D_NOPE = 192, D_V = 256 };
    if (check_batch(B, T, cu_q, q_pos) || k < 1 || H < 1) return -1;
    for (int t = 0; t < T; t++) {
        int b = seq_of(t, B, cu_q);
        for (int h = 0; h < H; h++) {
            const double *qn = q_nope + ((int64_t)t * H + h) * D_NOPE;
            const double *qr = q_rope + ((int64_t)t * H + h) * D_R;
            const double *wk = W_UK + (int64_t)h * D_NOPE * D_L;
            const double *wv = W_UV + (int64_t)h * D_V * D_L;
            double *o = out + ((int64_t)t * H + h) * D_V;
            double *z = malloc(sizeof(double) * (size_t)k);
            double *v = malloc(sizeof(double) * (size_t)k * D_V);
            int n = 0;
            double m = -INFINITY;
            for (int i = 0; i < k; i++) {
                int32_t j = idx[(int64_t)t * k + i];
                if (j < 0) continue;
                if (j > q_pos[t]) { free(z); free(v); return -2; }
                const uint16_t *c = kv_cache + (kv_off[b] + j) * (int64_t)D_ROW;
                double lat[D_L];
                for (int d = 0; d < D_L; d++) lat[d] = oracle_bf16_to_f64(c[d]);
                double acc = 0.0;
                for (int e = 0; e < D_NOPE; e++) {          /* q_nope . (W_UK c) */
                    double kn = 0.0;
                    for (int d = 0; d < D_L; d++) kn += wk[(int64_t)e * D_L + d] * lat[d];
                    acc += qn[e] * kn;
                }
                for (int d = 0; d < D_R; d++) acc += qr[d] * oracle_bf16_to_f64(c[D_L + d]);
                for (int e = 0; e < D_V; e++) {             /* V = W_UV c */
                    double vv = 0.0;
                    for (int d = 0; d < D_L; d++) vv += wv[(int64_t)e * D_L + d] * lat[d];
                    v[(int64_t)n * D_V + e] = vv;
                }
                z[n] = sm_scale * acc;
                if (z[n] > m) m = z[n];
                n++;
            }
            for (int e = 0; e < D_V; e++) o[e] = 0.0;
            double l = 0.0;
            for (int j = 0; j < n; j++) {
                double p = exp(z[j] - m);
                l += p;
                for (int e = 0; e < D_V; e++) o[e] += p * v[(int64_t)j * D_V + e];
            }
            if (n) for (int e = 0; e < D_V; e++) o[e] /= l;
            free(z);
            free(v);
        }
    }
    return 0;
}

/* ---------------------------------------------------------------- the chain */

int oracle_decode(const void *k_new, int k_dtype, const uint16_t *q_idx, const float *w,
                  const uint16_t *q_lat, const uint16_t *q_rope,
                  uint16_t *k_cache, const uint16_t *kv_cache,
                  int B, int T, const int32_t *cu_q, const int32_t *q_pos, const int64_t *kv_off,
                  int H_I, int H, int k, double sm_scale, int hadamard,
                  double *scores, int64_t ld, int32_t *idx, double *out, double *lse)
{
    int rc = oracle_k_append(k_new, k_dtype, B, T, cu_q, q_pos, kv_off, k_cache, hadamard);
    if (!rc) rc = oracle_indexer_score(q_idx, w, k_cache, B, T, cu_q, q_pos, kv_off, H_I,
                                       hadamard, scores, ld);
    if (!rc) rc = oracle_topk(scores, ld, T, q_pos, k, idx);
    if (!rc) rc = oracle_sparse_attn(q_lat, q_rope, kv_cache, B, T, cu_q, q_pos, kv_off, idx,
                                     k, H, sm_scale, out, lse);
    return rc;
}

/* ---------------------------------------------------------------- kpool indexer */

int oracle_kpool_write_rows(const uint16_t *k_new, const uint16_t *gate_new, int B, int T,
                            const int32_t *cu_q, const int32_t *q_pos, const int64_t *kv_off,
                            uint16_t *rows)
{
    if (check_batch(B, T, cu_q, q_pos)) return -1;
    for (int t = 0; t < T; t++) {
        int b = seq_of(t, B, cu_q);
        uint16_t *r = rows + (kv_off[b] + q_pos[t]) * (int64_t)ORACLE_KPOOL_ROW;
        for (int d = 0; d < D_I; d++) {
            r[d] = k_new[(int64_t)t * D_I + d];
            r[D_I + d] = gate_new[(int64_t)t * D_I + d];
        }
        r[2 * D_I] = 0x3C00;                               /* valid = 1.0 */
    }
    return 0;
}

static int row_valid(const uint16_t *r) { return oracle_f16_to_f64(r[2 * D_I]) != 0.0; }

int oracle_kpool_pool_key(const uint16_t *seq_rows, int64_t j, const float *ape, uint16_t *key)
{
    const uint16_t *r[ORACLE_KPOOL];
    int any = 0;
    for (int i = 0; i < ORACLE_KPOOL; i++) {
        r[i] = seq_rows + (j * ORACLE_KPOOL + i) * (int64_t)ORACLE_KPOOL_ROW;
        any |= row_valid(r[i]);
    }
    if (!any) return 0;
    for (int d = 0; d < D_I; d++) {
        /* softmax over the valid positions of (gate + ape), max-subtracted */
        double e[ORACLE_KPOOL], m = -INFINITY;
        for (int i = 0; i < ORACLE_KPOOL; i++) {
            e[i] = oracle_f16_to_f64(r[i][D_I + d]) + (double)ape[i * D_I + d];
            if (row_valid(r[i]) && e[i] > m) m = e[i];
        }
        double den = 0.0, num = 0.0;
        for (int i = 0; i < ORACLE_KPOOL; i++) {
            if (!row_valid(r[i])) continue;
            double a = exp(e[i] - m);
            den += a;
            num += a * oracle_f16_to_f64(r[i][d]);
        }
        key[d] = oracle_f64_to_f16(num / den);
    }
    return 1;
}

int oracle_kpool_select(const uint16_t *q_idx, const float *w, const uint16_t *rows, const float *ape,
                        int B, int T, const int32_t *cu_q, const int32_t *q_pos, const int64_t *kv_off,
                        int H_I, int top_k, int32_t *idx, double *pool_scores, int64_t ld_pools)
{
    if (check_batch(B, T, cu_q, q_pos) || H_I < 1 || top_k < 1) return -1;
    const int kp = top_k / ORACLE_KPOOL;                   /* pools selected */
    const int width = kp * ORACLE_KPOOL + ORACLE_KPOOL - 1;
    for (int t = 0; t < T; t++)
        if (pool_scores && (q_pos[t] + 1) / ORACLE_KPOOL > ld_pools) return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; t++) {
        const int b = seq_of(t, B, cu_q);
        const int p = q_pos[t];
        const int n_pools = (p + 1) / ORACLE_KPOOL;        /* complete pools visible */
        const uint16_t *seq_rows = rows + kv_off[b] * (int64_t)ORACLE_KPOOL_ROW;
        cand_t *c = malloc(sizeof(cand_t) * (size_t)(n_pools > 0 ? n_pools : 1));
        uint16_t *keys = malloc(sizeof(uint16_t) * (size_t)(n_pools > 0 ? n_pools : 1) * D_I);
        if (!c || !keys) { bad = 1; free(c); free(keys); continue; }
        if (pool_scores)
            for (int64_t j = 0; j < ld_pools; j++) pool_scores[(int64_t)t * ld_pools + j] = -INFINITY;
        int n_c = 0;
        for (int j = 0; j < n_pools; j++) {
            uint16_t *key = keys + (size_t)j * D_I;
            if (!oracle_kpool_pool_key(seq_rows, j, ape, key)) continue;
            double I = 0.0;
            for (int h = 0; h < H_I; h++) {
                double dot = 0.0;
                for (int d = 0; d < D_I; d++)
                    dot += oracle_f16_to_f64(q_idx[((int64_t)t * H_I + h) * D_I + d]) * oracle_f16_to_f64(key[d]);
                I += (double)w[(int64_t)t * H_I + h] * (dot > 0.0 ? dot : 0.0);
            }
            if (pool_scores) pool_scores[(int64_t)t * ld_pools + j] = I;
            c[n_c].v = I;
            c[n_c].s = j;
            n_c++;
        }
        /* the best floor(top_k / 4) pools by (score desc, pool asc), in pool order */
        qsort(c, (size_t)n_c, sizeof(cand_t), by_score_desc_pos_asc);
        int m = n_c < kp ? n_c : kp;
        int32_t *sel = malloc(sizeof(int32_t) * (size_t)(m > 0 ? m : 1));
        if (!sel) { bad = 1; free(c); free(keys); continue; }
        for (int i = 0; i < m; i++) sel[i] = c[i].s;
        qsort(sel, (size_t)m, sizeof(int32_t), by_pos);
        int32_t *out = idx + (int64_t)t * width;
        int n = 0;
        for (int i = 0; i < m; i++)                        /* each pool's valid positions */
            for (int r = 0; r < ORACLE_KPOOL; r++) {
                const int s = sel[i] * ORACLE_KPOOL + r;
                if (row_valid(seq_rows + (int64_t)s * ORACLE_KPOOL_ROW)) out[n++] = s;
            }
        for (int s = n_pools * ORACLE_KPOOL; s <= p; s++)  /* the tail, always */
            if (row_valid(seq_rows + (int64_t)s * ORACLE_KPOOL_ROW)) out[n++] = s;
        for (; n < width; n++) out[n] = -1;
        free(sel);
        free(c);
        free(keys);
    }
    return bad ? -1 : 0;
}
