/*
 * dsa_oracle.h -- CPU reference of the DeepSeek Sparse Attention hot path.
 *
 * TEST INFRASTRUCTURE.  This is the slow, plain, double-precision definition
 * that the CUDA path is checked against.  Only the tests, the smoke check and
 * the benchmark's CPU-baseline leg may load it.  It shares no code, header or
 * table with the CUDA library and never calls it.
 *
 * All pointers are host pointers.  Storage formats: fp16 and bf16 values are
 * passed as uint16_t bit patterns; results are double.  Batch description:
 *   B sequences, T query tokens; cu_q[B+1] query offsets per sequence;
 *   q_pos[T] absolute position of each query inside its sequence;
 *   kv_off[B] first row of each sequence in the pooled caches.
 * A query at position p sees the keys at positions 0..p (inclusive).
 *
 * Every function returns 0 on success and a negative code on a bad argument
 * (-1 bad size, -2 index out of range).
 *
 * Parity: every function is pinned by tests under tests/test_oracle_*.py.
 */
#ifndef DSA_ORACLE_H
#define DSA_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Storage conversions (exact decode; encode rounds to nearest, ties to even). */
double   oracle_f16_to_f64(uint16_t h);
double   oracle_bf16_to_f64(uint16_t b);
uint16_t oracle_f64_to_f16(double x);

/* Orthonormal Walsh-Hadamard transform of length 128, Sylvester (natural)
 * order: y = H x / sqrt(128), H[i][j] = (-1)^popcount(i & j). */
void oracle_fwht128(const double *x, double *y);

/* Indexer-key append: row kv_off[b] + q_pos[t] of k_cache receives
 * fp16(hadamard ? H k / sqrt(128) : k).  k_dtype 0 = float32, 1 = fp16. */
int oracle_k_append(const void *k_new, int k_dtype, int B, int T,
                    const int32_t *cu_q, const int32_t *q_pos, const int64_t *kv_off,
                    uint16_t *k_cache, int hadamard);

/* Lightning-indexer score
 *   I(t,s) = sum_h w[t,h] * max(0, q'[t,h] . k[s])  for s <= q_pos[t],
 * -inf for q_pos[t] < s < ld.  q' = H q / sqrt(128) (unrounded) when
 * hadamard_q, else q.  q_idx fp16 [T,H_I,128], w float32 [T,H_I],
 * k_cache fp16 [rows,128], scores double [T,ld]. */
int oracle_indexer_score(const uint16_t *q_idx, const float *w, const uint16_t *k_cache,
                         int B, int T, const int32_t *cu_q, const int32_t *q_pos,
                         const int64_t *kv_off, int H_I, int hadamard_q,
                         double *scores, int64_t ld);

/* Top-k per query row over the visible positions 0..q_pos[t]: a full sort by
 * (score descending, position ascending), the first min(k, q_pos[t]+1)
 * positions kept, written in ascending order, the rest of the row padded
 * with -1.  idx int32 [T,k]. */
int oracle_topk(const double *scores, int64_t ld, int T, const int32_t *q_pos,
                int k, int32_t *idx);

/* Top-k with the attention sink forced in (ik_llama_opt commit log, "GLM-5.2
 * DSA indexer: decode-correct via persistent indexer-K cache" (attention-sink
 * force-inclusion), "per-sequence attention sink" and "UPDATE 6 --
 * serving-correctness"): before the selection, the first n_sink positions of
 * the row's own sequence, counted from the sequence's first present position
 * anchor[row] (0 when anchor is NULL), get a boost taken as unbounded: their
 * scores become +inf, so they rank first and tie among themselves by
 * position.  Then exactly oracle_topk.  anchor is given per ROW (the caller
 * maps each row to its sequence's anchor). */
int oracle_topk_sink(const double *scores, int64_t ld, int T, const int32_t *q_pos,
                     int k, int n_sink, const int32_t *anchor, int32_t *idx);

/* Sparse MLA attention in the absorbed (latent) form over the selected rows:
 *   z_j = sm_scale * (q_lat[t,h] . c_j[0:512] + q_rope[t,h] . c_j[512:576])
 *   o[t,h] = sum_j softmax(z)_j * c_j[0:512],  lse[t,h] = log sum_j exp(z_j)
 * over j in idx[t, 0:k) (entries -1 skipped; a row with no entry gives o = 0,
 * lse = -inf).  Inputs as double: q_lat [T,H,512], q_rope [T,H,64];
 * kv_cache bf16 [rows,576].  out double [T,H,512]; lse may be NULL. */
int oracle_sparse_attn_f64(const double *q_lat, const double *q_rope, const uint16_t *kv_cache,
                           int B, int T, const int32_t *cu_q, const int32_t *q_pos,
                           const int64_t *kv_off, const int32_t *idx, int k, int H,
                           double sm_scale, double *out, double *lse);

/* Same with bf16 queries (the CUDA path's input format). */
int oracle_sparse_attn(const uint16_t *q_lat, const uint16_t *q_rope, const uint16_t *kv_cache,
                       int B, int T, const int32_t *cu_q, const int32_t *q_pos,
                       const int64_t *kv_off, const int32_t *idx, int k, int H,
                       double sm_scale, double *out, double *lse);

/* MLA-NoPE sparse attention (vllm-rdna PR #2 "Glm5Next (GLM-5.3-Flash) on
 * gfx1030", DSA = MLA-NoPE: the 512-d kv latent is cached per token and no
 * RoPE is applied anywhere), in the absorbed (latent) form:
 *   z_j = sm_scale * q_lat[t,h] . c_j[0:512],
 *   o[t,h] = sum_j softmax(z)_j * c_j,  lse[t,h] = log sum_j exp(z_j)
 * over j in idx[t, 0:k) as for oracle_sparse_attn_f64.  kv_latent bf16
 * [rows,512]; q_lat double [T,H,512]; out double [T,H,512]; lse may be NULL. */
int oracle_sparse_attn_nope_f64(const double *q_lat, const uint16_t *kv_latent,
                                int B, int T, const int32_t *cu_q, const int32_t *q_pos,
                                const int64_t *kv_off, const int32_t *idx, int k, int H,
                                double sm_scale, double *out, double *lse);

/* Same with bf16 queries. */
int oracle_sparse_attn_nope(const uint16_t *q_lat, const uint16_t *kv_latent,
                            int B, int T, const int32_t *cu_q, const int32_t *q_pos,
                            const int64_t *kv_off, const int32_t *idx, int k, int H,
                            double sm_scale, double *out, double *lse);

/* Dense causal MLA attention (absorbed form): softmax over every s <= q_pos[t]. */
int oracle_dense_attn_f64(const double *q_lat, const double *q_rope, const uint16_t *kv_cache,
                          int B, int T, const int32_t *cu_q, const int32_t *q_pos,
                          const int64_t *kv_off, int H, double sm_scale,
                          double *out, double *lse);

/* Unabsorbed MLA attention over the selected rows (tiny sizes only): each
 * row's latent is expanded through the per-head up-projections,
 *   K_nope[h] = W_UK[h] c[0:512] (192), K_rope = c[512:576] (64),
 *   V[h] = W_UV[h] c[0:512] (256),
 *   z = sm_scale * (q_nope[h] . K_nope[h] + q_rope[h] . K_rope),
 *   out[t,h] = sum_j softmax(z)_j V_j[h].
 * q_nope double [T,H,192], q_rope double [T,H,64], W_UK double [H,192,512],
 * W_UV double [H,256,512], out double [T,H,256]. */
int oracle_unabsorbed_attn(const double *q_nope, const double *q_rope, const uint16_t *kv_cache,
                           int B, int T, const int32_t *cu_q, const int32_t *q_pos,
                           const int64_t *kv_off, const double *W_UK, const double *W_UV,
                           const int32_t *idx, int k, int H, double sm_scale, double *out);

/* The whole step: append -> score -> top-k -> attention, in that order.
 * k_cache is updated in place.  scores (double [T, ld]) and idx are outputs
 * the caller provides; lse may be NULL. */
int oracle_decode(const void *k_new, int k_dtype, const uint16_t *q_idx, const float *w,
                  const uint16_t *q_lat, const uint16_t *q_rope,
                  uint16_t *k_cache, const uint16_t *kv_cache,
                  int B, int T, const int32_t *cu_q, const int32_t *q_pos, const int64_t *kv_off,
                  int H_I, int H, int k, double sm_scale, int hadamard,
                  double *scores, int64_t ld, int32_t *idx, double *out, double *lse);

/* Threads used by the row loops (OpenMP); returns the count in effect. */
int oracle_set_threads(int n);

#ifdef __cplusplus
}
#endif
/* ---------------------------------------------------------------- kpool indexer
 * GLM-5.3-Flash (vllm-rdna PR #2 "Glm5Next (GLM-5.3-Flash) on gfx1030", the
 * DSA layer bullet): a kpool indexer (32 heads x 128, topk 2048, kpool 4,
 * always_select_tail, pool compression softmax(gate+ape), tail <= 3 ->
 * width 2051) whose cache holds packed indexer rows of 257 fp16 values,
 * k (128) | gate (128) | valid (1).  Reading taken (the page gives only this
 * outline):
 *  - pools are the aligned runs of 4 positions [4j, 4j+4) of a sequence; a
 *    pool is visible to a query at position p when 4j + 3 <= p; the tail is
 *    the positions 4*floor((p+1)/4) .. p (at most 3);
 *  - the pooled key of pool j, per dim d: softmax over the pool's valid rows
 *    i of (gate[4j+i][d] + ape[i][d]) weighting k[4j+i][d], rounded once to
 *    fp16 (ape: [4][128] position-in-pool embedding, a model parameter);
 *    a pool with no valid row has no key;
 *  - pool scores follow the indexer formula on the pooled keys (no rotation,
 *    no extra scale constant);
 *  - top_k counts tokens: the floor(top_k / 4) best pools by (score desc,
 *    pool asc) are expanded to their valid positions, the valid tail
 *    positions are always added, the list is ascending and padded with -1 to
 *    width 4*floor(top_k/4) + 3 (2051 for top_k = 2048).
 */
#define ORACLE_KPOOL 4
#define ORACLE_KPOOL_ROW 257

/* Packed rows k|gate|1.0 of the new tokens at kv_off[b] + q_pos[t]. */
int oracle_kpool_write_rows(const uint16_t *k_new, const uint16_t *gate_new, int B, int T,
                            const int32_t *cu_q, const int32_t *q_pos, const int64_t *kv_off,
                            uint16_t *rows);

/* Pooled key of pool j of the sequence whose packed rows start at seq_rows.
 * Returns 1 and writes key[128] (fp16 bits) when the pool has a valid row,
 * else returns 0 and leaves key untouched. */
int oracle_kpool_pool_key(const uint16_t *seq_rows, int64_t j, const float *ape, uint16_t *key);

/* Selection of every query token: idx [T, width] token positions (ascending,
 * -1 padded), width = 4*floor(top_k/4) + 3.  pool_scores (nullable)
 * [T, ld_pools] receives the pool scores (-inf for pools not visible or
 * without a key). */
int oracle_kpool_select(const uint16_t *q_idx, const float *w, const uint16_t *rows, const float *ape,
                        int B, int T, const int32_t *cu_q, const int32_t *q_pos, const int64_t *kv_off,
                        int H_I, int top_k, int32_t *idx, double *pool_scores, int64_t ld_pools);

#endif
