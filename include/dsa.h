/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DeepSeek Sparse Attention hot path.
 *
 * The path: an fp16 single-head indexer-key cache, the lightning-indexer
 * score I(t,s) = sum_h w[t,h] * ReLU(q_I[t,h] . k_I[s]) under the causal mask
 * s <= pos(t), a top-k selection of positions, and softmax attention of every
 * query head over only the selected rows of the 576-wide MLA latent cache
 * (512 latent + 64 rope tail), returning the 512-d latent output.
 *
 * Sources (page title, section):
 *  [IDX]  ik_llama_opt commit log (src/llama-context.h page), commit "Add
 *         GLM-5.2/DeepSeek-V3.2 DSA lightning indexer": the score formula,
 *         the causal mask, ggml_top_k(min(top_k, n_tokens)).
 *  [KC]   same page, commit "GLM-5.2 DSA indexer: decode-correct via
 *         persistent indexer-K cache": the [128, kv_size] fp16 single-head
 *         key cache written at the token's slot before scoring; the
 *         Walsh-Hadamard rotation of q and k applied before the fp16 store.
 *  [MLA]  ds4 PR #523 "hy3: Metal decode path + shared gate/up fusion",
 *         milestone M3: 576-wide cached rows (kv_a latent + rotated rope
 *         tail) and glm_mla_attention_one (scores over nope + rope parts,
 *         one softmax across the candidate rows, values from the latent).
 *  [ABS]  ik_llama_opt commit log, "MLA tensor parallelism under -sm graph":
 *         wk_b / wv_b absorbed weights, so attention runs on the latent and
 *         the value up-projection is applied by the caller.
 *  [OPS]  vllm-rdna PR #2 "Glm5Next (GLM-5.3-Flash) on gfx1030",
 *         "Prohibitions honored": out-arguments into caller buffers, no
 *         blocking device-to-host copy, capture-safe calls.
 *
 * Conventions shared by every entry point
 *  - Pointers named in the signatures are DEVICE pointers unless stated;
 *    the caller owns every buffer.  The library never allocates, frees or
 *    synchronises; all work is enqueued on `stream` (NULL = legacy default
 *    stream) and returns before it runs.  No call reads device memory on the
 *    host.  A call may be captured into a CUDA graph if the caller keeps
 *    the arguments alive.
 *  - Storage types: dsa_f16 is an IEEE binary16 bit pattern, dsa_bf16 a
 *    bfloat16 bit pattern.  All tensors are dense, row-major, contiguous.
 *  - Fixed dims: indexer head dim 128, latent 512, rope tail 64, row 576.
 *    Supported: 1 <= H_I <= 64 indexer heads, 1 <= H <= 128 query heads
 *    (DeepSeek-V3.2, the other model the indexer commit names, has 128),
 *    1 <= k <= 65536.  Others return DSA_ERR_UNSUPPORTED.
 *  - Device pointers passed to the TMA engine (k_cache, kv_cache, q_lat,
 *    q_rope) must be 16-byte aligned, else DSA_ERR_MISALIGNED.
 *  - The attention results (out, lse) are written with plain stores and
 *    never read back, so they may also be pinned host memory that the
 *    driver maps into the device's address space at the same address
 *    (cuPointerGetAttribute reports the host address as its device pointer,
 *    as on NVLink-C2C systems): the result then reaches the host without a
 *    separate copy.  Whether a pointer is so mapped is the caller's to
 *    check; the library does not inspect pointers.
 *  - Host validation runs before anything is enqueued; a failing call
 *    enqueues nothing.  A failed launch returns DSA_ERR_CUDA.
 *  - Device-detected problems (a position outside the stated bounds, an
 *    index out of range, a bounded wait that gave up, shared memory that is
 *    not aligned as a kernel laid it out) never trap: the kernel
 *    skips the offending work, ORs a DSA_DEV_* bit into the status word at
 *    the start of the workspace and carries on.  dsa_read_device_status
 *    reads and clears it.
 *  - Inputs must be finite; NaN or Inf inputs give unspecified results.
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t dsa_f16;
typedef uint16_t dsa_bf16;

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARGUMENT = 1,   /* null pointer, bad size, bad enum */
    DSA_ERR_UNSUPPORTED = 2,        /* a dimension outside the supported set */
    DSA_ERR_MISALIGNED = 3,         /* a TMA-read pointer not 16-byte aligned */
    DSA_ERR_WORKSPACE_TOO_SMALL = 4,
    DSA_ERR_CUDA = 5,               /* a CUDA runtime call or launch failed */
    DSA_ERR_DEVICE = 6              /* dsa_read_device_status found DSA_DEV_* bits */
} dsa_status_t;

/* Bits of the device status word. */
enum {
    DSA_DEV_BAD_POSITION = 1u << 0, /* q_pos / kv_off / cu_q outside the stated bounds */
    DSA_DEV_BAD_INDEX    = 1u << 1, /* an idx entry not in {-1} U [0, q_pos[t]] */
    DSA_DEV_TIMEOUT      = 1u << 2, /* a bounded wait on an mbarrier gave up */
    DSA_DEV_SMEM_LAYOUT  = 1u << 3  /* a kernel found its shared memory not 1024-byte aligned (work skipped) */
};

/* dtype of new indexer keys */
enum { DSA_KEY_F32 = 0, DSA_KEY_F16 = 1 };

/* operations for dsa_workspace_size */
enum {
    DSA_OP_K_APPEND = 0,
    DSA_OP_INDEXER_SCORE = 1,
    DSA_OP_TOPK = 2,
    DSA_OP_SPARSE_ATTN = 3,
    DSA_OP_DECODE = 4,
    DSA_OP_KPOOL = 5          /* dsa_kpool_select and dsa_decode_kpool (k = top_k) */
};

/*
 * Variable-length batch.  B sequences, T query tokens in total; the tokens
 * of sequence b are t = cu_q[b] .. cu_q[b+1]-1.  Token t sits at absolute
 * position q_pos[t] within its sequence and sees the positions 0..q_pos[t]
 * (the inclusive causal mask of [IDX]).  Sequence b owns rows
 * kv_off[b] + s of both pooled caches (indexer keys and latent rows).
 * The host fields are upper bounds used to size grids and must hold:
 *   cu_q[b+1] - cu_q[b] <= max_q_per_seq,  q_pos[t] + 1 <= max_kv,
 *   kv_off[b] + q_pos[t] < cache_rows.
 * Positions are device data on purpose: a captured graph replays with new
 * positions without being rebuilt.
 */
typedef struct {
    int32_t batch;            /* B >= 1 (host) */
    int32_t total_q;          /* T >= 1 (host) */
    int32_t max_q_per_seq;    /* host upper bound, >= 1 */
    int32_t max_kv;           /* host upper bound of visible positions, >= 1 */
    int64_t cache_rows;       /* host: rows of each pooled cache */
    const int32_t *cu_q;      /* device [B+1], cu_q[0] = 0, cu_q[B] = T */
    const int32_t *q_pos;     /* device [T] */
    const int64_t *kv_off;    /* device [B] */
} dsa_batch_t;

/*
 * Indexer-key append ([KC]).  For every token t, writes
 *   k_cache[kv_off[b] + q_pos[t], :] = fp16_rne(hadamard ? H k_new[t] / sqrt(128) : k_new[t])
 * where H is the 128x128 Sylvester (natural order) Hadamard matrix.  The
 * rotation is exact before the single rounding to fp16.
 *   k_new    [T,128] float32 (k_dtype DSA_KEY_F32) or fp16 (DSA_KEY_F16)
 *   k_cache  [cache_rows,128] fp16, updated in place (only the T rows)
 *   ws       at least dsa_workspace_size(DSA_OP_K_APPEND) bytes (status word)
 */
dsa_status_t dsa_indexer_k_append(const void *k_new, int k_dtype, const dsa_batch_t *batch,
                                  dsa_f16 *k_cache, int hadamard,
                                  void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Lightning-indexer score, unfused ([IDX]; rotation per [KC]).
 *   scores[t, s] = sum_h w[t,h] * max(0, q'[t,h] . k_cache[kv_off[b]+s])   for s <= q_pos[t]
 *   scores[t, s] = -INFINITY                                               for q_pos[t] < s < ld_scores
 * with q' = H q_idx[t,h] / sqrt(128) when hadamard_q (the keys in the cache
 * are then expected rotated too), else q' = q_idx.  Products are formed
 * from fp16 operands and accumulated in float32; with hadamard_q the rotated
 * query is carried as two fp16 parts (hi + lo) so it keeps ~22 bits.
 *   q_idx   [T,H_I,128] fp16      w [T,H_I] float32
 *   k_cache [cache_rows,128] fp16 scores [T, ld_scores] float32, ld_scores >= max_kv
 * Materialises the whole score matrix: meant for tests and small batches.
 */
dsa_status_t dsa_indexer_score(const dsa_f16 *q_idx, const float *w, const dsa_f16 *k_cache,
                               const dsa_batch_t *batch, int H_I, int hadamard_q,
                               float *scores, int64_t ld_scores,
                               void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Top-k selection ([IDX]: ggml_top_k(min(top_k, n))).  For every token t the
 * positions s in 0..q_pos[t] are ranked by (scores[t,s] descending,
 * s ascending); -0.0 ranks equal to +0.0.  The first min(k, q_pos[t]+1) are
 * written to idx[t, :] in ascending order of s, the remainder is -1.  The
 * selected set is exact: bit-for-bit the same as a full sort of the given
 * float32 values.
 *   scores [T, ld_scores] float32 (only the visible prefix of each row is read)
 *   idx    [T, k] int32 (sequence-local positions)
 */
dsa_status_t dsa_topk(const float *scores, int64_t ld_scores, const dsa_batch_t *batch, int k,
                      int32_t *idx, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Top-k with the attention sink forced in ([SINK]: ik_llama_opt commit log,
 * "GLM-5.2 DSA indexer: per-sequence attention sink" and "UPDATE 6 --
 * serving-correctness": the first n_sink keys of the query's own sequence,
 * counted from the sequence's first present position, get a +1e20 boost
 * before the argsort so they always survive).  Here the boost is unbounded:
 * for token t of sequence b the positions [a_b, a_b + n_sink) within
 * [0, q_pos[t]] rank above every score and tie with one another (lower
 * position first); the rest of the selection is dsa_topk's.
 *   n_sink     >= 0 (0: exactly dsa_topk)
 *   sink_pos0  device int32 [B], a_b = max(0, sink_pos0[b]); NULL means a_b = 0
 * Errors: n_sink < 0 -> DSA_ERR_INVALID_ARGUMENT; sink_pos0 not 4-byte
 * aligned -> DSA_ERR_MISALIGNED; otherwise as dsa_topk.
 */
dsa_status_t dsa_topk_sink(const float *scores, int64_t ld_scores, const dsa_batch_t *batch, int k, int n_sink,
                           const int32_t *sink_pos0, int32_t *idx, void *ws, size_t ws_bytes,
                           cudaStream_t stream);

/*
 * Sparse MLA attention in the absorbed form ([MLA], [ABS]).  For token t and
 * head h, over the selected rows c_j = kv_cache[kv_off[b] + idx[t,j]]:
 *   z_j      = sm_scale * (q_lat[t,h] . c_j[0:512] + q_rope[t,h] . c_j[512:576])
 *   out[t,h] = sum_j softmax(z)_j * c_j[0:512]
 *   lse[t,h] = log(sum_j exp(z_j))                (natural log)
 * Entries idx = -1 are skipped; a token with no valid entry gets out = 0 and
 * lse = -INFINITY.  Entries outside [0, q_pos[t]] are skipped and flagged.
 *   q_lat [T,H,512] bf16, q_rope [T,H,64] bf16, kv_cache [cache_rows,576] bf16
 *   idx [T,k] int32, out [T,H,512] float32, lse [T,H] float32 or NULL
 * bf16 operands, float32 accumulation and softmax; the probabilities enter the
 * value product as bf16.
 */
dsa_status_t dsa_sparse_mla_attn(const dsa_bf16 *q_lat, const dsa_bf16 *q_rope,
                                 const dsa_bf16 *kv_cache, const dsa_batch_t *batch,
                                 const int32_t *idx, int k, int H, float sm_scale,
                                 float *out, float *lse, void *ws, size_t ws_bytes,
                                 cudaStream_t stream);

/*
 * MLA-NoPE sparse attention: vllm-rdna PR #2 "Glm5Next (GLM-5.3-Flash) on
 * gfx1030", whose DSA layers cache the 512-d kv latent per token and apply no
 * RoPE anywhere.  As dsa_sparse_mla_attn without the rope tail:
 *   z_j      = sm_scale * q_lat[t,h] . c_j,   c_j = kv_latent[kv_off[b] + idx[t,j]]
 *   out[t,h] = sum_j softmax(z)_j * c_j,  lse[t,h] = log(sum_j exp(z_j))
 *   q_lat [T,H,512] bf16, kv_latent [cache_rows,512] bf16 (1024-byte rows)
 * Everything else (idx, out, lse, workspace DSA_OP_SPARSE_ATTN, errors) as
 * dsa_sparse_mla_attn.
 */
dsa_status_t dsa_sparse_mla_attn_nope(const dsa_bf16 *q_lat, const dsa_bf16 *kv_latent,
                                      const dsa_batch_t *batch, const int32_t *idx, int k, int H,
                                      float sm_scale, float *out, float *lse, void *ws, size_t ws_bytes,
                                      cudaStream_t stream);

/*
 * The fused step ([IDX], [KC], [MLA]): append the new indexer keys, score
 * every query against its visible keys, select the top-k positions and
 * attend over them -- in that stream order, so each token's own key is in
 * the cache before scoring.  Decode (one token per sequence) and prefill
 * chunks (many tokens of a sequence) use the same call.  Scores are kept in
 * the workspace in slabs of query rows and never returned.
 *   k_new [T,128] (k_dtype), q_idx [T,H_I,128] fp16, w [T,H_I] float32,
 *   q_lat [T,H,512] bf16, q_rope [T,H,64] bf16,
 *   k_cache [cache_rows,128] fp16 (updated), kv_cache [cache_rows,576] bf16
 *   (already holding every row the queries can see, including their own),
 *   out [T,H,512] float32, lse [T,H] float32 or NULL, idx_out [T,k] int32 or NULL.
 * hadamard rotates both the appended keys and the queries.
 */
dsa_status_t dsa_decode(const void *k_new, int k_dtype, const dsa_f16 *q_idx, const float *w,
                        const dsa_bf16 *q_lat, const dsa_bf16 *q_rope,
                        dsa_f16 *k_cache, const dsa_bf16 *kv_cache,
                        const dsa_batch_t *batch, int H_I, int H, int k, float sm_scale,
                        int hadamard, float *out, float *lse, int32_t *idx_out,
                        void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Paged caches ([PAGE]: vllm-rdna PR #2 "Glm5Next (GLM-5.3-Flash) on
 * gfx1030": the latent cache and the indexer cache are two paged attention
 * groups of the serving engine, and the DSA backend gathers the selected
 * latents through the page table).  Position pos of sequence b is cache row
 *   block_table[b * max_blocks + pos / block_size] * block_size + pos % block_size
 * of both k_cache and kv_cache.
 *   block_table  device int32 [B, max_blocks]; entries of blocks a sequence
 *                does not reach are never read past max_kv; a negative
 *                entry marks an unmapped block (positions there are
 *                flagged DSA_DEV_BAD_POSITION / DSA_DEV_BAD_INDEX)
 *   block_size   a multiple of 64 (tiles load as 64-row halves unless it is
 *                a multiple of 128)
 *   max_blocks   >= ceil(max_kv / block_size)
 */
typedef struct {
    const int32_t *block_table;
    int32_t max_blocks;
    int32_t block_size;
} dsa_paging_t;

/*
 * dsa_decode over paged caches (see dsa_paging_t).  batch->kv_off is not
 * read (it may be NULL); batch->cache_rows is the row count of both pooled
 * caches.  Errors as dsa_decode, plus DSA_ERR_INVALID_ARGUMENT for a null
 * paging, a null block table, a block size that is not a positive multiple
 * of 64, or max_blocks * block_size < max_kv, and DSA_ERR_MISALIGNED for a
 * block table that is not 4-byte aligned.
 */
dsa_status_t dsa_decode_paged(const void *k_new, int k_dtype, const dsa_f16 *q_idx, const float *w,
                              const dsa_bf16 *q_lat, const dsa_bf16 *q_rope, dsa_f16 *k_cache,
                              const dsa_bf16 *kv_cache, const dsa_batch_t *batch, const dsa_paging_t *paging,
                              int H_I, int H, int k, float sm_scale, int hadamard, float *out, float *lse,
                              int32_t *idx_out, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * dsa_decode with the attention sink forced into every token's selection
 * ([SINK], as dsa_topk_sink: n_sink >= 0, sink_pos0 device int32 [B] or
 * NULL).  Same workspace, outputs and errors as dsa_decode.
 */
dsa_status_t dsa_decode_sink(const void *k_new, int k_dtype, const dsa_f16 *q_idx, const float *w,
                             const dsa_bf16 *q_lat, const dsa_bf16 *q_rope, dsa_f16 *k_cache,
                             const dsa_bf16 *kv_cache, const dsa_batch_t *batch, int H_I, int H, int k,
                             float sm_scale, int hadamard, int n_sink, const int32_t *sink_pos0, float *out,
                             float *lse, int32_t *idx_out, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * dsa_decode without a workspace, for callers that cannot allocate device
 * memory (a plugin inside a framework that owns all device allocations, code
 * running under stream capture where an allocation would break the capture,
 * an embedder with a memory budget fixed up front).  The paper has no
 * counterpart: this is an integration aid, not a step of the method.
 *
 * Arguments, results and errors are those of dsa_decode; the scratch that
 * dsa_decode would take from `ws` comes from a static 64 MiB device array
 * inside the library instead.  Every GPU that loads the library holds that
 * array until the process exits.  This call allocates nothing and calls no
 * allocating routine.
 *  - Limit: a batch whose dsa_workspace_size(DSA_OP_DECODE, ...) exceeds
 *    64 MiB (67108864 bytes) is refused with DSA_ERR_WORKSPACE_TOO_SMALL
 *    before anything touches the device.  Decode batches fit (for example
 *    8 sequences x 8192 positions, or 32 sequences of up to 65536 positions,
 *    top-2048); long prefill chunks need dsa_decode with a caller workspace.
 *  - Set-up: the first call on a device, with that device current, looks up
 *    the array's device address and clears its status block on `stream`.
 *    Make that first call before any stream capture.
 *  - Sharing: every call uses the same array and leaves its contents behind;
 *    calls whose work overlaps on the GPU (different streams without an
 *    ordering between them) race on it and must not be issued.
 *  - Device-side status bits of these calls accumulate in the array and are
 *    not reported; offending work is still skipped, never trapped.
 *  - The array's address is looked up once per device and kept: resetting a
 *    device (cudaDeviceReset) after the first call on it is not supported.
 */
dsa_status_t dsa_decode_noalloc(const void *k_new, int k_dtype, const dsa_f16 *q_idx, const float *w,
                                const dsa_bf16 *q_lat, const dsa_bf16 *q_rope,
                                dsa_f16 *k_cache, const dsa_bf16 *kv_cache,
                                const dsa_batch_t *batch, int H_I, int H, int k, float sm_scale,
                                int hadamard, float *out, float *lse, int32_t *idx_out,
                                cudaStream_t stream);

/*
 * kpool indexer of GLM-5.3-Flash (vllm-rdna PR #2 "Glm5Next (GLM-5.3-Flash)
 * on gfx1030", DSA layer bullet: kpool indexer 32h x 128, topk 2048, kpool 4,
 * always_select_tail, pool compression softmax(gate+ape), tail <= 3 -> width
 * 2051; two cache groups per DSA layer: the 512-wide latent and packed
 * indexer rows of 257 = k|gate|valid).  Reading taken where the page is only
 * an outline:
 *  - pools are the aligned runs of 4 positions [4j, 4j+4) of a sequence; a
 *    token at position p sees the complete pools j <= (p+1)/4 - 1; its tail
 *    is the positions 4*floor((p+1)/4) .. p (at most 3);
 *  - pooled key of pool j, per dim d: the softmax over the pool's valid rows
 *    i of (gate[4j+i][d] + ape[i][d]) weighting k[4j+i][d], rounded once to
 *    fp16 (computed in float64);
 *  - pools are scored by the indexer formula on their pooled keys (no
 *    rotation, no extra constant);
 *  - top_k counts tokens: the floor(top_k/4) best pools by (score desc, pool
 *    asc) are expanded to their valid positions and the valid tail positions
 *    always added, ascending, -1 padded to width 4*floor(top_k/4) + 3 (2051
 *    for top_k = 2048); the attention is the MLA-NoPE one over those rows.
 * Caches:
 *  idx_rows   fp16 [cache_rows, 257] (row stride 514 bytes): k (128) |
 *             gate (128) | valid (1; 0.0 = absent row, anything else =
 *             present); position s of sequence b at row kv_off[b] + s
 *  pool_keys  fp16 [pool_rows, 128]: pool j of sequence b at row
 *             kv_off[b]/4 + j; kv_off[b] must be a multiple of 4 and
 *             pool_rows * 4 >= max_kv (else DSA_ERR_INVALID_ARGUMENT; a
 *             kv_off that is not a multiple of 4 is flagged
 *             DSA_DEV_BAD_POSITION and its tokens skipped)
 *  ape        float32 [4, 128], the position-in-pool embedding
 * Supported: 1 <= top_k <= 4096, 1 <= H_I <= 64, 1 <= H <= 128.
 */

/*
 * Appends the tokens' packed rows (k_new | gate_new | 1.0 at kv_off[b] +
 * q_pos[t]) and writes the pooled key of every pool a token completes
 * (position = 3 mod 4), from the pool's rows as they are after the append.
 *   k_new, gate_new  fp16 [T, 128] (16-byte aligned)
 *   ws               at least dsa_workspace_size(DSA_OP_K_APPEND) bytes
 */
dsa_status_t dsa_kpool_append(const dsa_f16 *k_new, const dsa_f16 *gate_new, const float *ape,
                              const dsa_batch_t *batch, dsa_f16 *idx_rows, dsa_f16 *pool_keys, int64_t pool_rows,
                              void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * The kpool selection of every token: scores of its complete pools (the
 * indexer formula on pool_keys, q_idx [T,H_I,128] fp16, w [T,H_I] float32),
 * the floor(top_k/4) best pools, expanded with the tail into positions:
 *   idx   int32 [T, 4*floor(top_k/4) + 3], ascending, -1 padded
 * Selected sets follow the tie rule of dsa_topk on float32 pool scores.
 */
dsa_status_t dsa_kpool_select(const dsa_f16 *q_idx, const float *w, const dsa_f16 *idx_rows,
                              const dsa_f16 *pool_keys, int64_t pool_rows, const dsa_batch_t *batch, int H_I,
                              int top_k, int32_t *idx, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * The fused GLM-5.3-Flash DSA step: dsa_kpool_append, dsa_kpool_select and
 * MLA-NoPE attention (as dsa_sparse_mla_attn_nope) over the selected
 * positions of kv_latent [cache_rows, 512] bf16, in that stream order.
 *   q_lat [T,H,512] bf16, out [T,H,512] float32, lse [T,H] or NULL,
 *   idx_out [T, 4*floor(top_k/4) + 3] int32 or NULL
 * Workspace: dsa_workspace_size(DSA_OP_KPOOL, batch, H_I, H, top_k).
 */
dsa_status_t dsa_decode_kpool(const dsa_f16 *k_new, const dsa_f16 *gate_new, const float *ape,
                              const dsa_f16 *q_idx, const float *w, const dsa_bf16 *q_lat, dsa_f16 *idx_rows,
                              dsa_f16 *pool_keys, int64_t pool_rows, const dsa_bf16 *kv_latent,
                              const dsa_batch_t *batch, int H_I, int H, int top_k, float sm_scale, float *out,
                              float *lse, int32_t *idx_out, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Workspace bytes an operation needs for this batch (host only; batch
 * pointers are not read).  Every workspace starts with the 256-byte status
 * block; call dsa_workspace_init once on a new workspace.
 */
dsa_status_t dsa_workspace_size(int op, const dsa_batch_t *batch, int H_I, int H, int k,
                                size_t *bytes);

/*
 * Number of kernels one dsa_decode call enqueues for this batch (host only;
 * batch pointers are not read).  For launch accounting and tracing.
 */
dsa_status_t dsa_decode_launches(const dsa_batch_t *batch, int H_I, int H, int k, int *launches);

/* Zeroes the status block (enqueued on stream). */
dsa_status_t dsa_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Synchronises `stream`, copies the status word to *flags and clears it.
 * Returns DSA_ERR_DEVICE when any DSA_DEV_* bit was set, else DSA_OK.
 * This is the only call that synchronises; it is for tests and debugging.
 */
dsa_status_t dsa_read_device_status(void *ws, cudaStream_t stream, uint32_t *flags);

/* Static description of a status code. */
const char *dsa_status_string(dsa_status_t status);

/*
 * Profiling hook (not thread-safe).  When set, dsa_decode records
 * events[0..n) on its stream at stage boundaries: before the append, the
 * first score launch, the first top-k launch, the attention and the combine,
 * and after the last launch (6 events).  Calls that score in several
 * windows of query tokens also record events[6 + 2j] and events[7 + 2j]
 * just before and after the top-k launch of window j (when j < (n - 6) / 2).
 * Slots left unrecorded keep their previous timestamp.  n = 0 or
 * events = NULL disables it.
 */
dsa_status_t dsa_set_trace_events(cudaEvent_t *events, int n);

/*
 * Tracing hook (not thread-safe).  When dev_buf is a device buffer of 10
 * uint64 values, every kernel the library launches afterwards records the
 * globaltimer (ns) of its earliest CTA start into dev_buf[2*i] (atomic min)
 * and of its latest CTA end into dev_buf[2*i+1] (atomic max), i = 0 append,
 * 1 score, 2 top-k, 3 attention, 4 combine.  The caller initialises the
 * slots (start slots to UINT64_MAX, end slots to 0).  Unlike trace events
 * this leaves the launch order and overlap untouched.  NULL disables it.
 */
dsa_status_t dsa_set_timeline(void *dev_buf);

/*
 * Failure-path test hook (not thread-safe; for tests only).  Every bounded
 * wait in the kernels launched afterwards gives up after wait_limit_ns
 * nanoseconds (0 restores the default of one second).  With skip_copies set,
 * the producers of the score and attention kernels issue no copies at all,
 * so their consumers' first waits run out: the kernels then set
 * DSA_DEV_TIMEOUT, free their tensor memory and return, with nothing in
 * flight, and the context stays usable.  Outputs of such calls are
 * unspecified; the status word reports the timeout.  This exercises the
 * same code a real stall (a copy that never lands) would take, without
 * faulting or hanging the GPU.
 */
dsa_status_t dsa_set_test_faults(uint64_t wait_limit_ns, int skip_copies);

/* Library version, major * 10000 + minor * 100 + patch. */
int dsa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H */
