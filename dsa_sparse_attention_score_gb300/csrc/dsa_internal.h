// dsa_internal.h -- launchers shared between the kernel translation units and
// the C-ABI host layer.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "dsa.h"

namespace dsa {

// Launch with the programmatic-stream-serialization attribute when `pdl` is
// set: the kernel may start while its predecessor in the stream finishes and
// must call griddepcontrol.wait before reading the predecessor's output.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     bool pdl, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kSMs = 152;   // streaming multiprocessors of the target GPU

struct DevBatch {
    int B, T;
    int max_q, max_kv;
    int64_t cache_rows;
    const int32_t *cu_q;
    const int32_t *q_pos;
    const int64_t *kv_off;          // null with a block table
    unsigned long long *timeline;   // optional [2 * kTimelineSlots] start/end ns (tracing)
    // Paged caches: position pos of sequence seq lives at cache row
    // block_table[seq * max_blocks + pos / block_size] * block_size + pos % block_size.
    const int32_t *block_table;     // null: contiguous, row kv_off[seq] + pos
    int max_blocks, block_size;
    // Failure-path test hooks (dsa_set_test_faults): the limit of every
    // bounded wait, and whether the producers of the score and attention
    // kernels skip their copies so that the consumers' waits run out.
    uint64_t wait_ns;
    int skip_copies;
    // Pool mode (kpool indexer): the score and top-k kernels work on pools
    // of 2^pool_log2 positions -- a token at position p sees the complete
    // pools 0 .. ((p + 1) >> pool_log2) - 1 (none: -1, an empty row, not an
    // error) and sequence b's pools start at pool-cache row kv_off[b] >> pool_log2.
    int pool_log2;
};

// Cache row of position pos (0 <= pos < max_kv) of sequence seq, whose
// contiguous base is kv0 (unused with a block table); -1 for an unmapped
// block.
__device__ __forceinline__ int64_t cache_row(const DevBatch &b, int seq, int64_t kv0, int pos) {
    if (!b.block_table) return kv0 + pos;
    const int blk = __ldg(b.block_table + (int64_t)seq * b.max_blocks + pos / b.block_size);
    return blk < 0 ? -1 : (int64_t)blk * b.block_size + pos % b.block_size;
}
__device__ __forceinline__ int64_t seq_base(const DevBatch &b, int seq) {
    const int64_t kv0 = b.kv_off ? __ldg(b.kv_off + seq) : 0;
    return kv0 >> b.pool_log2;
}
// The last visible position (pool, in pool mode) of token t; -1 in pool mode
// when no pool is complete yet.
__device__ __forceinline__ int visible_last(const DevBatch &b, int t) {
    const int p = __ldg(b.q_pos + t);
    return b.pool_log2 ? ((p + 1) >> b.pool_log2) - 1 : p;
}
// A position that is out of range, as opposed to an empty row in pool mode.
__device__ __forceinline__ bool bad_last(const DevBatch &b, int last) {
    return b.pool_log2 ? last < -1 : last < 0;
}

// Tracing slots of the kernels (earliest CTA start, latest CTA end).
enum { kTlAppend = 0, kTlScore = 1, kTlTopk = 2, kTlAttn = 3, kTlCombine = 4, kTimelineSlots = 5 };

// Rows of a score/top-k slab: either one row per token (direct) or the rows
// (b, j - j0) of the local-token window [j0, j0 + J) of every sequence.
struct RowMap {
    int slab;     // 0 = direct (row = t), 1 = windowed
    int j0, J;
};

cudaError_t launch_k_append(const void *k_new, int k_dtype, const DevBatch &b, uint16_t *k_cache,
                            int hadamard, uint32_t *status, cudaStream_t stream);

// kpool indexer (GLM-5.3-Flash): packed rows k (128) | gate (128) | valid (1)
// of kKpoolRow fp16 values, pools of kKpool positions.
constexpr int kKpool = 4;
constexpr int kKpoolLog2 = 2;
constexpr int kKpoolRow = 257;
// phase 0 writes the tokens' packed rows (and, when `fused`, the pooled key
// of every pool a token completes); phase 1 writes only the pooled keys.
cudaError_t launch_kpool_append(const uint16_t *k_new, const uint16_t *gate_new, const float *ape,
                                const DevBatch &b, uint16_t *rows, uint16_t *pool_keys, int64_t pool_rows,
                                int phase, int fused, uint32_t *status, cudaStream_t stream);
// Selected pools (ascending, -1 padded, kp per token) -> token positions:
// each pool's valid positions, then the valid tail positions, -1 padded to width.
cudaError_t launch_kpool_expand(const int32_t *pool_idx, int kp, const uint16_t *rows, const DevBatch &b,
                                int width, int32_t *idx, uint32_t *status, cudaStream_t stream, bool pdl);
// In the launchers below `pdl` marks a launch that follows another kernel of
// the same call (programmatic dependent launch).

struct ScoreLaunch {
    const uint16_t *q_idx;   // fp16 [T, H_I, 128]
    const float *w;          // [T, H_I]
    int H_I;
    int hadamard_q;
    float *scores;           // [rows, ld]
    int64_t ld;
    int fill_masked;         // write -inf for visible-range complements up to ld
    RowMap rows;
    // What the preceding kernel of the same call wrote: 0 nothing this launch
    // reads or overwrites, 1 the tokens' own keys (the append), 2 anything
    // (a top-k still reading the score slab) -- then nothing starts before it ends.
    int depends;
    // Decode batches (one query token per sequence): the score kernel appends
    // each token's key itself instead of a separate append launch.
    int fuse_append;
    const void *k_new;       // [T, 128] of k_dtype
    int k_dtype;
    uint16_t *k_cache;       // written at the token's row
    int hadamard_k;
    // The kernel that follows is small: when this grid also fits in one wave,
    // trigger dependents at the start so that they fill the idle SMs.
    int early_ok;
};
cudaError_t launch_score(const ScoreLaunch &a, const CUtensorMap &k_map, const DevBatch &b,
                         uint32_t *status, cudaStream_t stream, bool pdl);

// n_sink > 0: the positions [a, a + n_sink) of each row's sequence are forced
// in, a = sink_pos0[seq] (device, [B]) or 0 when sink_pos0 is null.
cudaError_t launch_topk(const float *scores, int64_t ld, const DevBatch &b, RowMap rows, int k,
                        int32_t *idx, uint32_t *status, cudaStream_t stream, bool pdl, int n_sink = 0,
                        const int32_t *sink_pos0 = nullptr);

struct AttnLaunch {
    int rope = 1;            // 0: 512-wide latent rows without the rope tail
    const void *kv;          // the latent cache: [cache_rows, 576] (or 512) bf16
    int H, k;
    float sm_scale;
    const int32_t *idx;      // [T, k]
    float *out;              // [T, H, 512]
    float *lse;              // [T, H] or null
    int tiles_per_cta;       // attention row tiles handled by one CTA
    int n_split;             // CTAs per (token, head group)
    void *part_o;            // bf16 [T, n_split, groups*64, 512] when n_split > 1
    float *part_ml;          // [T, n_split, groups*64, 2]
};
cudaError_t launch_sparse_attn(const AttnLaunch &a, const CUtensorMap &q_lat_map,
                               const CUtensorMap &q_rope_map, const CUtensorMap &kv_map,
                               const DevBatch &b, uint32_t *status, cudaStream_t stream, bool pdl);
cudaError_t launch_attn_combine(const AttnLaunch &a, const DevBatch &b, cudaStream_t stream, bool pdl);

// Sets a kernel's dynamic shared-memory limit once per device; `slot`
// (0..kSmemAttrSlots-1) names the kernel instance.
constexpr int kSmemAttrSlots = 11;
cudaError_t ensure_smem_attr(const void *func, int slot, size_t bytes);

// Rows of one attention tile (the unit of the split across CTAs).
int attn_tile_rows();

// Shared-memory bytes of the attention kernel (for the host's occupancy set-up).
size_t sparse_attn_smem_bytes();
size_t score_smem_bytes(int n_rows, int hadamard_q, int n_stages);

}  // namespace dsa
