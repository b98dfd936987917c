// dsa_api.cu -- the C ABI declared in include/dsa.h: argument validation,
// workspace layout, TMA tensor maps and the launch order of each call.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "dsa_common.cuh"
#include "dsa_internal.h"

using namespace dsa;

namespace {

constexpr int kVersion = 10100;  // 1.1.0
constexpr size_t kAlign = 256;
constexpr int64_t kSlabBytes = int64_t(1) << 30;  // score slab budget in the workspace

cudaEvent_t *g_trace = nullptr;
int g_trace_n = 0;
unsigned long long *g_timeline = nullptr;
uint64_t g_wait_ns = kWaitLimitNs;    // failure-path test hooks (dsa_set_test_faults)
int g_skip_copies = 0;

constexpr int kMaxHeads = 128;        // query heads: one or two groups of 64 per token
constexpr int kMaxSplit = 128;        // split partials the combine kernel merges
constexpr int kKpoolMaxTopK = 4096;   // kpool: 1024 pools per token (the expansion's slots)

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

dsa_status_t check_batch(const dsa_batch_t *b, bool paged = false) {
    if (!b) return DSA_ERR_INVALID_ARGUMENT;
    if (b->batch < 1 || b->total_q < 1 || b->max_q_per_seq < 1 || b->max_kv < 1 || b->cache_rows < 1)
        return DSA_ERR_INVALID_ARGUMENT;
    if (b->cache_rows > INT32_MAX || (int64_t)b->batch * b->max_q_per_seq < b->total_q)
        return DSA_ERR_INVALID_ARGUMENT;
    if (!b->cu_q || !b->q_pos || (!b->kv_off && !paged)) return DSA_ERR_INVALID_ARGUMENT;
    return DSA_OK;
}

DevBatch dev_batch(const dsa_batch_t *b) {
    DevBatch d;
    d.B = b->batch;
    d.T = b->total_q;
    d.max_q = b->max_q_per_seq;
    d.max_kv = b->max_kv;
    d.cache_rows = b->cache_rows;
    d.cu_q = b->cu_q;
    d.q_pos = b->q_pos;
    d.kv_off = b->kv_off;
    d.timeline = g_timeline;
    d.block_table = nullptr;
    d.max_blocks = 0;
    d.block_size = 0;
    d.wait_ns = g_wait_ns;
    d.skip_copies = g_skip_copies;
    d.pool_log2 = 0;
    return d;
}

// ---------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D row-major tensor [rows, cols] of 16-bit elements, SWIZZLE_128B boxes.
bool make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t cols, uint64_t rows,
              uint32_t box_cols, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- workspace
struct Layout {
    size_t status = 0;
    size_t scores = 0, scores_bytes = 0;
    size_t idx = 0, idx_bytes = 0;
    size_t pool_idx = 0;      // kpool: selected pools [T, top_k / 4]
    size_t part_o = 0, part_o_bytes = 0;
    size_t part_ml = 0, part_ml_bytes = 0;
    size_t total = 0;
    int J = 0;            // slab window (local tokens per sequence)
    int64_t ld = 0;       // slab row stride (floats)
    int n_split = 1, tiles_per_cta = 1;
};

inline int head_groups(int H) { return (H + 63) / 64; }

// Splits of a token's selected rows across CTAs: with fewer (token, head
// group) pairs than SMs, up to one wave of CTAs (one per SM), each keeping at
// least two tiles so that its gathers overlap its arithmetic, and never more
// splits than the combine kernel merges.
void attn_split(int T, int H, int k, int *n_split, int *tpc) {
    const int n_tiles = (k + attn_tile_rows() - 1) / attn_tile_rows();
    const int64_t units = (int64_t)T * head_groups(H);
    int ns = 1;
    if (units < kSMs) ns = std::max(1, std::min((n_tiles + 1) / 2, (int)(kSMs / units)));
    ns = std::min(ns, kMaxSplit);
    int t = (n_tiles + ns - 1) / ns;
    ns = (n_tiles + t - 1) / t;
    *n_split = ns;
    *tpc = t;
}

// kpool: pools selected per token and the width of a token's position list.
inline int kpool_pools(int top_k) { return top_k / kKpool; }
inline int kpool_width(int top_k) { return kpool_pools(top_k) * kKpool + kKpool - 1; }

Layout layout(int op, const dsa_batch_t *b, int H, int k) {
    Layout L;
    size_t off = kStatusBytes;
    if (op == DSA_OP_KPOOL) {
        // score slab over pools, the selected pools, the expanded positions,
        // then the attention's split partials over those positions
        const int max_pools = std::max(1, b->max_kv / kKpool);
        L.ld = (int64_t)align_up((size_t)max_pools, 4);
        const int64_t row_bytes = L.ld * 4;
        int64_t J = std::max<int64_t>(1, kSlabBytes / (row_bytes * b->batch));
        L.J = (int)std::min<int64_t>(J, b->max_q_per_seq);
        L.scores = off;
        L.scores_bytes = (size_t)b->batch * L.J * row_bytes;
        off = align_up(off + L.scores_bytes, kAlign);
        L.pool_idx = off;
        off = align_up(off + (size_t)b->total_q * std::max(1, kpool_pools(k)) * 4, kAlign);
        L.idx = off;
        L.idx_bytes = (size_t)b->total_q * kpool_width(k) * 4;
        off = align_up(off + L.idx_bytes, kAlign);
        k = kpool_width(k);                          // the attention runs over the positions
    }
    if (op == DSA_OP_DECODE) {
        L.ld = (int64_t)align_up((size_t)b->max_kv, 4);
        const int64_t row_bytes = L.ld * 4;
        int64_t J = std::max<int64_t>(1, kSlabBytes / (row_bytes * b->batch));
        L.J = (int)std::min<int64_t>(J, b->max_q_per_seq);
        L.scores = off;
        L.scores_bytes = (size_t)b->batch * L.J * row_bytes;
        off = align_up(off + L.scores_bytes, kAlign);
        L.idx = off;
        L.idx_bytes = (size_t)b->total_q * k * 4;
        off = align_up(off + L.idx_bytes, kAlign);
    }
    if (op == DSA_OP_DECODE || op == DSA_OP_SPARSE_ATTN || op == DSA_OP_KPOOL) {
        attn_split(b->total_q, H, k, &L.n_split, &L.tiles_per_cta);
        if (L.n_split > 1) {
            const size_t rows = (size_t)b->total_q * L.n_split * head_groups(H) * 64;
            L.part_o = off;
            L.part_o_bytes = rows * D_L * 2;           // bf16
            off = align_up(off + L.part_o_bytes, kAlign);
            L.part_ml = off;
            L.part_ml_bytes = rows * 2 * 4;
            off = align_up(off + L.part_ml_bytes, kAlign);
        }
    }
    L.total = off;
    return L;
}

inline uint32_t *status_ptr(void *ws) { return reinterpret_cast<uint32_t *>(ws); }

dsa_status_t check_ws(void *ws, size_t ws_bytes, size_t need) {
    if (!ws) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned(ws, kAlign)) return DSA_ERR_MISALIGNED;
    if (ws_bytes < need) return DSA_ERR_WORKSPACE_TOO_SMALL;
    return DSA_OK;
}

// Inside a stream capture a plain event record only orders the graph; an
// external record node makes every replay record the event.
inline void trace(int i, cudaStream_t s) {
    if (!(g_trace && i < g_trace_n && g_trace[i])) return;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) cs = cudaStreamCaptureStatusNone;
    cudaEventRecordWithFlags(g_trace[i], s,
                             cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault);
}

#define DSA_TRY_CUDA(x)                      \
    do {                                     \
        if ((x) != cudaSuccess) return DSA_ERR_CUDA; \
    } while (0)

dsa_status_t run_attention(const dsa_bf16 *q_lat, const dsa_bf16 *q_rope, const dsa_bf16 *kv_cache,
                           const dsa_batch_t *batch, const int32_t *idx, int k, int H, float sm_scale,
                           float *out, float *lse, void *ws, const Layout &L, cudaStream_t stream,
                           bool traced, bool pdl, const dsa_paging_t *paging = nullptr, bool rope = true) {
    DevBatch db = dev_batch(batch);
    if (paging) {
        db.block_table = paging->block_table;
        db.max_blocks = paging->max_blocks;
        db.block_size = paging->block_size;
    }
    CUtensorMap ql, qr, kv;
    const uint64_t qrows = (uint64_t)batch->total_q * H;
    // without the rope tail the latent rows are D_L wide and the kernel never
    // reads the rope-query map (it gets the latent one)
    if (!make_map(&ql, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q_lat, D_L, qrows, 64, 64) ||
        !make_map(&qr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rope ? q_rope : q_lat, rope ? D_R : D_L, qrows, 64, 64) ||
        !make_map(&kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kv_cache, rope ? D_ROW : D_L,
                  (uint64_t)batch->cache_rows, 64, 1))
        return DSA_ERR_CUDA;
    AttnLaunch a{};
    a.rope = rope ? 1 : 0;
    a.kv = kv_cache;
    a.H = H;
    a.k = k;
    a.sm_scale = sm_scale;
    a.idx = idx;
    a.out = out;
    a.lse = lse;
    a.n_split = L.n_split;
    a.tiles_per_cta = L.tiles_per_cta;
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    a.part_o = L.n_split > 1 ? static_cast<void *>(w8 + L.part_o) : nullptr;
    a.part_ml = L.n_split > 1 ? reinterpret_cast<float *>(w8 + L.part_ml) : nullptr;
    DSA_TRY_CUDA(launch_sparse_attn(a, ql, qr, kv, db, status_ptr(ws), stream, pdl));
    if (traced) trace(4, stream);
    DSA_TRY_CUDA(launch_attn_combine(a, db, stream, true));
    return DSA_OK;
}

}  // namespace

namespace dsa {
cudaError_t ensure_smem_attr(const void *func, int slot, size_t bytes) {
    static std::mutex mu;
    static bool done[kSmemAttrSlots][64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || slot < 0 || slot >= kSmemAttrSlots) return cudaErrorInvalidValue;
    std::lock_guard<std::mutex> lock(mu);
    if (done[slot][dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) done[slot][dev] = true;
    return e;
}
}  // namespace dsa

extern "C" {

const char *dsa_status_string(dsa_status_t s) {
    switch (s) {
        case DSA_OK: return "ok";
        case DSA_ERR_INVALID_ARGUMENT: return "invalid argument";
        case DSA_ERR_UNSUPPORTED: return "unsupported dimension";
        case DSA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case DSA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case DSA_ERR_CUDA: return "CUDA error";
        case DSA_ERR_DEVICE: return "device reported an error in the status word";
    }
    return "unknown status";
}

int dsa_version(void) { return kVersion; }

dsa_status_t dsa_set_trace_events(cudaEvent_t *events, int n) {
    if (n < 0) return DSA_ERR_INVALID_ARGUMENT;
    g_trace = (n > 0) ? events : nullptr;
    g_trace_n = (events && n > 0) ? n : 0;
    return DSA_OK;
}

dsa_status_t dsa_set_timeline(void *dev_buf) {
    g_timeline = static_cast<unsigned long long *>(dev_buf);
    return DSA_OK;
}

dsa_status_t dsa_set_test_faults(uint64_t wait_limit_ns, int skip_copies) {
    g_wait_ns = wait_limit_ns ? wait_limit_ns : kWaitLimitNs;
    g_skip_copies = skip_copies ? 1 : 0;
    return DSA_OK;
}

dsa_status_t dsa_workspace_size(int op, const dsa_batch_t *batch, int H_I, int H, int k, size_t *bytes) {
    (void)H_I;
    if (!bytes || op < DSA_OP_K_APPEND || op > DSA_OP_KPOOL) return DSA_ERR_INVALID_ARGUMENT;
    if (!batch || batch->batch < 1 || batch->total_q < 1 || batch->max_q_per_seq < 1 || batch->max_kv < 1)
        return DSA_ERR_INVALID_ARGUMENT;
    if ((op == DSA_OP_TOPK || op == DSA_OP_SPARSE_ATTN || op == DSA_OP_DECODE) && (k < 1 || k > 65536))
        return DSA_ERR_UNSUPPORTED;
    if (op == DSA_OP_KPOOL && (k < 1 || k > kKpoolMaxTopK)) return DSA_ERR_UNSUPPORTED;
    if ((op == DSA_OP_SPARSE_ATTN || op == DSA_OP_DECODE || op == DSA_OP_KPOOL) && (H < 1 || H > kMaxHeads))
        return DSA_ERR_UNSUPPORTED;
    *bytes = layout(op, batch, H, k).total;
    return DSA_OK;
}

dsa_status_t dsa_decode_launches(const dsa_batch_t *batch, int H_I, int H, int k, int *launches) {
    (void)H_I;
    if (!launches || !batch || batch->batch < 1 || batch->total_q < 1 || batch->max_q_per_seq < 1 ||
        batch->max_kv < 1)
        return DSA_ERR_INVALID_ARGUMENT;
    if (k < 1 || k > 65536 || H < 1 || H > kMaxHeads) return DSA_ERR_UNSUPPORTED;
    const Layout L = layout(DSA_OP_DECODE, batch, H, k);
    const int slabs = (batch->max_q_per_seq + L.J - 1) / L.J;
    const bool combine = L.n_split > 1;
    *launches = (batch->max_q_per_seq == 1 ? 0 : 1) + 2 * slabs + 1 + (combine ? 1 : 0);
    return DSA_OK;
}

dsa_status_t dsa_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream) {
    dsa_status_t s = check_ws(ws, ws_bytes, kStatusBytes);
    if (s != DSA_OK) return s;
    DSA_TRY_CUDA(cudaMemsetAsync(ws, 0, kStatusBytes, stream));
    return DSA_OK;
}

dsa_status_t dsa_read_device_status(void *ws, cudaStream_t stream, uint32_t *flags) {
    if (!ws || !flags) return DSA_ERR_INVALID_ARGUMENT;
    uint32_t v = 0;
    DSA_TRY_CUDA(cudaStreamSynchronize(stream));
    DSA_TRY_CUDA(cudaMemcpy(&v, ws, sizeof v, cudaMemcpyDeviceToHost));
    DSA_TRY_CUDA(cudaMemset(ws, 0, sizeof v));
    *flags = v;
    return v ? DSA_ERR_DEVICE : DSA_OK;
}

dsa_status_t dsa_indexer_k_append(const void *k_new, int k_dtype, const dsa_batch_t *batch,
                                  dsa_f16 *k_cache, int hadamard, void *ws, size_t ws_bytes,
                                  cudaStream_t stream) {
    dsa_status_t s = check_batch(batch);
    if (s != DSA_OK) return s;
    if (!k_new || !k_cache || (k_dtype != DSA_KEY_F32 && k_dtype != DSA_KEY_F16))
        return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned(k_new, 16) || !aligned(k_cache, 16)) return DSA_ERR_MISALIGNED;
    if ((s = check_ws(ws, ws_bytes, kStatusBytes)) != DSA_OK) return s;
    DSA_TRY_CUDA(launch_k_append(k_new, k_dtype, dev_batch(batch), k_cache, hadamard != 0,
                                 status_ptr(ws), stream));
    return DSA_OK;
}

dsa_status_t dsa_indexer_score(const dsa_f16 *q_idx, const float *w, const dsa_f16 *k_cache,
                               const dsa_batch_t *batch, int H_I, int hadamard_q, float *scores,
                               int64_t ld_scores, void *ws, size_t ws_bytes, cudaStream_t stream) {
    dsa_status_t s = check_batch(batch);
    if (s != DSA_OK) return s;
    if (!q_idx || !w || !k_cache || !scores) return DSA_ERR_INVALID_ARGUMENT;
    if (H_I < 1 || H_I > 64) return DSA_ERR_UNSUPPORTED;
    if (ld_scores < batch->max_kv) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned(k_cache, 16) || !aligned(q_idx, 16) || !aligned(w, 4) || !aligned(scores, 4))
        return DSA_ERR_MISALIGNED;
    if ((s = check_ws(ws, ws_bytes, kStatusBytes)) != DSA_OK) return s;
    CUtensorMap km;
    if (!make_map(&km, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, k_cache, D_I, (uint64_t)batch->cache_rows, 64, 128))
        return DSA_ERR_CUDA;
    ScoreLaunch a{};
    a.q_idx = q_idx;
    a.w = w;
    a.H_I = H_I;
    a.hadamard_q = hadamard_q != 0;
    a.scores = scores;
    a.ld = ld_scores;
    a.fill_masked = 1;
    a.rows = RowMap{0, 0, batch->max_q_per_seq};
    DSA_TRY_CUDA(launch_score(a, km, dev_batch(batch), status_ptr(ws), stream, false));
    return DSA_OK;
}

static dsa_status_t topk_impl(const float *scores, int64_t ld_scores, const dsa_batch_t *batch, int k,
                              int n_sink, const int32_t *sink_pos0, int32_t *idx, void *ws, size_t ws_bytes,
                              cudaStream_t stream) {
    dsa_status_t s = check_batch(batch);
    if (s != DSA_OK) return s;
    if (!scores || !idx) return DSA_ERR_INVALID_ARGUMENT;
    if (k < 1 || k > 65536) return DSA_ERR_UNSUPPORTED;
    if (ld_scores < batch->max_kv) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned(scores, 4) || !aligned(idx, 4)) return DSA_ERR_MISALIGNED;
    if ((s = check_ws(ws, ws_bytes, kStatusBytes)) != DSA_OK) return s;
    if (n_sink < 0) return DSA_ERR_INVALID_ARGUMENT;
    if (sink_pos0 && !aligned(sink_pos0, 4)) return DSA_ERR_MISALIGNED;
    DSA_TRY_CUDA(launch_topk(scores, ld_scores, dev_batch(batch), RowMap{0, 0, 1}, k, idx,
                             status_ptr(ws), stream, false, n_sink, sink_pos0));
    return DSA_OK;
}

dsa_status_t dsa_topk(const float *scores, int64_t ld_scores, const dsa_batch_t *batch, int k,
                      int32_t *idx, void *ws, size_t ws_bytes, cudaStream_t stream) {
    return topk_impl(scores, ld_scores, batch, k, 0, nullptr, idx, ws, ws_bytes, stream);
}

dsa_status_t dsa_topk_sink(const float *scores, int64_t ld_scores, const dsa_batch_t *batch, int k, int n_sink,
                           const int32_t *sink_pos0, int32_t *idx, void *ws, size_t ws_bytes,
                           cudaStream_t stream) {
    return topk_impl(scores, ld_scores, batch, k, n_sink, sink_pos0, idx, ws, ws_bytes, stream);
}

dsa_status_t dsa_sparse_mla_attn_nope(const dsa_bf16 *q_lat, const dsa_bf16 *kv_latent,
                                      const dsa_batch_t *batch, const int32_t *idx, int k, int H,
                                      float sm_scale, float *out, float *lse, void *ws, size_t ws_bytes,
                                      cudaStream_t stream) {
    dsa_status_t s = check_batch(batch);
    if (s != DSA_OK) return s;
    if (!q_lat || !kv_latent || !idx || !out) return DSA_ERR_INVALID_ARGUMENT;
    if (H < 1 || H > kMaxHeads || k < 1 || k > 65536) return DSA_ERR_UNSUPPORTED;
    if ((int64_t)batch->total_q * H > INT32_MAX) return DSA_ERR_UNSUPPORTED;
    if (!aligned(q_lat, 16) || !aligned(kv_latent, 16) || !aligned(out, 16) || !aligned(idx, 4) ||
        (lse && !aligned(lse, 4)))
        return DSA_ERR_MISALIGNED;
    const Layout L = layout(DSA_OP_SPARSE_ATTN, batch, H, k);
    if ((s = check_ws(ws, ws_bytes, L.total)) != DSA_OK) return s;
    return run_attention(q_lat, nullptr, kv_latent, batch, idx, k, H, sm_scale, out, lse, ws, L, stream,
                         false, false, nullptr, false);
}

dsa_status_t dsa_sparse_mla_attn(const dsa_bf16 *q_lat, const dsa_bf16 *q_rope, const dsa_bf16 *kv_cache,
                                 const dsa_batch_t *batch, const int32_t *idx, int k, int H,
                                 float sm_scale, float *out, float *lse, void *ws, size_t ws_bytes,
                                 cudaStream_t stream) {
    dsa_status_t s = check_batch(batch);
    if (s != DSA_OK) return s;
    if (!q_lat || !q_rope || !kv_cache || !idx || !out) return DSA_ERR_INVALID_ARGUMENT;
    if (H < 1 || H > kMaxHeads || k < 1 || k > 65536) return DSA_ERR_UNSUPPORTED;
    if ((int64_t)batch->total_q * H > INT32_MAX) return DSA_ERR_UNSUPPORTED;
    if (!aligned(q_lat, 16) || !aligned(q_rope, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) ||
        !aligned(idx, 4) || (lse && !aligned(lse, 4)))
        return DSA_ERR_MISALIGNED;
    const Layout L = layout(DSA_OP_SPARSE_ATTN, batch, H, k);
    if ((s = check_ws(ws, ws_bytes, L.total)) != DSA_OK) return s;
    return run_attention(q_lat, q_rope, kv_cache, batch, idx, k, H, sm_scale, out, lse, ws, L, stream,
                         false, false);
}

static dsa_status_t decode_impl(const void *k_new, int k_dtype, const dsa_f16 *q_idx, const float *w,
                                const dsa_bf16 *q_lat, const dsa_bf16 *q_rope, dsa_f16 *k_cache,
                                const dsa_bf16 *kv_cache, const dsa_batch_t *batch, int H_I, int H, int k,
                                float sm_scale, int hadamard, int n_sink, const int32_t *sink_pos0, float *out,
                                float *lse, int32_t *idx_out, void *ws, size_t ws_bytes, cudaStream_t stream,
                                const dsa_paging_t *paging = nullptr) {
    dsa_status_t s = check_batch(batch, paging != nullptr);
    if (s != DSA_OK) return s;
    if (paging) {
        if (!paging->block_table || paging->block_size < 64 || paging->block_size % 64 != 0 ||
            (int64_t)paging->max_blocks * paging->block_size < batch->max_kv)
            return DSA_ERR_INVALID_ARGUMENT;
        if (!aligned(paging->block_table, 4)) return DSA_ERR_MISALIGNED;
    }
    if (n_sink < 0) return DSA_ERR_INVALID_ARGUMENT;
    if (sink_pos0 && !aligned(sink_pos0, 4)) return DSA_ERR_MISALIGNED;
    if (!k_new || !q_idx || !w || !q_lat || !q_rope || !k_cache || !kv_cache || !out)
        return DSA_ERR_INVALID_ARGUMENT;
    if (k_dtype != DSA_KEY_F32 && k_dtype != DSA_KEY_F16) return DSA_ERR_INVALID_ARGUMENT;
    if (H_I < 1 || H_I > 64 || H < 1 || H > kMaxHeads || k < 1 || k > 65536) return DSA_ERR_UNSUPPORTED;
    if ((int64_t)batch->total_q * H > INT32_MAX) return DSA_ERR_UNSUPPORTED;
    if (!aligned(k_new, 16) || !aligned(q_idx, 16) || !aligned(w, 4) || !aligned(q_lat, 16) ||
        !aligned(q_rope, 16) || !aligned(k_cache, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) ||
        (lse && !aligned(lse, 4)) || (idx_out && !aligned(idx_out, 4)))
        return DSA_ERR_MISALIGNED;
    const Layout L = layout(DSA_OP_DECODE, batch, H, k);
    if ((s = check_ws(ws, ws_bytes, L.total)) != DSA_OK) return s;

    DevBatch db = dev_batch(batch);
    if (paging) {
        db.block_table = paging->block_table;
        db.max_blocks = paging->max_blocks;
        db.block_size = paging->block_size;
    }
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    uint32_t *st = status_ptr(ws);
    float *slab = reinterpret_cast<float *>(w8 + L.scores);
    int32_t *idx = idx_out ? idx_out : reinterpret_cast<int32_t *>(w8 + L.idx);
    CUtensorMap km;
    // paged caches with blocks that are not a multiple of a 128-key tile
    // load each tile as two 64-row halves
    const uint32_t key_box_rows = (paging && paging->block_size % 128 != 0) ? 64 : 128;
    if (!make_map(&km, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, k_cache, D_I, (uint64_t)batch->cache_rows, 64, key_box_rows))
        return DSA_ERR_CUDA;

    // Decode batches (one query token per sequence) append inside the score
    // kernel; batches with several tokens per sequence append first.
    const bool fuse_append = batch->max_q_per_seq == 1;
    trace(0, stream);
    if (!fuse_append)
        DSA_TRY_CUDA(launch_k_append(k_new, k_dtype, db, k_cache, hadamard != 0, st, stream));
    for (int j0 = 0, win = 0; j0 < batch->max_q_per_seq; j0 += L.J, ++win) {
        ScoreLaunch a{};
        a.q_idx = q_idx;
        a.w = w;
        a.H_I = H_I;
        a.hadamard_q = hadamard != 0;
        a.scores = slab;
        a.ld = L.ld;
        a.fill_masked = 0;
        a.rows = RowMap{1, j0, L.J};
        a.depends = fuse_append ? 0 : (j0 == 0 ? 1 : 2);
        a.fuse_append = fuse_append;
        a.k_new = k_new;
        a.k_dtype = k_dtype;
        a.k_cache = k_cache;
        a.hadamard_k = hadamard != 0;
        // decode: the top-k that follows runs one small CTA group per sequence
        a.early_ok = fuse_append && (int64_t)batch->batch * ((batch->max_kv + 8191) / 8192) <= kSMs / 4;
        if (j0 == 0) trace(1, stream);
        DSA_TRY_CUDA(launch_score(a, km, db, st, stream, !(fuse_append && j0 == 0)));
        if (j0 == 0) trace(2, stream);
        trace(6 + 2 * win, stream);
        DSA_TRY_CUDA(launch_topk(slab, L.ld, db, a.rows, k, idx, st, stream, true, n_sink, sink_pos0));
        trace(7 + 2 * win, stream);
    }
    trace(3, stream);
    s = run_attention(q_lat, q_rope, kv_cache, batch, idx, k, H, sm_scale, out, lse, ws, L, stream, true, true,
                      paging);
    if (L.n_split <= 1) trace(4, stream);
    trace(5, stream);
    return s;
}

dsa_status_t dsa_decode(const void *k_new, int k_dtype, const dsa_f16 *q_idx, const float *w,
                        const dsa_bf16 *q_lat, const dsa_bf16 *q_rope, dsa_f16 *k_cache,
                        const dsa_bf16 *kv_cache, const dsa_batch_t *batch, int H_I, int H, int k,
                        float sm_scale, int hadamard, float *out, float *lse, int32_t *idx_out, void *ws,
                        size_t ws_bytes, cudaStream_t stream) {
    return decode_impl(k_new, k_dtype, q_idx, w, q_lat, q_rope, k_cache, kv_cache, batch, H_I, H, k, sm_scale,
                       hadamard, 0, nullptr, out, lse, idx_out, ws, ws_bytes, stream);
}

dsa_status_t dsa_decode_paged(const void *k_new, int k_dtype, const dsa_f16 *q_idx, const float *w,
                              const dsa_bf16 *q_lat, const dsa_bf16 *q_rope, dsa_f16 *k_cache,
                              const dsa_bf16 *kv_cache, const dsa_batch_t *batch, const dsa_paging_t *paging,
                              int H_I, int H, int k, float sm_scale, int hadamard, float *out, float *lse,
                              int32_t *idx_out, void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!paging) return DSA_ERR_INVALID_ARGUMENT;
    return decode_impl(k_new, k_dtype, q_idx, w, q_lat, q_rope, k_cache, kv_cache, batch, H_I, H, k, sm_scale,
                       hadamard, 0, nullptr, out, lse, idx_out, ws, ws_bytes, stream, paging);
}

dsa_status_t dsa_decode_sink(const void *k_new, int k_dtype, const dsa_f16 *q_idx, const float *w,
                             const dsa_bf16 *q_lat, const dsa_bf16 *q_rope, dsa_f16 *k_cache,
                             const dsa_bf16 *kv_cache, const dsa_batch_t *batch, int H_I, int H, int k,
                             float sm_scale, int hadamard, int n_sink, const int32_t *sink_pos0, float *out,
                             float *lse, int32_t *idx_out, void *ws, size_t ws_bytes, cudaStream_t stream) {
    return decode_impl(k_new, k_dtype, q_idx, w, q_lat, q_rope, k_cache, kv_cache, batch, H_I, H, k, sm_scale,
                       hadamard, n_sink, sink_pos0, out, lse, idx_out, ws, ws_bytes, stream);
}


// ---------------------------------------------------------------- kpool indexer

static dsa_status_t check_kpool_cache(const dsa_batch_t *batch, const dsa_f16 *idx_rows, const dsa_f16 *pool_keys,
                                      int64_t pool_rows) {
    if (!idx_rows || !pool_keys) return DSA_ERR_INVALID_ARGUMENT;
    if (pool_rows < 1 || pool_rows > INT32_MAX || pool_rows * kKpool < batch->max_kv) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned(idx_rows, 2) || !aligned(pool_keys, 16)) return DSA_ERR_MISALIGNED;
    return DSA_OK;
}

// The batch as the score and top-k kernels see it in pool mode.
static DevBatch pool_batch(const dsa_batch_t *batch, int64_t pool_rows) {
    DevBatch pb = dev_batch(batch);
    pb.pool_log2 = kKpoolLog2;
    pb.max_kv = std::max(1, batch->max_kv / kKpool);
    pb.cache_rows = pool_rows;
    return pb;
}

// Score windows of pools, their top-k, then the expansion into positions.
static dsa_status_t kpool_select_impl(const dsa_f16 *q_idx, const float *w, const dsa_f16 *idx_rows,
                                      const dsa_f16 *pool_keys, int64_t pool_rows, const dsa_batch_t *batch, int H_I,
                                      int top_k, int32_t *idx, void *ws, const Layout &L, cudaStream_t stream,
                                      bool after_append) {
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    uint32_t *st = status_ptr(ws);
    const int kp = kpool_pools(top_k);
    int32_t *pool_idx = reinterpret_cast<int32_t *>(w8 + L.pool_idx);
    const DevBatch pb = pool_batch(batch, pool_rows);
    bool pdl = after_append;
    if (kp > 0) {
        CUtensorMap km;
        if (!make_map(&km, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, pool_keys, D_I, (uint64_t)pool_rows, 64, 128))
            return DSA_ERR_CUDA;
        float *slab = reinterpret_cast<float *>(w8 + L.scores);
        for (int j0 = 0; j0 < batch->max_q_per_seq; j0 += L.J) {
            ScoreLaunch a{};
            a.q_idx = q_idx;
            a.w = w;
            a.H_I = H_I;
            a.scores = slab;
            a.ld = L.ld;
            a.rows = RowMap{1, j0, L.J};
            // the append wrote only each token's own last pool: with one token
            // per sequence the older pools' tiles need not wait for it
            a.depends = after_append ? (j0 == 0 ? 1 : 2) : (j0 == 0 ? 0 : 2);
            // one token per sequence: the top-k that follows is small
            a.early_ok = batch->max_q_per_seq == 1 &&
                         (int64_t)batch->batch * ((pb.max_kv + 8191) / 8192) <= kSMs / 4;
            DSA_TRY_CUDA(launch_score(a, km, pb, st, stream, pdl || j0 > 0));
            DSA_TRY_CUDA(launch_topk(slab, L.ld, pb, a.rows, kp, pool_idx, st, stream, true));
            pdl = true;
        }
    }
    DSA_TRY_CUDA(launch_kpool_expand(pool_idx, kp, idx_rows, dev_batch(batch), kpool_width(top_k), idx, st, stream,
                                     pdl));
    return DSA_OK;
}

dsa_status_t dsa_kpool_append(const dsa_f16 *k_new, const dsa_f16 *gate_new, const float *ape,
                              const dsa_batch_t *batch, dsa_f16 *idx_rows, dsa_f16 *pool_keys, int64_t pool_rows,
                              void *ws, size_t ws_bytes, cudaStream_t stream) {
    dsa_status_t s = check_batch(batch);
    if (s != DSA_OK) return s;
    if (!k_new || !gate_new || !ape) return DSA_ERR_INVALID_ARGUMENT;
    if ((s = check_kpool_cache(batch, idx_rows, pool_keys, pool_rows)) != DSA_OK) return s;
    if (!aligned(k_new, 16) || !aligned(gate_new, 16) || !aligned(ape, 4)) return DSA_ERR_MISALIGNED;
    if ((s = check_ws(ws, ws_bytes, kStatusBytes)) != DSA_OK) return s;
    const DevBatch db = dev_batch(batch);
    const bool fused = batch->max_q_per_seq == 1;   // one token per sequence: rows and keys in one pass
    DSA_TRY_CUDA(launch_kpool_append(k_new, gate_new, ape, db, idx_rows, pool_keys, pool_rows, 0, fused ? 1 : 0,
                                     status_ptr(ws), stream));
    if (!fused)
        DSA_TRY_CUDA(launch_kpool_append(k_new, gate_new, ape, db, idx_rows, pool_keys, pool_rows, 1, 0,
                                         status_ptr(ws), stream));
    return DSA_OK;
}

dsa_status_t dsa_kpool_select(const dsa_f16 *q_idx, const float *w, const dsa_f16 *idx_rows,
                              const dsa_f16 *pool_keys, int64_t pool_rows, const dsa_batch_t *batch, int H_I,
                              int top_k, int32_t *idx, void *ws, size_t ws_bytes, cudaStream_t stream) {
    dsa_status_t s = check_batch(batch);
    if (s != DSA_OK) return s;
    if (!q_idx || !w || !idx) return DSA_ERR_INVALID_ARGUMENT;
    if (H_I < 1 || H_I > 64 || top_k < 1 || top_k > kKpoolMaxTopK) return DSA_ERR_UNSUPPORTED;
    if ((s = check_kpool_cache(batch, idx_rows, pool_keys, pool_rows)) != DSA_OK) return s;
    if (!aligned(q_idx, 16) || !aligned(w, 4) || !aligned(idx, 4)) return DSA_ERR_MISALIGNED;
    const Layout L = layout(DSA_OP_KPOOL, batch, 64, top_k);
    if ((s = check_ws(ws, ws_bytes, L.total)) != DSA_OK) return s;
    return kpool_select_impl(q_idx, w, idx_rows, pool_keys, pool_rows, batch, H_I, top_k, idx, ws, L, stream, false);
}

dsa_status_t dsa_decode_kpool(const dsa_f16 *k_new, const dsa_f16 *gate_new, const float *ape,
                              const dsa_f16 *q_idx, const float *w, const dsa_bf16 *q_lat, dsa_f16 *idx_rows,
                              dsa_f16 *pool_keys, int64_t pool_rows, const dsa_bf16 *kv_latent,
                              const dsa_batch_t *batch, int H_I, int H, int top_k, float sm_scale, float *out,
                              float *lse, int32_t *idx_out, void *ws, size_t ws_bytes, cudaStream_t stream) {
    dsa_status_t s = check_batch(batch);
    if (s != DSA_OK) return s;
    if (!k_new || !gate_new || !ape || !q_idx || !w || !q_lat || !kv_latent || !out) return DSA_ERR_INVALID_ARGUMENT;
    if (H_I < 1 || H_I > 64 || H < 1 || H > kMaxHeads || top_k < 1 || top_k > kKpoolMaxTopK)
        return DSA_ERR_UNSUPPORTED;
    if ((int64_t)batch->total_q * H > INT32_MAX) return DSA_ERR_UNSUPPORTED;
    if ((s = check_kpool_cache(batch, idx_rows, pool_keys, pool_rows)) != DSA_OK) return s;
    if (!aligned(k_new, 16) || !aligned(gate_new, 16) || !aligned(ape, 4) || !aligned(q_idx, 16) ||
        !aligned(w, 4) || !aligned(q_lat, 16) || !aligned(kv_latent, 16) || !aligned(out, 16) ||
        (lse && !aligned(lse, 4)) || (idx_out && !aligned(idx_out, 4)))
        return DSA_ERR_MISALIGNED;
    const Layout L = layout(DSA_OP_KPOOL, batch, H, top_k);
    if ((s = check_ws(ws, ws_bytes, L.total)) != DSA_OK) return s;
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    int32_t *idx = idx_out ? idx_out : reinterpret_cast<int32_t *>(w8 + L.idx);
    const DevBatch db = dev_batch(batch);
    const bool fused = batch->max_q_per_seq == 1;
    DSA_TRY_CUDA(launch_kpool_append(k_new, gate_new, ape, db, idx_rows, pool_keys, pool_rows, 0, fused ? 1 : 0,
                                     status_ptr(ws), stream));
    if (!fused)
        DSA_TRY_CUDA(launch_kpool_append(k_new, gate_new, ape, db, idx_rows, pool_keys, pool_rows, 1, 0,
                                         status_ptr(ws), stream));
    if ((s = kpool_select_impl(q_idx, w, idx_rows, pool_keys, pool_rows, batch, H_I, top_k, idx, ws, L, stream,
                               true)) != DSA_OK)
        return s;
    return run_attention(q_lat, nullptr, kv_latent, batch, idx, kpool_width(top_k), H, sm_scale, out, lse, ws, L,
                         stream, false, true, nullptr, false);
}

}  // extern "C"
