// kpool.cu -- the GLM-5.3-Flash kpool indexer cache and the expansion of
// selected pools into token positions.
//
// vllm-rdna PR #2 "Glm5Next (GLM-5.3-Flash) on gfx1030", DSA layer bullet: a
// kpool indexer (32 heads x 128, topk 2048, kpool 4, always_select_tail, pool
// compression softmax(gate+ape), tail <= 3 -> width 2051) over packed indexer
// rows of 257 values, k | gate | valid.  Reading: pools are the aligned runs
// of 4 positions; the pooled key of a pool is, per dim d, the softmax over
// its valid rows i of (gate[i][d] + ape[i][d]) weighting k[i][d], rounded
// once to fp16; top_k counts tokens, so floor(top_k / 4) pools are selected,
// each expanded to its valid positions, and the valid tail positions (the
// incomplete last pool, at most 3) are always added.
//
// Here the pooled key is computed once, when a pool's fourth position is
// appended, and kept in a pool-key cache [pool rows, 128] fp16 (pool j of
// sequence b at row kv_off[b] / 4 + j), so that scoring streams a quarter of
// the keys through the tensor-core score kernel (in its pool mode).  The
// compression runs in float64, where the softmax and the weighted sum of four
// fp16 keys lose nothing that the single rounding to fp16 would keep.
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {

namespace {

__device__ __forceinline__ bool row_valid(const uint16_t *row) {
    return (row[2 * D_I] & 0x7FFFu) != 0;   // valid = any nonzero fp16
}

struct KpoolAppendParams {
    const uint16_t *k_new;     // fp16 [T, 128]
    const uint16_t *gate_new;  // fp16 [T, 128]
    const float *ape;          // [4, 128]
    uint16_t *rows;            // fp16 [cache_rows, 257]
    uint16_t *pool_keys;       // fp16 [pool_rows, 128]
    int64_t pool_rows;
    int phase, fused;
};

}  // namespace

// One CTA of 128 threads per token, thread d owning dim d: the token's
// packed row and, when it completes a pool, the pooled key (float64, whose
// issue rate on this part is low: spread one dim per thread).
__global__ void __launch_bounds__(128) kpool_append_kernel(const KpoolAppendParams a, const DevBatch b,
                                                           uint32_t *status) {
    tl_start(b.timeline, kTlAppend);
    // The score kernel that follows loads only older pools before it waits
    // for this grid: let it start now.
    pdl_trigger();
    const int t = blockIdx.x, d = threadIdx.x, lane = d & 31;
    const int seq = seq_of_warp(b.cu_q, b.B, t, lane);
    const int pos = __ldg(b.q_pos + t);
    const int64_t kv0 = b.kv_off ? __ldg(b.kv_off + seq) : 0;
    const bool ok = pos >= 0 && pos < b.max_kv && kv0 >= 0 && !(kv0 & (kKpool - 1)) && kv0 + pos < b.cache_rows;
    if (!ok && d == 0) flag(status, DSA_DEV_BAD_POSITION);
    const int64_t j = pos >> kKpoolLog2;
    const int64_t prow = (kv0 >> kKpoolLog2) + j;
    const bool completes = ok && (pos & (kKpool - 1)) == kKpool - 1 && (a.phase == 1 || a.fused);
    if (completes && prow >= a.pool_rows && d == 0) flag(status, DSA_DEV_BAD_POSITION);
    if (ok) {
        uint16_t *row = a.rows + (kv0 + pos) * kKpoolRow;
        const uint16_t kn = __ldg(a.k_new + (int64_t)t * D_I + d);
        const uint16_t gn = __ldg(a.gate_new + (int64_t)t * D_I + d);
        if (a.phase == 0) {                          // the packed row (514 bytes: 2-byte alignment)
            row[d] = kn;
            row[D_I + d] = gn;
            if (d == 0) row[2 * D_I] = 0x3C00u;      // valid = 1.0
        }
        if (completes && prow < a.pool_rows) {
            // pool j's rows 0..2 are in the cache; row 3 is this token's own
            const uint16_t *r0 = a.rows + (kv0 + j * kKpool) * kKpoolRow;
            double kv[kKpool], ex[kKpool], m = -INFINITY;
            bool valid[kKpool];
#pragma unroll
            for (int i = 0; i < kKpool; ++i) {
                const bool own = i == kKpool - 1;
                valid[i] = own ? true : row_valid(r0 + i * kKpoolRow);
                const uint16_t kb = own ? kn : r0[i * kKpoolRow + d];
                const uint16_t gb = own ? gn : r0[i * kKpoolRow + D_I + d];
                kv[i] = (double)__half2float(__ushort_as_half(kb));
                ex[i] = (double)__half2float(__ushort_as_half(gb)) + (double)__ldg(a.ape + i * D_I + d);
                if (valid[i] && ex[i] > m) m = ex[i];
            }
            double den = 0.0, num = 0.0;
#pragma unroll
            for (int i = 0; i < kKpool; ++i) {
                if (!valid[i]) continue;
                const double w = exp(ex[i] - m);
                den += w;
                num += w * kv[i];
            }
            a.pool_keys[prow * D_I + d] = __half_as_ushort(__double2half(num / den));
        }
    }
    __syncthreads();
    tl_end(b.timeline, kTlAppend);
}

// One CTA of 128 threads per token: thread i takes the selection slots
// [i s, (i + 1) s), s = kp / 128 (at most kMaxSlots); the counts of valid
// positions are scanned across the CTA so that positions are written in
// order.  All pool indices, then all validity flags, are loaded at once (two
// round trips instead of one chain per slot).
constexpr int kMaxSlots = 8;     // kp <= 1024 pools per token, top_k <= 4096

__global__ void __launch_bounds__(128) kpool_expand_kernel(const int32_t *__restrict__ pool_idx, int kp,
                                                           const uint16_t *__restrict__ rows, const DevBatch b,
                                                           int width, int32_t *__restrict__ idx, uint32_t *status) {
    __shared__ uint32_t warp_sum[4];
    const int t = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int32_t *out = idx + (int64_t)t * width;
    // a small grid: the attention that follows may start its prologue now
    pdl_trigger();
    const int seq = seq_of_warp(b.cu_q, b.B, t, lane);
    const int pos = __ldg(b.q_pos + t);
    const int64_t kv0 = b.kv_off ? __ldg(b.kv_off + seq) : 0;
    const bool ok = pos >= 0 && pos < b.max_kv && kv0 >= 0 && kv0 + pos < b.cache_rows;
    const int n_pools = ok ? (pos + 1) >> kKpoolLog2 : 0;
    const uint16_t *seq_rows = rows + (ok ? kv0 : 0) * kKpoolRow;
    // the tail's flags do not depend on the selection: load them first
    bool tail_v[kKpool - 1];
#pragma unroll
    for (int i = 0; i < kKpool - 1; ++i) {
        const int s = n_pools * kKpool + i;
        tail_v[i] = ok && s <= pos && row_valid(seq_rows + (int64_t)s * kKpoolRow);
    }
    pdl_wait();                                     // the pool selection comes from the preceding kernel
    if (!ok) {
        if (tid == 0) flag(status, DSA_DEV_BAD_POSITION);
        for (int i = tid; i < width; i += 128) out[i] = -1;
        return;
    }
    const int per = (kp + 127) / 128;
    const int lo = min(kp, tid * per);
    int pj[kMaxSlots];
#pragma unroll
    for (int u = 0; u < kMaxSlots; ++u) {
        const int i = lo + u;
        pj[u] = (u < per && i < kp) ? __ldg(pool_idx + (int64_t)t * kp + i) : -1;
        if (pj[u] >= n_pools) pj[u] = -1;           // out of range: nothing
    }
    uint32_t vmask[kMaxSlots];                      // valid positions of each slot's pool, 4 bits
#pragma unroll
    for (int u = 0; u < kMaxSlots; ++u) {
        uint32_t m = 0;
        if (pj[u] >= 0) {
#pragma unroll
            for (int r = 0; r < kKpool; ++r)
                m |= (uint32_t)row_valid(seq_rows + (int64_t)(pj[u] * kKpool + r) * kKpoolRow) << r;
        }
        vmask[u] = m;
    }
    uint32_t cnt = 0;
#pragma unroll
    for (int u = 0; u < kMaxSlots; ++u) cnt += __popc(vmask[u]);
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    uint32_t at = incl - cnt;
    for (int w = 0; w < warp; ++w) at += warp_sum[w];
    const uint32_t total = warp_sum[0] + warp_sum[1] + warp_sum[2] + warp_sum[3];
#pragma unroll
    for (int u = 0; u < kMaxSlots; ++u)
#pragma unroll
        for (int r = 0; r < kKpool; ++r)
            if (((vmask[u] >> r) & 1u) && at < (uint32_t)width) out[at++] = pj[u] * kKpool + r;
    // the tail, always; then padding
    uint32_t n = total;
#pragma unroll
    for (int i = 0; i < kKpool - 1; ++i) {
        if (tail_v[i] && tid == 0 && n < (uint32_t)width) out[n] = n_pools * kKpool + i;
        n += tail_v[i];
    }
    for (uint32_t i = n + tid; i < (uint32_t)width; i += 128) out[i] = -1;
}

cudaError_t launch_kpool_append(const uint16_t *k_new, const uint16_t *gate_new, const float *ape,
                                const DevBatch &b, uint16_t *rows, uint16_t *pool_keys, int64_t pool_rows,
                                int phase, int fused, uint32_t *status, cudaStream_t stream) {
    KpoolAppendParams a{k_new, gate_new, ape, rows, pool_keys, pool_rows, phase, fused};
    kpool_append_kernel<<<b.T, 128, 0, stream>>>(a, b, status);
    return cudaGetLastError();
}

cudaError_t launch_kpool_expand(const int32_t *pool_idx, int kp, const uint16_t *rows, const DevBatch &b,
                                int width, int32_t *idx, uint32_t *status, cudaStream_t stream, bool pdl) {
    if (kp > 128 * kMaxSlots) return cudaErrorInvalidValue;
    return launch_k(kpool_expand_kernel, dim3((unsigned)b.T), dim3(128), 0, stream, pdl, pool_idx, kp, rows, b,
                    width, idx, status);
}

}  // namespace dsa
