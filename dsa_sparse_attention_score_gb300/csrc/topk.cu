// topk.cu -- exact top-k of each query row of indexer scores.
//
// ik_llama_opt commit log, "Add GLM-5.2/DeepSeek-V3.2 DSA lightning indexer":
// the selection is ggml_top_k(min(top_k, n_tokens)) over the causally visible
// keys.  Ties go to the lower position and the output positions are
// ascending, so the result is the unique set a full sort by (score desc,
// position asc) would keep.
//
// One CTA per row.  Scores become order-preserving 32-bit keys (-0 folded
// onto +0).  Three histogram digits (11 + 11 + 10 bits) find the exact key tau
// of the k-th largest element and the number of keys strictly above it; an
// ordered compaction then keeps every key > tau plus the first
// (k - count_above) keys == tau in position order, writing positions in
// ascending order with warp ballots.
//
// Rows that fit are read once from global memory into shared memory and every
// pass runs there.  Longer rows take one global histogram pass for the first
// digit, copy only the keys of the threshold bin into shared memory for the
// other two digits, and finish with one global compaction pass.
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {

namespace {
constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kSmemCapMax = 49152;   // keys held in shared memory (192 KB)
constexpr int kSmemCapHybrid = 16384;

struct TopkSmem {
    uint32_t hist[2048];
    uint32_t warp_sum[kTopkWarps];
    uint32_t gt[kTopkWarps];
    uint32_t eq[kTopkWarps];
    uint32_t sel_bin;
    uint32_t sel_above;
    uint32_t n_cand;
};

__device__ __forceinline__ void hist_add(uint32_t *hist, uint32_t bin) { atomicAdd(hist + bin, 1u); }

// Bins are ranked from the top.  Finds the bin b* holding the kk-th largest
// key and the count of keys in bins above it.
__device__ void find_bin(TopkSmem &sm, int nbins, uint32_t kk) {
    const int per = nbins / kTopkThreads;               // 4 or 2 bins per thread
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hi = nbins - tid * per;                    // this thread covers [hi-per, hi)
    uint32_t local = 0;
    for (int i = 1; i <= per; ++i) local += sm.hist[hi - i];
    uint32_t incl = local;                               // inclusive scan, descending bins
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) sm.warp_sum[warp] = incl;
    __syncthreads();
    uint32_t before = 0;
    for (int w = 0; w < warp; ++w) before += sm.warp_sum[w];
    const uint32_t above = before + incl - local;        // keys in bins above this thread's range
    if (above < kk && kk <= above + local) {
        uint32_t acc = above;
        for (int i = 1; i <= per; ++i) {
            const uint32_t c = sm.hist[hi - i];
            if (acc + c >= kk) {
                sm.sel_bin = (uint32_t)(hi - i);
                sm.sel_above = acc;
                break;
            }
            acc += c;
        }
    }
    __syncthreads();
}

__device__ __forceinline__ void clear_hist(TopkSmem &sm, int nb) {
    for (int i = threadIdx.x; i < nb; i += kTopkThreads) sm.hist[i] = 0;
}

// Histogram of digit (key >> sh) & (nb-1) over the keys whose bits above the
// digit equal `prefix` (all keys when hsh >= 32).  Keys come from shared
// memory (`keys`) or from the float row in global memory.
template <bool kShared>
__device__ __forceinline__ void digit_hist(TopkSmem &sm, const uint32_t *keys, const float *row, int n,
                                           int sh, int nb, int hsh, uint32_t prefix) {
    constexpr int U = kShared ? 1 : 4;                   // loads in flight per thread
    for (int s0 = threadIdx.x; s0 < n; s0 += U * kTopkThreads) {
        uint32_t key[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + u * kTopkThreads;
            key[u] = s < n ? (kShared ? keys[s] : float_key(__ldg(row + s))) : 0u;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + u * kTopkThreads;
            if (s < n && (hsh >= 32 || (key[u] >> hsh) == prefix))
                hist_add(sm.hist, (key[u] >> sh) & (uint32_t)(nb - 1));
        }
    }
}

// Ordered compaction over positions 0..n-1: keeps keys > tau and the first
// need_eq keys == tau, writing positions in ascending order to out.
template <bool kShared>
__device__ void compact(TopkSmem &sm, const uint32_t *keys, const float *row, int n, uint32_t tau,
                        uint32_t need_eq, int32_t *out) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int seg = ((n + kTopkWarps - 1) / kTopkWarps + 31) & ~31;
    const int s_begin = min(n, warp * seg), s_end = min(n, s_begin + seg);
    uint32_t gt = 0, eq = 0;
    for (int s0 = s_begin; s0 < s_end; s0 += 32) {
        const int s = s0 + lane;
        const bool in = s < s_end;
        const uint32_t key = in ? (kShared ? keys[s] : float_key(__ldg(row + s))) : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, in && key > tau));
        eq += __popc(__ballot_sync(0xffffffffu, in && key == tau));
    }
    if (lane == 0) {
        sm.gt[warp] = gt;
        sm.eq[warp] = eq;
    }
    __syncthreads();
    uint32_t gt_before = 0, eq_before = 0;
    for (int w = 0; w < warp; ++w) {
        gt_before += sm.gt[w];
        eq_before += sm.eq[w];
    }
    uint32_t sel_before = gt_before + min(eq_before, need_eq);
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int s0 = s_begin; s0 < s_end; s0 += 32) {
        const int s = s0 + lane;
        const bool in = s < s_end;
        const uint32_t key = in ? (kShared ? keys[s] : float_key(__ldg(row + s))) : 0u;
        const bool is_gt = in && key > tau;
        const bool is_eq = in && key == tau;
        const uint32_t eq_ballot = __ballot_sync(0xffffffffu, is_eq);
        const uint32_t eq_rank = eq_before + __popc(eq_ballot & lt_mask);
        const bool sel = is_gt || (is_eq && eq_rank < need_eq);
        const uint32_t sel_ballot = __ballot_sync(0xffffffffu, sel);
        if (sel) out[sel_before + __popc(sel_ballot & lt_mask)] = s;
        eq_before += __popc(eq_ballot);
        sel_before += __popc(sel_ballot);
    }
}

}  // namespace

__device__ __forceinline__ void topk_row(const float *__restrict__ scores, int64_t ld, const DevBatch &b,
                                         RowMap rows, int k, int32_t *__restrict__ idx, uint32_t *status,
                                         int cap) {
    __shared__ TopkSmem sm;
    extern __shared__ uint32_t keys[];                   // cap keys
    const int tid = threadIdx.x;
    const int64_t r = blockIdx.x;
    int t;
    if (rows.slab) {
        const int seq = (int)(r / rows.J);
        const int j = rows.j0 + (int)(r % rows.J);
        if (seq >= b.B) return;
        const int q0 = __ldg(b.cu_q + seq), q1 = __ldg(b.cu_q + seq + 1);
        if (q0 < 0 || q1 > b.T || q1 < q0) return;     // flagged by the score pass
        if (j >= q1 - q0) return;
        t = q0 + j;
    } else {
        t = (int)r;
    }
    int32_t *out = idx + (int64_t)t * k;
    const int pos = __ldg(b.q_pos + t);
    if (pos < 0 || pos >= b.max_kv || (int64_t)pos >= ld) {
        if (tid == 0) flag(status, DSA_DEV_BAD_POSITION);
        for (int i = tid; i < k; i += kTopkThreads) out[i] = -1;
        return;
    }
    const int n = pos + 1;
    if (n <= k) {
        for (int i = tid; i < k; i += kTopkThreads) out[i] = i < n ? i : -1;
        return;
    }
    pdl_wait();                                          // the scores come from the preceding kernel
    const float *row = scores + r * ld;

    if (n <= cap) {
        // ---- whole row in shared memory
        for (int s0 = tid; s0 < n; s0 += 8 * kTopkThreads) {
            float f[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int s = s0 + u * kTopkThreads;
                f[u] = s < n ? __ldg(row + s) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int s = s0 + u * kTopkThreads;
                if (s < n) keys[s] = float_key(f[u]);
            }
        }
        clear_hist(sm, 2048);
        __syncthreads();
        uint32_t prefix = 0, above = 0, kk = (uint32_t)k;
        const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
#pragma unroll
        for (int pass = 0; pass < 3; ++pass) {
            const int nb = 1 << widths[pass];
            if (pass > 0) {
                clear_hist(sm, nb);
                __syncthreads();
            }
            digit_hist<true>(sm, keys, row, n, shifts[pass], nb, shifts[pass] + widths[pass], prefix);
            __syncthreads();
            find_bin(sm, nb, kk);
            prefix = (prefix << widths[pass]) | sm.sel_bin;
            above += sm.sel_above;
            kk -= sm.sel_above;
            __syncthreads();
        }
        compact<true>(sm, keys, row, n, prefix, (uint32_t)k - above, out);
        return;
    }

    // ---- long row: first digit from global memory
    clear_hist(sm, 2048);
    if (tid == 0) sm.n_cand = 0;
    __syncthreads();
    digit_hist<false>(sm, keys, row, n, 21, 2048, 32, 0);
    __syncthreads();
    find_bin(sm, 2048, (uint32_t)k);
    const uint32_t b1 = sm.sel_bin;
    uint32_t above = sm.sel_above;
    uint32_t kk = (uint32_t)k - above;
    const uint32_t c1 = sm.hist[b1];
    __syncthreads();
    uint32_t prefix = b1;
    if ((int)c1 <= cap) {
        // copy the threshold bin's keys, refine the two lower digits there
        for (int s0 = tid; s0 < n; s0 += 4 * kTopkThreads) {
            uint32_t key[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int s = s0 + u * kTopkThreads;
                key[u] = s < n ? float_key(__ldg(row + s)) : 0u;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int s = s0 + u * kTopkThreads;
                if (s < n && (key[u] >> 21) == b1) keys[atomicAdd(&sm.n_cand, 1u)] = key[u];
            }
        }
        __syncthreads();
        const int nc = (int)sm.n_cand;
        const int shifts[2] = {10, 0}, widths[2] = {11, 10};
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int nb = 1 << widths[pass];
            clear_hist(sm, nb);
            __syncthreads();
            digit_hist<true>(sm, keys, row, nc, shifts[pass], nb, shifts[pass] + widths[pass], prefix);
            __syncthreads();
            find_bin(sm, nb, kk);
            prefix = (prefix << widths[pass]) | sm.sel_bin;
            above += sm.sel_above;
            kk -= sm.sel_above;
            __syncthreads();
        }
    } else {
        const int shifts[2] = {10, 0}, widths[2] = {11, 10};
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int nb = 1 << widths[pass];
            clear_hist(sm, nb);
            __syncthreads();
            digit_hist<false>(sm, keys, row, n, shifts[pass], nb, shifts[pass] + widths[pass], prefix);
            __syncthreads();
            find_bin(sm, nb, kk);
            prefix = (prefix << widths[pass]) | sm.sel_bin;
            above += sm.sel_above;
            kk -= sm.sel_above;
            __syncthreads();
        }
    }
    compact<false>(sm, keys, row, n, prefix, (uint32_t)k - above, out);
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float *__restrict__ scores, int64_t ld,
                                                            DevBatch b, RowMap rows, int k,
                                                            int32_t *__restrict__ idx, uint32_t *status,
                                                            int cap) {
    tl_start(b.timeline, kTlTopk);
    topk_row(scores, ld, b, rows, k, idx, status, cap);
    __syncthreads();
    pdl_trigger();   // late: waiting dependents would share the SMs
    tl_end(b.timeline, kTlTopk);
}

cudaError_t launch_topk(const float *scores, int64_t ld, const DevBatch &b, RowMap rows, int k,
                        int32_t *idx, uint32_t *status, cudaStream_t stream, bool pdl) {
    const int64_t nrows = rows.slab ? (int64_t)b.B * rows.J : (int64_t)b.T;
    if (nrows <= 0) return cudaSuccess;
    if (nrows > 0x7fffffff) return cudaErrorInvalidConfiguration;
    int cap = b.max_kv <= kSmemCapMax ? b.max_kv : kSmemCapHybrid;
    cap = (cap + 3) & ~3;
    if (b.max_kv <= k) cap = 0;                          // every row is returned whole
    const size_t smem = (size_t)cap * 4;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(topk_kernel), 2,
                                     (size_t)kSmemCapMax * 4);
    if (e != cudaSuccess) return e;
    return launch_k(topk_kernel, dim3((unsigned)nrows), dim3(kTopkThreads), smem, stream, pdl, scores, ld, b,
                    rows, k, idx, status, cap);
}

}  // namespace dsa
