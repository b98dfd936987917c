// topk.cu -- exact top-k of each query row of indexer scores.
//
// ik_llama_opt commit log, "Add GLM-5.2/DeepSeek-V3.2 DSA lightning indexer":
// the selection is ggml_top_k(min(top_k, n_tokens)) over the causally visible
// keys.  Ties go to the lower position and the output positions are
// ascending, so the result is the unique set a full sort by (score desc,
// position asc) would keep.
//
// One CTA per row.  Scores become order-preserving 32-bit keys (-0 folded
// onto +0).  Three histogram passes (11 + 11 + 10 bits) find the exact key
// tau of the k-th largest element and the number of keys strictly above it;
// a final ordered compaction keeps every key > tau plus the first
// (k - count_above) keys == tau in position order, writing positions in
// ascending order with warp ballots.
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {

namespace {
constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;

struct TopkSmem {
    uint32_t hist[2048];
    uint32_t warp_sum[kTopkWarps];
    uint32_t gt[kTopkWarps];
    uint32_t eq[kTopkWarps];
    uint32_t sel_bin;
    uint32_t sel_above;
};

__device__ __forceinline__ void hist_add(uint32_t *hist, uint32_t bin) {
    const uint32_t peers = __match_any_sync(__activemask(), bin);
    if ((threadIdx.x & 31) == (uint32_t)(__ffs(peers) - 1)) atomicAdd(hist + bin, __popc(peers));
}

// Bins are ranked from the top.  Finds the bin b* holding the kk-th largest
// key and the count of keys in bins above it.
__device__ void find_bin(TopkSmem &sm, int nbins, uint32_t kk) {
    const int per = nbins / kTopkThreads;               // 4 or 2 bins per thread
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hi = nbins - tid * per;                    // this thread covers [hi-per, hi)
    uint32_t local = 0;
    for (int i = 1; i <= per; ++i) local += sm.hist[hi - i];
    // inclusive scan over threads in descending-bin order
    uint32_t incl = local;
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
}  // namespace

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float *__restrict__ scores,
                                                            int64_t ld, DevBatch b, RowMap rows,
                                                            int k, int32_t *__restrict__ idx,
                                                            uint32_t *status) {
    __shared__ TopkSmem sm;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t r = blockIdx.x;
    int t;
    if (rows.slab) {
        const int seq = (int)(r / rows.J);
        const int j = rows.j0 + (int)(r % rows.J);
        if (seq >= b.B) return;
        const int q0 = __ldg(b.cu_q + seq), q1 = __ldg(b.cu_q + seq + 1);
        if (q0 < 0 || q1 > b.T || q1 < q0) return;  // flagged by the score pass
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
    const float *row = scores + r * ld;
    if (n <= k) {
        for (int i = tid; i < k; i += kTopkThreads) out[i] = i < n ? i : -1;
        return;
    }

    // ---- radix select of the k-th largest key
    uint32_t prefix = 0, above_total = 0, kk = (uint32_t)k;
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
#pragma unroll
    for (int pass = 0; pass < 3; ++pass) {
        const int nb = 1 << widths[pass];
        for (int i = tid; i < nb; i += kTopkThreads) sm.hist[i] = 0;
        __syncthreads();
        const int sh = shifts[pass];
        const int hsh = sh + widths[pass];  // bits above this digit must match the prefix
        for (int s = tid; s < n; s += kTopkThreads) {
            const uint32_t key = float_key(__ldg(row + s));
            if (pass == 0 || (key >> hsh) == prefix) hist_add(sm.hist, (key >> sh) & (uint32_t)(nb - 1));
        }
        __syncthreads();
        find_bin(sm, nb, kk);
        prefix = (prefix << widths[pass]) | sm.sel_bin;
        above_total += sm.sel_above;
        kk -= sm.sel_above;
        __syncthreads();
    }
    const uint32_t tau = prefix;
    const uint32_t need_eq = (uint32_t)k - above_total;  // >= 1

    // ---- ordered compaction: warp w owns a contiguous segment
    const int seg = ((n + kTopkWarps - 1) / kTopkWarps + 31) & ~31;
    const int s_begin = min(n, warp * seg), s_end = min(n, s_begin + seg);
    uint32_t gt = 0, eq = 0;
    for (int s0 = s_begin; s0 < s_end; s0 += 32) {
        const int s = s0 + lane;
        uint32_t key = 0;
        if (s < s_end) key = float_key(__ldg(row + s));
        const bool in = s < s_end;
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
        uint32_t key = 0;
        if (in) key = float_key(__ldg(row + s));
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

cudaError_t launch_topk(const float *scores, int64_t ld, const DevBatch &b, RowMap rows, int k,
                        int32_t *idx, uint32_t *status, cudaStream_t stream) {
    const int64_t nrows = rows.slab ? (int64_t)b.B * rows.J : (int64_t)b.T;
    if (nrows <= 0) return cudaSuccess;
    if (nrows > 0x7fffffff) return cudaErrorInvalidConfiguration;
    topk_kernel<<<(unsigned)nrows, kTopkThreads, 0, stream>>>(scores, ld, b, rows, k, idx, status);
    return cudaGetLastError();
}

}  // namespace dsa
