// topk_impl.cuh -- exact top-k selection of one score row by one CTA, with
// the keys staged in shared memory (the fallback of topk.cu for rows longer
// than a cluster of CTAs holds in registers).
//
// ik_llama_opt commit log, "Add GLM-5.2/DeepSeek-V3.2 DSA lightning indexer":
// the selection is ggml_top_k(min(top_k, n_tokens)) over the causally visible
// keys.  Ties go to the lower position and the output positions are
// ascending, so the result is the unique set a full sort by (score desc,
// position asc) would keep.
//
// Scores become order-preserving 32-bit keys (-0 folded onto +0).  Three
// digits (11 + 11 + 10 bits) find the exact key tau of the k-th largest
// element and the number of keys strictly above it; an ordered compaction then
// keeps every key > tau plus the first (k - count_above) keys == tau in
// position order, writing positions in ascending order with warp ballots.
// Rows that fit are read once into shared memory and every pass runs there.
// Longer rows use the first digit's histogram (computed here, or supplied by
// the caller), copy only the keys of the threshold bin into shared memory for
// the two lower digits, and finish with one global compaction pass.
#pragma once

#include "dsa_common.cuh"

namespace dsa {
namespace topk {

// NT threads take part (thread index `tid` 0..NT-1); kBar < 0 synchronises
// with __syncthreads, else with named barrier kBar over the NT threads.
template <int NT>
struct Shared {
    uint32_t hist[2048];
    uint32_t warp_sum[NT / 32];
    uint32_t gt[NT / 32];
    uint32_t eq[NT / 32];
    uint32_t sel_bin;
    uint32_t sel_above;
    uint32_t n_cand;
};

template <int NT, int kBar>
__device__ __forceinline__ void sync() {
    if constexpr (kBar < 0) __syncthreads();
    else named_barrier(kBar, NT);
}

// Bins are ranked from the top.  Finds the bin b* holding the kk-th largest
// key and the count of keys in bins above it.
template <int NT, int kBar>
__device__ void find_bin(Shared<NT> &sm, int tid, int nbins, uint32_t kk) {
    const int per = nbins / NT;
    const int lane = tid & 31, warp = tid >> 5;
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
    sync<NT, kBar>();
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
    sync<NT, kBar>();
}

template <int NT>
__device__ __forceinline__ void clear_hist(Shared<NT> &sm, int tid, int nb) {
    for (int i = tid; i < nb; i += NT) sm.hist[i] = 0;
}

// A score row and its forced-in (attention-sink) positions [lo, hi), whose
// keys become the maximum key so that they rank first and tie by position.
struct RowSrc {
    const float *p;
    int lo, hi;
    __device__ __forceinline__ bool sink(int s) const { return s >= lo && s < hi; }
};

__device__ __forceinline__ uint32_t row_key(const RowSrc &row, int s) {
    return row.sink(s) ? 0xFFFFFFFFu : float_key(__ldcg(row.p + s));
}

// Histogram of digit (key >> sh) & (nb-1) over the keys whose bits above the
// digit equal `prefix` (all keys when hsh >= 32), from shared memory or from
// the float row in global memory.
template <int NT, bool kShared>
__device__ __forceinline__ void digit_hist(Shared<NT> &sm, int tid, const uint32_t *keys, const RowSrc &row, int n,
                                           int sh, int nb, int hsh, uint32_t prefix) {
    constexpr int U = kShared ? 1 : 8;                   // loads in flight per thread
    for (int s0 = tid; s0 < n; s0 += U * NT) {
        uint32_t key[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + u * NT;
            key[u] = s < n ? (kShared ? keys[s] : row_key(row, s)) : 0u;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + u * NT;
            if (s < n && (hsh >= 32 || (key[u] >> hsh) == prefix))
                atomicAdd(sm.hist + ((key[u] >> sh) & (uint32_t)(nb - 1)), 1u);
        }
    }
}

// Ordered compaction over positions 0..n-1: keeps keys > tau and the first
// need_eq keys == tau, writing positions in ascending order to out.
template <int NT, int kBar, bool kShared>
__device__ void compact(Shared<NT> &sm, int tid, const uint32_t *keys, const RowSrc &row, int n, uint32_t tau,
                        uint32_t need_eq, int32_t *out) {
    constexpr int W = NT / 32;
    const int lane = tid & 31, warp = tid >> 5;
    const int seg = ((n + W - 1) / W + 31) & ~31;
    const int s_begin = min(n, warp * seg), s_end = min(n, s_begin + seg);
    uint32_t gt = 0, eq = 0;
    for (int s0 = s_begin; s0 < s_end; s0 += 32) {
        const int s = s0 + lane;
        const bool in = s < s_end;
        const uint32_t key = in ? (kShared ? keys[s] : row_key(row, s)) : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, in && key > tau));
        eq += __popc(__ballot_sync(0xffffffffu, in && key == tau));
    }
    if (lane == 0) {
        sm.gt[warp] = gt;
        sm.eq[warp] = eq;
    }
    sync<NT, kBar>();
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
        const uint32_t key = in ? (kShared ? keys[s] : row_key(row, s)) : 0u;
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
    sync<NT, kBar>();
}

// Selects the top-k positions of row[0..n) into out[0..k).  n > k.
// keys: shared scratch for `cap` keys.  first_hist: optional histogram of the
// top 11 key bits of the row (global memory), which replaces the first pass.
template <int NT, int kBar>
__device__ void select_row(Shared<NT> &sm, int tid, uint32_t *keys, int cap, const RowSrc &row, int n, int k,
                           int32_t *out, const uint32_t *first_hist) {
    uint32_t prefix = 0, above = 0, kk = (uint32_t)k;
    const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
    if (n <= cap) {
        // ---- the whole row in shared memory
        for (int s0 = tid; s0 < n; s0 += 8 * NT) {
            float f[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int s = s0 + u * NT;
                f[u] = s < n ? __ldcg(row.p + s) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int s = s0 + u * NT;
                if (s < n) keys[s] = row.sink(s) ? 0xFFFFFFFFu : float_key(f[u]);
            }
        }
        if (first_hist) {
            for (int i = tid; i < 2048; i += NT) sm.hist[i] = __ldcg(first_hist + i);
        } else {
            clear_hist(sm, tid, 2048);
        }
        sync<NT, kBar>();
#pragma unroll
        for (int pass = 0; pass < 3; ++pass) {
            const int nb = 1 << widths[pass];
            if (pass > 0) {
                clear_hist(sm, tid, nb);
                sync<NT, kBar>();
            }
            if (pass > 0 || !first_hist) {
                digit_hist<NT, true>(sm, tid, keys, row, n, shifts[pass], nb, shifts[pass] + widths[pass], prefix);
                sync<NT, kBar>();
            }
            find_bin<NT, kBar>(sm, tid, nb, kk);
            prefix = (prefix << widths[pass]) | sm.sel_bin;
            above += sm.sel_above;
            kk -= sm.sel_above;
            sync<NT, kBar>();
        }
        compact<NT, kBar, true>(sm, tid, keys, row, n, prefix, (uint32_t)k - above, out);
        return;
    }

    // ---- long row: first digit from global memory (or the given histogram)
    if (tid == 0) sm.n_cand = 0;
    if (first_hist) {
        for (int i = tid; i < 2048; i += NT) sm.hist[i] = __ldcg(first_hist + i);
        sync<NT, kBar>();
    } else {
        clear_hist(sm, tid, 2048);
        sync<NT, kBar>();
        digit_hist<NT, false>(sm, tid, keys, row, n, 21, 2048, 32, 0);
        sync<NT, kBar>();
    }
    find_bin<NT, kBar>(sm, tid, 2048, (uint32_t)k);
    const uint32_t b1 = sm.sel_bin;
    above = sm.sel_above;
    kk = (uint32_t)k - above;
    const uint32_t c1 = sm.hist[b1];
    sync<NT, kBar>();
    prefix = b1;
    if ((int)c1 <= cap) {
        // copy the threshold bin's keys, refine the two lower digits there
        for (int s0 = tid; s0 < n; s0 += 8 * NT) {
            uint32_t key[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int s = s0 + u * NT;
                key[u] = s < n ? row_key(row, s) : 0u;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int s = s0 + u * NT;
                if (s < n && (key[u] >> 21) == b1) keys[atomicAdd(&sm.n_cand, 1u)] = key[u];
            }
        }
        sync<NT, kBar>();
        const int nc = (int)sm.n_cand;
#pragma unroll
        for (int pass = 1; pass < 3; ++pass) {
            const int nb = 1 << widths[pass];
            clear_hist(sm, tid, nb);
            sync<NT, kBar>();
            digit_hist<NT, true>(sm, tid, keys, row, nc, shifts[pass], nb, shifts[pass] + widths[pass], prefix);
            sync<NT, kBar>();
            find_bin<NT, kBar>(sm, tid, nb, kk);
            prefix = (prefix << widths[pass]) | sm.sel_bin;
            above += sm.sel_above;
            kk -= sm.sel_above;
            sync<NT, kBar>();
        }
    } else {
#pragma unroll
        for (int pass = 1; pass < 3; ++pass) {
            const int nb = 1 << widths[pass];
            clear_hist(sm, tid, nb);
            sync<NT, kBar>();
            digit_hist<NT, false>(sm, tid, keys, row, n, shifts[pass], nb, shifts[pass] + widths[pass], prefix);
            sync<NT, kBar>();
            find_bin<NT, kBar>(sm, tid, nb, kk);
            prefix = (prefix << widths[pass]) | sm.sel_bin;
            above += sm.sel_above;
            kk -= sm.sel_above;
            sync<NT, kBar>();
        }
    }
    compact<NT, kBar, false>(sm, tid, keys, row, n, prefix, (uint32_t)k - above, out);
}

}  // namespace topk
}  // namespace dsa
