// topk.cu -- exact top-k of score rows.
//
// ik_llama_opt commit log, "Add GLM-5.2/DeepSeek-V3.2 DSA lightning indexer":
// the selection is ggml_top_k(min(top_k, n_tokens)) over the causally visible
// keys.  Ties go to the lower position and the output positions are
// ascending, so the result is the unique set a full sort by (score desc,
// position asc) would keep.
//
// Main kernel (topk_cluster_kernel<NT, KPT>): a row is spread over a cluster
// of C CTAs of NT threads (C = 1..8); cluster thread g = rank * NT + tid
// holds the order-preserving keys of positions [g * e, (g + 1) * e) in
// registers, e <= KPT, read from memory once.  Three radix digits (11 + 11 +
// 10 bits) find the exact key tau of the k-th largest element: each pass
// counts the digit of the keys that still match the prefix into a shared
// histogram; in a cluster every CTA adds its counts into the histograms of
// all CTAs through distributed shared memory, so each finds the same bin
// after one cluster barrier.  The ordered compaction is one scan: per-thread
// counts of (key > tau, key == tau) are scanned within the CTA, CTA totals
// across the cluster, selected positions are staged in shared memory in
// output order and copied out coalesced.  Output order is position order
// because the cluster threads hold the row in order.
//
// Many rows longer than 16384 keys (k <= 4096), or any row longer than a
// cluster holds, go to topk_stream_kernel: one CTA per row places a candidate
// threshold from a sample of the row, streams the row once keeping the keys
// at or above it, and selects exactly among those.  topk_kernel (one CTA per
// row, keys staged in shared memory, see topk_impl.cuh) is the general
// fallback.
#include "dsa_common.cuh"
#include "dsa_internal.h"
#include "topk_impl.cuh"

#include <algorithm>

namespace dsa {

namespace {
constexpr int kTopkThreads = 512;
constexpr int kMaxCluster = 8;
constexpr int kSmemCapMax = 49152;   // keys held in shared memory by the fallback (192 KB)
constexpr int kSmemCapHybrid = 16384;

// The token of row r of a score slab, or -1.
__device__ __forceinline__ int row_token(const DevBatch &b, const RowMap &rows, int64_t r) {
    if (!rows.slab) return (int)r;
    const int seq = (int)(r / rows.J);
    const int j = rows.j0 + (int)(r % rows.J);
    if (seq >= b.B) return -1;
    const int q0 = __ldg(b.cu_q + seq), q1 = __ldg(b.cu_q + seq + 1);
    if (q0 >= 0 && q1 <= b.T && q1 >= q0 && j < q1 - q0) return q0 + j;   // bad bounds: flagged by the score pass
    return -1;
}
// Forced-in (attention-sink) positions of row r: [a, a + n_sink), a being the
// sequence's first present position (sink_pos0[seq], or 0 when not given).
__device__ __forceinline__ void row_sink(const DevBatch &b, const RowMap &rows, int64_t r, int t, int n_sink,
                                         const int32_t *sink_pos0, int &lo, int &hi) {
    lo = hi = 0;
    if (n_sink <= 0) return;
    const int sq = rows.slab ? (int)(r / rows.J) : seq_of(b.cu_q, b.B, t);
    const int a = sink_pos0 ? max(0, __ldg(sink_pos0 + sq)) : 0;
    lo = a;
    hi = (int)min((int64_t)a + n_sink, (int64_t)0x7fffffff);
}
}  // namespace

template <int NT>
struct ClusterSmem {
    uint32_t hist[2][2048];          // double-buffered digit histograms (cluster sums)
    uint32_t local[2048];            // this CTA's counts of a pass, when C > 1
    uint32_t warp_sum[NT / 32];
    uint32_t cta_total[kMaxCluster]; // packed (gt, eq) totals of the other CTAs, written remotely
    uint32_t sel_bin, sel_above;
};

// Bins are ranked from the top.  Finds the bin holding the kk-th largest key
// of `hist` and the count of keys in the bins above it.  Ends with a CTA
// barrier after which `hist` may be rewritten.
template <int NT>
__device__ __forceinline__ void find_bin(ClusterSmem<NT> &sm, const uint32_t *hist, int nb, uint32_t kk) {
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = nb / NT;
    const int hi = nb - tid * per;                       // this thread covers bins [hi - per, hi)
    uint32_t local = 0;
    for (int i = 1; i <= per; ++i) local += hist[hi - i];
    uint32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) sm.warp_sum[warp] = incl;
    __syncthreads();
    uint32_t ws = lane < NW ? sm.warp_sum[lane] : 0u;    // scan of the warp totals, in every warp
#pragma unroll
    for (int o = 1; o < NW; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, ws, o);
        if (lane >= o) ws += v;
    }
    const uint32_t wprev = __shfl_sync(0xffffffffu, ws, (warp + 31) & 31);
    const uint32_t above = (warp > 0 ? wprev : 0u) + incl - local;
    if (above < kk && kk <= above + local) {
        uint32_t acc = above;
        for (int i = 1; i <= per; ++i) {
            const uint32_t c = hist[hi - i];
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

template <int NT, int KPT>
__device__ __forceinline__ void select_cluster(ClusterSmem<NT> &sm, uint32_t *stage, const float *row, int n,
                                               int k, int32_t *out, int C, uint32_t crank, bool vec, int sink_lo,
                                               int sink_hi) {
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int GT = C * NT;
    const int e = ((n + GT - 1) / GT + 3) & ~3;          // keys per thread: a multiple of 4, <= KPT
    const int s0 = ((int)crank * NT + tid) * e;
    const int cnt = max(0, min(e, n - s0));

    for (int i = tid; i < 3 * 2048; i += NT) (&sm.hist[0][0])[i] = 0;
    // Every CTA of the cluster must run, and have cleared its histograms,
    // before any of them adds into another's: arrive now, wait after the loads.
    if (C > 1) cluster_arrive();

    // ---- this thread's keys, read once
    uint32_t key[KPT];
    if (vec) {
        // float4 loads: s0 is a multiple of 4 and the row stride a multiple of
        // 4 floats, so the last vector of a row ends inside the row's stride.
#pragma unroll
        for (int q = 0; q < KPT / 4; ++q) {
            float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
            if (4 * q < cnt) f = __ldcg(reinterpret_cast<const float4 *>(row + s0) + q);
            key[4 * q + 0] = float_key(f.x);
            key[4 * q + 1] = float_key(f.y);
            key[4 * q + 2] = float_key(f.z);
            key[4 * q + 3] = float_key(f.w);
        }
    } else {
#pragma unroll
        for (int j = 0; j < KPT; ++j) key[j] = j < cnt ? float_key(__ldcg(row + s0 + j)) : 0u;
    }
    if (sink_hi > sink_lo) {                             // forced-in positions rank first
#pragma unroll
        for (int j = 0; j < KPT; ++j)
            if (j < cnt && s0 + j >= sink_lo && s0 + j < sink_hi) key[j] = 0xFFFFFFFFu;
    }
    if (C > 1) cluster_wait();
    else __syncthreads();

    // ---- three digits: prefix ends as the exact key tau of the k-th largest.
    // Pass p sums into hist[p & 1].  In a cluster each CTA counts into
    // `local` first and then adds its counts into the sums of every CTA,
    // itself included, so that all of them find the same bin without a second
    // exchange (forwarding from the summed buffer would echo other CTAs'
    // counts while they arrive).
    uint32_t prefix = 0, above = 0, kk = (uint32_t)k;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int width = pass == 2 ? 10 : 11;
        const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nb = 1 << width;
        const int hsh = sh + width;                     // bits above the digit (32: none)
        uint32_t *H = sm.hist[pass & 1];
        uint32_t *cnt_to = C > 1 ? sm.local : H;
#pragma unroll
        for (int j = 0; j < KPT; ++j)
            if (j < cnt && (hsh >= 32 || (key[j] >> hsh) == prefix))
                atomicAdd(&cnt_to[(key[j] >> sh) & (uint32_t)(nb - 1)], 1u);
        __syncthreads();
        if (C > 1) {
            const uint32_t h0 = smem_u32(H);
            for (int i = tid; i < nb; i += NT) {
                const uint32_t v = sm.local[i];
                if (v) {
                    sm.local[i] = 0;                     // ready for the next pass
                    for (int r = 0; r < C; ++r) dsmem_add_u32(dsmem_map(h0 + 4u * (uint32_t)i, (uint32_t)r), v);
                }
            }
            cluster_sync_all();
        }
        find_bin<NT>(sm, H, nb, kk);
        prefix = (prefix << width) | sm.sel_bin;
        above += sm.sel_above;
        kk -= sm.sel_above;
        if (pass == 0)                                   // hist[0] again serves pass 2
            for (int i = tid; i < 2048; i += NT) H[i] = 0;
    }

    // ---- ordered compaction: keep key > tau and the first need_eq keys == tau
    const uint32_t tau = prefix, need_eq = (uint32_t)k - above;
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
        if (j < cnt) {
            gt += key[j] > tau;
            eq += key[j] == tau;
        }
    }
    const uint32_t packed = (gt << 16) | eq;           // a CTA holds at most 16384 keys
    uint32_t incl = packed;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) sm.warp_sum[warp] = incl;
    __syncthreads();
    uint32_t ws = lane < NW ? sm.warp_sum[lane] : 0u;
#pragma unroll
    for (int o = 1; o < NW; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, ws, o);
        if (lane >= o) ws += v;
    }
    const uint32_t wprev = __shfl_sync(0xffffffffu, ws, (warp + 31) & 31);
    const uint32_t total = __shfl_sync(0xffffffffu, ws, NW - 1);
    const uint32_t before = (warp > 0 ? wprev : 0u) + incl - packed;
    uint32_t low_gt = 0, low_eq = 0;                     // keys of the lower-ranked CTAs
    if (C > 1) {
        if (tid < C && tid > (int)crank)
            dsmem_st_u32(dsmem_map(smem_u32(&sm.cta_total[crank]), (uint32_t)tid), total);
        cluster_sync_all();                              // last cluster access
        for (int r = 0; r < (int)crank; ++r) {
            low_gt += sm.cta_total[r] >> 16;
            low_eq += sm.cta_total[r] & 0xFFFFu;
        }
    }
    const uint32_t cta_base = low_gt + min(low_eq, need_eq);          // selected before this CTA
    const uint32_t cta_sel = (total >> 16) + min(low_eq + (total & 0xFFFFu), need_eq) - min(low_eq, need_eq);
    uint32_t eq_before = low_eq + (before & 0xFFFFu);
    uint32_t sel = low_gt + (before >> 16) + min(eq_before, need_eq) - cta_base;
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
        if (j < cnt) {
            const bool is_eq = key[j] == tau;
            if (key[j] > tau || (is_eq && eq_before < need_eq)) stage[sel++] = (uint32_t)(s0 + j);
            eq_before += is_eq;
        }
    }
    __syncthreads();
    for (uint32_t i = tid; i < cta_sel; i += NT) out[cta_base + i] = (int32_t)stage[i];
}

template <int NT, int KPT>
__global__ void __launch_bounds__(NT) topk_cluster_kernel(const float *__restrict__ scores, int64_t ld, DevBatch b,
                                                          RowMap rows, int k, int32_t *__restrict__ idx,
                                                          uint32_t *status, int C, int vec, int early, int n_sink,
                                                          const int32_t *__restrict__ sink_pos0) {
    __shared__ ClusterSmem<NT> sm;
    extern __shared__ uint32_t stage[];                 // min(k, NT * KPT) selected positions
    tl_start(b.timeline, kTlTopk);
    // A grid of a few CTAs leaves most SMs idle: let the dependent kernel
    // start its prologue there right away.  A larger one triggers at its
    // end, since waiting dependents would share its SMs.
    if (early) pdl_trigger();
    const uint32_t crank = C > 1 ? cluster_rank() : 0u;
    const int64_t r = blockIdx.x / C;
    const int t = row_token(b, rows, r);               // uniform over the cluster
    if (t >= 0) {
        int32_t *out = idx + (int64_t)t * k;
        const int pos = visible_last(b, t);          // a pool index in pool mode
        const int g = (int)crank * NT + (int)threadIdx.x, GT = C * NT;
        if (pos < 0 || pos >= b.max_kv || (int64_t)pos >= ld) {
            // (in pool mode -1 is a token with no complete pool: an empty row)
            if (g == 0 && !(b.pool_log2 && pos == -1)) flag(status, DSA_DEV_BAD_POSITION);
            for (int i = g; i < k; i += GT) out[i] = -1;
        } else if (pos + 1 <= k) {
            for (int i = g; i < k; i += GT) out[i] = i <= pos ? i : -1;
        } else {
            int lo, hi;
            row_sink(b, rows, r, t, n_sink, sink_pos0, lo, hi);
            pdl_wait();                                // the scores come from the preceding kernel
            select_cluster<NT, KPT>(sm, stage, scores + r * ld, pos + 1, k, out, C, crank, vec != 0, lo, hi);
        }
    }
    __syncthreads();
    if (!early) pdl_trigger();
    tl_end(b.timeline, kTlTopk);
}

// Fallback for rows longer than a cluster holds in registers.
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float *__restrict__ scores, int64_t ld,
                                                            DevBatch b, RowMap rows, int k,
                                                            int32_t *__restrict__ idx, uint32_t *status,
                                                            int cap, int n_sink, const int32_t *__restrict__ sink_pos0) {
    __shared__ topk::Shared<kTopkThreads> sm;
    extern __shared__ uint32_t keys[];                   // cap keys
    tl_start(b.timeline, kTlTopk);
    const int tid = threadIdx.x;
    const int64_t r = blockIdx.x;
    const int t = row_token(b, rows, r);
    if (t >= 0) {
        int32_t *out = idx + (int64_t)t * k;
        const int pos = visible_last(b, t);
        if (pos < 0 || pos >= b.max_kv || (int64_t)pos >= ld) {
            if (tid == 0 && !(b.pool_log2 && pos == -1)) flag(status, DSA_DEV_BAD_POSITION);
            for (int i = tid; i < k; i += kTopkThreads) out[i] = -1;
        } else if (pos + 1 <= k) {
            for (int i = tid; i < k; i += kTopkThreads) out[i] = i <= pos ? i : -1;
        } else {
            int lo, hi;
            row_sink(b, rows, r, t, n_sink, sink_pos0, lo, hi);
            pdl_wait();
            topk::select_row<kTopkThreads, -1>(sm, tid, keys, cap, topk::RowSrc{scores + r * ld, lo, hi}, pos + 1, k,
                                               out, nullptr);
        }
    }
    __syncthreads();
    pdl_trigger();
    tl_end(b.timeline, kTlTopk);
}

namespace {
constexpr int kStreamRun = 16;                             // sampled runs of 16 keys (one 64-byte line) ...
constexpr int kStreamRuns = 256;                           // ... 4096 keys
constexpr int kStreamSample = kStreamRuns * kStreamRun;
// Shared memory of the candidates (score bits, position) of NT threads
// whose warps keep at most WCAP each.
template <int NT, int WCAP>
constexpr size_t stream_smem() { return (size_t)(NT / 32) * WCAP * 8; }
constexpr int kStreamUnroll = 5;                           // 128-key groups in flight per warp

template <int NT>
struct StreamSmem {
    topk::Shared<NT> sel;
    uint32_t wcnt[NT / 32];                                  // candidates kept per warp
    uint32_t wgt[NT / 32], weq[NT / 32];                     // per warp: keys above / equal to tau
};

// The float whose key is `key` (the inverse of float_key).
__device__ __forceinline__ float key_float(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Keeps the candidate at position p of one 32-key step of a warp (lane i
// holds position step + i), appending it to the warp's region in position
// order.  A key is kept when its score is not below tau_f (NaN scores are
// kept too: the exact passes rank them by key).  Appends past the region's
// capacity are dropped; the count wc still grows, which marks the overflow.
// kCheck: positions past w1 are dropped and attention-sink positions kept.
template <int WCAP, bool kCheck>
__device__ __forceinline__ void stream_keep(float f, int p, float tau_f, int w1, const topk::RowSrc &src,
                                            uint32_t lt, uint2 *wbuf, uint32_t &wc) {
    bool keep = !(f < tau_f);
    if (kCheck) keep = p < w1 && (keep || src.sink(p));
    const uint32_t bal = __ballot_sync(0xffffffffu, keep);
    const uint32_t at = wc + __popc(bal & lt);
    if (keep && at < (uint32_t)WCAP) wbuf[at] = make_uint2(__float_as_uint(f), (uint32_t)p);
    wc += __popc(bal);
}

// The key of a kept candidate: attention-sink positions rank first.
__device__ __forceinline__ uint32_t cand_key(const uint2 c, const topk::RowSrc &src) {
    return src.sink((int)c.y) ? 0xFFFFFFFFu : float_key(__uint_as_float(c.x));
}
}  // namespace

// Exact top-k of long rows in one pass over the row, by one CTA of NT threads
// whose warps keep at most WCAP candidates each:
//  A. a lower bound (22 leading bits) of the j-th largest of 4096 sample keys
//     (256 evenly spaced runs of 16 consecutive keys), j about 1.5 times
//     the expected sample rank of the row's k-th key, is a threshold tau_lo;
//  B. every warp streams its contiguous segment of the row and appends the
//     scores not below tau_lo, with their positions, in position order to
//     its own region of shared memory;
//  C. when at least k keys are kept, the row's k-th key is >= tau_lo, so every
//     key the selection needs (and every key tied with the k-th) was kept: a
//     three-digit radix select over the kept keys gives the exact tau;
//  D. an ordered compaction of the kept keys writes the positions.
// A region that overflows, or fewer than k kept keys, sends the row to the
// general path (topk::select_row), so the result is exact whatever the data.
template <int NT, int WCAP>
__global__ void __launch_bounds__(NT, 1024 / NT)
    topk_stream_kernel(const float *__restrict__ scores, int64_t ld, DevBatch b, RowMap rows, int k,
                       int32_t *__restrict__ idx, uint32_t *status, int n_sink, const int32_t *__restrict__ sink_pos0) {
    constexpr int W = NT / 32;
    __shared__ StreamSmem<NT> sm;
    extern __shared__ uint2 cand[];                      // kept (score bits, position) [W * WCAP]
    uint32_t *skey = reinterpret_cast<uint32_t *>(cand);  // the samples' keys, before the pass
    tl_start(b.timeline, kTlTopk);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t r = blockIdx.x;
    const int t = row_token(b, rows, r);
    if (t >= 0) {
        int32_t *out = idx + (int64_t)t * k;
        const int pos = visible_last(b, t);
        if (pos < 0 || pos >= b.max_kv || (int64_t)pos >= ld) {
            if (tid == 0 && !(b.pool_log2 && pos == -1)) flag(status, DSA_DEV_BAD_POSITION);
            for (int i = tid; i < k; i += NT) out[i] = -1;
        } else if (pos + 1 <= k) {
            for (int i = tid; i < k; i += NT) out[i] = i <= pos ? i : -1;
        } else {
            int slo, shi;
            row_sink(b, rows, r, t, n_sink, sink_pos0, slo, shi);
            pdl_wait();                                  // the scores come from the preceding kernel
            const int n = pos + 1;
            const topk::RowSrc src{scores + r * ld, slo, shi};

            // ---- A: sample threshold
            const int m = min(n, kStreamSample);
            {
                // every key of a short row, else run c of 16 keys from c (n - 16) / 255 rounded down to 16
                uint32_t sk[kStreamSample / NT];
                const uint32_t run_step = (uint32_t)(n - kStreamRun) / (kStreamRuns - 1);
                const uint32_t run_rem = (uint32_t)(n - kStreamRun) % (kStreamRuns - 1);
#pragma unroll
                for (int u = 0; u < kStreamSample / NT; ++u) {
                    const int i = tid + u * NT;
                    const uint32_t c = (uint32_t)i / kStreamRun;
                    // c (n - 16) / 255 without 64-bit arithmetic: c step + c rem / 255
                    const int s = n <= kStreamSample
                                      ? i
                                      : (int)((c * run_step + c * run_rem / (kStreamRuns - 1)) & ~(uint32_t)(kStreamRun - 1)) +
                                            (i & (kStreamRun - 1));
                    sk[u] = i < m ? topk::row_key(src, s) : 0u;
                }
#pragma unroll
                for (int u = 0; u < kStreamSample / NT; ++u) {
                    const int i = tid + u * NT;
                    if (i < m) skey[i] = sk[u];
                }
            }
            // about 1.5 times the sample rank of the row's k-th key, plus a margin
            const int64_t jr = 3 * (((int64_t)k * m + n - 1) / n) / 2 + 16;
            const int j = jr < m ? (int)jr : m;
            uint32_t prefix = 0, kk = (uint32_t)j;
            {
                // two digits of 11 bits, from the top: the bin holding the j-th largest sample
#pragma unroll 1
                for (int pass = 0; pass < 2; ++pass) {
                    const int sh = pass == 0 ? 21 : 10, wd = 11, nb = 1 << wd;
                    topk::clear_hist(sm.sel, tid, nb);
                    __syncthreads();
                    topk::digit_hist<NT, true>(sm.sel, tid, skey, src, m, sh, nb, sh + wd, prefix);
                    __syncthreads();
                    topk::find_bin<NT, -1>(sm.sel, tid, nb, kk);
                    prefix = (prefix << wd) | sm.sel.sel_bin;
                    kk -= sm.sel.sel_above;
                    __syncthreads();
                }
            }
            prefix <<= 10;                               // the bin's lowest key
            const float tau_f = key_float(prefix);       // keys >= prefix <=> scores not below tau_f

            // ---- B: one pass over the row, warp segments of whole 128-key groups
            const int seg = ((n + W - 1) / W + 127) & ~127;
            const int w0 = min(n, warp * seg), w1 = min(n, w0 + seg);
            uint2 *wbuf = cand + warp * WCAP;
            uint32_t wc = 0;
            const uint32_t lt = (1u << lane) - 1u;
            int base = w0;
            if (!(src.lo < src.hi && src.lo < w1 && src.hi > w0)) {
                // whole blocks with no sink position: no per-key checks
                for (; base + 128 * kStreamUnroll <= w1; base += 128 * kStreamUnroll) {
                    float v[4 * kStreamUnroll];
#pragma unroll
                    for (int u = 0; u < 4 * kStreamUnroll; ++u) v[u] = __ldcg(src.p + base + 32 * u + lane);
#pragma unroll
                    for (int u = 0; u < 4 * kStreamUnroll; ++u)
                        stream_keep<WCAP, false>(v[u], base + 32 * u + lane, tau_f, w1, src, lt, wbuf, wc);
                }
            }
            for (; base < w1; base += 128 * kStreamUnroll) {
                float v[4 * kStreamUnroll];
#pragma unroll
                for (int u = 0; u < 4 * kStreamUnroll; ++u) {
                    const int p = base + 32 * u + lane;
                    v[u] = p < w1 ? __ldcg(src.p + p) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 4 * kStreamUnroll; ++u)
                    stream_keep<WCAP, true>(v[u], base + 32 * u + lane, tau_f, w1, src, lt, wbuf, wc);
            }
            const bool ovf = wc > (uint32_t)WCAP;
            if (lane == 0) sm.wcnt[warp] = ovf ? (uint32_t)WCAP + 1u : wc;
            __syncthreads();
            uint32_t kept = 0;
            bool bad = false;
#pragma unroll
            for (int w = 0; w < W; ++w) {
                bad |= sm.wcnt[w] > (uint32_t)WCAP;
                kept += sm.wcnt[w];
            }
            bad |= kept < (uint32_t)k;                   // tau_lo above the k-th key: not enough kept

            if (!bad) {
                // ---- C: exact select among the kept keys
                uint32_t tp = 0, above = 0;
                kk = (uint32_t)k;
#pragma unroll 1
                for (int pass = 0; pass < 3; ++pass) {
                    const int sh = pass == 0 ? 21 : pass == 1 ? 10 : 0, wd = pass == 2 ? 10 : 11;
                    const int nb = 1 << wd, hsh = sh + wd;
                    topk::clear_hist(sm.sel, tid, nb);
                    __syncthreads();
                    for (uint32_t i = lane; i < wc; i += 32) {       // each warp over its own kept keys
                        const uint32_t key = cand_key(wbuf[i], src);
                        if (hsh >= 32 || (key >> hsh) == tp) atomicAdd(&sm.sel.hist[(key >> sh) & (uint32_t)(nb - 1)], 1u);
                    }
                    __syncthreads();
                    topk::find_bin<NT, -1>(sm.sel, tid, nb, kk);
                    tp = (tp << wd) | sm.sel.sel_bin;
                    above += sm.sel.sel_above;
                    kk -= sm.sel.sel_above;
                    __syncthreads();
                }
                const uint32_t tau = tp, need_eq = (uint32_t)k - above;

                // ---- D: ordered compaction, warp by warp over its region
                uint32_t gt = 0, eq = 0;
                for (uint32_t i0 = 0; i0 < wc; i0 += 32) {
                    const uint32_t i = i0 + lane;
                    const uint32_t key = i < wc ? cand_key(wbuf[i], src) : 0u;
                    gt += __popc(__ballot_sync(0xffffffffu, i < wc && key > tau));
                    eq += __popc(__ballot_sync(0xffffffffu, i < wc && key == tau));
                }
                if (lane == 0) {
                    sm.wgt[warp] = gt;
                    sm.weq[warp] = eq;
                }
                __syncthreads();
                uint32_t gt_before = 0, eq_before = 0;
                for (int w = 0; w < warp; ++w) {
                    gt_before += sm.wgt[w];
                    eq_before += sm.weq[w];
                }
                uint32_t sel_before = gt_before + min(eq_before, need_eq);
                for (uint32_t i0 = 0; i0 < wc; i0 += 32) {
                    const uint32_t i = i0 + lane;
                    const bool in = i < wc;
                    const uint2 c = in ? wbuf[i] : make_uint2(0u, 0u);
                    const uint32_t key = in ? cand_key(c, src) : 0u;
                    const bool is_gt = in && key > tau, is_eq = in && key == tau;
                    const uint32_t eq_ballot = __ballot_sync(0xffffffffu, is_eq);
                    const uint32_t eq_rank = eq_before + __popc(eq_ballot & lt);
                    const bool sel = is_gt || (is_eq && eq_rank < need_eq);
                    const uint32_t sel_ballot = __ballot_sync(0xffffffffu, sel);
                    if (sel) out[sel_before + __popc(sel_ballot & lt)] = (int32_t)c.y;
                    eq_before += __popc(eq_ballot);
                    sel_before += __popc(sel_ballot);
                }
            } else {
                // the general path, with the whole dynamic shared memory as its key scratch
                topk::select_row<NT, -1>(sm.sel, tid, reinterpret_cast<uint32_t *>(cand), 2 * W * WCAP,
                                                     src, n, k, out, nullptr);
            }
        }
    }
    __syncthreads();
    pdl_trigger();
    tl_end(b.timeline, kTlTopk);
}

template <int NT, int WCAP>
cudaError_t launch_stream(const float *scores, int64_t ld, const DevBatch &b, const RowMap &rows, int k, int32_t *idx,
                          uint32_t *status, cudaStream_t stream, bool pdl, int64_t nrows, int n_sink,
                          const int32_t *sink_pos0, int slot) {
    constexpr size_t smem = stream_smem<NT, WCAP>();
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(topk_stream_kernel<NT, WCAP>), slot, smem);
    if (e != cudaSuccess) return e;
    return launch_k(topk_stream_kernel<NT, WCAP>, dim3((unsigned)nrows), dim3(NT), smem, stream, pdl, scores, ld, b,
                    rows, k, idx, status, n_sink, sink_pos0);
}

namespace {

template <int NT, int KPT>
cudaError_t launch_cluster(const float *scores, int64_t ld, const DevBatch &b, RowMap rows, int k, int32_t *idx,
                           uint32_t *status, cudaStream_t stream, bool pdl, int64_t nrows, int C, int vec,
                           int n_sink, const int32_t *sink_pos0) {
    if (nrows * C > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const size_t stage = (size_t)std::min(k, NT * KPT) * 4;
    constexpr int slot = NT == 256 ? 5 : KPT == 16 ? 6 : KPT == 32 ? 7 : KPT == 8 ? 9 : 10;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(topk_cluster_kernel<NT, KPT>), slot,
                                     (size_t)NT * KPT * 4);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nrows * C));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = stage;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)C;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = C > 1 ? 2 : 1;
    const int early = nrows * C <= kSMs / 4 ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, topk_cluster_kernel<NT, KPT>, scores, ld, b, rows, k, idx, status, C, vec, early,
                              n_sink, sink_pos0);
}

}  // namespace

// Explicit configuration (threads per CTA, keys per thread, cluster size);
// nt * kpt * C must cover the longest row.
cudaError_t launch_topk_cfg(const float *scores, int64_t ld, const DevBatch &b, RowMap rows, int k, int32_t *idx,
                            uint32_t *status, cudaStream_t stream, bool pdl, int nt, int kpt, int C, int n_sink,
                            const int32_t *sink_pos0) {
    const int64_t nrows = rows.slab ? (int64_t)b.B * rows.J : (int64_t)b.T;
    if (nrows <= 0) return cudaSuccess;
    if (C < 1 || C > kMaxCluster || (int64_t)nt * kpt * C < b.max_kv) return cudaErrorInvalidValue;
    const int vec = (ld % 4 == 0 && reinterpret_cast<uintptr_t>(scores) % 16 == 0) ? 1 : 0;
    if (nt == 512 && kpt == 4)
        return launch_cluster<512, 4>(scores, ld, b, rows, k, idx, status, stream, pdl, nrows, C, vec, n_sink,
                                      sink_pos0);
    if (nt == 512 && kpt == 8)
        return launch_cluster<512, 8>(scores, ld, b, rows, k, idx, status, stream, pdl, nrows, C, vec, n_sink,
                                      sink_pos0);
    if (nt == 512 && kpt == 16)
        return launch_cluster<512, 16>(scores, ld, b, rows, k, idx, status, stream, pdl, nrows, C, vec, n_sink,
                                                   sink_pos0);
    if (nt == 512 && kpt == 32)
        return launch_cluster<512, 32>(scores, ld, b, rows, k, idx, status, stream, pdl, nrows, C, vec, n_sink,
                                                   sink_pos0);
    if (nt == 256 && kpt == 32)
        return launch_cluster<256, 32>(scores, ld, b, rows, k, idx, status, stream, pdl, nrows, C, vec, n_sink,
                                                   sink_pos0);
    return cudaErrorInvalidValue;
}

cudaError_t launch_topk(const float *scores, int64_t ld, const DevBatch &b, RowMap rows, int k,
                        int32_t *idx, uint32_t *status, cudaStream_t stream, bool pdl, int n_sink,
                        const int32_t *sink_pos0) {
    const int64_t nrows = rows.slab ? (int64_t)b.B * rows.J : (int64_t)b.T;
    if (nrows <= 0) return cudaSuccess;
    if (nrows > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const int64_t n_max = b.max_kv;                      // no row is longer
    // Rows up to 8192 keys: one CTA per row -- 256 threads (several CTAs per
    // SM) when rows are plentiful, 512 when latency matters.  Longer rows:
    // 512 x 32 keys per CTA in clusters of up to 8 CTAs (measured on GB300:
    // 4 x 16384 beats 8 x 8192 for 64k-key rows; clusters never pay for
    // 8192-key rows).
    if (n_max <= 8192) {
        if (nrows >= 2 * kSMs)
            return launch_topk_cfg(scores, ld, b, rows, k, idx, status, stream, pdl, 256, 32, 1, n_sink, sink_pos0);
        // the smallest register array that holds the row: the per-key loops
        // run over all KPT slots (measured on GB300, 2048-key pool rows: 512 x 8
        // instead of 512 x 16 took 2.7 us off the kpool decode top-k)
        const int kpt = n_max <= 512 * 4 ? 4 : n_max <= 512 * 8 ? 8 : 16;
        return launch_topk_cfg(scores, ld, b, rows, k, idx, status, stream, pdl, 512, kpt, 1, n_sink, sink_pos0);
    }
    const bool vec = ld % 4 == 0 && reinterpret_cast<uintptr_t>(scores) % 16 == 0;
    const bool cluster_fits = n_max <= (int64_t)kMaxCluster * 512 * 32;
    if (n_max > 512 * 32 && vec && k <= 4096 && (nrows >= kSMs || !cluster_fits)) {
        // many long rows: one streaming pass per row (see topk_stream_kernel).
        // Fewer rows than SMs keep the cluster path, which spreads a row's
        // latency chain over several CTAs.  Four CTAs of 256 threads share an
        // SM when k <= 2048 (so that one row's selection overlaps the others'
        // passes), two of 512 up to k = 4096.
        if (k <= 2048) return launch_stream<256, 704>(scores, ld, b, rows, k, idx, status, stream, pdl, nrows, n_sink,
                                                      sink_pos0, 8);
        return launch_stream<512, 768>(scores, ld, b, rows, k, idx, status, stream, pdl, nrows, n_sink, sink_pos0, 0);
    }
    // up to 65536 keys: clusters of up to 8 CTAs with 16 keys per thread
    // (measured on GB300, ragged decode rows of 4k-64k keys: 25.1 -> 17.0 us
    // against 4 CTAs of 32 keys per thread: half the work per thread in every
    // pass outweighs the wider histogram exchange)
    if (n_max <= (int64_t)kMaxCluster * 512 * 16)
        return launch_topk_cfg(scores, ld, b, rows, k, idx, status, stream, pdl, 512, 16,
                               (int)((n_max + 512 * 16 - 1) / (512 * 16)), n_sink, sink_pos0);
    if (cluster_fits)
        return launch_topk_cfg(scores, ld, b, rows, k, idx, status, stream, pdl, 512, 32,
                               (int)((n_max + 512 * 32 - 1) / (512 * 32)), n_sink, sink_pos0);
    int cap = kSmemCapHybrid;
    const size_t smem = (size_t)cap * 4;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(topk_kernel), 2, (size_t)kSmemCapMax * 4);
    if (e != cudaSuccess) return e;
    return launch_k(topk_kernel, dim3((unsigned)nrows), dim3(kTopkThreads), smem, stream, pdl, scores, ld, b,
                    rows, k, idx, status, cap, n_sink, sink_pos0);
}

}  // namespace dsa
