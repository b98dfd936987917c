// score.cu -- lightning-indexer score on the 5th-generation tensor cores.
//
// ik_llama_opt commit log, "Add GLM-5.2/DeepSeek-V3.2 DSA lightning indexer":
//   scores = relu(indexer_k . indexer_q), scaled per-head weights, summed over
//   heads, plus the causal mask.  The keys come from the persistent fp16
//   single-head cache of "decode-correct via persistent indexer-K cache"
//   (rotated queries when the cache holds rotated keys).
//
// One CTA owns a group of up to G query tokens of one sequence and a chunk of
// consecutive 128-key tiles.  Per tile the tensor core computes
//     D[key, (token, head)] = k_tile[128 x 128] . Q[(token, head) x 128]^T
// (M = 128 keys, K = 128, HP = H_I rounded up to 16) in one or two steps
// ("halves") of N = NP <= 256 columns, each step into the other of two TMEM
// accumulators, so the epilogue of one step overlaps the MMA of the next and
// the TMA loads run ahead.  Two halves (G * HP = 2 * NP) use each key tile
// for twice the tokens, halving the key bytes per flop (measured on GB300,
// 4096 tokens after 4096: 0.47 -> 0.44 ms).  In the epilogue each thread owns
// one key row (its TMEM lane) and reduces sum_h w * max(0, D) for each of its
// tokens in registers -- no cross-thread reduction.
//
// Warp roles: warp 0 issues TMA loads (a ring of 2-4 32 KB key tiles),
// warp 1 allocates TMEM and issues MMAs, the 4 or 16 warps after them stage
// the queries and run the epilogue.  All waits are bounded (1 s by default)
// and end in DSA_DEV_TIMEOUT.
#include <algorithm>

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {

namespace {

constexpr int kMaxStages = 4;        // depth of the key-tile ring (runtime: 2..4)
constexpr int kMaxGroup = 32;        // tokens per group: 2 halves x 256 columns / 16 padded heads
constexpr size_t kSmemLimit = 232448;   // opt-in shared memory per CTA (227 KB)
constexpr int kTileKeys = 128;
constexpr int kTileBytes = kTileKeys * D_I * 2;  // 32 KB: two 64-column SW128 boxes
// Epilogue warps per CTA: 16 (four per TMEM lane quarter, splitting each
// step's tokens) for multi-token groups -- measured on GB300 the epilogue
// needs them to keep pace with the tensor core; 4 (several CTAs per SM) for
// one-token decode groups.
template <int kEpi> struct ScoreCfg {
    static constexpr int kEpiWarps = kEpi;
    static constexpr int kThreads = 64 + 32 * kEpi;
    static constexpr int kQuarterWarps = kEpi / 4;   // epilogue warps per TMEM lane quarter
    // 16-column blocks per TMEM round trip: all 64 heads with registers to
    // spare (four epilogue warps), 32 heads under the 16-warp register cap
    static constexpr int kBlocksPerTrip = kEpi == 4 ? 4 : 2;
};

struct ScoreParams {
    const uint16_t *q_idx;
    const float *w;
    float *scores;
    int64_t ld;
    DevBatch b;
    uint32_t *status;
    RowMap rows;
    int H_I, HP, G;           // heads, padded heads, tokens per group
    int NQ, NP, halves;       // query operand rows G*HP; MMA N of a step NQ/halves (<= 256); steps per tile
    int hadamard_q;
    int fill_masked;
    int depends;
    int fuse_append;
    const void *k_new;
    int k_dtype;
    uint16_t *k_cache;
    int hadamard_k;
    int tiles_per_cta;
    int stages;
    int early;                // trigger dependents at the start (see launch_score)
    int balance;              // one token per sequence: CTAs shared out by sequence length (see below)
    int groups_per_seq;
    uint32_t tmem_cols;
};

struct Smem {
    uint4 new_key[16];        // the appended key row (fp16, row-major), fused-append mode
    float4 w4[128];           // head weights of the group's tokens (HP per token)
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t q_ready;
    uint32_t tmem_base;
    int32_t abort_flag;
    int32_t meta_q0, meta_q1, meta_max_p;
    int64_t meta_kv0;
    int32_t spec_tok, spec_pos;   // a token whose stored position is already loaded (-1: none)
    int32_t pos[kMaxGroup];
    int64_t out_row[kMaxGroup];
    uint32_t bal_warp[32];    // balanced chunking: per-warp sums
    int32_t bal_seq, bal_lo, bal_hi;
};

// Two halves of 256 columns (a 512-row query operand) leave room for a
// 3-deep ring -- with no slack for realigning the dynamic shared memory.
static_assert(512 * 256 + 3 * kTileBytes + sizeof(Smem) <= kSmemLimit, "score ring does not fit");

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Smem &sm,
                                         uint32_t *status, uint64_t limit_ns) {
    if (*(volatile int32_t *)&sm.abort_flag) return false;
    if (mbar_wait(bar, parity, limit_ns)) return true;
    *(volatile int32_t *)&sm.abort_flag = 1;
    flag(status, DSA_DEV_TIMEOUT);
    return false;
}

// One 128-element query row is held 4 values per lane (lane l: 4l..4l+3).
__device__ __forceinline__ uint2 load_q_row(const uint16_t *src, bool valid, int lane) {
    return valid ? __ldg(reinterpret_cast<const uint2 *>(src) + lane) : make_uint2(0u, 0u);
}

// Rotate (optionally) a query row, split it into fp16 hi (+ lo) parts and
// store them at row n of the SW128 K-major operand.
__device__ __forceinline__ void store_q_row(uint2 x, int hadamard, uint8_t *q_hi, uint8_t *q_lo, int NQ,
                                            int n, int lane) {
    float v[4];
    v[0] = __half2float(__ushort_as_half((unsigned short)(x.x & 0xFFFF)));
    v[1] = __half2float(__ushort_as_half((unsigned short)(x.x >> 16)));
    v[2] = __half2float(__ushort_as_half((unsigned short)(x.y & 0xFFFF)));
    v[3] = __half2float(__ushort_as_half((unsigned short)(x.y >> 16)));
    uint16_t hi[4], lo[4];
    if (hadamard) {
        float a, c;
        a = v[0]; c = v[1]; v[0] = a + c; v[1] = a - c;
        a = v[2]; c = v[3]; v[2] = a + c; v[3] = a - c;
        a = v[0]; c = v[2]; v[0] = a + c; v[2] = a - c;
        a = v[1]; c = v[3]; v[1] = a + c; v[3] = a - c;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float other = __shfl_xor_sync(0xffffffffu, v[e], m);
                v[e] = upper ? other - v[e] : v[e] + other;
            }
        }
        const float scale = 0.08838834764831845f;  // 1/sqrt(128)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float y = v[e] * scale;
            const __half h = __float2half_rn(y);
            hi[e] = __half_as_ushort(h);
            lo[e] = __half_as_ushort(__float2half_rn(y - __half2float(h)));
        }
    } else {
        hi[0] = (uint16_t)(x.x & 0xFFFF); hi[1] = (uint16_t)(x.x >> 16);
        hi[2] = (uint16_t)(x.y & 0xFFFF); hi[3] = (uint16_t)(x.y >> 16);
    }
    // element 4*lane: K block lane/16, chunk (lane%16)/2, half-chunk lane%2
    const int kb = lane >> 4;
    const uint32_t off = (uint32_t)kb * (uint32_t)(NQ * 128) +
                         sw128_offset((uint32_t)n, (uint32_t)((lane & 15) >> 1)) + (lane & 1) * 8;
    uint2 o;
    o.x = (uint32_t)hi[0] | ((uint32_t)hi[1] << 16);
    o.y = (uint32_t)hi[2] | ((uint32_t)hi[3] << 16);
    *reinterpret_cast<uint2 *>(q_hi + off) = o;
    if (hadamard) {
        o.x = (uint32_t)lo[0] | ((uint32_t)lo[1] << 16);
        o.y = (uint32_t)lo[2] | ((uint32_t)lo[3] << 16);
        *reinterpret_cast<uint2 *>(q_lo + off) = o;
    }
}

// The token's new key in storage form: lane l returns fp16 elements 4l..4l+3
// of fp16(hadamard ? H k / sqrt(128) : k).  The transform runs in float64,
// where every partial sum of the butterflies is exact for fp16 inputs, so the
// single rounding to fp16 happens on the exact value.
__device__ __forceinline__ uint2 appended_key(const void *k_new, int k_dtype, int t, int hadamard, int lane) {
    double v[4];
    if (k_dtype == DSA_KEY_F32) {
        const float4 x = __ldg(reinterpret_cast<const float4 *>(k_new) + (int64_t)t * 32 + lane);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else {
        const uint2 x = __ldg(reinterpret_cast<const uint2 *>(k_new) + (int64_t)t * 32 + lane);
        v[0] = __half2float(__ushort_as_half((unsigned short)(x.x & 0xFFFF)));
        v[1] = __half2float(__ushort_as_half((unsigned short)(x.x >> 16)));
        v[2] = __half2float(__ushort_as_half((unsigned short)(x.y & 0xFFFF)));
        v[3] = __half2float(__ushort_as_half((unsigned short)(x.y >> 16)));
    }
    if (hadamard) {
        double a, c;
        a = v[0]; c = v[1]; v[0] = a + c; v[1] = a - c;
        a = v[2]; c = v[3]; v[2] = a + c; v[3] = a - c;
        a = v[0]; c = v[2]; v[0] = a + c; v[2] = a - c;
        a = v[1]; c = v[3]; v[1] = a + c; v[3] = a - c;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const double other = __shfl_xor_sync(0xffffffffu, v[e], m);
                v[e] = upper ? other - v[e] : v[e] + other;
            }
        }
        const double scale = 1.0 / sqrt(128.0);
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] *= scale;
    }
    uint2 o;
    o.x = (uint32_t)__half_as_ushort(__double2half(v[0])) | ((uint32_t)__half_as_ushort(__double2half(v[1])) << 16);
    o.y = (uint32_t)__half_as_ushort(__double2half(v[2])) | ((uint32_t)__half_as_ushort(__double2half(v[3])) << 16);
    return o;
}

}  // namespace

template <int kEpi>
__global__ void __launch_bounds__(ScoreCfg<kEpi>::kThreads, kEpi >= 8 ? 1 : 2)
    score_kernel(const ScoreParams p, const __grid_constant__ CUtensorMap k_map) {
    constexpr int kEpiWarps = ScoreCfg<kEpi>::kEpiWarps;
    constexpr int kQuarterWarps = ScoreCfg<kEpi>::kQuarterWarps;
    constexpr int kBT = ScoreCfg<kEpi>::kBlocksPerTrip;
    // The operand region (SW128 atoms: 1024-byte aligned) starts the dynamic
    // shared memory, then the control block.  The launch requests no slack
    // for realignment (the deepest ring leaves a few hundred bytes of the
    // 227 KB), so a misaligned window skips the work and says so.
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) flag(p.status, DSA_DEV_SMEM_LAYOUT);
        return;
    }
    uint8_t *base = smem_raw;
    const int q_bytes = p.NQ * 256;                      // two 64-column K blocks
    uint8_t *q_hi = base;
    uint8_t *q_lo = base + q_bytes;                      // used with hadamard_q
    uint8_t *stages = base + q_bytes * (p.hadamard_q ? 2 : 1);
    const int n_stages = p.stages;
    Smem &sm = *reinterpret_cast<Smem *>(stages + n_stages * kTileBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DevBatch &b = p.b;
    tl_start(b.timeline, kTlScore);
    if (p.early) pdl_trigger();
    if (warp == 0 && lane == 0) tma_prefetch_desc(&k_map);   // fetched while the batch data loads

    // Barriers and tensor memory.  Balanced decode grids set up while their
    // batch loads are in flight; the others once the positions are known:
    // on GB300 (batched decode, 8 x 8192 keys, cold L2) allocating the tensor
    // memory at the start made this kernel 0.7 us faster but left the
    // attention kernel that follows 5-6 us slower, for a reason not found.
    auto set_up = [&]() {
        if (threadIdx.x == 64) {
            for (int s = 0; s < n_stages; ++s) {
                mbar_init(smem_u32(&sm.full[s]), 1);
                mbar_init(smem_u32(&sm.empty[s]), 1);
            }
            for (int s = 0; s < 2; ++s) {
                mbar_init(smem_u32(&sm.acc_full[s]), 1);
                mbar_init(smem_u32(&sm.acc_empty[s]), kEpiWarps);
            }
            mbar_init(smem_u32(&sm.q_ready), kEpiWarps);
            sm.abort_flag = 0;
            fence_mbar_init();
        }
        if (warp == 1) {
            tmem_alloc(smem_u32(&sm.tmem_base), p.tmem_cols);
            tmem_relinquish();
        }
    };
    // Every return after the set-up gives the tensor memory back.
    bool have_tmem = false;
    auto release = [&](uint32_t tm) {
        if (have_tmem && warp == 1) {
            tc_fence_after();
            tmem_dealloc(tm, p.tmem_cols);
        }
    };
    // The last visible position of a token from its stored position.
    auto visible = [&](int q) { return b.pool_log2 ? ((q + 1) >> b.pool_log2) - 1 : q; };

    // ---- which tokens and keys this CTA covers (uniform across the CTA).
    // One-token groups (decode) load their token's position in the same round
    // trip as the batch offsets, on the guess that sequence s's token is
    // token s (every sequence has exactly one); the guess is checked, and a
    // wrong one costs a second load.
    int seq, grp, tile_lo = 0, tile_cnt = p.tiles_per_cta;
    uint32_t tmem;
    if (p.balance) {
        // One token per sequence, at most one sequence per thread: sequence s,
        // whose token sees n_s key tiles, gets c_s = min(ceil(n_s / 2),
        // 1 + n_s (G - B) / sum n) of the G CTAs (at most G in all, each with
        // two tiles or more), CTA j of them the tiles [j n_s / c_s,
        // (j + 1) n_s / c_s): every CTA streams about the same number of tiles
        // however the lengths differ.  Every CTA computes the same shares.
        const int nthreads = (int)blockDim.x, tid = (int)threadIdx.x;
        const int G = (int)gridDim.x;
        uint32_t n_s = 0;
        int my_q0 = 0, my_q1 = 0, my_raw = -1;
        int64_t my_kv = 0;
        int guess = -1;
        if (tid < b.B) {
            my_q0 = __ldg(b.cu_q + tid);
            my_q1 = __ldg(b.cu_q + tid + 1);
            guess = __ldg(b.q_pos + min(tid, b.T - 1));
            my_kv = seq_base(b, tid);
        }
        set_up();
        if (tid < b.B) {
            // a sequence that gets no CTA is checked here (a sequence may have
            // no token; pool mode: -1 is an empty row)
            bool bad = my_q0 < 0 || my_q1 > b.T || my_q1 < my_q0 || my_q1 - my_q0 > b.max_q;
            if (!bad && my_q1 > my_q0) {
                my_raw = my_q0 == tid ? guess : __ldg(b.q_pos + my_q0);
                const int pos = visible(my_raw);
                if (pos >= 0 && pos < b.max_kv) n_s = (uint32_t)(pos / kTileKeys) + 1u;
                else bad = !(b.pool_log2 && pos == -1);
            }
            if (bad && blockIdx.x == 0) flag(p.status, DSA_DEV_BAD_POSITION);
        }
        if (tid == 0) sm.bal_seq = -1;
        uint32_t v = n_s;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) sm.bal_warp[warp] = v;
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        tmem = sm.tmem_base;
        have_tmem = true;
        uint32_t total = 0;
        for (int w = 0; w < nthreads / 32; ++w) total += sm.bal_warp[w];
        uint32_t c_s = 0;
        if (n_s > 0) {
            const uint64_t share = 1u + (uint64_t)n_s * (uint64_t)(G - b.B) / total;
            const uint64_t half = (n_s + 1u) / 2u;
            c_s = (uint32_t)(share < half ? share : half);
        }
        uint32_t incl = c_s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        __syncthreads();                                 // the totals above are read
        if (lane == 31) sm.bal_warp[warp] = incl;
        __syncthreads();
        uint32_t pre = incl - c_s;
        for (int w = 0; w < warp; ++w) pre += sm.bal_warp[w];
        const uint32_t cta = blockIdx.x;
        if (c_s > 0 && pre <= cta && cta < pre + c_s) {
            // the owning thread knows the sequence's offsets and position
            const uint32_t j = cta - pre;
            sm.bal_seq = tid;
            sm.bal_lo = (int)(j * n_s / c_s);
            sm.bal_hi = (int)((j + 1u) * n_s / c_s);
            sm.meta_q0 = my_q0;
            sm.meta_q1 = my_q1;
            sm.meta_kv0 = my_kv;
            sm.spec_tok = my_q0;
            sm.spec_pos = my_raw;
        }
        __syncthreads();
        if (sm.bal_seq < 0) {                            // more CTAs than shares
            release(tmem);
            return;
        }
        seq = sm.bal_seq;
        grp = 0;
        tile_lo = sm.bal_lo;
        tile_cnt = sm.bal_hi - sm.bal_lo;
    } else {
        seq = blockIdx.y / p.groups_per_seq;
        // later groups of a sequence see more keys: launch them first, so that
        // the last wave holds the shortest CTAs (measured on GB300, 4096 tokens
        // after 4096: 3% off the scoring)
        grp = p.groups_per_seq - 1 - (int)(blockIdx.y % p.groups_per_seq);
        if (seq >= b.B) return;
        if (threadIdx.x == 0) {                   // independent loads, one round trip
            const int q0 = __ldg(b.cu_q + seq);
            const int q1 = __ldg(b.cu_q + seq + 1);
            const int64_t kv0 = seq_base(b, seq);
            const bool guess = p.G == 1 && seq < b.T;
            const int gp = guess ? __ldg(b.q_pos + seq) : -1;
            sm.meta_q0 = q0;
            sm.meta_q1 = q1;
            sm.meta_kv0 = kv0;
            sm.spec_tok = guess ? seq : -1;
            sm.spec_pos = gp;
        }
        __syncthreads();
        tmem = 0;
    }
    const int q0 = sm.meta_q0, q1 = sm.meta_q1;
    const int64_t kv0 = sm.meta_kv0;
    const int n_seq = q1 - q0;
    if (q0 < 0 || q1 > b.T || n_seq < 0 || n_seq > b.max_q) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && grp == 0) flag(p.status, DSA_DEV_BAD_POSITION);
        release(tmem);
        return;
    }
    const int win_lo = p.rows.slab ? p.rows.j0 : 0;
    const int win_hi = p.rows.slab ? min(p.rows.j0 + p.rows.J, n_seq) : n_seq;
    const int j_lo = win_lo + grp * p.G;
    const int j_hi = min(j_lo + p.G, win_hi);
    if (j_lo >= j_hi) {
        release(tmem);
        return;
    }
    const int g = j_hi - j_lo;
    const int tph = p.G / p.halves;               // tokens per half
    const int hv = (p.halves == 2 && g > tph) ? 2 : 1;   // MMA steps per tile
    if ((int)threadIdx.x < g) {                   // the group's positions, in parallel
        const int i = threadIdx.x;
        const int t = q0 + j_lo + i;
        const int pos = visible(t == sm.spec_tok ? sm.spec_pos : __ldg(b.q_pos + t));   // a pool index in pool mode
        bool ok = pos >= 0 && pos < b.max_kv && kv0 >= 0;
        if (ok) {
            const int64_t row = cache_row(b, seq, kv0, pos);
            ok = row >= 0 && row < b.cache_rows;
        }
        const bool empty = b.pool_log2 && pos == -1;  // no complete pool yet: nothing to score
        if (!ok && !empty) flag(p.status, DSA_DEV_BAD_POSITION);
        sm.pos[i] = ok ? pos : -1;
        sm.out_row[i] = p.rows.slab ? (int64_t)seq * p.rows.J + (j_lo + i - p.rows.j0) : (int64_t)t;
    }
    __syncthreads();
    if (!p.balance) {
        set_up();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        tmem = sm.tmem_base;
        have_tmem = true;
    }
    int max_p = -1;
    for (int i = 0; i < g; ++i) max_p = max(max_p, sm.pos[i]);
    const int64_t chunk0 = p.balance ? (int64_t)tile_lo * kTileKeys : (int64_t)blockIdx.x * p.tiles_per_cta * kTileKeys;
    int n_mma = 0;
    if (max_p >= chunk0)
        n_mma = (int)min((int64_t)tile_cnt, (max_p - chunk0) / kTileKeys + 1);
    int n_tiles = n_mma;
    if (p.fill_masked) {
        const int64_t left = p.ld - chunk0;
        n_tiles = left <= 0 ? 0 : (int)min((int64_t)tile_cnt, (left + kTileKeys - 1) / kTileKeys);
        n_tiles = max(n_tiles, n_mma);
    }
    if (n_tiles == 0) {
        release(tmem);
        return;
    }
    // With a single query token in the sequence, only the tile holding its own
    // (just appended) key depends on the preceding kernel; otherwise all do.
    int first_dependent = n_mma;
    if (p.depends == 2 || (p.depends == 1 && n_seq > 1)) first_dependent = 0;
    else if (p.depends == 1 && n_mma > 0 && (max_p - chunk0) / kTileKeys < tile_cnt)
        first_dependent = n_mma - 1;
    // Fused append: this CTA holds the tile of the token's own position.
    const int append_tile = (p.fuse_append && n_seq == 1 && n_mma > 0 &&
                             (max_p - chunk0) / kTileKeys < tile_cnt) ? n_mma - 1 : -1;

    if (warp == 0) {
        // ---------------- TMA producer (issues nothing under the failure-path
        // test hook, so that the MMA issuer's first wait runs out)
        if (lane == 0 && !b.skip_copies) {
            for (int i = 0; i < n_mma; ++i) {
                const int s = i % n_stages;
                const uint32_t k = (uint32_t)(i / n_stages);
                if (i == first_dependent) pdl_wait();
                if (!wait_bar(smem_u32(&sm.empty[s]), (k & 1) ^ 1, sm, p.status, b.wait_ns)) break;
                const uint32_t full = smem_u32(&sm.full[s]);
                mbar_arrive_expect_tx(full, kTileBytes);
                const uint32_t dst = smem_u32(stages + s * kTileBytes);
                const int p0 = (int)(chunk0 + (int64_t)i * kTileKeys);
                if (!b.block_table) {
                    const int32_t row = (int32_t)(kv0 + p0);
                    tma_load_2d(dst, &k_map, full, 0, row);
                    tma_load_2d(dst + kTileBytes / 2, &k_map, full, 64, row);
                } else {
                    // paged: a 128-key tile is one block span when the block
                    // size is a multiple of 128, else two 64-row halves (the
                    // map's box is then 64 rows).  Positions past the
                    // sequence's blocks load the fill value (row cache_rows).
                    const int halves = b.block_size % kTileKeys == 0 ? 1 : 2;
                    for (int h = 0; h < halves; ++h) {
                        const int ph = p0 + h * 64;
                        int64_t r = ph < b.max_kv ? cache_row(b, seq, kv0, ph) : -1;
                        if (r < 0 || r >= b.cache_rows) r = b.cache_rows;
                        tma_load_2d(dst + h * 8192, &k_map, full, 0, (int32_t)r);
                        tma_load_2d(dst + kTileBytes / 2 + h * 8192, &k_map, full, 64, (int32_t)r);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer.  It first computes the appended key (its
        // load and rotation overlap the tile loads the producer has issued).
        if (append_tile >= 0) {
            const int t = q0 + j_lo;
            const uint2 kv = appended_key(p.k_new, p.k_dtype, t, p.hadamard_k, lane);
            reinterpret_cast<uint2 *>(p.k_cache + cache_row(b, seq, kv0, max_p) * D_I)[lane] = kv;   // persist
            reinterpret_cast<uint2 *>(sm.new_key)[lane] = kv;                        // staging
            __syncwarp();
        }
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(128, p.NP, false, false, false);
            const uint32_t qh = smem_u32(q_hi), ql = smem_u32(q_lo);
            const uint32_t qblk = (uint32_t)p.NQ * 128u;
            // the 8 (16 with the lo query part) MMAs of one step: keys of stage
            // buffer a0 against query rows [qrow0, qrow0 + NP) into column d
            auto issue_step = [&](uint32_t d, uint32_t a0, uint32_t qrow0) {
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint32_t koff = (uint32_t)(kb * (kTileBytes / 2) + ks * 32);
                        const uint64_t ad = sdesc_sw128(a0 + koff, 16, 1024);
                        const uint32_t boff = (uint32_t)kb * qblk + qrow0 * 128u + (uint32_t)ks * 32;
                        umma_f16(d, ad, sdesc_sw128(qh + boff, 16, 1024), idesc, (kb | ks) != 0);
                        if (p.hadamard_q) umma_f16(d, ad, sdesc_sw128(ql + boff, 16, 1024), idesc, 1);
                    }
                }
            };
            // replace the stale cache row loaded by TMA with the new key
            auto patch_append = [&](int i, int s) {
                const uint32_t r = (uint32_t)(max_p - (chunk0 + (int64_t)i * kTileKeys));
                uint8_t *tile = stages + s * kTileBytes;
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    *reinterpret_cast<uint4 *>(tile + (c >> 3) * (kTileBytes / 2) + sw128_offset(r, c & 7)) =
                        sm.new_key[c];
                fence_proxy_async_smem();
            };
            if (!wait_bar(smem_u32(&sm.q_ready), 0, sm, p.status, b.wait_ns)) {
                // the loops below are skipped
            } else if constexpr (kEpi == 4) {
                tc_fence_after();
                // one token: one step per tile, the stage released before the
                // accumulator is signalled (measured on GB300, ragged
                // long-context decode: 7 us per step faster than the general
                // loop; issuing the step from a rolled loop over its K slices
                // was slower by 0.4 us)
                for (int i = 0; i < n_mma; ++i) {
                    const int s = i % n_stages;
                    const uint32_t k = (uint32_t)(i / n_stages);
                    const int buf = i & 1;
                    const uint32_t ka = (uint32_t)(i >> 1);
                    if (!wait_bar(smem_u32(&sm.acc_empty[buf]), (ka & 1) ^ 1, sm, p.status, b.wait_ns)) break;
                    if (!wait_bar(smem_u32(&sm.full[s]), k & 1, sm, p.status, b.wait_ns)) break;
                    tc_fence_after();
                    if (i == append_tile) patch_append(i, s);
                    issue_step(tmem + (uint32_t)(buf * p.NP), smem_u32(stages + s * kTileBytes), 0);
                    umma_commit(smem_u32(&sm.empty[s]));
                    umma_commit(smem_u32(&sm.acc_full[buf]));
                }
            } else {
                tc_fence_after();
                for (int i = 0; i < n_mma; ++i) {
                    const int s = i % n_stages;
                    const uint32_t k = (uint32_t)(i / n_stages);
                    if (!wait_bar(smem_u32(&sm.full[s]), k & 1, sm, p.status, b.wait_ns)) break;
                    tc_fence_after();
                    if (i == append_tile) patch_append(i, s);
                    const uint32_t a0 = smem_u32(stages + s * kTileBytes);
                    bool ok = true;
#pragma unroll 1
                    for (int h = 0; h < hv; ++h) {
                        const uint32_t u = (uint32_t)(i * hv + h);   // MMA step: accumulator u & 1
                        if (!wait_bar(smem_u32(&sm.acc_empty[u & 1]), ((u >> 1) & 1) ^ 1, sm, p.status, b.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_step(tmem + (u & 1) * (uint32_t)p.NP, a0, (uint32_t)(h * p.NP));
                        umma_commit(smem_u32(&sm.acc_full[u & 1]));
                    }
                    if (!ok) break;
                    umma_commit(smem_u32(&sm.empty[s]));   // the tile's last MMA step read it
                }
            }
        }
    } else {
        // ---------------- query staging + epilogue
        const int ew = warp - 2;  // 0..kEpiWarps-1
        // head weights: this thread's first one is loaded beside the first
        // query rows (one round trip for both), the rest (none for the
        // shapes launched: NQ <= 32 kEpiWarps) after them
        auto weight_at = [&](int i) -> float {
            const int tok = i / p.HP, h = i % p.HP;
            return (tok < g && h < p.H_I && sm.pos[tok] >= 0) ? __ldg(p.w + (int64_t)(q0 + j_lo + tok) * p.H_I + h)
                                                                : 0.f;
        };
        const int wi0 = (int)threadIdx.x - 64;
        const float w0 = wi0 < p.NQ ? weight_at(wi0) : 0.f;
        // stage query rows n = tok*HP + h; each warp keeps 8 row loads in flight
        for (int n0 = ew; n0 < p.NQ; n0 += 8 * kEpiWarps) {
            uint2 x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int n = n0 + u * kEpiWarps;
                const int tok = n / p.HP, h = n % p.HP;
                const bool valid = n < p.NQ && tok < g && h < p.H_I;
                x[u] = load_q_row(p.q_idx + ((int64_t)(q0 + j_lo + (valid ? tok : 0)) * p.H_I + (valid ? h : 0)) * D_I,
                                  valid, lane);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int n = n0 + u * kEpiWarps;
                if (n < p.NQ) store_q_row(x[u], p.hadamard_q, q_hi, q_lo, p.NQ, n, lane);
            }
        }
        if (wi0 < p.NQ) reinterpret_cast<float *>(sm.w4)[wi0] = w0;
        for (int i = wi0 + 32 * kEpiWarps; i < p.NQ; i += 32 * kEpiWarps) reinterpret_cast<float *>(sm.w4)[i] = weight_at(i);
        fence_proxy_async_smem();
        named_barrier(1, 32 * kEpiWarps);     // weights and positions visible to all epilogue warps
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.q_ready));

        const int quarter = warp & 3;         // TMEM lanes this warp may access
        const int part = ew >> 2;             // which part of each half's tokens
        const int r = quarter * 32 + lane;    // key row within a tile
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const int hp16 = p.HP >> 4;
        const int tpw = (tph + kQuarterWarps - 1) / kQuarterWarps;
        const int lo_h = min(tph, part * tpw), hi_h = min(tph, lo_h + tpw);   // within a half
        bool aborted = false;
        const uint32_t n_steps = (uint32_t)(n_mma * hv);
        for (uint32_t u = 0; u < n_steps; ++u) {     // MMA step u: tile u / hv, half u % hv, accumulator u & 1
            const int i = hv == 2 ? (int)(u >> 1) : (int)u;
            const int h = (int)u & (hv - 1);
            const int64_t s = chunk0 + (int64_t)i * kTileKeys + r;
            const int buf = (int)(u & 1);
            if (!wait_bar(smem_u32(&sm.acc_full[buf]), (u >> 1) & 1, sm, p.status, b.wait_ns)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const int tok_lo = min(g, h * tph + lo_h), tok_hi = min(g, h * tph + hi_h);
            // kBT 16-column loads per TMEM round trip, accumulated in head order
            for (int tok = tok_lo; tok < tok_hi; ++tok) {
                const uint32_t col = tmem + lane_addr + (uint32_t)(buf * p.NP + (tok - h * tph) * p.HP);
                const float4 *wt = sm.w4 + (tok * p.HP >> 2);   // broadcast 16-byte loads
                float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int c0 = 0; c0 < 4; c0 += kBT) {
                    if (c0 < hp16) {
                        uint32_t v[kBT][16];
#pragma unroll
                        for (int c = 0; c < kBT; ++c)
                            if (c0 + c < hp16) tmem_ld16(col + 16 * (c0 + c), v[c]);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < kBT; ++c) {
                            if (c0 + c < hp16) {
#pragma unroll
                                for (int j = 0; j < 16; j += 4) {
                                    const float4 w = wt[4 * (c0 + c) + (j >> 2)];
                                    const float2 r01 = make_float2(fmaxf(__uint_as_float(v[c][j]), 0.f),
                                                                   fmaxf(__uint_as_float(v[c][j + 1]), 0.f));
                                    const float2 r23 = make_float2(fmaxf(__uint_as_float(v[c][j + 2]), 0.f),
                                                                   fmaxf(__uint_as_float(v[c][j + 3]), 0.f));
                                    acc2 = __ffma2_rn(make_float2(w.x, w.y), r01, acc2);
                                    acc2 = __ffma2_rn(make_float2(w.z, w.w), r23, acc2);
                                }
                            }
                        }
                    }
                }
                const float acc = acc2.x + acc2.y;
                const int pos = sm.pos[tok];
                float *dst = p.scores + sm.out_row[tok] * p.ld;
                if (s <= pos) dst[s] = acc;
                else if (p.fill_masked && s < p.ld) dst[s] = -INFINITY;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.acc_empty[buf]));
        }
        // tiles beyond every token's position (fill_masked)
        for (int i = n_mma; i < n_tiles && !aborted; ++i) {
            const int64_t s = chunk0 + (int64_t)i * kTileKeys + r;
            for (int h = 0; h < hv; ++h)
                for (int tok = min(g, h * tph + lo_h); tok < min(g, h * tph + hi_h); ++tok)
                    if (s < p.ld) p.scores[sm.out_row[tok] * p.ld + s] = -INFINITY;
        }
    }

    tc_fence_before();
    __syncwarp();                  // lanes of warps 0 and 1 arrive from different paths
    __syncthreads();
    // A CTA whose tiles did not depend on the preceding kernel never waited
    // for it; waiting here keeps this grid from completing before it, so that
    // kernels further down the stream may rely on it having completed too.
    if (p.depends && threadIdx.x == 0) pdl_wait();
    if (!p.early) pdl_trigger();   // late: waiting dependents would share the SMs
    tl_end(b.timeline, kTlScore);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, p.tmem_cols);
    }
}

size_t score_smem_bytes(int n_rows, int hadamard_q, int n_stages) {
    return (size_t)n_rows * 256 * (hadamard_q ? 2 : 1) + (size_t)n_stages * kTileBytes + sizeof(Smem);
}

cudaError_t launch_score(const ScoreLaunch &a, const CUtensorMap &k_map, const DevBatch &b,
                         uint32_t *status, cudaStream_t stream, bool pdl) {
    ScoreParams p{};
    p.q_idx = a.q_idx;
    p.w = a.w;
    p.scores = a.scores;
    p.ld = a.ld;
    p.b = b;
    p.status = status;
    p.rows = a.rows;
    p.H_I = a.H_I;
    p.HP = (a.H_I + 15) / 16 * 16;
    const int n_max = a.hadamard_q ? 128 : 256;             // MMA N of one step
    const int window = a.rows.slab ? a.rows.J : b.max_q;
    const int g1 = max(1, min(n_max / p.HP, window));       // tokens per step
    // Multi-token groups without the rotation's second (lo) operand take two
    // steps per key tile; with it the doubled query operand would not leave
    // room for the ring.
    p.halves = (!a.hadamard_q && g1 > 1 && window > g1) ? 2 : 1;
    p.G = g1 * p.halves;
    p.NP = g1 * p.HP;
    p.NQ = p.G * p.HP;
    if (p.G > kMaxGroup) return cudaErrorInvalidConfiguration;
    p.hadamard_q = a.hadamard_q;
    p.fill_masked = a.fill_masked;
    p.depends = a.depends;
    p.fuse_append = a.fuse_append;
    p.k_new = a.k_new;
    p.k_dtype = a.k_dtype;
    p.k_cache = a.k_cache;
    p.hadamard_k = a.hadamard_k;
    p.groups_per_seq = (window + p.G - 1) / p.G;
    uint32_t cols = 32;
    while (cols < (uint32_t)(2 * p.NP)) cols <<= 1;
    p.tmem_cols = cols;

    const int64_t span = a.fill_masked ? a.ld : (int64_t)b.max_kv;
    const int64_t tiles = (span + kTileKeys - 1) / kTileKeys;
    const int64_t work = tiles * (int64_t)b.B * p.groups_per_seq;
    // About two CTAs' worth of tiles per SM.
    int64_t tpc = (work + 2 * 152 - 1) / (2 * 152);
    tpc = std::max<int64_t>(2, std::min<int64_t>(64, tpc));
    p.tiles_per_cta = (int)tpc;
    // One-token groups (decode variant, launched two CTAs per SM) use a
    // 2-deep ring so that two CTAs fit: measured on GB300 on the ragged
    // long-context decode, 90 us against 128 us with a 4-deep ring at one CTA
    // per SM.
    p.stages = (p.G == 1 || tpc <= 2) ? 2 : kMaxStages;
    while (p.stages > 2 && score_smem_bytes(p.NQ, p.hadamard_q, p.stages) > kSmemLimit) --p.stages;
    int64_t chunks = (tiles + tpc - 1) / tpc;
    int64_t groups = (int64_t)b.B * p.groups_per_seq;
    if (groups > 65535 || chunks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    // One token per sequence (decode) with long rows (chunks of more than two
    // tiles): a grid of one wave (two CTAs per SM) whose CTAs share the
    // sequences' tiles out by length on the device, so that ragged batches do
    // not leave a few SMs streaming the longest sequences (see the kernel;
    // measured on GB300, 32 sequences of 4k-64k keys: 75.1 -> 57.1 us).  With
    // short rows the fixed chunks are already even and the shares' extra
    // round trip would cost more (8 x 8192 keys: 8.8 -> 10.6 us).  Shares
    // need one sequence per thread.
    p.balance = (p.G == 1 && b.max_q == 1 && !a.fill_masked && tpc > 2 && b.B <= ScoreCfg<4>::kThreads &&
                 b.B < kSMs) ? 1 : 0;
    if (p.balance) {
        chunks = 2 * kSMs;
        groups = 1;
    }

    const size_t smem = score_smem_bytes(p.NQ, p.hadamard_q, p.stages);
    if (smem > kSmemLimit) return cudaErrorInvalidConfiguration;
    const size_t smem_max = kSmemLimit;
    dim3 grid((unsigned)chunks, (unsigned)groups);
    // One wave of this kernel (decode variant: two CTAs per SM) followed by a
    // small dependent grid: that grid can start on the SMs left free.
    p.early = (a.early_ok && p.G == 1 && chunks * groups <= 2 * kSMs) ? 1 : 0;
    if (p.G == 1) {                                    // one token per group: lean decode variant
        cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(score_kernel<4>), 3, smem_max);
        if (e != cudaSuccess) return e;
        return launch_k(score_kernel<4>, grid, dim3(ScoreCfg<4>::kThreads), smem, stream, pdl, p, k_map);
    }
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(score_kernel<16>), 4, smem_max);
    if (e != cudaSuccess) return e;
    return launch_k(score_kernel<16>, grid, dim3(ScoreCfg<16>::kThreads), smem, stream, pdl, p, k_map);
}

}  // namespace dsa
