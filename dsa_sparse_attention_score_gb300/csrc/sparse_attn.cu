// sparse_attn.cu -- sparse MLA attention over the selected latent rows.
//
// ds4 PR #523 "hy3: Metal decode path + shared gate/up fusion", milestone M3
// (glm_mla_attention_one): each cached row is 576 wide -- the 512-d kv latent
// plus the 64-d rotated rope tail; scores use both parts, one softmax runs over
// the candidate rows, values come from the latent.  In the absorbed form of
// ik_llama_opt "MLA tensor parallelism under -sm graph" (wk_b / wv_b) the
// queries arrive pre-multiplied by W_UK and the output stays in the latent:
//     z_j = sm_scale * (q_lat . c_j[0:512] + q_rope . c_j[512:576]),
//     o   = sum_j softmax(z)_j c_j[0:512].
//
// One CTA per (token, head group, split) handles a run of 64-row tiles of the
// token's selected positions, with a group of 64 of the token's heads on the
// N side of every MMA (up to 128 heads run as two groups that share nothing
// but the L2 lines of the gathered rows):
//     S^T[row, head]  = C[row, 0:576] . Q[head, 0:576]^T        (M=64, N=64, K=576)
//     O^T[dim, head] += C[row, dim]^T . P^T[row, head]           (M=4x128, N=64, K=64)
// A gathered tile C sits in shared memory as nine 64-column SWIZZLE_128B
// blocks (TMA tile::gather4, four rows per request).  Without a rope tail
// (MLA-NoPE: vllm-rdna PR #2 "Glm5Next (GLM-5.3-Flash) on gfx1030", 512-d
// latent rows) eight blocks are gathered and multiplied, and the ninth only
// holds P^T.  The same bytes serve as
// the K-major A operand of S^T and, for the latent blocks, as the MN-major A
// operand of O^T, so V is never copied.  The rope block is dead once S^T is
// computed and holds P^T (bf16) for the second MMA.
//
// Two tile buffers (2 x 72 KB) beside the queries (72 KB): four producer
// warps gather tile i+1 while the tensor core and the softmax warps work on
// tile i; the MMA warp issues S^T and O^T products as their inputs arrive,
// so the softmax of one tile overlaps the score product of the next.  Softmax
// runs in eight warps; an M=64 accumulator puts row m in TMEM lane
// 32 (m / 16) + m % 16, so lanes 0..15 of each lane quarter hold 16 key rows,
// read by the two warps of the quarter (heads 0..31 and 32..63), each warp's
// two halves taking 16 heads.
// The per-head running maximum is only raised when a tile exceeds it by more
// than 2^8 (lazy rescale of the TMEM accumulator); the final normalisation
// makes the result exact either way.  With several splits per token, each
// split's unnormalised output O (rounded to bf16, which keeps float32's
// exponent range) and its (m, l) in float32 go to the workspace, and a
// combine kernel merges them.
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {

namespace {

constexpr int kHeads = 64;                    // heads per CTA (padded)
constexpr int kRows = 64;                     // gathered rows per tile
constexpr int kBlocks = 9;                    // 576 / 64 columns
constexpr int kQBlockBytes = kHeads * 128;    // 8 KB
constexpr int kCBlockBytes = kRows * 128;     // 8 KB
constexpr int kQBytes = kBlocks * kQBlockBytes;
constexpr int kCBytes = kBlocks * kCBlockBytes;   // one tile buffer
constexpr int kBufs = 2;
constexpr int kSoftmaxWarps = 8;              // warps 0..7: two per TMEM lane quarter
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kMmaWarp = 8;
constexpr int kProducerWarps = 4;             // warps 9..12
constexpr int kThreads = 32 * (kSoftmaxWarps + 1 + kProducerWarps);
constexpr int kProducers = 32 * kProducerWarps;
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t kTmemCols = 512;           // S: 2 x 64 cols, O^T: 4 x 64 cols
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;

struct AttnParams {
    const uint8_t *kv;       // the latent cache (16-byte aligned rows), for the cp.async gather
    const int32_t *idx;
    float *out;
    float *lse;
    uint16_t *part_o;        // [T, n_split, groups, 64, 512] bf16, unnormalised
    float *part_ml;          // [T, n_split, groups, 64, 2]
    DevBatch b;
    uint32_t *status;
    int H, k;
    int groups;              // head groups of 64 per token (1 or 2)
    float scale_log2;        // sm_scale * log2(e)
    int tiles_per_cta, n_split, n_tiles;
    int rope;                // 1: 576-wide rows with the rope tail; 0: 512-wide latent rows
    int async_copy;          // gather rows with cp.async (1) or TMA tile::gather4 (0)
};

struct Ctl {
    uint64_t q_full;
    uint64_t c_full[kBufs];
    uint64_t c_empty[kBufs];
    uint64_t s_full[kBufs];
    uint64_t p_full[kBufs];
    uint64_t o_full;
    uint32_t tmem_base;
    int32_t abort_flag;
    float red[4][kHeads];
    float m[kHeads];
    float alpha[kHeads];
    float2 ma[kHeads];       // (m, alpha) of the current tile, read together
    int32_t resc[2];         // any head of warp 0 / 1 rescaled in this tile
    float l[kHeads];
    float inv_l[kHeads];     // 1 / l (0 for an empty row)
    int32_t warp_alive[kSoftmaxWarps];
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Ctl &c, uint32_t *status,
                                         uint64_t limit_ns) {
    if (*(volatile int32_t *)&c.abort_flag) return false;
    if (mbar_wait(bar, parity, limit_ns)) return true;
    *(volatile int32_t *)&c.abort_flag = 1;
    flag(status, DSA_DEV_TIMEOUT);
    return false;
}

// Transposing butterfly reduction across each 16-lane half of a warp, whose
// lanes hold 16 values each (lanes 0..15: heads 0..15, lanes 16..31: heads
// 16..31 of the warp's 32): lane L ends up with the reduction over its half
// of head L.
template <bool kMax>
__device__ __forceinline__ float half_reduce_16(const float (&x)[16], int lane) {
    float a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) a[i] = x[i];
#pragma unroll
    for (int half = 8; half >= 1; half >>= 1) {
        const bool up = lane & half;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < half) {
                const float keep = up ? a[half + i] : a[i];
                const float send = up ? a[i] : a[half + i];
                const float o = __shfl_xor_sync(0xffffffffu, send, half);
                a[i] = kMax ? fmaxf(keep, o) : keep + o;
            }
        }
    }
    return a[0];
}

// One producer warp copies 16 rows of a tile (tile rows r0 .. r0 + 15) whose
// cache rows lanes 0..15 hold in my_row, CPR 16-byte chunks per row (72 with
// the rope tail, 64 without), into the nine-block SWIZZLE_128B layout the
// MMAs read.  Within each group of four rows, warp instruction i copies flat
// chunks 32 i .. 32 i + 31, so every warp instruction reads at most two rows'
// contiguous runs of bytes; the addresses are set up once per i and advance
// by a constant per group.
template <int CPR>
__device__ __forceinline__ void copy_rows16(uint32_t cb, const uint8_t *kv, int32_t my_row, int r0, int lane) {
    // Four rows at a time: their 4 * CPR chunks are PER per lane, and lane l's
    // i-th chunk sits at the same (row in the group, chunk) in every group.
    // r0 is a multiple of 8, so a row's swizzle phase is (4 g + rg) mod 8:
    // odd groups flip bit 2 of the chunk index, i.e. bit 6 of the address.
    constexpr int PER = 4 * CPR / 32;
    static_assert(4 * CPR % 32 == 0, "a group of four rows is a whole number of warp-wide copies");
#pragma unroll 1
    for (int i = 0; i < PER; ++i) {
        const int f = lane + 32 * i;
        const int rg = f / CPR, c = f - rg * CPR;
        const uint32_t d0 = cb + (uint32_t)(c >> 3) * kCBlockBytes + sw128_offset((uint32_t)(r0 + rg), (uint32_t)(c & 7));
        const uint8_t *src = kv + c * 16;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int32_t row = __shfl_sync(0xffffffffu, my_row, 4 * g + rg);
            cp_async16((d0 + (uint32_t)g * 512u) ^ ((uint32_t)(g & 1) << 6), src + (int64_t)row * (CPR * 16));
        }
    }
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_kernel(const AttnParams p, const __grid_constant__ CUtensorMap q_lat_map,
                       const __grid_constant__ CUtensorMap q_rope_map,
                       const __grid_constant__ CUtensorMap kv_map) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *q_s = base;
    uint8_t *c_s = base + kQBytes;                       // kBufs tile buffers
    Ctl &ctl = *reinterpret_cast<Ctl *>(c_s + kBufs * kCBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DevBatch &b = p.b;
    const int t = blockIdx.x / p.groups;
    const int hg = blockIdx.x - t * p.groups;            // head group: heads h0 .. h0 + nh - 1
    const int h0 = hg * kHeads, nh = min(kHeads, p.H - h0);
    const int split = blockIdx.y;
    if (t >= b.T) return;
    // this CTA's slice of the split partials
    const int64_t part_idx = ((int64_t)t * p.n_split + split) * p.groups + hg;
    tl_start(b.timeline, kTlAttn);
    const int pos = __ldg(b.q_pos + t);
    const int seq = seq_of_warp(b.cu_q, b.B, t, lane);
    const int64_t kv0 = seq_base(b, seq);
    const int tile_lo = split * p.tiles_per_cta;
    const int tile_hi = min(p.n_tiles, tile_lo + p.tiles_per_cta);
    int64_t own_row = -1;                                // the token's own row: fallback for skipped entries
    if (pos >= 0 && pos < b.max_kv && kv0 >= 0) own_row = cache_row(b, seq, kv0, pos);
    const bool pos_ok = own_row >= 0 && own_row < b.cache_rows;
    if (!pos_ok || tile_lo >= tile_hi) {
        if (!pos_ok && threadIdx.x == 0 && split == 0) flag(p.status, DSA_DEV_BAD_POSITION);
        // Empty contribution.
        if (p.n_split > 1) {
            for (int i = threadIdx.x; i < kHeads * D_L / 2; i += kThreads)
                reinterpret_cast<uint32_t *>(p.part_o + part_idx * kHeads * D_L)[i] = 0u;
            if (threadIdx.x < kHeads) {
                float *ml = p.part_ml + (part_idx * kHeads + threadIdx.x) * 2;
                ml[0] = -INFINITY;
                ml[1] = 0.f;
            }
        } else {
            for (int i = threadIdx.x; i < nh * D_L; i += kThreads) p.out[((int64_t)t * p.H + h0) * D_L + i] = 0.f;
            if (p.lse && threadIdx.x < nh) p.lse[(int64_t)t * p.H + h0 + threadIdx.x] = -INFINITY;
        }
        return;
    }
    const int n_my = tile_hi - tile_lo;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&ctl.q_full), 1);
        for (int i = 0; i < kBufs; ++i) {
            // a tile lands when its bytes arrive (TMA) or when every producer
            // has seen its own copies complete (cp.async)
            mbar_init(smem_u32(&ctl.c_full[i]), p.async_copy ? kProducers : 1);
            mbar_init(smem_u32(&ctl.c_empty[i]), 1);
            mbar_init(smem_u32(&ctl.s_full[i]), 1);
            mbar_init(smem_u32(&ctl.p_full[i]), kSoftmaxWarps);
        }
        mbar_init(smem_u32(&ctl.o_full), 1);
        ctl.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&ctl.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kMmaWarp + 1 && lane == 0) {
        tma_prefetch_desc(&kv_map);
        tma_prefetch_desc(&q_lat_map);
        tma_prefetch_desc(&q_rope_map);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;
    const int32_t *idx_row = p.idx + (int64_t)t * p.k;

    if (warp > kMmaWarp) {
        // ---------------- producers: queries once, then gathered row tiles.
        // A tile is 16 row quads x 9 column blocks = 144 gather4 requests
        // (8 blocks, 128 requests, without the rope tail); producer thread pl
        // sends requests pl and pl + 128.
        // Under the failure-path test hook nothing is copied, so that the
        // consumers' waits run out.
        const int pl = (int)threadIdx.x - 32 * (kMmaWarp + 1);
        const bool copy = !b.skip_copies;
        if (pl == 0 && copy) {
            // query rows of the head group; rows past the token's heads (the
            // next token's, or zero fill past the tensor) only feed padded
            // accumulator columns that are never stored
            const uint32_t qf = smem_u32(&ctl.q_full);
            mbar_arrive_expect_tx(qf, p.rope ? kQBytes : kQBytes - kQBlockBytes);
            const int32_t qrow = t * p.H + h0;
            for (int kb = 0; kb < 8; ++kb)
                tma_load_2d(smem_u32(q_s + kb * kQBlockBytes), &q_lat_map, qf, kb * 64, qrow);
            if (p.rope) tma_load_2d(smem_u32(q_s + 8 * kQBlockBytes), &q_rope_map, qf, 0, qrow);
        }
        // Cache row of entry e of the token's index row: the row itself when it
        // is a visible position, else (padding, or out of range: flagged) the
        // token's own row, whose scores the softmax masks.
        auto row_of = [&](int e, bool report) -> int32_t {
            const int32_t v = e < p.k ? __ldg(idx_row + e) : -1;
            bool ok = v >= 0 && v <= pos;
            int64_t row;
            if (!b.block_table) {
                row = kv0 + (ok ? v : pos);          // in range: the position check covers v <= pos
            } else {
                row = ok ? cache_row(b, seq, kv0, v) : own_row;
                if (row < 0 || row >= b.cache_rows) {
                    ok = false;
                    row = own_row;
                }
            }
            if (!ok && v != -1 && report) flag(p.status, DSA_DEV_BAD_INDEX);
            return (int32_t)row;
        };
        pdl_wait();                                  // the indices come from the preceding kernel
        if (p.async_copy) {
            // cp.async gather: warp pw copies tile rows 16 pw .. 16 pw + 15,
            // then waits for its own copies, fences them for the tensor core
            // and arrives; the tile is full when all 128 producers have.
            // Decode CTAs of more than two tiles also ask L2 for their rows
            // of the next tile as soon as the current tile's copies are out:
            // that tile's buffer frees only after the current one's value
            // product, and its gather then reads L2 instead of HBM (measured
            // on GB300, ragged decode: attention 31.0 -> 29.4 us).  Prefill
            // CTAs skip it -- neighbouring tokens already share rows through
            // L2, and the extra requests only slowed the gathers (long
            // prefill attention 10.48 -> 10.96 ms) -- and so do CTAs of two
            // tiles, whose second tile would compete with the first for HBM.
            const int pw = pl >> 5;
            const bool ahead = n_my > 2 && b.max_q == 1;
            const uint32_t row_bytes = p.rope ? kBlocks * 128u : (kBlocks - 1) * 128u;
            // (Without the look-ahead a tile's rows are looked up before its
            // buffer is free, where the index loads hide behind the wait:
            // looking them up between the copies and their completion cost
            // the prefill chunk 5% of its attention time.)
            int32_t next_row = (ahead && lane < 16) ? row_of(tile_lo * kRows + 16 * pw + lane, true) : 0;
            for (int it = 0; it < n_my; ++it) {
                const int buf = it & 1;
                const uint32_t use = (uint32_t)(it >> 1);
                const int32_t my_row = ahead ? next_row
                                             : (lane < 16 ? row_of((tile_lo + it) * kRows + 16 * pw + lane, true) : 0);
                if (!wait_bar(smem_u32(&ctl.c_empty[buf]), (use & 1u) ^ 1u, ctl, p.status, b.wait_ns)) break;
                if (!copy) continue;
                const uint32_t cb = smem_u32(c_s + buf * kCBytes);
                if (p.rope) copy_rows16<kBlocks * 8>(cb, p.kv, my_row, 16 * pw, lane);
                else copy_rows16<(kBlocks - 1) * 8>(cb, p.kv, my_row, 16 * pw, lane);
                cp_async_commit();
                if (ahead && it + 1 < n_my && lane < 16) {
                    next_row = row_of((tile_lo + it + 1) * kRows + 16 * pw + lane, true);
                    prefetch_l2_bulk(p.kv + (int64_t)next_row * row_bytes, row_bytes);
                }
                cp_async_wait_all();
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&ctl.c_full[buf]));
            }
        } else {
            // TMA gather: a tile is 16 row quads x 9 column blocks = 144
            // gather4 requests (8 blocks, 128 requests, without the rope
            // tail); producer thread pl sends requests pl and pl + 128.  Their
            // rows are looked up before the buffer is free, so the copies go
            // out as soon as it is.
            const int nb = p.rope ? kBlocks : kBlocks - 1;   // column blocks gathered per row
            const int n_req = (kRows / 4) * nb;                // gather4 requests per tile
            constexpr int kReq = ((kRows / 4) * kBlocks + kProducers - 1) / kProducers;
            for (int it = 0; it < n_my; ++it) {
                const int buf = it & 1;
                const uint32_t use = (uint32_t)(it >> 1);
                int32_t rr[kReq][4];
#pragma unroll
                for (int u = 0; u < kReq; ++u) {
                    const int q = pl + u * kProducers;
                    if (q >= n_req) break;
                    const int quad = p.rope ? q / kBlocks : q >> 3, kb = p.rope ? q % kBlocks : q & 7;
#pragma unroll
                    for (int j = 0; j < 4; ++j) rr[u][j] = row_of((tile_lo + it) * kRows + quad * 4 + j, kb == 0);
                }
                if (!wait_bar(smem_u32(&ctl.c_empty[buf]), (use & 1u) ^ 1u, ctl, p.status, b.wait_ns)) break;
                if (!copy) continue;
                const uint32_t full = smem_u32(&ctl.c_full[buf]);
                if (pl == 0) mbar_arrive_expect_tx(full, p.rope ? kCBytes : kCBytes - kCBlockBytes);
#pragma unroll
                for (int u = 0; u < kReq; ++u) {
                    const int q = pl + u * kProducers;
                    if (q >= n_req) break;
                    const int quad = p.rope ? q / kBlocks : q >> 3, kb = p.rope ? q % kBlocks : q & 7;
                    tma_gather4(smem_u32(c_s + buf * kCBytes + kb * kCBlockBytes + quad * 512), &kv_map, full,
                                kb * 64, rr[u][0], rr[u][1], rr[u][2], rr[u][3]);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer.  S^T(i) needs tile i gathered and the S
        // buffer it reuses read by softmax(i - 2); O^T(i) needs P^T(i).  The two
        // streams are issued in whatever order their inputs arrive, so that an
        // O^T product (which frees a tile buffer for the next gather) never
        // waits behind a gather.
        // Block (try_wait suspends the thread) until the queries and the first
        // tile have landed: an early-launched grid would otherwise spin through
        // the whole of the preceding kernels.
        if (lane == 0 && wait_bar(smem_u32(&ctl.q_full), 0, ctl, p.status, b.wait_ns) &&
            wait_bar(smem_u32(&ctl.c_full[0]), 0, ctl, p.status, b.wait_ns)) {
            const uint32_t id_s = idesc_f16(kRows, kHeads, true, false, false);
            const uint32_t id_o = idesc_f16(128, kHeads, true, true, true);
            const uint32_t qa = smem_u32(q_s), ca = smem_u32(c_s);
            // Descriptors differ only in their start address (bits 0..13, in
            // 16-byte units, no carry: shared addresses are below 256 KB), so
            // each product adds a constant offset to a base descriptor.
            const uint64_t s_a0 = sdesc_sw128(ca, 16, 1024), s_b0 = sdesc_sw128(qa, 16, 1024);
            const uint64_t o_a0 = sdesc_sw128(ca, kCBlockBytes, 1024), o_b0 = sdesc_sw128(ca + 8 * kCBlockBytes,
                                                                                          kCBlockBytes, 1024);
            const int s_blocks = p.rope ? kBlocks : kBlocks - 1;
            int s_next = 0, o_next = 0;
            uint64_t t_last = global_ns();
            while (o_next < n_my) {
                bool progress = false;
                if (s_next < n_my && s_next <= o_next + 1 &&
                    mbar_test(smem_u32(&ctl.c_full[s_next & 1]), (uint32_t)(s_next >> 1) & 1u)) {
                    const int buf = s_next & 1;
                    tc_fence_after();
                    uint64_t ad = s_a0 + (uint64_t)((buf * kCBytes) >> 4), bd = s_b0;
                    const uint32_t d_s = tmem + kColS + buf * kHeads;
#pragma unroll 1
                    for (int kb = 0; kb < s_blocks; ++kb) {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            umma_f16(d_s, ad + (uint64_t)(ks * 2), bd + (uint64_t)(ks * 2), id_s, (kb | ks) != 0);
                        ad += (uint64_t)(kCBlockBytes >> 4);
                        bd += (uint64_t)(kQBlockBytes >> 4);
                    }
                    umma_commit(smem_u32(&ctl.s_full[buf]));
                    ++s_next;
                    progress = true;
                }
                if (o_next < s_next &&
                    mbar_test(smem_u32(&ctl.p_full[o_next & 1]), (uint32_t)(o_next >> 1) & 1u)) {
                    const int buf = o_next & 1;
                    tc_fence_after();
                    const uint64_t boff = (uint64_t)((buf * kCBytes) >> 4);
                    const uint32_t acc0 = o_next > 0 ? 1u : 0u;
                    uint64_t ad = o_a0 + boff;
                    const uint64_t bd = o_b0 + boff;
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
#pragma unroll
                        for (int ks = 0; ks < kRows / 16; ++ks)
                            umma_f16(tmem + kColO + c * kHeads, ad + (uint64_t)(ks * (2048 >> 4)),
                                     bd + (uint64_t)(ks * (2048 >> 4)), id_o, (acc0 | (uint32_t)ks) ? 1u : 0u);
                        ad += (uint64_t)((2 * kCBlockBytes) >> 4);
                    }
                    umma_commit(smem_u32(&ctl.c_empty[buf]));
                    umma_commit(smem_u32(&ctl.o_full));
                    ++o_next;
                    progress = true;
                }
                if (progress) {
                    t_last = global_ns();
                } else if (*(volatile int32_t *)&ctl.abort_flag) {
                    break;
                } else if (global_ns() - t_last > b.wait_ns) {
                    *(volatile int32_t *)&ctl.abort_flag = 1;
                    flag(p.status, DSA_DEV_TIMEOUT);
                    break;
                }
            }
        }
    } else {
        // ---------------- softmax and epilogue (warps 0..7)
        const int tx = (int)threadIdx.x;                   // 0..255
        const int quarter = warp & 3;                      // TMEM lanes 32*quarter .. 32*quarter+31
        const int part = warp >> 2;                        // heads 32*part .. 32*part+31
        // An M=64 accumulator keeps rows in lanes 0..15 of each quarter; the
        // two halves of the warp read the same 16 rows, 16 heads each.
        const int hb = 32 * part + 16 * (lane >> 4);       // this thread's first head
        const int hl = 32 * part + lane;                   // the head this lane reduces
        const int r = quarter * 16 + (lane & 15);          // row within the tile
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        if (tx < kHeads) ctl.m[tx] = -INFINITY;
        pdl_wait();
        bool alive = true;
        named_barrier(1, kSoftmaxThreads);
        float lpart[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) lpart[h] = 0.f;
        // Every softmax thread runs the same sequence of named barriers whatever
        // happens; `alive` (warp-uniform) only gates tensor-memory and shared
        // memory work after a bounded wait gave up.
        for (int it = 0; it < n_my; ++it) {
            const int buf = it & 1;
            const int e = (tile_lo + it) * kRows + r;
            const int32_t v = e < p.k ? __ldg(idx_row + e) : -1;
            const bool valid = v >= 0 && v <= pos;
            if (alive) alive = wait_bar(smem_u32(&ctl.s_full[buf]), (uint32_t)(it >> 1) & 1u, ctl, p.status, b.wait_ns);
            alive = __all_sync(0xffffffffu, alive);
            float x[16];
            if (alive) {
                tc_fence_after();
                uint32_t u[16];
                tmem_ld16x2_16(tmem + lane_addr + kColS + buf * kHeads + 32 * part, u);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < 16; ++h) x[h] = valid ? __uint_as_float(u[h]) * p.scale_log2 : -INFINITY;
            } else {
#pragma unroll
                for (int h = 0; h < 16; ++h) x[h] = -INFINITY;
            }
            // per-head tile maximum across the 64 rows: lane L gets head 32 part + L
            ctl.red[quarter][hl] = half_reduce_16<true>(x, lane);
            named_barrier(1, kSoftmaxThreads);
            if (tx < kHeads) {
                const int h = tx;
                const float tmax = fmaxf(fmaxf(ctl.red[0][h], ctl.red[1][h]), fmaxf(ctl.red[2][h], ctl.red[3][h]));
                const float mo = ctl.m[h];
                float mn = mo, al = 1.f;
                if (tmax > mo + kRescaleLog2 || (mo == -INFINITY && tmax != -INFINITY)) {
                    mn = tmax;
                    al = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
                }
                ctl.m[h] = mn;
                ctl.alpha[h] = al;
                ctl.ma[h] = make_float2(mn, al);
                const bool any = __any_sync(0xffffffffu, al != 1.f);
                if (lane == 0) ctl.resc[warp] = any ? 1 : 0;
            }
            named_barrier(1, kSoftmaxThreads);
            const bool rescale = ctl.resc[0] | ctl.resc[1];   // identical in every thread
            uint32_t pk[8];
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const int h = hb + j;
                const float2 a0 = ctl.ma[h], a1 = ctl.ma[h + 1];
                const float p0 = (a0.x == -INFINITY) ? 0.f : exp2f(x[j] - a0.x);
                const float p1 = (a1.x == -INFINITY) ? 0.f : exp2f(x[j + 1] - a1.x);
                lpart[j] = lpart[j] * a0.y + p0;
                lpart[j + 1] = lpart[j + 1] * a1.y + p1;
                const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                pk[j / 2] = *reinterpret_cast<const uint32_t *>(&pb);
            }
            if (alive) {
                // P^T row r into the (now dead) rope block, MN-major SW128: 64
                // heads = 128 bytes, this thread's 16 heads = chunks hb/8, hb/8 + 1.
                uint8_t *prow = c_s + buf * kCBytes + 8 * kCBlockBytes;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    uint4 q4;
                    q4.x = pk[4 * j]; q4.y = pk[4 * j + 1]; q4.z = pk[4 * j + 2]; q4.w = pk[4 * j + 3];
                    *reinterpret_cast<uint4 *>(prow + sw128_offset((uint32_t)r, (uint32_t)(hb / 8 + j))) = q4;
                }
            }
            if (rescale && it > 0) {
                // Heads whose maximum moved: rescale their O^T columns once the
                // previous tile's PV product has landed.  O^T is an M=128
                // accumulator: every lane of the warp owns one output dim; the
                // two warps of a quarter take 32 heads each.
                if (alive) alive = wait_bar(smem_u32(&ctl.o_full), (uint32_t)(it - 1) & 1u, ctl, p.status, b.wait_ns);
                alive = __all_sync(0xffffffffu, alive);
                if (alive) {
                    tc_fence_after();
#pragma unroll 1
                    for (int cq = 0; cq < 8; ++cq) {             // 4 dim blocks x 2 groups of 16 heads
                        uint32_t u[16];
                        const int hq = part * 32 + (cq & 1) * 16;
                        const uint32_t addr = tmem + lane_addr + kColO + (cq >> 1) * kHeads + hq;
                        tmem_ld16(addr, u);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            u[j] = __float_as_uint(__uint_as_float(u[j]) * ctl.alpha[hq + j]);
                        tmem_st16(addr, u);
                    }
                    tmem_wait_st();
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl.p_full[buf]));
        }
        // ---- final: O^T of the last tile, row sums, outputs
        if (alive) alive = wait_bar(smem_u32(&ctl.o_full), (uint32_t)(n_my - 1) & 1u, ctl, p.status, b.wait_ns);
        alive = __all_sync(0xffffffffu, alive);
        ctl.red[quarter][hl] = half_reduce_16<false>(lpart, lane);
        named_barrier(1, kSoftmaxThreads);
        if (tx < kHeads) {
            const float l = ctl.red[0][tx] + ctl.red[1][tx] + ctl.red[2][tx] + ctl.red[3][tx];
            ctl.l[tx] = l;
            ctl.inv_l[tx] = l > 0.f ? 1.f / l : 0.f;
        }
        if (lane == 0) ctl.warp_alive[warp] = alive ? 1 : 0;
        named_barrier(1, kSoftmaxThreads);
        bool all_alive = true;
#pragma unroll
        for (int w = 0; w < kSoftmaxWarps; ++w) all_alive = all_alive && ctl.warp_alive[w];
        if (all_alive) {
            // This CTA's [head][dim] block straight from TMEM: thread (quarter,
            // lane) holds output dim c*128 + quarter*32 + lane of every head,
            // so each warp store writes one head's contiguous run of dims; the
            // two warps of a quarter store 32 heads each.  The output (one
            // split) is normalised and float32; a split's partial is
            // unnormalised bf16 (measured on GB300, batched decode: the
            // per-element 1 / l multiply there cost 3.6 us per CTA, pairing
            // lanes for 4-byte stores 0.9 us).
            tc_fence_after();
            const int H = p.H;
            const int rd = quarter * 32 + lane;
            if (p.n_split == 1) {
                // 16 heads at a time: their 1 / l in registers, then the 16
                // accumulator columns of each 128-dim block
                float *dst = p.out + ((int64_t)t * H + h0) * D_L;
#pragma unroll 1
                for (int q = 2 * part; q < 2 * part + 2; ++q) {
                    float inv[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) inv[jj] = ctl.inv_l[q * 16 + jj];
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t u[16];
                        tmem_ld16(tmem + lane_addr + kColO + c * kHeads + q * 16, u);
                        tmem_wait_ld();
                        const int d = c * 128 + rd;
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int h = q * 16 + jj;
                            if (h < nh) dst[h * D_L + d] = __uint_as_float(u[jj]) * inv[jj];
                        }
                    }
                }
            } else {
                uint16_t *dst = p.part_o + part_idx * kHeads * D_L;
                for (int c = 0; c < 4; ++c) {
                    const int d = c * 128 + rd;
                    uint32_t u[32];
                    tmem_ld32(tmem + lane_addr + kColO + c * kHeads + part * 32, u);
                    tmem_wait_ld();
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        dst[(part * 32 + jj) * D_L + d] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(u[jj])));
                }
            }
            if (tx < kHeads) {
                const int h = tx;
                const float l = ctl.l[h], m = ctl.m[h];
                if (p.n_split > 1) {
                    float *ml = p.part_ml + (part_idx * kHeads + h) * 2;
                    ml[0] = l > 0.f ? m : -INFINITY;
                    ml[1] = l;
                } else if (p.lse && h < nh) {
                    p.lse[(int64_t)t * H + h0 + h] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
                }
            }
        }
    }

    tc_fence_before();
    __syncwarp();                  // lanes of the MMA warp arrive from different paths
    __syncthreads();
    // Dependents launch only now: CTAs of the next grid waiting on this one
    // would share the SMs and slow it down.
    pdl_trigger();
    tl_end(b.timeline, kTlAttn);
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Merge split partials: o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
// NF partial rows are loaded at a time.  With NF = 4 (up to four splits)
// the kernel fits in 32 registers, so 16 CTAs share an SM and a grid of
// thousands of (token, head) CTAs runs in one wave; NF = 16 keeps five CTAs
// per SM.
template <int NF>
__global__ void __launch_bounds__(128, NF <= 4 ? 16 : 5) attn_combine_kernel(const uint16_t *__restrict__ part_o,
                                                                            const float *__restrict__ part_ml,
                                                                            int n_split, int H, int groups,
                                                                            float *out, float *lse,
                                                                            unsigned long long *timeline) {
    __shared__ float wgt[128];
    __shared__ float ml[2][128];
    const int t = blockIdx.x, h = blockIdx.y;
    // partial row of (split s, head h): ((t * n_split + s) * groups + h / 64) * 64 + h % 64
    const int64_t hoff = (int64_t)(h / kHeads) * kHeads + h % kHeads;
    const int64_t stride = (int64_t)groups * kHeads;     // partial rows per split
    const int64_t base = (int64_t)t * n_split * stride + hoff;
    tl_start(timeline, kTlCombine);
    pdl_wait();
    for (int s = threadIdx.x; s < n_split; s += 128) {      // all split statistics at once
        ml[0][s] = __ldg(part_ml + (base + s * stride) * 2);
        ml[1][s] = __ldg(part_ml + (base + s * stride) * 2 + 1);
    }
    __syncthreads();
    float M = -INFINITY;
    for (int s = 0; s < n_split; ++s) M = fmaxf(M, ml[0][s]);
    float L = 0.f;
    for (int s = 0; s < n_split; ++s) {
        const float w = ml[0][s] == -INFINITY ? 0.f : exp2f(ml[0][s] - M);
        L += w * ml[1][s];
        if (threadIdx.x == 0) wgt[s] = w;
    }
    __syncthreads();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < n_split; s0 += NF) {              // NF loads in flight
        uint2 o[NF];
#pragma unroll
        for (int u = 0; u < NF; ++u)
            if (s0 + u < n_split)
                o[u] = __ldg(reinterpret_cast<const uint2 *>(part_o + (base + (s0 + u) * stride) * D_L) + threadIdx.x);
#pragma unroll
        for (int u = 0; u < NF; ++u) {
            if (s0 + u < n_split) {
                const float w = wgt[s0 + u];
                const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&o[u].x));
                const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&o[u].y));
                acc.x += w * a.x; acc.y += w * a.y; acc.z += w * c.x; acc.w += w * c.y;
            }
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
    reinterpret_cast<float4 *>(out + ((int64_t)t * H + h) * D_L)[threadIdx.x] = acc;
    if (lse && threadIdx.x == 0)
        lse[(int64_t)t * H + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
    __syncthreads();
    tl_end(timeline, kTlCombine);
}

size_t sparse_attn_smem_bytes() { return 1024 + kQBytes + kBufs * kCBytes + sizeof(Ctl); }

int attn_tile_rows() { return kRows; }

cudaError_t launch_sparse_attn(const AttnLaunch &a, const CUtensorMap &q_lat_map,
                               const CUtensorMap &q_rope_map, const CUtensorMap &kv_map,
                               const DevBatch &b, uint32_t *status, cudaStream_t stream, bool pdl) {
    AttnParams p{};
    p.kv = static_cast<const uint8_t *>(a.kv);
    p.idx = a.idx;
    p.out = a.out;
    p.lse = a.lse;
    p.part_o = static_cast<uint16_t *>(a.part_o);
    p.part_ml = a.part_ml;
    p.b = b;
    p.status = status;
    p.H = a.H;
    p.k = a.k;
    p.groups = (a.H + kHeads - 1) / kHeads;
    p.scale_log2 = a.sm_scale * 1.4426950408889634f;
    p.tiles_per_cta = a.tiles_per_cta;
    p.n_split = a.n_split;
    p.n_tiles = (a.k + kRows - 1) / kRows;
    p.rope = a.rope;
    // Gather path: cp.async reads each row through L2 at the load/store
    // units' rate; TMA tile::gather4 issues one 512-byte request at a time.
    p.async_copy = 1;
    const size_t smem = sparse_attn_smem_bytes();
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(sparse_attn_kernel), 1, smem);
    if (e != cudaSuccess) return e;
    if (a.n_split > 65535 || p.groups < 1 || p.groups > 2 || (int64_t)b.T * p.groups > 0x7fffffff)
        return cudaErrorInvalidConfiguration;
    dim3 grid((unsigned)(b.T * p.groups), (unsigned)a.n_split);
    return launch_k(sparse_attn_kernel, grid, dim3(kThreads), smem, stream, pdl, p, q_lat_map, q_rope_map, kv_map);
}

cudaError_t launch_attn_combine(const AttnLaunch &a, const DevBatch &b, cudaStream_t stream, bool pdl) {
    if (a.n_split <= 1) return cudaSuccess;
    if (a.n_split > 128) return cudaErrorInvalidConfiguration;
    const int groups = (a.H + kHeads - 1) / kHeads;
    dim3 grid((unsigned)b.T, (unsigned)a.H);
    if (a.n_split <= 4)
        return launch_k(attn_combine_kernel<4>, grid, dim3(128), 0, stream, pdl, (const uint16_t *)a.part_o,
                        (const float *)a.part_ml, a.n_split, a.H, groups, a.out, a.lse, b.timeline);
    return launch_k(attn_combine_kernel<16>, grid, dim3(128), 0, stream, pdl, (const uint16_t *)a.part_o,
                    (const float *)a.part_ml, a.n_split, a.H, groups, a.out, a.lse, b.timeline);
}

}  // namespace dsa
