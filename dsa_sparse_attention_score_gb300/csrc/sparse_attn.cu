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
// One CTA per (token, split) handles a run of 128-row tiles of the token's
// selected positions, with the token's 64 heads on the N side of every MMA:
//     S^T[row, head]  = C[row, 0:576] . Q[head, 0:576]^T        (M=128, N=64, K=576)
//     O^T[dim, head] += C[row, dim]^T . P^T[row, head]           (M=4x128, N=64, K=128)
// The gathered tile C sits in shared memory as nine 64-column SWIZZLE_128B
// blocks (TMA tile::gather4, four rows per instruction).  The same bytes serve
// as the K-major A operand of S^T and, for the latent blocks, as the MN-major
// A operand of O^T, so V is never copied.  The rope block is dead once S^T is
// computed and holds P^T (bf16) for the second MMA.  Softmax runs in four
// warps, one key row per thread, with a per-head running maximum that is
// only raised when a tile exceeds it by more than 2^8 (lazy rescale of the
// TMEM accumulator); the final normalisation makes the result exact either
// way.  With several splits per token, unnormalised partials (O, m, l) go to
// the workspace and a combine kernel merges them.
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {

namespace {

constexpr int kHeads = 64;                    // heads per CTA (padded)
constexpr int kRows = 128;                    // gathered rows per tile
constexpr int kBlocks = 9;                    // 576 / 64 columns
constexpr int kQBlockBytes = kHeads * 128;    // 8 KB
constexpr int kCBlockBytes = kRows * 128;     // 16 KB
constexpr int kQBytes = kBlocks * kQBlockBytes;
constexpr int kCBytes = kBlocks * kCBlockBytes;
constexpr int kThreads = 192;                 // producer, MMA, 4 softmax warps
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t kTmemCols = 512;           // S: 64 cols, O^T: 4 x 64 cols
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 64;

struct AttnParams {
    const int32_t *idx;
    float *out;
    float *lse;
    float *part_o;
    float *part_ml;
    DevBatch b;
    uint32_t *status;
    int H, k;
    float scale_log2;        // sm_scale * log2(e)
    int tiles_per_cta, n_split, n_tiles;
    int clustered;           // the n_split CTAs of a token form one cluster and reduce in DSMEM
};

struct Ctl {
    uint64_t q_full;
    uint64_t c_full[kBlocks];
    uint64_t c_empty[kBlocks];
    uint64_t s_full;
    uint64_t p_full;
    uint64_t o_full;
    uint32_t tmem_base;
    int32_t abort_flag;
    float red[4][kHeads];
    float m[kHeads];
    float alpha[kHeads];
    float l[kHeads];
    float gm[kHeads];        // cluster-wide maximum per head
    float gl[kHeads];        // cluster-wide softmax denominator per head
    float sc[kHeads];        // this CTA's scale 2^(m - gm)
    int32_t warp_alive[4];
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Ctl &c, uint32_t *status) {
    if (*(volatile int32_t *)&c.abort_flag) return false;
    if (mbar_wait(bar, parity)) return true;
    *(volatile int32_t *)&c.abort_flag = 1;
    flag(status, DSA_DEV_TIMEOUT);
    return false;
}

// Transposing butterfly reduction of 64 per-lane values across a warp:
// lane L ends up with the reduction of heads 2L and 2L+1 in v[0], v[1].
template <bool kMax>
__device__ __forceinline__ void warp_reduce_64(const float (&x)[64], int lane, float &r0, float &r1) {
    float a[32];
    {
        const bool up = lane & 16;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float keep = up ? x[32 + i] : x[i];
            const float send = up ? x[i] : x[32 + i];
            const float o = __shfl_xor_sync(0xffffffffu, send, 16);
            a[i] = kMax ? fmaxf(keep, o) : keep + o;
        }
    }
#pragma unroll
    for (int half = 16, bit = 8; half >= 2; half >>= 1, bit >>= 1) {
        const bool up = lane & bit;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i < half) {
                const float keep = up ? a[half + i] : a[i];
                const float send = up ? a[i] : a[half + i];
                const float o = __shfl_xor_sync(0xffffffffu, send, bit);
                a[i] = kMax ? fmaxf(keep, o) : keep + o;
            }
        }
    }
    r0 = a[0];
    r1 = a[1];
}

// One tile needs 288 gather4 requests (32 row quads x 9 column blocks).
// Lane `gl` of the `kIssuers` issuing lanes sends requests gl, gl + kIssuers,
// ... after the block it writes has been released by the previous tile.
constexpr int kIssueWarps = 5;                 // producer + the four softmax warps
constexpr int kIssuers = 32 * kIssueWarps;

__device__ __forceinline__ bool issue_tile_gathers(int gl, int tile, const int32_t *idx_row, int k, int pos,
                                                   int64_t kv0, uint32_t parity, uint8_t *c_s, Ctl &ctl,
                                                   const CUtensorMap *kv_map, uint32_t *status) {
    for (int q = gl; q < 32 * kBlocks; q += kIssuers) {
        const int kb = q >> 5, quad = q & 31;
        if (!wait_bar(smem_u32(&ctl.c_empty[kb]), parity, ctl, status)) return false;
        int32_t rr[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = tile * kRows + quad * 4 + j;
            const int32_t v = e < k ? __ldg(idx_row + e) : -1;
            const bool ok = v >= 0 && v <= pos;
            if (!ok && v != -1 && kb == 0) flag(status, DSA_DEV_BAD_INDEX);
            rr[j] = (int32_t)(kv0 + (ok ? v : 0));
        }
        tma_gather4(smem_u32(c_s + kb * kCBlockBytes + quad * 512), kv_map, smem_u32(&ctl.c_full[kb]), kb * 64,
                    rr[0], rr[1], rr[2], rr[3]);
    }
    return true;
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
    uint8_t *c_s = base + kQBytes;
    Ctl &ctl = *reinterpret_cast<Ctl *>(c_s + kCBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const DevBatch &b = p.b;
    const int t = blockIdx.x;
    const int split = blockIdx.y;
    if (t >= b.T) return;
    tl_start(b.timeline, kTlAttn);
    const int pos = __ldg(b.q_pos + t);
    const int seq = seq_of_warp(b.cu_q, b.B, t, lane);
    const int64_t kv0 = __ldg(b.kv_off + seq);
    const int tile_lo = split * p.tiles_per_cta;
    const int tile_hi = min(p.n_tiles, tile_lo + p.tiles_per_cta);
    const bool pos_ok = pos >= 0 && pos < b.max_kv && kv0 >= 0 && kv0 + pos < b.cache_rows;
    if (!pos_ok || tile_lo >= tile_hi) {
        if (!pos_ok && threadIdx.x == 0 && split == 0) flag(p.status, DSA_DEV_BAD_POSITION);
        // Empty contribution.
        if (p.n_split > 1) {
            for (int i = threadIdx.x; i < kHeads * D_L; i += kThreads)
                p.part_o[((int64_t)t * p.n_split + split) * kHeads * D_L + i] = 0.f;
            if (threadIdx.x < kHeads) {
                float *ml = p.part_ml + (((int64_t)t * p.n_split + split) * kHeads + threadIdx.x) * 2;
                ml[0] = -INFINITY;
                ml[1] = 0.f;
            }
        } else {
            for (int i = threadIdx.x; i < p.H * D_L; i += kThreads) p.out[(int64_t)t * p.H * D_L + i] = 0.f;
            if (p.lse && threadIdx.x < p.H) p.lse[(int64_t)t * p.H + threadIdx.x] = -INFINITY;
        }
        return;
    }
    const int n_my = tile_hi - tile_lo;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&ctl.q_full), 1);
        for (int i = 0; i < kBlocks; ++i) {
            mbar_init(smem_u32(&ctl.c_full[i]), 1);
            mbar_init(smem_u32(&ctl.c_empty[i]), 1);
        }
        mbar_init(smem_u32(&ctl.s_full), 1);
        mbar_init(smem_u32(&ctl.p_full), 4);
        mbar_init(smem_u32(&ctl.o_full), 1);
        ctl.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&kv_map);
        tma_prefetch_desc(&q_lat_map);
        tma_prefetch_desc(&q_rope_map);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;
    const int32_t *idx_row = p.idx + (int64_t)t * p.k;

    if (warp == 0) {
        // ---------------- producer: queries once, then gathered row tiles
        if (lane == 0) {
            const uint32_t qf = smem_u32(&ctl.q_full);
            mbar_arrive_expect_tx(qf, kQBytes);
            const int32_t qrow = t * p.H;
            for (int kb = 0; kb < 8; ++kb)
                tma_load_2d(smem_u32(q_s + kb * kQBlockBytes), &q_lat_map, qf, kb * 64, qrow);
            tma_load_2d(smem_u32(q_s + 8 * kQBlockBytes), &q_rope_map, qf, 0, qrow);
        }
        pdl_wait();                                  // the indices come from the preceding kernel
        for (int it = 0; it < n_my; ++it) {
            const uint32_t par = ((uint32_t)it & 1u) ^ 1u;
            if (lane == 0) {
                bool ok = true;
                for (int kb = 0; kb < kBlocks && ok; ++kb) {
                    ok = wait_bar(smem_u32(&ctl.c_empty[kb]), par, ctl, p.status);
                    if (ok) mbar_arrive_expect_tx(smem_u32(&ctl.c_full[kb]), kCBlockBytes);
                }
                if (!ok) break;
            }
            __syncwarp();
            if (!issue_tile_gathers(lane, tile_lo + it, idx_row, p.k, pos, kv0, par, c_s, ctl, &kv_map, p.status))
                break;
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0 && wait_bar(smem_u32(&ctl.q_full), 0, ctl, p.status)) {
            const uint32_t id_s = idesc_f16(128, kHeads, true, false, false);
            const uint32_t id_o = idesc_f16(128, kHeads, true, true, true);
            const uint32_t qa = smem_u32(q_s), ca = smem_u32(c_s);
            for (int it = 0; it < n_my; ++it) {
                const uint32_t par = (uint32_t)it & 1u;
                bool ok = true;
                for (int kb = 0; kb < kBlocks && ok; ++kb) {
                    if (!wait_bar(smem_u32(&ctl.c_full[kb]), par, ctl, p.status)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t ad = sdesc_sw128(ca + kb * kCBlockBytes + ks * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(qa + kb * kQBlockBytes + ks * 32, 16, 1024);
                        umma_f16(tmem + kColS, ad, bd, id_s, (kb | ks) != 0);
                    }
                }
                if (!ok) break;
                umma_commit(smem_u32(&ctl.s_full));
                if (!wait_bar(smem_u32(&ctl.p_full), par, ctl, p.status)) break;
                tc_fence_after();
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t ad =
                            sdesc_sw128(ca + (2 * c) * kCBlockBytes + ks * 2048, kCBlockBytes, 1024);
                        const uint64_t bd =
                            sdesc_sw128(ca + 8 * kCBlockBytes + ks * 2048, kCBlockBytes, 1024);
                        umma_f16(tmem + kColO + c * kHeads, ad, bd, id_o, (it > 0 || ks > 0) ? 1u : 0u);
                    }
                    umma_commit(smem_u32(&ctl.c_empty[2 * c]));
                    umma_commit(smem_u32(&ctl.c_empty[2 * c + 1]));
                }
                umma_commit(smem_u32(&ctl.c_empty[8]));
                umma_commit(smem_u32(&ctl.o_full));
            }
        }
    } else {
        // ---------------- softmax and epilogue (warps 2..5)
        const int tx = (int)threadIdx.x - 64;              // 0..127
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;                 // row within the tile
        const int sw = warp - 2;                           // 0..3
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        if (tx < kHeads) ctl.m[tx] = -INFINITY;
        pdl_wait();
        const int gl = 32 + tx;                            // issuing lane id (producer warp owns 0..31)
        bool alive = issue_tile_gathers(gl, tile_lo, idx_row, p.k, pos, kv0, 1u, c_s, ctl, &kv_map, p.status);
        alive = __all_sync(0xffffffffu, alive);
        named_barrier(1, 128);
        float lpart[kHeads];
#pragma unroll
        for (int h = 0; h < kHeads; ++h) lpart[h] = 0.f;
        // Every softmax thread runs the same sequence of named barriers whatever
        // happens; `alive` (warp-uniform) only gates tensor-memory and shared
        // memory work after a bounded wait gave up.
        for (int it = 0; it < n_my; ++it) {
            const uint32_t par = (uint32_t)it & 1u;
            const int e = (tile_lo + it) * kRows + r;
            const int32_t v = e < p.k ? __ldg(idx_row + e) : -1;
            const bool valid = v >= 0 && v <= pos;
            if (alive) alive = wait_bar(smem_u32(&ctl.s_full), par, ctl, p.status);
            alive = __all_sync(0xffffffffu, alive);
            float x[kHeads];
            if (alive) {
                tc_fence_after();
                uint32_t u0[32], u1[32];
                tmem_ld32(tmem + lane_addr + kColS, u0);
                tmem_ld32(tmem + lane_addr + kColS + 32, u1);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < 32; ++h) {
                    x[h] = valid ? __uint_as_float(u0[h]) * p.scale_log2 : -INFINITY;
                    x[32 + h] = valid ? __uint_as_float(u1[h]) * p.scale_log2 : -INFINITY;
                }
            } else {
#pragma unroll
                for (int h = 0; h < kHeads; ++h) x[h] = -INFINITY;
            }
            // per-head tile maximum across the 128 rows
            float m0, m1;
            warp_reduce_64<true>(x, lane, m0, m1);
            ctl.red[sw][2 * lane] = m0;
            ctl.red[sw][2 * lane + 1] = m1;
            named_barrier(1, 128);
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
            }
            named_barrier(1, 128);
            bool rescale = false;      // identical in every thread: all read the same alphas
            uint32_t pk[32];
#pragma unroll
            for (int h = 0; h < kHeads; h += 2) {
                const float mh0 = ctl.m[h], mh1 = ctl.m[h + 1];
                const float a0 = ctl.alpha[h], a1 = ctl.alpha[h + 1];
                rescale |= (a0 != 1.f) || (a1 != 1.f);
                const float p0 = (mh0 == -INFINITY) ? 0.f : exp2f(x[h] - mh0);
                const float p1 = (mh1 == -INFINITY) ? 0.f : exp2f(x[h + 1] - mh1);
                lpart[h] = lpart[h] * a0 + p0;
                lpart[h + 1] = lpart[h + 1] * a1 + p1;
                const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                pk[h / 2] = *reinterpret_cast<const uint32_t *>(&pb);
            }
            if (alive) {
                // P^T row r into the (now dead) rope block, MN-major SW128: 64 heads = 128 bytes.
                uint8_t *prow = c_s + 8 * kCBlockBytes;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint4 q4;
                    q4.x = pk[4 * j]; q4.y = pk[4 * j + 1]; q4.z = pk[4 * j + 2]; q4.w = pk[4 * j + 3];
                    *reinterpret_cast<uint4 *>(prow + sw128_offset((uint32_t)r, (uint32_t)j)) = q4;
                }
            }
            if (rescale && it > 0) {
                // Heads whose maximum moved: rescale their O^T columns once the
                // previous tile's PV product has landed.
                if (alive) alive = wait_bar(smem_u32(&ctl.o_full), par ^ 1u, ctl, p.status);
                alive = __all_sync(0xffffffffu, alive);
                if (alive) {
                    tc_fence_after();
                    for (int c = 0; c < 4; ++c) {
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint32_t u[32];
                            const uint32_t addr = tmem + lane_addr + kColO + c * kHeads + half * 32;
                            tmem_ld32(addr, u);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                u[j] = __float_as_uint(__uint_as_float(u[j]) * ctl.alpha[half * 32 + j]);
                            tmem_st32(addr, u);
                        }
                    }
                    tmem_wait_st();
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl.p_full));
            if (it + 1 < n_my && alive) {
                // this warp's share of the next tile's gathers, as its blocks free up
                alive = issue_tile_gathers(gl, tile_lo + it + 1, idx_row, p.k, pos, kv0, par, c_s,
                                           ctl, &kv_map, p.status);
            }
            alive = __all_sync(0xffffffffu, alive);
        }
        // ---- final: O^T of the last tile, row sums, outputs
        const uint32_t last_par = (uint32_t)(n_my - 1) & 1u;
        if (alive) alive = wait_bar(smem_u32(&ctl.o_full), last_par, ctl, p.status);
        alive = __all_sync(0xffffffffu, alive);
        float l0, l1;
        warp_reduce_64<false>(lpart, lane, l0, l1);
        ctl.red[sw][2 * lane] = l0;
        ctl.red[sw][2 * lane + 1] = l1;
        named_barrier(1, 128);
        if (tx < kHeads) ctl.l[tx] = ctl.red[0][tx] + ctl.red[1][tx] + ctl.red[2][tx] + ctl.red[3][tx];
        if (lane == 0) ctl.warp_alive[sw] = alive ? 1 : 0;
        named_barrier(1, 128);
        if (alive && !p.clustered) {
            // Stage this CTA's [head][dim] block in the dead gathered tile and
            // write it with one bulk copy: unnormalised partials when the token
            // is split, the normalised output otherwise.
            tc_fence_after();
            const int H = p.H;
            const int rows = p.n_split > 1 ? kHeads : H;
            float *stage = reinterpret_cast<float *>(c_s);
            for (int c = 0; c < 4; ++c) {
                const int d = c * 128 + r;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t u[32];
                    tmem_ld32(tmem + lane_addr + kColO + c * kHeads + half * 32, u);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int h = half * 32 + j;
                        float o = __uint_as_float(u[j]);
                        if (p.n_split == 1) {
                            const float l = ctl.l[h];
                            o = l > 0.f ? o / l : 0.f;
                        }
                        if (h < rows) stage[h * D_L + d] = o;
                    }
                }
            }
            fence_proxy_async_smem();
        }
        named_barrier(1, 128);                       // every warp, whatever its state
        const bool all_alive = ctl.warp_alive[0] && ctl.warp_alive[1] && ctl.warp_alive[2] && ctl.warp_alive[3];
        if (all_alive && !p.clustered) {
            const int H = p.H;
            const int rows = p.n_split > 1 ? kHeads : H;
            if (tx == 0) {
                float *dst = p.n_split > 1 ? p.part_o + ((int64_t)t * p.n_split + split) * kHeads * D_L
                                           : p.out + (int64_t)t * H * D_L;
                const uint32_t bytes = (uint32_t)(rows * D_L * 4);
                for (uint32_t off = 0; off < bytes; off += 32768)
                    bulk_s2g(reinterpret_cast<uint8_t *>(dst) + off, smem_u32(c_s) + off, min(32768u, bytes - off));
                bulk_commit();
                bulk_wait_all();
            }
            if (tx < kHeads) {
                const int h = tx;
                const float l = ctl.l[h], m = ctl.m[h];
                if (p.n_split > 1) {
                    float *ml = p.part_ml + (((int64_t)t * p.n_split + split) * kHeads + h) * 2;
                    ml[0] = l > 0.f ? m : -INFINITY;
                    ml[1] = l;
                } else if (p.lse && h < H) {
                    p.lse[(int64_t)t * H + h] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (p.clustered) {
        // ---- split-KV reduction inside the cluster (the token's n_split CTAs):
        // every CTA scales its unnormalised O^T by 2^(m - M) and sends each
        // output slice to the CTA that owns it; owners sum the slices in a
        // fixed order and write the normalised result.
        const int CS = p.n_split;
        const uint32_t my = cluster_rank();
        const bool ok = ctl.warp_alive[0] && ctl.warp_alive[1] && ctl.warp_alive[2] && ctl.warp_alive[3];
        const int tx = (int)threadIdx.x - 64;
        if (!ok && tx >= 0 && tx < kHeads) {                // a CTA that gave up contributes nothing
            ctl.m[tx] = -INFINITY;
            ctl.l[tx] = 0.f;
        }
        cluster_sync_all();                                  // every m, l final; every PV done
        const int dpo = D_L / CS;                            // output dims owned per CTA
        const uint32_t slot_bytes = (uint32_t)(kHeads * dpo * 4);
        const uint32_t recv = smem_u32(c_s);                 // the dead gathered tile holds the slots
        if (warp >= 2) {
            if (tx < kHeads) {
                float M = -INFINITY;
                for (int c = 0; c < CS; ++c) M = fmaxf(M, dsmem_ld_f32(dsmem_map(smem_u32(&ctl.m[tx]), c)));
                float L = 0.f;
                for (int c = 0; c < CS; ++c) {
                    const float mc = dsmem_ld_f32(dsmem_map(smem_u32(&ctl.m[tx]), c));
                    const float lc = dsmem_ld_f32(dsmem_map(smem_u32(&ctl.l[tx]), c));
                    if (mc != -INFINITY) L += exp2f(mc - M) * lc;
                }
                ctl.gm[tx] = M;
                ctl.gl[tx] = L;
                ctl.sc[tx] = ctl.m[tx] == -INFINITY ? 0.f : exp2f(ctl.m[tx] - M);
            }
            named_barrier(1, 128);
            const int quarter = warp & 3;
            const int r = quarter * 32 + (threadIdx.x & 31);
            const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
            if (ok) tc_fence_after();
            for (int c = 0; c < 4; ++c) {
                const int d = c * 128 + r;
                const uint32_t owner = (uint32_t)(d / dpo);
                const uint32_t dst = dsmem_map(recv + my * slot_bytes, owner) + (uint32_t)((d % dpo) * 4);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t u[32];
                    if (ok) {
                        tmem_ld32(tmem + lane_addr + kColO + c * kHeads + half * 32, u);
                        tmem_wait_ld();
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int h = half * 32 + j;
                        const float v = ok ? __uint_as_float(u[j]) * ctl.sc[h] : 0.f;
                        dsmem_st_f32(dst + (uint32_t)(h * dpo * 4), v);
                    }
                }
            }
        }
        cluster_sync_all();                                  // every slice delivered
        if (warp >= 2) {
            const int H = p.H;
            const uint8_t *slots = c_s;
            for (int e = tx; e < kHeads * dpo; e += 128) {
                const int h = e / dpo, dd = e % dpo;
                float acc = 0.f;
                for (int c = 0; c < CS; ++c)
                    acc += *reinterpret_cast<const float *>(slots + c * slot_bytes + (h * dpo + dd) * 4);
                if (h < H) {
                    const float L = ctl.gl[h];
                    p.out[((int64_t)t * H + h) * D_L + my * dpo + dd] = L > 0.f ? acc / L : 0.f;
                }
            }
            if (my == 0 && p.lse && tx < H) {
                const float L = ctl.gl[tx];
                p.lse[(int64_t)t * H + tx] = L > 0.f ? (ctl.gm[tx] + log2f(L)) * 0.69314718055994531f : -INFINITY;
            }
        }
    }
    // Dependents launch only now: CTAs of the next grid waiting on this one
    // would share the SMs and slow it down.
    pdl_trigger();
    tl_end(b.timeline, kTlAttn);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Merge split partials: o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
__global__ void __launch_bounds__(128) attn_combine_kernel(const float *__restrict__ part_o,
                                                           const float *__restrict__ part_ml,
                                                           int n_split, int H, float *out, float *lse,
                                                           unsigned long long *timeline) {
    __shared__ float wgt[128];
    __shared__ float ml[2][128];
    const int t = blockIdx.x, h = blockIdx.y;
    const int64_t base = (int64_t)t * n_split;
    tl_start(timeline, kTlCombine);
    pdl_wait();
    for (int s = threadIdx.x; s < n_split; s += 128) {      // all split statistics at once
        ml[0][s] = __ldg(part_ml + ((base + s) * kHeads + h) * 2);
        ml[1][s] = __ldg(part_ml + ((base + s) * kHeads + h) * 2 + 1);
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
    for (int s0 = 0; s0 < n_split; s0 += 16) {              // 16 loads in flight
        float4 o[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
            if (s0 + u < n_split)
                o[u] = __ldg(reinterpret_cast<const float4 *>(part_o + ((base + s0 + u) * kHeads + h) * D_L) +
                             threadIdx.x);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            if (s0 + u < n_split) {
                const float w = wgt[s0 + u];
                acc.x += w * o[u].x; acc.y += w * o[u].y; acc.z += w * o[u].z; acc.w += w * o[u].w;
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

size_t sparse_attn_smem_bytes() { return 1024 + kQBytes + kCBytes + sizeof(Ctl); }

cudaError_t launch_sparse_attn(const AttnLaunch &a, const CUtensorMap &q_lat_map,
                               const CUtensorMap &q_rope_map, const CUtensorMap &kv_map,
                               const DevBatch &b, uint32_t *status, cudaStream_t stream, bool pdl) {
    AttnParams p{};
    p.idx = a.idx;
    p.out = a.out;
    p.lse = a.lse;
    p.part_o = a.part_o;
    p.part_ml = a.part_ml;
    p.b = b;
    p.status = status;
    p.H = a.H;
    p.k = a.k;
    p.scale_log2 = a.sm_scale * 1.4426950408889634f;
    p.tiles_per_cta = a.tiles_per_cta;
    p.n_split = a.n_split;
    p.n_tiles = (a.k + kRows - 1) / kRows;
    const size_t smem = sparse_attn_smem_bytes();
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(sparse_attn_kernel), 1, smem);
    if (e != cudaSuccess) return e;
    if (a.n_split > 65535) return cudaErrorInvalidConfiguration;
    p.clustered = a.clustered;
    dim3 grid((unsigned)b.T, (unsigned)a.n_split);
    if (!a.clustered)
        return launch_k(sparse_attn_kernel, grid, dim3(kThreads), smem, stream, pdl, p, q_lat_map, q_rope_map,
                        kv_map);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)a.n_split;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, sparse_attn_kernel, p, q_lat_map, q_rope_map, kv_map);
}

// Whether the n_split CTAs of a token can run as one cluster on this device
// (cluster sizes above 8 need the non-portable opt-in and a GPC with that
// many free SMs).  Cached per device and size.
bool attn_cluster_ok(int n_split) {
    if (n_split < 2 || n_split > 16 || (n_split & (n_split - 1))) return false;
    static int cache[64][17];                 // 0 unknown, 1 yes, 2 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    int &c = cache[dev][n_split];
    if (c) return c == 1;
    c = 2;
    const size_t smem = sparse_attn_smem_bytes();
    if (ensure_smem_attr(reinterpret_cast<const void *>(sparse_attn_kernel), 1, smem) != cudaSuccess) return false;
    if (n_split > 8 && cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                           cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, (unsigned)n_split);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)n_split;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sparse_attn_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (n > 0) c = 1;
    return n > 0;
}

cudaError_t launch_attn_combine(const AttnLaunch &a, const DevBatch &b, cudaStream_t stream, bool pdl) {
    if (a.n_split <= 1 || a.clustered) return cudaSuccess;
    if (a.n_split > 128) return cudaErrorInvalidConfiguration;
    dim3 grid((unsigned)b.T, (unsigned)a.H);
    return launch_k(attn_combine_kernel, grid, dim3(128), 0, stream, pdl, (const float *)a.part_o,
                    (const float *)a.part_ml, a.n_split, a.H, a.out, a.lse, b.timeline);
}

}  // namespace dsa
