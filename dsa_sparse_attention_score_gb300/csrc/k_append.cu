// k_append.cu -- indexer-key append with optional Walsh-Hadamard rotation.
//
// ik_llama_opt commit log, "GLM-5.2 DSA indexer: decode-correct via persistent
// indexer-K cache": the batch's (Hadamard-rotated) indexer keys are written to
// the fp16 single-head key cache at the tokens' own slots before scoring; the
// rotation is orthonormal and improves the precision of the fp16 cache.
//
// One warp per new key row.  Lane l holds elements 4l..4l+3.  The 128-point
// transform runs as 7 butterfly stages in float64: two inside a lane, five
// across lanes by shuffles.  For fp16 inputs every partial sum is exact in
// float64 (multiples of 2^-24 below 2^23), so the only rounding is the final
// one to fp16 after the 1/sqrt(128) scale -- the value the definition gives.
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {

__global__ void __launch_bounds__(128) k_append_kernel(const void *__restrict__ k_new, int k_dtype,
                                                       DevBatch b, uint16_t *__restrict__ k_cache,
                                                       int hadamard, uint32_t *status) {
    pdl_trigger();  // the score kernel may start its prologue now
    tl_start(b.timeline, kTlAppend);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 4 + warp;
    if (t >= b.T) return;
    // Independent loads first: position, this lane's four key values, and the
    // sequence lookup (one cu_q entry per lane); then the sequence's offset.
    const int32_t pos = __ldg(b.q_pos + t);
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
    const int s = seq_of_warp(b.cu_q, b.B, t, lane);
    const int64_t kv0 = seq_base(b, s);
    const int64_t row = (pos >= 0 && pos < b.max_kv && kv0 >= 0) ? cache_row(b, s, kv0, pos) : -1;
    if (row < 0 || row >= b.cache_rows) {
        if (lane == 0) flag(status, DSA_DEV_BAD_POSITION);
        return;
    }
    if (hadamard) {
        // element index i = 4*lane + e: bits 0-1 are e, bits 2-6 are the lane.
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
    uint16_t h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) h[e] = __half_as_ushort(__double2half(v[e]));
    uint2 out;
    out.x = (uint32_t)h[0] | ((uint32_t)h[1] << 16);
    out.y = (uint32_t)h[2] | ((uint32_t)h[3] << 16);
    reinterpret_cast<uint2 *>(k_cache + row * D_I)[lane] = out;
    __syncwarp();
    if (lane == 0 && b.timeline) atomicMax(b.timeline + 2 * kTlAppend + 1, (unsigned long long)global_ns());
}

cudaError_t launch_k_append(const void *k_new, int k_dtype, const DevBatch &b, uint16_t *k_cache,
                            int hadamard, uint32_t *status, cudaStream_t stream) {
    const int blocks = (b.T + 3) / 4;
    k_append_kernel<<<blocks, 128, 0, stream>>>(k_new, k_dtype, b, k_cache, hadamard, status);
    return cudaGetLastError();
}

}  // namespace dsa
