/*
 * decode_from_files.c -- a plain C caller of the DSA library: one dsa_decode
 * step on inputs read from files, outputs written to files.  Nothing but the
 * C ABI of include/dsa.h and the CUDA runtime (device memory, copies).
 *
 *   decode_from_files DIR
 *
 * DIR holds meta.bin and one raw little-endian file per tensor:
 *   meta.bin     int32 B, T, max_q_per_seq, max_kv, H_I, H, k, hadamard;
 *                int64 cache_rows; float sm_scale
 *   cu_q.bin int32 [B+1]   q_pos.bin int32 [T]   kv_off.bin int64 [B]
 *   k_new.bin f32 [T,128]  q_idx.bin f16 [T,H_I,128]  w.bin f32 [T,H_I]
 *   q_lat.bin bf16 [T,H,512]  q_rope.bin bf16 [T,H,64]
 *   k_cache.bin f16 [rows,128]  kv_cache.bin bf16 [rows,576]
 * and receives out.bin f32 [T,H,512], lse.bin f32 [T,H], idx.bin int32 [T,k],
 * k_cache_out.bin f16 [rows,128] (the cache with the step's keys appended).
 * Exit status 0 when every call returned DSA_OK and the device status word
 * is clean.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "dsa.h"

static char g_dir[4096];

static const char *path_of(const char *name) {
    static char buf[4200];
    snprintf(buf, sizeof buf, "%s/%s", g_dir, name);
    return buf;
}

/* Reads exactly `bytes` bytes of DIR/name into a new device buffer. */
static void *upload(const char *name, size_t bytes) {
    FILE *f = fopen(path_of(name), "rb");
    if (!f) { fprintf(stderr, "cannot open %s\n", name); exit(2); }
    void *h = malloc(bytes ? bytes : 1);
    if (!h || fread(h, 1, bytes, f) != bytes) { fprintf(stderr, "short read %s\n", name); exit(2); }
    fclose(f);
    void *d = NULL;
    if (cudaMalloc(&d, bytes ? bytes : 1) != cudaSuccess ||
        cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
        fprintf(stderr, "device copy of %s failed\n", name);
        exit(2);
    }
    free(h);
    return d;
}

static void download(const char *name, const void *d, size_t bytes) {
    void *h = malloc(bytes ? bytes : 1);
    if (!h || cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) {
        fprintf(stderr, "copy back of %s failed\n", name);
        exit(2);
    }
    FILE *f = fopen(path_of(name), "wb");
    if (!f || fwrite(h, 1, bytes, f) != bytes) { fprintf(stderr, "cannot write %s\n", name); exit(2); }
    fclose(f);
    free(h);
}

int main(int argc, char **argv) {
    if (argc != 2) { fprintf(stderr, "usage: %s DIR\n", argv[0]); return 2; }
    snprintf(g_dir, sizeof g_dir, "%s", argv[1]);

    int32_t m[8];
    int64_t cache_rows;
    float sm_scale;
    FILE *f = fopen(path_of("meta.bin"), "rb");
    if (!f || fread(m, sizeof m, 1, f) != 1 || fread(&cache_rows, sizeof cache_rows, 1, f) != 1 ||
        fread(&sm_scale, sizeof sm_scale, 1, f) != 1) {
        fprintf(stderr, "bad meta.bin\n");
        return 2;
    }
    fclose(f);
    const int B = m[0], T = m[1], max_q = m[2], max_kv = m[3], H_I = m[4], H = m[5], K = m[6], had = m[7];
    const size_t rows = (size_t)cache_rows;

    dsa_batch_t batch;
    batch.batch = B;
    batch.total_q = T;
    batch.max_q_per_seq = max_q;
    batch.max_kv = max_kv;
    batch.cache_rows = cache_rows;
    batch.cu_q = upload("cu_q.bin", (size_t)(B + 1) * 4);
    batch.q_pos = upload("q_pos.bin", (size_t)T * 4);
    batch.kv_off = upload("kv_off.bin", (size_t)B * 8);

    const float *k_new = upload("k_new.bin", (size_t)T * 128 * 4);
    const dsa_f16 *q_idx = upload("q_idx.bin", (size_t)T * H_I * 128 * 2);
    const float *w = upload("w.bin", (size_t)T * H_I * 4);
    const dsa_bf16 *q_lat = upload("q_lat.bin", (size_t)T * H * 512 * 2);
    const dsa_bf16 *q_rope = upload("q_rope.bin", (size_t)T * H * 64 * 2);
    dsa_f16 *k_cache = upload("k_cache.bin", rows * 128 * 2);
    const dsa_bf16 *kv_cache = upload("kv_cache.bin", rows * 576 * 2);

    float *out = NULL, *lse = NULL;
    int32_t *idx = NULL;
    void *ws = NULL;
    size_t ws_bytes = 0;
    if (cudaMalloc((void **)&out, (size_t)T * H * 512 * 4) != cudaSuccess ||
        cudaMalloc((void **)&lse, (size_t)T * H * 4) != cudaSuccess ||
        cudaMalloc((void **)&idx, (size_t)T * K * 4) != cudaSuccess) {
        fprintf(stderr, "output allocation failed\n");
        return 2;
    }

    dsa_status_t st = dsa_workspace_size(DSA_OP_DECODE, &batch, H_I, H, K, &ws_bytes);
    if (st == DSA_OK && cudaMalloc(&ws, ws_bytes) != cudaSuccess) st = DSA_ERR_CUDA;
    if (st == DSA_OK) st = dsa_workspace_init(ws, ws_bytes, NULL);
    if (st == DSA_OK)
        st = dsa_decode(k_new, DSA_KEY_F32, q_idx, w, q_lat, q_rope, k_cache, kv_cache, &batch, H_I, H, K,
                        sm_scale, had, out, lse, idx, ws, ws_bytes, NULL);
    uint32_t flags = 0;
    if (st == DSA_OK) st = dsa_read_device_status(ws, NULL, &flags);
    printf("dsa_decode: %s, device flags %u\n", dsa_status_string(st), (unsigned)flags);
    if (st != DSA_OK) return 1;

    download("out.bin", out, (size_t)T * H * 512 * 4);
    download("lse.bin", lse, (size_t)T * H * 4);
    download("idx.bin", idx, (size_t)T * K * 4);
    download("k_cache_out.bin", k_cache, rows * 128 * 2);
    return 0;
}
