// noalloc.cu -- dsa_decode for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: a plugin inside a
// host framework that owns every device allocation and exposes no allocator,
// code that runs while a stream is being captured into a CUDA graph (where a
// cudaMalloc would break the capture), or an embedder with a fixed memory
// budget decided before the model starts.  dsa_decode_noalloc serves them: it
// runs exactly the kernels of dsa_decode, with the scratch those kernels need
// (status word, score slab, selected indices, split-attention partials) taken
// from one file-scope device array of fixed size instead of a caller buffer.
//
// The array is static device memory: every GPU that loads the library holds
// its 64 MiB until the process exits.  Nothing here calls cudaMalloc,
// cudaFree or any allocating library routine.
#include <mutex>

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_setup_mu;
void *g_scratch_ptr[kMaxDevices] = {};   // the address whose status block was last cleared

// Device address of the scratch array on the current device, looked up on
// every call (a device reset reloads the module, and the array may move);
// its status block is cleared whenever the address is new.
dsa_status_t scratch_for_current_device(cudaStream_t stream, void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSA_ERR_CUDA;
    void *p = nullptr;
    // In host code the array's name is only a stand-in; the runtime maps it
    // to this device's copy.
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch_ptr[dev] != p) {
        if (cudaMemsetAsync(p, 0, dsa::kStatusBytes, stream) != cudaSuccess) return DSA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = p;
    return DSA_OK;
}

}  // namespace

extern "C" dsa_status_t dsa_decode_noalloc(const void *k_new, int k_dtype, const dsa_f16 *q_idx,
                                           const float *w, const dsa_bf16 *q_lat, const dsa_bf16 *q_rope,
                                           dsa_f16 *k_cache, const dsa_bf16 *kv_cache,
                                           const dsa_batch_t *batch, int H_I, int H, int k,
                                           float sm_scale, int hadamard, float *out, float *lse,
                                           int32_t *idx_out, cudaStream_t stream) {
    // Size check first: a batch whose scratch would not fit is refused before
    // the device is touched.
    size_t need = 0;
    dsa_status_t s = dsa_workspace_size(DSA_OP_DECODE, batch, H_I, H, k, &need);
    if (s != DSA_OK) return s;
    if (need > kNoallocScratchBytes) return DSA_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    if ((s = scratch_for_current_device(stream, &scratch)) != DSA_OK) return s;
    return dsa_decode(k_new, k_dtype, q_idx, w, q_lat, q_rope, k_cache, kv_cache, batch, H_I, H, k,
                      sm_scale, hadamard, out, lse, idx_out, scratch, kNoallocScratchBytes, stream);
}
