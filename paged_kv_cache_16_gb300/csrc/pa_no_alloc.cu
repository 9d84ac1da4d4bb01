// pa_attention_no_alloc: the attention entry point for callers that cannot
// allocate device memory.
//
// Who needs it: an engine that sizes its paged KV pool at start-up to take
// nearly all free device memory has no room left for a per-step workspace,
// and a hot path that must not call cudaMalloc / cudaFree (those calls can
// synchronise the whole device and stall every stream) cannot create one on
// demand.  Such callers still own q, the caches, the block table and the
// output; only the scratch space moves into the library.
//
// The scratch is one file-scope device array of PA_NO_ALLOC_SCRATCH_BYTES,
// created on a device when this module is loaded there and kept until the
// process exits.  Its device address is looked up once per device (on the
// first call made with that device current) and passed to the same kernels
// pa_attention launches.  Nothing here allocates: no cudaMalloc, no
// cudaMallocHost, no cudaFree, no event creation.
#include <cstring>
#include <mutex>

#include "plan.h"

namespace {

constexpr size_t kScratchBytes = PA_NO_ALLOC_SCRATCH_BYTES;

// Shared by every call on a device; keeps the last call's contents.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once).
pa_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PA_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" pa_status pa_attention_no_alloc(const pa_plan_t *plan, const void *q, const void *key_cache,
                                           const void *value_cache, const int32_t *block_table, void *out,
                                           int32_t *device_error_word, void *stream_) {
    using namespace pa;
    if (!plan) return PA_ERR_INVALID_ARGUMENT;
    pa_plan_s *P = const_cast<pa_plan_s *>(plan);
    if (P->T == 0) {
        // nothing to attend; the error word still receives this call's bits (none)
        if (device_error_word && (!aligned(device_error_word, 4) ||
                                  cudaMemsetAsync(device_error_word, 0, sizeof(int32_t),
                                                  static_cast<cudaStream_t>(stream_)) != cudaSuccess))
            return aligned(device_error_word, 4) ? PA_ERR_CUDA : PA_ERR_INVALID_ARGUMENT;
        return PA_OK;
    }
    if (!q || !key_cache || !value_cache || !block_table || !out) return PA_ERR_INVALID_ARGUMENT;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) ||
        !aligned(block_table, 4) || (device_error_word && !aligned(device_error_word, 4)))
        return PA_ERR_INVALID_ARGUMENT;
    if (P->ws_bytes > kScratchBytes) return PA_ERR_WORKSPACE_TOO_SMALL;  // plan needs more than the array
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    void *scratch = nullptr;
    pa_status st = scratch_address(&scratch);
    if (st != PA_OK) return st;
    std::lock_guard<std::mutex> lock(P->mu);
    uint8_t *ws = static_cast<uint8_t *>(scratch);

    // The error word must start at zero; metadata and partials are fully
    // rewritten by this call before they are read.
    if (cudaMemsetAsync(ws, 0, sizeof(int32_t), stream) != cudaSuccess) return PA_ERR_CUDA;
    if (P->blob_bytes &&
        cudaMemcpyAsync(ws + kWorkspaceHeader, P->blob.data(), P->blob_bytes, cudaMemcpyHostToDevice, stream) !=
            cudaSuccess)
        return PA_ERR_CUDA;

    // one stream only: no library stream or event is created for this call
    const pa_status es = enqueue_attention(P, q, key_cache, value_cache, block_table, out, ws, stream, false,
                                           KvUpdate{}, false);
    if (es != PA_OK) return es;
    const int32_t *err = reinterpret_cast<const int32_t *>(ws);
    if (device_error_word &&
        cudaMemcpyAsync(device_error_word, err, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}
