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
    if (P->T == 0) return PA_OK;
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

    int32_t *err = reinterpret_cast<int32_t *>(ws);
    const int32_t *part_offset = reinterpret_cast<const int32_t *>(ws + P->off_part);
    float *o_part = reinterpret_cast<float *>(ws + P->off_opart);
    float2 *ml_part = reinterpret_cast<float2 *>(ws + P->off_ml);
    uint16_t *out16 = static_cast<uint16_t *>(out);

    CUtensorMap tm_k, tm_v;
    const uint64_t rows = static_cast<uint64_t>(P->num_blocks) * kBlockSize;
    if (!make_map(&tm_k, key_cache, P->D, P->Hkv, rows, 1, kBlockSize) ||
        !make_map(&tm_v, value_cache, P->D, P->Hkv, rows, 1, kBlockSize))
        return PA_ERR_CUDA;
    if (!P->tiles.empty()) {
        CUtensorMap tm_q;
        if (!make_map(&tm_q, q, P->D, P->Hq, P->T, P->G, kTileRows / P->G)) return PA_ERR_CUDA;
        ExtendParams ep{};
        ep.out = out16;
        ep.block_table = block_table;
        ep.tiles = reinterpret_cast<const ExtendTile *>(ws + P->off_tiles);
        ep.part_offset = part_offset;
        ep.o_part = o_part;
        ep.ml_part = ml_part;
        ep.err = err;
        ep.num_tiles = static_cast<int32_t>(P->tiles.size());
        ep.max_blocks = P->max_blocks;
        ep.num_blocks = P->num_blocks;
        ep.num_heads_q = P->Hq;
        ep.group = P->G;
        ep.n_groups = P->n_groups;
        ep.heads_per_group = P->HG;
        ep.scale_log2 = P->scale_log2;
        if (launch_extend(P->D, tm_q, tm_k, tm_v, ep, stream) != cudaSuccess) return PA_ERR_CUDA;
    }
    if (!P->items.empty()) {
        DecodeParams dp{};
        dp.q = static_cast<const uint16_t *>(q);
        dp.out = out16;
        dp.block_table = block_table;
        dp.items = reinterpret_cast<const DecodeItem *>(ws + P->off_items);
        dp.cta_begin = reinterpret_cast<const int32_t *>(ws + P->off_cta);
        dp.part_offset = part_offset;
        dp.o_part = o_part;
        dp.ml_part = ml_part;
        dp.err = err;
        dp.max_blocks = P->max_blocks;
        dp.num_blocks = P->num_blocks;
        dp.num_heads_q = P->Hq;
        dp.group = P->G;
        dp.n_groups = P->n_groups;
        dp.scale_log2 = P->scale_log2;
        const int ncta = static_cast<int>(P->cta_begin.size()) - 1;
        if (launch_decode(P->D, P->HG, ncta, tm_k, tm_v, dp, stream) != cudaSuccess) return PA_ERR_CUDA;
    }
    if (!P->merges.empty()) {
        MergeParams mp{};
        mp.out = out16;
        mp.rows = reinterpret_cast<const MergeRow *>(ws + P->off_merges);
        mp.o_part = o_part;
        mp.ml_part = ml_part;
        mp.num_rows = static_cast<int32_t>(P->merges.size());
        mp.num_heads_q = P->Hq;
        mp.max_heads = P->HG * P->G;
        if (launch_merge(P->D, mp, stream) != cudaSuccess) return PA_ERR_CUDA;
    }
    if (device_error_word &&
        cudaMemcpyAsync(device_error_word, err, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}
