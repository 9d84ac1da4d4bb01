// Native graph executor (pa_graph_*): graph mode of the page "vLLM 源码完全拆解
// （十六）" (fourth walk-through) without a framework around it.  The execution
// of one fixed shape is captured once into two CUDA graphs; each step plans on
// the host, copies the plan's metadata image into the page-locked buffer the
// next graph uploads from, and launches that graph.  Two images and two
// graphs alternate so that the host prepares step n+1 while step n may still
// run; an event per graph says when its image (and host I/O buffers) may be
// rewritten.
//
// Built on the public C ABI only (pa_plan_fixed, pa_upload_metadata[_from],
// pa_slot_mapping, pa_write_kv[_fp8], pa_attention[_with_kv_update]_launch):
// the graphs hold exactly the launches a caller capturing by hand would get.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <utility>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/pa.h"

struct pa_graph_s {
    pa_batch_desc model{};        // model fields of the creation step (array pointers unused)
    pa_fixed_shape shape{};
    pa_graph_buffers bufs{};
    pa_plan_t *capture_plan = nullptr;
    void *workspace = nullptr;
    size_t ws_bytes = 0;
    int64_t *slots = nullptr;
    void *image[2] = {nullptr, nullptr};   // page-locked, device-mapped metadata images
    size_t image_bytes = 0;
    cudaGraphExec_t exec[2] = {nullptr, nullptr};
    cudaEvent_t done[2] = {nullptr, nullptr};
    bool launched[2] = {false, false};
    cudaStream_t cap = nullptr;
    int turn = 0;
    // staged host input (shape.decode_prefix_tokens > 0): the bytes of the
    // input image the decode stream needs are copied first, the rows from the
    // prefix on after them on a second stream, and only the work that reads
    // those rows waits for them
    bool staged = false;
    std::vector<std::pair<size_t, size_t>> early, late;   // [begin, end) byte ranges of the image
    cudaStream_t cap_late = nullptr;
    cudaEvent_t early_in = nullptr, late_in = nullptr;
    cudaEvent_t late_out = nullptr, late_copied = nullptr;   // rows from the prefix on: final, copied back
};

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool page_locked(const void *p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

// the fields a captured graph bakes in
bool same_model(const pa_batch_desc &a, const pa_batch_desc &b) {
    return a.num_heads_q == b.num_heads_q && a.num_heads_kv == b.num_heads_kv && a.head_dim == b.head_dim &&
           a.block_size == b.block_size && a.num_blocks == b.num_blocks &&
           a.max_blocks_per_req == b.max_blocks_per_req && a.softmax_scale == b.softmax_scale &&
           a.num_sms == b.num_sms && a.kv_cache_dtype == b.kv_cache_dtype && a.k_scale == b.k_scale &&
           a.v_scale == b.v_scale;
}

pa_status check_buffers(const pa_graph_buffers &b) {
    if (!b.q || !b.key || !b.value || !b.out || !b.query_start_loc || !b.num_computed || !b.block_table ||
        !b.key_cache || !b.value_cache)
        return PA_ERR_INVALID_ARGUMENT;
    if (!aligned16(b.q) || !aligned16(b.key) || !aligned16(b.value) || !aligned16(b.out) ||
        !aligned16(b.key_cache) || !aligned16(b.value_cache))
        return PA_ERR_INVALID_ARGUMENT;
    const bool any_in = b.host_in[0] || b.host_in[1] || b.device_in || b.in_bytes;
    const bool all_in = b.host_in[0] && b.host_in[1] && b.device_in && b.in_bytes;
    const bool any_out = b.host_out[0] || b.host_out[1] || b.out_bytes;
    const bool all_out = b.host_out[0] && b.host_out[1] && b.out_bytes;
    if (any_in != all_in || any_out != all_out) return PA_ERR_INVALID_ARGUMENT;
    for (int i = 0; i < 2; ++i) {
        if (all_in && !page_locked(b.host_in[i])) return PA_ERR_INVALID_ARGUMENT;
        if (all_out && !page_locked(b.host_out[i])) return PA_ERR_INVALID_ARGUMENT;
    }
    return PA_OK;
}

// The step's launches over the graph's buffers, as a caller would enqueue
// them: fused write + attention, or slot mapping, cache write, attention;
// the output rows go to `out`.
pa_status enqueue_step(const pa_graph_s *g, const pa_plan_t *plan, void *out, cudaStream_t s) {
    const pa_graph_buffers &b = g->bufs;
    if (b.fused)
        return pa_attention_with_kv_update_launch(plan, b.q, b.key, b.value, b.key_cache, b.value_cache,
                                                  b.block_table, g->slots, out, g->workspace, g->ws_bytes, s);
    const pa_batch_desc &m = g->model;
    pa_status st = pa_slot_mapping(b.query_start_loc, b.num_computed, b.block_table, g->shape.max_reqs,
                                   g->shape.max_tokens, m.max_blocks_per_req, m.block_size, g->slots, s);
    if (st != PA_OK) return st;
    const int64_t num_slots = static_cast<int64_t>(m.num_blocks) * m.block_size;
    int32_t *err = static_cast<int32_t *>(g->workspace);
    if (m.kv_cache_dtype == PA_KV_FP8_E4M3)
        st = pa_write_kv_fp8(b.key, b.value, g->slots, g->shape.max_tokens, m.num_heads_kv, m.head_dim, b.key_cache,
                             b.value_cache, num_slots, m.k_scale, m.v_scale, err, s);
    else
        st = pa_write_kv(b.key, b.value, g->slots, g->shape.max_tokens, m.num_heads_kv, m.head_dim, b.key_cache,
                         b.value_cache, num_slots, err, s);
    if (st != PA_OK) return st;
    return pa_attention_launch(plan, b.q, b.key_cache, b.value_cache, b.block_table, out, g->workspace,
                               g->ws_bytes, s);
}

// The device address of host_out[i] when the kernels can store the output
// straight into it: out_bytes spans the whole output buffer, so every row a
// step can write lies inside it.  The stores cross the host link while the
// step runs (the tiles' rows while the decode stream still streams) instead
// of one copy after it.  nullptr: copy device `out` back at the end.
void *direct_host_out(const pa_graph_s *g, int i) {
    const pa_graph_buffers &b = g->bufs;
    if (!b.out_bytes || g->staged) return nullptr;
    const size_t full = static_cast<size_t>(g->shape.max_tokens) * g->model.num_heads_q * g->model.head_dim * 2;
    void *dptr = nullptr;
    if (b.out_bytes < full || cudaHostGetDevicePointer(&dptr, b.host_out[i], 0) != cudaSuccess || !aligned16(dptr)) {
        cudaGetLastError();
        return nullptr;
    }
    return dptr;
}

// Staging of the host input: the rows from decode_prefix_tokens on of q, key
// and value, where those buffers lie inside device_in, are copied late;
// everything else in the image (the other rows, the metadata arrays) first.
void plan_staging(pa_graph_s *g) {
    const pa_graph_buffers &b = g->bufs;
    const int64_t P = g->shape.decode_prefix_tokens, T = g->shape.max_tokens;
    if (!b.fused || !b.in_bytes || P <= 0 || P >= T) return;
    const size_t dq = static_cast<size_t>(g->model.num_heads_q) * g->model.head_dim * 2;
    const size_t dkv = static_cast<size_t>(g->model.num_heads_kv) * g->model.head_dim * 2;
    const uintptr_t base = reinterpret_cast<uintptr_t>(b.device_in);
    std::vector<std::pair<size_t, size_t>> span, late;
    for (const auto &buf : {std::make_pair(b.q, dq), std::make_pair(b.key, dkv), std::make_pair(b.value, dkv)}) {
        const uintptr_t p = reinterpret_cast<uintptr_t>(buf.first);
        if (p < base || p + buf.second * T > base + b.in_bytes) return;   // not inside the image: one copy
        span.emplace_back(p - base, p - base + buf.second * T);
        late.emplace_back(p - base + buf.second * P, p - base + buf.second * T);
    }
    std::sort(span.begin(), span.end());
    for (size_t k = 1; k < span.size(); ++k)
        if (span[k].first < span[k - 1].second) return;                  // overlapping buffers: one copy
    std::sort(late.begin(), late.end());
    size_t at = 0;
    for (const auto &r : late) {
        if (r.first > at) g->early.emplace_back(at, r.first);
        at = r.second;
    }
    if (at < b.in_bytes) g->early.emplace_back(at, b.in_bytes);
    g->late = late;
    g->staged = true;
}

cudaError_t copy_ranges(const std::vector<std::pair<size_t, size_t>> &ranges, void *dst, const void *src,
                        cudaStream_t s) {
    for (const auto &r : ranges) {
        const cudaError_t e = cudaMemcpyAsync(static_cast<char *>(dst) + r.first, static_cast<const char *>(src) + r.first,
                                              r.second - r.first, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Capture graph i on the capture stream.  The capture is always ended, also
// after a failed call inside it.
pa_status capture(pa_graph_s *g, int i) {
    const pa_graph_buffers &b = g->bufs;
    if (cudaStreamBeginCapture(g->cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return PA_ERR_CUDA;
    pa_status st = PA_OK;
    // one copy each way (splitting them over parallel streams measured
    // slower), or, staged, the early part and the metadata upload (which
    // reads its image over the same host link) and only then the late rows
    if (g->staged) {
        if (copy_ranges(g->early, b.device_in, b.host_in[i], g->cap) != cudaSuccess) st = PA_ERR_CUDA;
        if (st == PA_OK) st = pa_upload_metadata_from(g->image[i], g->image_bytes, g->workspace, g->ws_bytes, g->cap);
        if (st == PA_OK && (cudaEventRecord(g->early_in, g->cap) != cudaSuccess ||
                            cudaStreamWaitEvent(g->cap_late, g->early_in, 0) != cudaSuccess ||
                            copy_ranges(g->late, b.device_in, b.host_in[i], g->cap_late) != cudaSuccess ||
                            cudaEventRecord(g->late_in, g->cap_late) != cudaSuccess))
            st = PA_ERR_CUDA;
    } else {
        if (b.in_bytes && cudaMemcpyAsync(b.device_in, b.host_in[i], b.in_bytes, cudaMemcpyHostToDevice, g->cap) !=
                              cudaSuccess)
            st = PA_ERR_CUDA;
        if (st == PA_OK) st = pa_upload_metadata_from(g->image[i], g->image_bytes, g->workspace, g->ws_bytes, g->cap);
    }
    void *direct = direct_host_out(g, i);
    void *out = direct ? direct : b.out;
    // staged with a whole-output host buffer: the rows from the prefix on are
    // copied back on the second stream as soon as the tiles have written
    // them, while the decode stream still runs; rows [0, P) after the step
    const size_t row_bytes = static_cast<size_t>(g->model.num_heads_q) * g->model.head_dim * 2;
    const size_t full = static_cast<size_t>(g->shape.max_tokens) * row_bytes;
    const bool split_back = g->staged && b.out_bytes >= full;
    if (st == PA_OK && g->staged)
        st = pa_attention_with_kv_update_launch_staged(g->capture_plan, b.q, b.key, b.value, b.key_cache,
                                                        b.value_cache, b.block_table, g->slots, out, g->workspace,
                                                        g->ws_bytes, g->cap, g->late_in,
                                                        split_back ? g->late_out : nullptr);
    else if (st == PA_OK)
        st = enqueue_step(g, g->capture_plan, out, g->cap);
    if (st == PA_OK && split_back) {
        const size_t early = static_cast<size_t>(g->shape.decode_prefix_tokens) * row_bytes;
        if (cudaStreamWaitEvent(g->cap_late, g->late_out, 0) != cudaSuccess ||
            cudaMemcpyAsync(static_cast<char *>(b.host_out[i]) + early, static_cast<const char *>(b.out) + early,
                            full - early, cudaMemcpyDeviceToHost, g->cap_late) != cudaSuccess ||
            cudaEventRecord(g->late_copied, g->cap_late) != cudaSuccess ||
            cudaMemcpyAsync(b.host_out[i], b.out, early, cudaMemcpyDeviceToHost, g->cap) != cudaSuccess ||
            cudaStreamWaitEvent(g->cap, g->late_copied, 0) != cudaSuccess)
            st = PA_ERR_CUDA;
    } else if (st == PA_OK && b.out_bytes && !direct &&
               cudaMemcpyAsync(b.host_out[i], b.out, b.out_bytes, cudaMemcpyDeviceToHost, g->cap) != cudaSuccess) {
        st = PA_ERR_CUDA;
    }
    cudaGraph_t graph = nullptr;
    const cudaError_t end = cudaStreamEndCapture(g->cap, &graph);
    if (st == PA_OK && (end != cudaSuccess || graph == nullptr)) st = PA_ERR_CUDA;
    if (st == PA_OK && cudaGraphInstantiate(&g->exec[i], graph, 0) != cudaSuccess) {
        g->exec[i] = nullptr;
        st = PA_ERR_CUDA;
    }
    if (graph) cudaGraphDestroy(graph);
    if (st != PA_OK) cudaGetLastError();
    return st;
}

}  // namespace

extern "C" {

pa_status pa_graph_create(const pa_batch_desc *desc, const pa_fixed_shape *shape, const pa_graph_buffers *bufs,
                          pa_graph_t **out) {
    if (out) *out = nullptr;
    if (!desc || !shape || !bufs || !out) return PA_ERR_INVALID_ARGUMENT;
    pa_status st = check_buffers(*bufs);
    if (st != PA_OK) return st;
    pa_graph_s *g = new (std::nothrow) pa_graph_s;
    if (!g) return PA_ERR_CUDA;
    g->model = *desc;
    g->model.query_start_loc = g->model.seq_lens = g->model.num_computed_tokens = nullptr;
    g->model.block_table_host = nullptr;
    g->shape = *shape;
    g->bufs = *bufs;
    st = pa_plan_fixed(desc, shape, &g->capture_plan, &g->ws_bytes);
    if (st != PA_OK) {
        delete g;
        return st;
    }
    g->image_bytes = (pa_plan_metadata_bytes(g->capture_plan) + 15) & ~static_cast<size_t>(15);
    if (g->image_bytes == 0) g->image_bytes = 16;
    bool ok = cudaMalloc(&g->workspace, g->ws_bytes) == cudaSuccess &&
              cudaMemset(g->workspace, 0, g->ws_bytes) == cudaSuccess &&
              cudaMalloc(reinterpret_cast<void **>(&g->slots), sizeof(int64_t) * g->shape.max_tokens) == cudaSuccess &&
              cudaStreamCreateWithFlags(&g->cap, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; ok && i < 2; ++i)
        ok = cudaHostAlloc(&g->image[i], g->image_bytes, cudaHostAllocMapped) == cudaSuccess &&
             cudaEventCreateWithFlags(&g->done[i], cudaEventDisableTiming) == cudaSuccess;
    plan_staging(g);
    if (ok && g->staged)
        ok = cudaStreamCreateWithFlags(&g->cap_late, cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&g->early_in, cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&g->late_in, cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&g->late_out, cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&g->late_copied, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        pa_graph_destroy(g);
        return PA_ERR_CUDA;
    }
    for (int i = 0; i < 2 && st == PA_OK; ++i)
        st = pa_plan_copy_metadata(g->capture_plan, g->image[i], g->image_bytes);
    // eager upload: prepares the kernels before the first capture
    if (st == PA_OK) st = pa_upload_metadata(g->capture_plan, g->workspace, g->ws_bytes, g->cap);
    if (st == PA_OK && cudaStreamSynchronize(g->cap) != cudaSuccess) st = PA_ERR_CUDA;
    for (int i = 0; i < 2 && st == PA_OK; ++i) st = capture(g, i);
    if (st != PA_OK) {
        pa_graph_destroy(g);
        return st;
    }
    *out = g;
    return PA_OK;
}

pa_status pa_graph_step(pa_graph_t *g, const pa_batch_desc *desc, void *stream) {
    if (!g || !desc) return PA_ERR_INVALID_ARGUMENT;
    if (!same_model(g->model, *desc)) return PA_ERR_INVALID_ARGUMENT;
    const int i = g->turn;
    if (g->launched[i] && cudaEventSynchronize(g->done[i]) != cudaSuccess) return PA_ERR_CUDA;
    pa_plan_t *plan = nullptr;
    size_t ws = 0;
    pa_status st = pa_plan_fixed(desc, &g->shape, &plan, &ws);
    if (st != PA_OK) return st;
    if (ws > g->ws_bytes || pa_plan_metadata_bytes(plan) > g->image_bytes) st = PA_ERR_INVALID_ARGUMENT;
    if (st == PA_OK) st = pa_plan_copy_metadata(plan, g->image[i], g->image_bytes);
    pa_plan_destroy(plan);
    if (st != PA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaGraphLaunch(g->exec[i], s) != cudaSuccess || cudaEventRecord(g->done[i], s) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    g->launched[i] = true;
    g->turn = 1 - i;
    return PA_OK;
}

int32_t pa_graph_turn(const pa_graph_t *g) { return g ? g->turn : 0; }

pa_status pa_graph_wait(pa_graph_t *g, int32_t turn) {
    if (!g || turn < 0 || turn > 1) return PA_ERR_INVALID_ARGUMENT;
    if (g->launched[turn] && cudaEventSynchronize(g->done[turn]) != cudaSuccess) return PA_ERR_CUDA;
    return PA_OK;
}

void *pa_graph_workspace(const pa_graph_t *g) { return g ? g->workspace : nullptr; }

int64_t *pa_graph_slot_mapping(const pa_graph_t *g) { return g ? g->slots : nullptr; }

void pa_graph_destroy(pa_graph_t *g) {
    if (!g) return;
    for (int i = 0; i < 2; ++i) {
        if (g->launched[i]) cudaEventSynchronize(g->done[i]);
        if (g->exec[i]) cudaGraphExecDestroy(g->exec[i]);
        if (g->done[i]) cudaEventDestroy(g->done[i]);
        if (g->image[i]) cudaFreeHost(g->image[i]);
    }
    if (g->cap) {
        cudaStreamSynchronize(g->cap);
        cudaStreamDestroy(g->cap);
    }
    if (g->cap_late) {
        cudaStreamSynchronize(g->cap_late);
        cudaStreamDestroy(g->cap_late);
    }
    if (g->early_in) cudaEventDestroy(g->early_in);
    if (g->late_in) cudaEventDestroy(g->late_in);
    if (g->late_out) cudaEventDestroy(g->late_out);
    if (g->late_copied) cudaEventDestroy(g->late_copied);
    if (g->workspace) cudaFree(g->workspace);
    if (g->slots) cudaFree(g->slots);
    if (g->capture_plan) pa_plan_destroy(g->capture_plan);
    cudaGetLastError();
    delete g;
}

}  // extern "C"
