// Bandwidth-trivial kernels of the step: slot mapping, the KV-cache scatter,
// block zeroing, the FP8 block expansion and the merge of partition partials.
#include "dev.cuh"

namespace pa {
namespace {

// slot of every scheduled token ("vLLM 推理流程分析" §5.1.2 compute_slot_mapping):
// the request is found by binary search over query_start_loc.
__global__ void slot_mapping_kernel(const int32_t *__restrict__ qsl,
                                    const int32_t *__restrict__ num_computed,
                                    const int32_t *__restrict__ block_table, int32_t num_reqs,
                                    int32_t num_tokens, int32_t max_blocks, int32_t block_size,
                                    int64_t *__restrict__ slots) {
    const int32_t t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= num_tokens) return;
    if (t >= qsl[num_reqs]) {            // padding of a launch sized for a token capacity
        slots[t] = -1;
        return;
    }
    int32_t lo = 0, hi = num_reqs - 1;  // last r with qsl[r] <= t
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (qsl[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int32_t pos = num_computed[lo] + (t - qsl[lo]);
    const int32_t blk = block_table[static_cast<int64_t>(lo) * max_blocks + pos / block_size];
    slots[t] = static_cast<int64_t>(blk) * block_size + pos % block_size;
}

// reshape_and_cache ("vLLM 推理流程分析" §6.3): one thread moves one 16-byte
// chunk of one token's key row and the same chunk of its value row.
// Consecutive threads touch consecutive chunks, so loads and stores coalesce.
__global__ void write_kv_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                                const int64_t *__restrict__ slots, int64_t total_chunks,
                                int32_t chunks_per_row, uint4 *__restrict__ key_cache,
                                uint4 *__restrict__ value_cache, int64_t num_slots,
                                int32_t *err) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
         i < total_chunks; i += stride) {
        const int64_t t = i / chunks_per_row;
        const int32_t c = static_cast<int32_t>(i - t * chunks_per_row);
        // the source chunks do not depend on the slot: loaded together with it
        const uint4 kv = __ldcs(key + i);
        const uint4 vv = __ldcs(value + i);
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (err != nullptr && c == 0) atomicOr(err, kErrSlotRange);
            continue;
        }
        key_cache[slot * chunks_per_row + c] = kv;
        value_cache[slot * chunks_per_row + c] = vv;
    }
}

// reshape_and_cache into E4M3 caches ("vLLM 推理流程分析" §6.3, FP8 conversion
// with k_scale / v_scale): one thread turns 16 bf16 elements of a token's key
// row (and of its value row) into 16 codes, code = E4M3(bf16 / scale) with the
// quotient rounded once in IEEE binary32.
__device__ __forceinline__ uint4 quantize16(uint4 a, uint4 b, float scale) {
    const uint2 lo = dev::e4m3_quantize8(a, scale), hi = dev::e4m3_quantize8(b, scale);
    return make_uint4(lo.x, lo.y, hi.x, hi.y);
}

__global__ void write_kv_fp8_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                                    const int64_t *__restrict__ slots, int64_t total_chunks,
                                    int32_t chunks_per_row, uint4 *__restrict__ key_cache,
                                    uint4 *__restrict__ value_cache, int64_t num_slots, float k_scale,
                                    float v_scale, int32_t *err) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total_chunks; i += stride) {
        const int64_t t = i / chunks_per_row;
        const int32_t c = static_cast<int32_t>(i - t * chunks_per_row);
        // the source chunks do not depend on the slot: loaded together with it
        const uint4 k0 = __ldcs(key + 2 * i), k1 = __ldcs(key + 2 * i + 1);
        const uint4 v0 = __ldcs(value + 2 * i), v1 = __ldcs(value + 2 * i + 1);
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (err != nullptr && c == 0) atomicOr(err, kErrSlotRange);
            continue;
        }
        key_cache[slot * chunks_per_row + c] = quantize16(k0, k1, k_scale);
        value_cache[slot * chunks_per_row + c] = quantize16(v0, v1, v_scale);
    }
}

// E4M3 cache blocks read by the tensor-core tiles, expanded to bf16 scratch
// blocks: the code values themselves (exact in bf16; the scales are applied
// by the attention kernels).  One CTA per block.
__device__ __forceinline__ void expand16(const uint4 codes, uint4 *dst) {
    const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t h0 = dev::e4m3x2_to_f16x2(w[i] & 0xFFFFu);
        const uint32_t h1 = dev::e4m3x2_to_f16x2(w[i] >> 16);
        o[2 * i] = dev::pack_bf16x2(dev::f16_lo(h0), dev::f16_hi(h0));
        o[2 * i + 1] = dev::pack_bf16x2(dev::f16_lo(h1), dev::f16_hi(h1));
    }
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

__global__ void dequant_kernel(DequantParams p) {
    dev::grid_launch_dependents();
    dev::grid_dep_wait();
    const int32_t n = p.counts[kCountDequant];
    const int32_t chunks = p.block_elems / 16;
    for (int32_t i = blockIdx.x; i < n; i += gridDim.x) {
        const DequantItem it = p.items[i];
        const int32_t src = p.block_table[static_cast<int64_t>(it.req) * p.max_blocks + it.block];
        uint4 *kd = reinterpret_cast<uint4 *>(p.key_out + static_cast<int64_t>(it.dst) * p.block_elems);
        uint4 *vd = reinterpret_cast<uint4 *>(p.value_out + static_cast<int64_t>(it.dst) * p.block_elems);
        if (src < 0 || src >= p.num_blocks) {
            if (threadIdx.x == 0) atomicOr(p.err, kErrBlockRange);
            for (int32_t c = threadIdx.x; c < 2 * chunks; c += blockDim.x) kd[c] = vd[c] = make_uint4(0, 0, 0, 0);
            continue;
        }
        const uint4 *ks = reinterpret_cast<const uint4 *>(p.key_cache + static_cast<int64_t>(src) * p.block_elems);
        const uint4 *vs = reinterpret_cast<const uint4 *>(p.value_cache + static_cast<int64_t>(src) * p.block_elems);
        // a thread's chunks of the block are all loaded before any is
        // stored: one round trip to memory instead of one per chunk
        constexpr int U = 4;
        for (int32_t c0 = threadIdx.x; c0 < chunks; c0 += U * blockDim.x) {
            uint4 kx[U], vx[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int32_t c = c0 + u * static_cast<int32_t>(blockDim.x);
                if (c < chunks) {
                    kx[u] = __ldg(ks + c);
                    vx[u] = __ldg(vs + c);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int32_t c = c0 + u * static_cast<int32_t>(blockDim.x);
                if (c < chunks) {
                    expand16(kx[u], kd + 2 * c);
                    expand16(vx[u], vd + 2 * c);
                }
            }
        }
    }
}

// Fused cache update, extend rows (pa_attention_with_kv_update): token e of
// the runs' concatenation lies in the last run with wbegin <= e; its slot
// comes from the block table as in slot mapping ("vLLM 推理流程分析" §5.1.2),
// and its row is stored as pa_write_kv / pa_write_kv_fp8 store it (§6.3).
// One thread per 16-byte output chunk.
__global__ void write_runs_kernel(WriteParams p) {
    dev::grid_launch_dependents();
    dev::grid_dep_wait();
    // runs [r0, nruns) and their tokens [e0, ntok)
    int32_t r0 = 0, nruns = p.counts[kCountWriteRuns];
    int64_t e0 = 0, ntok = p.counts[kCountWriteTokens];
    if (p.part == 1) {
        nruns = p.counts[kCountWriteRunsEarly];
        ntok = p.counts[kCountWriteTokensEarly];
    } else if (p.part == 2) {
        r0 = p.counts[kCountWriteRunsEarly];
        e0 = p.counts[kCountWriteTokensEarly];
    }
    const int32_t cpr = p.kv8 ? p.row_elems / 16 : p.row_elems / 8;   // output chunks per row
    const int64_t total = (ntok - e0) * cpr;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int32_t e = static_cast<int32_t>(e0 + i / cpr);
        const int32_t c = static_cast<int32_t>(i % cpr);
        int32_t lo = r0, hi = nruns - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (p.runs[mid].wbegin <= e) lo = mid; else hi = mid - 1;
        }
        const WriteRun run = p.runs[lo];
        const int32_t t = run.t0 + (e - run.wbegin);
        const int32_t pos = run.pos0 + (e - run.wbegin);
        // the source chunks do not depend on the block id: load them first,
        // so that they and the block-table read share one round trip
        const uint4 *k = reinterpret_cast<const uint4 *>(p.key) + static_cast<int64_t>(t) * (p.row_elems / 8);
        const uint4 *v = reinterpret_cast<const uint4 *>(p.value) + static_cast<int64_t>(t) * (p.row_elems / 8);
        const int32_t sc = p.kv8 ? 2 * c : c;
        const uint4 k0 = __ldcs(k + sc), v0 = __ldcs(v + sc);
        uint4 k1 = make_uint4(0, 0, 0, 0), v1 = k1;
        if (p.kv8) {
            k1 = __ldcs(k + sc + 1);
            v1 = __ldcs(v + sc + 1);
        }
        const int32_t blk = p.block_table[static_cast<int64_t>(run.req) * p.max_blocks + pos / kBlockSize];
        if (blk < 0 || blk >= p.num_blocks) {
            if (c == 0) atomicOr(p.err, kErrBlockRange);
            continue;
        }
        const int64_t slot = static_cast<int64_t>(blk) * kBlockSize + pos % kBlockSize;
        if (c == 0 && p.slots_out != nullptr) p.slots_out[t] = slot;
        uint4 *kd = static_cast<uint4 *>(p.key_cache) + slot * cpr + c;
        uint4 *vd = static_cast<uint4 *>(p.value_cache) + slot * cpr + c;
        if (p.kv8) {
            *kd = quantize16(k0, k1, p.k_scale);
            *vd = quantize16(v0, v1, p.v_scale);
        } else {
            *kd = k0;
            *vd = v0;
        }
    }
}

// Metadata upload: the plan's pinned host image, read across the host link
// by the SMs themselves (no copy-engine round trip), into the workspace.
// Uncached loads: a recycled host buffer must never be served from a line
// cached for an earlier plan.
__global__ void upload_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int64_t n16) {
    dev::grid_launch_dependents();   // the next kernel may start its prologue (it waits for this one)
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) {
        uint4 v;
        asm volatile("ld.global.cv.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "l"(src + i));
        dst[i] = v;
    }
}

// Zeroing of newly allocated blocks ("vLLM 推理流程分析" §4 new_block_ids_to_zero,
// §5.1.1 _zero_block_ids): one CTA per listed id, 16-byte stores over the
// block's K and V bytes.
__global__ void zero_blocks_kernel(const int32_t *__restrict__ ids, int32_t num_blocks, int64_t chunks,
                                   uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache, int32_t *err) {
    const int32_t b = ids[blockIdx.x];
    if (b < 0) return;
    if (b >= num_blocks) {
        if (err != nullptr && threadIdx.x == 0) atomicOr(err, kErrBlockRange);
        return;
    }
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x) {
        key_cache[b * chunks + c] = z;
        value_cache[b * chunks + c] = z;
    }
}

// Merge of partition partials (page "vLLM 源码完全拆解（十六）", third
// walk-through: per-partition (m_r, l_r, o_r) combined with exponential
// rescaling).  One warp per (token, query head); m is in log2 units.
template <int D>
__global__ void merge_kernel(MergeParams p) {
    dev::grid_launch_dependents();
    dev::grid_dep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t total = static_cast<int64_t>(p.counts[kCountMerges]) * p.max_heads;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x / 32;
    for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < total; w += stride) {
        const MergeRow row = p.rows[w / p.max_heads];
        const int hi = static_cast<int>(w % p.max_heads);
        if (hi >= row.hq_count) continue;
        dev::merge_head<D>(p.out + static_cast<int64_t>(row.token) * p.num_heads_q * D, p.o_part, p.ml_part,
                           row.slot0, row.count, p.num_heads_q, row.hq_begin + hi, lane);
    }
}

}  // namespace

cudaError_t launch_slot_mapping(const int32_t *qsl, const int32_t *num_computed,
                                const int32_t *block_table, int32_t num_reqs, int32_t num_tokens,
                                int32_t max_blocks, int32_t block_size, int64_t *slots,
                                cudaStream_t stream) {
    if (num_tokens <= 0) return cudaSuccess;
    const int threads = 256;
    const int blocks = (num_tokens + threads - 1) / threads;
    slot_mapping_kernel<<<blocks, threads, 0, stream>>>(qsl, num_computed, block_table, num_reqs,
                                                        num_tokens, max_blocks, block_size, slots);
    return cudaGetLastError();
}

cudaError_t launch_write_kv(const void *key, const void *value, const int64_t *slots,
                            int32_t num_tokens, int32_t row_elems, void *key_cache,
                            void *value_cache, int64_t num_slots, int32_t *err,
                            cudaStream_t stream) {
    if (num_tokens <= 0) return cudaSuccess;
    const int32_t chunks_per_row = row_elems * 2 / 16;
    const int64_t total = static_cast<int64_t>(num_tokens) * chunks_per_row;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 152 * 16) blocks = 152 * 16;  // grid-stride beyond ~16 waves of CTAs
    write_kv_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value), slots, total,
        chunks_per_row, static_cast<uint4 *>(key_cache), static_cast<uint4 *>(value_cache),
        num_slots, err);
    return cudaGetLastError();
}

cudaError_t launch_write_kv_fp8(const void *key, const void *value, const int64_t *slots, int32_t num_tokens,
                                int32_t row_elems, void *key_cache, void *value_cache, int64_t num_slots,
                                float k_scale, float v_scale, int32_t *err, cudaStream_t stream) {
    if (num_tokens <= 0) return cudaSuccess;
    const int32_t chunks_per_row = row_elems / 16;        // 16 codes per output chunk
    const int64_t total = static_cast<int64_t>(num_tokens) * chunks_per_row;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    write_kv_fp8_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value), slots, total, chunks_per_row,
        static_cast<uint4 *>(key_cache), static_cast<uint4 *>(value_cache), num_slots, k_scale, v_scale, err);
    return cudaGetLastError();
}

cudaError_t launch_dequant(int grid, const DequantParams &p, cudaStream_t stream, bool pdl) {
    if (grid <= 0) return cudaSuccess;
    return launch_ex(dequant_kernel, dim3(grid), dim3(256), 0, stream, pdl, p);
}

cudaError_t launch_merge(int head_dim, int grid, const MergeParams &p, cudaStream_t stream, bool pdl) {
    if (grid <= 0) return cudaSuccess;
    if (head_dim == 128) return launch_ex(merge_kernel<128>, dim3(grid), dim3(256), 0, stream, pdl, p);
    if (head_dim == 64) return launch_ex(merge_kernel<64>, dim3(grid), dim3(256), 0, stream, pdl, p);
    return cudaErrorInvalidValue;
}

cudaError_t launch_upload(const void *src, void *dst, size_t bytes, cudaStream_t stream) {
    if (bytes == 0) return cudaSuccess;
    if (bytes % 16 != 0) return cudaErrorInvalidValue;
    const int64_t n16 = static_cast<int64_t>(bytes / 16);
    const int threads = 256;
    int64_t blocks = (n16 + threads - 1) / threads;
    if (blocks > 64) blocks = 64;
    upload_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(static_cast<const uint4 *>(src),
                                                                        static_cast<uint4 *>(dst), n16);
    return cudaGetLastError();
}

cudaError_t launch_write_runs(int grid, const WriteParams &p, cudaStream_t stream, bool pdl) {
    if (grid <= 0) return cudaSuccess;
    return launch_ex(write_runs_kernel, dim3(grid), dim3(256), 0, stream, pdl, p);
}

cudaError_t launch_zero_blocks(const int32_t *ids, int32_t num_ids, int32_t num_blocks, int64_t block_bytes,
                               void *key_cache, void *value_cache, int32_t *err, cudaStream_t stream) {
    if (num_ids <= 0) return cudaSuccess;
    zero_blocks_kernel<<<num_ids, 256, 0, stream>>>(ids, num_blocks, block_bytes / 16,
                                                    static_cast<uint4 *>(key_cache),
                                                    static_cast<uint4 *>(value_cache), err);
    return cudaGetLastError();
}

}  // namespace pa
