// Internal work-list records shared by the host planner and the kernels.
// Everything here is plain old data: the planner fills host arrays of these,
// pa_attention copies them into the workspace, the kernels read them there.
#pragma once
#include <utility>
#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace pa {

constexpr int kBlockSize = 16;     // tokens per cache block
constexpr int kTileKeys = 128;     // keys per tensor-core tile (8 blocks)
constexpr int kTileRows = 128;     // query rows per tensor-core sub-tile (two per CTA)
constexpr int kMaxDecodeHeads = 8; // kv heads one decode CTA serves
constexpr int kMmaRows = 16;       // rows of one decode MMA tile: (query token, head) pairs
constexpr int kMaxSmallQ = 8;      // longest row (query tokens) the decode kernel takes

// Split-KV decode kernel resources, shared by the planner (which sizes the
// persistent grid without touching a device) and the kernel.  kv8: E4M3
// caches (one byte per element).
constexpr int decode_stage_bytes(int d, int hg, bool kv8) { return 2 * hg * 16 * d * (kv8 ? 1 : 2); }
constexpr int decode_stages(int d, int hg, bool kv8) {
    return kv8 ? (200 * 1024 / decode_stage_bytes(d, hg, kv8) > 6 ? 6 : 200 * 1024 / decode_stage_bytes(d, hg, kv8))
               : (decode_stage_bytes(d, hg, kv8) * 4 <= 200 * 1024   ? 4
                  : decode_stage_bytes(d, hg, kv8) * 3 <= 200 * 1024 ? 3
                                                                       : 2);
}
constexpr int decode_threads(int hg) { return (hg + 1) * 32; }
// stages, their full_k / full_v / empty barriers and the fused update's
// row_ready barrier, plus 1024-byte alignment slack
constexpr int decode_smem_bytes(int d, int hg, bool kv8) {
    return decode_stages(d, hg, kv8) * decode_stage_bytes(d, hg, kv8) + (3 * decode_stages(d, hg, kv8) + 1) * 8 +
           1024;
}
constexpr int kSmemPerSm = 233472;  // 228 KiB of shared memory per SM
constexpr int decode_ctas_per_sm_static(int d, int hg, bool kv8) {
    return (kSmemPerSm / (decode_smem_bytes(d, hg, kv8) + 1024)) < (2048 / decode_threads(hg))
               ? (kSmemPerSm / (decode_smem_bytes(d, hg, kv8) + 1024))
               : (2048 / decode_threads(hg));
}

// Device error word bits (mirrors PA_DEVERR_* of pa.h).
constexpr int kErrSlotRange = 0x1;
constexpr int kErrBlockRange = 0x2;
constexpr int kErrTimeout = 0x4;

// One contiguous run of one request's key blocks for one group of kv heads,
// processed by one persistent CTA of the split-KV decode kernel.
struct DecodeItem {
    int32_t token;       // query row (q / out row)
    int32_t req;         // block-table row
    int32_t page_begin;  // first logical block of the run
    int32_t page_end;    // one past the last logical block of the run
    int32_t key_end;     // keys >= key_end are masked (one past the last token's position)
    int32_t head_group;  // kv heads [head_group*HG, head_group*HG + HG)
    int32_t part;        // partial index of this run (-1: write bf16 output)
    int32_t n_tok;       // query tokens token .. token + n_tok - 1 (n_tok * G <= 16); token i
                         // sees keys < key_end - (n_tok - 1 - i)
};

// One CTA tile of up to 256 query rows (2 x 128/G consecutive tokens x the
// G query heads of one kv head) against the key range [key_begin, key_end)
// of one request's context.
struct ExtendTile {
    int32_t t0;          // first token of the tile
    int32_t n_tok;       // tokens of the tile that belong to it (<= 256/G)
    int32_t req;         // block-table row the keys are read through
    int32_t pos0;        // absolute position of token t0 (causal bound)
    int32_t key_begin;   // block aligned
    int32_t key_end;
    int32_t kv_head;
    int32_t part;        // partial index (-1: write bf16 output)
    int32_t causal;      // 0: every key of the range is visible (shared prefix)
    int32_t pad[3];
};

// The query heads [hq_begin, hq_begin + hq_count) of one token whose output
// is the merge of `count` partial results starting at partial slot `slot0`.
struct MergeRow {
    int32_t token;
    int32_t slot0;
    int32_t count;
    int32_t hq_begin;
    int32_t hq_count;
    int32_t pad[3];
};

// Layout of the workspace:
//   [0, 256)            error word and reserved
//   meta blob           part_offset[T] | cta_begin[ncta+1] | DecodeItem[] |
//                       ExtendTile[] | MergeRow[]        (each 16-byte aligned)
//   o_part              float [num_slots][Hq][D]
//   ml_part             float2 [num_slots][Hq]  (log2-domain max, sum)
struct DecodeParams {
    const uint16_t *q;
    uint16_t *out;
    const int32_t *block_table;
    const DecodeItem *items;
    const int32_t *cta_begin;   // [gridDim.x + 1] item ranges per CTA
    const int32_t *part_offset; // [T][n_groups] first partial slot of (token, head group)
    float *o_part;
    float2 *ml_part;
    int32_t *err;
    int32_t max_blocks;
    int32_t num_blocks;
    int32_t num_heads_q;
    int32_t group;              // G = Hq / Hkv
    int32_t n_groups;           // kv-head groups (Hkv / heads per group)
    float scale_log2;           // softmax_scale * k_scale * log2(e)
    float out_scale;            // v_scale (1 for bf16 caches)
    // fused cache update (new_k != null): the CTA holding a decode row's last
    // page stores the row's new K/V into the caches and into its stage
    const uint16_t *new_k;      // [T][Hkv][D] bf16
    const uint16_t *new_v;
    void *cache_k;
    void *cache_v;
    int64_t *slots_out;         // optional [T]
    int32_t num_heads_kv;
    float k_scale, v_scale;     // E4M3 quantisation scales of the write
};

struct ExtendParams {
    uint16_t *out;
    const int32_t *block_table;
    const ExtendTile *tiles;
    const int32_t *part_offset;
    float *o_part;
    float2 *ml_part;
    int32_t *err;
    const int32_t *cta_tile_begin;  // [grid + 1]: CTA c runs tiles cta_tiles[begin[c] .. begin[c+1])
    const int32_t *cta_tiles;       // tile indices, each CTA's longest first
    int32_t max_blocks;
    int32_t num_blocks;
    int32_t num_heads_q;
    int32_t group;
    int32_t n_groups;
    int32_t heads_per_group;    // kv heads per head group (indexes part_offset)
    float scale_log2;           // softmax_scale * k_scale * log2(e)
    float out_scale;            // v_scale (1 for bf16 caches)
};

// FP8 caches: one cache block the tensor-core tiles read, expanded to bf16.
struct DequantItem {
    int32_t req;                // block-table row of the source block
    int32_t block;              // logical block index in that row
    int32_t dst;                // block index in the bf16 scratch caches
    int32_t pad;
};

struct DequantParams {
    const uint8_t *key_cache;   // E4M3 caches
    const uint8_t *value_cache;
    uint16_t *key_out;          // bf16 scratch caches [n_dst][16][Hkv][D]
    uint16_t *value_out;
    const int32_t *block_table;
    const DequantItem *items;
    int32_t *err;
    const int32_t *counts;      // device work counts (MetaCounts)
    int32_t max_blocks;
    int32_t num_blocks;
    int32_t block_elems;        // 16 * Hkv * D
};

struct MergeParams {
    uint16_t *out;
    const MergeRow *rows;
    const float *o_part;
    const float2 *ml_part;
    const int32_t *counts;      // device work counts (MetaCounts)
    int32_t num_heads_q;
    int32_t max_heads;          // largest hq_count of any row
};

// Work counts at the head of the uploaded metadata: kernels launched on a
// grid sized for a capacity read their real counts here.
enum MetaCount : int {
    kCountTiles = 0,
    kCountMerges = 1,
    kCountDequant = 2,
    kCountTokens = 3,
    kCountWriteRuns = 4,     // extend rows whose new K/V the fused write kernel stores
    kCountWriteTokens = 5,   // their tokens in total
    kCountWriteRunsEarly = 6,    // leading runs: the small rows' (read by the decode stream)
    kCountWriteTokensEarly = 7,  // their tokens
    kNumCounts = 8
};

// Fused cache update: the new tokens of one small or extend row, stored by
// the write kernel before the decode stream or the tensor-core tiles read
// them (one-token decode rows are stored by the decode kernel itself).  The
// small rows' runs come first.
struct WriteRun {
    int32_t t0;          // first token row
    int32_t n_tok;       // tokens
    int32_t req;         // block-table row
    int32_t pos0;        // position of the first token (num_computed)
    int32_t wbegin;      // tokens of the runs before this one
    int32_t pad[3];
};

// The fused write of extend-row tokens (pa_attention_with_kv_update).
struct WriteParams {
    const uint16_t *key;        // [T][Hkv][D] bf16
    const uint16_t *value;
    void *key_cache;            // bf16 or E4M3 caches
    void *value_cache;
    const int32_t *block_table;
    const WriteRun *runs;
    const int32_t *counts;
    int64_t *slots_out;         // optional [T]
    int32_t *err;
    int32_t row_elems;          // Hkv * D
    int32_t max_blocks;
    int32_t num_blocks;
    int32_t kv8;
    float k_scale, v_scale;     // E4M3 quantisation (code of x / scale)
    int32_t part;               // runs to store: 0 all, 1 the early ones, 2 the rest
};

// Launch with programmatic stream serialisation when `pdl` (the kernel calls
// grid_dep_wait before touching data of earlier kernels, which is a no-op for
// a plain launch).  Plain launches follow a wait on another stream's event.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             bool pdl, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args &&...args) {
    return launch_ex(kernel, grid, block, smem, stream, true, std::forward<Args>(args)...);
}

// Launchers (each returns the launch's cudaError_t).
cudaError_t launch_slot_mapping(const int32_t *qsl, const int32_t *num_computed,
                                const int32_t *block_table, int32_t num_reqs, int32_t num_tokens,
                                int32_t max_blocks, int32_t block_size, int64_t *slots,
                                cudaStream_t stream);
cudaError_t launch_write_kv(const void *key, const void *value, const int64_t *slots,
                            int32_t num_tokens, int32_t row_elems, void *key_cache,
                            void *value_cache, int64_t num_slots, int32_t *err,
                            cudaStream_t stream);
cudaError_t launch_write_kv_fp8(const void *key, const void *value, const int64_t *slots, int32_t num_tokens,
                                int32_t row_elems, void *key_cache, void *value_cache, int64_t num_slots,
                                float k_scale, float v_scale, int32_t *err, cudaStream_t stream);
// The grid-sized launchers take the CTA count to launch; kernels read their
// real work counts from the device (MetaCount), so a grid sized for a
// capacity is as correct as an exact one.
cudaError_t launch_dequant(int grid, const DequantParams &p, cudaStream_t stream, bool pdl = true);
// Decode kernel: head_dim D, heads per CTA hg, E4M3 caches (kv8).  Returns
// cudaErrorInvalidValue for an unsupported combination.
cudaError_t launch_decode(int head_dim, int hg, bool kv8, int num_ctas, const CUtensorMap &tm_k,
                          const CUtensorMap &tm_v, const DecodeParams &p, cudaStream_t stream);
cudaError_t launch_extend(int head_dim, int grid, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                          const CUtensorMap &tm_v, const ExtendParams &p, cudaStream_t stream, bool pdl = true);
cudaError_t launch_merge(int head_dim, int grid, const MergeParams &p, cudaStream_t stream, bool pdl = true);
// Copy `bytes` (a multiple of 16) from device-accessible pinned host memory
// to device memory with a kernel.
cudaError_t launch_upload(const void *src, void *dst, size_t bytes, cudaStream_t stream);
// Fused write of extend-row tokens: grid-stride over their 16-element chunks.
cudaError_t launch_write_runs(int grid, const WriteParams &p, cudaStream_t stream, bool pdl = true);
// Zero the K and V entries of the listed blocks (ids < 0 skipped).
cudaError_t launch_zero_blocks(const int32_t *ids, int32_t num_ids, int32_t num_blocks, int64_t block_bytes,
                               void *key_cache, void *value_cache, int32_t *err, cudaStream_t stream);
// One-time per-process kernel attributes (dynamic shared memory sizes) of the
// kernels a plan launches, so that later launches can be captured.
cudaError_t prepare_decode(int head_dim, int hg, bool kv8);
cudaError_t prepare_extend(int head_dim);

}  // namespace pa
