// The plan object behind the opaque pa_plan_t of pa.h (host only), and the
// host helpers the entry points share.
#pragma once
#include <mutex>
#include <vector>

#include "../../include/pa.h"
#include "pa_internal.h"

struct pa_plan_s {
    // step shape
    int32_t R = 0, Hq = 0, Hkv = 0, D = 0, num_blocks = 0, max_blocks = 0;
    int32_t T = 0, G = 0, HG = 1, n_groups = 1, num_sms = 0;
    int32_t n_prefix = 0;         // num_common_prefix_blocks (cascade when > 0)
    int32_t prefix_req = -1;      // block-table row of the shared prefix
    int32_t prefix_splits = 0;
    float scale_log2 = 0.f;     // softmax_scale * k_scale * log2(e)
    bool kv8 = false;           // E4M3 caches
    float out_scale = 1.f;      // v_scale for E4M3 caches
    float k_scale = 1.f, v_scale = 1.f;   // E4M3 quantisation scales of the fused write
    // work lists
    std::vector<int32_t> part_offset;   // [T * n_groups]
    std::vector<int32_t> cta_begin;     // [ncta + 1]
    std::vector<pa::DecodeItem> items;
    std::vector<pa::ExtendTile> tiles;
    std::vector<pa::MergeRow> merges;
    std::vector<int32_t> cta_tile_begin;      // persistent tensor-core CTAs: [ext_ctas + 1]
    std::vector<int32_t> cta_tiles;           // their tile lists
    int32_t ext_ctas = 0;                     // grid of the tensor-core kernel
    bool fork = false;                        // tiles on a second stream, beside the decode kernel
    std::vector<pa::WriteRun> write_runs;     // small, then extend rows (fused cache update)
    int32_t write_tokens = 0;
    int32_t decode_prefix = 0;                // fixed shapes: decode-stream rows lie below it (0: no bound)
    int32_t write_runs_early = 0;             // leading runs: the small rows' (the decode stream reads them)
    int32_t write_tokens_early = 0;           // and their tokens
    std::vector<int32_t> scratch_table;       // E4M3: [rows][max_blocks] bf16 scratch block ids
    std::vector<pa::DequantItem> dequant;     // E4M3: blocks to expand each call
    int32_t num_scratch_blocks = 0;
    int32_t num_slots = 0;
    // workspace layout
    size_t off_part = 0, off_cta = 0, off_items = 0, off_tiles = 0, off_merges = 0;
    size_t off_scrtab = 0, off_dequant = 0, off_kscr = 0, off_vscr = 0, off_runs = 0;
    size_t off_ctb = 0, off_ctiles = 0;
    size_t blob_bytes = 0, off_opart = 0, off_ml = 0, ws_bytes = 0;
    // launch shape: exact sizes for pa_plan, capacities for pa_plan_fixed
    bool fixed = false;
    int32_t ncta = 0;                   // decode CTAs
    int32_t cap_tokens = 0, cap_items = 0, cap_tiles = 0, cap_merges = 0, cap_dequant = 0;
    int32_t cap_slots = 0, cap_scr_rows = 0, cap_runs = 0;
    bool prepared = false;              // kernel attributes set (pa_upload_metadata)
    std::vector<uint8_t> blob;          // host image of the metadata blob
    void *pinned = nullptr;             // pinned staging copy used for async uploads
    void *pinned_dev = nullptr;         // its device-side address (read by the upload kernel)
    size_t pinned_cap = 0;
    cudaEvent_t upload_evt = nullptr;   // recorded after each upload from `pinned`
    pa_plan_info info{};
    // timing
    bool timing = false;
    std::vector<cudaEvent_t> ev_start[4], ev_stop[4];
    std::mutex mu;
};

namespace pa {

constexpr size_t kWorkspaceHeader = 256;  // error word + reserved, then the metadata blob

// 3-D bf16 tensor map over [outer][mid][D] with a box of [box_outer][box_mid][64]
// and 128-byte swizzling (false if the driver entry point is unavailable or
// the encoding is rejected).
bool make_map(CUtensorMap *tm, const void *ptr, uint64_t d, uint64_t mid, uint64_t outer, uint32_t box_mid,
              uint32_t box_outer);

// Enqueue every kernel of one attention call on `stream`; the metadata blob
// must already be (or be about to be, in stream order) at ws + header.
// `timed` records the plan's per-kernel timing events when they are enabled.
// For a fixed-shape plan every launch and argument depends on the plan's
// capacities only.
// Fused cache update (pa_attention_with_kv_update): the step's new rows.
struct KvUpdate {
    const void *key = nullptr;      // [T][Hkv][D] bf16; null = no update
    const void *value = nullptr;
    int64_t *slots_out = nullptr;   // optional [T]
    // staged inputs: rows from P->decode_prefix on are complete once this
    // event fires; their cache write and the tiles wait for it on the side
    // stream (null: every input is complete in stream order)
    cudaEvent_t late_rows = nullptr;
    cudaEvent_t late_out_ready = nullptr;   // optional: recorded once out rows from the prefix on are final
};

// allow_fork = false keeps every launch on `stream` (a plan whose tiles run
// side by side with the decode kernel then runs them one after the other,
// with the same work cut and the same results).
pa_status enqueue_attention(pa_plan_s *P, const void *q, const void *key_cache, const void *value_cache,
                            const int32_t *block_table, void *out, uint8_t *ws, cudaStream_t stream, bool timed,
                            const KvUpdate &update = KvUpdate{}, bool allow_fork = true);

// The second stream (and its fork / join events) of this host thread on the
// current device, created on first use; null if creation fails.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
SideStream *side_stream();

// Set the kernel attributes the plan's launches need (once per plan).
pa_status prepare_plan(pa_plan_s *P);

}  // namespace pa
