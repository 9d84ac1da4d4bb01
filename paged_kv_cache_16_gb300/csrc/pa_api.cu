// C ABI of the paged-KV step: metadata validation and planning (host), and
// the enqueueing of the device kernels.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <queue>
#include <new>
#include <vector>

#include <cudaTypedefs.h>

#include "../../include/pa.h"
#include "plan.h"

using namespace pa;

namespace pa {

// cuTensorMapEncodeTiled from the driver, fetched once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D bf16 tensor map over [outer][mid][D] with a box of [box_outer][box_mid][64]
// and 128-byte swizzling.
bool make_map(CUtensorMap *tm, const void *ptr, uint64_t d, uint64_t mid, uint64_t outer,
              uint32_t box_mid, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {d, mid, outer};
    cuuint64_t strides[2] = {d * 2, mid * d * 2};
    cuuint32_t box[3] = {64, box_mid, box_outer};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor map of a paged cache for the decode stream: dimensions (element,
// row, kv head) over [rows][Hkv][D], box [box_heads][16 rows][128 bytes].  One
// box brings the 16 rows of a block for box_heads kv heads, each head's rows
// a contiguous, 128-byte-swizzled [16][128 B] tile in shared memory.
bool make_map_kv(CUtensorMap *tm, const void *ptr, uint64_t d, uint64_t hkv, uint64_t rows, uint32_t box_heads,
                 bool u8) {
    auto fn = encode_fn();
    if (!fn) return false;
    const uint64_t es = u8 ? 1 : 2;
    cuuint64_t dims[3] = {d, rows, hkv};
    cuuint64_t strides[2] = {hkv * d * es, d * es};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(kBlockSize), box_heads};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(tm, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr),
                    dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace pa

namespace {

constexpr size_t kHeader = kWorkspaceHeader;

// Pinned staging buffers for the per-call metadata upload, recycled across
// plans.  A plan takes a buffer on its first pa_attention call and hands it
// back when destroyed; the buffer is given out again only after the last copy
// from it has completed on the device (its event has fired), so destroying a
// plan never waits and never frees pinned memory on the hot path.
class StagingPool {
  public:
    bool acquire(size_t bytes, void **ptr, size_t *cap, cudaEvent_t *ev) {
        std::lock_guard<std::mutex> lock(mu_);
        for (size_t i = 0; i < free_.size(); ++i) {
            if (free_[i].cap >= bytes && cudaEventQuery(free_[i].ev) == cudaSuccess) {
                *ptr = free_[i].ptr;
                *cap = free_[i].cap;
                *ev = free_[i].ev;
                free_.erase(free_.begin() + static_cast<long>(i));
                return true;
            }
        }
        const size_t rounded = align(bytes, size_t(64) << 10);
        if (cudaMallocHost(ptr, rounded) != cudaSuccess) return false;
        if (cudaEventCreateWithFlags(ev, cudaEventDisableTiming) != cudaSuccess) {
            cudaFreeHost(*ptr);
            return false;
        }
        *cap = rounded;
        return true;
    }
    void release(void *ptr, size_t cap, cudaEvent_t ev) {
        std::lock_guard<std::mutex> lock(mu_);
        free_.push_back({ptr, cap, ev});
        if (free_.size() > kMaxFree) {  // bound the pool: retire the oldest
            Buf old = free_.front();
            free_.erase(free_.begin());
            cudaEventSynchronize(old.ev);
            cudaEventDestroy(old.ev);
            cudaFreeHost(old.ptr);
        }
    }

  private:
    struct Buf {
        void *ptr;
        size_t cap;
        cudaEvent_t ev;
    };
    static size_t align(size_t x, size_t a) { return (x + a - 1) / a * a; }
    static constexpr size_t kMaxFree = 32;
    std::mutex mu_;
    std::vector<Buf> free_;
};

StagingPool &staging() {
    static StagingPool *pool = new StagingPool();  // never destroyed: outlives CUDA teardown
    return *pool;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }


int heads_per_group(int hkv) {
    for (int hg = kMaxDecodeHeads; hg > 1; hg >>= 1)
        if (hkv % hg == 0) return hg;
    return 1;
}

pa_status validate(const pa_batch_desc *d) {
    if (d->num_reqs < 0 || d->num_heads_q <= 0 || d->num_heads_kv <= 0 || d->num_blocks <= 0 ||
        d->max_blocks_per_req <= 0 || d->block_size <= 0 || d->head_dim <= 0)
        return PA_ERR_INVALID_ARGUMENT;
    if (d->num_heads_q % d->num_heads_kv != 0) return PA_ERR_INVALID_ARGUMENT;
    if (!(d->softmax_scale > 0.f) || !std::isfinite(d->softmax_scale)) return PA_ERR_INVALID_ARGUMENT;
    if (d->num_common_prefix_blocks < 0 || d->num_sms < 0) return PA_ERR_INVALID_ARGUMENT;
    if (d->query_start_loc == nullptr || (d->num_reqs > 0 && (d->seq_lens == nullptr ||
                                                              d->num_computed_tokens == nullptr)))
        return PA_ERR_INVALID_ARGUMENT;
    const int32_t *qsl = d->query_start_loc;
    if (qsl[0] != 0) return PA_ERR_INVALID_ARGUMENT;
    for (int32_t r = 0; r < d->num_reqs; ++r) {
        const int64_t q_len = static_cast<int64_t>(qsl[r + 1]) - qsl[r];
        if (q_len < 0) return PA_ERR_INVALID_ARGUMENT;
        if (d->seq_lens[r] < 0 || d->num_computed_tokens[r] < 0) return PA_ERR_INVALID_ARGUMENT;
        if (static_cast<int64_t>(d->num_computed_tokens[r]) + q_len != d->seq_lens[r])
            return PA_ERR_INVALID_ARGUMENT;
        const int64_t need = (static_cast<int64_t>(d->seq_lens[r]) + d->block_size - 1) / d->block_size;
        if (need > d->max_blocks_per_req) return PA_ERR_INVALID_ARGUMENT;
        if (d->block_table_host) {
            // one unsigned compare per id (negative ids wrap to large ones),
            // branch-free so that the compiler vectorises it
            const int32_t *row = d->block_table_host + static_cast<int64_t>(r) * d->max_blocks_per_req;
            const uint32_t nb = static_cast<uint32_t>(d->num_blocks);
            uint32_t bad = 0;
            for (int64_t b = 0; b < need; ++b) bad |= static_cast<uint32_t>(row[b]) >= nb ? 1u : 0u;
            if (bad) return PA_ERR_INVALID_ARGUMENT;
        }
    }
    const int32_t n = d->num_common_prefix_blocks;
    if (n > 0) {
        if (n > d->max_blocks_per_req) return PA_ERR_INVALID_ARGUMENT;
        int32_t ref = -1;
        for (int32_t r = 0; r < d->num_reqs; ++r) {
            if (qsl[r + 1] == qsl[r]) continue;
            if (static_cast<int64_t>(n) * d->block_size > d->num_computed_tokens[r]) return PA_ERR_INVALID_ARGUMENT;
            if (d->block_table_host) {
                if (ref < 0) {
                    ref = r;
                    continue;
                }
                const int32_t *a = d->block_table_host + static_cast<int64_t>(ref) * d->max_blocks_per_req;
                const int32_t *b = d->block_table_host + static_cast<int64_t>(r) * d->max_blocks_per_req;
                for (int32_t i = 0; i < n; ++i)
                    if (a[i] != b[i]) return PA_ERR_INVALID_ARGUMENT;
            }
        }
    }
    if (d->kv_cache_dtype != PA_KV_BF16 && d->kv_cache_dtype != PA_KV_FP8_E4M3) return PA_ERR_INVALID_ARGUMENT;
    if (d->kv_cache_dtype == PA_KV_FP8_E4M3 &&
        (!(d->k_scale > 0.f) || !std::isfinite(d->k_scale) || !(d->v_scale > 0.f) || !std::isfinite(d->v_scale)))
        return PA_ERR_INVALID_ARGUMENT;
    // supported shapes
    if (d->block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
    if (d->kv_cache_dtype == PA_KV_FP8_E4M3 && d->head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (d->head_dim != 64 && d->head_dim != 128) return PA_ERR_UNSUPPORTED;
    const int G = d->num_heads_q / d->num_heads_kv;
    if (G > kTileRows) return PA_ERR_UNSUPPORTED;   // a tensor-core sub-tile holds at least one token
    if (static_cast<int64_t>(d->num_blocks) * d->block_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

// A unit of the split-KV decode kernel: n_tok <= 16 / G consecutive query
// tokens of one request whose G heads fill the 16 rows of one MMA tile; the
// unit reads keys [0, key_end), key_end = one past its last token's position.
struct DecodeUnit {
    int32_t r, t0, n_tok, key_end;
};

// Cut the concatenated decode runs into ncta equal contiguous shares.
// pieces[u * n_groups + grp] receives the number of runs unit u was cut into;
// item_unit[i] the unit of item i.
// work_ctas: at most that many CTAs get work (0: num_sms x CTAs per SM).
// fixed_ncta > 0: the grid has exactly that many CTAs; the shares past the
// ones the work needs are empty.
// Decode cut costs in quarters of one block's streaming time.  The fixed
// cost of an item (about 1.3 us on GB300, fitted: 32-96 KB all cut the
// E4M3 decode workload's kernel time by 5-6% against an equal cut, 64 KB
// the most) is what one SM streams meanwhile when the whole GPU streams
// (about 45 GB/s per SM): 64 KB, 2 blocks of E4M3 codes for 8 kv heads of
// 128 dims.  It counts for E4M3 caches only,
// whose consumers run close to their per-SM limit (about 52 GB/s); a bf16
// SM streams twice what the HBM share needs and absorbs it (an item cost
// there made the decode workload 1.3% slower).
constexpr int64_t kPageCost = 4;
constexpr int64_t kItemBytes = 64 * 1024;

// Shortest cascade prefix tile, in 128-key steps.
constexpr int kMinPrefixSteps = 8;

void plan_decode(pa_plan_s *P, const std::vector<DecodeUnit> &units, std::vector<int32_t> &pieces,
                 std::vector<int32_t> &item_unit, int64_t work_ctas, int64_t fixed_ncta) {
    struct Run { int32_t u, grp, pb, pe; };
    std::vector<Run> runs;
    runs.reserve(units.size() * P->n_groups);
    const int32_t kb = P->n_prefix;  // first block of the suffix work
    int64_t total = 0;
    for (int grp = 0; grp < P->n_groups; ++grp)
        for (size_t u = 0; u < units.size(); ++u) {
            const int32_t pe = (units[u].key_end + kBlockSize - 1) / kBlockSize;
            if (pe <= kb) continue;
            runs.push_back({static_cast<int32_t>(u), grp, kb, pe});
            total += pe - kb;
        }
    pieces.assign(units.size() * P->n_groups, 0);
    item_unit.clear();
    P->cta_begin.assign(1, 0);
    if (total == 0) {
        if (fixed_ncta > 0) P->cta_begin.assign(static_cast<size_t>(fixed_ncta) + 1, 0);
        return;
    }
    const int cps = std::max(1, decode_ctas_per_sm_static(P->D, P->HG, P->kv8));
    const int64_t min_pages = 4;
    const int64_t cap = work_ctas > 0 ? work_ctas : static_cast<int64_t>(P->num_sms) * cps;
    int64_t ncta = std::min<int64_t>(cap, (total + min_pages - 1) / min_pages);
    ncta = std::max<int64_t>(ncta, 1);
    if (fixed_ncta > 0) ncta = std::min(ncta, fixed_ncta);
    // The cut is equal in cost, not in pages: an item costs its pages plus a
    // fixed start-up and finish (q loads, the fused row store, the epilogue),
    // so a CTA that holds the end of one run and the start of the next gets
    // fewer pages.  Costs are in quarter blocks.  Cutting a run at a CTA
    // boundary makes at most one item per run plus one per CTA.
    const int64_t page_bytes = 2LL * kBlockSize * P->HG * P->D * (P->kv8 ? 1 : 2);   // K and V
    const int64_t item_cost = P->kv8 ? (kPageCost * kItemBytes + page_bytes / 2) / page_bytes : 0;
    const int64_t total_cost =
        kPageCost * total + item_cost * (static_cast<int64_t>(runs.size()) + ncta - 1);
    P->items.reserve(runs.size() + static_cast<size_t>(ncta));
    item_unit.reserve(runs.size() + static_cast<size_t>(ncta));
    P->cta_begin.reserve(static_cast<size_t>(std::max(ncta, fixed_ncta)) + 1);
    size_t run = 0;
    int32_t cursor = runs.empty() ? 0 : runs[0].pb;
    int64_t spent = 0;   // cost given to the CTAs so far
    for (int64_t c = 0; c < ncta; ++c) {
        const bool last = c + 1 == ncta;
        const int64_t target = total_cost * (c + 1) / ncta;   // cumulative cost at this CTA's end
        while (run < runs.size()) {
            const Run &R = runs[run];
            const DecodeUnit &U = units[R.u];
            const int64_t room = last ? R.pe - cursor : (target - spent - item_cost) / kPageCost;   // pages
            if (room <= 0) break;
            const int32_t take = static_cast<int32_t>(std::min<int64_t>(room, R.pe - cursor));
            DecodeItem it{};
            it.token = U.t0;
            it.req = U.r;
            it.page_begin = cursor;
            it.page_end = cursor + take;
            it.key_end = U.key_end;
            it.head_group = R.grp;
            it.part = pieces[static_cast<size_t>(R.u) * P->n_groups + R.grp]++;
            it.n_tok = U.n_tok;
            P->items.push_back(it);
            item_unit.push_back(R.u);
            cursor += take;
            spent += item_cost + kPageCost * take;
            if (cursor >= R.pe) {
                ++run;
                if (run < runs.size()) cursor = runs[run].pb;
            }
        }
        P->cta_begin.push_back(static_cast<int32_t>(P->items.size()));
    }
    while (static_cast<int64_t>(P->cta_begin.size()) < fixed_ncta + 1)
        P->cta_begin.push_back(static_cast<int32_t>(P->items.size()));
}

// Step-time model used to split the SMs between the tensor-core tiles and
// the split-KV decode stream when a step has both (times in microseconds,
// constants measured on GB300 at full clock).  The tiles are bound by the
// tensor pipe of the SMs they run on, the decode stream by HBM once it has
// enough SMs (each SM streams about 90 GB/s of bf16 blocks, 52 GB/s of E4M3
// codes), so running the two side by side on disjoint SMs costs about
// the longer of the two instead of their sum.
// Side by side the two slow each other down a little (the tiles' K/V
// re-reads and the decode stream share L2 and HBM): the side constants below
// were measured that way.  With E4M3 caches the tile stream first makes the
// bf16 copies of the tiles' blocks (three bytes moved per code).
constexpr double kTileStepUs = 1.85;          // one 128-key step of a 256-row tile on one SM
constexpr double kTileStepSideUs = 2.15;      // the same beside the bf16 decode stream
constexpr double kTileStepSideFp8Us = 1.80;   // the same beside the E4M3 decode stream
constexpr double kDequantUsPerBlock = 0.05;   // bf16 copy of one E4M3 block (K and V, all kv heads)
constexpr double kHbmBytesPerUs = 7.0e6;      // decode stream at the HBM limit
constexpr double kHbmSideBytesPerUs = 6.7e6;  // the same beside the tiles
constexpr double kSmBf16BytesPerUs = 9.0e4;   // decode stream of one SM, bf16 caches
constexpr double kSmFp8BytesPerUs = 5.2e4;    // decode stream of one SM, E4M3 caches
constexpr double kForkUs = 5.0;               // cost of the second stream (fork, join, plain launches)
constexpr double kHostLinkBytesPerUs = 2.0e5;  // page-locked host <-> device copy (staged inputs)
// Share of the tiles' output copy-back counted on their path: the copy
// overlaps the decode stream's tail, so only part of it lengthens the step
// (mixed step from host memory to host memory: 1.018 / 0.997 / 1.059 ms
// for 0 / 0.25 / 0.5, 1.100 ms for all of it).
constexpr double kOutLeadWeight = 0.25;

struct StepModel {
    double tile_units = 0, tile_max = 0;      // sum and largest tile cost (128-key steps + 1)
    double decode_bytes = 0, sm_rate = 0;
    double side_step = kTileStepSideUs;       // tile step beside the decode stream
    double tile_lead = 0;                     // tile-stream work before the tiles (E4M3 copies)
    double tiles(int ctas, bool side) const {
        return ctas <= 0 ? 1e30
                         : tile_lead + std::max(tile_units / ctas, tile_max) * (side ? side_step : kTileStepUs);
    }
    double decode(int sms, bool side) const {
        return sms <= 0 ? 1e30
                        : std::max(decode_bytes / (sms * sm_rate),
                                   decode_bytes / (side ? kHbmSideBytesPerUs : kHbmBytesPerUs));
    }
};

// Extend CTAs for a step that runs tiles and decode side by side on
// num_sms SMs: the split with the shortest modelled step; among near-equal
// splits the one whose tiles finish with some slack before the decode
// stream (the model is a few percent off either way).
int split_sms(const StepModel &m, int num_sms, int max_tile_ctas, double *t_out) {
    const int hi = std::min(num_sms - 1, max_tile_ctas);
    double best = 1e30;
    int arg = 1;
    for (int e = 1; e <= hi; ++e) {
        const double t = std::max(m.tiles(e, true), m.decode(num_sms - e, true));
        if (t < best) { best = t; arg = e; }
    }
    for (int e = 1; e <= hi; ++e)
        if (m.tiles(e, true) <= 0.85 * best && m.decode(num_sms - e, true) <= 1.01 * best) { arg = e; break; }
    *t_out = best;
    return arg;
}

pa_status build_plan(pa_plan_s *P, const pa_batch_desc *d, const pa_fixed_shape *shape) {
    P->fixed = shape != nullptr;
    P->R = d->num_reqs;
    P->Hq = d->num_heads_q;
    P->Hkv = d->num_heads_kv;
    P->D = d->head_dim;
    P->num_blocks = d->num_blocks;
    P->max_blocks = d->max_blocks_per_req;
    P->T = d->num_reqs > 0 ? d->query_start_loc[d->num_reqs] : 0;
    P->G = P->Hq / P->Hkv;
    P->HG = heads_per_group(P->Hkv);
    P->n_groups = P->Hkv / P->HG;
    P->kv8 = d->kv_cache_dtype == PA_KV_FP8_E4M3;
    P->scale_log2 = d->softmax_scale * (P->kv8 ? d->k_scale : 1.f) * 1.4426950408889634f;
    P->out_scale = P->kv8 ? d->v_scale : 1.f;
    P->k_scale = P->kv8 ? d->k_scale : 1.f;
    P->v_scale = P->kv8 ? d->v_scale : 1.f;
    P->num_sms = d->num_sms;
    if (P->num_sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&P->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return PA_ERR_CUDA;
    }
    if (P->fixed && (P->T > shape->max_tokens || P->R > shape->max_reqs)) return PA_ERR_CAPACITY;
    const int32_t *qsl = d->query_start_loc;
    // q_len 1: decode rows.  2..kMaxSmallQ (speculative verify): on the
    // split-KV decode kernel when the row fits one 16-row unit, or when it
    // needs several units (each re-reads the row's keys) but the tensor-core
    // tiles of all such rows would not fill the GPU; else, and for longer
    // rows, tensor-core tiles.
    // A decode unit is one MMA tile of 16 (token, head) rows, so the decode
    // kernel takes groups of at most 16 query heads; larger groups (e.g. a
    // single kv head shared by 32 query heads) run every row on the tiles.
    const int32_t tg = std::max(1, kMmaRows / P->G);   // tokens per decode unit
    std::vector<int32_t> decode_rows, small_rows, extend_rows, multi_unit;
    decode_rows.reserve(static_cast<size_t>(P->R));
    for (int32_t r = 0; r < P->R; ++r) {
        const int32_t q_len = qsl[r + 1] - qsl[r];
        if (q_len > 0 && P->G > kMmaRows) extend_rows.push_back(r);
        else if (q_len == 1) decode_rows.push_back(r);
        else if (q_len > 1 && q_len <= tg) small_rows.push_back(r);
        else if (q_len > 1 && q_len <= kMaxSmallQ) multi_unit.push_back(r);
        else if (q_len > 1) extend_rows.push_back(r);
    }
    const bool multi_on_decode = static_cast<int64_t>(multi_unit.size()) * P->Hkv < P->num_sms;
    for (int32_t r : multi_unit) (multi_on_decode ? small_rows : extend_rows).push_back(r);
    std::sort(small_rows.begin(), small_rows.end());
    std::sort(extend_rows.begin(), extend_rows.end());
    std::vector<char> on_decode(static_cast<size_t>(P->R), 0);
    for (int32_t r : decode_rows) on_decode[r] = 1;
    for (int32_t r : small_rows) on_decode[r] = 1;
    const bool cascade = d->num_common_prefix_blocks > 0 && P->T > 0;
    P->n_prefix = cascade ? d->num_common_prefix_blocks : 0;
    const int32_t kb_keys = P->n_prefix * kBlockSize;
    for (int32_t r = 0; r < P->R; ++r)
        if (qsl[r + 1] > qsl[r]) { P->prefix_req = r; break; }

    // ---------------------------------------------------- tensor-core tiles
    const int tpt = 2 * (kTileRows / P->G);   // tokens per CTA tile: two 128-row sub-tiles
    if (cascade) {
        const int n_key_tiles = (kb_keys + kTileKeys - 1) / kTileKeys;
        const int token_tiles = (P->T + tpt - 1) / tpt;
        const int units = P->Hkv * token_tiles;
        // key splits: enough tiles to spread over the SMs, but none shorter
        // than kMinPrefixSteps key tiles, whose fixed cost (Q load, pipeline
        // fill, fp32 partial write) is worth several steps (cascade workload:
        // 4 splits of 8 steps 0.088 ms per step, 8 of 4 steps 0.102 ms)
        int splits = static_cast<int>(std::lround(static_cast<double>(P->num_sms) / units));
        splits = std::max(1, std::min({splits, n_key_tiles / kMinPrefixSteps, n_key_tiles}));
        const int chunk = (n_key_tiles + splits - 1) / splits;      // key tiles per split
        splits = (n_key_tiles + chunk - 1) / chunk;
        P->prefix_splits = splits;
        for (int h = 0; h < P->Hkv; ++h)
            for (int tt = 0; tt < token_tiles; ++tt)
                for (int s = 0; s < splits; ++s) {
                    ExtendTile t{};
                    t.t0 = tt * tpt;
                    t.n_tok = std::min(tpt, P->T - t.t0);
                    t.req = P->prefix_req;
                    t.pos0 = 0;
                    t.key_begin = s * chunk * kTileKeys;
                    t.key_end = std::min(kb_keys, (s + 1) * chunk * kTileKeys);
                    t.kv_head = h;
                    t.part = s;
                    t.causal = 0;
                    P->tiles.push_back(t);
                }
        P->info.num_prefix_tiles = static_cast<int32_t>(P->tiles.size());
    }
    {
        size_t n = P->tiles.size();
        for (int32_t r : extend_rows) n += static_cast<size_t>(P->Hkv) * ((qsl[r + 1] - qsl[r] + tpt - 1) / tpt);
        P->tiles.reserve(n);
    }
    for (int32_t r : extend_rows) {
        const int32_t q_len = qsl[r + 1] - qsl[r];
        for (int h = 0; h < P->Hkv; ++h)
            for (int32_t m0 = 0; m0 < q_len; m0 += tpt) {
                ExtendTile t{};
                t.t0 = qsl[r] + m0;
                t.n_tok = std::min(tpt, q_len - m0);
                t.req = r;
                t.pos0 = d->num_computed_tokens[r] + m0;
                t.key_begin = kb_keys;
                t.key_end = std::min(d->seq_lens[r], t.pos0 + t.n_tok);
                t.kv_head = h;
                t.part = cascade ? P->prefix_splits : -1;
                t.causal = 1;
                P->tiles.push_back(t);
            }
    }
    // longest key ranges first: the last wave is made of short tiles (a
    // stable order: keys (INT32_MAX - range, index) sorted, then one move)
    {
        std::vector<uint64_t> key(P->tiles.size());
        for (size_t i = 0; i < key.size(); ++i)
            key[i] = (static_cast<uint64_t>(INT32_MAX - (P->tiles[i].key_end - P->tiles[i].key_begin)) << 32) | i;
        std::sort(key.begin(), key.end());
        std::vector<ExtendTile> sorted(key.size());
        for (size_t i = 0; i < key.size(); ++i) sorted[i] = P->tiles[static_cast<uint32_t>(key[i])];
        P->tiles.swap(sorted);
    }

    // E4M3 caches: the tiles read bf16 copies of the blocks they touch, one
    // scratch block-table row per request the tiles read through
    if (P->kv8 && !P->tiles.empty()) {
        std::vector<int32_t> row_of(static_cast<size_t>(P->R), -1), lo, hi, reqs;
        for (const ExtendTile &t : P->tiles) {
            int32_t &row = row_of[t.req];
            if (row < 0) {
                row = static_cast<int32_t>(reqs.size());
                reqs.push_back(t.req);
                lo.push_back(INT32_MAX);
                hi.push_back(0);
            }
            lo[row] = std::min(lo[row], t.key_begin / kBlockSize);
            hi[row] = std::max(hi[row], (t.key_end + kBlockSize - 1) / kBlockSize);
        }
        P->scratch_table.assign(reqs.size() * static_cast<size_t>(P->max_blocks), 0);
        for (size_t row = 0; row < reqs.size(); ++row)
            for (int32_t b = lo[row]; b < hi[row]; ++b) {
                DequantItem di{};
                di.req = reqs[row];
                di.block = b;
                di.dst = P->num_scratch_blocks++;
                P->scratch_table[row * P->max_blocks + b] = di.dst;
                P->dequant.push_back(di);
            }
        for (ExtendTile &t : P->tiles) t.req = row_of[t.req];
    }

    // ------------------------------------------------------ decode units
    std::vector<DecodeUnit> units;
    units.reserve(decode_rows.size() + small_rows.size() * 2);
    for (int32_t r = 0; r < P->R; ++r) {
        const int32_t q_len = qsl[r + 1] - qsl[r];
        if (!on_decode[r]) continue;
        for (int32_t j = 0; j < q_len; j += tg) {
            const int32_t n = std::min(tg, q_len - j);
            units.push_back({r, qsl[r] + j, n, d->num_computed_tokens[r] + j + n});
        }
    }
    // staged inputs: the decode stream may read rows below the shape's
    // decode prefix only
    P->decode_prefix = P->fixed ? shape->decode_prefix_tokens : 0;
    if (P->decode_prefix > 0)
        for (const DecodeUnit &u : units)
            if (u.t0 + u.n_tok > P->decode_prefix) return PA_ERR_CAPACITY;
    const int cps = std::max(1, decode_ctas_per_sm_static(P->D, P->HG, P->kv8));

    // ------------------------------------------ tile costs and the SM split
    // cost of a tile: its 128-key steps (as the kernel counts them) plus one
    // for the Q load and epilogue
    std::vector<std::pair<int64_t, int32_t>> cost;
    cost.reserve(P->tiles.size());
    StepModel model;
    {
        const int tpt_rows = kTileRows / P->G;
        for (size_t i = 0; i < P->tiles.size(); ++i) {
            const ExtendTile &t = P->tiles[i];
            int n_tiles = 0;
            for (int sub = 0; sub < 2; ++sub) {
                const int first = sub * tpt_rows;
                if (first >= t.n_tok) continue;
                const int last = std::min(t.n_tok, first + tpt_rows);
                const int kend = t.causal ? std::min(t.key_end, t.pos0 + last) : t.key_end;
                n_tiles = std::max(n_tiles, (kend - t.key_begin + kTileKeys - 1) / kTileKeys);
            }
            cost.push_back({n_tiles + 1, static_cast<int32_t>(i)});
            model.tile_units += n_tiles + 1;
            model.tile_max = std::max<double>(model.tile_max, n_tiles + 1);
        }
        const int64_t row_bytes = static_cast<int64_t>(P->Hkv) * P->D * (P->kv8 ? 1 : 2) * 2;
        for (const DecodeUnit &u : units)
            model.decode_bytes += static_cast<double>(std::max(0, u.key_end - kb_keys)) * row_bytes;
        model.sm_rate = P->kv8 ? kSmFp8BytesPerUs : kSmBf16BytesPerUs;
        if (P->kv8) {
            model.side_step = kTileStepSideFp8Us;
            model.tile_lead = kDequantUsPerBlock * P->num_scratch_blocks;
        }
        // staged inputs: the tiles start once the rows from the decode prefix
        // on (q, key, value) have crossed the host link, and their output
        // rows cross it back after them
        if (P->decode_prefix > 0 && P->decode_prefix < P->T)
            model.tile_lead += static_cast<double>(P->T - P->decode_prefix) *
                               (P->Hq + 2 * P->Hkv + kOutLeadWeight * P->Hq) * P->D * 2 / kHostLinkBytesPerUs;
    }
    const int64_t n_tiles_all = static_cast<int64_t>(P->tiles.size());
    if (P->fixed && n_tiles_all > shape->max_extend_tiles) return PA_ERR_CAPACITY;
    const bool have_tiles = n_tiles_all > 0, have_decode = model.decode_bytes > 0;
    // grids: eager plans are sized by the work, fixed-shape plans by their
    // capacities (the decode grid is always num_sms x CTAs per SM)
    const int64_t tile_grid_cap = P->fixed ? std::min<int64_t>(shape->max_extend_tiles, P->num_sms)
                                           : std::min<int64_t>(n_tiles_all, P->num_sms);
    // The work cut: split the SMs when the model says running the two side
    // by side pays, else every CTA of both grids gets work.  The cut depends
    // on the step only, so a fixed-shape plan and a plain plan of the same
    // step cut (and compute) identically.  The launch topology: plain plans
    // put the tiles on a second stream exactly when the cut is split;
    // fixed-shape plans with tiles always do (their launches cannot depend on
    // the step), and an unsplit step then has both grids compete for the SMs.
    int64_t tile_work_ctas = std::min<int64_t>(n_tiles_all, P->num_sms);   // CTAs that get tiles
    int64_t decode_work_ctas = 0;                                           // 0: all
    bool split = false;
    if (have_tiles && have_decode && P->num_sms >= 2) {
        double t_split = 0;
        const int e = split_sms(model, P->num_sms, static_cast<int>(std::min<int64_t>(n_tiles_all, P->num_sms - 1)),
                                &t_split);
        const double t_seq = model.tiles(static_cast<int>(tile_work_ctas), false) + model.decode(P->num_sms, false);
        if (t_split + kForkUs < t_seq) {
            split = true;
            tile_work_ctas = e;
            decode_work_ctas = P->num_sms - e;
        }
    }
    P->fork = P->fixed ? shape->max_extend_tiles > 0 && P->num_sms >= 2 : split;
    P->ext_ctas = static_cast<int32_t>(std::max<int64_t>(P->fixed ? tile_grid_cap : tile_work_ctas, 0));
    P->info.num_extend_ctas = static_cast<int32_t>(have_tiles ? tile_work_ctas : 0);
    P->info.side_by_side = P->fork ? 1 : 0;

    // ------------------------------- persistent tensor-core CTAs (LPT)
    // each tile goes to the least loaded of the first tile_work_ctas CTAs,
    // longest tiles first; the grid's other CTAs get nothing
    {
        // counts per CTA, then the tiles in assignment order (a counting
        // sort: no per-CTA lists to grow)
        P->cta_tile_begin.assign(static_cast<size_t>(P->ext_ctas) + 1, 0);
        P->cta_tiles.clear();
        if (P->ext_ctas > 0 && have_tiles) {
            // costs in descending order, equal costs by index (stable)
            std::vector<uint64_t> order(cost.size());
            for (size_t k = 0; k < cost.size(); ++k)
                order[k] = (static_cast<uint64_t>(INT32_MAX - cost[k].first) << 32) | static_cast<uint32_t>(k);
            std::sort(order.begin(), order.end());
            // min-heap of (work so far, CTA) packed as work << 32 | CTA (the
            // work of all tiles, in steps, is far below 2^32)
            if (model.tile_units >= 4294967296.0) return PA_ERR_UNSUPPORTED;
            std::vector<uint64_t> heap(static_cast<size_t>(tile_work_ctas));
            for (int32_t c = 0; c < tile_work_ctas; ++c) heap[static_cast<size_t>(c)] = static_cast<uint64_t>(c);
            std::vector<int32_t> cta_of(cost.size());
            std::vector<std::pair<int64_t, int32_t>> by_cost(cost.size());
            for (size_t k = 0; k < cost.size(); ++k) {
                by_cost[k] = cost[static_cast<uint32_t>(order[k])];
                const uint64_t top = heap.front();   // least loaded, lowest index among equals
                const int32_t c = static_cast<int32_t>(top & 0xFFFFFFFFu);
                cta_of[k] = c;
                ++P->cta_tile_begin[static_cast<size_t>(c) + 1];
                // replace the root and sift it down
                const uint64_t v = top + (static_cast<uint64_t>(by_cost[k].first) << 32);
                size_t i = 0;
                const size_t n = heap.size();
                for (;;) {
                    size_t l = 2 * i + 1;
                    if (l >= n) break;
                    if (l + 1 < n && heap[l + 1] < heap[l]) ++l;
                    if (heap[l] >= v) break;
                    heap[i] = heap[l];
                    i = l;
                }
                heap[i] = v;
            }
            cost.swap(by_cost);
            for (size_t c = 1; c < P->cta_tile_begin.size(); ++c) P->cta_tile_begin[c] += P->cta_tile_begin[c - 1];
            P->cta_tiles.resize(cost.size());
            std::vector<int32_t> pos(P->cta_tile_begin.begin(), P->cta_tile_begin.end() - 1);
            for (size_t k = 0; k < cost.size(); ++k) P->cta_tiles[pos[cta_of[k]]++] = cost[k].second;
        }
    }

    // ------------------------------------------------------------- decode
    std::vector<int32_t> pieces, item_unit;
    plan_decode(P, units, pieces, item_unit, decode_work_ctas, P->fixed ? static_cast<int64_t>(P->num_sms) * cps : 0);

    // ----------------------- fused cache update of small and extend rows
    // the small rows (read by the decode stream) first, then the extend rows
    // (read by the tiles only), each in token order
    std::vector<int32_t> multi_rows(small_rows);
    multi_rows.insert(multi_rows.end(), extend_rows.begin(), extend_rows.end());
    for (int32_t r : multi_rows) {
        WriteRun w{};
        w.t0 = qsl[r];
        w.n_tok = qsl[r + 1] - qsl[r];
        w.req = r;
        w.pos0 = d->num_computed_tokens[r];
        w.wbegin = P->write_tokens;
        P->write_tokens += w.n_tok;
        P->write_runs.push_back(w);
    }
    // the small rows' runs are stored before the decode stream starts; with a
    // second stream the extend rows' runs are stored there, before the tiles
    P->write_runs_early = static_cast<int32_t>(small_rows.size());
    for (int32_t k = 0; k < P->write_runs_early; ++k) P->write_tokens_early += P->write_runs[k].n_tok;

    // ----------------------------------------------------- partial slots
    std::vector<int32_t> count(static_cast<size_t>(P->T) * P->n_groups, 0);
    for (size_t u = 0; u < units.size(); ++u)
        for (int grp = 0; grp < P->n_groups; ++grp) {
            const int32_t k = pieces[u * P->n_groups + grp];
            for (int32_t t = units[u].t0; t < units[u].t0 + units[u].n_tok; ++t)
                count[static_cast<size_t>(t) * P->n_groups + grp] = cascade ? P->prefix_splits + k : (k > 1 ? k : 0);
        }
    if (cascade)
        for (int32_t r : extend_rows)
            for (int32_t t = qsl[r]; t < qsl[r + 1]; ++t)
                for (int grp = 0; grp < P->n_groups; ++grp)
                    count[static_cast<size_t>(t) * P->n_groups + grp] = P->prefix_splits + 1;
    for (size_t i = 0; i < P->items.size(); ++i) {
        DecodeItem &it = P->items[i];
        const int32_t k = pieces[static_cast<size_t>(item_unit[i]) * P->n_groups + it.head_group];
        if (cascade) it.part += P->prefix_splits;
        else if (k == 1) it.part = -1;
    }
    P->part_offset.assign(count.size(), 0);
    P->merges.reserve(units.size() * P->n_groups + (cascade ? count.size() : 0));
    int64_t slots = 0;
    for (size_t i = 0; i < count.size(); ++i) {
        P->part_offset[i] = static_cast<int32_t>(slots);
        slots += count[i];
        if (count[i] > 0) {
            MergeRow m{};
            m.token = static_cast<int32_t>(i / P->n_groups);
            m.slot0 = P->part_offset[i];
            m.count = count[i];
            m.hq_begin = static_cast<int32_t>(i % P->n_groups) * P->HG * P->G;
            m.hq_count = P->HG * P->G;
            // staged inputs: rows from the decode prefix on are final when
            // the tiles finish, so none of them may be merged
            if (P->decode_prefix > 0 && m.token >= P->decode_prefix) return PA_ERR_CAPACITY;
            P->merges.push_back(m);
        }
    }
    if (slots > INT32_MAX) return PA_ERR_UNSUPPORTED;
    P->num_slots = static_cast<int32_t>(slots);

    // ------------------------------------------------- launch shape
    P->ncta = static_cast<int32_t>(P->cta_begin.size()) - 1;
    const int32_t scr_rows = P->max_blocks > 0 ? static_cast<int32_t>(P->scratch_table.size() / P->max_blocks) : 0;
    if (P->fixed) {
        // decode units: at least one token each, and a request of at most
        // kMaxSmallQ tokens makes at most ceil(kMaxSmallQ / tg) of them; the
        // equal cut adds at most one item per CTA
        const int64_t max_units = std::min<int64_t>(shape->max_tokens, static_cast<int64_t>(shape->max_reqs) *
                                                                            ((kMaxSmallQ + tg - 1) / tg));
        const int64_t items_cap = static_cast<int64_t>(P->ncta) + max_units * P->n_groups;
        const int64_t merges_cap = static_cast<int64_t>(shape->max_tokens) * P->n_groups;
        const int64_t slots_cap = shape->max_partial_slots > 0
                                      ? shape->max_partial_slots
                                      : static_cast<int64_t>(P->ncta) + 2 * merges_cap;
        if (items_cap > INT32_MAX || merges_cap > INT32_MAX || slots_cap > INT32_MAX) return PA_ERR_UNSUPPORTED;
        P->cap_tokens = shape->max_tokens;
        P->cap_items = static_cast<int32_t>(items_cap);
        P->cap_tiles = shape->max_extend_tiles;
        P->cap_merges = static_cast<int32_t>(merges_cap);
        P->cap_dequant = P->kv8 && P->cap_tiles > 0 ? shape->max_dequant_blocks : 0;
        P->cap_slots = static_cast<int32_t>(slots_cap);
        P->cap_scr_rows = P->kv8 && P->cap_tiles > 0 ? shape->max_reqs : 0;
        // a row of several query tokens makes T exceed the request count
        P->cap_runs = shape->max_tokens > shape->max_reqs ? shape->max_reqs : 0;
        if (static_cast<int64_t>(P->items.size()) > P->cap_items ||
            static_cast<int64_t>(P->tiles.size()) > P->cap_tiles ||
            static_cast<int64_t>(P->merges.size()) > P->cap_merges || P->num_scratch_blocks > P->cap_dequant ||
            P->num_slots > P->cap_slots || scr_rows > P->cap_scr_rows ||
            static_cast<int64_t>(P->write_runs.size()) > P->cap_runs)
            return PA_ERR_CAPACITY;
    } else {
        P->cap_tokens = P->T;
        P->cap_items = static_cast<int32_t>(P->items.size());
        P->cap_tiles = static_cast<int32_t>(P->tiles.size());
        P->cap_merges = static_cast<int32_t>(P->merges.size());
        P->cap_dequant = P->num_scratch_blocks;
        P->cap_slots = P->num_slots;
        P->cap_scr_rows = scr_rows;
        P->cap_runs = static_cast<int32_t>(P->write_runs.size());
    }

    // ------------------------------------------------- workspace layout
    // (every size below is a capacity: for a fixed-shape plan the layout
    // depends on the shape only)
    size_t off = kHeader;
    auto place = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 16); return o; };
    const size_t off_counts = place(kNumCounts * sizeof(int32_t));
    P->off_part = place(static_cast<size_t>(P->cap_tokens) * P->n_groups * sizeof(int32_t));
    P->off_cta = place(P->cta_begin.size() * sizeof(int32_t));
    P->off_items = place(static_cast<size_t>(P->cap_items) * sizeof(DecodeItem));
    P->off_tiles = place(static_cast<size_t>(P->cap_tiles) * sizeof(ExtendTile));
    P->off_merges = place(static_cast<size_t>(P->cap_merges) * sizeof(MergeRow));
    P->off_scrtab = place(static_cast<size_t>(P->cap_scr_rows) * P->max_blocks * sizeof(int32_t));
    P->off_dequant = place(static_cast<size_t>(P->cap_dequant) * sizeof(DequantItem));
    P->off_runs = place(static_cast<size_t>(P->cap_runs) * sizeof(WriteRun));
    P->off_ctb = place(P->cta_tile_begin.size() * sizeof(int32_t));
    P->off_ctiles = place(static_cast<size_t>(P->cap_tiles) * sizeof(int32_t));
    P->blob_bytes = off - kHeader;
    off = align_up(off, 256);
    P->off_opart = off;
    off = align_up(off + static_cast<size_t>(P->cap_slots) * P->Hq * P->D * sizeof(float), 256);
    P->off_ml = off;
    off = align_up(off + static_cast<size_t>(P->cap_slots) * P->Hq * sizeof(float2), 1024);
    const size_t scratch_bytes = static_cast<size_t>(P->cap_dequant) * kBlockSize * P->Hkv * P->D * 2;
    P->off_kscr = off;
    off = align_up(off + scratch_bytes, 1024);
    P->off_vscr = off;
    off = align_up(off + scratch_bytes, 256);
    P->ws_bytes = off;
    P->blob.assign(P->blob_bytes, 0);
    auto put = [&](size_t at, const void *src, size_t n) {
        if (n) std::memcpy(P->blob.data() + (at - kHeader), src, n);
    };
    int32_t counts[kNumCounts] = {};
    counts[kCountTiles] = static_cast<int32_t>(P->tiles.size());
    counts[kCountMerges] = static_cast<int32_t>(P->merges.size());
    counts[kCountDequant] = static_cast<int32_t>(P->dequant.size());
    counts[kCountTokens] = P->T;
    counts[kCountWriteRuns] = static_cast<int32_t>(P->write_runs.size());
    counts[kCountWriteTokens] = P->write_tokens;
    counts[kCountWriteRunsEarly] = P->write_runs_early;
    counts[kCountWriteTokensEarly] = P->write_tokens_early;
    put(off_counts, counts, sizeof counts);
    put(P->off_part, P->part_offset.data(), P->part_offset.size() * sizeof(int32_t));
    put(P->off_cta, P->cta_begin.data(), P->cta_begin.size() * sizeof(int32_t));
    put(P->off_items, P->items.data(), P->items.size() * sizeof(DecodeItem));
    put(P->off_tiles, P->tiles.data(), P->tiles.size() * sizeof(ExtendTile));
    put(P->off_merges, P->merges.data(), P->merges.size() * sizeof(MergeRow));
    put(P->off_scrtab, P->scratch_table.data(), P->scratch_table.size() * sizeof(int32_t));
    put(P->off_dequant, P->dequant.data(), P->dequant.size() * sizeof(DequantItem));
    put(P->off_runs, P->write_runs.data(), P->write_runs.size() * sizeof(WriteRun));
    put(P->off_ctb, P->cta_tile_begin.data(), P->cta_tile_begin.size() * sizeof(int32_t));
    put(P->off_ctiles, P->cta_tiles.data(), P->cta_tiles.size() * sizeof(int32_t));

    // ------------------------------------------------------------- info
    pa_plan_info &I = P->info;
    I.num_tokens = P->T;
    I.num_decode_rows = static_cast<int32_t>(decode_rows.size());
    I.num_extend_rows = static_cast<int32_t>(extend_rows.size());
    I.num_small_q_rows = static_cast<int32_t>(small_rows.size());
    I.num_decode_ctas = P->ncta;
    I.num_decode_items = static_cast<int32_t>(P->items.size());
    I.num_extend_tiles = static_cast<int32_t>(P->tiles.size());
    I.num_partial_slots = P->num_slots;
    I.num_merge_rows = static_cast<int32_t>(P->merges.size());
    I.kernels_per_call = (P->ncta > 0 ? 1 : 0) + (P->cap_tiles > 0 ? 1 : 0) + (P->cap_merges > 0 ? 1 : 0) +
                         (P->cap_dequant > 0 ? 1 : 0);
    I.num_dequant_blocks = P->num_scratch_blocks;
    const int64_t row_bytes = static_cast<int64_t>(P->Hkv) * P->D * 2 * (P->kv8 ? 1 : 2);   // K and V
    for (const DecodeUnit &u : units) I.decode_kv_bytes += std::max(0, u.key_end - kb_keys) * row_bytes;
    I.prefix_kv_bytes = cascade ? kb_keys * row_bytes : 0;
    double pairs = 0.0;   // sum over the row's queries i of (num_computed + i + 1 - prefix keys)
    for (int32_t r : extend_rows) {
        const double q_len = qsl[r + 1] - qsl[r];
        pairs += q_len * (d->num_computed_tokens[r] + 1 - kb_keys) + q_len * (q_len - 1) / 2;
    }
    I.extend_flops = 4.0 * P->D * P->Hq * pairs;
    I.prefix_flops = cascade ? 4.0 * P->D * P->Hq * static_cast<double>(P->T) * kb_keys : 0.0;
    return PA_OK;
}

cudaError_t record(pa_plan_s *P, int kind, bool start, cudaStream_t stream) {
    if (!P->timing) return cudaSuccess;
    cudaEvent_t e;
    cudaError_t err = cudaEventCreate(&e);
    if (err != cudaSuccess) return err;
    (start ? P->ev_start : P->ev_stop)[kind].push_back(e);
    return cudaEventRecord(e, stream);
}

void clear_timing(pa_plan_s *P) {
    for (int k = 0; k < 4; ++k) {
        for (auto e : P->ev_start[k]) cudaEventDestroy(e);
        for (auto e : P->ev_stop[k]) cudaEventDestroy(e);
        P->ev_start[k].clear();
        P->ev_stop[k].clear();
    }
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

namespace pa {

SideStream *side_stream() {
    // one per host thread and device, created on first use and kept for the
    // thread's lifetime (never destroyed: a thread may outlive nothing here,
    // but the CUDA context may be torn down before thread-local destructors)
    constexpr int kMaxDevices = 64;
    thread_local SideStream slots[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    SideStream &ss = slots[dev];
    if (!ss.stream) {
        cudaStream_t st = nullptr;
        cudaEvent_t fork = nullptr, join = nullptr;
        if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
        if (cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess) {
            if (fork) cudaEventDestroy(fork);
            cudaStreamDestroy(st);
            return nullptr;
        }
        ss.stream = st;
        ss.fork = fork;
        ss.join = join;
    }
    return &ss;
}

pa_status prepare_plan(pa_plan_s *P) {
    if (P->prepared) return PA_OK;
    if (P->ncta > 0 && prepare_decode(P->D, P->HG, P->kv8) != cudaSuccess) return PA_ERR_CUDA;
    if (P->cap_tiles > 0 && prepare_extend(P->D) != cudaSuccess) return PA_ERR_CUDA;
    if (P->fork && side_stream() == nullptr) return PA_ERR_CUDA;
    P->prepared = true;
    return PA_OK;
}

pa_status enqueue_attention(pa_plan_s *P, const void *q, const void *key_cache, const void *value_cache,
                            const int32_t *block_table, void *out, uint8_t *ws, cudaStream_t stream, bool timed,
                            const KvUpdate &update, bool allow_fork) {
    auto rec = [&](int kind, bool start, cudaStream_t st) { return timed ? record(P, kind, start, st) : cudaSuccess; };
    int32_t *err = reinterpret_cast<int32_t *>(ws);
    const int32_t *counts = reinterpret_cast<const int32_t *>(ws + kHeader);
    const int32_t *part_offset = reinterpret_cast<const int32_t *>(ws + P->off_part);
    float *o_part = reinterpret_cast<float *>(ws + P->off_opart);
    float2 *ml_part = reinterpret_cast<float2 *>(ws + P->off_ml);
    uint16_t *out16 = static_cast<uint16_t *>(out);
    const int sms = std::max(1, P->num_sms);

    // decode stream: one box per block and 128-byte column slice covers the
    // CTA's HG kv heads; tensor-core tiles (bf16 caches): one box per block,
    // kv head and 64-column half
    CUtensorMap tm_k{}, tm_v{}, tm_dk{}, tm_dv{};
    const uint64_t rows = static_cast<uint64_t>(P->num_blocks) * kBlockSize;
    if (P->ncta > 0 && (!make_map_kv(&tm_dk, key_cache, P->D, P->Hkv, rows, P->HG, P->kv8) ||
                        !make_map_kv(&tm_dv, value_cache, P->D, P->Hkv, rows, P->HG, P->kv8)))
        return PA_ERR_CUDA;
    if (P->cap_tiles > 0 && !P->kv8 &&
        (!make_map(&tm_k, key_cache, P->D, P->Hkv, rows, 1, kBlockSize) ||
         !make_map(&tm_v, value_cache, P->D, P->Hkv, rows, 1, kBlockSize)))
        return PA_ERR_CUDA;

    const bool fork = P->fork && allow_fork && P->cap_tiles > 0;
    // staged inputs (rows from the decode prefix on complete at late_rows):
    // with a second stream only the tiles' side waits; without one, all
    const bool staged = update.late_rows != nullptr;
    if (staged && !fork && cudaStreamWaitEvent(stream, update.late_rows, 0) != cudaSuccess) return PA_ERR_CUDA;
    WriteParams wp{};
    int write_grid = 0;
    if (update.key != nullptr && P->cap_runs > 0) {
        // fused cache update of the small and extend rows' new tokens (the
        // decode stream and the tiles read them); one-token decode rows' are
        // stored by the decode kernel itself
        wp.key = static_cast<const uint16_t *>(update.key);
        wp.value = static_cast<const uint16_t *>(update.value);
        wp.key_cache = const_cast<void *>(key_cache);
        wp.value_cache = const_cast<void *>(value_cache);
        wp.block_table = block_table;
        wp.runs = reinterpret_cast<const WriteRun *>(ws + P->off_runs);
        wp.counts = counts;
        wp.slots_out = update.slots_out;
        wp.err = err;
        wp.row_elems = P->Hkv * P->D;
        wp.max_blocks = P->max_blocks;
        wp.num_blocks = P->num_blocks;
        wp.kv8 = P->kv8 ? 1 : 0;
        wp.k_scale = P->k_scale;
        wp.v_scale = P->v_scale;
        const int64_t chunks = static_cast<int64_t>(std::max(1, P->fixed ? P->cap_tokens : P->write_tokens)) *
                               (P->kv8 ? wp.row_elems / 16 : wp.row_elems / 8);
        write_grid = static_cast<int>(std::min<int64_t>((chunks + 255) / 256, 16 * sms));
        // with a second stream: here the small rows' runs (the decode stream
        // reads them), the extend rows' on the tile stream before the tiles
        // (after late_rows when staged); without one, all of them here
        wp.part = fork ? 1 : 0;
        if ((!fork || P->fixed || P->write_runs_early > 0) &&
            launch_write_runs(write_grid, wp, stream) != cudaSuccess)
            return PA_ERR_CUDA;
    }
    // Side by side: the write of the extend rows, the tiles (and, for E4M3
    // caches, the bf16 copies of their blocks) go to a second stream that
    // starts after everything enqueued so far (metadata upload, write of the
    // small rows), while the decode kernel runs on the other SMs; the merge
    // waits for both.
    cudaStream_t tile_stream = stream;
    SideStream *side = nullptr;
    if (fork) {
        side = side_stream();
        if (!side || cudaEventRecord(side->fork, stream) != cudaSuccess ||
            cudaStreamWaitEvent(side->stream, side->fork, 0) != cudaSuccess)
            return PA_ERR_CUDA;
        tile_stream = side->stream;
        if (staged && cudaStreamWaitEvent(tile_stream, update.late_rows, 0) != cudaSuccess) return PA_ERR_CUDA;
        wp.part = 2;
        if (write_grid > 0 && launch_write_runs(write_grid, wp, tile_stream, false) != cudaSuccess)
            return PA_ERR_CUDA;
    }
    if (P->cap_tiles > 0) {
        // E4M3: the tiles read bf16 copies of their blocks, made here
        CUtensorMap tm_tk = tm_k, tm_tv = tm_v;
        const int32_t *tile_table = block_table;
        int32_t tile_blocks = P->num_blocks;
        if (P->kv8) {
            DequantParams qp{};
            qp.key_cache = static_cast<const uint8_t *>(key_cache);
            qp.value_cache = static_cast<const uint8_t *>(value_cache);
            qp.key_out = reinterpret_cast<uint16_t *>(ws + P->off_kscr);
            qp.value_out = reinterpret_cast<uint16_t *>(ws + P->off_vscr);
            qp.block_table = block_table;
            qp.items = reinterpret_cast<const DequantItem *>(ws + P->off_dequant);
            qp.err = err;
            qp.counts = counts;
            qp.max_blocks = P->max_blocks;
            qp.num_blocks = P->num_blocks;
            qp.block_elems = kBlockSize * P->Hkv * P->D;
            if (launch_dequant(std::min(P->cap_dequant, 8 * sms), qp, tile_stream, !fork) != cudaSuccess)
                return PA_ERR_CUDA;
            const uint64_t srows = static_cast<uint64_t>(std::max(1, P->cap_dequant)) * kBlockSize;
            if (!make_map(&tm_tk, ws + P->off_kscr, P->D, P->Hkv, srows, 1, kBlockSize) ||
                !make_map(&tm_tv, ws + P->off_vscr, P->D, P->Hkv, srows, 1, kBlockSize))
                return PA_ERR_CUDA;
            tile_table = reinterpret_cast<const int32_t *>(ws + P->off_scrtab);
            tile_blocks = P->cap_dequant;
        }
        CUtensorMap tm_q;
        if (!make_map(&tm_q, q, P->D, P->Hq, std::max(1, P->cap_tokens), P->G, kTileRows / P->G)) return PA_ERR_CUDA;
        ExtendParams ep{};
        ep.out = out16;
        ep.block_table = tile_table;
        ep.tiles = reinterpret_cast<const ExtendTile *>(ws + P->off_tiles);
        ep.part_offset = part_offset;
        ep.o_part = o_part;
        ep.ml_part = ml_part;
        ep.err = err;
        ep.cta_tile_begin = reinterpret_cast<const int32_t *>(ws + P->off_ctb);
        ep.cta_tiles = reinterpret_cast<const int32_t *>(ws + P->off_ctiles);
        ep.max_blocks = P->max_blocks;
        ep.num_blocks = tile_blocks;
        ep.num_heads_q = P->Hq;
        ep.group = P->G;
        ep.n_groups = P->n_groups;
        ep.heads_per_group = P->HG;
        ep.scale_log2 = P->scale_log2;
        ep.out_scale = P->out_scale;
        if (rec(1, true, tile_stream) != cudaSuccess) return PA_ERR_CUDA;
        if (launch_extend(P->D, P->ext_ctas, tm_q, tm_tk, tm_tv, ep, tile_stream, !fork) != cudaSuccess)
            return PA_ERR_CUDA;
        if (rec(1, false, tile_stream) != cudaSuccess) return PA_ERR_CUDA;
        // staged: the rows from the decode prefix on are the tiles' alone
        // (no merge row), final here
        if (fork && update.late_out_ready && cudaEventRecord(update.late_out_ready, tile_stream) != cudaSuccess)
            return PA_ERR_CUDA;
        if (fork && cudaEventRecord(side->join, tile_stream) != cudaSuccess) return PA_ERR_CUDA;
    }
    if (P->ncta > 0) {
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
        dp.out_scale = P->out_scale;
        dp.new_k = static_cast<const uint16_t *>(update.key);
        dp.new_v = static_cast<const uint16_t *>(update.value);
        dp.cache_k = const_cast<void *>(key_cache);
        dp.cache_v = const_cast<void *>(value_cache);
        dp.slots_out = update.slots_out;
        dp.num_heads_kv = P->Hkv;
        dp.k_scale = P->k_scale;
        dp.v_scale = P->v_scale;
        if (rec(0, true, stream) != cudaSuccess) return PA_ERR_CUDA;
        if (launch_decode(P->D, P->HG, P->kv8, P->ncta, tm_dk, tm_dv, dp, stream) != cudaSuccess) return PA_ERR_CUDA;
        if (rec(0, false, stream) != cudaSuccess) return PA_ERR_CUDA;
    }
    if (fork && cudaStreamWaitEvent(stream, side->join, 0) != cudaSuccess) return PA_ERR_CUDA;
    if (P->cap_merges > 0) {
        MergeParams mp{};
        mp.out = out16;
        mp.rows = reinterpret_cast<const MergeRow *>(ws + P->off_merges);
        mp.o_part = o_part;
        mp.ml_part = ml_part;
        mp.counts = counts;
        mp.num_heads_q = P->Hq;
        mp.max_heads = P->HG * P->G;
        const int64_t warps = static_cast<int64_t>(P->cap_merges) * mp.max_heads;   // 8 warps per CTA
        const int grid = static_cast<int>(std::min<int64_t>((warps + 7) / 8, 16 * sms));
        if (rec(2, true, stream) != cudaSuccess) return PA_ERR_CUDA;
        if (launch_merge(P->D, grid, mp, stream, !fork) != cudaSuccess) return PA_ERR_CUDA;
        if (rec(2, false, stream) != cudaSuccess) return PA_ERR_CUDA;
    }
    if (!fork && update.late_out_ready && cudaEventRecord(update.late_out_ready, stream) != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}

}  // namespace pa

extern "C" {

const char *pa_status_string(pa_status s) {
    switch (s) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARGUMENT: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape";
        case PA_ERR_CUDA: return "CUDA runtime error";
        case PA_ERR_DEVICE_CHECK: return "device-side check failed";
        case PA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case PA_ERR_CAPACITY: return "step exceeds the plan's fixed capacity";
    }
    return "unknown status";
}

pa_status pa_plan(const pa_batch_desc *desc, pa_plan_t **out, size_t *workspace_bytes) {
    if (out) *out = nullptr;
    if (desc == nullptr || out == nullptr || workspace_bytes == nullptr) return PA_ERR_INVALID_ARGUMENT;
    pa_status st = validate(desc);
    if (st != PA_OK) return st;
    pa_plan_s *P = new (std::nothrow) pa_plan_s();
    if (!P) return PA_ERR_INVALID_ARGUMENT;
    st = build_plan(P, desc, nullptr);
    if (st != PA_OK) {
        delete P;
        return st;
    }
    *out = P;
    *workspace_bytes = P->ws_bytes;
    return PA_OK;
}

pa_status pa_plan_fixed(const pa_batch_desc *desc, const pa_fixed_shape *shape, pa_plan_t **out,
                        size_t *workspace_bytes) {
    if (out) *out = nullptr;
    if (desc == nullptr || shape == nullptr || out == nullptr || workspace_bytes == nullptr)
        return PA_ERR_INVALID_ARGUMENT;
    if (shape->max_tokens <= 0 || shape->max_reqs <= 0 || shape->max_extend_tiles < 0 ||
        shape->max_dequant_blocks < 0 || shape->max_partial_slots < 0 || shape->decode_prefix_tokens < 0)
        return PA_ERR_INVALID_ARGUMENT;
    pa_status st = validate(desc);
    if (st != PA_OK) return st;
    if (desc->kv_cache_dtype == PA_KV_FP8_E4M3 && shape->max_extend_tiles > 0 && shape->max_dequant_blocks == 0)
        return PA_ERR_INVALID_ARGUMENT;   // FP8 tiles read bf16 copies: they need room
    pa_plan_s *P = new (std::nothrow) pa_plan_s();
    if (!P) return PA_ERR_INVALID_ARGUMENT;
    st = build_plan(P, desc, shape);
    if (st != PA_OK) {
        delete P;
        return st;
    }
    *out = P;
    *workspace_bytes = P->ws_bytes;
    return PA_OK;
}

void pa_plan_destroy(pa_plan_t *P) {
    if (!P) return;
    if (P->pinned) staging().release(P->pinned, P->pinned_cap, P->upload_evt);
    clear_timing(P);
    delete P;
}

pa_status pa_plan_get_info(const pa_plan_t *P, pa_plan_info *info) {
    if (!P || !info) return PA_ERR_INVALID_ARGUMENT;
    *info = P->info;
    return PA_OK;
}

pa_status pa_slot_mapping(const int32_t *qsl, const int32_t *num_computed, const int32_t *block_table,
                          int32_t num_reqs, int32_t num_tokens, int32_t max_blocks_per_req,
                          int32_t block_size, int64_t *slot_mapping, void *stream) {
    if (num_tokens < 0 || num_reqs < 0 || max_blocks_per_req <= 0 || block_size <= 0)
        return PA_ERR_INVALID_ARGUMENT;
    if (num_tokens == 0) return PA_OK;
    if (num_reqs == 0 || !qsl || !num_computed || !block_table || !slot_mapping) return PA_ERR_INVALID_ARGUMENT;
    cudaError_t e = launch_slot_mapping(qsl, num_computed, block_table, num_reqs, num_tokens, max_blocks_per_req,
                                        block_size, slot_mapping, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_write_kv(const void *key, const void *value, const int64_t *slot_mapping, int32_t num_tokens,
                      int32_t num_heads_kv, int32_t head_dim, void *key_cache, void *value_cache,
                      int64_t num_slots, int32_t *device_error_word, void *stream) {
    if (num_tokens < 0 || num_heads_kv <= 0 || head_dim <= 0 || num_slots < 0) return PA_ERR_INVALID_ARGUMENT;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !slot_mapping || !key_cache || !value_cache) return PA_ERR_INVALID_ARGUMENT;
    const int64_t row_bytes = static_cast<int64_t>(num_heads_kv) * head_dim * 2;
    if (row_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16))
        return PA_ERR_INVALID_ARGUMENT;
    cudaError_t e = launch_write_kv(key, value, slot_mapping, num_tokens, num_heads_kv * head_dim, key_cache,
                                    value_cache, num_slots, device_error_word, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_write_kv_fp8(const void *key, const void *value, const int64_t *slot_mapping, int32_t num_tokens,
                          int32_t num_heads_kv, int32_t head_dim, void *key_cache, void *value_cache,
                          int64_t num_slots, float k_scale, float v_scale, int32_t *device_error_word,
                          void *stream) {
    if (num_tokens < 0 || num_heads_kv <= 0 || head_dim <= 0 || num_slots < 0) return PA_ERR_INVALID_ARGUMENT;
    if (!(k_scale > 0.f) || !std::isfinite(k_scale) || !(v_scale > 0.f) || !std::isfinite(v_scale))
        return PA_ERR_INVALID_ARGUMENT;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !slot_mapping || !key_cache || !value_cache) return PA_ERR_INVALID_ARGUMENT;
    if ((static_cast<int64_t>(num_heads_kv) * head_dim) % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16))
        return PA_ERR_INVALID_ARGUMENT;
    cudaError_t e = launch_write_kv_fp8(key, value, slot_mapping, num_tokens, num_heads_kv * head_dim, key_cache,
                                        value_cache, num_slots, k_scale, v_scale, device_error_word,
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

namespace {

pa_status check_launch_args(const pa_plan_s *P, const void *q, const void *key_cache, const void *value_cache,
                            const int32_t *block_table, const void *out, const void *workspace,
                            size_t workspace_bytes) {
    if (!q || !key_cache || !value_cache || !block_table || !out || !workspace) return PA_ERR_INVALID_ARGUMENT;
    if (!aligned(workspace, 256) || !aligned(q, 16) || !aligned(out, 16) || !aligned(key_cache, 16) ||
        !aligned(value_cache, 16) || !aligned(block_table, 4))
        return PA_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < P->ws_bytes) return PA_ERR_WORKSPACE_TOO_SMALL;
    return PA_OK;
}

// metadata upload (pinned, stream ordered); the caller holds P->mu
pa_status upload(pa_plan_s *P, uint8_t *ws, cudaStream_t stream, bool timed) {
    if (!P->blob_bytes) return PA_OK;
    if (!P->pinned) {
        if (!staging().acquire(P->blob_bytes, &P->pinned, &P->pinned_cap, &P->upload_evt)) return PA_ERR_CUDA;
        std::memcpy(P->pinned, P->blob.data(), P->blob_bytes);
    }
    if (!P->pinned_dev && cudaHostGetDevicePointer(&P->pinned_dev, P->pinned, 0) != cudaSuccess) return PA_ERR_CUDA;
    if (timed && record(P, 3, true, stream) != cudaSuccess) return PA_ERR_CUDA;
    if (launch_upload(P->pinned_dev, ws + kHeader, P->blob_bytes, stream) != cudaSuccess) return PA_ERR_CUDA;
    if (timed && record(P, 3, false, stream) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaEventRecord(P->upload_evt, stream) != cudaSuccess) return PA_ERR_CUDA;
    return PA_OK;
}

}  // namespace

pa_status pa_attention(const pa_plan_t *plan, const void *q, const void *key_cache, const void *value_cache,
                       const int32_t *block_table, void *out, void *workspace, size_t workspace_bytes,
                       void *stream_) {
    if (!plan) return PA_ERR_INVALID_ARGUMENT;
    pa_plan_s *P = const_cast<pa_plan_s *>(plan);
    if (P->T == 0 && !P->fixed) return PA_OK;
    pa_status st = check_launch_args(P, q, key_cache, value_cache, block_table, out, workspace, workspace_bytes);
    if (st != PA_OK) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    std::lock_guard<std::mutex> lock(P->mu);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if ((st = prepare_plan(P)) != PA_OK) return st;
    if ((st = upload(P, ws, stream, true)) != PA_OK) return st;
    return enqueue_attention(P, q, key_cache, value_cache, block_table, out, ws, stream, true);
}

pa_status pa_upload_metadata(const pa_plan_t *plan, void *workspace, size_t workspace_bytes, void *stream_) {
    if (!plan || !workspace) return PA_ERR_INVALID_ARGUMENT;
    pa_plan_s *P = const_cast<pa_plan_s *>(plan);
    if (!aligned(workspace, 256)) return PA_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < P->ws_bytes) return PA_ERR_WORKSPACE_TOO_SMALL;
    std::lock_guard<std::mutex> lock(P->mu);
    pa_status st = prepare_plan(P);
    if (st != PA_OK) return st;
    return upload(P, static_cast<uint8_t *>(workspace), static_cast<cudaStream_t>(stream_), false);
}

size_t pa_plan_metadata_bytes(const pa_plan_t *plan) { return plan ? plan->blob_bytes : 0; }

pa_status pa_plan_copy_metadata(const pa_plan_t *plan, void *host_dst, size_t bytes) {
    if (!plan || (!host_dst && plan->blob_bytes)) return PA_ERR_INVALID_ARGUMENT;
    pa_plan_s *P = const_cast<pa_plan_s *>(plan);
    if (bytes < P->blob_bytes) return PA_ERR_INVALID_ARGUMENT;
    if (P->blob_bytes) std::memcpy(host_dst, P->blob.data(), P->blob_bytes);
    return PA_OK;
}

pa_status pa_upload_metadata_from(const void *host_src, size_t bytes, void *workspace, size_t workspace_bytes,
                                  void *stream_) {
    if (!workspace || !aligned(workspace, 256) || bytes % 16 != 0 || (bytes && (!host_src || !aligned(host_src, 16))))
        return PA_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < kHeader + bytes) return PA_ERR_WORKSPACE_TOO_SMALL;
    if (!bytes) return PA_OK;
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, host_src) != cudaSuccess || attr.type != cudaMemoryTypeHost) {
        cudaGetLastError();   // clear the error of an unregistered pointer
        return PA_ERR_INVALID_ARGUMENT;
    }
    void *dev_src = nullptr;
    if (cudaHostGetDevicePointer(&dev_src, const_cast<void *>(host_src), 0) != cudaSuccess) return PA_ERR_CUDA;
    return launch_upload(dev_src, static_cast<uint8_t *>(workspace) + kHeader, bytes,
                         static_cast<cudaStream_t>(stream_)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_attention_launch(const pa_plan_t *plan, const void *q, const void *key_cache, const void *value_cache,
                              const int32_t *block_table, void *out, void *workspace, size_t workspace_bytes,
                              void *stream_) {
    if (!plan) return PA_ERR_INVALID_ARGUMENT;
    pa_plan_s *P = const_cast<pa_plan_s *>(plan);
    if (P->T == 0 && !P->fixed) return PA_OK;
    pa_status st = check_launch_args(P, q, key_cache, value_cache, block_table, out, workspace, workspace_bytes);
    if (st != PA_OK) return st;
    std::lock_guard<std::mutex> lock(P->mu);
    if ((st = prepare_plan(P)) != PA_OK) return st;
    return enqueue_attention(P, q, key_cache, value_cache, block_table, out, static_cast<uint8_t *>(workspace),
                             static_cast<cudaStream_t>(stream_), false);
}

pa_status pa_attention_with_kv_update(const pa_plan_t *plan, const void *q, const void *key, const void *value,
                                      void *key_cache, void *value_cache, const int32_t *block_table,
                                      int64_t *slot_mapping, void *out, void *workspace, size_t workspace_bytes,
                                      void *stream_) {
    if (!plan) return PA_ERR_INVALID_ARGUMENT;
    pa_plan_s *P = const_cast<pa_plan_s *>(plan);
    if (P->T == 0 && !P->fixed) return PA_OK;
    pa_status st = check_launch_args(P, q, key_cache, value_cache, block_table, out, workspace, workspace_bytes);
    if (st != PA_OK) return st;
    if (!key || !value || !aligned(key, 16) || !aligned(value, 16) || (slot_mapping && !aligned(slot_mapping, 8)))
        return PA_ERR_INVALID_ARGUMENT;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    std::lock_guard<std::mutex> lock(P->mu);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if ((st = prepare_plan(P)) != PA_OK) return st;
    if ((st = upload(P, ws, stream, true)) != PA_OK) return st;
    KvUpdate u;
    u.key = key;
    u.value = value;
    u.slots_out = slot_mapping;
    return enqueue_attention(P, q, key_cache, value_cache, block_table, out, ws, stream, true, u);
}

pa_status pa_attention_with_kv_update_launch(const pa_plan_t *plan, const void *q, const void *key,
                                             const void *value, void *key_cache, void *value_cache,
                                             const int32_t *block_table, int64_t *slot_mapping, void *out,
                                             void *workspace, size_t workspace_bytes, void *stream_) {
    if (!plan) return PA_ERR_INVALID_ARGUMENT;
    pa_plan_s *P = const_cast<pa_plan_s *>(plan);
    if (P->T == 0 && !P->fixed) return PA_OK;
    pa_status st = check_launch_args(P, q, key_cache, value_cache, block_table, out, workspace, workspace_bytes);
    if (st != PA_OK) return st;
    if (!key || !value || !aligned(key, 16) || !aligned(value, 16) || (slot_mapping && !aligned(slot_mapping, 8)))
        return PA_ERR_INVALID_ARGUMENT;
    std::lock_guard<std::mutex> lock(P->mu);
    if ((st = prepare_plan(P)) != PA_OK) return st;
    KvUpdate u;
    u.key = key;
    u.value = value;
    u.slots_out = slot_mapping;
    return enqueue_attention(P, q, key_cache, value_cache, block_table, out, static_cast<uint8_t *>(workspace),
                             static_cast<cudaStream_t>(stream_), false, u);
}

pa_status pa_attention_with_kv_update_launch_staged(const pa_plan_t *plan, const void *q, const void *key,
                                                    const void *value, void *key_cache, void *value_cache,
                                                    const int32_t *block_table, int64_t *slot_mapping, void *out,
                                                    void *workspace, size_t workspace_bytes, void *stream_,
                                                    void *late_rows, void *late_out_ready) {
    if (!plan || !late_rows || !plan->fixed || plan->decode_prefix <= 0) return PA_ERR_INVALID_ARGUMENT;
    pa_plan_s *P = const_cast<pa_plan_s *>(plan);
    pa_status st = check_launch_args(P, q, key_cache, value_cache, block_table, out, workspace, workspace_bytes);
    if (st != PA_OK) return st;
    if (!key || !value || !aligned(key, 16) || !aligned(value, 16) || (slot_mapping && !aligned(slot_mapping, 8)))
        return PA_ERR_INVALID_ARGUMENT;
    std::lock_guard<std::mutex> lock(P->mu);
    if ((st = prepare_plan(P)) != PA_OK) return st;
    KvUpdate u;
    u.key = key;
    u.value = value;
    u.slots_out = slot_mapping;
    u.late_rows = static_cast<cudaEvent_t>(late_rows);
    u.late_out_ready = static_cast<cudaEvent_t>(late_out_ready);
    return enqueue_attention(P, q, key_cache, value_cache, block_table, out, static_cast<uint8_t *>(workspace),
                             static_cast<cudaStream_t>(stream_), false, u);
}

pa_status pa_zero_blocks(const int32_t *block_ids, int32_t num_ids, int32_t num_blocks, int32_t num_heads_kv,
                         int32_t head_dim, int32_t kv_cache_dtype, void *key_cache, void *value_cache,
                         int32_t *device_error_word, void *stream) {
    if (num_ids < 0 || num_blocks < 0 || num_heads_kv <= 0 || head_dim <= 0) return PA_ERR_INVALID_ARGUMENT;
    if (kv_cache_dtype != PA_KV_BF16 && kv_cache_dtype != PA_KV_FP8_E4M3) return PA_ERR_INVALID_ARGUMENT;
    if (num_ids == 0) return PA_OK;
    if (!block_ids || !key_cache || !value_cache || !aligned(key_cache, 16) || !aligned(value_cache, 16) ||
        !aligned(block_ids, 4))
        return PA_ERR_INVALID_ARGUMENT;
    const int64_t block_bytes =
        static_cast<int64_t>(kBlockSize) * num_heads_kv * head_dim * (kv_cache_dtype == PA_KV_FP8_E4M3 ? 1 : 2);
    if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    cudaError_t e = launch_zero_blocks(block_ids, num_ids, num_blocks, block_bytes, key_cache, value_cache,
                                       device_error_word, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_check_device_errors(int32_t *word, int32_t *bits, void *stream_) {
    if (bits) *bits = 0;
    if (!word) return PA_ERR_INVALID_ARGUMENT;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    int32_t host = 0;
    if (cudaMemcpyAsync(&host, word, sizeof host, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaMemsetAsync(word, 0, sizeof host, stream) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PA_ERR_CUDA;
    if (bits) *bits = host;
    return host == 0 ? PA_OK : PA_ERR_DEVICE_CHECK;
}

pa_status pa_plan_enable_timing(pa_plan_t *P, int32_t enable) {
    if (!P) return PA_ERR_INVALID_ARGUMENT;
    std::lock_guard<std::mutex> lock(P->mu);
    clear_timing(P);
    P->timing = enable != 0;
    return PA_OK;
}

pa_status pa_plan_kernel_times(pa_plan_t *P, double ms_total[4], int32_t launches[4]) {
    if (!P || !ms_total || !launches) return PA_ERR_INVALID_ARGUMENT;
    std::lock_guard<std::mutex> lock(P->mu);
    for (int k = 0; k < 4; ++k) {
        ms_total[k] = 0.0;
        launches[k] = static_cast<int32_t>(P->ev_stop[k].size());
        for (size_t i = 0; i < P->ev_stop[k].size(); ++i) {
            if (cudaEventSynchronize(P->ev_stop[k][i]) != cudaSuccess) return PA_ERR_CUDA;
            float ms = 0.f;
            if (cudaEventElapsedTime(&ms, P->ev_start[k][i], P->ev_stop[k][i]) != cudaSuccess) return PA_ERR_CUDA;
            ms_total[k] += ms;
        }
    }
    return PA_OK;
}

}  // extern "C"
