// Split-KV decode attention: one query token per request, keys streamed
// block by block from the paged caches.
//
// Shape of the work (page "vLLM 推理流程分析" §6.2 / §10.2: a decode query
// reads every earlier K/V row through the block table; page
// "vLLM 源码完全拆解（十六）", third walk-through: stable softmax over the
// pages, partition partials (m, l, o) merged afterwards).
//
// GB300 mapping:
//  * persistent CTAs, one per SM; the planner cuts the concatenation of all
//    decode requests' key blocks into contiguous runs, one per CTA, equal in
//    bytes (E4M3 caches: equal in bytes plus a fixed cost per item), so every
//    SM streams about the same (runs that split a request produce partials
//    for the merge kernel);
//  * one CTA serves HG kv heads; a producer warp streams each 16-token block
//    as one TMA box per 128-byte column slice ([HG heads][16 rows][128 B],
//    128-byte swizzle, each head's rows one contiguous tile) for K and for V
//    into an NS-stage mbarrier ring.  Large boxes matter: the TMA unit's
//    per-box cost caps an SM at about 54 GB/s with one box per head, while
//    [8 heads] boxes reach the HBM limit from about 100 SMs on;
//  * one consumer warp per kv head: the G query heads of the group form the
//    rows of a 16x16 bf16 MMA tile (G <= 16), so each K/V row loaded from HBM
//    is used by all G heads; S = Q K^T and O += P V run on the tensor cores
//    (mma.sync), the online softmax in fp32 registers with quad shuffles.
//    E4M3 caches: codes converted in registers to f16 MMA operands; items of
//    at most 8 query rows compute the transposed products (keys as MMA rows),
//    which halves their MMAs.
#include <type_traits>

#include "dev.cuh"

namespace pa {
namespace {

using namespace dev;

template <int D, int HG, bool KV8>
struct DecodeCfg {
    static constexpr int EB = KV8 ? 1 : 2;                 // bytes per cache element
    static constexpr int NH = D * EB / 128;                // 128-byte boxes per cache row
    static constexpr int CPE = 128 / EB;                   // elements per box row
    static constexpr int BOX = 16 * 128;                   // one head's [16 rows][128 B] tile
    static constexpr int SLICE = HG * BOX;                 // one TMA box: a column slice of all HG heads
    static constexpr int TSTAGE = NH * SLICE;              // K (or V) bytes per block: [slice][head][row]
    static constexpr int STAGE = decode_stage_bytes(D, HG, KV8);
    static constexpr int NS = decode_stages(D, HG, KV8);
    static constexpr int THREADS = decode_threads(HG);
    static constexpr int SMEM = decode_smem_bytes(D, HG, KV8);
};

// bf16 pair -> f16 pair (saturating at the largest finite f16)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) { return pack_f16x2_sat(bf16_lo(w), bf16_hi(w)); }

// Fused cache update of one decode row (pa_attention_with_kv_update; the
// fused dispatch of "vLLM 推理流程分析" §6.1, the write of §6.3): the item
// whose run holds a decode row's last page stores the row's new K and V
// (E4M3: quantised exactly as pa_write_kv_fp8 does) when it starts, one warp
// per kv head, before the producer loads that page, which then reads the new
// row from the cache like every other row.  Every other slot a decode row
// reads was written by an earlier step.
__device__ __forceinline__ int new_row_page(const DecodeItem &item) {
    const int lp = (item.key_end - 1) / kBlockSize;
    return item.n_tok == 1 && item.key_end > 0 && item.page_begin <= lp && lp < item.page_end ? lp : -1;
}

template <int D, bool KV8>
__device__ __forceinline__ void store_new_row(const DecodeParams &p, const DecodeItem &item, int lp, int kvh,
                                              int lane) {
    const int32_t blk = __ldg(p.block_table + static_cast<int64_t>(item.req) * p.max_blocks + lp);
    const int64_t slot = static_cast<int64_t>(blk) * kBlockSize + (item.key_end - 1) % kBlockSize;
    const bool ok = blk >= 0 && blk < p.num_blocks;   // else: not stored (the page load reports it)
    if (ok && lane < D / 8) {
        const int64_t src = (static_cast<int64_t>(item.token) * p.num_heads_kv + kvh) * D;
        const int64_t dst = (slot * p.num_heads_kv + kvh) * D;
        const uint4 k = __ldg(reinterpret_cast<const uint4 *>(p.new_k + src) + lane);
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.new_v + src) + lane);
        if constexpr (KV8) {
            reinterpret_cast<uint2 *>(static_cast<uint8_t *>(p.cache_k) + dst)[lane] = e4m3_quantize8(k, p.k_scale);
            reinterpret_cast<uint2 *>(static_cast<uint8_t *>(p.cache_v) + dst)[lane] = e4m3_quantize8(v, p.v_scale);
        } else {
            reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.cache_k) + dst)[lane] = k;
            reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.cache_v) + dst)[lane] = v;
        }
    }
    if (kvh == 0 && lane == 0 && p.slots_out != nullptr && ok) p.slots_out[item.token] = slot;
    fence_proxy_async_global();   // the stores before the async-proxy (TMA) load of the page
}

template <int D, int HG, bool KV8, bool FUSED>
__global__ void __launch_bounds__((HG + 1) * 32, 1)
decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const DecodeParams p) {
    using C = DecodeCfg<D, HG, KV8>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int abort_flag;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;           // stages, 1024-aligned
    const uint32_t bar0 = base + C::NS * C::STAGE;   // full_k | full_v | empty | row_ready
    auto full_k = [&](int s) { return bar0 + 8u * s; };
    auto full_v = [&](int s) { return bar0 + 8u * (C::NS + s); };
    auto empty = [&](int s) { return bar0 + 8u * (2 * C::NS + s); };
    const uint32_t row_ready = bar0 + 8u * (3 * C::NS);   // fused update: new rows stored (HG arrivals)
    auto stage = [&](int s) { return base + static_cast<uint32_t>(s) * C::STAGE; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    grid_launch_dependents();
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(full_k(s), 1);
            mbar_init(full_v(s), 1);
            mbar_init(empty(s), HG);
        }
        mbar_init(row_ready, HG);
        fence_barrier_init();
    } else if (threadIdx.x == 32 * HG) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    // everything below reads or writes what earlier kernels of the stream
    // produce or consume (work list, caches, partials)
    grid_dep_wait();
    __syncthreads();

    const int item_begin = p.cta_begin[blockIdx.x];
    const int item_end = p.cta_begin[blockIdx.x + 1];

    if (warp == HG) {
        // ------------------------------------------------------ producer --
        int issued = 0;
        int rows_waited = 0;            // fused update: row_ready phases consumed
        // the stream is read once: its lines go first when L2 needs room, so
        // it does not push out what other kernels of the step (tensor-core
        // tiles beside it, partials, metadata) keep re-reading
        const uint64_t evict_first = policy_evict_first();
        bool ok = true;
        for (int it = item_begin; it < item_end && ok; ++it) {
            const DecodeItem item = p.items[it];
            const int32_t *bt = p.block_table + static_cast<int64_t>(item.req) * p.max_blocks;
            const int h0 = item.head_group * HG;
            const int new_page = FUSED ? new_row_page(item) : -1;   // load only after its new rows are stored
            int32_t blk_lane = 0;       // block id of page (window + lane), 32 pages at a time
            int window = item.page_begin - 32;
            for (int pg = item.page_begin; pg < item.page_end; ++pg) {
                if (pg - window >= 32) {
                    window = pg;
                    blk_lane = pg + lane < item.page_end ? bt[pg + lane] : 0;
                }
                const int s = issued % C::NS;
                const int n = issued / C::NS;
                if (n > 0 && !warp_wait(empty(s), (n & 1) ^ 1, &abort_flag)) {
                    if (lane == 0) raise_abort(&abort_flag, p.err, kErrTimeout);
                    ok = false;
                    break;
                }
                const int32_t blk = __shfl_sync(0xffffffffu, blk_lane, pg - window);
                const bool valid = blk >= 0 && blk < p.num_blocks;
                if (pg == new_page) {
                    if (!warp_wait(row_ready, rows_waited & 1, &abort_flag)) {
                        if (lane == 0) raise_abort(&abort_flag, p.err, kErrTimeout);
                        ok = false;
                        break;
                    }
                    ++rows_waited;
                }
                if (lane == 0) {
                    if (valid) {
                        mbar_arrive_expect_tx(full_k(s), C::TSTAGE);
                        mbar_arrive_expect_tx(full_v(s), C::TSTAGE);
                    } else {
                        atomicOr(p.err, kErrBlockRange);
                        mbar_arrive(full_k(s));
                        mbar_arrive(full_v(s));
                    }
                }
                __syncwarp();
                if (valid && lane < 2 * C::NH) {
                    const int tensor = lane / C::NH;
                    const int slice = lane % C::NH;
                    const uint32_t dst = stage(s) + tensor * C::TSTAGE + slice * C::SLICE;
                    const uint32_t bar = tensor ? full_v(s) : full_k(s);
                    tma_load_3d_hint(dst, tensor ? &tm_v : &tm_k, slice * C::CPE, blk * kBlockSize, h0, bar, evict_first);
                }
                ++issued;
            }
        }
        // Never leave the CTA with TMA writes in flight.
        if (lane == 0) {
            for (int k = issued - 1; k >= 0 && k >= issued - C::NS; --k) {
                const int s = k % C::NS, n = k / C::NS;
                if (!mbar_wait(full_k(s), n & 1, nullptr) || !mbar_wait(full_v(s), n & 1, nullptr))
                    atomicOr(p.err, kErrTimeout);
            }
        }
    } else if constexpr (KV8) {
        // ------------------------------------------- consumers (E4M3) --
        // Two cache blocks (32 keys) per softmax round.  K codes feed the
        // f16 MMAs as B fragments directly: the contraction index is permuted
        // so that a lane's four k-values of a step are the four adjacent
        // codes d = 16kk + 4t .. 16kk + 4t + 3 of one key (one 32-bit load).
        // V codes are B fragments of O += P V the same way: n-tile 4a + i
        // holds the dims 32a + 4n + i (n = 0..7 its column), so one 32-bit
        // load of a key row feeds four n-tiles and a byte permute pairs the
        // codes of keys 2t and 2t + 1 (and 2t + 8, 2t + 9).  The row sums l
        // come from one more MMA of P against a column of ones, so they add
        // exactly the f16 weights the value MMAs use.
        const int g = lane >> 2;
        const int t4 = lane & 3;
        const int G = p.group;
        // MMA row r = (token r / G, head r % G)
        constexpr uint32_t kOnes = 0x3C003C00u;  // f16x2 (1, 1)
        const uint32_t k_lane = g * 128u + 4u * t4;   // key g at +0, key g + 8 at +1024
        const uint32_t va_lane = 256u * t4 + 16u * (g >> 2) + 4u * (g & 3);             // key 2t
        const uint32_t vb_lane = 256u * t4 + 128u + 16u * ((g >> 2) ^ 1) + 4u * (g & 3);  // key 2t + 1
        const float sl2 = p.scale_log2;  // > 0: the maximum of raw scores scales
        int consumed = 0;
        bool ok = true;
        for (int it = item_begin; it < item_end && ok; ++it) {
            const DecodeItem item = p.items[it];
            const int kvh = item.head_group * HG + warp;
            const int nrow = item.n_tok * G;
            if (nrow <= 8) {
                // Items of at most 8 query rows (decode rows): the transposed
                // products S^T = K Q^T and O^T += V^T P^T.  The 16 keys of a
                // block are the MMA rows and the query rows its 8 columns, so
                // a block takes half the MMAs of the row-major form (whose 16
                // rows would be mostly empty for one query token).  Lane
                // (g, t) holds the scores of keys g and g + 8 for query rows
                // n0 = 2t and n1 = 2t + 1.  The K codes as loaded above are
                // the A fragments (same contraction order, so Q^T is row g's
                // q); P^T reaches the B fragment of the value MMA through an
                // 8x8 transpose per half block.  O^T m-tile 4h + i holds the
                // dims 64h + 4r + i (r = 0..15 its row), so one 32-bit load
                // of a value row feeds four m-tiles.
                const int n0 = 2 * t4, n1 = 2 * t4 + 1;
                const uint16_t *qg =
                    p.q + (static_cast<int64_t>(item.token + g / G) * p.num_heads_q + kvh * G + g % G) * D;
                uint32_t qt[D / 16][2];
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int c = kk * 16 + 4 * t4;
                    qt[kk][0] = g < nrow ? bf16x2_to_f16x2(__ldg(reinterpret_cast<const uint32_t *>(qg + c))) : 0u;
                    qt[kk][1] = g < nrow ? bf16x2_to_f16x2(__ldg(reinterpret_cast<const uint32_t *>(qg + c + 2))) : 0u;
                }
                float ot[D / 16][4];
#pragma unroll
                for (int j = 0; j < D / 16; ++j) ot[j][0] = ot[j][1] = ot[j][2] = ot[j][3] = 0.f;
                float lt[4] = {0.f, 0.f, 0.f, 0.f};
                float ma = -INFINITY, mb = -INFINITY;   // running maxima of rows n0 and n1 (scaled)
                // causal limits of rows n0 and n1: token i sees keys < key_end - (n_tok - 1 - i)
                const int lim_a = min(item.key_end, item.key_end - (item.n_tok - 1 - n0 / G));
                const int lim_b = min(item.key_end, item.key_end - (item.n_tok - 1 - n1 / G));
                const int lim_lo = item.key_end - (item.n_tok - 1);
                if constexpr (FUSED) {
                    const int lp = new_row_page(item);
                    if (lp >= 0) {
                        store_new_row<D, true>(p, item, lp, kvh, lane);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(row_ready);
                    }
                }
                auto qk_t = [&](uint32_t kb, float (&s)[4]) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t x = kb + k_lane + (static_cast<uint32_t>(kk ^ g) << 4);
                        uint32_t a[4];
                        e4m3x4_to_f16x2x2(lds_u32(x), a[0], a[2]);
                        e4m3x4_to_f16x2x2(lds_u32(x + 1024u), a[1], a[3]);
                        mma_f16_16816(s, a, qt[kk][0], qt[kk][1]);
                    }
                };
                // O^T += V^T P^T for one block: lane (g, t) loads the value
                // rows of keys 2t, 2t + 1, 2t + 8, 2t + 9 at the logical bytes
                // 64h + 32jr + 4g (dims of rows g + 8jr of m-tiles 4h + i);
                // MASKED zeroes the codes of rows at or past `valid`
                auto pv_t = [&](auto masked, uint32_t vb, uint32_t b0, uint32_t b1, int valid) {
                    const uint32_t r0 = vb + 256u * t4;
                    uint32_t mA = ~0u, mB = ~0u, mC = ~0u, mD = ~0u;
                    if constexpr (decltype(masked)::value) {
                        mA = 2 * t4 < valid ? ~0u : 0u;
                        mB = 2 * t4 + 1 < valid ? ~0u : 0u;
                        mC = 2 * t4 + 8 < valid ? ~0u : 0u;
                        mD = 2 * t4 + 9 < valid ? ~0u : 0u;
                    }
#pragma unroll
                    for (int h = 0; h < D / 64; ++h) {
                        uint32_t a[4][4];
#pragma unroll
                        for (int jr = 0; jr < 2; ++jr) {
                            const uint32_t chunk = 4u * h + 2u * jr + static_cast<uint32_t>(g >> 2);
                            const uint32_t ce = ((chunk ^ (2u * t4)) << 4) + 4u * (g & 3);        // rows 2t, 2t + 8
                            const uint32_t co = ((chunk ^ (2u * t4 + 1u)) << 4) + 4u * (g & 3);   // rows 2t + 1, 2t + 9
                            uint32_t wA = lds_u32(r0 + ce), wB = lds_u32(r0 + 128u + co);
                            uint32_t wC = lds_u32(r0 + 1024u + ce), wD = lds_u32(r0 + 1152u + co);
                            if constexpr (decltype(masked)::value) {
                                wA &= mA; wB &= mB; wC &= mC; wD &= mD;
                            }
                            e4m3x4_to_f16x2x2(prmt(wA, wB, 0x5140u), a[0][jr], a[1][jr]);
                            e4m3x4_to_f16x2x2(prmt(wA, wB, 0x7362u), a[2][jr], a[3][jr]);
                            e4m3x4_to_f16x2x2(prmt(wC, wD, 0x5140u), a[0][2 + jr], a[1][2 + jr]);
                            e4m3x4_to_f16x2x2(prmt(wC, wD, 0x7362u), a[2][2 + jr], a[3][2 + jr]);
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) mma_f16_16816(ot[4 * h + i], a[i], b0, b1);
                    }
                    const uint32_t ones[4] = {kOnes, kOnes, kOnes, kOnes};
                    mma_f16_16816(lt, ones, b0, b1);   // every row: the f16 weights' sums of n0, n1
                };
                auto round_t = [&](auto two_c, int pg) -> bool {
                    constexpr bool TWO = decltype(two_c)::value;
                    const int s0 = consumed % C::NS, s1 = (consumed + 1) % C::NS;
                    const uint32_t par0 = (consumed / C::NS) & 1, par1 = ((consumed + 1) / C::NS) & 1;
                    if (!warp_wait(full_k(s0), par0, &abort_flag) || (TWO && !warp_wait(full_k(s1), par1, &abort_flag)))
                        return false;
                    if (!warp_wait(full_v(s0), par0, &abort_flag) || (TWO && !warp_wait(full_v(s1), par1, &abort_flag)))
                        return false;
                    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
                    qk_t(stage(s0) + warp * C::BOX, sa);
                    if constexpr (TWO) qk_t(stage(s1) + warp * C::BOX, sb);
                    const int loaded = TWO ? 2 * kBlockSize : kBlockSize;
                    const int valid_keys = min(item.key_end - pg * kBlockSize, loaded);   // V rows past it may be anything
                    if (!TWO || lim_lo - pg * kBlockSize < 2 * kBlockSize) {
                        // keys past the context or a row's causal limit drop out
                        const int va = min(lim_a - pg * kBlockSize, loaded), vb = min(lim_b - pg * kBlockSize, loaded);
                        if (g >= va) sa[0] = -INFINITY;
                        if (g >= vb) sa[1] = -INFINITY;
                        if (g + 8 >= va) sa[2] = -INFINITY;
                        if (g + 8 >= vb) sa[3] = -INFINITY;
                        if constexpr (TWO) {
                            if (g + 16 >= va) sb[0] = -INFINITY;
                            if (g + 16 >= vb) sb[1] = -INFINITY;
                            if (g + 24 >= va) sb[2] = -INFINITY;
                            if (g + 24 >= vb) sb[3] = -INFINITY;
                        }
                    }
                    float mx0 = fmaxf(sa[0], sa[2]), mx1 = fmaxf(sa[1], sa[3]);
                    if constexpr (TWO) {
                        mx0 = max3(mx0, sb[0], sb[2]);
                        mx1 = max3(mx1, sb[1], sb[3]);
                    }
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1) {   // over the keys: lanes of the same t
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
                    }
                    mx0 *= sl2;
                    mx1 *= sl2;
                    // rescale only when the running maximum grows by more than 2^8
                    const bool need0 = mx0 > ma + 8.f;
                    const bool need1 = mx1 > mb + 8.f;
                    if (__any_sync(0xffffffffu, need0 || need1)) {
                        float a0 = 1.f, a1 = 1.f;
                        if (need0) { a0 = ex2(ma - mx0); ma = mx0; }
                        if (need1) { a1 = ex2(mb - mx1); mb = mx1; }
#pragma unroll
                        for (int j = 0; j < D / 16; ++j) {
                            ot[j][0] *= a0; ot[j][1] *= a1; ot[j][2] *= a0; ot[j][3] *= a1;
                        }
                        lt[0] *= a0; lt[1] *= a1; lt[2] *= a0; lt[3] *= a1;
                    }
                    const float ra = ma == -INFINITY ? 0.f : ma;
                    const float rb = mb == -INFINITY ? 0.f : mb;
                    // P^T of a block as B fragments: the packed weights of keys
                    // g (and g + 8) x rows (n0, n1), transposed 8x8
                    auto weights = [&](const float (&s)[4], uint32_t &b0, uint32_t &b1) {
                        b0 = movmatrix_trans(pack_f16x2(ex2(fmaf(s[0], sl2, -ra)), ex2(fmaf(s[1], sl2, -rb))));
                        b1 = movmatrix_trans(pack_f16x2(ex2(fmaf(s[2], sl2, -ra)), ex2(fmaf(s[3], sl2, -rb))));
                    };
                    uint32_t pa0, pa1;
                    weights(sa, pa0, pa1);
                    const uint32_t vb0 = stage(s0) + C::TSTAGE + warp * C::BOX;
                    if (valid_keys < kBlockSize) pv_t(std::true_type{}, vb0, pa0, pa1, valid_keys);
                    else pv_t(std::false_type{}, vb0, pa0, pa1, kBlockSize);
                    if constexpr (TWO) {
                        uint32_t pb0, pb1;
                        weights(sb, pb0, pb1);
                        const uint32_t vb1 = stage(s1) + C::TSTAGE + warp * C::BOX;
                        if (valid_keys < 2 * kBlockSize) pv_t(std::true_type{}, vb1, pb0, pb1, valid_keys - kBlockSize);
                        else pv_t(std::false_type{}, vb1, pb0, pb1, kBlockSize);
                    }
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(empty(s0));
                        if constexpr (TWO) mbar_arrive(empty(s1));
                    }
                    consumed += TWO ? 2 : 1;
                    return true;
                };
                int pg = item.page_begin;
                for (; ok && pg + 1 < item.page_end; pg += 2) ok = round_t(std::true_type{}, pg);
                if (ok && pg < item.page_end) ok = round_t(std::false_type{}, pg);
                if (!ok) {
                    if (lane == 0) raise_abort(&abort_flag, p.err, kErrTimeout);
                    break;
                }
                // rows n0 and n1: lane holds dims 64h + 32jr + 4g + i in
                // ot[4h + i][2jr] (row n0) and ot[4h + i][2jr + 1] (row n1)
                const float inv0 = lt[0] > 0.f ? p.out_scale / lt[0] : 0.f;
                const float inv1 = lt[1] > 0.f ? p.out_scale / lt[1] : 0.f;
                const bool has0 = n0 < nrow, has1 = n1 < nrow;
                const int tokA = n0 / G, tokB = n1 / G;
                const int headA = kvh * G + n0 % G, headB = kvh * G + n1 % G;
                if (item.part < 0) {
                    uint16_t *oa = p.out + (static_cast<int64_t>(item.token + tokA) * p.num_heads_q + headA) * D;
                    uint16_t *ob = p.out + (static_cast<int64_t>(item.token + tokB) * p.num_heads_q + headB) * D;
#pragma unroll
                    for (int h = 0; h < D / 64; ++h)
#pragma unroll
                        for (int jr = 0; jr < 2; ++jr) {
                            const int d = 64 * h + 32 * jr + 4 * g;
                            if (has0)
                                *reinterpret_cast<uint2 *>(oa + d) =
                                    make_uint2(pack_bf16x2(ot[4 * h][2 * jr] * inv0, ot[4 * h + 1][2 * jr] * inv0),
                                               pack_bf16x2(ot[4 * h + 2][2 * jr] * inv0, ot[4 * h + 3][2 * jr] * inv0));
                            if (has1)
                                *reinterpret_cast<uint2 *>(ob + d) =
                                    make_uint2(pack_bf16x2(ot[4 * h][2 * jr + 1] * inv1, ot[4 * h + 1][2 * jr + 1] * inv1),
                                               pack_bf16x2(ot[4 * h + 2][2 * jr + 1] * inv1, ot[4 * h + 3][2 * jr + 1] * inv1));
                        }
                } else {
                    const int64_t slotA = has0 ? static_cast<int64_t>(p.part_offset[(item.token + tokA) * p.n_groups + item.head_group]) + item.part : 0;
                    const int64_t slotB = has1 ? static_cast<int64_t>(p.part_offset[(item.token + tokB) * p.n_groups + item.head_group]) + item.part : 0;
                    float *opa = p.o_part + (slotA * p.num_heads_q + headA) * D;
                    float *opb = p.o_part + (slotB * p.num_heads_q + headB) * D;
#pragma unroll
                    for (int h = 0; h < D / 64; ++h)
#pragma unroll
                        for (int jr = 0; jr < 2; ++jr) {
                            const int d = 64 * h + 32 * jr + 4 * g;
                            if (has0)
                                *reinterpret_cast<float4 *>(opa + d) =
                                    make_float4(ot[4 * h][2 * jr] * inv0, ot[4 * h + 1][2 * jr] * inv0,
                                                ot[4 * h + 2][2 * jr] * inv0, ot[4 * h + 3][2 * jr] * inv0);
                            if (has1)
                                *reinterpret_cast<float4 *>(opb + d) =
                                    make_float4(ot[4 * h][2 * jr + 1] * inv1, ot[4 * h + 1][2 * jr + 1] * inv1,
                                                ot[4 * h + 2][2 * jr + 1] * inv1, ot[4 * h + 3][2 * jr + 1] * inv1);
                        }
                    if (g == 0) {
                        if (has0) p.ml_part[slotA * p.num_heads_q + headA] = make_float2(ma, lt[0]);
                        if (has1) p.ml_part[slotB * p.num_heads_q + headB] = make_float2(mb, lt[1]);
                    }
                }
                continue;
            }
            const int tok0 = g / G, tok1 = (g + 8) / G;
            const int head0 = kvh * G + g % G, head1 = kvh * G + (g + 8) % G;
            const uint16_t *q0 = p.q + (static_cast<int64_t>(item.token + tok0) * p.num_heads_q + head0) * D;
            const uint16_t *q1 = p.q + (static_cast<int64_t>(item.token + tok1) * p.num_heads_q + head1) * D;
            // causal limit of each row: token i sees keys < key_end - (n_tok - 1 - i)
            const int lim0 = min(item.key_end, item.key_end - (item.n_tok - 1 - tok0));
            const int lim1 = min(item.key_end, item.key_end - (item.n_tok - 1 - tok1));
            const int lim_min = item.key_end - (item.n_tok - 1);
            uint32_t qf[D / 16][4];
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int c = kk * 16 + 4 * t4;
                auto ld = [&](const uint16_t *row, int col) {
                    return bf16x2_to_f16x2(__ldg(reinterpret_cast<const uint32_t *>(row + col)));
                };
                qf[kk][0] = g < nrow ? ld(q0, c) : 0u;
                qf[kk][1] = g + 8 < nrow ? ld(q1, c) : 0u;
                qf[kk][2] = g < nrow ? ld(q0, c + 2) : 0u;
                qf[kk][3] = g + 8 < nrow ? ld(q1, c + 2) : 0u;
            }
            float o[D / 8][4];
#pragma unroll
            for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
            float lacc[4] = {0.f, 0.f, 0.f, 0.f};
            float m0 = -INFINITY, m1 = -INFINITY;
            if constexpr (FUSED) {
                const int lp = new_row_page(item);
                if (lp >= 0) {
                    store_new_row<D, true>(p, item, lp, kvh, lane);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(row_ready);
                }
            }

            auto qk = [&](uint32_t kb, float (&a)[4], float (&b)[4]) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t x = kb + k_lane + (static_cast<uint32_t>(kk ^ g) << 4);
                    uint32_t k0, k1, k2, k3;
                    e4m3x4_to_f16x2x2(lds_u32(x), k0, k1);
                    e4m3x4_to_f16x2x2(lds_u32(x + 1024u), k2, k3);
                    mma_f16_16816(a, qf[kk], k0, k1);
                    mma_f16_16816(b, qf[kk], k2, k3);
                }
            };
            // O += P V for one block; MASKED zeroes the codes of rows at or
            // past `valid` (0-weight x NaN would poison the MMA)
            auto pv = [&](auto masked, uint32_t vb, const uint32_t (&pf)[4], int valid) {
                const uint32_t ra = vb + va_lane, rb = vb + vb_lane;
                uint32_t mA = ~0u, mB = ~0u, mC = ~0u, mD = ~0u;
                if constexpr (decltype(masked)::value) {
                    mA = 2 * t4 < valid ? ~0u : 0u;
                    mB = 2 * t4 + 1 < valid ? ~0u : 0u;
                    mC = 2 * t4 + 8 < valid ? ~0u : 0u;
                    mD = 2 * t4 + 9 < valid ? ~0u : 0u;
                }
#pragma unroll
                for (int a = 0; a < D / 32; ++a) {
                    const uint32_t xa = static_cast<uint32_t>(a ^ t4) << 5;
                    uint32_t wA = lds_u32(ra + xa), wB = lds_u32(rb + xa);
                    uint32_t wC = lds_u32(ra + 1024u + xa), wD = lds_u32(rb + 1024u + xa);
                    if constexpr (decltype(masked)::value) {
                        wA &= mA; wB &= mB; wC &= mC; wD &= mD;
                    }
                    uint32_t b0[4], b1[4];
                    e4m3x4_to_f16x2x2(prmt(wA, wB, 0x5140u), b0[0], b0[1]);
                    e4m3x4_to_f16x2x2(prmt(wA, wB, 0x7362u), b0[2], b0[3]);
                    e4m3x4_to_f16x2x2(prmt(wC, wD, 0x5140u), b1[0], b1[1]);
                    e4m3x4_to_f16x2x2(prmt(wC, wD, 0x7362u), b1[2], b1[3]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) mma_f16_16816(o[4 * a + i], pf, b0[i], b1[i]);
                }
                mma_f16_16816(lacc, pf, kOnes, kOnes);
            };
            // one softmax round over one (TWO = false) or two cache blocks
            auto round = [&](auto two_c, int pg) -> bool {
                constexpr bool TWO = decltype(two_c)::value;
                const int s0 = consumed % C::NS, s1 = (consumed + 1) % C::NS;
                const uint32_t par0 = (consumed / C::NS) & 1, par1 = ((consumed + 1) / C::NS) & 1;
                if (!warp_wait(full_k(s0), par0, &abort_flag) || (TWO && !warp_wait(full_k(s1), par1, &abort_flag)))
                    return false;
                // the round's V blocks too (they land with the K blocks): one
                // scheduling region per round, so value loads and conversions
                // can interleave with the softmax
                if (!warp_wait(full_v(s0), par0, &abort_flag) || (TWO && !warp_wait(full_v(s1), par1, &abort_flag)))
                    return false;
                float sc[4][4];
#pragma unroll
                for (int j = 0; j < 4; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
                qk(stage(s0) + warp * C::BOX, sc[0], sc[1]);
                if constexpr (TWO) qk(stage(s1) + warp * C::BOX, sc[2], sc[3]);
                // keys past the context (their codes may be NaN) or past the
                // blocks loaded drop out; raw scores, scaled inside ex2
                const int loaded = TWO ? 2 * kBlockSize : kBlockSize;
                const int valid_keys = min(item.key_end - pg * kBlockSize, loaded);   // V rows past it may be anything
                if (!TWO || lim_min - pg * kBlockSize < 2 * kBlockSize) {
                    const int valid0 = min(lim0 - pg * kBlockSize, loaded), valid1 = min(lim1 - pg * kBlockSize, loaded);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (j * 8 + 2 * t4 + (e & 1) >= (e < 2 ? valid0 : valid1)) sc[j][e] = -INFINITY;
                }
                constexpr int NT = TWO ? 4 : 2;
                float mx0 = fmaxf(sc[0][0], sc[0][1]), mx1 = fmaxf(sc[0][2], sc[0][3]);
#pragma unroll
                for (int j = 1; j < NT; ++j) {
                    mx0 = fmaxf(mx0, fmaxf(sc[j][0], sc[j][1]));
                    mx1 = fmaxf(mx1, fmaxf(sc[j][2], sc[j][3]));
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2)) * sl2;
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2)) * sl2;
                // rescale only when the running maximum grows by more than 2^8
                const bool need0 = mx0 > m0 + 8.f;
                const bool need1 = mx1 > m1 + 8.f;
                if (__any_sync(0xffffffffu, need0 || need1)) {
                    float a0 = 1.f, a1 = 1.f;
                    if (need0) { a0 = ex2(m0 - mx0); m0 = mx0; }
                    if (need1) { a1 = ex2(m1 - mx1); m1 = mx1; }
#pragma unroll
                    for (int j = 0; j < D / 8; ++j) {
                        o[j][0] *= a0; o[j][1] *= a0; o[j][2] *= a1; o[j][3] *= a1;
                    }
                    lacc[0] *= a0; lacc[1] *= a0; lacc[2] *= a1; lacc[3] *= a1;
                }
                const float r0 = m0 == -INFINITY ? 0.f : m0;
                const float r1 = m1 == -INFINITY ? 0.f : m1;
                uint32_t pa[2][4];
#pragma unroll
                for (int b = 0; b < NT / 2; ++b) {
                    pa[b][0] = pack_f16x2(ex2(fmaf(sc[2 * b][0], sl2, -r0)), ex2(fmaf(sc[2 * b][1], sl2, -r0)));
                    pa[b][1] = pack_f16x2(ex2(fmaf(sc[2 * b][2], sl2, -r1)), ex2(fmaf(sc[2 * b][3], sl2, -r1)));
                    pa[b][2] = pack_f16x2(ex2(fmaf(sc[2 * b + 1][0], sl2, -r0)), ex2(fmaf(sc[2 * b + 1][1], sl2, -r0)));
                    pa[b][3] = pack_f16x2(ex2(fmaf(sc[2 * b + 1][2], sl2, -r1)), ex2(fmaf(sc[2 * b + 1][3], sl2, -r1)));
                }
                const uint32_t vb0 = stage(s0) + C::TSTAGE + warp * C::BOX;
                if (valid_keys < kBlockSize) pv(std::true_type{}, vb0, pa[0], valid_keys);
                else pv(std::false_type{}, vb0, pa[0], kBlockSize);
                if constexpr (TWO) {
                    const uint32_t vb1 = stage(s1) + C::TSTAGE + warp * C::BOX;
                    if (valid_keys < 2 * kBlockSize) pv(std::true_type{}, vb1, pa[1], valid_keys - kBlockSize);
                    else pv(std::false_type{}, vb1, pa[1], kBlockSize);
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(empty(s0));
                    if constexpr (TWO) mbar_arrive(empty(s1));
                }
                consumed += TWO ? 2 : 1;
                return true;
            };
            int pg = item.page_begin;
            for (; ok && pg + 1 < item.page_end; pg += 2) ok = round(std::true_type{}, pg);
            if (ok && pg < item.page_end) ok = round(std::false_type{}, pg);
            if (!ok) {
                if (lane == 0) raise_abort(&abort_flag, p.err, kErrTimeout);
                break;
            }
            // ------------------------------------------------ finalize --
            const float l0 = lacc[0], l1 = lacc[2];
            const float inv0 = l0 > 0.f ? p.out_scale / l0 : 0.f;
            const float inv1 = l1 > 0.f ? p.out_scale / l1 : 0.f;
            const bool has0 = g < nrow, has1 = g + 8 < nrow;
            // lane holds dims 32a + 8t .. 32a + 8t + 7 of rows g and g + 8:
            // o[4a + i][0 / 2] -> dim 32a + 8t + i, o[4a + i][1 / 3] -> + 4
            if (item.part < 0) {
                uint16_t *orow0 = p.out + (static_cast<int64_t>(item.token + tok0) * p.num_heads_q + head0) * D;
                uint16_t *orow1 = p.out + (static_cast<int64_t>(item.token + tok1) * p.num_heads_q + head1) * D;
#pragma unroll
                for (int a = 0; a < D / 32; ++a) {
                    const int d = 32 * a + 8 * t4;
                    if (has0)
                        *reinterpret_cast<uint4 *>(orow0 + d) =
                            make_uint4(pack_bf16x2(o[4 * a][0] * inv0, o[4 * a + 1][0] * inv0),
                                       pack_bf16x2(o[4 * a + 2][0] * inv0, o[4 * a + 3][0] * inv0),
                                       pack_bf16x2(o[4 * a][1] * inv0, o[4 * a + 1][1] * inv0),
                                       pack_bf16x2(o[4 * a + 2][1] * inv0, o[4 * a + 3][1] * inv0));
                    if (has1)
                        *reinterpret_cast<uint4 *>(orow1 + d) =
                            make_uint4(pack_bf16x2(o[4 * a][2] * inv1, o[4 * a + 1][2] * inv1),
                                       pack_bf16x2(o[4 * a + 2][2] * inv1, o[4 * a + 3][2] * inv1),
                                       pack_bf16x2(o[4 * a][3] * inv1, o[4 * a + 1][3] * inv1),
                                       pack_bf16x2(o[4 * a + 2][3] * inv1, o[4 * a + 3][3] * inv1));
                }
            } else {
                const int64_t slot0 = has0 ? static_cast<int64_t>(p.part_offset[(item.token + tok0) * p.n_groups + item.head_group]) + item.part : 0;
                const int64_t slot1 = has1 ? static_cast<int64_t>(p.part_offset[(item.token + tok1) * p.n_groups + item.head_group]) + item.part : 0;
                float *op0 = p.o_part + (slot0 * p.num_heads_q + head0) * D;
                float *op1 = p.o_part + (slot1 * p.num_heads_q + head1) * D;
#pragma unroll
                for (int a = 0; a < D / 32; ++a) {
                    const int d = 32 * a + 8 * t4;
                    if (has0) {
                        float4 *dst = reinterpret_cast<float4 *>(op0 + d);
                        dst[0] = make_float4(o[4 * a][0] * inv0, o[4 * a + 1][0] * inv0, o[4 * a + 2][0] * inv0, o[4 * a + 3][0] * inv0);
                        dst[1] = make_float4(o[4 * a][1] * inv0, o[4 * a + 1][1] * inv0, o[4 * a + 2][1] * inv0, o[4 * a + 3][1] * inv0);
                    }
                    if (has1) {
                        float4 *dst = reinterpret_cast<float4 *>(op1 + d);
                        dst[0] = make_float4(o[4 * a][2] * inv1, o[4 * a + 1][2] * inv1, o[4 * a + 2][2] * inv1, o[4 * a + 3][2] * inv1);
                        dst[1] = make_float4(o[4 * a][3] * inv1, o[4 * a + 1][3] * inv1, o[4 * a + 2][3] * inv1, o[4 * a + 3][3] * inv1);
                    }
                }
                if (t4 == 0) {
                    if (has0) p.ml_part[slot0 * p.num_heads_q + head0] = make_float2(m0, l0);
                    if (has1) p.ml_part[slot1 * p.num_heads_q + head1] = make_float2(m1, l1);
                }
            }
        }
    } else {
        // ------------------------------------------------ consumers (bf16) --
        // MMA rows g and g + 8 are (query token, head) pairs: row r is token
        // r / G of the item and head r % G of the kv head's group
        const int g = lane >> 2;
        const int t4 = lane & 3;
        const int G = p.group;
        int consumed = 0;
        bool ok = true;
        for (int it = item_begin; it < item_end && ok; ++it) {
            const DecodeItem item = p.items[it];
            const int kvh = item.head_group * HG + warp;
            const int nrow = item.n_tok * G;
            const int tok0 = g / G, tok1 = (g + 8) / G;
            const int head0 = kvh * G + g % G, head1 = kvh * G + (g + 8) % G;
            const uint16_t *q0 = p.q + (static_cast<int64_t>(item.token + tok0) * p.num_heads_q + head0) * D;
            const uint16_t *q1 = p.q + (static_cast<int64_t>(item.token + tok1) * p.num_heads_q + head1) * D;
            // causal limit of each row: token i sees keys < key_end - (n_tok - 1 - i)
            const int lim0 = min(item.key_end, item.key_end - (item.n_tok - 1 - tok0));
            const int lim1 = min(item.key_end, item.key_end - (item.n_tok - 1 - tok1));
            uint32_t qf[D / 16][4];
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int c = kk * 16 + 2 * t4;
                qf[kk][0] = g < nrow ? __ldg(reinterpret_cast<const uint32_t *>(q0 + c)) : 0u;
                qf[kk][1] = g + 8 < nrow ? __ldg(reinterpret_cast<const uint32_t *>(q1 + c)) : 0u;
                qf[kk][2] = g < nrow ? __ldg(reinterpret_cast<const uint32_t *>(q0 + c + 8)) : 0u;
                qf[kk][3] = g + 8 < nrow ? __ldg(reinterpret_cast<const uint32_t *>(q1 + c + 8)) : 0u;
            }
            float o[D / 8][4];
#pragma unroll
            for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
            float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
            if constexpr (FUSED) {
                const int lp = new_row_page(item);
                if (lp >= 0) {
                    store_new_row<D, false>(p, item, lp, kvh, lane);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(row_ready);
                }
            }

            for (int pg = item.page_begin; pg < item.page_end; ++pg, ++consumed) {
                const int s = consumed % C::NS;
                const uint32_t par = (consumed / C::NS) & 1;
                if (!warp_wait(full_k(s), par, &abort_flag)) {
                    if (lane == 0) raise_abort(&abort_flag, p.err, kErrTimeout);
                    ok = false;
                    break;
                }
                const uint32_t kb = stage(s) + warp * C::BOX;   // this head's tile of slice 0
                const uint32_t vb = kb + C::TSTAGE;
                // S = Q K^T over this block's 16 keys (two n-tiles of 8 keys)
                float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int mi = lane >> 3;
                    const int key = (mi >> 1) * 8 + (lane & 7);
                    const int chunk = (kk % 4) * 2 + (mi & 1);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(sw128(kb + (kk / 4) * C::SLICE, key, chunk), b0, b1, b2, b3);
                    mma_bf16_16816(sc[0], qf[kk], b0, b1);
                    mma_bf16_16816(sc[1], qf[kk], b2, b3);
                }
                // mask keys past each row's limit, scale to log2 units
                const int key0 = pg * kBlockSize;
                const int valid_keys = item.key_end - key0;  // >= 1: rows past it may hold anything
                const int valid0 = lim0 - key0, valid1 = lim1 - key0;
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = j * 8 + 2 * t4 + (e & 1);
                        sc[j][e] = key < (e < 2 ? valid0 : valid1) ? sc[j][e] * p.scale_log2 : -INFINITY;
                    }
                float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
                float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                // Rescale only when the running maximum grows by more than 2^8;
                // otherwise keep the stale reference (weights stay <= 256).
                const bool need0 = mx0 > m0 + 8.f;
                const bool need1 = mx1 > m1 + 8.f;
                float a0 = 1.f, a1 = 1.f;
                if (need0) { a0 = ex2(m0 - mx0); m0 = mx0; l0 *= a0; }
                if (need1) { a1 = ex2(m1 - mx1); m1 = mx1; l1 *= a1; }
                if (__any_sync(0xffffffffu, need0 || need1)) {
#pragma unroll
                    for (int j = 0; j < D / 8; ++j) {
                        o[j][0] *= a0; o[j][1] *= a0; o[j][2] *= a1; o[j][3] *= a1;
                    }
                }
                const float r0 = m0 == -INFINITY ? 0.f : m0;
                const float r1 = m1 == -INFINITY ? 0.f : m1;
                uint32_t pa[4];
                pa[0] = pack_bf16x2(ex2(sc[0][0] - r0), ex2(sc[0][1] - r0));
                pa[1] = pack_bf16x2(ex2(sc[0][2] - r1), ex2(sc[0][3] - r1));
                pa[2] = pack_bf16x2(ex2(sc[1][0] - r0), ex2(sc[1][1] - r0));
                pa[3] = pack_bf16x2(ex2(sc[1][2] - r1), ex2(sc[1][3] - r1));
                l0 += bf16_lo(pa[0]) + bf16_hi(pa[0]) + bf16_lo(pa[2]) + bf16_hi(pa[2]);
                l1 += bf16_lo(pa[1]) + bf16_hi(pa[1]) + bf16_lo(pa[3]) + bf16_hi(pa[3]);

                if (!warp_wait(full_v(s), par, &abort_flag)) {
                    if (lane == 0) raise_abort(&abort_flag, p.err, kErrTimeout);
                    ok = false;
                    break;
                }
                if (valid_keys < kBlockSize) {
                    // rows past the context may hold anything (even NaN); zero
                    // them so that 0-weight * row stays 0 inside the MMA
                    const int bad = kBlockSize - valid_keys;
                    for (int i = lane; i < bad * C::NH * 8; i += 32) {
                        const int row = valid_keys + i / (C::NH * 8);
                        const int half = (i / 8) % C::NH;
                        const int ch = i % 8;
                        const uint32_t a = vb + half * C::SLICE + row * 128 + ch * 16;
                        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                // O += P V
#pragma unroll
                for (int np = 0; np < D / 16; ++np) {
                    const int mi = lane >> 3;
                    const int key = (mi & 1) * 8 + (lane & 7);
                    const int chunk = 2 * np + (mi >> 1);
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4_trans(sw128(vb + (chunk / 8) * C::SLICE, key, chunk % 8), b0, b1, b2, b3);
                    mma_bf16_16816(o[2 * np], pa, b0, b1);
                    mma_bf16_16816(o[2 * np + 1], pa, b2, b3);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty(s));
            }
            if (!ok) break;
            // ------------------------------------------------ finalize --
            l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
            l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
            const float inv0 = l0 > 0.f ? p.out_scale / l0 : 0.f;
            const float inv1 = l1 > 0.f ? p.out_scale / l1 : 0.f;
            const bool has0 = g < nrow, has1 = g + 8 < nrow;
            if (item.part < 0) {
                uint16_t *orow0 = p.out + (static_cast<int64_t>(item.token + tok0) * p.num_heads_q + head0) * D;
                uint16_t *orow1 = p.out + (static_cast<int64_t>(item.token + tok1) * p.num_heads_q + head1) * D;
#pragma unroll
                for (int j = 0; j < D / 8; ++j) {
                    const int d = j * 8 + 2 * t4;
                    if (has0) *reinterpret_cast<uint32_t *>(orow0 + d) = pack_bf16x2(o[j][0] * inv0, o[j][1] * inv0);
                    if (has1) *reinterpret_cast<uint32_t *>(orow1 + d) = pack_bf16x2(o[j][2] * inv1, o[j][3] * inv1);
                }
            } else {
                const int64_t slot0 = has0 ? static_cast<int64_t>(p.part_offset[(item.token + tok0) * p.n_groups + item.head_group]) + item.part : 0;
                const int64_t slot1 = has1 ? static_cast<int64_t>(p.part_offset[(item.token + tok1) * p.n_groups + item.head_group]) + item.part : 0;
                float *op0 = p.o_part + (slot0 * p.num_heads_q + head0) * D;
                float *op1 = p.o_part + (slot1 * p.num_heads_q + head1) * D;
#pragma unroll
                for (int j = 0; j < D / 8; ++j) {
                    const int d = j * 8 + 2 * t4;
                    if (has0) *reinterpret_cast<float2 *>(op0 + d) = make_float2(o[j][0] * inv0, o[j][1] * inv0);
                    if (has1) *reinterpret_cast<float2 *>(op1 + d) = make_float2(o[j][2] * inv1, o[j][3] * inv1);
                }
                if (t4 == 0) {
                    if (has0) p.ml_part[slot0 * p.num_heads_q + head0] = make_float2(m0, l0);
                    if (has1) p.ml_part[slot1 * p.num_heads_q + head1] = make_float2(m1, l1);
                }
            }
        }
    }
    __syncthreads();
}

template <int D, int HG, bool KV8, bool FUSED>
cudaError_t configure() {
    static bool configured = false;  // attribute is per function, set once per process
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, HG, KV8, FUSED>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, DecodeCfg<D, HG, KV8>::SMEM);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return cudaSuccess;
}

template <int D, int HG, bool KV8>
cudaError_t configure_both() {
    cudaError_t e = configure<D, HG, KV8, false>();
    return e == cudaSuccess ? configure<D, HG, KV8, true>() : e;
}

template <int D, int HG, bool KV8>
cudaError_t launch_t(int num_ctas, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                     const DecodeParams &p, cudaStream_t stream) {
    using C = DecodeCfg<D, HG, KV8>;
    cudaError_t e = configure_both<D, HG, KV8>();
    if (e != cudaSuccess) return e;
    if (p.new_k != nullptr)
        return launch_pdl(decode_kernel<D, HG, KV8, true>, dim3(num_ctas), dim3(C::THREADS),
                          C::SMEM, stream, tm_k, tm_v, p);
    return launch_pdl(decode_kernel<D, HG, KV8, false>, dim3(num_ctas), dim3(C::THREADS),
                      C::SMEM, stream, tm_k, tm_v, p);
}

}  // namespace

#define PA_DECODE_CASES(X)                                                                                  \
    X(64, 1, false) X(64, 2, false) X(64, 4, false) X(64, 8, false) X(128, 1, false) X(128, 2, false)      \
    X(128, 4, false) X(128, 8, false) X(128, 1, true) X(128, 2, true) X(128, 4, true) X(128, 8, true)

cudaError_t prepare_decode(int head_dim, int hg, bool kv8) {
#define X(d, h, f) \
    if (head_dim == d && hg == h && kv8 == f) return configure_both<d, h, f>();
    PA_DECODE_CASES(X)
#undef X
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode(int head_dim, int hg, bool kv8, int num_ctas, const CUtensorMap &tm_k,
                                          const CUtensorMap &tm_v, const DecodeParams &p, cudaStream_t stream) {
    if (num_ctas <= 0) return cudaSuccess;
#define X(d, h, f) \
    if (head_dim == d && hg == h && kv8 == f) return launch_t<d, h, f>(num_ctas, tm_k, tm_v, p, stream);
    PA_DECODE_CASES(X)
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace pa
