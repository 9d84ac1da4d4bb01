// Extend / chunked-prefill attention on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), and the shared-prefix stage of
// the cascade route.
//
// What one CTA computes (page "vLLM 推理流程分析" §6.2: varlen causal
// attention through block_table; §10.1: a token sees itself and earlier
// tokens; §5.1.2: positions = num_computed + offset in the chunk):
//   up to 256 query rows = 2 sub-tiles of 128 rows, each 128/G consecutive
//   tokens x the G query heads of one kv head, against keys
//   [key_begin, key_end) of one request's context, read through the block
//   table in tiles of 128 keys (8 blocks).  Row (i, g) at absolute position
//   pos0 + i sees key j iff j <= pos0 + i (causal tiles); shared-prefix tiles
//   see their whole key range.  Both sub-tiles share every K/V tile loaded.
//
// Per 128-key tile and sub-tile t:
//   S_t = Q_t K^T        tcgen05.mma M=128 N=128 K=D, A and B from shared memory
//   P_t = exp2(S_t*scale*log2e - m)   softmax warpgroup t, one row per thread,
//                        written back to tensor memory over S_t as bf16 pairs
//   O_t += P_t V         tcgen05.mma M=128 N=D K=128, A from tensor memory
// Warp roles: warp 0 TMA producer (Q once, K and V blocks into 2- and 3-stage
// rings; a V stage is released as soon as both PVs reading it are done),
// warp 1 MMA issuer (one thread) and tensor-memory owner (warps 2-3 idle:
// warpgroup 0 gives its registers to the softmax warpgroups), warps 4-7
// softmax of sub-tile 0, warps 8-11 softmax of sub-tile 1.  The MMA thread
// alternates between the sub-tiles, so the tensor core works on one while
// the other's softmax runs.  Its issue blocks at the pipe's rate (about one
// M128 N128 K16 MMA per 64 cycles), so a wait between two MMA groups idles
// the pipe: the barriers it needs next (the next K and V tiles, the other
// sub-tile's P) are tested once in the middle of each group instead.  The running max only moves (and O is rescaled) when it
// grows by more than 2^8, which keeps every weight <= 256.
//
// Tensor memory (512 columns x 128 lanes, fp32): S_0 [0,128), S_1 [128,256)
// (P_t in the first 64 columns of S_t), O_0 [256,256+D), O_1 [384,384+D).
// Shared memory tiles are 128-byte-swizzled [rows][64 elements] halves:
// Q_t (A, K-major), K (B, K-major), V (B, MN-major).
#include "dev.cuh"

namespace pa {
namespace {

using namespace dev;

template <int D>
struct ExtCfg {
    static constexpr int NH = D / 64;
    static constexpr int HALF = 128 * 128;            // [128 rows][64] bf16 half tile
    static constexpr int QB = NH * HALF;              // one Q sub-tile
    static constexpr int KVB = NH * HALF;             // K (or V) tile bytes per stage
    static constexpr int NSK = 2;                     // K stages
    static constexpr int NSV = 3;                     // V stages (V waits longest for its stage)
    static constexpr int THREADS = 384;               // 3 warpgroups
    // registers per thread after the split (launch: 168 x 384 = 64512):
    // 120 x 128 for the load / MMA warpgroup + 192 x 256 for the two softmax
    // warpgroups = 64512
    static constexpr int REGS_CTRL = 120;
    static constexpr int REGS_SOFTMAX = 192;
    static_assert(REGS_CTRL * 128 + REGS_SOFTMAX * 256 <= 168 * 384, "register split exceeds the launch");
    static constexpr int TILE_SMEM = 2 * QB + (NSK + NSV) * KVB;
    // one CTA per SM: it owns all 512 tensor-memory columns
    static constexpr int SMEM = (TILE_SMEM + 2048 < 120 * 1024) ? 120 * 1024 : TILE_SMEM + 2048;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t IDESC_QK = idesc_bf16(128, 128, false, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
};


__device__ __forceinline__ uint32_t col_s(int t) { return static_cast<uint32_t>(t) * 128u; }
__device__ __forceinline__ uint32_t col_o(int t) { return 256u + static_cast<uint32_t>(t) * 128u; }

// barrier indices.  K and V stages are released separately: a K stage as
// soon as the QK^T MMAs reading it finish, a V stage after the PV MMAs, so the
// next K tile is loaded while the current tile's softmax and PV still run.
// The CTA is persistent: rings, barriers and tensor memory carry over from one
// tile to the next, and the next tile's Q is loaded as soon as the current
// tile's last QK^T has read Q (QEMPTY), under the tile's last PV, softmax and
// epilogue.
enum : int {
    B_QFULL = 0,
    B_QEMPTY = 1,
    B_KFULL = 2,    // +stage (2)
    B_VFULL = 4,    // +stage (3)
    B_KEMPTY = 7,   // +stage (2)
    B_VEMPTY = 9,   // +stage (3)
    B_SFULL = 12,   // +sub-tile
    B_PFULL = 14,   // +sub-tile
    B_ODONE = 16,   // +sub-tile
    B_DRAIN = 18,
    NUM_BARS = 19
};

// key tiles each sub-tile of a CTA tile needs (0 for an empty sub-tile)
struct TileShape {
    int n_sub[2];
    int n_tiles;
};
__device__ __forceinline__ TileShape tile_shape(const ExtendTile &tile, int tpt) {
    TileShape sh;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int first = t * tpt;
        if (first >= tile.n_tok) {
            sh.n_sub[t] = 0;
            continue;
        }
        const int last = min(tile.n_tok, first + tpt);   // one past the sub-tile's last token
        const int kend = tile.causal ? min(tile.key_end, tile.pos0 + last) : tile.key_end;
        sh.n_sub[t] = (kend - tile.key_begin + kTileKeys - 1) / kTileKeys;
    }
    sh.n_tiles = max(sh.n_sub[0], sh.n_sub[1]);
    return sh;
}

template <int D>
__global__ void __launch_bounds__(384, 1)
extend_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const ExtendParams p) {
    using C = ExtCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int abort_flag;
    __shared__ uint32_t tmem_base_slot;
    __shared__ __align__(8) uint64_t bars[NUM_BARS];

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    auto q_s = [&](int t) { return base + static_cast<uint32_t>(t) * C::QB; };
    auto k_s = [&](int s) { return base + 2 * C::QB + static_cast<uint32_t>(s) * C::KVB; };
    auto v_s = [&](int s) { return base + 2 * C::QB + static_cast<uint32_t>(C::NSK + s) * C::KVB; };
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    grid_launch_dependents();
    grid_dep_wait();    // the work list and caches come from earlier kernels of the stream
    // this CTA's tiles, longest first (the planner's greedy assignment)
    const int tile_begin = p.cta_tile_begin[blockIdx.x];
    const int tile_end = p.cta_tile_begin[blockIdx.x + 1];
    if (tile_begin >= tile_end) return;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.group;
    const int tpt = kTileRows / G;                    // tokens per 128-row sub-tile

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(bar(B_QFULL), 1);
        mbar_init(bar(B_QEMPTY), 1);
        for (int s = 0; s < C::NSK; ++s) {
            mbar_init(bar(B_KFULL + s), 1);
            mbar_init(bar(B_KEMPTY + s), 1);
        }
        for (int s = 0; s < C::NSV; ++s) {
            mbar_init(bar(B_VFULL + s), 1);
            mbar_init(bar(B_VEMPTY + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(B_SFULL + t), 1);
            mbar_init(bar(B_PFULL + t), 128);
            mbar_init(bar(B_ODONE + t), 1);
        }
        mbar_init(bar(B_DRAIN), 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_base_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_slot;
    if (warp < 4) {
      // warpgroup 0: loads and MMA issue, with few registers
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REGS_CTRL));
      if (warp == 0) {
        // -------------------------------------------------------- producer --
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
        }
        int issued[2] = {0, 0};   // K and V tiles whose loads were issued (over all tiles)
        int n_q_loads = 0;
        bool ok = true;
        for (int ti = tile_begin; ti < tile_end && ok; ++ti) {
            const ExtendTile tile = p.tiles[p.cta_tiles[ti]];
            const TileShape sh = tile_shape(tile, tpt);
            // Q of this tile, once the previous tile's QK^T no longer read Q
            if (n_q_loads > 0 && !warp_wait(bar(B_QEMPTY), (n_q_loads - 1) & 1, &abort_flag)) {
                if (lane == 0) raise_abort(&abort_flag, p.err, kErrTimeout);
                break;
            }
            const int n_q = sh.n_sub[1] > 0 ? 2 : 1;
            // each box is tpt tokens x G heads x 64 dims: tpt * G rows of
            // 128 bytes (128 rows unless G does not divide 128)
            if (lane == 0) mbar_arrive_expect_tx(bar(B_QFULL), n_q * C::NH * tpt * G * 128);
            __syncwarp();
            if (lane < n_q * C::NH) {
                const int t = lane / C::NH, half = lane % C::NH;
                tma_load_3d(q_s(t) + half * C::HALF, &tm_q, half * 64, tile.kv_head * G, tile.t0 + t * tpt,
                            bar(B_QFULL));
            }
            ++n_q_loads;
            const int32_t *bt = p.block_table + static_cast<int64_t>(tile.req) * p.max_blocks;
            // block ids of 32 pages (4 key tiles) per load: the producer's
            // dependent block-table read happens once per window, not per tile
            const int pg_end = (tile.key_end + kBlockSize - 1) / kBlockSize;
            int32_t win = 0;
            int win0 = -64;
            for (int j = 0; j < sh.n_tiles; ++j) {
                const int kt0 = tile.key_begin + j * kTileKeys;
                const int pg0 = kt0 / kBlockSize;
                const int pages = min(8, (tile.key_end - kt0 + kBlockSize - 1) / kBlockSize);
                if (pg0 + 8 > win0 + 32) {
                    win0 = pg0;
                    win = pg0 + lane < pg_end ? bt[pg0 + lane] : 0;
                }
                const int32_t mine_blk = __shfl_sync(0xffffffffu, win, (pg0 - win0 + (lane & 7)) & 31);
                int32_t blk = 0;
                bool valid = false;
                if (lane < pages) {
                    blk = mine_blk;
                    valid = blk >= 0 && blk < p.num_blocks;
                }
                const unsigned vmask = __ballot_sync(0xffffffffu, valid);
                const uint32_t bytes = __popc(vmask) * kBlockSize * 128 * C::NH;
                if (lane == 0 && __popc(vmask) != pages) atomicOr(p.err, kErrBlockRange);
                static_assert(8 * C::NH <= 32, "one TMA box per lane");
                const int page = lane / C::NH;
                const int half = lane % C::NH;
                const int32_t b = __shfl_sync(0xffffffffu, blk, page & 7);  // every lane takes part
                const bool mine = lane < 8 * C::NH && ((vmask >> page) & 1u);
#pragma unroll
                for (int tensor = 0; tensor < 2; ++tensor) {
                    const int ns = tensor ? C::NSV : C::NSK;
                    const int s = issued[tensor] % ns, n = issued[tensor] / ns;
                    const int empty = tensor ? B_VEMPTY : B_KEMPTY;
                    const int full = tensor ? B_VFULL : B_KFULL;
                    if (n > 0 && !warp_wait(bar(empty + s), (n & 1) ^ 1, &abort_flag)) {
                        if (lane == 0) raise_abort(&abort_flag, p.err, kErrTimeout);
                        ok = false;
                        break;
                    }
                    if (lane == 0) mbar_arrive_expect_tx(bar(full + s), bytes);
                    __syncwarp();
                    if (mine)
                        tma_load_3d((tensor ? v_s(s) : k_s(s)) + half * C::HALF + page * 2048,
                                    tensor ? &tm_v : &tm_k, half * 64, tile.kv_head, b * kBlockSize, bar(full + s));
                    ++issued[tensor];
                }
                if (!ok) break;
            }
        }
        if (lane == 0) {
            // no TMA write may outlive the CTA
            if (n_q_loads > 0 && !mbar_wait(bar(B_QFULL), (n_q_loads - 1) & 1, nullptr)) atomicOr(p.err, kErrTimeout);
            for (int tensor = 0; tensor < 2; ++tensor) {
                const int ns = tensor ? C::NSV : C::NSK;
                for (int k = issued[tensor] - 1; k >= 0 && k >= issued[tensor] - ns; --k) {
                    const int s = k % ns, n = k / ns;
                    if (!mbar_wait(bar((tensor ? B_VFULL : B_KFULL) + s), n & 1, nullptr))
                        atomicOr(p.err, kErrTimeout);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer --
        if (lane == 0) {
            int kc = 0, vc = 0;          // K and V tiles consumed (over all tiles)
            int pc[2] = {0, 0};          // P tiles consumed per sub-tile
            int n_q = 0;                 // Q tiles consumed
            bool ok = true;
            // operand descriptors built once; each MMA only moves the start
            // address (the issuing thread shares its issue slots with two
            // softmax warps, so every instruction here counts)
            const uint64_t q_desc[2] = {sdesc_sw128(q_s(0), 16, 1024), sdesc_sw128(q_s(1), 16, 1024)};
            const uint64_t k_desc0 = sdesc_sw128(k_s(0), 16, 1024);
            const uint64_t v_desc0 = sdesc_sw128(v_s(0), C::HALF, 1024);
            // readiness of the barriers the thread needs next, polled (one
            // test each) between MMAs, where the pipe still holds queued work
            bool p_ready[2] = {false, false}, k_ready = false, v_ready = false;
            auto poll = [&](bool &flag, int b, int parity) {
                if (!flag) flag = mbar_test_wait(bar(b), static_cast<uint32_t>(parity));
            };
            auto qk = [&](int t, int s, auto mid) {
                const uint64_t a0 = q_desc[t];
                const uint64_t b0 = sdesc_advance(k_desc0, static_cast<uint32_t>(s) * C::KVB);
                const uint32_t d = tmem + col_s(t);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * C::HALF + (kk % 4) * 32;
                    tc_mma(d, sdesc_advance(a0, off), sdesc_advance(b0, off), C::IDESC_QK, kk > 0 ? 1u : 0u);
                    if (kk == D / 32 - 1) mid();
                }
                tc_commit(bar(B_SFULL + t));
            };
            auto pv = [&](int t, int sv, bool first, auto mid) -> bool {
                if (!p_ready[t] && !mbar_wait_spin(bar(B_PFULL + t), pc[t] & 1, &abort_flag)) return false;
                p_ready[t] = false;
                ++pc[t];
                tc_fence_after();
                const uint64_t b0 = sdesc_advance(v_desc0, static_cast<uint32_t>(sv) * C::KVB);
                const uint32_t d = tmem + col_o(t), a = tmem + col_s(t);
#pragma unroll
                for (int kk = 0; kk < kTileKeys / 16; ++kk) {
                    tc_mma_ts(d, a + kk * 8, sdesc_advance(b0, kk * 2048), C::IDESC_PV, (!first || kk > 0) ? 1u : 0u);
                    if (kk == 3) mid();
                }
                return true;
            };
            auto nothing = [] {};
            for (int ti = tile_begin; ti < tile_end && ok; ++ti) {
                const ExtendTile tile = p.tiles[p.cta_tiles[ti]];
                const TileShape sh = tile_shape(tile, tpt);
                ok = mbar_wait_spin(bar(B_QFULL), n_q & 1, &abort_flag);
                ++n_q;
                if (!ok || sh.n_tiles == 0) {
                    if (ok) tc_commit(bar(B_QEMPTY));
                    continue;
                }
                // QK^T still to issue in this tile; Q is released after the last
                int q_left = sh.n_sub[0] + sh.n_sub[1];
                ok = mbar_wait_spin(bar(B_KFULL + kc % C::NSK), (kc / C::NSK) & 1, &abort_flag);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int t = 0; t < 2; ++t)
                    if (sh.n_sub[t] > 0) {
                        qk(t, kc % C::NSK, nothing);
                        if (--q_left == 0) tc_commit(bar(B_QEMPTY));
                    }
                tc_commit(bar(B_KEMPTY + kc % C::NSK));   // K tile 0 read by both QK^T
                ++kc;
                for (int j = 0; j < sh.n_tiles && ok; ++j) {
                    const int sv = vc % C::NSV;
                    const int t_last = j < sh.n_sub[1] ? 1 : 0;   // last sub-tile that reads V tile j
                    const bool k_next = j + 1 < sh.n_tiles;
                    bool k_used = false;
                    if (!v_ready) ok = mbar_wait_spin(bar(B_VFULL + sv), (vc / C::NSV) & 1, &abort_flag);
                    v_ready = false;
#pragma unroll
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (j >= sh.n_sub[t]) continue;
                        // during PV_0: the next K tile; during PV_1: the next V tile
                        if (t == 0)
                            ok = pv(0, sv, j == 0, [&] { if (k_next) poll(k_ready, B_KFULL + kc % C::NSK, (kc / C::NSK) & 1); });
                        else
                            ok = pv(1, sv, j == 0, [&] { poll(v_ready, B_VFULL + (vc + 1) % C::NSV, ((vc + 1) / C::NSV) & 1); });
                        if (!ok) break;
                        if (t == t_last) tc_commit(bar(B_VEMPTY + sv));   // V tile j read by both PV
                        if (j + 1 < sh.n_sub[t]) {
                            if (!k_ready) {
                                ok = mbar_wait_spin(bar(B_KFULL + kc % C::NSK), (kc / C::NSK) & 1, &abort_flag);
                                if (!ok) break;
                                k_ready = true;
                            }
                            k_used = true;
                            tc_fence_after();
                            // overwrites S_t: issued after the PV that reads P_t.
                            // During QK_0 poll P_1 of this step, during QK_1 P_0 of the next
                            if (t == 0)
                                qk(0, kc % C::NSK, [&] { if (j < sh.n_sub[1]) poll(p_ready[1], B_PFULL + 1, pc[1] & 1); });
                            else
                                qk(1, kc % C::NSK, [&] { poll(p_ready[0], B_PFULL + 0, pc[0] & 1); });
                            if (--q_left == 0) tc_commit(bar(B_QEMPTY));
                        } else {
                            tc_commit(bar(B_ODONE + t));
                        }
                    }
                    if (ok && k_used) {
                        tc_commit(bar(B_KEMPTY + kc % C::NSK));   // K tile j+1 read by both QK^T
                        ++kc;
                        k_ready = false;
                    }
                    ++vc;
                }
            }
            if (!ok) raise_abort(&abort_flag, p.err, kErrTimeout);
            // every MMA of this CTA must finish before tensor memory is released
            tc_commit(bar(B_DRAIN));
            if (!mbar_wait(bar(B_DRAIN), 0, nullptr)) atomicOr(p.err, kErrTimeout);
        }
        __syncwarp();
      }
    } else {
        // ------------------------------------------- softmax + epilogue --
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REGS_SOFTMAX));
        const int t = (warp - 4) / 4;            // sub-tile of this warpgroup
        const int quarter = warp & 3;            // tensor-memory lanes 32*quarter .. +31
        const int row = quarter * 32 + lane;
        const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        int scnt = 0, ocnt = 0;                  // S tiles and outputs consumed by this sub-tile
        int vbase = 0;                           // V tiles of the previous tiles of this CTA
        bool ok = true;
        for (int ti = tile_begin; ti < tile_end && ok; ++ti) {
            const ExtendTile tile = p.tiles[p.cta_tiles[ti]];
            const TileShape sh = tile_shape(tile, tpt);
            const int i = t * tpt + row / G;         // token of this row within the tile
            const int gq = row % G;
            // rows past tpt * G (when G does not divide 128) are padding
            const bool tok_valid = row < tpt * G && i < tile.n_tok;
            const int pos_lim = tile.causal ? tile.pos0 + i + 1 : 0x7fffffff;  // keys < pos_lim
            const int row_end = min(tile.key_end, pos_lim);
            const int n_mine = t ? sh.n_sub[1] : sh.n_sub[0];
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < n_mine; ++j) {
                if (!warp_wait(bar(B_SFULL + t), scnt & 1, &abort_flag)) { ok = false; break; }
                ++scnt;
                tc_fence_after();
                const int kt0 = tile.key_begin + j * kTileKeys;
                const int lim = row_end - kt0;       // columns < lim are visible
                // the whole S row in registers: four loads, one wait
                uint32_t sr[128];
                tmem_ld32(t_row + col_s(t) + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                tmem_ld32(t_row + col_s(t) + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                tmem_ld32(t_row + col_s(t) + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
                tmem_ld32(t_row + col_s(t) + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
                tmem_wait_ld();
                if (lim < kTileKeys) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= lim) sr[c] = __float_as_uint(-INFINITY);
                }
                // row max: 3-input max, four chains
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int c = 0; c < 128; c += 8) {
                    mx0 = max3(mx0, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
                    mx1 = max3(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
                    mx2 = max3(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
                    mx3 = max3(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
                }
                const float mxs = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * p.scale_log2;
                const bool need = mxs > m + 8.f;
                float alpha = 1.f;
                if (need) {
                    alpha = ex2(m - mxs);
                    m = mxs;
                    l *= alpha;
                }
                const float nref = m == -INFINITY ? 0.f : -m;
                // P = exp2(s*scale - m) as bf16 pairs, packed in place (entry e
                // takes columns 2e and 2e+1, which are read before entry e is
                // written), then stored over the first 64 columns of S; the
                // scale-and-shift and the row sum run on packed fp32 pairs
                const uint64_t scale2 = f32x2(p.scale_log2, p.scale_log2), shift2 = f32x2(nref, nref);
                uint64_t la = f32x2(0.f, 0.f), lb = la;
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    float x0, x1;
                    f32x2_split(fma_f32x2(f32x2(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])), scale2,
                                          shift2),
                                x0, x1);
                    const float p0 = ex2(x0), p1 = ex2(x1);
                    if (e & 1) lb = add_f32x2(lb, f32x2(p0, p1));
                    else la = add_f32x2(la, f32x2(p0, p1));
                    sr[e] = pack_bf16x2(p0, p1);
                }
                float a0, a1, b0, b1;
                f32x2_split(la, a0, a1);
                f32x2_split(lb, b0, b1);
                l += (a0 + b0) + (a1 + b1);
                tmem_st32(t_row + col_s(t) + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                tmem_st32(t_row + col_s(t) + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                if (j >= 1 && __any_sync(0xffffffffu, need)) {
                    // O_t holds the tiles before j (their PV completed before S_t(j) did)
#pragma unroll 1
                    for (int c = 0; c < D; c += 32) {
                        uint32_t orr[32];
                        tmem_ld32(t_row + col_o(t) + c, orr);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                        tmem_st32(t_row + col_o(t) + c, orr);
                    }
                }
                tmem_wait_st();
                // value rows past the end of the key range may hold anything
                // (unwritten slots, stale blocks, NaN): zero them so that
                // 0 * row stays 0 inside the MMA.  Each sub-tile that reads
                // the last V tile zeroes them before handing over its P, so
                // the PV after it sees zeros (both write the same zeros).
                const int valid_keys = tile.key_end - kt0;
                if (valid_keys < kTileKeys && j == sh.n_tiles - 1) {
                    const int vi = vbase + j;
                    const int s = vi % C::NSV;
                    if (!warp_wait(bar(B_VFULL + s), (vi / C::NSV) & 1, &abort_flag)) { ok = false; break; }
                    if (row >= valid_keys) {
#pragma unroll
                        for (int h = 0; h < C::NH; ++h)
#pragma unroll
                            for (int ch = 0; ch < 8; ++ch) {
                                const uint32_t a = v_s(s) + h * C::HALF + row * 128 + ch * 16;
                                asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
                            }
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                mbar_arrive(bar(B_PFULL + t));
            }
            if (!ok) break;
            vbase += sh.n_tiles;
            // ------------------------------------------------- epilogue --
            if (n_mine == 0) continue;
            if (!warp_wait(bar(B_ODONE + t), ocnt & 1, &abort_flag)) { ok = false; break; }
            ++ocnt;
            tc_fence_after();
            const float inv = l > 0.f ? p.out_scale / l : 0.f;
            const int tok = tile.t0 + i;
            const int h = tile.kv_head * G + gq;
            int64_t slot = -1;
            if (tile.part >= 0 && tok_valid)
                slot = static_cast<int64_t>(p.part_offset[tok * p.n_groups + tile.kv_head / p.heads_per_group]) +
                       tile.part;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t orr[32];
                tmem_ld32(t_row + col_o(t) + c, orr);
                tmem_wait_ld();
                if (!tok_valid) continue;
                if (tile.part < 0) {
                    uint16_t *dst = p.out + (static_cast<int64_t>(tok) * p.num_heads_q + h) * D + c;
#pragma unroll
                    for (int q8 = 0; q8 < 2; ++q8) {
                        uint32_t w[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            w[e] = pack_bf16x2(__uint_as_float(orr[q8 * 16 + 2 * e]) * inv,
                                               __uint_as_float(orr[q8 * 16 + 2 * e + 1]) * inv);
                        st_global_v8(dst + q8 * 16, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
                    }
                } else {
                    float *dst = p.o_part + (slot * p.num_heads_q + h) * D + c;
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8)
                        st_global_v8(dst + q8 * 8, __float_as_uint(__uint_as_float(orr[q8 * 8 + 0]) * inv),
                                     __float_as_uint(__uint_as_float(orr[q8 * 8 + 1]) * inv),
                                     __float_as_uint(__uint_as_float(orr[q8 * 8 + 2]) * inv),
                                     __float_as_uint(__uint_as_float(orr[q8 * 8 + 3]) * inv),
                                     __float_as_uint(__uint_as_float(orr[q8 * 8 + 4]) * inv),
                                     __float_as_uint(__uint_as_float(orr[q8 * 8 + 5]) * inv),
                                     __float_as_uint(__uint_as_float(orr[q8 * 8 + 6]) * inv),
                                     __float_as_uint(__uint_as_float(orr[q8 * 8 + 7]) * inv));
                }
            }
            if (tok_valid && tile.part >= 0) p.ml_part[slot * p.num_heads_q + h] = make_float2(m, l);
            tc_fence_before();
        }
        if (!ok) raise_abort(&abort_flag, p.err, kErrTimeout);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D>
cudaError_t configure() {
    static bool configured = false;  // attribute is per function, set once per process
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(extend_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             ExtCfg<D>::SMEM);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return cudaSuccess;
}

template <int D>
cudaError_t launch_t(int grid, const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                     const ExtendParams &p, cudaStream_t stream, bool pdl) {
    using C = ExtCfg<D>;
    cudaError_t e = configure<D>();
    if (e != cudaSuccess) return e;
    return launch_ex(extend_kernel<D>, dim3(grid), dim3(C::THREADS), C::SMEM, stream, pdl, tm_q, tm_k, tm_v, p);
}

}  // namespace

cudaError_t prepare_extend(int head_dim) {
    if (head_dim == 128) return configure<128>();
    if (head_dim == 64) return configure<64>();
    return cudaErrorInvalidValue;
}

cudaError_t launch_extend(int head_dim, int grid, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                          const CUtensorMap &tm_v, const ExtendParams &p, cudaStream_t stream, bool pdl) {
    if (grid <= 0) return cudaSuccess;
    if (head_dim == 128) return launch_t<128>(grid, tm_q, tm_k, tm_v, p, stream, pdl);
    if (head_dim == 64) return launch_t<64>(grid, tm_q, tm_k, tm_v, p, stream, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace pa
