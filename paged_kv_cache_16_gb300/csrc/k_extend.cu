// Extend / chunked-prefill attention tile on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), and the shared-prefix stage of
// the cascade route.
//
// What one CTA computes (page "vLLM 推理流程分析" §6.2: varlen causal
// attention through block_table; §10.1: a token sees itself and earlier
// tokens; §5.1.2: positions = num_computed + offset in the chunk):
//   128 query rows = 128/G consecutive tokens x the G query heads of one kv
//   head, against keys [key_begin, key_end) of one request's context, read
//   through the block table in tiles of 128 keys (8 blocks).  Row (i, g) at
//   absolute position pos0 + i sees key j iff j <= pos0 + i (causal tiles);
//   shared-prefix tiles see their whole key range.
//
// Per 128-key tile:  S = Q K^T   (tcgen05.mma, M=128 N=128 K=D, S in TMEM)
//                    P = exp2(S*scale*log2e - m)  (4 softmax warps, one row each)
//                    O += P V    (tcgen05.mma, M=128 N=D K=128, O in TMEM)
// Warp roles: warp 0 TMA producer (Q once, K/V blocks into a 2-stage ring),
// warp 1 MMA issuer (one thread) and TMEM owner, warps 2-5 softmax,
// correction and epilogue.  S is double-buffered in TMEM so the QK^T of tile
// j+1 overlaps the softmax of tile j.  The running max is only moved (and O
// rescaled) when it grows by more than 2^8, which keeps every weight <= 256.
//
// Shared memory tiles are 128-byte-swizzled [rows][64 elements] halves:
//   Q  (A, K-major), K (B, K-major), P (A, K-major), V (B, MN-major).
#include "dev.cuh"

namespace pa {
namespace {

using namespace dev;

template <int D>
struct ExtCfg {
    static constexpr int NH = D / 64;
    static constexpr int HALF = 128 * 128;            // [128 rows][64] bf16 half tile
    static constexpr int QB = NH * HALF;              // Q tile bytes
    static constexpr int KVB = NH * HALF;             // K (or V) tile bytes per stage
    static constexpr int PB = 2 * HALF;               // P tile: 128 rows x 128 keys
    static constexpr int NS = 2;
    static constexpr int THREADS = 192;
    static constexpr int TILE_SMEM = QB + NS * 2 * KVB + PB;
    // keep one CTA per SM: it owns all 512 TMEM columns
    static constexpr int SMEM = (TILE_SMEM + 2048 < 120 * 1024) ? 120 * 1024 : TILE_SMEM + 2048;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_O = 256;
    static constexpr uint32_t IDESC_QK = idesc_bf16(128, 128, false, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
};

// barrier indices
enum : int {
    B_Q = 0,
    B_KFULL = 1,   // +stage
    B_VFULL = 3,   // +stage
    B_KVEMPTY = 5, // +stage
    B_SFULL = 7,   // +buffer
    B_SFREE = 9,   // +buffer
    B_PFULL = 11,
    B_ODONE = 12,
    B_DRAIN = 13,
    NUM_BARS = 14
};

template <int D>
__global__ void __launch_bounds__(192, 1)
extend_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const ExtendParams p) {
    using C = ExtCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int abort_flag;
    __shared__ uint32_t tmem_base_slot;
    __shared__ __align__(8) uint64_t bars[NUM_BARS];

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t q_s = base;
    auto k_s = [&](int s) { return base + C::QB + static_cast<uint32_t>(s) * 2 * C::KVB; };
    auto v_s = [&](int s) { return k_s(s) + C::KVB; };
    const uint32_t p_s = base + C::QB + C::NS * 2 * C::KVB;
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const ExtendTile tile = p.tiles[blockIdx.x];
    const int G = p.group;
    const int n_tiles = (tile.key_end - tile.key_begin + kTileKeys - 1) / kTileKeys;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bar(B_KFULL + s), 1);
            mbar_init(bar(B_VFULL + s), 1);
            mbar_init(bar(B_KVEMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_SFULL + b), 1);
            mbar_init(bar(B_SFREE + b), 128);
        }
        mbar_init(bar(B_PFULL), 128);
        mbar_init(bar(B_ODONE), 1);
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

    if (warp == 0) {
        // -------------------------------------------------------- producer --
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            mbar_arrive_expect_tx(bar(B_Q), C::QB);
        }
        __syncwarp();
        if (lane < C::NH)
            tma_load_3d(q_s + lane * C::HALF, &tm_q, lane * 64, tile.kv_head * G, tile.t0, bar(B_Q));
        const int32_t *bt = p.block_table + static_cast<int64_t>(tile.req) * p.max_blocks;
        int issued = 0;
        for (int j = 0; j < n_tiles; ++j) {
            const int s = j % C::NS;
            const int n = j / C::NS;
            if (n > 0 && !warp_wait(bar(B_KVEMPTY + s), (n & 1) ^ 1, &abort_flag)) {
                if (lane == 0) raise_abort(&abort_flag, p.err, kErrTimeout);
                break;
            }
            const int kt0 = tile.key_begin + j * kTileKeys;
            const int pages = min(8, (tile.key_end - kt0 + kBlockSize - 1) / kBlockSize);
            int32_t blk = 0;
            bool valid = false;
            if (lane < pages) {
                blk = bt[kt0 / kBlockSize + lane];
                valid = blk >= 0 && blk < p.num_blocks;
            }
            const unsigned vmask = __ballot_sync(0xffffffffu, valid);
            if (lane == 0) {
                if (__popc(vmask) != pages) atomicOr(p.err, kErrBlockRange);
                const uint32_t bytes = __popc(vmask) * kBlockSize * 128 * C::NH;
                mbar_arrive_expect_tx(bar(B_KFULL + s), bytes);
                mbar_arrive_expect_tx(bar(B_VFULL + s), bytes);
            }
            __syncwarp();
            static_assert(2 * 8 * C::NH <= 32, "one TMA box per lane");
            {
                const int tensor = lane / (8 * C::NH);
                const int rem = lane % (8 * C::NH);
                const int page = rem / C::NH;
                const int half = rem % C::NH;
                const int32_t b = __shfl_sync(0xffffffffu, blk, page);  // every lane takes part
                if (lane < 2 * 8 * C::NH && ((vmask >> page) & 1u)) {
                    const uint32_t dst = (tensor ? v_s(s) : k_s(s)) + half * C::HALF + page * 2048;
                    tma_load_3d(dst, tensor ? &tm_v : &tm_k, half * 64, tile.kv_head, b * kBlockSize,
                                bar(tensor ? B_VFULL + s : B_KFULL + s));
                }
            }
            ++issued;
        }
        if (lane == 0) {
            // no TMA write may outlive the CTA
            if (!mbar_wait(bar(B_Q), 0, nullptr)) atomicOr(p.err, kErrTimeout);
            for (int k = issued - 1; k >= 0 && k >= issued - C::NS; --k) {
                const int s = k % C::NS, n = k / C::NS;
                if (!mbar_wait(bar(B_KFULL + s), n & 1, nullptr) ||
                    !mbar_wait(bar(B_VFULL + s), n & 1, nullptr))
                    atomicOr(p.err, kErrTimeout);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer --
        if (lane == 0) {
            bool ok = mbar_wait(bar(B_Q), 0, &abort_flag);
            tc_fence_after();
            auto pv = [&](int jj) -> bool {
                const int s = jj % C::NS;
                if (!mbar_wait(bar(B_PFULL), jj & 1, &abort_flag)) return false;
                if (!mbar_wait(bar(B_VFULL + s), (jj / C::NS) & 1, &abort_flag)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kTileKeys / 16; ++kk) {
                    const uint64_t a = sdesc_sw128(p_s + (kk / 4) * C::HALF + (kk % 4) * 32, 16, 1024);
                    const uint64_t b = sdesc_sw128(v_s(s) + kk * 2048, C::HALF, 1024);
                    tc_mma(tmem + C::COL_O, a, b, C::IDESC_PV, (jj > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar(B_ODONE));
                tc_commit(bar(B_KVEMPTY + s));
                return true;
            };
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int s = j % C::NS;
                const int sb = j & 1;
                ok = mbar_wait(bar(B_KFULL + s), (j / C::NS) & 1, &abort_flag);
                if (ok && j >= 2) ok = mbar_wait(bar(B_SFREE + sb), ((j >> 1) - 1) & 1, &abort_flag);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t a = sdesc_sw128(q_s + (kk / 4) * C::HALF + (kk % 4) * 32, 16, 1024);
                    const uint64_t b = sdesc_sw128(k_s(s) + (kk / 4) * C::HALF + (kk % 4) * 32, 16, 1024);
                    tc_mma(tmem + sb * 128, a, b, C::IDESC_QK, kk > 0 ? 1u : 0u);
                }
                tc_commit(bar(B_SFULL + sb));
                if (j >= 1) ok = pv(j - 1);
            }
            if (ok && n_tiles > 0) ok = pv(n_tiles - 1);
            if (!ok) raise_abort(&abort_flag, p.err, kErrTimeout);
            // every MMA of this CTA must finish before TMEM is released
            tc_commit(bar(B_DRAIN));
            if (!mbar_wait(bar(B_DRAIN), 0, nullptr)) atomicOr(p.err, kErrTimeout);
        }
        __syncwarp();
    } else {
        // ------------------------------------------- softmax + epilogue --
        const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31
        const int row = quarter * 32 + lane;
        const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const int i = row / G;
        const int gq = row % G;
        const bool tok_valid = i < tile.n_tok;
        const int pos_lim = tile.causal ? tile.pos0 + i + 1 : 0x7fffffff;  // keys < pos_lim
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const int sb = j & 1;
            const int s = j % C::NS;
            if (!warp_wait(bar(B_SFULL + sb), (j >> 1) & 1, &abort_flag)) { ok = false; break; }
            tc_fence_after();
            uint32_t sr[128];
            tmem_ld32(t_row + sb * 128 + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
            tmem_ld32(t_row + sb * 128 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
            tmem_ld32(t_row + sb * 128 + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
            tmem_ld32(t_row + sb * 128 + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar(B_SFREE + sb));

            const int kt0 = tile.key_begin + j * kTileKeys;
            const int lim = min(tile.key_end, pos_lim) - kt0;   // columns < lim are visible
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 128; ++c) {
                const float v = c < lim ? __uint_as_float(sr[c]) * p.scale_log2 : -INFINITY;
                sr[c] = __float_as_uint(v);
                mx = fmaxf(mx, v);
            }
            const bool need = mx > m + 8.f;
            float alpha = 1.f;
            if (need) {
                alpha = ex2(m - mx);
                m = mx;
                l *= alpha;
            }
            const float ref = m == -INFINITY ? 0.f : m;
            if (j >= 1) {
                // PV of the previous tile must be done: O is final for it and
                // the P buffer is free again
                if (!warp_wait(bar(B_ODONE), (j - 1) & 1, &abort_flag)) { ok = false; break; }
                tc_fence_after();
                if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
                    for (int c = 0; c < D; c += 32) {
                        uint32_t orr[32];
                        tmem_ld32(t_row + C::COL_O + c, orr);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                        tmem_st32(t_row + C::COL_O + c, orr);
                    }
                    tmem_wait_st();
                }
            }
            // P row -> shared memory (bf16, 128-byte swizzled, K-major)
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    w[e] = pack_bf16x2(ex2(__uint_as_float(sr[c * 8 + 2 * e]) - ref),
                                       ex2(__uint_as_float(sr[c * 8 + 2 * e + 1]) - ref));
                    l += bf16_lo(w[e]) + bf16_hi(w[e]);
                }
                const uint32_t a = sw128(p_s + (c / 8) * C::HALF, row, c % 8);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w[0]), "r"(w[1]),
                             "r"(w[2]), "r"(w[3])
                             : "memory");
            }
            // value rows past the end of the key range may hold anything
            // (unwritten slots, stale blocks, NaN): zero them so that
            // 0 * row stays 0 inside the MMA
            const int valid_keys = tile.key_end - kt0;
            if (valid_keys < kTileKeys) {
                if (!warp_wait(bar(B_VFULL + s), (j / C::NS) & 1, &abort_flag)) { ok = false; break; }
                if (row >= valid_keys) {
#pragma unroll
                    for (int h = 0; h < C::NH; ++h)
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            const uint32_t a = v_s(s) + h * C::HALF + row * 128 + ch * 16;
                            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0)
                                         : "memory");
                        }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B_PFULL));
        }
        if (!ok) raise_abort(&abort_flag, p.err, kErrTimeout);
        // ----------------------------------------------------- epilogue --
        if (ok && n_tiles > 0 && warp_wait(bar(B_ODONE), (n_tiles - 1) & 1, &abort_flag)) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int t = tile.t0 + i;
            const int h = tile.kv_head * G + gq;
            int64_t slot = -1;
            if (tile.part >= 0 && tok_valid)
                slot = static_cast<int64_t>(p.part_offset[t * p.n_groups + tile.kv_head / p.heads_per_group]) +
                       tile.part;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t orr[32];
                tmem_ld32(t_row + C::COL_O + c, orr);
                tmem_wait_ld();
                if (!tok_valid) continue;
                if (tile.part < 0) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out + (static_cast<int64_t>(t) * p.num_heads_q + h) * D + c);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(orr[q4 * 8 + 0]) * inv, __uint_as_float(orr[q4 * 8 + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(orr[q4 * 8 + 2]) * inv, __uint_as_float(orr[q4 * 8 + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(orr[q4 * 8 + 4]) * inv, __uint_as_float(orr[q4 * 8 + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(orr[q4 * 8 + 6]) * inv, __uint_as_float(orr[q4 * 8 + 7]) * inv);
                        dst[q4] = w;
                    }
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(p.o_part + (slot * p.num_heads_q + h) * D + c);
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4)
                        dst[q4] = make_float4(__uint_as_float(orr[q4 * 4 + 0]) * inv, __uint_as_float(orr[q4 * 4 + 1]) * inv,
                                              __uint_as_float(orr[q4 * 4 + 2]) * inv, __uint_as_float(orr[q4 * 4 + 3]) * inv);
                }
            }
            if (tok_valid && tile.part >= 0) p.ml_part[slot * p.num_heads_q + h] = make_float2(m, l);
        } else if (n_tiles > 0) {
            raise_abort(&abort_flag, p.err, kErrTimeout);
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D>
cudaError_t launch_t(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                     const ExtendParams &p, cudaStream_t stream) {
    using C = ExtCfg<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(extend_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    extend_kernel<D><<<p.num_tiles, C::THREADS, C::SMEM, stream>>>(tm_q, tm_k, tm_v, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_extend(int head_dim, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                          const CUtensorMap &tm_v, const ExtendParams &p, cudaStream_t stream) {
    if (p.num_tiles <= 0) return cudaSuccess;
    if (head_dim == 128) return launch_t<128>(tm_q, tm_k, tm_v, p, stream);
    if (head_dim == 64) return launch_t<64>(tm_q, tm_k, tm_v, p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
