// Short-query GDPA forward: O = act(scale Q K^T) V for batches whose query sets each fit one
// query tile (bf16 inputs, GDPA modes, no bias, no causal mask or window).
//
// GDPA replaces the softmax by an element-wise activation with no row statistics (aihot.vn
// GEM article, "Generalized Dot-Product Attention (GDPA)": two matrix products with an
// activation between them), and its production shapes pair short query sets with long
// key/value histories.  A forward over 128-row query tiles leaves most TMEM lanes on
// padding rows there (a query set of q rows fills q of 128).  Since no statistic runs
// along a query row, this kernel forms the scores transposed instead, with the keys on
// the lanes, so every lane holds a real key row:
//   S^T = K_t Q^T          TMEM, lanes = 128 key rows, BQ query columns (double-buffered)
//   P^T = act(S^T)         two bf16 terms, bf16(P^T) and the remainder, to two shared-memory
//                          tiles (rows = keys), 0 where masked
//   O^T += V_t^T P^T       TMEM, lanes = head-dim rows, over all key tiles: one product of
//                          N = 2 BQ whose B is the two terms' tiles side by side, so V is
//                          read once per K-step; the epilogue adds the two halves
// GDPA's output is a sum over keys with no normalisation, so P's bf16 rounding would add up
// over a long key range; the second term carries P to about 16 significant bits, as in the
// query-tile forward.
// and writes O (the transpose of O^T) once per item.  Item = (sequence, head) with all of
// its key tiles; the query set's Q rows stay in shared memory.
// O^T's product has M = 128 lanes; at head_dim 64 the V tile has one 64-column block and the
// descriptor's block stride is 0, so lanes 64-127 repeat lanes 0-63 and are not written out.
// TMEM: S^T [0, BQ) and [BQ, 2 BQ), O^T [2 BQ, 4 BQ) (high term's columns, then the low
// term's): 256 columns at BQ = 64 (two CTAs share an SM), 512 at BQ = 128.
//
// CTA = BQ/32 activation warpgroups (thread = key row = TMEM lane; warpgroup g owns query
// columns [32 g, 32 g + 32); in the epilogue thread = head-dim row, the same columns), then a
// TMA producer warp and an MMA issuer warp: 10 warps at BQ = 64, 18 at BQ = 128, where the
// activation's chain of dependent exponent and reciprocal operations needs the extra warps
// to hide its latency.
#include <algorithm>

#include <cuda_bf16.h>

#include "jfa_internal.h"
#include "ptx.cuh"
#include "tilemath.cuh"

namespace jfa {

namespace {

template <int D, int BQ>
struct FsCfg {
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static_assert(BQ == 64 || BQ == 128, "query tile of 64 or 128 rows");
    static constexpr int BN = kFwdBN;  // key rows per tile
    static constexpr int kRowBytes = D * 2;
    static constexpr int kCB = kRowBytes / 128;  // 128-byte column blocks of a head row
    static constexpr int kBoxCols = 64;
    static constexpr int kKVTile = BN * kRowBytes;
    static constexpr int kQTile = BQ * kRowBytes;
    // P^T tiles (the high and low bf16 terms), bf16 [BN keys][BQ queries] as 64-query column
    // blocks of BN x 128 bytes, 128-byte swizzled: the MN-major B of O^T's product.
    static constexpr int kPTile = BN * BQ * 2;
    static constexpr int WG = BQ / 32;  // activation warpgroups, 32 query columns each
    static constexpr int kCompWarps = 4 * WG;
    static constexpr int kOffK = 0;  // two stages
    static constexpr int kOffV = 2 * kKVTile;  // two stages
    static constexpr int kOffQ = 4 * kKVTile;
    static constexpr int kOffP = kOffQ + kQTile;
    static constexpr int kOffBar = kOffP + 2 * kPTile;
    static constexpr int kNumBars = 20;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemNeed = kOffMisc + 16 + 1024;  // tmem slot, abort flag; alignment of the base
    static constexpr int kCols = 32;  // query columns per thread
    static constexpr uint32_t kTmS = 0, kTmO = 2 * BQ;
    static constexpr uint32_t kTmCols = 4 * BQ <= 256 ? 256 : 512;
    // Two CTAs per SM where TMEM and shared memory allow it; otherwise shared memory keeps a
    // second CTA off the SM (it would wait on the TMEM allocation).
    static constexpr int kCtasPerSm = (kTmCols == 256 && 2 * (kSmemNeed + 1024) <= 228 * 1024) ? 2 : 1;
    static constexpr int kSmemBytes = (kCtasPerSm == 1 && kSmemNeed < 120 * 1024) ? 120 * 1024 : kSmemNeed;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static constexpr uint32_t kIdescS = make_idesc(kFmtBF16, BN, BQ, false, false);
    static constexpr uint32_t kIdescO = make_idesc(kFmtBF16, 128, 2 * BQ, true, true);
    static constexpr int kProdWarp = kCompWarps, kMmaWarp = kCompWarps + 1, kThreads = (kCompWarps + 2) * 32;
};

enum {
    FS_K_FULL = 0,   // +stage
    FS_K_EMPTY = 2,  // +stage
    FS_V_FULL = 4,   // +stage
    FS_V_EMPTY = 6,  // +stage
    FS_Q_FULL = 8,
    FS_Q_EMPTY = 9,
    FS_S_FULL = 10,   // +buffer
    FS_S_FREE = 12,   // +buffer: every activation warp has read the S^T buffer
    FS_P_FULL = 14,   // every activation warp has written its rows of the P^T tiles
    FS_P_FREE = 15,   // O^T's product has read the P^T tiles
    FS_O_FULL = 16,   // the item's last O^T product is done
    FS_O_EMPTY = 17,  // every warp has read O^T
    FS_DRAIN = 18,
};

// GELU: the activation is tanh-GELU, else SiLU (a template parameter, so that the activation
// pass is straight-line code).
template <int D, int BQ, typename OT, bool GELU>
__global__ void __launch_bounds__(FsCfg<D, BQ>::kThreads, FsCfg<D, BQ>::kCtasPerSm)
    jfa_fwd_short_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using C = FsCfg<D, BQ>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sK = sbase + C::kOffK, sV = sbase + C::kOffV, sQ = sbase + C::kOffQ, sP = sbase + C::kOffP;
    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * uint32_t(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(FS_K_FULL + s), 1);
            mbar_init(bar(FS_K_EMPTY + s), 1);
            mbar_init(bar(FS_V_FULL + s), 1);
            mbar_init(bar(FS_V_EMPTY + s), 1);
            mbar_init(bar(FS_S_FULL + s), 1);
            mbar_init(bar(FS_S_FREE + s), C::kCompWarps);
        }
        mbar_init(bar(FS_Q_FULL), 1);
        mbar_init(bar(FS_Q_EMPTY), 1);
        mbar_init(bar(FS_P_FULL), C::kCompWarps);
        mbar_init(bar(FS_P_FREE), 1);
        mbar_init(bar(FS_O_FULL), 1);
        mbar_init(bar(FS_O_EMPTY), C::kCompWarps);
        mbar_init(bar(FS_DRAIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == C::kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmCols);
        tmem_relinquish();
    }
    if (warp == C::kProdWarp && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int it_begin = p.cta_off[blockIdx.x];
    const int it_end = p.cta_off[blockIdx.x + 1];
    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(p.status, kStatusTimeout);
    };
    auto warp_wait = [&](int b, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait_bounded(bar(b), parity, abort_flag));
    };

    if (warp == C::kProdWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t kv_it = 0, item_it = 0;
            uint32_t k_extra = 0;  // 1: the last K load went out but its V load did not
            bool ok = true;
            auto load_kv = [&](int h, int row) -> bool {
                const uint32_t st = kv_it & 1, ph = ((kv_it >> 1) & 1) ^ 1;
                if (!mbar_wait_bounded(bar(FS_K_EMPTY + st), ph, abort_flag)) return false;
                mbar_arrive_expect_tx(bar(FS_K_FULL + st), C::kKVTile);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb)
                    tma_load_2d(sK + st * C::kKVTile + cb * C::BN * 128, &tmK, bar(FS_K_FULL + st),
                                h * D + cb * C::kBoxCols, row);
                if (!mbar_wait_bounded(bar(FS_V_EMPTY + st), ph, abort_flag)) {
                    k_extra = 1;
                    return false;
                }
                mbar_arrive_expect_tx(bar(FS_V_FULL + st), C::kKVTile);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb)
                    tma_load_2d(sV + st * C::kKVTile + cb * C::BN * 128, &tmV, bar(FS_V_FULL + st),
                                h * D + cb * C::kBoxCols, row);
                ++kv_it;
                return true;
            };
            for (int it = it_begin; it < it_end && ok; ++it) {
                const int4 w = p.items[it];
                if (!short_fwd_item_ok(w, p, BQ)) {  // not an item of this plan: skipped by every role
                    atomicOr(p.status, kStatusBounds);
                    continue;
                }
                const int b = w.x, h = w.y, n = w.w;
                const int q0 = p.q_off[b], q_len = p.q_off[b + 1] - q0, kv0 = p.kv_off[b];
                if (q_len == 0 || n == 0) continue;  // nothing to read
                if (!load_kv(h, kv0)) { ok = false; break; }
                if (!mbar_wait_bounded(bar(FS_Q_EMPTY), (item_it & 1) ^ 1, abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(FS_Q_FULL), C::kQTile);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb)
                    tma_load_2d(sQ + cb * BQ * 128, &tmQ, bar(FS_Q_FULL), h * D + cb * C::kBoxCols, q0);
                ++item_it;
                for (int t = 1; t < n; ++t)
                    if (!load_kv(h, kv0 + t * C::BN)) { ok = false; break; }
            }
            if (!ok) fail();
            // Drain: wait until every load this thread issued has landed.
            drain_ring(bar(FS_Q_FULL), item_it, 1);
            drain_ring(bar(FS_K_FULL), kv_it + k_extra, 2);
            drain_ring(bar(FS_V_FULL), kv_it, 2);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        uint32_t kv_it = 0, item_it = 0;
        bool ok = true;
        const SDesc dQk = sdesc_sw128(sQ, 16, 1024);
        // O^T = V^T P^T: V as an MN-major A over 128 head-dim lanes (64-column blocks BN * 128
        // bytes apart; one block at head_dim 64, read for both halves), the P^T tile as an
        // MN-major B (64-query blocks BN * 128 bytes apart).
        // both terms' tiles as one B of 2 BQ columns: 64-query blocks BN * 128 bytes apart, the
        // low term's right after the high term's
        const SDesc dPm = sdesc_sw128(sP, C::BN * 128, 1024);
        auto koff = [](int s, int rows) -> uint32_t {
            return uint32_t(((s * 32) >> 7) * rows * 128 + ((s * 32) & 127));
        };
        // S^T(g) = K Q^T into buffer g & 1, once the activation warps have read it two tiles ago.
        auto issue_s = [&](uint32_t g, bool last_of_item) -> bool {
            const uint32_t st = g & 1;
            if (!warp_wait(FS_K_FULL + st, (g >> 1) & 1)) return false;
            if (g >= 2 && !warp_wait(FS_S_FREE + st, ((g >> 1) - 1) & 1)) return false;
            tc_fence_after();
            if (elect_one()) {
                const SDesc ka = sdesc_sw128(sK + st * C::kKVTile, 16, 1024);
#pragma unroll
                for (int s = 0; s < D / 16; ++s)
                    mma_ss(tmem + C::kTmS + st * BQ, ka, koff(s, C::BN), dQk, koff(s, BQ), C::kIdescS, s > 0);
                tc_commit(bar(FS_S_FULL + st));
                tc_commit(bar(FS_K_EMPTY + st));
                if (last_of_item) tc_commit(bar(FS_Q_EMPTY));
            }
            __syncwarp();
            return true;
        };
        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 w = p.items[it];
            if (!short_fwd_item_ok(w, p, BQ)) continue;
            const int b = w.x, n = w.w;
            const int q_len = p.q_off[b + 1] - p.q_off[b];
            if (q_len == 0 || n == 0) continue;
            if (!warp_wait(FS_Q_FULL, item_it & 1)) { ok = false; break; }
            const uint32_t g0 = kv_it;
            if (!issue_s(g0, n == 1)) { ok = false; break; }
            for (int t = 0; t < n && ok; ++t) {
                const uint32_t g = g0 + uint32_t(t), st = g & 1;
                // the next tile's scores run while the activation warps work on this one
                if (t + 1 < n && !issue_s(g + 1, t + 2 == n)) { ok = false; break; }
                // O^T += V^T P^T once the P^T tile is written; the item's first product also
                // waits for the previous item's O^T to have been read out.
                if (!warp_wait(FS_V_FULL + st, (g >> 1) & 1) || !warp_wait(FS_P_FULL, g & 1)) { ok = false; break; }
                if (t == 0 && item_it > 0 && !warp_wait(FS_O_EMPTY, (item_it - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                if (elect_one()) {
                    const SDesc va = sdesc_sw128(sV + st * C::kKVTile, D == 128 ? C::BN * 128 : 0, 1024);
#pragma unroll
                    for (int s = 0; s < C::BN / 16; ++s)
                        mma_ss(tmem + C::kTmO, va, uint32_t(s) * 2048u, dPm, uint32_t(s) * 2048u, C::kIdescO,
                               t > 0 || s > 0);
                    tc_commit(bar(FS_P_FREE));
                    tc_commit(bar(FS_V_EMPTY + st));
                    if (t == n - 1) tc_commit(bar(FS_O_FULL));
                }
                __syncwarp();
            }
            if (!ok) break;
            kv_it += uint32_t(n);
            ++item_it;
        }
        if (!ok) fail();
        if (elect_one()) tc_commit(bar(FS_DRAIN));
        __syncwarp();
        mbar_wait_bounded(bar(FS_DRAIN), 0, nullptr);
    } else {
        // ------------------------------------------------------------ activation, epilogue
        constexpr int NC = C::kCols;
        constexpr int NK = NC / 32;
        const int wg = warp >> 2, quarter = warp & 3;
        const int r = quarter * 32 + lane;  // key row of a tile; head-dim row in the epilogue
        const int c0 = wg * NC;
        const uint32_t lane_base = uint32_t(quarter * 32) << 16;
        const size_t row_stride = size_t(p.H) * D;
        uint32_t kv_it = 0, item_it = 0;
        bool ok = true;
        // this thread's 16-byte piece q (0..3) of chunk k in its row of the P^T tile
        auto p_addr = [&](int k, int q) -> uint32_t {
            const int c = c0 + 32 * k;
            const int piece = (c & 63) / 8 + q;
            return sP + uint32_t((c >> 6) * C::BN * 128 + r * 128 + ((piece ^ (r & 7)) << 4));
        };
        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 w = p.items[it];
            if (!short_fwd_item_ok(w, p, BQ)) continue;
            const int b = w.x, h = w.y, n = w.w;
            const int q0 = p.q_off[b], q_len = p.q_off[b + 1] - q0;
            const int kv0 = p.kv_off[b], kv_len = p.kv_off[b + 1] - kv0;
            (void)kv0;
            if (q_len == 0) continue;
            OT* o_item = reinterpret_cast<OT*>(p.O) + (size_t(q0) * size_t(p.H) + size_t(h)) * D;
            if (n == 0) {  // no key: O = 0; thread = head-dim row r, its warpgroup's query rows
                if (r < D)
                    for (int q = c0; q < min(q_len, c0 + NC); ++q) o_item[size_t(q) * row_stride + r] = OT(0.f);
                continue;
            }
            const int hi_q = min(NC, max(0, q_len - c0));  // valid local query columns [0, hi_q)
            for (int t = 0; t < n; ++t, ++kv_it) {
                const uint32_t g = kv_it, st = g & 1;
                const int hi = (t * C::BN + r < kv_len) ? hi_q : 0;
                const bool full = __all_sync(0xffffffffu, hi == NC);
                bool zc[NK];
#pragma unroll
                for (int k = 0; k < NK; ++k) zc[k] = !full && __all_sync(0xffffffffu, hi <= 32 * k);
                if (!warp_wait(FS_S_FULL + st, (g >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                uint32_t pk[NK][16], pl[NK][16];  // bf16(P^T) and the remainder
#pragma unroll
                for (int k = 0; k < NK; ++k) {
                    if (zc[k]) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) pk[k][c] = pl[k][c] = 0u;
                        continue;
                    }
                    float sv[32];
                    {
                        uint32_t (&ra)[32] = *reinterpret_cast<uint32_t(*)[32]>(sv);
                        tmem_ld32(tmem + lane_base + C::kTmS + st * BQ + uint32_t(c0 + 32 * k), ra);
                        tmem_ld_wait(ra);
                    }
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const int cc = 32 * k + c;
                        float2 a = gdpa_act2<GELU>(make_float2(sv[c], sv[c + 1]), p.scale);
                        if (!full) a = make_float2(cc < hi ? a.x : 0.f, cc + 1 < hi ? a.y : 0.f);
                        const uint32_t u = pack_bf16x2(a.x, a.y);
                        pk[k][c >> 1] = u;
                        const float2 rem =
                            add2(a, make_float2(-__uint_as_float(u << 16), -__uint_as_float(u & 0xffff0000u)));
                        pl[k][c >> 1] = pack_bf16x2(rem.x, rem.y);
                    }
                }
                // the S^T buffer is read: the tile after next may score into it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(FS_S_FREE + st));
                // P^T into the shared tile once the previous tile's O^T product has read it
                if (g > 0 && !warp_wait(FS_P_FREE, (g - 1) & 1)) { ok = false; break; }
#pragma unroll
                for (int k = 0; k < NK; ++k)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        st_shared_v4(p_addr(k, q), pk[k][4 * q], pk[k][4 * q + 1], pk[k][4 * q + 2], pk[k][4 * q + 3]);
                        st_shared_v4(p_addr(k, q) + C::kPTile, pl[k][4 * q], pl[k][4 * q + 1], pl[k][4 * q + 2],
                                     pl[k][4 * q + 3]);
                    }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(FS_P_FULL));
            }
            if (!ok) break;
            // O = (O^T)^T: thread = head-dim row r (lanes past D repeat lower ones), its
            // warpgroup's query columns; each store instruction writes one query row's D/32
            // consecutive elements across the warp.
            if (!warp_wait(FS_O_FULL, item_it & 1)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < NK; ++k) {
                if (32 * k >= hi_q) break;
                uint32_t ov[32], ol[32];
                tmem_ld32(tmem + lane_base + C::kTmO + uint32_t(c0 + 32 * k), ov);
                tmem_ld32(tmem + lane_base + C::kTmO + uint32_t(BQ + c0 + 32 * k), ol);
                tmem_ld_wait(ov);
                tmem_ld_wait(ol);
                if (r < D) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const int q = c0 + 32 * k + c;
                        if (q < q_len)
                            o_item[size_t(q) * row_stride + r] = OT(__uint_as_float(ov[c]) + __uint_as_float(ol[c]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(FS_O_EMPTY));
            ++item_it;
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kMmaWarp) tmem_dealloc(tmem, C::kTmCols);
}

template <int D, int BQ, typename OT, bool GELU>
cudaError_t launch_fs_a(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const FwdParams& p,
                        int grid, cudaStream_t st) {
    using C = FsCfg<D, BQ>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(jfa_fwd_short_kernel<D, BQ, OT, GELU>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    jfa_fwd_short_kernel<D, BQ, OT, GELU><<<grid, C::kThreads, C::kSmemBytes, st>>>(tmQ, tmK, tmV, p);
    return cudaGetLastError();
}

template <int D, int BQ, typename OT>
cudaError_t launch_fs_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const FwdParams& p,
                        int grid, cudaStream_t st) {
    return p.mode == JFA_GDPA_GELU_TANH ? launch_fs_a<D, BQ, OT, true>(tmQ, tmK, tmV, p, grid, st)
                                        : launch_fs_a<D, BQ, OT, false>(tmQ, tmK, tmV, p, grid, st);
}

template <typename OT>
cudaError_t launch_fs_o(int D, int bq, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                        const FwdParams& p, int grid, cudaStream_t st) {
    if (D == 64 && bq == 64) return launch_fs_t<64, 64, OT>(tmQ, tmK, tmV, p, grid, st);
    if (D == 64 && bq == 128) return launch_fs_t<64, 128, OT>(tmQ, tmK, tmV, p, grid, st);
    if (D == 128 && bq == 128) return launch_fs_t<128, 128, OT>(tmQ, tmK, tmV, p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace

int short_fwd_ctas_per_sm(int D, int bq) {
    if (D == 64 && bq == 64) return FsCfg<64, 64>::kCtasPerSm;
    if (D == 64 && bq == 128) return FsCfg<64, 128>::kCtasPerSm;
    if (D == 128 && bq == 128) return FsCfg<128, 128>::kCtasPerSm;
    return 0;
}

cudaError_t launch_fwd_short(int o_dtype, int D, int bq, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                             const CUtensorMap& tmV, const FwdParams& p, int grid, cudaStream_t st) {
    if (p.mode == JFA_SOFTMAX) return cudaErrorInvalidValue;
    if (o_dtype == JFA_BF16) return launch_fs_o<__nv_bfloat16>(D, bq, tmQ, tmK, tmV, p, grid, st);
    if (o_dtype == JFA_F32) return launch_fs_o<float>(D, bq, tmQ, tmK, tmV, p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace jfa
