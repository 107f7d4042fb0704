// Short-query backward: dQ, dK and dV in one pass for batches whose query sets each fit
// one query tile (bf16 inputs).
//
// The GEM articles' cross-attention and GDPA shapes pair short query sets with long
// key/value histories (aihot.vn GEM article, "Generalized Dot-Product Attention (GDPA)":
// short or asymmetric K/V break the pipeline assumptions of the self-attention kernels).
// There every key tile sees a single query step, so a kernel over key tiles spends each
// item on a short dependent chain and on per-item set-up, and dQ needs either a second
// pass or reduce-adds from every key tile.  This kernel takes one (sequence, head) per
// work item instead: the item's Q and dO rows (at most BQ of them) stay in shared
// memory, its key tiles stream past them, and dQ accumulates in TMEM across all of
// them.  dQ is written once per item, with no accumulator in memory and no atomics,
// so every result is the same bit for bit on every run.  Per key tile t:
//   S^T  = K_t Q^T          TMEM X, lanes = key rows, BQ columns
//   P^T  = exp2(S^T - lse) or act(S^T)              bf16, packed over X
//   dP^T = V_t dO^T         TMEM Y
//   dS^T = P^T (dP^T - Delta) or act'(S^T) dP^T     bf16, to the dS tile (shared memory)
//   dV_t = P^T dO           TMEM Y (A from TMEM X; the compute warps have read dP^T)
//   dK_t = dS^T Q           TMEM Z (A = the dS tile read K-major)
//   dQ  += dS K_t           TMEM W (A = the dS tile read MN-major, 128 query lanes)
// and the compute warps write dV_t and dK_t (times scale) to memory.  After the last
// tile they write dQ (times scale).
// TMEM: X [0, BQ), Y [BQ, BQ + max(BQ, D)), Z next D columns, W next D columns: 256
// columns at (D, BQ) = (64, 64), so two CTAs share an SM; 512 otherwise.
//
// CTA = 10 warps: 0-7 compute (thread = key row = TMEM lane; warpgroup g owns query
// columns [g BQ/2, (g+1) BQ/2) of a tile, and in the epilogues head-dim columns
// [g D/2, (g+1) D/2), with thread = key row for dK/dV and = query row for dQ), 8 TMA
// producer, 9 MMA issuer.
#include <algorithm>

#include "bwd_common.cuh"
#include "jfa_internal.h"
#include "ptx.cuh"
#include "tilemath.cuh"

namespace jfa {

namespace {

template <int D, int BQ>
struct ShCfg {
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static_assert(BQ == 64 || BQ == 128, "query tile of 64 or 128 rows");
    static constexpr int BN = kBwdBN;  // key rows per tile
    static constexpr int kRowBytes = D * 2;
    static constexpr int kCB = kRowBytes / 128;  // 128-byte column blocks of a head row
    static constexpr int kBoxCols = 64;          // bf16 elements per 128-byte box row
    static constexpr int kKVTile = BN * kRowBytes;
    static constexpr int kQTile = BQ * kRowBytes;
    // dS tile, bf16 [BN keys][BQ queries] as 64-query column blocks of BN x 128 bytes,
    // 128-byte swizzled: K-major for dK's A (rows = keys), MN-major for dQ's A.
    static constexpr int kDSTile = BN * BQ * 2;
    static constexpr int kCompWarps = 8;
    static constexpr int kOffK = 0;  // two stages
    static constexpr int kOffV = 2 * kKVTile;
    static constexpr int kOffQ = kOffV + kKVTile;
    static constexpr int kOffDO = kOffQ + kQTile;
    static constexpr int kOffDS = kOffDO + kQTile;
    static constexpr int kOffStage = kOffDS + kDSTile;  // 2 KB per compute warp: regrouped stores
    static constexpr int kOffBar = kOffStage + kCompWarps * 2048;
    static constexpr int kNumBars = 16;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kCols = BQ / 2;  // query columns per compute thread
    // tmem slot + abort flag (16 B); per compute warp: -lse (log2 units) and -Delta of its
    // warpgroup's columns
    static constexpr int kMiscBytes = 16 + kCompWarps * 2 * kCols * 4;
    static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + alignment of the base
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static constexpr uint32_t kTmX = 0, kTmY = BQ, kTmZ = BQ + (BQ > D ? BQ : D), kTmW = kTmZ + D;
    static constexpr uint32_t kTmCols = kTmW + D <= 256 ? 256 : 512;
    // Two CTAs per SM where both TMEM and shared memory allow it; otherwise shared memory
    // keeps a second CTA off the SM (it would wait on the TMEM allocation).
    static constexpr int kCtasPerSm = (kTmCols == 256 && 2 * (kSmemBytes + 1024) <= 228 * 1024) ? 2 : 1;
    static_assert(kCtasPerSm == 2 || kSmemBytes > 114 * 1024, "one CTA per SM must fill shared memory");
    static constexpr uint32_t kIdescS = make_idesc(kFmtBF16, BN, BQ, false, false);
    static constexpr uint32_t kIdescAcc = make_idesc(kFmtBF16, BN, D, false, true);
    static constexpr uint32_t kIdescDQ = make_idesc(kFmtBF16, 128, D, true, true);
    static constexpr int kEpiCols = D / 2;  // dK/dV/dQ columns each warpgroup writes
    static constexpr int kProdWarp = kCompWarps, kMmaWarp = kCompWarps + 1, kThreads = (kCompWarps + 2) * 32;
};

enum {
    SH_K_FULL = 0,  // +stage
    SH_K_EMPTY = 2, // +stage
    SH_V_FULL = 4,
    SH_V_EMPTY = 5,
    SH_QD_FULL = 6,
    SH_QD_EMPTY = 7,
    SH_S_FULL = 8,
    SH_DP_FULL = 9,
    SH_DS_FULL = 10,   // every compute warp wrote P^T to X and its dS rows (so has read dP^T)
    SH_DV_FULL = 11,   // dV(t) done: Y holds dV, X may be rewritten
    SH_ACC_FULL = 12,  // dK(t) and dQ(t) done: Z holds dK, the dS tile and K stage are free
    SH_ACC_EMPTY = 13, // every compute warp has read dV and dK: Y and Z are free
    SH_DQ_EMPTY = 14,  // every compute warp has read the item's dQ out of W
    SH_DRAIN = 15,
};

// TMEM column, relative to X, of the 16 bf16 P^T values of K-step s (16 queries) once the
// compute threads have packed their values in place: warpgroup g owns columns
// [g NC, (g+1) NC) and writes its NC packed values to the first NC/2 of them.
template <int NC>
__device__ __forceinline__ uint32_t packed_col_nc(int s) {
    return uint32_t(NC * (s / (NC / 16)) + 8 * (s % (NC / 16)));
}

// MODE: JFA_SOFTMAX, JFA_GDPA_GELU_TANH or JFA_GDPA_SILU (a template parameter, so that the
// activation pass is straight-line code).
template <int D, int BQ, int MODE>
__global__ void __launch_bounds__(320, ShCfg<D, BQ>::kCtasPerSm)
    jfa_bwd_short_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                         const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV,
                         const BwdParams p) {
    using C = ShCfg<D, BQ>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sK = sbase + C::kOffK, sV = sbase + C::kOffV, sQ = sbase + C::kOffQ, sDO = sbase + C::kOffDO;
    const uint32_t sDS = sbase + C::kOffDS;
    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * uint32_t(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    float* misc_f = reinterpret_cast<float*>(smem + C::kOffMisc + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(SH_K_FULL + s), 1);
            mbar_init(bar(SH_K_EMPTY + s), 1);
        }
        mbar_init(bar(SH_V_FULL), 1);
        mbar_init(bar(SH_V_EMPTY), 1);
        mbar_init(bar(SH_QD_FULL), 1);
        mbar_init(bar(SH_QD_EMPTY), 1);
        mbar_init(bar(SH_S_FULL), 1);
        mbar_init(bar(SH_DP_FULL), 1);
        mbar_init(bar(SH_DS_FULL), C::kCompWarps);
        mbar_init(bar(SH_DV_FULL), 1);
        mbar_init(bar(SH_ACC_FULL), 1);
        mbar_init(bar(SH_ACC_EMPTY), C::kCompWarps);
        mbar_init(bar(SH_DQ_EMPTY), C::kCompWarps);
        mbar_init(bar(SH_DRAIN), 1);
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
        tma_prefetch_desc(&tmdO);
        tma_prefetch_desc(&tmDK);
        tma_prefetch_desc(&tmDV);
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
            // K and V of the item's tile t (load kv_it of the rings)
            auto load_kv = [&](int h, int row) -> bool {
                const uint32_t st = kv_it & 1;
                if (!mbar_wait_bounded(bar(SH_K_EMPTY + st), ((kv_it >> 1) & 1) ^ 1, abort_flag)) return false;
                mbar_arrive_expect_tx(bar(SH_K_FULL + st), C::kKVTile);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb)
                    tma_load_2d(sK + st * C::kKVTile + cb * C::BN * 128, &tmK, bar(SH_K_FULL + st),
                                h * D + cb * C::kBoxCols, row);
                if (!mbar_wait_bounded(bar(SH_V_EMPTY), (kv_it & 1) ^ 1, abort_flag)) {
                    k_extra = 1;
                    return false;
                }
                mbar_arrive_expect_tx(bar(SH_V_FULL), C::kKVTile);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb)
                    tma_load_2d(sV + cb * C::BN * 128, &tmV, bar(SH_V_FULL), h * D + cb * C::kBoxCols, row);
                ++kv_it;
                return true;
            };
            for (int it = it_begin; it < it_end && ok; ++it) {
                const int4 w = p.items[it];
                if (!short_item_ok(w, p, BQ)) {  // not an item of this plan: skipped by every role
                    atomicOr(p.status, kStatusBounds);
                    continue;
                }
                const int b = w.x, h = w.y, n = w.w;
                const int q0 = p.q_off[b], q_len = p.q_off[b + 1] - q0, kv0 = p.kv_off[b];
                if (q_len == 0 || n == 0) continue;  // zero rows only, written by the compute warps
                // The first key tile goes out before the wait for the Q/dO buffer, so that it
                // loads while the previous item's last products run.
                if (!load_kv(h, kv0)) { ok = false; break; }
                if (!mbar_wait_bounded(bar(SH_QD_EMPTY), (item_it & 1) ^ 1, abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(SH_QD_FULL), 2 * C::kQTile);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb) {
                    tma_load_2d(sQ + cb * BQ * 128, &tmQ, bar(SH_QD_FULL), h * D + cb * C::kBoxCols, q0);
                    tma_load_2d(sDO + cb * BQ * 128, &tmdO, bar(SH_QD_FULL), h * D + cb * C::kBoxCols, q0);
                }
                ++item_it;
                for (int t = 1; t < n; ++t)
                    if (!load_kv(h, kv0 + t * C::BN)) { ok = false; break; }
            }
            if (!ok) fail();
            // Drain: wait until every load this thread issued has landed.
            drain_ring(bar(SH_QD_FULL), item_it, 1);
            drain_ring(bar(SH_K_FULL), kv_it + k_extra, 2);
            drain_ring(bar(SH_V_FULL), kv_it, 1);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the schedule, so descriptors and counters stay
        // warp-uniform; one elected lane issues every MMA and commit.
        uint32_t kv_it = 0, item_it = 0;
        bool ok = true;
        const SDesc dVa = sdesc_sw128(sV, 16, 1024);
        const SDesc dKa0 = sdesc_sw128(sK, 16, 1024), dKa1 = sdesc_sw128(sK + C::kKVTile, 16, 1024);
        const SDesc dKm0 = sdesc_sw128(sK, C::BN * 128, 1024), dKm1 = sdesc_sw128(sK + C::kKVTile, C::BN * 128, 1024);
        const SDesc dQk = sdesc_sw128(sQ, 16, 1024), dOk = sdesc_sw128(sDO, 16, 1024);
        const SDesc dQm = sdesc_sw128(sQ, BQ * 128, 1024), dOm = sdesc_sw128(sDO, BQ * 128, 1024);
        // The dS tile as dK's K-major A, and as dQ's MN-major A over 128 query lanes: two
        // 64-query blocks BN * 128 bytes apart; a 64-query tile has one block, read for
        // both halves (lanes 64-127 then repeat lanes 0-63 and are never written out).
        const SDesc dSk = sdesc_sw128(sDS, 16, 1024);
        const SDesc dSm = sdesc_sw128(sDS, BQ == 128 ? C::BN * 128 : 0, 1024);
        // K step s of a contraction over 128-byte rows: 128-byte column block (s*32)>>7 of an
        // operand with `rows` rows, (s*32)&127 bytes into the row.
        auto koff = [](int s, int rows) -> uint32_t {
            return uint32_t(((s * 32) >> 7) * rows * 128 + ((s * 32) & 127));
        };
        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 w = p.items[it];
            if (!short_item_ok(w, p, BQ)) continue;
            const int b = w.x, n = w.w;
            const int q_len = p.q_off[b + 1] - p.q_off[b];
            if (q_len == 0 || n == 0) continue;
            if (!warp_wait(SH_QD_FULL, item_it & 1)) { ok = false; break; }
            for (int t = 0; t < n; ++t) {
                const uint32_t st = kv_it & 1;
                // S^T = K Q^T into X, once dV of the previous tile has read P^T there.
                if (!warp_wait(SH_K_FULL + st, (kv_it >> 1) & 1)) { ok = false; break; }
                if (kv_it > 0 && !warp_wait(SH_DV_FULL, (kv_it - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                if (elect_one()) {
                    const SDesc ka = st ? dKa1 : dKa0;
#pragma unroll
                    for (int s = 0; s < D / 16; ++s)
                        mma_ss(tmem + C::kTmX, ka, koff(s, C::BN), dQk, koff(s, BQ), C::kIdescS, s > 0);
                    tc_commit(bar(SH_S_FULL));
                }
                __syncwarp();
                // dP^T = V dO^T into Y, once the epilogue of the previous tile has read Y and Z.
                if (!warp_wait(SH_V_FULL, kv_it & 1)) { ok = false; break; }
                if (kv_it > 0 && !warp_wait(SH_ACC_EMPTY, (kv_it - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int s = 0; s < D / 16; ++s)
                        mma_ss(tmem + C::kTmY, dVa, koff(s, C::BN), dOk, koff(s, BQ), C::kIdescS, s > 0);
                    tc_commit(bar(SH_DP_FULL));
                    tc_commit(bar(SH_V_EMPTY));
                }
                __syncwarp();
                // dV, dK and dQ once P^T is in X and dS in shared memory; the first dQ of an
                // item also waits for the previous item's dQ to have been read out of W.
                if (!warp_wait(SH_DS_FULL, kv_it & 1)) { ok = false; break; }
                if (t == 0 && item_it > 0 && !warp_wait(SH_DQ_EMPTY, (item_it - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int s = 0; s < BQ / 16; ++s)
                        mma_ts(tmem + C::kTmY, tmem + C::kTmX + packed_col_nc<C::kCols>(s), dOm, uint32_t(s) * 2048u,
                               C::kIdescAcc, s > 0);
                    tc_commit(bar(SH_DV_FULL));
#pragma unroll
                    for (int s = 0; s < BQ / 16; ++s)
                        mma_ss(tmem + C::kTmZ, dSk, koff(s, C::BN), dQm, uint32_t(s) * 2048u, C::kIdescAcc, s > 0);
                    const SDesc km = st ? dKm1 : dKm0;
#pragma unroll
                    for (int s = 0; s < C::BN / 16; ++s)
                        mma_ss(tmem + C::kTmW, dSm, uint32_t(s) * 2048u, km, uint32_t(s) * 2048u, C::kIdescDQ,
                               t > 0 || s > 0);
                    tc_commit(bar(SH_ACC_FULL));
                    tc_commit(bar(SH_K_EMPTY + st));
                    if (t == n - 1) tc_commit(bar(SH_QD_EMPTY));
                }
                __syncwarp();
                ++kv_it;
            }
            if (!ok) break;
            ++item_it;
        }
        if (!ok) fail();
        if (elect_one()) tc_commit(bar(SH_DRAIN));
        __syncwarp();
        mbar_wait_bounded(bar(SH_DRAIN), 0, nullptr);
    } else {
        // ------------------------------------------------------------ P^T, dS, epilogues
        constexpr int NC = C::kCols;
        constexpr int NK = NC / 32;  // 32-column chunks per thread
        const int wg = warp >> 2, quarter = warp & 3;
        const int r = quarter * 32 + lane;  // key row of a tile (TMEM lane); query row for dQ
        const int c0 = wg * NC;
        const uint32_t lane_base = uint32_t(quarter * 32) << 16;
        const uint32_t tX = tmem + lane_base + C::kTmX + uint32_t(c0);
        const uint32_t tY = tmem + lane_base + C::kTmY + uint32_t(c0);
        float* lse_s = misc_f + warp * 2 * NC;  // -lse (log2 units) per column
        float* del_s = lse_s + NC;              // -Delta per column
        const uint32_t stg = sbase + uint32_t(C::kOffStage + warp * 2048);
        constexpr bool GDPA = MODE != JFA_SOFTMAX, softmax = !GDPA;
        constexpr bool gelu = MODE == JFA_GDPA_GELU_TANH;
        const float xs = softmax ? p.scale_log2 : p.scale;
        const size_t row_stride = size_t(p.H) * D;  // elements between consecutive token rows
        uint32_t kv_it = 0;
        bool ok = true;
        // This thread's 16-byte piece q (0..3) of chunk k in its row of the dS tile: global
        // query column c0 + 32k + 8q, in the 64-query block (c0 + 32k) / 64, swizzled.
        auto ds_addr = [&](int k, int q) -> uint32_t {
            const int c = c0 + 32 * k;
            const int piece = (c & 63) / 8 + q;
            return sDS + uint32_t((c >> 6) * C::BN * 128 + r * 128 + ((piece ^ (r & 7)) << 4));
        };

        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 w = p.items[it];
            if (!short_item_ok(w, p, BQ)) continue;
            const int b = w.x, h = w.y, n = w.w;
            const int q0 = p.q_off[b], q_len = p.q_off[b + 1] - q0;
            const int kv0 = p.kv_off[b], kv_len = p.kv_off[b + 1] - kv0;
            if (q_len == 0) {  // no query: dK = dV = 0 for every key row
                for (int t = 0; t < n; ++t) {
                    const int j = t * C::BN + r;
                    if (j < kv_len) {
                        const size_t o = (size_t(kv0 + j) * size_t(p.H) + size_t(h)) * D + size_t(wg * C::kEpiCols);
                        zero_bf16_row(reinterpret_cast<__nv_bfloat16*>(p.dV) + o, C::kEpiCols);
                        zero_bf16_row(reinterpret_cast<__nv_bfloat16*>(p.dK) + o, C::kEpiCols);
                    }
                }
                continue;
            }
            if (n == 0) {  // no key: dQ = 0 for every query row
                if (r < q_len)
                    zero_bf16_row(reinterpret_cast<__nv_bfloat16*>(p.dQ) +
                                      (size_t(q0 + r) * size_t(p.H) + size_t(h)) * D + size_t(wg * C::kEpiCols),
                                  C::kEpiCols);
                continue;
            }
            // Row terms of this warpgroup's query columns, 0 past the end of the query set.
            __syncwarp();
#pragma unroll
            for (int k = 0; k < NK; ++k) {
                const int c = c0 + 32 * k + lane;
                const bool v = softmax && c < q_len;
                const size_t ridx = (size_t(q0) + size_t(v ? c : 0)) * size_t(p.H) + size_t(h);
                lse_s[32 * k + lane] = v ? -p.lse[ridx] * 1.4426950408889634f : 0.f;
                del_s[32 * k + lane] = v ? -p.delta[ridx] : 0.f;
            }
            __syncwarp();
            const int hi_q = min(NC, max(0, q_len - c0));  // valid local columns [0, hi_q)

            for (int t = 0; t < n; ++t, ++kv_it) {
                const bool key_valid = t * C::BN + r < kv_len;
                const int hi = key_valid ? hi_q : 0;
                const bool full = __all_sync(0xffffffffu, hi == NC);
                // chunks masked for every key row of the warp: P^T = dS = 0, nothing loaded
                bool zc[NK];
#pragma unroll
                for (int k = 0; k < NK; ++k) zc[k] = !full && __all_sync(0xffffffffu, hi <= 32 * k);

                if (!warp_wait(SH_S_FULL, kv_it & 1)) { ok = false; break; }
                tc_fence_after();
                float pv[NC];  // P (softmax) or act' (GDPA), for the dS phase
#pragma unroll
                for (int k = 0; k < NK; ++k) {
                    uint32_t pk[16];
                    if (zc[k]) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) pk[c] = 0u;
#pragma unroll
                        for (int c = 32 * k; c < 32 * k + 32; ++c) pv[c] = 0.f;
                    } else {
                        {
                            uint32_t (&ra)[32] = *reinterpret_cast<uint32_t(*)[32]>(pv + 32 * k);
                            tmem_ld32(tX + 32u * k, ra);
                            tmem_ld_wait(ra);
                        }
                        if constexpr (softmax) {
                            const float2 xs2 = make_float2(xs, xs);
#pragma unroll
                            for (int c = 32 * k; c < 32 * k + 32; c += 4) {
                                const float4 l4 = *reinterpret_cast<const float4*>(lse_s + c);
                                const float2 e0 = fma2(make_float2(pv[c], pv[c + 1]), xs2, make_float2(l4.x, l4.y));
                                const float2 e1 = fma2(make_float2(pv[c + 2], pv[c + 3]), xs2, make_float2(l4.z, l4.w));
                                pv[c] = ex2_approx(e0.x);
                                pv[c + 1] = ex2_approx(e0.y);
                                pv[c + 2] = ex2_approx(e1.x);
                                pv[c + 3] = ex2_approx(e1.y);
                            }
                            if (!full) {
#pragma unroll
                                for (int c = 32 * k; c < 32 * k + 32; ++c) pv[c] = c < hi ? pv[c] : 0.f;
                            }
#pragma unroll
                            for (int c = 0; c < 32; c += 2) pk[c >> 1] = pack_bf16x2(pv[32 * k + c], pv[32 * k + c + 1]);
                        } else {
#pragma unroll
                            for (int c = 0; c < 32; c += 2) {
                                const int cc = 32 * k + c;
                                float2 a, d;
                                gdpa_act_grad2<gelu>(make_float2(pv[cc], pv[cc + 1]), xs, a, d);
                                const bool v0 = full || cc < hi, v1 = full || cc + 1 < hi;
                                pk[c >> 1] = pack_bf16x2(v0 ? a.x : 0.f, v1 ? a.y : 0.f);
                                pv[cc] = v0 ? d.x : 0.f;
                                pv[cc + 1] = v1 ? d.y : 0.f;
                            }
                        }
                    }
                    tmem_st16(tX + 16u * k, pk);
                }
                tmem_st_wait();

                if (!warp_wait(SH_DP_FULL, kv_it & 1)) { ok = false; break; }
                tc_fence_after();
                // dS = P^T (dP^T - Delta) (softmax) or act' dP^T (GDPA), into this thread's row
                // of the dS tile.
#pragma unroll
                for (int k = 0; k < NK; ++k) {
                    uint32_t pd[16];
                    if (zc[k]) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) pd[c] = 0u;
                    } else {
                        float dp[32];
                        {
                            uint32_t (&ra)[32] = *reinterpret_cast<uint32_t(*)[32]>(dp);
                            tmem_ld32(tY + 32u * k, ra);
                            tmem_ld_wait(ra);
                        }
                        if constexpr (softmax) {
#pragma unroll
                            for (int c = 0; c < 32; c += 4) {
                                const float4 d4 = *reinterpret_cast<const float4*>(del_s + 32 * k + c);
                                const float* pp = pv + 32 * k + c;
                                const float2 a = mul2(make_float2(pp[0], pp[1]),
                                                      add2(make_float2(dp[c], dp[c + 1]), make_float2(d4.x, d4.y)));
                                const float2 b2 = mul2(make_float2(pp[2], pp[3]),
                                                       add2(make_float2(dp[c + 2], dp[c + 3]), make_float2(d4.z, d4.w)));
                                pd[c >> 1] = pack_bf16x2(a.x, a.y);
                                pd[(c >> 1) + 1] = pack_bf16x2(b2.x, b2.y);
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < 32; c += 2) {
                                const float2 a = mul2(make_float2(pv[32 * k + c], pv[32 * k + c + 1]),
                                                      make_float2(dp[c], dp[c + 1]));
                                pd[c >> 1] = pack_bf16x2(a.x, a.y);
                            }
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) st_shared_v4(ds_addr(k, q), pd[4 * q], pd[4 * q + 1], pd[4 * q + 2], pd[4 * q + 3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(SH_DS_FULL));

                // Epilogue of the tile: dV as soon as its product is done, then dK (times scale),
                // 32 columns at a time through the staging.  A warp whose 32 key rows all lie in
                // the sequence writes an accumulator's first chunk with one TMA store of the
                // staged box and any second chunk (head_dim 128) row by row: with one 2 KB
                // staging per warp a second box would wait for the first to be read, which
                // measured slower.  A warp holding the sequence's end stores row by row (a box
                // cannot skip the rows that belong to the next sequence).  Before the staging is
                // written, the lane that issued the previous box waits until it has been read.
                const uint32_t valid = __ballot_sync(0xffffffffu, key_valid);
                const int ky = kv0 + t * C::BN + quarter * 32;  // the warp's first key row
                const size_t off0 = (size_t(ky) * size_t(p.H) + size_t(h)) * D + size_t(wg * C::kEpiCols);
#pragma unroll
                for (int u = 0; u < 2; ++u) {  // dV, then dK
                    if (!warp_wait(u ? SH_ACC_FULL : SH_DV_FULL, kv_it & 1)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int cc = 0; cc < C::kEpiCols / 32; ++cc) {
                        uint32_t rr[32];
                        tmem_ld32(tmem + lane_base + (u ? C::kTmZ : C::kTmY) + uint32_t(wg * C::kEpiCols + 32 * cc), rr);
                        tmem_ld_wait(rr);
                        if (!valid) continue;
                        if (lane == 0) bulk_wait_read();
                        __syncwarp();
                        if (valid == 0xffffffffu && cc == 0) {
                            stage_chunk_bf16(stg, rr, u ? p.scale : 1.f, lane);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_2d(u ? &tmDK : &tmDV, stg, h * D + wg * C::kEpiCols + 32 * cc, ky);
                                bulk_commit();
                            }
                        } else {
                            store_chunk_bf16(stg, rr, u ? p.scale : 1.f, lane, valid,
                                             reinterpret_cast<__nv_bfloat16*>(u ? p.dK : p.dV) + off0 + 32 * cc,
                                             row_stride);
                        }
                    }
                }
                if (!ok) break;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(SH_ACC_EMPTY));
            }
            if (!ok) break;
            // dQ of the item (times scale): thread = query row r; the last tile's ACC_FULL,
            // waited for above, covers the last product into W.
            {
                const uint32_t valid = __ballot_sync(0xffffffffu, r < q_len);
                if (valid) {
                    const size_t off0 =
                        (size_t(q0 + quarter * 32) * size_t(p.H) + size_t(h)) * D + size_t(wg * C::kEpiCols);
#pragma unroll
                    for (int cc = 0; cc < C::kEpiCols / 32; ++cc) {
                        uint32_t rr[32];
                        tmem_ld32(tmem + lane_base + C::kTmW + uint32_t(wg * C::kEpiCols + 32 * cc), rr);
                        tmem_ld_wait(rr);
                        if (lane == 0) bulk_wait_read();
                        __syncwarp();
                        store_chunk_bf16(stg, rr, p.scale, lane, valid,
                                         reinterpret_cast<__nv_bfloat16*>(p.dQ) + off0 + 32 * cc, row_stride);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(SH_DQ_EMPTY));
        }
        if (!ok) fail();
        // Every store this warp's lane issued has completed before the CTA exits.
        if (lane == 0) bulk_wait_done();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kMmaWarp) tmem_dealloc(tmem, C::kTmCols);
}

template <int D, int BQ, int MODE>
cudaError_t launch_short_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const CUtensorMap& tmdO, const CUtensorMap& tmDK, const CUtensorMap& tmDV, const BwdParams& p,
                           int grid, cudaStream_t st) {
    using C = ShCfg<D, BQ>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(jfa_bwd_short_kernel<D, BQ, MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    jfa_bwd_short_kernel<D, BQ, MODE><<<grid, C::kThreads, C::kSmemBytes, st>>>(tmQ, tmK, tmV, tmdO, tmDK, tmDV, p);
    return cudaGetLastError();
}

}  // namespace

int short_ctas_per_sm(int D, int bq) {
    if (D == 64 && bq == 64) return ShCfg<64, 64>::kCtasPerSm;
    if (D == 64 && bq == 128) return ShCfg<64, 128>::kCtasPerSm;
    if (D == 128 && bq == 128) return ShCfg<128, 128>::kCtasPerSm;
    return 0;
}

template <int D, int BQ>
static cudaError_t launch_short_m(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                  const CUtensorMap& tmdO, const CUtensorMap& tmDK, const CUtensorMap& tmDV,
                                  const BwdParams& p, int grid, cudaStream_t st) {
    if (p.mode == JFA_SOFTMAX) return launch_short_t<D, BQ, JFA_SOFTMAX>(tmQ, tmK, tmV, tmdO, tmDK, tmDV, p, grid, st);
    if (p.mode == JFA_GDPA_GELU_TANH)
        return launch_short_t<D, BQ, JFA_GDPA_GELU_TANH>(tmQ, tmK, tmV, tmdO, tmDK, tmDV, p, grid, st);
    return launch_short_t<D, BQ, JFA_GDPA_SILU>(tmQ, tmK, tmV, tmdO, tmDK, tmDV, p, grid, st);
}

cudaError_t launch_bwd_short(int D, int bq, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const CUtensorMap& tmdO, const CUtensorMap& tmDK, const CUtensorMap& tmDV,
                             const BwdParams& p, int grid, cudaStream_t st) {
    if (D == 64 && bq == 64) return launch_short_m<64, 64>(tmQ, tmK, tmV, tmdO, tmDK, tmDV, p, grid, st);
    if (D == 64 && bq == 128) return launch_short_m<64, 128>(tmQ, tmK, tmV, tmdO, tmDK, tmDV, p, grid, st);
    if (D == 128 && bq == 128) return launch_short_m<128, 128>(tmQ, tmK, tmV, tmdO, tmDK, tmDV, p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace jfa
