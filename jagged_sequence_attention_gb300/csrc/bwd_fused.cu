// Fused backward kernel: dK, dV and dQ in one pass over key tiles (bf16 inputs).
//
// The backward of the GEM articles' jagged flash attention is parallelised over
// key/value tiles (kerneldigest.dev summary, "Arquitectura del Sistema": backward-pass
// parallelisation), and the vibekk.com article names "backward accumulation" as the
// bottleneck left once padding is gone (section 第一轮瓶颈迁移): every key tile adds a
// part of every query row's dQ.  This kernel forms that part on the tensor core next to
// dK and dV and adds it into a jagged fp32 accumulator [T_q, H, D] in L2 (no padded
// buffer); a conversion pass scales it and writes dQ in bf16.  Compared with a second
// pass over query tiles, which recomputes S and dP to form dQ on chip, it issues five
// products per tile pair instead of seven, and moves 64 KB of fp32 reduce-adds per tile
// pair instead (L2 absorbs them at about 7 TB/s on GB300).
//
// Persistent over (sequence, head, 128-row key tile).  K and V stay in shared memory;
// 128-row query tiles stream through a two-stage Q ring and a one-stage dO buffer.
// Per step i (query tile i):
//   S^T  = K Q_i^T      TMEM X, lanes = key rows
//   P^T  = exp2(S^T - lse) or act(S^T)            bf16, written back over X
//   dP^T = V dO_i^T     TMEM Y
//   dS^T = P^T (dP^T - Delta) or act'(S^T) dP^T   bf16, to shared memory (one tile)
//   dV  += P^T dO_i     (A from TMEM X)
//   dK  += dS^T Q_i     (A = the dS tile read K-major)
//   dQ_i = dS K         (A = the same dS tile read MN-major; into TMEM Y, whose dP^T the
//                        compute warps have read), then drained by the compute warps:
//                        TMEM -> registers (Y released) -> 32 x 32 fp32 boxes staged in
//                        the dS tile -> TMA tensor reduce-adds into the accumulator, so
//                        the compute warps issue no per-element global traffic
// TMEM: dV [0,128), dK [128,256), X [256,384), Y [384,512).
// Issue order per step: S(i+1), dK(i), dQ(i), dP(i+1), dV(i+1).  dP(i+1) waits for the
// drain of dQ(i) out of Y; the compute warps drain dQ(i) after step i+1's P^T phase, so
// that dK(i) and dQ(i) run on the tensor core while P^T(i+1) is formed.
//
// CTA = 10 warps: 0-7 compute (thread = key row = TMEM lane; warpgroup g owns query
// columns [64g, 64g+64) of a step, and in the drain, head-dim columns [g D/2, (g+1) D/2)
// of dQ_i with thread = query row), 8 TMA producer, 9 MMA issuer.
#include <algorithm>

#include "bwd_common.cuh"
#include "jfa_internal.h"
#include "ptx.cuh"
#include "tilemath.cuh"

namespace jfa {

namespace {

template <int D>
struct FuCfg {
    static constexpr int BN = kBwdBN;  // key rows (TMEM lanes of dK, dV, S^T, dP^T)
    static constexpr int BM = kBwdBM;  // query rows per step (TMEM lanes of dQ)
    static constexpr int kRowBytes = D * 2;
    static_assert(kRowBytes % 128 == 0 && kRowBytes <= 256, "head row must be 128 or 256 bytes");
    static constexpr int kCB = kRowBytes / 128;  // 128-byte column blocks of a row
    static constexpr int kBoxCols = 64;          // bf16 elements per 128-byte box row
    static constexpr int kKVTile = BN * kRowBytes;
    static constexpr int kQTile = BM * kRowBytes;
    // dS tile, bf16 [BN keys][BM queries] as two 128-byte column blocks of 64 queries,
    // 128-byte swizzled: K-major for dK's A (rows = keys), MN-major for dQ's A.
    static constexpr int kDSTile = BN * BM * 2;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kKVTile;
    static constexpr int kOffQ = 2 * kKVTile;          // + stage * kQTile
    static constexpr int kOffDO = kOffQ + 2 * kQTile;  // one stage
    static constexpr int kOffDS = kOffDO + kQTile;
    static constexpr int kOffBar = kOffDS + kDSTile;
    static constexpr int kNumBars = 24;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kCompWarps = kDkdvCompWarps;
    static constexpr int kCols = BM / 2;  // query columns per compute thread
    // tmem slot + abort flag (16 B); per compute warp: -lse and -Delta of its columns, the
    // head's bias row and a step's bias-by-relative-position table (kCols + 32 entries)
    static constexpr int kRelTab = kCols + 32;
    static constexpr int kWarpMisc = 2 * kCols + 32 + kRelTab;
    static constexpr int kMiscBytes = 16 + kCompWarps * kWarpMisc * 4;
    // per compute warp: a 2 KB buffer through which the epilogue's stores are regrouped
    static constexpr int kOffStage = (kOffMisc + kMiscBytes + 127) / 128 * 128;
    static constexpr int kSmemNeed = kOffStage + kCompWarps * 2048 + 1024;
    static constexpr int kSmemBytes = kSmemNeed > 120 * 1024 ? kSmemNeed : 120 * 1024;
    static_assert(kSmemNeed <= 227 * 1024, "shared memory budget");
    static constexpr int kDSteps = D / 16;   // contraction over head_dim
    static constexpr int kQSteps = BM / 16;  // contraction over query rows
    static constexpr int kKSteps = BN / 16;  // contraction over key rows (dQ)
    static_assert(kQSteps == 8 && kCols == 64, "chunked dK/dV issue assumes 128-row query steps");
    // dQ drain: each warp owns 32 query rows x D/2 columns, in 32-column chunks staged
    // through its 4 KB part of the dS tile
    static constexpr int kDrainChunks = D / 64;
    static_assert(kCompWarps * 4096 == kDSTile, "drain staging covers the dS tile");
    static constexpr uint32_t kTmDV = 0, kTmDK = 128, kTmX = 256, kTmY = 384;
    static constexpr uint32_t kIdescS = make_idesc(kFmtBF16, BN, BM, false, false);
    static constexpr uint32_t kIdescAcc = make_idesc(kFmtBF16, BN, D, false, true);
    static constexpr uint32_t kIdescDQ = make_idesc(kFmtBF16, BM, D, true, true);
    static constexpr int kEpiCols = D / 2;  // dK/dV columns each warpgroup writes
    static constexpr int kProdWarp = kCompWarps, kMmaWarp = kCompWarps + 1, kThreads = (kCompWarps + 2) * 32;
};

enum {
    FU_K_FULL = 0,
    FU_V_FULL = 1,
    FU_K_EMPTY = 2,  // the item's last dQ product is done: K may be overwritten
    FU_Q_FULL = 3,   // +stage
    FU_Q_EMPTY = 5,  // +stage
    FU_DO_FULL = 7,
    FU_DO_EMPTY = 8,
    FU_S_FULL = 9,
    FU_P_FULL = 10,  // +chunk: columns [32k, 32k+32) of both warpgroups' P^T are in TMEM
    FU_DP_FULL = 12,
    FU_DS_FULL = 13,  // +chunk: the chunk's dS is in shared memory
    FU_X_FREE = 15,   // dV(i) done: the S^T/P^T columns may be rewritten
    FU_DQK_DONE = 16, // dK(i) and dQ(i) done: dQ(i) is in Y and the dS tile is no longer read
    FU_DQ_EMPTY = 17, // every compute warp has drained dQ(i): Y and the dS tile are free
    FU_ACC_FULL = 18,
    FU_ACC_EMPTY = 19,
    FU_DRAIN = 20,
    FU_V_EMPTY = 21,  // the item's last dP product is done: V may be overwritten
};

template <int D, bool GDPA>
__global__ void __launch_bounds__(320, 1)
    jfa_bwd_fused_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                         const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmDK,
                         const __grid_constant__ CUtensorMap tmDV, const BwdParams p) {
    using C = FuCfg<D>;
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
        mbar_init(bar(FU_K_FULL), 1);
        mbar_init(bar(FU_V_FULL), 1);
        mbar_init(bar(FU_K_EMPTY), 1);
        mbar_init(bar(FU_V_EMPTY), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(FU_Q_FULL + s), 1);
            mbar_init(bar(FU_Q_EMPTY + s), 1);
            mbar_init(bar(FU_P_FULL + s), C::kCompWarps);
            mbar_init(bar(FU_DS_FULL + s), C::kCompWarps);
        }
        mbar_init(bar(FU_DO_FULL), 1);
        mbar_init(bar(FU_DO_EMPTY), 1);
        mbar_init(bar(FU_S_FULL), 1);
        mbar_init(bar(FU_DP_FULL), 1);
        mbar_init(bar(FU_X_FREE), 1);
        mbar_init(bar(FU_DQK_DONE), 1);
        mbar_init(bar(FU_DQ_EMPTY), C::kCompWarps);
        mbar_init(bar(FU_ACC_FULL), 1);
        mbar_init(bar(FU_ACC_EMPTY), C::kCompWarps);
        mbar_init(bar(FU_DRAIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == C::kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == C::kProdWarp && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmdO);
        tma_prefetch_desc(&tmDQ);
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
            // Loads issued so far, per buffer (the drain below waits for each one's last).
            // An item's loads go out in the order in which their buffers come free at the
            // end of the previous item: its first Q tile (a ring stage freed a step
            // earlier), V (after the last dP), its first dO tile (after the last dV), and K
            // (after the last dQ), so that only K's load stands between one item's last
            // product and the next item's first.
            uint32_t n_q = 0, n_do = 0, n_k = 0, n_v = 0;
            bool ok = true;
            auto load_q = [&](int h, int y) -> bool {
                const uint32_t st = n_q & 1, ph = (n_q >> 1) & 1;
                if (!mbar_wait_bounded(bar(FU_Q_EMPTY + st), ph ^ 1, abort_flag)) return false;
                mbar_arrive_expect_tx(bar(FU_Q_FULL + st), C::kQTile);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb)
                    tma_load_2d(sQ + st * C::kQTile + cb * C::BM * 128, &tmQ, bar(FU_Q_FULL + st),
                                h * D + cb * C::kBoxCols, y);
                ++n_q;
                return true;
            };
            auto load_do = [&](int h, int y) -> bool {
                if (!mbar_wait_bounded(bar(FU_DO_EMPTY), (n_do & 1) ^ 1, abort_flag)) return false;
                mbar_arrive_expect_tx(bar(FU_DO_FULL), C::kQTile);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb)
                    tma_load_2d(sDO + cb * C::BM * 128, &tmdO, bar(FU_DO_FULL), h * D + cb * C::kBoxCols, y);
                ++n_do;
                return true;
            };
            // K or V of key rows [y, y + BN)
            auto load_kv = [&](bool is_k, int h, int y) -> bool {
                uint32_t& cnt = is_k ? n_k : n_v;
                if (!mbar_wait_bounded(bar(is_k ? FU_K_EMPTY : FU_V_EMPTY), (cnt & 1) ^ 1, abort_flag)) return false;
                const uint32_t full = bar(is_k ? FU_K_FULL : FU_V_FULL);
                mbar_arrive_expect_tx(full, C::kKVTile);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb)
                    tma_load_2d((is_k ? sK : sV) + cb * C::BN * 128, is_k ? &tmK : &tmV, full,
                                h * D + cb * C::kBoxCols, y);
                ++cnt;
                return true;
            };
            for (int it = it_begin; it < it_end && ok; ++it) {
                const int4 w = p.items[it];
                if (!kv_item_ok(w, p, false)) {  // not an item of this plan: skipped by every role
                    atomicOr(p.status, kStatusBounds);
                    continue;
                }
                const int n = w.w;
                if (n == 0) continue;
                const int b = w.x, h = w.y, nt = w.z;
                const int q0 = p.q_off[b], kv0 = p.kv_off[b];
                int first_qt, nq;  // query tiles [first_qt, first_qt + n) see this key tile
                query_tile_range(p.q_off[b + 1] - q0, p.kv_off[b + 1] - kv0, nt, p.causal, p.window, first_qt, nq);
                const int y0 = q0 + first_qt * C::BM, ykv = kv0 + nt * C::BN;
                if (!load_q(h, y0) || !load_kv(false, h, ykv) || !load_do(h, y0) || !load_kv(true, h, ykv)) {
                    ok = false;
                    break;
                }
                for (int i = 1; i < n; ++i) {
                    const int y = q0 + (first_qt + i) * C::BM;
                    if (!load_q(h, y) || !load_do(h, y)) { ok = false; break; }
                }
            }
            if (!ok) fail();
            // Drain: wait until every load this thread issued has landed.
            if (n_k > 0) mbar_wait_bounded(bar(FU_K_FULL), (n_k - 1) & 1, nullptr);
            if (n_v > 0) mbar_wait_bounded(bar(FU_V_FULL), (n_v - 1) & 1, nullptr);
            drain_ring(bar(FU_Q_FULL), n_q, 2);
            drain_ring(bar(FU_DO_FULL), n_do, 1);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the schedule, so descriptors and counters stay
        // warp-uniform; one elected lane (always lane 0) issues every MMA and commit.
        uint32_t step_it = 0, item_it = 0, dv_cnt = 0;
        bool ok = true;
        const SDesc dKa = sdesc_sw128(sK, 16, 1024), dVa = sdesc_sw128(sV, 16, 1024);
        const SDesc dQk0 = sdesc_sw128(sQ, 16, 1024), dQk1 = sdesc_sw128(sQ + C::kQTile, 16, 1024);
        const SDesc dOk = sdesc_sw128(sDO, 16, 1024);
        const SDesc dQm0 = sdesc_sw128(sQ, C::BM * 128, 1024), dQm1 = sdesc_sw128(sQ + C::kQTile, C::BM * 128, 1024);
        const SDesc dOm = sdesc_sw128(sDO, C::BM * 128, 1024);
        // the dS tile as dK's K-major A, and as dQ's MN-major A (64-query blocks BN * 128
        // bytes apart); K as dQ's MN-major B (64-column blocks BN * 128 bytes apart)
        const SDesc dSk = sdesc_sw128(sDS, 16, 1024), dSm = sdesc_sw128(sDS, C::BN * 128, 1024);
        const SDesc dKm = sdesc_sw128(sK, C::BN * 128, 1024);
        // K step s of a contraction over a 128-byte-row operand: 128-byte column block
        // (s*32)>>7, (s*32)&127 bytes into the row; both operands have 128 rows.
        auto koff = [](int s) -> uint32_t { return uint32_t(((s * 32) >> 7) * 128 * 128 + ((s * 32) & 127)); };
        // S^T(g) = K Q^T into X, once dV of the previous step has read P^T there.
        auto issue_s = [&](uint32_t g) -> bool {
            const uint32_t st = g & 1, ph = (g >> 1) & 1;
            if (!warp_wait(FU_Q_FULL + st, ph)) return false;
            if (dv_cnt > 0 && !warp_wait(FU_X_FREE, (dv_cnt - 1) & 1)) return false;
            tc_fence_after();
            const SDesc dq = st ? dQk1 : dQk0;
            if (elect_one()) {
#pragma unroll
                for (int s = 0; s < C::kDSteps; ++s) mma_ss(tmem + C::kTmX, dKa, koff(s), dq, koff(s), C::kIdescS, s > 0);
                tc_commit(bar(FU_S_FULL));
            }
            __syncwarp();
            return true;
        };
        // dP^T(g) = V dO^T into Y, once every compute warp has drained dQ(g-1) out of Y;
        // after an item's last one, V is released to the next item's load.
        auto issue_dp = [&](uint32_t g, bool last) -> bool {
            if (!warp_wait(FU_DO_FULL, g & 1)) return false;
            if (g > 0 && !warp_wait(FU_DQ_EMPTY, (g - 1) & 1)) return false;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int s = 0; s < C::kDSteps; ++s) mma_ss(tmem + C::kTmY, dVa, koff(s), dOk, koff(s), C::kIdescS, s > 0);
                tc_commit(bar(FU_DP_FULL));
                if (last) tc_commit(bar(FU_V_EMPTY));
            }
            __syncwarp();
            return true;
        };
        // The K-steps (16 query rows each) that read chunk c of warpgroup w's 64 columns:
        // query rows 64w + 32c .. + 31, K-steps 4w + 2c, +1.
        auto chunk_step = [](int c, int i) -> int { return 4 * (i >> 1) + 2 * c + (i & 1); };
        // dV += P^T dO with P^T read from TMEM, chunk by chunk as the compute warps
        // finish it; the first step of an item waits for the epilogue of the previous
        // item to have read the accumulators.
        auto issue_dv = [&](uint32_t g, bool first) -> bool {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (!warp_wait(FU_P_FULL + c, g & 1)) return false;
                if (c == 0 && first && !warp_wait(FU_ACC_EMPTY, (item_it & 1) ^ 1)) return false;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int s = chunk_step(c, i);
                        mma_ts(tmem + C::kTmDV, tmem + C::kTmX + packed_col(s), dOm, s * 16 * 128, C::kIdescAcc,
                               (!first || c > 0 || i > 0));
                    }
                    if (c == 1) {
                        tc_commit(bar(FU_X_FREE));
                        tc_commit(bar(FU_DO_EMPTY));
                    }
                }
                __syncwarp();
            }
            ++dv_cnt;
            return true;
        };
        // dK += dS^T Q (chunk by chunk as the dS tile fills), then dQ(g) = dS K into Y.
        auto issue_dk_dq = [&](uint32_t g, bool first) -> bool {
            const uint32_t st = g & 1;
            const SDesc dq = st ? dQm1 : dQm0;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (!warp_wait(FU_DS_FULL + c, g & 1)) return false;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int s = chunk_step(c, i);
                        mma_ss(tmem + C::kTmDK, dSk, koff(s), dq, s * 16 * 128, C::kIdescAcc, (!first || c > 0 || i > 0));
                    }
                    if (c == 1) {
                        tc_commit(bar(FU_Q_EMPTY + st));
#pragma unroll
                        for (int s = 0; s < C::kKSteps; ++s)
                            mma_ss(tmem + C::kTmY, dSm, s * 16 * 128, dKm, s * 16 * 128, C::kIdescDQ, s > 0);
                        tc_commit(bar(FU_DQK_DONE));
                    }
                }
                __syncwarp();
            }
            return true;
        };
        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 wi = p.items[it];
            if (!kv_item_ok(wi, p, false)) continue;
            const int n = wi.w;
            if (n == 0) continue;
            if (!warp_wait(FU_K_FULL, item_it & 1) || !warp_wait(FU_V_FULL, item_it & 1)) { ok = false; break; }
            tc_fence_after();
            const uint32_t g0 = step_it;
            if (!issue_s(g0) || !issue_dp(g0, n == 1) || !issue_dv(g0, true)) { ok = false; break; }
            for (int i = 0; i < n && ok; ++i) {
                const uint32_t g = g0 + uint32_t(i);
                if (i + 1 < n && !issue_s(g + 1)) { ok = false; break; }
                if (!issue_dk_dq(g, i == 0)) { ok = false; break; }
                if (i + 1 < n && (!issue_dp(g + 1, i + 2 == n) || !issue_dv(g + 1, false))) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            if (elect_one()) {
                tc_commit(bar(FU_ACC_FULL));
                tc_commit(bar(FU_K_EMPTY));
            }
            __syncwarp();
            step_it += uint32_t(n);
            ++item_it;
        }
        if (!ok) fail();
        if (elect_one()) tc_commit(bar(FU_DRAIN));
        __syncwarp();
        mbar_wait_bounded(bar(FU_DRAIN), 0, nullptr);
    } else {
        // ------------------------------------------------------------ P^T, dS, dQ drain, epilogue
        // Thread = key row r (TMEM lane); warpgroup wg owns query columns [c0, c0+64).
        constexpr int NC = C::kCols;
        const int wg = warp >> 2;
        const int r = (warp & 3) * 32 + lane;
        const int c0 = wg * NC;
        const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
        const uint32_t tX = tmem + lane_base + C::kTmX + uint32_t(c0);
        const uint32_t tY = tmem + lane_base + C::kTmY + uint32_t(c0);
        float* lse_s = misc_f + warp * C::kWarpMisc;  // -lse (log2 units) per column
        float* del_s = lse_s + NC;                      // -Delta per column
        float* bias_w = del_s + NC;                     // the head's bias row (log2 units for softmax)
        float* rtab = bias_w + 32;                      // bias by relative position, per step
        // This thread's row of the dS tile: key r, warpgroup wg's 64-query block, 128-byte
        // swizzled (16-byte piece q of the row at position q ^ (r & 7)).
        const uint32_t ds_row = sDS + uint32_t(wg * C::BN * 128 + r * 128);
        // This warp's 4 KB of the dS tile, the drain's staging once dK and dQ have read it.
        const uint32_t stg = sDS + uint32_t(warp * 4096);
        // Element (lane, c) has relative position rbase(lane 0) - lane + c: rtab[k] holds
        // the bias of rbase(lane 0) - 31 + k, so the lane reads rrow[c], rrow = rtab + 31 - lane.
        const float* rrow = rtab + 31 - lane;
        constexpr bool softmax = !GDPA;
        const bool gelu = p.mode == JFA_GDPA_GELU_TANH;
        uint32_t step_it = 0, item_it = 0;
        bool ok = true;

        // dQ(g) of query rows [qrow0, qrow0 + 128) of a sequence whose first row is dq_y0 (of
        // dq_len rows), at accumulator column dq_x0 (this warpgroup's half of head h), 32
        // columns at a time: TMEM Y -> registers -> this warp's staging (the 128-byte-swizzled
        // box layout) -> a TMA reduce-add into the accumulator.  Y is released for the next dP
        // once its last columns are read.  The staging was last read by a box before this
        // warp wrote its dS rows there, which waited for that, so only a second box waits.
        // The box covers all 32 rows: rows
        // past the sequence end hold zeros (their dS is 0), and adding a zero leaves any value
        // of the accumulator as it is (it starts at +0, so no sum in it is ever -0); rows past
        // the accumulator's end are clipped by the tensor map.  A warp whose rows all lie past
        // the end adds nothing.
        auto drain = [&](uint32_t g, int dq_x0, int dq_y0, int dq_len, int qrow0) -> bool {
            if (!warp_wait(FU_DQK_DONE, g & 1)) return false;
            tc_fence_after();
            const int wrow0 = qrow0 + (warp & 3) * 32;  // this warp's first query row
#pragma unroll
            for (int k = 0; k < C::kDrainChunks; ++k) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + C::kTmY + uint32_t(wg * (D / 2) + 32 * k), v);
                tmem_ld_wait(v);
                if (k + 1 == C::kDrainChunks) {  // the last read of Y: release it for the next dP
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(FU_DQ_EMPTY));
                }
                if (k > 0) {  // the previous box has left the staging
                    if (lane == 0) bulk_wait_read();
                    __syncwarp();
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    st_shared_v4(stg + uint32_t(lane * 128 + ((q ^ (lane & 7)) << 4)), v[4 * q], v[4 * q + 1],
                                 v[4 * q + 2], v[4 * q + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && wrow0 < dq_len) {
                    tma_reduce_add_2d(&tmDQ, stg, dq_x0 + 32 * k, dq_y0 + wrow0);
                    bulk_commit();
                }
            }
            return true;
        };

        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 w = p.items[it];
            if (!kv_item_ok(w, p, false)) continue;
            const int n = w.w, b = w.x, h = w.y, nt = w.z;
            const int kv0 = p.kv_off[b], kv_len = p.kv_off[b + 1] - kv0;
            const int q0 = p.q_off[b], q_len = p.q_off[b + 1] - q0;
            int first_qt, nq;  // query tiles [first_qt, first_qt + n) see this key tile
            query_tile_range(q_len, kv_len, nt, p.causal, p.window, first_qt, nq);
            const int dq_x0 = h * D + wg * (D / 2);  // accumulator column of this warpgroup's half
            const int j = nt * C::BN + r;  // key row within the sequence
            const bool key_valid = j < kv_len;
            const size_t krow = (size_t(kv0) + size_t(key_valid ? j : 0)) * size_t(p.H) + size_t(h);
            __nv_bfloat16* dv_row = reinterpret_cast<__nv_bfloat16*>(p.dV) + krow * D + wg * C::kEpiCols;
            __nv_bfloat16* dk_row = reinterpret_cast<__nv_bfloat16*>(p.dK) + krow * D + wg * C::kEpiCols;
            if (n == 0) {  // no query sees this key tile: its gradients are zero
                if (key_valid) {
                    zero_bf16_row(dv_row, C::kEpiCols);
                    zero_bf16_row(dk_row, C::kEpiCols);
                }
                continue;
            }
            if (p.bias) {
                __syncwarp();
                bias_w[lane] = p.bias[h * 32 + lane] * (softmax ? 1.4426950408889634f : 1.0f);
                __syncwarp();
            }
            // Row terms (lse, Delta) of this warpgroup's query columns: lane l holds columns
            // c0 + l and c0 + 32 + l, loaded one step ahead as they are (bit k of rv: column
            // valid).
            float rl[2] = {0.f, 0.f}, rd[2] = {0.f, 0.f};
            uint32_t rv = 0;
            auto fetch = [&](int qrow0) {
                rv = 0;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int c = qrow0 + c0 + 32 * k + lane;
                    const bool v = c < q_len;
                    const size_t ridx = (size_t(q0) + size_t(v ? c : 0)) * size_t(p.H) + size_t(h);
                    if constexpr (softmax) {
                        rl[k] = p.lse[ridx];
                        rd[k] = p.delta[ridx];
                    }
                    rv |= uint32_t(v) << k;
                }
            };
            fetch(first_qt * C::BM);
            for (int i = 0; i < n; ++i) {
                const uint32_t g = step_it + uint32_t(i);
                const int qrow0 = (first_qt + i) * C::BM;
                const int diag = kv_len - q_len;
                // -lse in log2 units and -Delta of this step's columns (0 past the end)
                const float cur_nl0 = (softmax && (rv & 1u)) ? -rl[0] * 1.4426950408889634f : 0.f;
                const float cur_nl1 = (softmax && (rv & 2u)) ? -rl[1] * 1.4426950408889634f : 0.f;
                __syncwarp();
                del_s[lane] = (softmax && (rv & 1u)) ? -rd[0] : 0.f;
                del_s[32 + lane] = (softmax && (rv & 2u)) ? -rd[1] : 0.f;
                if (i + 1 < n) fetch(qrow0 + C::BM);
                // subtraction scheme: valid local columns are [lo, hi)
                int hi = key_valid ? min(NC, q_len - qrow0 - c0) : 0;
                // sliding window: query i sees key j only while j >= i' - W, i.e. i <= j - diag + W
                if (p.window >= 0) hi = min(hi, j - diag + p.window + 1 - qrow0 - c0);
                const int lo = p.causal ? max(0, j - diag - qrow0 - c0) : 0;
                const bool full = __all_sync(0xffffffffu, lo == 0 && hi == NC);
                const int rbase = qrow0 + c0 + diag - j;  // relative position of local column 0
                const float xs = softmax ? p.scale_log2 : p.scale;
                // Bias per 32-column chunk: one value when every lane's chunk sits in one
                // bucket, else read per element from the relative-position table.  Lane k
                // tests chunk k for the whole warp: over the warp's keys, chunk k spans
                // relative positions rbase(lane 0) + 32k - 31 .. + 62.
                bool cconst[2] = {true, true};
                float cbias[2] = {0.f, 0.f};
                if (p.bias) {
                    const int rb0 = __shfl_sync(0xffffffffu, rbase, 0);
                    int bk = 0;
                    const uint32_t cm = warp_const_chunks(lane < 2, rb0 + 32 * lane - 31, bk);
                    const float bv = bias_w[bk];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        cconst[k] = (cm >> k) & 1u;
                        cbias[k] = __shfl_sync(0xffffffffu, bv, k);
                    }
                }
                // Staged addend of column c: -lse, plus the chunk's bias when that is one
                // value for the whole warp (it then is the same for every lane).
                lse_s[lane] = cur_nl0 + (cconst[0] ? cbias[0] : 0.f);
                lse_s[32 + lane] = cur_nl1 + (cconst[1] ? cbias[1] : 0.f);
                if (!(cconst[0] && cconst[1])) {
                    const int r0 = __shfl_sync(0xffffffffu, rbase, 0) - 31;
#pragma unroll
                    for (int m = 0; m < C::kRelTab / 32; ++m)
                        rtab[lane + 32 * m] = bias_w[relpos_bucket(r0 + lane + 32 * m)];
                }
                __syncwarp();

                // A 32-column chunk masked for every key row of the warp has P^T = dS = 0:
                // softmax zeroes P and forms dS = 0 on the common path; GDPA also skips the
                // chunk's loads and dS arithmetic.
                const bool zc[2] = {!full && __all_sync(0xffffffffu, hi <= 0 || lo >= 32),
                                    !full && __all_sync(0xffffffffu, hi <= 32 || lo >= NC)};
                if (!warp_wait(FU_S_FULL, g & 1)) { ok = false; break; }
                tc_fence_after();
                float pv[NC];
                {
                    uint32_t (&ra)[32] = *reinterpret_cast<uint32_t(*)[32]>(pv);
                    uint32_t (&rb)[32] = *reinterpret_cast<uint32_t(*)[32]>(pv + 32);
                    if constexpr (GDPA) {  // GDPA: a zero chunk is not even loaded
                        if (!zc[0]) tmem_ld32(tX, ra);
                        if (!zc[1]) tmem_ld32(tX + 32u, rb);
                        if (!(zc[0] && zc[1])) {
                            tmem_ld_wait(ra);
                            tmem_ld_wait(rb);
                        }
                    } else {
                        tmem_ld32(tX, ra);
                        tmem_ld32(tX + 32u, rb);
                        tmem_ld_wait(ra);
                        tmem_ld_wait(rb);
                    }
                }
                // P^T = exp2(xs * s + bias - lse) (softmax; pv keeps P) or act(scale * s +
                // bias) (GDPA; pv keeps act' for dS), one 32-column chunk at a time, packed
                // over the warpgroup's own S^T columns (already read) and signalled at once.
                const float2 xs2 = make_float2(xs, xs);
                const bool fast = full && cconst[0] && cconst[1];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    uint32_t pk[16];
                    if (softmax && fast) {
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
#pragma unroll
                        for (int c = 0; c < 32; c += 2) pk[c >> 1] = pack_bf16x2(pv[32 * k + c], pv[32 * k + c + 1]);
                    } else if (zc[k]) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) pk[c] = 0u;
                        if constexpr (softmax) {  // P^T = 0, so dS of the chunk comes out 0
#pragma unroll
                            for (int c = 32 * k; c < 32 * k + 32; ++c) pv[c] = 0.f;
                        }
                    } else if (softmax) {
#pragma unroll
                        for (int c = 32 * k; c < 32 * k + 32; c += 4) {
                            const float4 l4 = *reinterpret_cast<const float4*>(lse_s + c);
                            float2 a0 = make_float2(l4.x, l4.y), a1 = make_float2(l4.z, l4.w);
                            if (!cconst[k]) {
                                a0 = add2(a0, make_float2(rrow[c], rrow[c + 1]));
                                a1 = add2(a1, make_float2(rrow[c + 2], rrow[c + 3]));
                            }
                            const float2 e0 = fma2(make_float2(pv[c], pv[c + 1]), xs2, a0);
                            const float2 e1 = fma2(make_float2(pv[c + 2], pv[c + 3]), xs2, a1);
                            pv[c] = ex2_approx(e0.x);
                            pv[c + 1] = ex2_approx(e0.y);
                            pv[c + 2] = ex2_approx(e1.x);
                            pv[c + 3] = ex2_approx(e1.y);
                        }
                        if (!full) {
#pragma unroll
                            for (int c = 32 * k; c < 32 * k + 32; ++c) pv[c] = (c >= lo && c < hi) ? pv[c] : 0.f;
                        }
#pragma unroll
                        for (int c = 0; c < 32; c += 2) pk[c >> 1] = pack_bf16x2(pv[32 * k + c], pv[32 * k + c + 1]);
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; c += 2) {
                            const int cc = 32 * k + c;
                            float a0, a1, d0, d1;
                            const bool v0 = full || (cc >= lo && cc < hi), v1 = full || (cc + 1 >= lo && cc + 1 < hi);
                            const float b0 = cconst[k] ? cbias[k] : rrow[cc];
                            const float b1 = cconst[k] ? cbias[k] : rrow[cc + 1];
                            gdpa_act_grad(gelu, fmaf(pv[cc], xs, b0), a0, d0);
                            gdpa_act_grad(gelu, fmaf(pv[cc + 1], xs, b1), a1, d1);
                            pk[c >> 1] = pack_bf16x2(v0 ? a0 : 0.f, v1 ? a1 : 0.f);
                            pv[cc] = v0 ? d0 : 0.f;
                            pv[cc + 1] = v1 ? d1 : 0.f;
                        }
                    }
                    tmem_st16(tX + 16u * k, pk);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(FU_P_FULL + k));
                }

                // dQ of the previous step, drained once this step's P^T is out, so that dK and dQ
                // of the previous step run on the tensor core during the P^T phase; Y must be
                // free before dP of this step is issued.
                if (i > 0 && !drain(g - 1, dq_x0, q0, q_len, qrow0 - C::BM)) { ok = false; break; }

                if (!warp_wait(FU_DP_FULL, g & 1)) { ok = false; break; }
                tc_fence_after();
                // This warp's rows of the dS tile are its dQ staging: the last box must have
                // left it before dS is written there.
                if (lane == 0) bulk_wait_read();
                __syncwarp();
                // dS = P^T (dP^T - Delta) (softmax) or act' dP^T (GDPA), 32 columns at a time,
                // into this thread's row of the dS tile (pieces 4k .. 4k+3 of the row).
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    uint32_t pd[16];
                    bool zero = false;
                    if constexpr (GDPA) zero = zc[k];
                    if (zero) {  // dS = 0: written without reading dP^T
#pragma unroll
                        for (int c = 0; c < 16; ++c) pd[c] = 0u;
                    } else {
                        float dp[32];
                        {
                            uint32_t (&ra)[32] = *reinterpret_cast<uint32_t(*)[32]>(dp);
                            tmem_ld32(tY + 32u * k, ra);
                            tmem_ld_wait(ra);
                        }
                        if (softmax) {
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
                    for (int q = 0; q < 4; ++q)
                        st_shared_v4(ds_row + uint32_t((((4 * k + q) ^ (r & 7))) << 4), pd[4 * q], pd[4 * q + 1],
                                     pd[4 * q + 2], pd[4 * q + 3]);
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(FU_DS_FULL + k));
                }
            }
            if (!ok) break;
            // dQ of the item's last step
            if (!drain(step_it + uint32_t(n) - 1, dq_x0, q0, q_len, (first_qt + n - 1) * C::BM)) { ok = false; break; }
            // Epilogue: dV and dK (times scale) of this key row, the warpgroup's half of D.
            if (!warp_wait(FU_ACC_FULL, item_it & 1)) { ok = false; break; }
            tc_fence_after();
            {
                const uint32_t valid = __ballot_sync(0xffffffffu, key_valid);
                if (D == 128 && valid == 0xffffffffu) {
                    // Every key row of the warp lies in the sequence: each accumulator's 32 rows x
                    // 64 columns are packed into the staging (the 128-byte-swizzled box layout)
                    // and written by one TMA store.  (A box cannot skip rows, so a warp holding
                    // the sequence's end, whose later rows belong to the next sequence, takes the
                    // row-by-row path below.)
                    const int ky = kv0 + nt * C::BN + (warp & 3) * 32;  // the warp's first key row
#pragma unroll
                    for (int t = 0; t < 2; ++t) {  // dV, then dK
                        const float mul = t ? p.scale : 1.f;
                        uint32_t w[32];  // bf16 pairs of columns (2k, 2k + 1)
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            uint32_t rr[32];
                            tmem_ld32(tmem + lane_base + (t ? C::kTmDK : C::kTmDV) + uint32_t(wg * 64 + 32 * cc), rr);
                            tmem_ld_wait(rr);
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                w[16 * cc + i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * mul,
                                                             __uint_as_float(rr[2 * i + 1]) * mul);
                        }
                        if (lane == 0) bulk_wait_read();  // the staging's previous box has been read
                        __syncwarp();
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            st_shared_v4(stg + uint32_t(lane * 128 + ((q ^ (lane & 7)) << 4)), w[4 * q], w[4 * q + 1],
                                         w[4 * q + 2], w[4 * q + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(t ? &tmDK : &tmDV, stg, h * D + wg * 64, ky);
                            bulk_commit();
                        }
                    }
                } else {
                    const uint32_t stage_w = sbase + uint32_t(C::kOffStage + warp * 2048);
                    const size_t off0 =
                        ((size_t(kv0) + size_t(nt * C::BN + (warp & 3) * 32)) * size_t(p.H) + size_t(h)) * D +
                        size_t(wg * C::kEpiCols);
                    const size_t stride = size_t(p.H) * D;
#pragma unroll
                    for (int cc = 0; cc < C::kEpiCols / 32; ++cc) {
#pragma unroll
                        for (int t = 0; t < 2; ++t) {  // dV, then dK
                            uint32_t rr[32];
                            tmem_ld32(tmem + lane_base + (t ? C::kTmDK : C::kTmDV) + uint32_t(wg * C::kEpiCols + 32 * cc),
                                      rr);
                            tmem_ld_wait(rr);
                            store_chunk_bf16(stage_w, rr, t ? p.scale : 1.f, lane, valid,
                                             reinterpret_cast<__nv_bfloat16*>(t ? p.dK : p.dV) + off0 + 32 * cc, stride);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(FU_ACC_EMPTY));
            step_it += uint32_t(n);
            ++item_it;
        }
        if (!ok) fail();
        // Every dQ reduce-add this warp issued has completed before the CTA exits.
        if (lane == 0) bulk_wait_done();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kMmaWarp) tmem_dealloc(tmem, 512);
}

template <int D, bool GDPA>
cudaError_t launch_fused_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const CUtensorMap& tmdO, const CUtensorMap& tmDQ, const CUtensorMap& tmDK,
                           const CUtensorMap& tmDV, const BwdParams& p, int grid, cudaStream_t st) {
    using C = FuCfg<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(jfa_bwd_fused_kernel<D, GDPA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    jfa_bwd_fused_kernel<D, GDPA><<<grid, C::kThreads, C::kSmemBytes, st>>>(tmQ, tmK, tmV, tmdO, tmDQ, tmDK, tmDV, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_fused(int D, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const CUtensorMap& tmdO, const CUtensorMap& tmDQ, const CUtensorMap& tmDK,
                             const CUtensorMap& tmDV, const BwdParams& p, int grid, cudaStream_t st) {
    const bool sm = p.mode == JFA_SOFTMAX;
    if (D == 128)
        return sm ? launch_fused_t<128, false>(tmQ, tmK, tmV, tmdO, tmDQ, tmDK, tmDV, p, grid, st)
                  : launch_fused_t<128, true>(tmQ, tmK, tmV, tmdO, tmDQ, tmDK, tmDV, p, grid, st);
    if (D == 64)
        return sm ? launch_fused_t<64, false>(tmQ, tmK, tmV, tmdO, tmDQ, tmDK, tmDV, p, grid, st)
                  : launch_fused_t<64, true>(tmQ, tmK, tmV, tmdO, tmDQ, tmDK, tmDV, p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace jfa
