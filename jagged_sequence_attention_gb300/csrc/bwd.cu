// Backward kernels for jagged flash attention / GDPA on sm_103a.
//
// The backward is parallelised over key/value tiles, as the kerneldigest.dev summary
// of the GEM work describes for JFA ("paralelización de backward pass", section
// "Arquitectura del Sistema"), and it accumulates no gradient into a padded tensor:
// the vibekk.com article names that "backward accumulation" among the bottlenecks
// left once padding is gone (section 第一轮瓶颈迁移).  For bf16 inputs it runs as
// three launches:
//
//   preprocess  Delta_i = sum_d dO_id O_id (softmax only)
//   dK/dV       this file: persistent over (sequence, head, 128-row key tile).  K and V
//               stay in shared memory while 128-row query tiles stream through:
//                 S^T  = K Q_i^T      (TMEM, lanes = key rows)
//                 dP^T = V dO_i^T     (TMEM)
//                 P^T  = exp2(S^T - lse) or act(S^T), written back over S^T as bf16
//                 dS^T = P^T (dP^T - Delta) or act'(S^T) dP^T, written over dP^T
//                 dV  += P^T dO_i,  dK += dS^T Q_i   (A operand read from TMEM)
//   dQ          bwd_dq.cu: persistent over (sequence, head, 128-row query tile), the
//               forward's geometry: dQ = sum over key tiles of dS K_j, in TMEM.
//
// The dQ pass recomputes S and dP instead of adding into a shared fp32 dQ buffer
// from every key tile: that costs two extra tensor-core products per tile pair but
// removes the atomic traffic (key tiles x query rows x D x 4 bytes, about 0.4 TB for
// a million-token causal batch), a workspace of T_q x H x D floats and a conversion
// pass.  Every product is 128 x 128 x D or 128 x D x 128, the tensor core's full
// rate; P and dS never go through shared memory.
//
// dK/dV CTA = 10 warps: 0-7 compute (warpgroup g owns query columns [64g, 64g+64) of
// a step; thread = key row = TMEM lane) and write the dK/dV epilogue, 8 TMA producer,
// 9 MMA issuer.  TMEM: dV [0,128), dK [128,256), S^T/P^T [256,384), dP^T/dS^T
// [384,512).  Issue order per step: S(i+1), dK(i), dP(i+1), dV(i+1); each product
// that must wait for a TMEM region to be consumed finds another product queued
// ahead of it.  P^T and dS^T are signalled per 32-column chunk, so dV and dK start on
// the first chunk while the second is being formed.
#include <algorithm>

#include "bwd_common.cuh"
#include "jfa_internal.h"
#include "ptx.cuh"
#include "tilemath.cuh"

namespace jfa {

namespace {

template <int D>
struct KvCfg {
    static constexpr int BN = kBwdBN;  // key rows (TMEM lanes)
    static constexpr int BM = kBwdBM;  // query rows per step
    static constexpr int kRowBytes = D * 2;
    static_assert(kRowBytes % 128 == 0 && kRowBytes <= 256, "head row must be 128 or 256 bytes");
    static constexpr int kCB = kRowBytes / 128;  // 128-byte column blocks of a row
    static constexpr int kBoxCols = 64;          // bf16 elements per 128-byte box row
    static constexpr int kKVTile = BN * kRowBytes;
    static constexpr int kQTile = BM * kRowBytes;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kKVTile;
    static constexpr int kOffQ = 2 * kKVTile;          // + stage * kQTile
    static constexpr int kOffDO = kOffQ + 2 * kQTile;  // + stage * kQTile
    static constexpr int kOffBar = kOffDO + 2 * kQTile;
    static constexpr int kNumBars = 24;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kCompWarps = kDkdvCompWarps;
    static constexpr int kCols = BM / 2;  // query columns per compute thread
    // tmem slot + abort flag (16 B); per compute warp: -lse and -Delta of its columns, the
    // head's bias row, a step's bias-by-relative-position table (kCols + 32 entries) and
    // the item's bias-table gradient by bucket (32 entries)
    static constexpr int kRelTab = kCols + 32;
    static constexpr int kWarpMisc = 2 * kCols + 32 + kRelTab + 32;
    static constexpr int kMiscBytes = 16 + kCompWarps * kWarpMisc * 4;
    // per compute warp: a 2 KB buffer through which the epilogue's stores are regrouped
    static constexpr int kOffStage = (kOffMisc + kMiscBytes + 127) / 128 * 128;
    static constexpr int kSmemNeed = kOffStage + kCompWarps * 2048 + 1024;
    // At least 120 KB so that exactly one CTA fits on an SM: it allocates all 512 TMEM columns.
    static constexpr int kSmemBytes = kSmemNeed > 120 * 1024 ? kSmemNeed : 120 * 1024;
    static constexpr int kDSteps = D / 16;   // contraction over head_dim
    static constexpr int kQSteps = BM / 16;  // contraction over query rows
    // dV/dK issue their K-steps per (warpgroup, 32-column chunk): 2 x 2 x 2 steps
    static_assert(kQSteps == 8 && kCols == 64, "chunked dV/dK issue assumes 128-row query steps");
    static constexpr uint32_t kTmDV = 0, kTmDK = 128, kTmX = 256, kTmY = 384;
    static constexpr uint32_t kIdescS = make_idesc(kFmtBF16, BN, BM, false, false);
    static constexpr uint32_t kIdescAcc = make_idesc(kFmtBF16, BN, D, false, true);
    static constexpr int kEpiCols = D / 2;  // dK/dV columns each warpgroup writes
    static constexpr int kProdWarp = kCompWarps, kMmaWarp = kCompWarps + 1, kThreads = (kCompWarps + 2) * 32;
};

enum {
    KV_K_FULL = 0,
    KV_V_FULL = 1,
    KV_KV_EMPTY = 2,
    KV_Q_FULL = 3,    // +stage
    KV_Q_EMPTY = 5,   // +stage
    KV_DO_FULL = 7,   // +stage
    KV_DO_EMPTY = 9,  // +stage
    KV_S_FULL = 11,
    KV_P_FULL = 12,   // +chunk: columns [32k, 32k+32) of both warpgroups' P^T are in TMEM
    KV_DP_FULL = 14,
    KV_DS_FULL = 15,  // +chunk, as for P^T
    KV_X_FREE = 17,   // dV(i) done: the S^T/P^T columns may be rewritten
    KV_Y_FREE = 18,   // dK(i) done: the dP^T/dS^T columns may be rewritten
    KV_ACC_FULL = 19,
    KV_ACC_EMPTY = 20,
    KV_DRAIN = 21,
};

// Warp sum by xor-shuffles: every lane receives the total, in the same order each run.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// DBIAS: also accumulate the gradient of the relative-position bias table, the sum of
// dS over the allowed pairs of each bucket, into per-(CTA, warp) partial tables that a
// second kernel sums in a fixed order (so the result is the same on every run).
// DENSE: the bias is the dense per-pair array p.dense, read per element; with p.ddense
// set, dS of every allowed pair is also stored there (its gradient).
// SHARED: shared key/value; an item is a user's key tile and its steps, read from
// p.steps, are the (query set, query tile) pairs of all the user's query sets, so that
// dK and dV accumulate the broadcast's gradient in TMEM and are written once.
template <int D, bool GDPA, bool DBIAS, bool DENSE, bool SHARED>
__global__ void __launch_bounds__(320, 1)
    jfa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                        const BwdParams p) {
    using C = KvCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sK = sbase + C::kOffK, sV = sbase + C::kOffV, sQ = sbase + C::kOffQ, sDO = sbase + C::kOffDO;
    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * uint32_t(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    float* misc_f = reinterpret_cast<float*>(smem + C::kOffMisc + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(bar(KV_K_FULL), 1);
        mbar_init(bar(KV_V_FULL), 1);
        mbar_init(bar(KV_KV_EMPTY), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(KV_Q_FULL + s), 1);
            mbar_init(bar(KV_Q_EMPTY + s), 1);
            mbar_init(bar(KV_DO_FULL + s), 1);
            mbar_init(bar(KV_DO_EMPTY + s), 1);
        }
        mbar_init(bar(KV_S_FULL), 1);
        mbar_init(bar(KV_P_FULL), C::kCompWarps);
        mbar_init(bar(KV_P_FULL + 1), C::kCompWarps);
        mbar_init(bar(KV_DP_FULL), 1);
        mbar_init(bar(KV_DS_FULL), C::kCompWarps);
        mbar_init(bar(KV_DS_FULL + 1), C::kCompWarps);
        mbar_init(bar(KV_X_FREE), 1);
        mbar_init(bar(KV_Y_FREE), 1);
        mbar_init(bar(KV_ACC_FULL), 1);
        mbar_init(bar(KV_ACC_EMPTY), C::kCompWarps);
        mbar_init(bar(KV_DRAIN), 1);
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
            uint32_t step_it = 0, item_it = 0;
            uint32_t q_extra = 0;  // 1: the last step's Q load went out but its dO load did not
            bool ok = true;
            for (int it = it_begin; it < it_end && ok; ++it) {
                const int4 w = p.items[it];
                if (!kv_item_ok(w, p, SHARED)) {  // not an item of this plan: skipped by every role
                    atomicOr(p.status, kStatusBounds);
                    continue;
                }
                const int n = w.w;
                if (n == 0) continue;
                const int b = w.x, h = w.y, nt = w.z;  // b: key/value sequence (shared: the user)
                const int q0 = SHARED ? 0 : p.q_off[b], kv0 = p.kv_off[b];
                int first_qt = 0, nq;  // query tiles [first_qt, first_qt + n) see this key tile
                if (!SHARED) query_tile_range(p.q_off[b + 1] - q0, p.kv_off[b + 1] - kv0, nt, p.causal, p.window, first_qt, nq);
                const int s0 = SHARED ? p.step_off[p.ktile_off[b] + nt] : 0;
                if (!mbar_wait_bounded(bar(KV_KV_EMPTY), (item_it & 1) ^ 1, abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(KV_K_FULL), C::kKVTile);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb)
                    tma_load_2d(sK + cb * C::BN * 128, &tmK, bar(KV_K_FULL), h * D + cb * C::kBoxCols, kv0 + nt * C::BN);
                mbar_arrive_expect_tx(bar(KV_V_FULL), C::kKVTile);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb)
                    tma_load_2d(sV + cb * C::BN * 128, &tmV, bar(KV_V_FULL), h * D + cb * C::kBoxCols, kv0 + nt * C::BN);
                ++item_it;
                for (int i = 0; i < n; ++i, ++step_it) {
                    const uint32_t st = step_it & 1, ph = (step_it >> 1) & 1;
                    int y;
                    if constexpr (SHARED) {
                        const int2 stp = p.steps[s0 + i];
                        y = p.q_off[stp.x] + stp.y * C::BM;
                    } else {
                        y = q0 + (first_qt + i) * C::BM;
                    }
                    if (!mbar_wait_bounded(bar(KV_Q_EMPTY + st), ph ^ 1, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(bar(KV_Q_FULL + st), C::kQTile);
#pragma unroll
                    for (int cb = 0; cb < C::kCB; ++cb)
                        tma_load_2d(sQ + st * C::kQTile + cb * C::BM * 128, &tmQ, bar(KV_Q_FULL + st),
                                    h * D + cb * C::kBoxCols, y);
                    if (!mbar_wait_bounded(bar(KV_DO_EMPTY + st), ph ^ 1, abort_flag)) {
                        q_extra = 1;
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(KV_DO_FULL + st), C::kQTile);
#pragma unroll
                    for (int cb = 0; cb < C::kCB; ++cb)
                        tma_load_2d(sDO + st * C::kQTile + cb * C::BM * 128, &tmdO, bar(KV_DO_FULL + st),
                                    h * D + cb * C::kBoxCols, y);
                }
            }
            if (!ok) fail();
            // Drain: wait until every load this thread issued has landed.
            if (item_it > 0) {
                mbar_wait_bounded(bar(KV_K_FULL), (item_it - 1) & 1, nullptr);
                mbar_wait_bounded(bar(KV_V_FULL), (item_it - 1) & 1, nullptr);
            }
            drain_ring(bar(KV_Q_FULL), step_it + q_extra, 2);
            drain_ring(bar(KV_DO_FULL), step_it, 2);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the schedule, so descriptors and counters stay
        // warp-uniform; one elected lane (always lane 0) issues every MMA and commit.
        uint32_t step_it = 0, item_it = 0, dv_cnt = 0, dk_cnt = 0;
        bool ok = true;
        const SDesc dKa = sdesc_sw128(sK, 16, 1024), dVa = sdesc_sw128(sV, 16, 1024);
        // Descriptors of both ring stages, selected by value (no indexed array, which
        // would live in local memory).
        const SDesc dQk0 = sdesc_sw128(sQ, 16, 1024), dQk1 = sdesc_sw128(sQ + C::kQTile, 16, 1024);
        const SDesc dOk0 = sdesc_sw128(sDO, 16, 1024), dOk1 = sdesc_sw128(sDO + C::kQTile, 16, 1024);
        const SDesc dQm0 = sdesc_sw128(sQ, C::BM * 128, 1024), dQm1 = sdesc_sw128(sQ + C::kQTile, C::BM * 128, 1024);
        const SDesc dOm0 = sdesc_sw128(sDO, C::BM * 128, 1024), dOm1 = sdesc_sw128(sDO + C::kQTile, C::BM * 128, 1024);
        // K step s of a head_dim contraction: 128-byte column block (s*32)>>7,
        // (s*32)&127 bytes into the row; both operands have 128 rows.
        auto koff = [](int s) -> uint32_t { return uint32_t(((s * 32) >> 7) * 128 * 128 + ((s * 32) & 127)); };
        // S^T(g) = K Q^T into the S^T columns, once dV of the previous step has read P^T there.
        auto issue_s = [&](uint32_t g) -> bool {
            const uint32_t st = g & 1, ph = (g >> 1) & 1;
            if (!warp_wait(KV_Q_FULL + st, ph)) return false;
            if (dv_cnt > 0 && !warp_wait(KV_X_FREE, (dv_cnt - 1) & 1)) return false;
            tc_fence_after();
            const SDesc dq = st ? dQk1 : dQk0;
            if (elect_one()) {
#pragma unroll
                for (int s = 0; s < C::kDSteps; ++s) mma_ss(tmem + C::kTmX, dKa, koff(s), dq, koff(s), C::kIdescS, s > 0);
                tc_commit(bar(KV_S_FULL));
            }
            __syncwarp();
            return true;
        };
        // dP^T(g) = V dO^T into the dP^T columns, once dK of the previous step has read dS^T there.
        auto issue_dp = [&](uint32_t g) -> bool {
            const uint32_t st = g & 1, ph = (g >> 1) & 1;
            if (!warp_wait(KV_DO_FULL + st, ph)) return false;
            if (dk_cnt > 0 && !warp_wait(KV_Y_FREE, (dk_cnt - 1) & 1)) return false;
            tc_fence_after();
            const SDesc dO = st ? dOk1 : dOk0;
            if (elect_one()) {
#pragma unroll
                for (int s = 0; s < C::kDSteps; ++s) mma_ss(tmem + C::kTmY, dVa, koff(s), dO, koff(s), C::kIdescS, s > 0);
                tc_commit(bar(KV_DP_FULL));
            }
            __syncwarp();
            return true;
        };
        // The K-steps (16 query rows each) that read chunk c of the packed operand:
        // warpgroup w's chunk c covers query rows 64w + 32c .. + 31, K-steps 4w + 2c, +1.
        auto chunk_step = [](int c, int i) -> int { return 4 * (i >> 1) + 2 * c + (i & 1); };
        // dV += P^T dO with P^T read from TMEM, chunk by chunk as the compute warps
        // finish it; the first step of an item waits for the epilogue of the previous
        // item to have read the accumulators.
        auto issue_dv = [&](uint32_t g, bool first) -> bool {
            const uint32_t st = g & 1;
            const SDesc dO = st ? dOm1 : dOm0;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (!warp_wait(KV_P_FULL + c, g & 1)) return false;
                if (c == 0 && first && !warp_wait(KV_ACC_EMPTY, (item_it & 1) ^ 1)) return false;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int s = chunk_step(c, i);
                        mma_ts(tmem + C::kTmDV, tmem + C::kTmX + packed_col(s), dO, s * 16 * 128, C::kIdescAcc,
                               (!first || c > 0 || i > 0));
                    }
                    if (c == 1) {
                        tc_commit(bar(KV_X_FREE));
                        tc_commit(bar(KV_DO_EMPTY + st));
                    }
                }
                __syncwarp();
            }
            ++dv_cnt;
            return true;
        };
        // dK += dS^T Q with dS^T read from TMEM, chunk by chunk.
        auto issue_dk = [&](uint32_t g, bool first) -> bool {
            const uint32_t st = g & 1;
            const SDesc dq = st ? dQm1 : dQm0;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (!warp_wait(KV_DS_FULL + c, g & 1)) return false;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int s = chunk_step(c, i);
                        mma_ts(tmem + C::kTmDK, tmem + C::kTmY + packed_col(s), dq, s * 16 * 128, C::kIdescAcc,
                               (!first || c > 0 || i > 0));
                    }
                    if (c == 1) {
                        tc_commit(bar(KV_Y_FREE));
                        tc_commit(bar(KV_Q_EMPTY + st));
                    }
                }
                __syncwarp();
            }
            ++dk_cnt;
            return true;
        };
        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 wi = p.items[it];
            if (!kv_item_ok(wi, p, SHARED)) continue;
            const int n = wi.w;
            if (n == 0) continue;
            if (!warp_wait(KV_K_FULL, item_it & 1) || !warp_wait(KV_V_FULL, item_it & 1)) { ok = false; break; }
            tc_fence_after();
            const uint32_t g0 = step_it;
            if (!issue_s(g0) || !issue_dp(g0) || !issue_dv(g0, true)) { ok = false; break; }
            for (int i = 0; i < n && ok; ++i) {
                const uint32_t g = g0 + uint32_t(i);
                // S^T(i+1) goes ahead of dK(i): it needs only dV(i) to have read P^T, so it runs
                // while the compute warps form dS^T(i), and their next P^T phase starts as soon
                // as dS^T(i) is done instead of after dK(i) and S^T(i+1) have run.
                if (i + 1 < n && !issue_s(g + 1)) { ok = false; break; }
                if (!issue_dk(g, i == 0)) { ok = false; break; }
                if (i + 1 < n && (!issue_dp(g + 1) || !issue_dv(g + 1, false))) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            if (elect_one()) {
                tc_commit(bar(KV_ACC_FULL));
                tc_commit(bar(KV_KV_EMPTY));
            }
            __syncwarp();
            step_it += uint32_t(n);
            ++item_it;
        }
        if (!ok) fail();
        if (elect_one()) tc_commit(bar(KV_DRAIN));
        __syncwarp();
        mbar_wait_bounded(bar(KV_DRAIN), 0, nullptr);
    } else {
        // ------------------------------------------------------------ P^T, dS^T, epilogue
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
        float* dacc_w = rtab + C::kRelTab;              // the item's table gradient by bucket
        // This warp's partial table gradient [H][32], owned by this warp alone.
        float* dpart = DBIAS ? p.dbias_part + (size_t(blockIdx.x) * C::kCompWarps + size_t(warp)) * size_t(p.H) * 32
                             : nullptr;
        // Gradient of warp-constant chunks: a per-thread sum for each chunk slot, tagged
        // with the (warp-uniform) bucket it belongs to, flushed when the bucket changes.
        float dacc[2] = {0.f, 0.f};
        int dtag[2] = {-1, -1};
        auto dflush = [&](int k) {
            if (dtag[k] >= 0) {
                const float v = warp_sum(dacc[k]);
                if (lane == 0) dacc_w[dtag[k]] += v;
            }
            dacc[k] = 0.f;
        };
        if constexpr (DBIAS) {
            dacc_w[lane] = 0.f;
            for (int e = lane; e < p.H * 32; e += 32) dpart[e] = 0.f;
            __syncwarp();
        }
        // Element (lane, c) has relative position rbase(lane 0) - lane + c: rtab[k] holds
        // the bias of rbase(lane 0) - 31 + k, so the lane reads rrow[c], rrow = rtab + 31 - lane.
        const float* rrow = rtab + 31 - lane;
        constexpr bool softmax = !GDPA;  // the other mode's code is not compiled in
        const bool gelu = p.mode == JFA_GDPA_GELU_TANH;
        uint32_t step_it = 0, item_it = 0;
        bool ok = true;
        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 w = p.items[it];
            if (!kv_item_ok(w, p, SHARED)) continue;
            const int n = w.w, b = w.x, h = w.y, nt = w.z;  // b: key/value sequence (shared: the user)
            const int kv0 = p.kv_off[b], kv_len = p.kv_off[b + 1] - kv0;
            // The query sequence of the item (not shared), or of each step (shared).
            const int q0 = SHARED ? 0 : p.q_off[b], q_len = SHARED ? 0 : p.q_off[b + 1] - q0;
            int first_qt = 0, nq;  // query tiles [first_qt, first_qt + n) see this key tile
            if (!SHARED) query_tile_range(q_len, kv_len, nt, p.causal, p.window, first_qt, nq);
            const int s0 = SHARED ? p.step_off[p.ktile_off[b] + nt] : 0;
            const int j = nt * C::BN + r;  // key row within the sequence
            const bool key_valid = j < kv_len;
            // Step i: query sequence sb (rows from sq0, sq_len of them), first row sqrow0.
            auto step_q = [&](int i, int& sb, int& sq0, int& sq_len, int& sqrow0) {
                if constexpr (SHARED) {
                    const int2 stp = p.steps[s0 + i];
                    sb = stp.x;
                    sq0 = p.q_off[sb];
                    sq_len = p.q_off[sb + 1] - sq0;
                    sqrow0 = stp.y * C::BM;
                } else {
                    sb = b;
                    sq0 = q0;
                    sq_len = q_len;
                    sqrow0 = (first_qt + i) * C::BM;
                }
            };
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
            // valid).  Nothing reads the loaded registers until that step, so the load's
            // latency is never waited for.
            float rl[2] = {0.f, 0.f}, rd[2] = {0.f, 0.f};
            uint32_t rv = 0;
            auto fetch = [&](int fq0, int fq_len, int qrow0) {
                rv = 0;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int c = qrow0 + c0 + 32 * k + lane;
                    const bool v = c < fq_len;
                    const size_t ridx = (size_t(fq0) + size_t(v ? c : 0)) * size_t(p.H) + size_t(h);
                    if constexpr (softmax) {
                        rl[k] = p.lse[ridx];
                        rd[k] = p.delta[ridx];
                    }
                    rv |= uint32_t(v) << k;
                }
            };
            {
                int fb, fq0, fql, fr0;
                step_q(0, fb, fq0, fql, fr0);
                fetch(fq0, fql, fr0);
            }
            for (int i = 0; i < n; ++i) {
                const uint32_t g = step_it + uint32_t(i);
                int sb, sq0, sq_len, qrow0;  // the step's query sequence and first query row
                step_q(i, sb, sq0, sq_len, qrow0);
                const int diag = kv_len - sq_len;
                // -lse in log2 units and -Delta of this step's columns (0 past the end)
                const float cur_nl0 = (softmax && (rv & 1u)) ? -rl[0] * 1.4426950408889634f : 0.f;
                const float cur_nl1 = (softmax && (rv & 2u)) ? -rl[1] * 1.4426950408889634f : 0.f;
                __syncwarp();
                del_s[lane] = (softmax && (rv & 1u)) ? -rd[0] : 0.f;
                del_s[32 + lane] = (softmax && (rv & 2u)) ? -rd[1] : 0.f;
                if (i + 1 < n) {
                    int fb, fq0, fql, fr0;
                    step_q(i + 1, fb, fq0, fql, fr0);
                    fetch(fq0, fql, fr0);
                }
                // dense bias / gradient of key j: element (query row i) at [i * kv_len]
                const size_t dbase = DENSE ? size_t(h) * size_t(p.n_pairs) + size_t(p.pair_off[sb]) +
                                                 size_t(key_valid ? j : 0)
                                           : 0;
                // subtraction scheme: valid local columns are [lo, hi)
                int hi = key_valid ? min(NC, sq_len - qrow0 - c0) : 0;
                // sliding window: query i sees key j only while j >= i' - W, i.e. i <= j - diag + W
                if (p.window >= 0) hi = min(hi, j - diag + p.window + 1 - qrow0 - c0);
                const int lo = p.causal ? max(0, j - diag - qrow0 - c0) : 0;
                const bool full = __all_sync(0xffffffffu, lo == 0 && hi == NC);
                const int rbase = qrow0 + c0 + diag - j;  // relative position of local column 0
                const float xs = softmax ? p.scale_log2 : p.scale;
                // dense bias of local column c: dsrc[c * kv_len] (read only for c in [lo, hi))
                const float* dsrc = DENSE ? p.dense + dbase + size_t(qrow0 + c0) * size_t(kv_len) : nullptr;
                // Bias per 32-column chunk: one value when every lane's chunk sits in
                // one bucket, else read per element from the relative-position table.
                // Lane k tests chunk k for the whole warp: over the warp's keys, chunk k
                // spans relative positions rbase(lane 0) + 32k - 31 .. + 62.
                bool cconst[2] = {true, true};
                float cbias[2] = {0.f, 0.f};
                int cbk[2] = {0, 0};  // the bucket of a warp-constant chunk (DBIAS)
                if (p.bias) {
                    const int rb0 = __shfl_sync(0xffffffffu, rbase, 0);
                    int bk = 0;
                    const uint32_t cm = warp_const_chunks(lane < 2, rb0 + 32 * lane - 31, bk);
                    const float bv = bias_w[bk];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        cconst[k] = (cm >> k) & 1u;
                        cbias[k] = __shfl_sync(0xffffffffu, bv, k);
                        if constexpr (DBIAS) cbk[k] = __shfl_sync(0xffffffffu, bk, k);
                    }
                }
                // Staged addend of column c: -lse, plus the chunk's bias when that is
                // one value for the whole warp (it then is the same for every lane).
                lse_s[lane] = cur_nl0 + (cconst[0] ? cbias[0] : 0.f);
                lse_s[32 + lane] = cur_nl1 + (cconst[1] ? cbias[1] : 0.f);
                if (!(cconst[0] && cconst[1])) {
                    const int r0 = __shfl_sync(0xffffffffu, rbase, 0) - 31;
#pragma unroll
                    for (int m = 0; m < C::kRelTab / 32; ++m)
                        rtab[lane + 32 * m] = bias_w[relpos_bucket(r0 + lane + 32 * m)];
                }
                __syncwarp();

                // A 32-column chunk masked for every key row of the warp (query rows past the
                // sequence's end, or all before the causal diagonal, or no valid key row) has
                // P^T = dS^T = 0: it skips the exponent or activation and writes zeros (steps
                // with no masked column never test this).  Softmax zeroes P and forms dS^T = 0
                // on the common path; GDPA also skips the chunk's loads and dS^T arithmetic.
                // Each is the faster of the two forms for its mode.
                const bool zc[2] = {!full && __all_sync(0xffffffffu, hi <= 0 || lo >= 32),
                                    !full && __all_sync(0xffffffffu, hi <= 32 || lo >= NC)};
                if (!warp_wait(KV_S_FULL, g & 1)) { ok = false; break; }
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
                // bias) (GDPA; pv keeps act' for dS), one 32-column chunk at a time: each
                // chunk is packed over the warpgroup's own S^T columns (already read) and
                // signalled at once, so dV can start on it while the next chunk is formed.
                const float2 xs2 = make_float2(xs, xs);
                // Fast steps (no column masked, both chunks' bias warp-constant) take a
                // branch-free copy of the exponent loop.
                const bool fast = !DENSE && full && cconst[0] && cconst[1];
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
                        if constexpr (softmax) {  // P^T = 0, so dS^T of the chunk comes out 0
#pragma unroll
                            for (int c = 32 * k; c < 32 * k + 32; ++c) pv[c] = 0.f;
                        }
                    } else if (softmax) {
                        // exponent = xs * s + (bias - lse): the staged addend already holds
                        // the bias of a warp-constant chunk; other chunks add it per element
                        // from the relative-position table.
#pragma unroll
                        for (int c = 32 * k; c < 32 * k + 32; c += 4) {
                            const float4 l4 = *reinterpret_cast<const float4*>(lse_s + c);
                            float2 a0 = make_float2(l4.x, l4.y), a1 = make_float2(l4.z, l4.w);
                            if constexpr (DENSE) {
                                float bv[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    bv[e] = (c + e >= lo && c + e < hi) ? __ldg(dsrc + size_t(c + e) * size_t(kv_len)) : 0.f;
                                const float2 l2e = make_float2(1.4426950408889634f, 1.4426950408889634f);
                                a0 = fma2(make_float2(bv[0], bv[1]), l2e, a0);
                                a1 = fma2(make_float2(bv[2], bv[3]), l2e, a1);
                            } else if (!cconst[k]) {
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
                            float b0, b1;
                            if constexpr (DENSE) {
                                b0 = v0 ? __ldg(dsrc + size_t(cc) * size_t(kv_len)) : 0.f;
                                b1 = v1 ? __ldg(dsrc + size_t(cc + 1) * size_t(kv_len)) : 0.f;
                            } else {
                                b0 = cconst[k] ? cbias[k] : rrow[cc];
                                b1 = cconst[k] ? cbias[k] : rrow[cc + 1];
                            }
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
                    if (lane == 0) mbar_arrive(bar(KV_P_FULL + k));
                }

                if (!warp_wait(KV_DP_FULL, g & 1)) { ok = false; break; }
                tc_fence_after();
                // dS^T = P^T (dP^T - Delta) (softmax) or act' dP^T (GDPA), 32 columns at a
                // time, packed over the warpgroup's own dP^T columns (already read).
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    if constexpr (GDPA) {
                        if (zc[k]) {  // dS^T = 0: written without reading dP^T
                            uint32_t pd[16];
#pragma unroll
                            for (int c = 0; c < 16; ++c) pd[c] = 0u;
                            tmem_st16(tY + 16u * k, pd);
                            tmem_st_wait();
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(bar(KV_DS_FULL + k));
                            continue;
                        }
                    }
                    float dp[32];
                    {
                        uint32_t (&ra)[32] = *reinterpret_cast<uint32_t(*)[32]>(dp);
                        tmem_ld32(tY + 32u * k, ra);
                        tmem_ld_wait(ra);
                    }
                    uint32_t pd[16];
                    float2 cs = make_float2(0.f, 0.f);  // the chunk's dS sum (DBIAS)
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
                            if constexpr (DBIAS || DENSE) {  // keep dS (fp32) for a bias gradient
                                dp[c] = a.x;
                                dp[c + 1] = a.y;
                                dp[c + 2] = b2.x;
                                dp[c + 3] = b2.y;
                            }
                            if constexpr (DBIAS) cs = add2(cs, add2(a, b2));
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; c += 2) {
                            const float2 a = mul2(make_float2(pv[32 * k + c], pv[32 * k + c + 1]),
                                                  make_float2(dp[c], dp[c + 1]));
                            pd[c >> 1] = pack_bf16x2(a.x, a.y);
                            if constexpr (DBIAS || DENSE) {
                                dp[c] = a.x;
                                dp[c + 1] = a.y;
                            }
                            if constexpr (DBIAS) cs = add2(cs, a);
                        }
                    }
                    tmem_st16(tY + 16u * k, pd);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(KV_DS_FULL + k));
                    if constexpr (DENSE) {
                        // gradient of the dense bias: dS of the allowed pairs (lanes hold
                        // consecutive keys, so each column's store is one 128-byte line)
                        if (p.ddense) {
                            float* gdst = p.ddense + dbase + size_t(qrow0 + c0 + 32 * k) * size_t(kv_len);
#pragma unroll
                            for (int c = 0; c < 32; ++c)
                                if (32 * k + c >= lo && 32 * k + c < hi) gdst[size_t(c) * size_t(kv_len)] = dp[c];
                        }
                    }
                    if constexpr (DBIAS) {
                        // Table gradient of this chunk (dS is exactly 0 at masked pairs).
                        if (cconst[k]) {
                            if (cbk[k] != dtag[k]) {
                                dflush(k);
                                dtag[k] = cbk[k];
                            }
                            dacc[k] += cs.x + cs.y;
                        } else {
                            // Element (lane l, column c) lies on diagonal d = c - l + 31 of the
                            // chunk, relative position rlo + d.  Lane m gathers diagonals m and
                            // m + 32: from column c it takes lane (c + 31 - m) mod 32's element.
                            const int rlo = __shfl_sync(0xffffffffu, rbase, 0) + 32 * k - 31;
                            float g0 = 0.f, g1 = 0.f;
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                const float v = __shfl_sync(0xffffffffu, dp[c], (c + 31 - lane) & 31);
                                if (lane >= c) g0 += v; else g1 += v;
                            }
                            const int b0 = relpos_bucket(rlo + lane), b1 = relpos_bucket(rlo + lane + 32);
                            const int bmin = __reduce_min_sync(0xffffffffu, min(b0, b1));
                            const int bmax = __reduce_max_sync(0xffffffffu, max(b0, b1));
                            for (int kb = bmin; kb <= bmax; ++kb) {
                                const float v = warp_sum((b0 == kb ? g0 : 0.f) + (b1 == kb ? g1 : 0.f));
                                if (lane == 0) dacc_w[kb] += v;
                            }
                        }
                    }
                }
            }
            if (!ok) break;
            if constexpr (DBIAS) {
                // the item's table gradient into this warp's partial table of head h
                dflush(0);
                dflush(1);
                dtag[0] = dtag[1] = -1;
                __syncwarp();
                dpart[h * 32 + lane] += dacc_w[lane];
                dacc_w[lane] = 0.f;
                __syncwarp();
            }
            // Epilogue: dV and dK (times scale) of this key row, the warpgroup's half of D.
            if (!warp_wait(KV_ACC_FULL, item_it & 1)) { ok = false; break; }
            tc_fence_after();
            {
                const uint32_t stage_w = sbase + uint32_t(C::kOffStage + warp * 2048);
                const uint32_t valid = __ballot_sync(0xffffffffu, key_valid);
                // this warp's first key row (kv0 + key0) * H + h, then rows H * D elements apart
                const size_t off0 = ((size_t(kv0) + size_t(nt * C::BN + (warp & 3) * 32)) * size_t(p.H) + size_t(h)) * D +
                                    size_t(wg * C::kEpiCols);
                const size_t stride = size_t(p.H) * D;
#pragma unroll
                for (int cc = 0; cc < C::kEpiCols / 32; ++cc) {
#pragma unroll
                    for (int t = 0; t < 2; ++t) {  // dV, then dK
                        uint32_t rr[32];
                        tmem_ld32(tmem + lane_base + (t ? C::kTmDK : C::kTmDV) + uint32_t(wg * C::kEpiCols + 32 * cc), rr);
                        tmem_ld_wait(rr);
                        store_chunk_bf16(stage_w, rr, t ? p.scale : 1.f, lane, valid,
                                         reinterpret_cast<__nv_bfloat16*>(t ? p.dK : p.dV) + off0 + 32 * cc, stride);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(KV_ACC_EMPTY));
            step_it += uint32_t(n);
            ++item_it;
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kMmaWarp) tmem_dealloc(tmem, 512);
}

// Eight consecutive elements of a 16-byte aligned row, as floats (one or two 16-byte
// read-only loads).
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p)), b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Delta_i = sum_d dO_id * O_id for each (row, head): D/8 lanes per row, eight elements
// (16-byte loads) each, reduced across the lanes.
template <typename TO, typename T, int D>
__global__ void jfa_bwd_pre_kernel(const TO* __restrict__ O, const T* __restrict__ dO, float* __restrict__ delta,
                                   int64_t rows) {
    constexpr int kLanes = D / 8;
    static_assert(kLanes >= 1 && kLanes <= 32 && (32 % kLanes) == 0, "row lanes must tile a warp");
    const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t row = gid / kLanes;
    const int sub = int(gid % kLanes);
    float acc = 0.f;
    if (row < rows) {
        float o[8], g[8];
        load8(O + row * D + sub * 8, o);
        load8(dO + row * D + sub * 8, g);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc = fmaf(o[k], g[k], acc);
    }
#pragma unroll
    for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && sub == 0) delta[row] = acc;
}

// fp32 inputs: dQ = scale * accumulator.
template <typename T>
__global__ void jfa_bwd_post_kernel(const float4* __restrict__ acc, T* __restrict__ dQ, int64_t n4, float scale) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += int64_t(gridDim.x) * blockDim.x) {
        const float4 v = acc[i];
        if constexpr (sizeof(T) == 2) {
            uint2 u;
            u.x = pack_bf16x2(v.x * scale, v.y * scale);
            u.y = pack_bf16x2(v.z * scale, v.w * scale);
            reinterpret_cast<uint2*>(dQ)[i] = u;
        } else {
            reinterpret_cast<float4*>(dQ)[i] = make_float4(v.x * scale, v.y * scale, v.z * scale, v.w * scale);
        }
    }
}

// One thread per (head, bucket): the sum over the partial tables, slot by slot.
__global__ void jfa_dbias_reduce_kernel(const float* __restrict__ part, int64_t n_slots, int H, float* dbias) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= H * 32) return;
    float acc = 0.f;
    for (int64_t s = 0; s < n_slots; ++s) acc += part[s * H * 32 + e];
    dbias[e] = acc;
}

// fp32 path: one partial per work item; the item's head selects the row it adds to.
__global__ void jfa_dbias_reduce_items_kernel(const float* __restrict__ part, const int4* __restrict__ items,
                                              int64_t n_items, int H, float* dbias) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= H * 32) return;
    const int h = e >> 5, k = e & 31;
    float acc = 0.f;
    for (int64_t it = 0; it < n_items; ++it)
        if (items[it].y == h) acc += part[it * 32 + k];
    dbias[e] = acc;
}

template <int D, bool GDPA, bool DBIAS, bool DENSE, bool SHARED>
cudaError_t launch_dkdv_t_m(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const CUtensorMap& tmdO, const BwdParams& p, int grid, cudaStream_t st) {
    using C = KvCfg<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(jfa_bwd_dkdv_kernel<D, GDPA, DBIAS, DENSE, SHARED>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    jfa_bwd_dkdv_kernel<D, GDPA, DBIAS, DENSE, SHARED><<<grid, C::kThreads, C::kSmemBytes, st>>>(tmQ, tmK, tmV, tmdO, p);
    return cudaGetLastError();
}

template <int D, bool SHARED>
cudaError_t launch_dkdv_t_s(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const CUtensorMap& tmdO, const BwdParams& p, int grid, cudaStream_t st) {
    const bool sm = p.mode == JFA_SOFTMAX;
    if (p.dense)
        return sm ? launch_dkdv_t_m<D, false, false, true, SHARED>(tmQ, tmK, tmV, tmdO, p, grid, st)
                  : launch_dkdv_t_m<D, true, false, true, SHARED>(tmQ, tmK, tmV, tmdO, p, grid, st);
    if (p.dbias_part)
        return sm ? launch_dkdv_t_m<D, false, true, false, SHARED>(tmQ, tmK, tmV, tmdO, p, grid, st)
                  : launch_dkdv_t_m<D, true, true, false, SHARED>(tmQ, tmK, tmV, tmdO, p, grid, st);
    return sm ? launch_dkdv_t_m<D, false, false, false, SHARED>(tmQ, tmK, tmV, tmdO, p, grid, st)
              : launch_dkdv_t_m<D, true, false, false, SHARED>(tmQ, tmK, tmV, tmdO, p, grid, st);
}

template <int D>
cudaError_t launch_dkdv_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const CUtensorMap& tmdO, const BwdParams& p, int grid, cudaStream_t st) {
    return p.steps ? launch_dkdv_t_s<D, true>(tmQ, tmK, tmV, tmdO, p, grid, st)
                   : launch_dkdv_t_s<D, false>(tmQ, tmK, tmV, tmdO, p, grid, st);
}

template <typename TO, typename T, int D>
cudaError_t launch_pre_t(const void* O, const void* dO, float* delta, int64_t rows, cudaStream_t st) {
    const int64_t threads = rows * (D / 8);
    const int block = 256;
    const int64_t grid = (threads + block - 1) / block;
    jfa_bwd_pre_kernel<TO, T, D><<<unsigned(grid), block, 0, st>>>(static_cast<const TO*>(O),
                                                                   static_cast<const T*>(dO), delta, rows);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_pre(int dtype, int o_dtype, int D, const void* O, const void* dO, float* delta, float* dq_acc,
                           int64_t Tq, int H, int mode, cudaStream_t st) {
    using bf16 = __nv_bfloat16;
    const int64_t rows = Tq * H;
    if (dq_acc) {  // fp32 inputs: the dQ accumulator starts at zero
        cudaError_t e = cudaMemsetAsync(dq_acc, 0, size_t(rows) * size_t(D) * 4, st);
        if (e != cudaSuccess) return e;
    }
    if (mode != JFA_SOFTMAX) return cudaSuccess;
    const bool of = o_dtype == JFA_F32;
    if (dtype == JFA_BF16 && D == 128)
        return of ? launch_pre_t<float, bf16, 128>(O, dO, delta, rows, st)
                  : launch_pre_t<bf16, bf16, 128>(O, dO, delta, rows, st);
    if (dtype == JFA_BF16 && D == 64)
        return of ? launch_pre_t<float, bf16, 64>(O, dO, delta, rows, st)
                  : launch_pre_t<bf16, bf16, 64>(O, dO, delta, rows, st);
    if (dtype == JFA_F32 && D == 32 && of) return launch_pre_t<float, float, 32>(O, dO, delta, rows, st);
    if (dtype == JFA_F32 && D == 64 && of) return launch_pre_t<float, float, 64>(O, dO, delta, rows, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_main(int dtype, int D, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const CUtensorMap& tmdO, const BwdParams& p, int grid, cudaStream_t st) {
    if (dtype == JFA_BF16 && D == 128) return launch_dkdv_t<128>(tmQ, tmK, tmV, tmdO, p, grid, st);
    if (dtype == JFA_BF16 && D == 64) return launch_dkdv_t<64>(tmQ, tmK, tmV, tmdO, p, grid, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_dbias_reduce(const float* part, int64_t n_slots, int H, float* dbias, cudaStream_t st) {
    const int n = H * 32;
    jfa_dbias_reduce_kernel<<<(n + 255) / 256, 256, 0, st>>>(part, n_slots, H, dbias);
    return cudaGetLastError();
}

cudaError_t launch_dbias_reduce_items(const float* part, const int4* items, int64_t n_items, int H, float* dbias,
                                      cudaStream_t st) {
    const int n = H * 32;
    jfa_dbias_reduce_items_kernel<<<(n + 255) / 256, 256, 0, st>>>(part, items, n_items, H, dbias);
    return cudaGetLastError();
}

cudaError_t launch_bwd_post(int dtype, int D, const float* dq_acc, void* dQ, int64_t Tq, int H, float scale,
                            cudaStream_t st) {
    const int64_t n4 = Tq * H * D / 4;
    if (n4 == 0) return cudaSuccess;
    const int block = 256;
    const int64_t grid = std::min<int64_t>((n4 + block - 1) / block, 152 * 16);
    if (dtype == JFA_BF16)
        jfa_bwd_post_kernel<__nv_bfloat16><<<unsigned(grid), block, 0, st>>>(
            reinterpret_cast<const float4*>(dq_acc), static_cast<__nv_bfloat16*>(dQ), n4, scale);
    else
        jfa_bwd_post_kernel<float><<<unsigned(grid), block, 0, st>>>(reinterpret_cast<const float4*>(dq_acc),
                                                                     static_cast<float*>(dQ), n4, scale);
    return cudaGetLastError();
}

}  // namespace jfa
