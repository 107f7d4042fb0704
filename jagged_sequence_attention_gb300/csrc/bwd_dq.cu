// dQ pass of the bf16 backward: jagged flash attention / GDPA on sm_103a.
//
// Persistent over (sequence, head, 128-row query tile) with the forward's key-tile
// schedule (all key tiles, or up to the causal diagonal under the subtraction
// scheme the kerneldigest.dev summary names, section "Arquitectura del Sistema").
// For each key tile K_j, V_j:
//   S  = Q K_j^T     (TMEM, lanes = query rows; double-buffered)
//   dP = dO V_j^T    (TMEM)
//   dS = P (dP - Delta), P = exp2(S - lse)  (softmax)  or  act'(S) dP  (GDPA),
//        written back over S as bf16
//   dQ += dS K_j     (TMEM accumulator, A operand read from TMEM)
// and dQ = scale * accumulator is written once per tile: no atomics, no fp32 buffer.
//
// CTA = 10 warps: 0-7 compute (warpgroup g owns key columns [64g, 64g+64) of a tile;
// thread = query row = TMEM lane) and write the dQ epilogue, 8 TMA producer, 9 MMA
// issuer.  TMEM: S/dS buffers [0,128) and [128,256), dP [256,384), dQ [384,512).
// Issue order per key tile: S(j+1), dQ(j), dP(j+1): the next scores are computed
// while dS(j) is formed, and dP(j+1) while dQ(j) accumulates.
#include "bwd_common.cuh"
#include "jfa_internal.h"
#include "ptx.cuh"
#include "tilemath.cuh"

namespace jfa {

namespace {

// Every start is the first position of its bucket or above: (1 + s)^2 >= 2^b, and s - 1 is
// below it (s^2 < 2^b); checked here when the library is built.
constexpr bool bucket_starts_hold() {
    for (int b = 0; b < 32; ++b) {
        const long long st = relpos_bucket_start(b);
        if ((1 + st) * (1 + st) < (1LL << b) || (st > 0 && st * st >= (1LL << b))) return false;
    }
    return true;
}
static_assert(bucket_starts_hold(), "relative-position bucket starts");

// relpos_bucket_start(b) for every bucket, looked up with a warp-uniform index
struct BucketStarts {
    int v[32];
    constexpr BucketStarts() : v() {
        for (int b = 0; b < 32; ++b) v[b] = relpos_bucket_start(b);
    }
};
__constant__ BucketStarts kBucketStart = BucketStarts();

template <int D>
struct QCfg {
    static constexpr int BM = kFwdBM;  // query rows (TMEM lanes)
    static constexpr int BN = kFwdBN;  // key rows per step
    static constexpr int kRowBytes = D * 2;
    static_assert(kRowBytes % 128 == 0 && kRowBytes <= 256, "head row must be 128 or 256 bytes");
    static constexpr int kCB = kRowBytes / 128;
    static constexpr int kBoxCols = 64;
    static constexpr int kQTile = BM * kRowBytes;
    static constexpr int kKVTile = BN * kRowBytes;
    static constexpr int kOffQ = 0;
    static constexpr int kOffDO = kQTile;
    // K is read by S(j) and, a compute phase later, by dQ(j): three stages let K(j+3)
    // load while S(j+1), dQ(j+1), dP(j+2) and S(j+2) run.  V is read by dP(j) only.
    static constexpr int kKStages = 3, kVStages = 2;
    static constexpr int kOffK = 2 * kQTile;                  // + stage * kKVTile
    static constexpr int kOffV = kOffK + kKStages * kKVTile;  // + stage * kKVTile
    static constexpr int kOffBar = kOffV + kVStages * kKVTile;
    static constexpr int kNumBars = 24;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kCompWarps = 8;
    static constexpr int kCols = BN / 2;  // key columns per compute thread
    // tmem slot + abort flag (16 B); per compute warp: the head's bias row
    static constexpr int kMiscBytes = 16 + kCompWarps * 32 * 4;
    static constexpr int kSmemNeed = kOffMisc + kMiscBytes + 1024;
    static_assert(kSmemNeed <= 227 * 1024, "shared memory budget");
    // At least 120 KB so that exactly one CTA fits on an SM: it allocates all 512 TMEM columns.
    static constexpr int kSmemBytes = kSmemNeed > 120 * 1024 ? kSmemNeed : 120 * 1024;
    static constexpr int kDSteps = D / 16;   // contraction over head_dim
    static constexpr int kKSteps = BN / 16;  // contraction over key rows
    // dQ issues its K-steps per (warpgroup, 32-column chunk): 2 x 2 x 2 steps
    static_assert(kKSteps == 8 && kCols == 64, "chunked dQ issue assumes 128-key tiles");
    static constexpr uint32_t kTmDP = 256, kTmDQ = 384;
    static constexpr uint32_t kIdescS = make_idesc(kFmtBF16, BM, BN, false, false);
    static constexpr uint32_t kIdescDQ = make_idesc(kFmtBF16, BM, D, false, true);
    static constexpr int kEpiCols = D / 2;  // dQ columns each warpgroup writes
    static constexpr int kProdWarp = kCompWarps, kMmaWarp = kCompWarps + 1, kThreads = (kCompWarps + 2) * 32;
};

enum {
    DQ_Q_FULL = 0,
    DQ_DO_FULL = 1,
    DQ_QDO_EMPTY = 2,
    DQ_K_FULL = 3,    // +stage (3)
    DQ_K_EMPTY = 6,   // +stage (3)
    DQ_V_FULL = 9,    // +stage (2)
    DQ_V_EMPTY = 11,  // +stage (2)
    DQ_S_FULL = 13,   // +buffer
    DQ_SB_FREE = 15,  // +buffer: the dQ product that read dS from the buffer is done
    DQ_DP_FULL = 17,
    DQ_DS_FULL = 18,  // +chunk: key columns [32k, 32k+32) of both warpgroups' dS are in TMEM
    DQ_ACC_FULL = 20,
    DQ_ACC_EMPTY = 21,
    DQ_DRAIN = 22,
};

// DENSE: the bias is the dense per-pair array p.dense, read per element.
template <int D, bool GDPA, bool DENSE>
__global__ void __launch_bounds__(320, 1)
    jfa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                      const BwdParams p) {
    using C = QCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::kOffQ, sDO = sbase + C::kOffDO, sK = sbase + C::kOffK, sV = sbase + C::kOffV;
    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * uint32_t(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    float* misc_f = reinterpret_cast<float*>(smem + C::kOffMisc + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(bar(DQ_Q_FULL), 1);
        mbar_init(bar(DQ_DO_FULL), 1);
        mbar_init(bar(DQ_QDO_EMPTY), 1);
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(bar(DQ_K_FULL + s), 1);
            mbar_init(bar(DQ_K_EMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(DQ_V_FULL + s), 1);
            mbar_init(bar(DQ_V_EMPTY + s), 1);
            mbar_init(bar(DQ_S_FULL + s), 1);
            mbar_init(bar(DQ_SB_FREE + s), 1);
        }
        mbar_init(bar(DQ_DP_FULL), 1);
        mbar_init(bar(DQ_DS_FULL), C::kCompWarps);
        mbar_init(bar(DQ_DS_FULL + 1), C::kCompWarps);
        mbar_init(bar(DQ_ACC_FULL), 1);
        mbar_init(bar(DQ_ACC_EMPTY), C::kCompWarps);
        mbar_init(bar(DQ_DRAIN), 1);
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
            uint32_t kv_it = 0, item_it = 0;
            uint32_t k_extra = 0;  // 1: the last step's K load went out but its V load did not
            bool ok = true;
            for (int it = it_begin; it < it_end && ok; ++it) {
                const int4 w = p.items[it];
                if (!dq_item_ok(w, p)) {  // not an item of this plan: skipped by every role
                    atomicOr(p.status, kStatusBounds);
                    continue;
                }
                const int n = w.w;
                if (n == 0) continue;
                const int b = w.x, h = w.y, tq = w.z;
                const int kb = p.kv_map ? p.kv_map[b] : b;  // key/value sequence (shared: the user)
                const int q0 = p.q_off[b], kv0 = p.kv_off[kb];
                int kf, nk;  // key tiles [kf, kf + n)
                key_tile_range(p.q_off[b + 1] - q0, p.kv_off[kb + 1] - kv0, tq, p.causal, p.window, kf, nk);
                if (!mbar_wait_bounded(bar(DQ_QDO_EMPTY), (item_it & 1) ^ 1, abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(DQ_Q_FULL), C::kQTile);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb)
                    tma_load_2d(sQ + cb * C::BM * 128, &tmQ, bar(DQ_Q_FULL), h * D + cb * C::kBoxCols, q0 + tq * C::BM);
                mbar_arrive_expect_tx(bar(DQ_DO_FULL), C::kQTile);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb)
                    tma_load_2d(sDO + cb * C::BM * 128, &tmdO, bar(DQ_DO_FULL), h * D + cb * C::kBoxCols,
                                q0 + tq * C::BM);
                ++item_it;
                for (int j = 0; j < n; ++j, ++kv_it) {
                    const uint32_t kst = kv_it % 3, kph = (kv_it / 3) & 1;
                    const uint32_t st = kv_it & 1, ph = (kv_it >> 1) & 1;
                    const int y = kv0 + (kf + j) * C::BN;
                    if (!mbar_wait_bounded(bar(DQ_K_EMPTY + kst), kph ^ 1, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(bar(DQ_K_FULL + kst), C::kKVTile);
#pragma unroll
                    for (int cb = 0; cb < C::kCB; ++cb)
                        tma_load_2d(sK + kst * C::kKVTile + cb * C::BN * 128, &tmK, bar(DQ_K_FULL + kst),
                                    h * D + cb * C::kBoxCols, y);
                    if (!mbar_wait_bounded(bar(DQ_V_EMPTY + st), ph ^ 1, abort_flag)) {
                        k_extra = 1;
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(DQ_V_FULL + st), C::kKVTile);
#pragma unroll
                    for (int cb = 0; cb < C::kCB; ++cb)
                        tma_load_2d(sV + st * C::kKVTile + cb * C::BN * 128, &tmV, bar(DQ_V_FULL + st),
                                    h * D + cb * C::kBoxCols, y);
                }
            }
            if (!ok) fail();
            // Drain: wait until every load this thread issued has landed.
            if (item_it > 0) {
                mbar_wait_bounded(bar(DQ_Q_FULL), (item_it - 1) & 1, nullptr);
                mbar_wait_bounded(bar(DQ_DO_FULL), (item_it - 1) & 1, nullptr);
            }
            drain_ring(bar(DQ_K_FULL), kv_it + k_extra, 3);
            drain_ring(bar(DQ_V_FULL), kv_it, 2);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the schedule, so descriptors and counters stay
        // warp-uniform; one elected lane (always lane 0) issues every MMA and commit.
        uint32_t kv_it = 0, item_it = 0;
        bool ok = true;
        const SDesc dQa = sdesc_sw128(sQ, 16, 1024), dOa = sdesc_sw128(sDO, 16, 1024);
        // Descriptors of every ring stage, selected by value (no indexed array, which
        // would live in local memory).
        const SDesc dKk0 = sdesc_sw128(sK, 16, 1024), dKk1 = sdesc_sw128(sK + C::kKVTile, 16, 1024),
                    dKk2 = sdesc_sw128(sK + 2 * C::kKVTile, 16, 1024);
        const SDesc dVk0 = sdesc_sw128(sV, 16, 1024), dVk1 = sdesc_sw128(sV + C::kKVTile, 16, 1024);
        const SDesc dKm0 = sdesc_sw128(sK, C::BN * 128, 1024), dKm1 = sdesc_sw128(sK + C::kKVTile, C::BN * 128, 1024),
                    dKm2 = sdesc_sw128(sK + 2 * C::kKVTile, C::BN * 128, 1024);
        auto koff = [](int s) -> uint32_t { return uint32_t(((s * 32) >> 7) * 128 * 128 + ((s * 32) & 127)); };
        // S(g) = Q K^T into buffer g&1, once the dQ product that read that buffer is done.
        auto issue_s = [&](uint32_t g) -> bool {
            const uint32_t sb = g & 1, ph = (g >> 1) & 1, kst = g % 3;
            if (!warp_wait(DQ_K_FULL + kst, (g / 3) & 1) || !warp_wait(DQ_SB_FREE + sb, ph ^ 1)) return false;
            tc_fence_after();
            const SDesc dk = kst == 0 ? dKk0 : kst == 1 ? dKk1 : dKk2;
            if (elect_one()) {
#pragma unroll
                for (int s = 0; s < C::kDSteps; ++s) mma_ss(tmem + sb * 128u, dQa, koff(s), dk, koff(s), C::kIdescS, s > 0);
                tc_commit(bar(DQ_S_FULL + sb));
            }
            __syncwarp();
            return true;
        };
        // dP(g) = dO V^T; the compute threads read dP(g-1) before signalling dS(g-1),
        // which the issuer waited for before getting here.
        auto issue_dp = [&](uint32_t g) -> bool {
            const uint32_t st = g & 1, ph = (g >> 1) & 1;
            if (!warp_wait(DQ_V_FULL + st, ph)) return false;
            tc_fence_after();
            const SDesc dv = st ? dVk1 : dVk0;
            if (elect_one()) {
#pragma unroll
                for (int s = 0; s < C::kDSteps; ++s) mma_ss(tmem + C::kTmDP, dOa, koff(s), dv, koff(s), C::kIdescS, s > 0);
                tc_commit(bar(DQ_DP_FULL));
                tc_commit(bar(DQ_V_EMPTY + st));
            }
            __syncwarp();
            return true;
        };
        // dQ += dS K with dS read from buffer g&1; the first product of an item waits
        // for the previous item's epilogue to have read the accumulator.
        auto issue_dq = [&](uint32_t g, bool first) -> bool {
            const uint32_t sb = g & 1, kst = g % 3;
            const SDesc dk = kst == 0 ? dKm0 : kst == 1 ? dKm1 : dKm2;
            // chunk c of warpgroup w covers key rows 64w + 32c .. + 31: K-steps 4w + 2c, +1
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (!warp_wait(DQ_DS_FULL + c, g & 1)) return false;
                if (c == 0 && first && !warp_wait(DQ_ACC_EMPTY, (item_it & 1) ^ 1)) return false;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int s = 4 * (i >> 1) + 2 * c + (i & 1);
                        mma_ts(tmem + C::kTmDQ, tmem + sb * 128u + packed_col(s), dk, s * 16 * 128, C::kIdescDQ,
                               (!first || c > 0 || i > 0));
                    }
                    if (c == 1) {
                        tc_commit(bar(DQ_SB_FREE + sb));
                        tc_commit(bar(DQ_K_EMPTY + kst));
                    }
                }
                __syncwarp();
            }
            return true;
        };
        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 wi = p.items[it];
            if (!dq_item_ok(wi, p)) continue;
            const int n = wi.w;
            if (n == 0) continue;
            if (!warp_wait(DQ_Q_FULL, item_it & 1) || !warp_wait(DQ_DO_FULL, item_it & 1)) { ok = false; break; }
            tc_fence_after();
            const uint32_t g0 = kv_it;
            if (!issue_s(g0) || !issue_dp(g0)) { ok = false; break; }
            for (int j = 0; j < n && ok; ++j) {
                const uint32_t g = g0 + uint32_t(j);
                if (j + 1 < n && !issue_s(g + 1)) { ok = false; break; }
                if (!issue_dq(g, j == 0)) { ok = false; break; }
                if (j + 1 < n && !issue_dp(g + 1)) { ok = false; break; }
            }
            if (!ok) break;
            if (elect_one()) {
                tc_commit(bar(DQ_ACC_FULL));
                tc_commit(bar(DQ_QDO_EMPTY));
            }
            __syncwarp();
            kv_it += uint32_t(n);
            ++item_it;
        }
        if (!ok) fail();
        if (elect_one()) tc_commit(bar(DQ_DRAIN));
        __syncwarp();
        mbar_wait_bounded(bar(DQ_DRAIN), 0, nullptr);
    } else {
        // ------------------------------------------------------------ dS, epilogue
        // Thread = query row t of the tile (TMEM lane); warpgroup wg owns key columns
        // [c0, c0+64) of every key tile.
        constexpr int NC = C::kCols;
        const int wg = warp >> 2;
        const int t = (warp & 3) * 32 + lane;
        const int c0 = wg * NC;
        const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
        float* bias_w = misc_f + warp * 32;
        constexpr bool softmax = !GDPA;  // the other mode's code is not compiled in
        const bool gelu = p.mode == JFA_GDPA_GELU_TANH;
        uint32_t kv_it = 0, item_it = 0;
        bool ok = true;
        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 w = p.items[it];
            if (!dq_item_ok(w, p)) continue;
            const int n = w.w, b = w.x, h = w.y, tq = w.z;
            const int q0 = p.q_off[b], q_len = p.q_off[b + 1] - q0;
            const int kb = p.kv_map ? p.kv_map[b] : b;
            const int kv_len = p.kv_off[kb + 1] - p.kv_off[kb];
            const int diag = kv_len - q_len;
            const int row = tq * C::BM + t;
            const bool row_valid = row < q_len;
            const size_t orow = (size_t(q0) + size_t(row_valid ? row : 0)) * size_t(p.H) + size_t(h);
            __nv_bfloat16* dq_row = reinterpret_cast<__nv_bfloat16*>(p.dQ) + orow * D + wg * C::kEpiCols;
            if (n == 0) {  // the tile sees no key: dQ is zero
                if (row_valid) zero_bf16_row(dq_row, C::kEpiCols);
                continue;
            }
            if (p.bias) {
                __syncwarp();
                bias_w[lane] = p.bias[h * 32 + lane] * (softmax ? 1.4426950408889634f : 1.0f);
                __syncwarp();
            }
            const float lse_row = (softmax && row_valid) ? p.lse[orow] * 1.4426950408889634f : 0.f;
            // dense bias of this row (read only inside its allowed columns)
            const float* drow = DENSE ? p.dense + size_t(h) * size_t(p.n_pairs) + size_t(p.pair_off[b]) +
                                            size_t(row_valid ? row : 0) * size_t(kv_len)
                                      : nullptr;
            const float del_row = (softmax && row_valid) ? p.delta[orow] : 0.f;
            const float xs = softmax ? p.scale_log2 : p.scale;
            int kf, nk;  // key tiles [kf, kf + n)
            key_tile_range(q_len, kv_len, tq, p.causal, p.window, kf, nk);
            for (int j = 0; j < n; ++j) {
                const uint32_t g = kv_it + uint32_t(j), sb = g & 1;
                const int col0 = (kf + j) * C::BN + c0;
                int lim = kv_len - col0;  // subtraction scheme: local columns >= lim are masked
                if (p.causal) lim = min(lim, row + diag + 1 - col0);
                if (!row_valid) lim = 0;
                // sliding window: local columns below lo are masked
                const int lo = p.window >= 0 ? row + diag - p.window - col0 : 0;
                const bool full = __all_sync(0xffffffffu, lim >= NC && lo <= 0);
                const int rb = row + diag - col0;  // relative position of local column 0
                // Lane k tests chunk k for the whole warp: over the warp's rows, chunk k
                // spans relative positions rb(lane 0) - 32k - 31 .. + 62.
                // A chunk that is not one bucket but exactly two (the warp's positions all >= 0,
                // its lowest one bucket below its highest) takes its bias per lane from a column
                // threshold: columns c <= rb - start(upper bucket) are in the upper bucket.
                bool cconst[2] = {true, true}, two[2] = {false, false};
                float cbias[2] = {0.f, 0.f}, clow[2] = {0.f, 0.f};
                int cstart[2] = {0, 0};
                if (p.bias) {
                    const int rb0 = __shfl_sync(0xffffffffu, rb, 0);
                    int bk = 0;
                    const int lo_k = rb0 - 32 * lane - 31;  // lane k < 2: chunk k's lowest position
                    const uint32_t cm = warp_const_chunks(lane < 2, lo_k, bk);
                    const uint32_t tm =
                        __ballot_sync(0xffffffffu, lane < 2 && lo_k >= 0 && relpos_bucket(lo_k) == bk - 1);
                    const float bv = bias_w[bk], bv_low = bias_w[bk > 0 ? bk - 1 : 0];
                    const int st = kBucketStart.v[lane < 2 ? bk : 0];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        cconst[k] = (cm >> k) & 1u;
                        two[k] = (tm >> k) & 1u;
                        cbias[k] = __shfl_sync(0xffffffffu, bv, k);
                        clow[k] = __shfl_sync(0xffffffffu, bv_low, k);
                        cstart[k] = __shfl_sync(0xffffffffu, st, k);
                    }
                }
                const uint32_t tS = tmem + lane_base + sb * 128u + uint32_t(c0);

                if (!warp_wait(DQ_S_FULL + sb, (g >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                float pv[NC];
                {
                    uint32_t (&ra)[32] = *reinterpret_cast<uint32_t(*)[32]>(pv);
                    uint32_t (&rb2)[32] = *reinterpret_cast<uint32_t(*)[32]>(pv + 32);
                    tmem_ld32(tS, ra);
                    tmem_ld32(tS + 32u, rb2);
                    tmem_ld_wait(ra);
                    tmem_ld_wait(rb2);
                }
                // softmax: pv = P = exp2(xs * s + bias - lse); GDPA: pv = act'(scale * s + bias)
                const bool fast = !DENSE && full && cconst[0] && cconst[1];
                if (softmax && DENSE) {
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        const float bv = (c >= lo && c < lim) ? __ldg(drow + col0 + c) : 0.f;
                        pv[c] = ex2_approx(fmaf(pv[c], xs, fmaf(bv, 1.4426950408889634f, -lse_row)));
                    }
                } else if (softmax && fast) {
                    // branch-free copy for steps with no masked column and warp-constant bias
                    const float2 xs2 = make_float2(xs, xs);
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const float2 add = make_float2(cbias[k] - lse_row, cbias[k] - lse_row);
#pragma unroll
                        for (int c = 32 * k; c < 32 * k + 32; c += 2) {
                            const float2 e = fma2(make_float2(pv[c], pv[c + 1]), xs2, add);
                            pv[c] = ex2_approx(e.x);
                            pv[c + 1] = ex2_approx(e.y);
                        }
                    }
                } else if (softmax) {
                    const float2 xs2 = make_float2(xs, xs);
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        if (cconst[k]) {
                            const float2 add = make_float2(cbias[k] - lse_row, cbias[k] - lse_row);
#pragma unroll
                            for (int c = 32 * k; c < 32 * k + 32; c += 2) {
                                const float2 e = fma2(make_float2(pv[c], pv[c + 1]), xs2, add);
                                pv[c] = ex2_approx(e.x);
                                pv[c + 1] = ex2_approx(e.y);
                            }
                        } else if (two[k]) {
                            const float ahi = cbias[k] - lse_row, alo = clow[k] - lse_row;
                            const int t = rb - cstart[k];  // columns c <= t: the upper bucket
#pragma unroll
                            for (int c = 32 * k; c < 32 * k + 32; c += 2) {
                                const float2 add = make_float2(c <= t ? ahi : alo, c + 1 <= t ? ahi : alo);
                                const float2 e = fma2(make_float2(pv[c], pv[c + 1]), xs2, add);
                                pv[c] = ex2_approx(e.x);
                                pv[c + 1] = ex2_approx(e.y);
                            }
                        } else {
#pragma unroll
                            for (int c = 32 * k; c < 32 * k + 32; ++c)
                                pv[c] = ex2_approx(fmaf(pv[c], xs, bias_w[relpos_bucket(rb - c)] - lse_row));
                        }
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
#pragma unroll
                        for (int c = 32 * k; c < 32 * k + 32; ++c) {
                            float a, da;
                            float bv;
                            if constexpr (DENSE)
                                bv = (c >= lo && c < lim) ? __ldg(drow + col0 + c) : 0.f;
                            else
                                bv = cconst[k] ? cbias[k] : bias_w[relpos_bucket(rb - c)];
                            gdpa_act_grad(gelu, fmaf(pv[c], xs, bv), a, da);
                            pv[c] = da;
                        }
                    }
                }
                if (!fast && !full) {
#pragma unroll
                    for (int c = 0; c < NC; ++c) pv[c] = (c >= lo && c < lim) ? pv[c] : 0.f;
                }

                if (!warp_wait(DQ_DP_FULL, g & 1)) { ok = false; break; }
                tc_fence_after();
                // dS = P (dP - Delta) (softmax) or act' dP (GDPA), 32 columns at a time,
                // packed over the warpgroup's own S columns (already read).
                const float2 nd = make_float2(-del_row, -del_row);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    float dp[32];
                    {
                        uint32_t (&ra)[32] = *reinterpret_cast<uint32_t(*)[32]>(dp);
                        tmem_ld32(tmem + lane_base + C::kTmDP + uint32_t(c0) + 32u * k, ra);
                        tmem_ld_wait(ra);
                    }
                    uint32_t pd[16];
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const float2 d2 = make_float2(dp[c], dp[c + 1]);
                        const float2 a = mul2(make_float2(pv[32 * k + c], pv[32 * k + c + 1]), softmax ? add2(d2, nd) : d2);
                        pd[c >> 1] = pack_bf16x2(a.x, a.y);
                    }
                    tmem_st16(tS + 16u * k, pd);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(DQ_DS_FULL + k));
                }
            }
            if (!ok) break;
            // Epilogue: dQ = scale * accumulator, the warpgroup's half of D.
            if (!warp_wait(DQ_ACC_FULL, item_it & 1)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < C::kEpiCols / 32; ++cc) {
                uint32_t rr[32];
                float v[32];
                tmem_ld32(tmem + lane_base + C::kTmDQ + uint32_t(wg * C::kEpiCols + 32 * cc), rr);
                tmem_ld_wait(rr);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(rr[e]);
                if (row_valid) store_bf16_row(dq_row + 32 * cc, v, 32, p.scale);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(DQ_ACC_EMPTY));
            kv_it += uint32_t(n);
            ++item_it;
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kMmaWarp) tmem_dealloc(tmem, 512);
}

template <int D, bool GDPA, bool DENSE>
cudaError_t launch_dq_t_m(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                        const CUtensorMap& tmdO, const BwdParams& p, int grid, cudaStream_t st) {
    using C = QCfg<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e =
            cudaFuncSetAttribute(jfa_bwd_dq_kernel<D, GDPA, DENSE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    jfa_bwd_dq_kernel<D, GDPA, DENSE><<<grid, C::kThreads, C::kSmemBytes, st>>>(tmQ, tmK, tmV, tmdO, p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_dq_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                        const CUtensorMap& tmdO, const BwdParams& p, int grid, cudaStream_t st) {
    if (p.dense)
        return p.mode == JFA_SOFTMAX ? launch_dq_t_m<D, false, true>(tmQ, tmK, tmV, tmdO, p, grid, st)
                                     : launch_dq_t_m<D, true, true>(tmQ, tmK, tmV, tmdO, p, grid, st);
    return p.mode == JFA_SOFTMAX ? launch_dq_t_m<D, false, false>(tmQ, tmK, tmV, tmdO, p, grid, st)
                                 : launch_dq_t_m<D, true, false>(tmQ, tmK, tmV, tmdO, p, grid, st);
}

}  // namespace

cudaError_t launch_bwd_dq(int dtype, int D, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const CUtensorMap& tmdO, const BwdParams& p, int grid, cudaStream_t st) {
    if (dtype == JFA_BF16 && D == 128) return launch_dq_t<128>(tmQ, tmK, tmV, tmdO, p, grid, st);
    if (dtype == JFA_BF16 && D == 64) return launch_dq_t<64>(tmQ, tmK, tmV, tmdO, p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace jfa
