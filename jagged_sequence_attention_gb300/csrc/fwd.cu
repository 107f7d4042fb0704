// Forward kernel: jagged flash attention / GDPA on sm_103a.
//
// Computes, per (sequence, head, pair of 128-row query tiles) work item, the
// attention of the GEM articles' "Jagged Sequence Flash Attention" (aihot.vn, that
// section): directly on packed values plus offsets, never materialising a padded
// tensor.  Masking follows the "subtraction scheme" the kerneldigest.dev summary
// names (section "Arquitectura del Sistema"): for a key tile starting at column c0
// the kernel subtracts c0 from the sequence's key length (and from the row's causal
// limit) and masks columns at or beyond what remains -- no mask tensor, no padding.
// The GDPA mode (aihot.vn, "Generalized Dot-Product Attention (GDPA)") swaps the
// online softmax for an elementwise GELU/SiLU with no normalisation.
//
// CTA = 18 warps, persistent, one CTA per SM, work list from the planner.  Two query
// tiles (A: rows 256p..256p+127, B: the next 128) share every K/V tile, so each K/V
// byte loaded feeds two products, and the two tiles' softmax warps ping-pong around the
// tensor core.  Two warps share each row (thread = row = TMEM lane): one takes score
// columns [0, 64) and O columns [0, D/2), the other the rest, so a tile's softmax runs
// on two warps per scheduler; they exchange row maxima and sums through shared memory.
//   warps 0-3   tile A, columns [0, 64): softmax/activation, correction, epilogue
//   warps 4-7   tile B, columns [0, 64)
//   warps 8-11  tile A, columns [64, 128)
//   warps 12-15 tile B, columns [64, 128)
//   warp 16     TMA producer: Q_A, Q_B once per item; K_j, V_j through 2-stage rings
//   warp 17     tcgen05.mma issuer and TMEM owner
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256,256+D), O_B [384,384+D).
// P is written back over its own S columns as packed bf16 (64 columns; GDPA adds the
// rounding remainder in the next 64) and read by O += P V straight from TMEM.  The
// MMA issue order S_A(j) S_B(j) PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) ... keeps the
// tensor core on one tile while the other tile's softmax runs.
#include "jfa_internal.h"
#include "ptx.cuh"
#include "tilemath.cuh"

namespace jfa {

template <int D>
struct FwdCfg {
    static constexpr int BM = kFwdBM, BN = kFwdBN;
    static constexpr int kRowBytes = D * 2;
    static_assert(kRowBytes % 128 == 0 && kRowBytes <= 256, "head row must be 128 or 256 bytes");
    static constexpr int kCB = kRowBytes / 128;  // 128-byte column blocks of a tile
    static constexpr int kBoxCols = 64;          // bf16 elements per 128-byte box row
    static constexpr int kQBytes = BM * kRowBytes;
    static constexpr int kKVBytes = BN * kRowBytes;
    static constexpr int kStages = 2;
    static constexpr int kOffQ = 0;  // + tile * kQBytes
    static constexpr int kOffK = kOffQ + 2 * kQBytes;
    static constexpr int kOffV = kOffK + kStages * kKVBytes;
    static constexpr int kOffBar = kOffV + kStages * kKVBytes;
    static constexpr int kNumBars = 32;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    // softmax warps: 2 tiles x 2 column halves x 4 row quarters
    static constexpr int kSoftWarps = 16;
    // tmem slot + abort flag; per softmax warp: the head's bias row (32) and a tile's
    // bias-by-relative-position table (160), with a copy shifted by one entry (so that every
    // lane reads its column pairs as aligned 8-byte loads)
    static constexpr int kBiasRow = 32, kBiasTab = 160;
    static constexpr int kWarpBias = kBiasRow + 2 * kBiasTab;
    // ... for split items, tile 1's row max and two partial sums (two buffers of 3 x BM
    // floats), and the pair exchanges (two buffers of 2 halves x 8 pairs x 32 floats)
    static constexpr int kMiscBytes = 16 + kSoftWarps * kWarpBias * 4 + 2 * 3 * BM * 4 + 2 * 2 * 8 * 32 * 4;
    static constexpr int kSmemNeed = kOffMisc + kMiscBytes + 1024;
    // At least 120 KB so that exactly one CTA fits on an SM: the CTA allocates all
    // 512 TMEM columns.
    static constexpr int kSmemBytes = kSmemNeed > 120 * 1024 ? kSmemNeed : 120 * 1024;
    static constexpr int kUmmaK = 16;
    static constexpr int kQKSteps = D / kUmmaK;
    static constexpr int kPVSteps = BN / kUmmaK;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kIdescQK = make_idesc(kFmtBF16, BM, BN, false, false);
    static constexpr uint32_t kIdescPV = make_idesc(kFmtBF16, BM, D, false, true);
    static constexpr int kThreads = (kSoftWarps + 2) * 32;
    static constexpr int kProdWarp = kSoftWarps, kMmaWarp = kSoftWarps + 1;
    __host__ __device__ static constexpr uint32_t tmem_s(int x) { return x ? 128u : 0u; }
    __host__ __device__ static constexpr uint32_t tmem_o(int x) { return x ? 384u : 256u; }
};

// TMEM column (within a tile's S/P columns) of the 16 P values of PV K-step s: P of
// S chunk k (32 columns) occupies the chunk's first 16 columns, two bf16 per column,
// and the GDPA rounding remainder the next 16.
__device__ __forceinline__ uint32_t p_col(int s) { return uint32_t(32 * (s >> 1) + 8 * (s & 1)); }

// Barrier slots.
enum {
    B_Q_FULL = 0,
    B_Q_EMPTY = 1,
    B_K_FULL = 2,   // +stage
    B_K_EMPTY = 4,  // +stage
    B_V_FULL = 6,
    B_V_EMPTY = 8,
    B_S_FULL = 10,   // +tile
    B_P_FULL = 12,   // +tile
    B_O_DONE = 14,   // +tile: a P V product of the tile finished
    B_O_EMPTY = 16,  // +tile: the tile's epilogue has read O
    B_DRAIN = 18,
    B_COMBINE = 19,  // split item: tile 1's last P V done and its row max/sums written
    B_XCH = 20,      // +pair: the two warps of a row group have written their exchange values
    B_NEVER = 28,    // nothing arrives here (the timeout test's stall, test builds only)
};

template <typename T>
__device__ __forceinline__ void store_row(T* dst, const float* v, int n);

template <>
__device__ __forceinline__ void store_row<__nv_bfloat16>(__nv_bfloat16* dst, const float* v, int n) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (int i = 0; i < n / 8; ++i) {
        uint4 u;
        u.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
        u.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
        u.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
        u.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
        d4[i] = u;
    }
}

template <>
__device__ __forceinline__ void store_row<float>(float* dst, const float* v, int n) {
    float4* d4 = reinterpret_cast<float4*>(dst);
    for (int i = 0; i < n / 4; ++i) d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

// WIN: a sliding window may be set (p.window >= 0).  Without it the window arithmetic
// folds away at compile time, so the plain causal and non-causal paths carry none of it.
// DENSE: the bias is the dense per-pair array p.dense (read per element, both passes).
// SPLIT: the work list holds split items (fwd_split_item, see below); without it the
// split code compiles away and the kernel is the plain two-tile pipeline.
template <int D, typename OT, bool GDPA, bool WIN, bool DENSE, bool SPLIT>
__global__ void __launch_bounds__(576, 1)
    jfa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::kOffQ, sK = sbase + C::kOffK, sV = sbase + C::kOffV;
    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * uint32_t(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    float* bias_s = reinterpret_cast<float*>(smem + C::kOffMisc + 16);
    constexpr bool gdpa = GDPA;
    const int window = WIN ? p.window : -1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q_FULL), 1);
        mbar_init(bar(B_Q_EMPTY), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_K_FULL + s), 1);
            mbar_init(bar(B_K_EMPTY + s), 1);
            mbar_init(bar(B_V_FULL + s), 1);
            mbar_init(bar(B_V_EMPTY + s), 1);
            mbar_init(bar(B_S_FULL + s), 1);
            mbar_init(bar(B_P_FULL + s), 8);
            mbar_init(bar(B_O_DONE + s), 1);
            mbar_init(bar(B_O_EMPTY + s), 8);
        }
        mbar_init(bar(B_DRAIN), 1);
        mbar_init(bar(B_COMBINE), 8);
        for (int q = 0; q < 8; ++q) mbar_init(bar(B_XCH + q), 2);
        mbar_init(bar(B_NEVER), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == C::kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
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

    if (warp == C::kProdWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t kv_it = 0, item_it = 0;
            uint32_t k_extra = 0;  // 1: the last step's K load went out but its V load did not
            bool ok = true;
            for (int it = it_begin; it < it_end && ok; ++it) {
                const int4 w = p.items[it];
                if (!fwd_item_ok(w, p, window)) {  // not an item of this plan: skipped by every role
                    atomicOr(p.status, kStatusBounds);
                    continue;
                }
                const int n = w.w;
                if (n == 0) continue;
                const int b = w.x, h = w.y, pr = w.z;
                const int kb = p.kv_map ? p.kv_map[b] : b;  // key/value sequence (shared: the user)
                const int q0 = p.q_off[b], q_len = p.q_off[b + 1] - q0, kv0 = p.kv_off[kb];
                const int kv_len = p.kv_off[kb + 1] - kv0;
                const int ntiles = (2 * pr + 1) * C::BM < q_len ? 2 : 1;
                int f0, ns, na, nb;  // the pair streams key tiles [f0, f0 + n)
                pair_stream(q_len, kv_len, pr, p.causal, window, f0, ns, na, nb);
                if (!mbar_wait_bounded(bar(B_Q_EMPTY), (item_it & 1) ^ 1, abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(B_Q_FULL), C::kQBytes * ntiles);
                for (int tq = 0; tq < ntiles; ++tq)
#pragma unroll
                    for (int cb = 0; cb < C::kCB; ++cb)
                        tma_load_2d(sQ + tq * C::kQBytes + cb * C::BM * 128, &tmQ, bar(B_Q_FULL),
                                    h * D + cb * C::kBoxCols, q0 + (2 * pr + tq) * C::BM);
                ++item_it;
                // A split item (fwd_split_item) streams the two halves of its key range
                // interleaved: tile 0's half at even steps, tile 1's at odd.
                const bool split = SPLIT && fwd_split_item(q_len, pr, na);
                const int half0 = (na + 1) / 2;
                for (int j = 0; j < n; ++j, ++kv_it) {
                    const uint32_t st = kv_it & 1, ph = (kv_it >> 1) & 1;
                    const int kt = split ? ((j & 1) ? half0 + (j >> 1) : (j >> 1)) : j;
                    const int y = kv0 + (f0 + kt) * C::BN;
                    if (!mbar_wait_bounded(bar(B_K_EMPTY + st), ph ^ 1, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(bar(B_K_FULL + st), C::kKVBytes);
#pragma unroll
                    for (int cb = 0; cb < C::kCB; ++cb)
                        tma_load_2d(sK + st * C::kKVBytes + cb * C::BN * 128, &tmK, bar(B_K_FULL + st),
                                    h * D + cb * C::kBoxCols, y);
                    if (!mbar_wait_bounded(bar(B_V_EMPTY + st), ph ^ 1, abort_flag)) {
                        k_extra = 1;
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(B_V_FULL + st), C::kKVBytes);
#pragma unroll
                    for (int cb = 0; cb < C::kCB; ++cb)
                        tma_load_2d(sV + st * C::kKVBytes + cb * C::BN * 128, &tmV, bar(B_V_FULL + st),
                                    h * D + cb * C::kBoxCols, y);
                }
            }
            if (!ok) fail();
            // Drain: wait until every load this thread issued has landed.
            if (item_it > 0) mbar_wait_bounded(bar(B_Q_FULL), (item_it - 1) & 1, nullptr);
            drain_ring(bar(B_K_FULL), kv_it + k_extra, 2);
            drain_ring(bar(B_V_FULL), kv_it, 2);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the schedule, so descriptors and counters stay
        // warp-uniform; one elected lane (always lane 0) issues every MMA and commit.
        auto wwait = [&](int b, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait_bounded(bar(b), parity, abort_flag));
        };
        uint32_t kv_it = 0, item_it = 0;
        uint32_t pv_cnt0 = 0, pv_cnt1 = 0, items_x0 = 0, items_x1 = 0;
        bool ok = true;
#ifdef JFA_TEST_STALL_MMA
        // Test builds only (the bounded-wait test): before its first product the issuer waits
        // on a barrier that nothing arrives on, so that this pipeline wait runs out and every
        // role of the CTA winds down and reports the timeout.
        if (it_begin < it_end && !wwait(B_NEVER, 0)) ok = false;
#endif
        // Descriptors of every operand tile, built once; each MMA below adds a
        // compile-time byte offset to the low half.
        const SDesc dQ0 = sdesc_sw128(sQ, 16, 1024), dQ1 = sdesc_sw128(sQ + C::kQBytes, 16, 1024);
        const SDesc dK0 = sdesc_sw128(sK, 16, 1024), dK1 = sdesc_sw128(sK + C::kKVBytes, 16, 1024);
        const SDesc dV0 = sdesc_sw128(sV, C::BN * 128, 1024), dV1 = sdesc_sw128(sV + C::kKVBytes, C::BN * 128, 1024);
        // S_x = Q_x K^T into the tile's S columns; first waits for the tile's
        // previous P V product, which reads P from those columns.
        // qx: the query tile the product reads (tile x's own, or tile 0 in a split item)
        auto issue_s = [&](int x, uint32_t st, int qx) -> bool {
            const uint32_t pc = x ? pv_cnt1 : pv_cnt0;
            if (pc > 0 && !wwait(B_O_DONE + x, (pc - 1) & 1)) return false;
            tc_fence_after();
            const SDesc dq = qx ? dQ1 : dQ0, dk = st ? dK1 : dK0;
            const uint32_t d_tmem = tmem + C::tmem_s(x);
            if (elect_one()) {
#pragma unroll
                for (int s = 0; s < C::kQKSteps; ++s) {
                    // K step s: 128-byte column block (s*32)>>7, (s*32)&127 bytes into the row
                    mma_ss(d_tmem, dq, ((s * 32) >> 7) * C::BM * 128 + ((s * 32) & 127), dk,
                           ((s * 32) >> 7) * C::BN * 128 + ((s * 32) & 127), C::kIdescQK, s > 0);
                }
                tc_commit(bar(B_S_FULL + x));
            }
            __syncwarp();
            return true;
        };
        // O_x += P_x V with P read from TMEM; GDPA adds the remainder product.
        auto issue_pv = [&](int x, uint32_t st, bool first) -> bool {
            const uint32_t pc = x ? pv_cnt1 : pv_cnt0, ix = x ? items_x1 : items_x0;
            if (!wwait(B_P_FULL + x, pc & 1)) return false;
            if (first && !wwait(B_O_EMPTY + x, (ix & 1) ^ 1)) return false;
            tc_fence_after();
            const SDesc dv = st ? dV1 : dV0;
            const uint32_t d_tmem = tmem + C::tmem_o(x), a_tmem = tmem + C::tmem_s(x);
            if (elect_one()) {
#pragma unroll
                for (int s = 0; s < C::kPVSteps; ++s)
                    mma_ts(d_tmem, a_tmem + p_col(s), dv, s * C::kUmmaK * 128, C::kIdescPV, (!first || s > 0));
                if (gdpa) {
#pragma unroll
                    for (int s = 0; s < C::kPVSteps; ++s)
                        mma_ts(d_tmem, a_tmem + p_col(s) + 16u, dv, s * C::kUmmaK * 128, C::kIdescPV, 1u);
                }
                tc_commit(bar(B_O_DONE + x));
            }
            __syncwarp();
            if (x) ++pv_cnt1; else ++pv_cnt0;
            return true;
        };
        auto commit = [&](int b) {
            if (elect_one()) tc_commit(bar(b));
            __syncwarp();
        };
        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 w = p.items[it];
            if (!fwd_item_ok(w, p, window)) continue;
            const int n = w.w;
            if (n == 0) continue;
            const int b = w.x, pr = w.z;
            const int kb = p.kv_map ? p.kv_map[b] : b;
            const int q_len = p.q_off[b + 1] - p.q_off[b], kv_len = p.kv_off[kb + 1] - p.kv_off[kb];
            // Each tile's key range inside the pair's stream [f0, f0 + n): tile x is active
            // for stream steps [off_x, off_x + nx_x).
            int fa, nx0, fb, nx1, f0, ns, na2, nb2;
            key_tile_range(q_len, kv_len, 2 * pr, p.causal, window, fa, nx0);
            key_tile_range(q_len, kv_len, 2 * pr + 1, p.causal, window, fb, nx1);
            pair_stream(q_len, kv_len, pr, p.causal, window, f0, ns, na2, nb2);
            const int off0 = fa - f0, off1 = fb - f0;
            // A split item (fwd_split_item: a pair holding one query tile with two or more key
            // tiles; a longer sequence's odd last tile only with a long key range): both tiles'
            // products read query tile 0; tile 0 takes the even stream steps, tile 1 the odd.
            const bool split = SPLIT && fwd_split_item(q_len, pr, nx0);
            if (!wwait(B_Q_FULL, item_it & 1)) { ok = false; break; }
            if (!split) {
                auto act0 = [&](int j) { return j >= off0 && j < off0 + nx0; };
                auto act1 = [&](int j) { return j >= off1 && j < off1 + nx1; };
                // prologue: S of key tile 0
                {
                    const uint32_t st = kv_it & 1, ph = (kv_it >> 1) & 1;
                    if (!wwait(B_K_FULL + st, ph)) { ok = false; break; }
                    if (act0(0) && !issue_s(0, st, 0)) { ok = false; break; }
                    if (act1(0) && !issue_s(1, st, 1)) { ok = false; break; }
                    commit(B_K_EMPTY + st);
                    if (n == 1) commit(B_Q_EMPTY);
                }
                for (int j = 0; j < n && ok; ++j) {
                    const uint32_t g = kv_it + j, st = g & 1, ph = (g >> 1) & 1;
                    const uint32_t g1 = g + 1, st1 = g1 & 1, ph1 = (g1 >> 1) & 1;
                    if (!wwait(B_V_FULL + st, ph)) { ok = false; break; }
                    if (act0(j) && !issue_pv(0, st, j == off0)) { ok = false; break; }
                    if (j + 1 < n && !wwait(B_K_FULL + st1, ph1)) { ok = false; break; }
                    if (act0(j + 1) && !issue_s(0, st1, 0)) { ok = false; break; }
                    if (act1(j) && !issue_pv(1, st, j == off1)) { ok = false; break; }
                    commit(B_V_EMPTY + st);
                    if (act1(j + 1) && !issue_s(1, st1, 1)) { ok = false; break; }
                    if (j + 1 < n) {
                        commit(B_K_EMPTY + st1);
                        if (j + 2 == n) commit(B_Q_EMPTY);
                    }
                }
            } else {
                // step j: tile x = j & 1 computes P V of stream step j, then S of step j + 2
                // (S of steps 0 and 1 in the prologue); every S reads query tile 0.  The
                // producer streams tile 0's half of the key range at even steps, tile 1's at odd.
                {
                    const uint32_t st = kv_it & 1, ph = (kv_it >> 1) & 1;
                    if (!wwait(B_K_FULL + st, ph)) { ok = false; break; }
                    if (!issue_s(0, st, 0)) { ok = false; break; }
                    commit(B_K_EMPTY + st);
                    const uint32_t g1 = kv_it + 1, st1 = g1 & 1, ph1 = (g1 >> 1) & 1;
                    if (!wwait(B_K_FULL + st1, ph1)) { ok = false; break; }
                    if (!issue_s(1, st1, 0)) { ok = false; break; }
                    commit(B_K_EMPTY + st1);
                    if (n == 2) commit(B_Q_EMPTY);
                }
                for (int j = 0; j < n && ok; ++j) {
                    const int x = j & 1;
                    const uint32_t g = kv_it + j, st = g & 1, ph = (g >> 1) & 1;
                    const uint32_t g2 = g + 2, st2 = g2 & 1, ph2 = (g2 >> 1) & 1;
                    if (!wwait(B_V_FULL + st, ph)) { ok = false; break; }
                    if (!issue_pv(x, st, j < 2)) { ok = false; break; }
                    commit(B_V_EMPTY + st);
                    if (j + 2 < n) {
                        if (!wwait(B_K_FULL + st2, ph2)) { ok = false; break; }
                        if (!issue_s(x, st2, 0)) { ok = false; break; }
                        commit(B_K_EMPTY + st2);
                        if (j + 3 == n) commit(B_Q_EMPTY);
                    }
                }
            }
            kv_it += n;
            ++item_it;
            items_x0 += nx0 > 0 ? 1 : 0;
            items_x1 += (nx1 > 0 || split) ? 1 : 0;
        }
        if (!ok) fail();
        // Drain all issued MMAs before TMEM is released.
        commit(B_DRAIN);
        mbar_wait_bounded(bar(B_DRAIN), 0, nullptr);
    } else {
        // ------------------------------------------------------------ softmax / epilogue
        // Two warps share each 32-row group of a tile: the warp with hf = 0 takes score
        // columns [0, 64) and O columns [0, D/2), the one with hf = 1 the rest.  They
        // exchange their partial row max (softmax) each step and their partial row sums at
        // the end through shared memory, behind a bounded wait on their pair's barrier.
        const int x = (warp >> 2) & 1;         // query tile of this warp
        const int hf = warp >> 3;              // column half
        const int pair = warp & 7;             // the two warps holding these rows
        const int t = (warp & 3) * 32 + lane;  // row in the tile == TMEM lane
        constexpr int HC = C::BN / 2;          // score columns per thread
        constexpr int OC = D / 2;              // O columns per thread
        const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
        const uint32_t tSt = tmem + lane_base + C::tmem_s(x);  // the tile's S columns
        const uint32_t tS = tSt + uint32_t(HC * hf);           // this warp's half
        const uint32_t tO = tmem + lane_base + C::tmem_o(x) + uint32_t(OC * hf);
        constexpr bool softmax = !GDPA;
        uint32_t s_cnt = 0;
        uint32_t split_cnt = 0;  // split items seen (phase of B_COMBINE, exchange buffer)
        uint32_t x_cnt = 0;      // exchanges with the partner warp (phase of its barrier)
        float* comb_s = bias_s + C::kSoftWarps * C::kWarpBias;  // [2][m, l0, l1][BM]
        float* xch_s = comb_s + 2 * 3 * C::BM;                                  // [2][2][8][32]
        // The partner warp's value of a per-row float this warp also passes in.
        auto exchange = [&](float v, float& other) -> bool {
            float* buf = xch_s + (x_cnt & 1) * 512 + pair * 32;
            buf[hf * 256 + lane] = v;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_XCH + pair));
            // The partner is normally a few hundred cycles away at most: spin inline (a call
            // to the parked slow-path wait would save this warp's live scores around it),
            // bounded by an iteration count and the CTA's abort flag.
            bool done = false;
            for (uint32_t spin = 0; spin < (1u << 26) && !done; ++spin) {
                done = mbar_try_wait(bar(B_XCH + pair), x_cnt & 1);
                if (!done && (spin & 1023u) == 1023u && *abort_flag) break;
            }
            const bool ok = __all_sync(0xffffffffu, done);
            ++x_cnt;
            if (ok) other = buf[(hf ^ 1) * 256 + lane];
            return ok;
        };
        bool ok = true;
        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 w = p.items[it];
            if (!fwd_item_ok(w, p, window)) continue;
            const int b = w.x, h = w.y, pr = w.z;
            const int q0 = p.q_off[b], q_len = p.q_off[b + 1] - q0;
            const int kb = p.kv_map ? p.kv_map[b] : b;
            const int kv_len = p.kv_off[kb + 1] - p.kv_off[kb];
            // Split item (fwd_split_item): both tiles'
            // warps take tile 0's rows, tile x one half of its key range (the first
            // (na + 1) / 2 key tiles, or the rest) with its own max, sum and O; tile 0's
            // warps combine the two at the end.  The tile loop is the same in both cases.
            int kfa, na;
            key_tile_range(q_len, kv_len, 2 * pr, p.causal, window, kfa, na);
            const bool split = SPLIT && fwd_split_item(q_len, pr, na);
            const int tile = split ? 2 * pr : 2 * pr + x;
            if (tile * C::BM >= q_len) continue;  // tile B of a short last pair
            int kf, n;  // this tile's key tiles [kf, kf + n)
            if (split) {
                kf = kfa + (x ? (na + 1) / 2 : 0);
                n = x ? na / 2 : (na + 1) / 2;
            } else {
                key_tile_range(q_len, kv_len, tile, p.causal, window, kf, n);
            }
            const int row = tile * C::BM + t;
            const bool row_valid = row < q_len;
            const int diag = kv_len - q_len;
            // dense bias of this row (row-major [q_len, kv_len] block of head h, sequence b)
            const float* drow = nullptr;
            if constexpr (DENSE)
                drow = p.dense + size_t(h) * size_t(p.n_pairs) + size_t(p.pair_off[b]) +
                       size_t(row_valid ? row : 0) * size_t(kv_len);
            // Each warp keeps its own copy of the head's bias row (log2 units for
            // softmax) and its maximum, so no cross-warp barrier is needed.
            float* btab = bias_s + warp * C::kWarpBias;
            float* rtab = btab + C::kBiasRow;
            float bmax = 0.f;
            if (p.bias) {
                __syncwarp();
                const float bv = p.bias[h * 32 + lane] * (softmax ? 1.4426950408889634f : 1.0f);
                btab[lane] = bv;
                bmax = bv;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
                __syncwarp();
            }
            const size_t orow = (size_t(q0) + size_t(row)) * size_t(p.H) + size_t(h);
            if (n == 0) {
                if (row_valid) {
                    float z[32];
#pragma unroll
                    for (int d = 0; d < 32; ++d) z[d] = 0.f;
                    for (int c = 0; c < OC / 32; ++c)
                        store_row<OT>(reinterpret_cast<OT*>(p.O) + orow * D + OC * hf + c * 32, z, 32);
                    if (p.lse && hf == 0) p.lse[orow] = -INFINITY;
                }
                continue;
            }
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < n; ++j) {
                // The step's masks and bias lookups depend on its position only, so they are
                // formed while the tensor core computes its scores.
                const int col0 = (kf + j) * C::BN;
                int lim = kv_len - col0;  // subtraction scheme: columns >= lim are masked
                if (p.causal) lim = min(lim, row + diag + 1 - col0);
                if (DENSE && !row_valid) lim = 0;  // never read a dense bias past the sequence
                // sliding window: columns below row + diag - W are masked
                const int lo = (WIN && (!DENSE || window >= 0)) ? row + diag - window - col0 : 0;
                const int rbase = row + diag - col0;  // relative position of column 0
                const bool full = __all_sync(0xffffffffu, lim >= C::BN && lo <= 0);
                const float xs = softmax ? p.scale_log2 : p.scale;
                // Bias per 32-column chunk: a constant when every lane's chunk sits in
                // one bucket (warp-uniform flag per chunk); otherwise read per element
                // from a table of the bias by relative position built for this tile.
                // Lane k tests chunk k for the whole warp: over the warp's rows, chunk k
                // spans relative positions rbase(lane 0) - 32k - 31 .. + 62.
                uint32_t hmask = 3u;  // bit k: this warp's chunk k (tile chunk 2 hf + k) has a constant bias
                float cb[2] = {0.f, 0.f};
                if (p.bias) {
                    const int rb0 = __shfl_sync(0xffffffffu, rbase, 0);
                    int bk = 0;
                    const int kl = 2 * hf + (lane & 1);  // lanes 0, 1 test this warp's chunks
                    hmask = warp_const_chunks(lane < 2, rb0 - 32 * kl - 31, bk) & 3u;
                    const float bv = btab[bk];
#pragma unroll
                    for (int k = 0; k < 2; ++k) cb[k] = __shfl_sync(0xffffffffu, bv, k);
                }
                if (hmask != 3u) {
                    // rtab[i] = bias(r) for r = (lane 0's rbase) - 127 + i, i in [0, 160): element
                    // (lane, c) is rtab[lane + 127 - c]; and rtab[160 + i] = rtab[i + 1].
                    const int r0 = __shfl_sync(0xffffffffu, rbase, 0) - (C::BN - 1);
                    __syncwarp();
#pragma unroll
                    for (int m2 = 0; m2 < C::kBiasTab / 32; ++m2) {
                        const int i = lane + 32 * m2;
                        const float v = btab[relpos_bucket(r0 + i)];
                        rtab[i] = v;
                        if (i > 0) rtab[C::kBiasTab + i - 1] = v;
                    }
                    __syncwarp();
                }
                // Columns (c, c + 1), c even, as one aligned float2 (bias of c + 1, bias of c) at
                // rpair - c: even lanes read the table at lane + 126 - c, odd lanes the shifted
                // copy at lane + 125 - c.
                const float* rpair = (lane & 1) ? rtab + C::kBiasTab + lane + (C::BN - 3) : rtab + lane + (C::BN - 2);
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar(B_S_FULL + x), s_cnt & 1, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // this warp's two chunks: 32-column chunks kk = 2 hf + k of the tile, loaded
                // at once and kept in registers through both passes
                uint32_t sr[2][32];
                tmem_ld32(tS, sr[0]);
                tmem_ld32(tS + 32u, sr[1]);
                // In place: the scores of this warp's chunk k (tile chunk kk) become the
                // scaled, biased and masked scores minus `shift` (masked: -inf).
                auto to_x = [&](uint32_t (&r)[32], int k, float shift) {
                    const int kk = 2 * hf + k;
                    if constexpr (DENSE) {
                        // per-element bias, read only inside the row's allowed columns
                        const float bs = softmax ? 1.4426950408889634f : 1.0f;
                        const int lk = lim - 32 * kk, lok = lo - 32 * kk;
                        const float* src = drow + col0 + 32 * kk;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const bool in = i >= lok && i < lk;
                            const float bv = in ? __ldg(src + i) : 0.f;
                            r[i] = __float_as_uint(in ? fmaf(__uint_as_float(r[i]), xs, fmaf(bv, bs, -shift)) : -INFINITY);
                        }
                        return;
                    }
                    if (hmask & (1u << k)) {
                        const float2 sc = make_float2(xs, xs), add = make_float2(cb[k] - shift, cb[k] - shift);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 t2 = fma2(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), sc, add);
                            r[i] = __float_as_uint(t2.x);
                            r[i + 1] = __float_as_uint(t2.y);
                        }
                    } else {
                        const float2 sc = make_float2(xs, xs), ns = make_float2(-shift, -shift);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const float2 bb = *reinterpret_cast<const float2*>(rpair - (32 * kk + i));
                            const float2 t2 = fma2(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])), sc,
                                                   add2(make_float2(bb.y, bb.x), ns));
                            r[i] = __float_as_uint(t2.x);
                            r[i + 1] = __float_as_uint(t2.y);
                        }
                    }
                    if (!full) {
                        const int lk = lim - 32 * kk, lok = lo - 32 * kk;
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = (i >= lok && i < lk) ? r[i] : __float_as_uint(-INFINITY);
                    }
                };
                tmem_ld_wait(sr[0]);
                tmem_ld_wait(sr[1]);
                if constexpr (softmax) {
                    // pass 1: an upper bound of this half's row max from the raw scores (one
                    // FMNMX per element): xs * max(s) + the chunk's bias (constant, or the
                    // head's largest); the exact max for a dense bias.  Any m >= the true max
                    // gives the same P / l.  The partner's half completes the row.
                    const bool fast = !DENSE && full && hmask == 3u;
                    float mx = -INFINITY;
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int kk = 2 * hf + k;
                        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                        if (DENSE) {
                            to_x(sr[k], k, 0.f);  // exact x, kept for pass 2
#pragma unroll
                            for (int i = 0; i < 32; i += 2)
                                m4[(i >> 1) & 3] = fmax3(m4[(i >> 1) & 3], __uint_as_float(sr[k][i]), __uint_as_float(sr[k][i + 1]));
                            mx = fmaxf(mx, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
                            continue;
                        }
                        if (fast || full) {
#pragma unroll
                            for (int i = 0; i < 32; i += 2)
                                m4[(i >> 1) & 3] = fmax3(m4[(i >> 1) & 3], __uint_as_float(sr[k][i]), __uint_as_float(sr[k][i + 1]));
                        } else {
                            const int lk = lim - 32 * kk, lok = lo - 32 * kk;
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                m4[i & 3] = fmaxf(m4[i & 3], (i >= lok && i < lk) ? __uint_as_float(sr[k][i]) : -INFINITY);
                        }
                        const float mk = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                        mx = fmaxf(mx, fmaf(mk, xs, (hmask & (1u << k)) ? cb[k] : bmax));
                    }
                    float mo;
                    if (!exchange(mx, mo)) { ok = false; break; }
                    mx = fmaxf(mx, mo);
                    // Lazy rescaling: keep the running max unless it grows by more than 2^8;
                    // both O and l use the same stale max, so the final O / l is unchanged.
                    float m_new = m;
                    if (mx > m + 8.f) m_new = mx;
                    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                    const float alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_use);
                    const bool need_rescale = (m_new != m) && j > 0;
                    m = m_new;
                    // O of this tile is stable here: S_x(j) was issued after P_x(j-1) V
                    // completed, and P V of step j waits for this tile's P.
                    if (__any_sync(0xffffffffu, need_rescale)) {
#pragma unroll 1
                        for (int c = 0; c < OC / 8; ++c) {
                            uint32_t r[8];
                            tmem_ld8(tO + c * 8u, r);
                            tmem_ld_wait(r);
#pragma unroll
                            for (int i = 0; i < 8; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                            tmem_st8(tO + c * 8u, r);
                        }
                    }
                    // pass 2: P = exp2(x - m) (packed FMA folds in -m), packed row sum,
                    // P -> the chunk's first 16 TMEM columns
                    float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    if (!DENSE) {
                        // the raw scores again (cheaper than keeping 64 registers live across
                        // the exchange and the rescale)
                        tmem_ld32(tS, sr[0]);
                        tmem_ld32(tS + 32u, sr[1]);
                        tmem_ld_wait(sr[0]);
                        tmem_ld_wait(sr[1]);
                    }
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int kk = 2 * hf + k;
                        uint32_t pk[16];
                        if (!DENSE && full && (hmask & (1u << k))) {
                            const float2 xs2 = make_float2(xs, xs), add = make_float2(cb[k] - m_use, cb[k] - m_use);
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                const float2 t2 = fma2(make_float2(__uint_as_float(sr[k][i]), __uint_as_float(sr[k][i + 1])), xs2, add);
                                const float2 e2 = make_float2(ex2_approx(t2.x), ex2_approx(t2.y));
                                rs[(i >> 1) & 1] = add2(rs[(i >> 1) & 1], e2);
                                pk[i >> 1] = pack_bf16x2(e2.x, e2.y);
                            }
                        } else if (!DENSE && full) {
                            // no column masked, bias per element: the same single loop with the
                            // bias pair read from the table
                            const float2 xs2 = make_float2(xs, xs), nm = make_float2(-m_use, -m_use);
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                const float2 bb = *reinterpret_cast<const float2*>(rpair - (32 * kk + i));
                                const float2 t2 = fma2(make_float2(__uint_as_float(sr[k][i]), __uint_as_float(sr[k][i + 1])), xs2,
                                                       add2(make_float2(bb.y, bb.x), nm));
                                const float2 e2 = make_float2(ex2_approx(t2.x), ex2_approx(t2.y));
                                rs[(i >> 1) & 1] = add2(rs[(i >> 1) & 1], e2);
                                pk[i >> 1] = pack_bf16x2(e2.x, e2.y);
                            }
                        } else {
                            if (DENSE) {
                                const float2 sh = make_float2(-m_use, -m_use);
#pragma unroll
                                for (int i = 0; i < 32; i += 2) {
                                    const float2 t2 = add2(make_float2(__uint_as_float(sr[k][i]), __uint_as_float(sr[k][i + 1])), sh);
                                    sr[k][i] = __float_as_uint(t2.x);
                                    sr[k][i + 1] = __float_as_uint(t2.y);
                                }
                            } else {
                                to_x(sr[k], k, m_use);
                            }
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                const float2 e2 = make_float2(ex2_approx(__uint_as_float(sr[k][i])), ex2_approx(__uint_as_float(sr[k][i + 1])));
                                rs[(i >> 1) & 1] = add2(rs[(i >> 1) & 1], e2);
                                pk[i >> 1] = pack_bf16x2(e2.x, e2.y);
                            }
                        }
                        tmem_st16(tSt + 32u * kk, pk);
                    }
                    const float2 r01 = add2(rs[0], rs[1]);
                    l = l * alpha + (r01.x + r01.y);
                } else {
                    // GDPA: P = act(x), one pass; remainder P - bf16(P) beside it.
                    const bool gelu = p.mode == JFA_GDPA_GELU_TANH;
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int kk = 2 * hf + k;
                        to_x(sr[k], k, 0.f);
                        uint32_t pk[16], pl[16];
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            // masked entries are -inf here: contribute exactly 0
                            const float v0 = __uint_as_float(sr[k][i]), v1 = __uint_as_float(sr[k][i + 1]);
                            const float a0 = v0 == -INFINITY ? 0.f : gdpa_act(gelu, v0);
                            const float a1 = v1 == -INFINITY ? 0.f : gdpa_act(gelu, v1);
                            const uint32_t u = pack_bf16x2(a0, a1);
                            pk[i >> 1] = u;
                            pl[i >> 1] = pack_bf16x2(a0 - __uint_as_float(u << 16), a1 - __uint_as_float(u & 0xffff0000u));
                        }
                        tmem_st16(tSt + 32u * kk, pk);
                        tmem_st16(tSt + 32u * kk + 16u, pl);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_P_FULL + x));
                ++s_cnt;
            }
            if (!ok) break;
            // Epilogue: wait for the tile's last P V product, read O, release it.
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar(B_O_DONE + x), (s_cnt - 1) & 1, abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (split) {
                // Tile 1's warps hand over the row max and their partial sums; tile 0's warps
                // combine both halves of the key range over their O columns:
                // O = (O0 2^(m0-m) + O1 2^(m1-m)) / (l0 2^(m0-m) + l1 2^(m1-m)), m = max(m0, m1)
                // (GDPA: O = O0 + O1), then release both O accumulators.
                float* comb = comb_s + (split_cnt & 1) * 3 * C::BM;
                ++split_cnt;
                if (x == 1) {
                    if (hf == 0) comb[t] = m;
                    comb[(1 + hf) * C::BM + t] = l;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_COMBINE));
                    continue;
                }
                float l0 = l;
                if constexpr (softmax) {
                    float lo2;
                    if (!exchange(l, lo2)) { ok = false; break; }
                    l0 = l + lo2;
                }
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar(B_COMBINE), (split_cnt - 1) & 1, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float c0 = 1.f, c1 = 1.f, mm = m, ll = l0;
                if constexpr (softmax) {
                    const float m1 = comb[t], l1 = comb[C::BM + t] + comb[2 * C::BM + t];
                    mm = fmaxf(m, m1);
                    const float a0 = m == -INFINITY ? 0.f : ex2_approx(m - mm);
                    const float a1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - mm);
                    ll = fmaf(l0, a0, l1 * a1);
                    const float inv = ll > 0.f ? 1.f / ll : 0.f;
                    c0 = a0 * inv;
                    c1 = a1 * inv;
                }
                const uint32_t tO1 = tmem + lane_base + C::tmem_o(1) + uint32_t(OC * hf);
                OT* orow_p = reinterpret_cast<OT*>(p.O) + orow * D + OC * hf;
#pragma unroll
                for (int c = 0; c < OC / 32; ++c) {
                    uint32_t r0[32], r1[32];
                    float v[32];
                    tmem_ld32(tO + c * 32u, r0);
                    tmem_ld32(tO1 + c * 32u, r1);
                    tmem_ld_wait(r0);
                    tmem_ld_wait(r1);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = fmaf(__uint_as_float(r0[i]), c0, __uint_as_float(r1[i]) * c1);
                    if (row_valid) store_row<OT>(orow_p + c * 32, v, 32);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(B_O_EMPTY + 0));
                    mbar_arrive(bar(B_O_EMPTY + 1));
                }
                if (row_valid && softmax && p.lse && hf == 0)
                    p.lse[orow] = ll > 0.f ? (mm + __log2f(ll)) * 0.6931471805599453f : -INFINITY;
                continue;
            }
            {
                float lt = l;  // the row's sum over both halves (softmax)
                if constexpr (softmax) {
                    float lo2;
                    if (!exchange(l, lo2)) { ok = false; break; }
                    lt = l + lo2;
                }
                const float inv = (softmax && lt > 0.f) ? 1.f / lt : (softmax ? 0.f : 1.f);
                OT* orow_p = reinterpret_cast<OT*>(p.O) + orow * D + OC * hf;
#pragma unroll
                for (int c = 0; c < OC / 32; ++c) {
                    uint32_t r[32];
                    float v[32];
                    tmem_ld32(tO + c * 32u, r);
                    tmem_ld_wait(r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * inv;
                    if (row_valid) store_row<OT>(orow_p + c * 32, v, 32);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_O_EMPTY + x));
                if (row_valid && softmax && p.lse && hf == 0)
                    p.lse[orow] = lt > 0.f ? (m + __log2f(lt)) * 0.6931471805599453f : -INFINITY;
            }
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kMmaWarp) tmem_dealloc(tmem, C::kTmemCols);
}

template <int D, typename OT, bool GDPA, bool WIN, bool DENSE, bool SPLIT>
static cudaError_t launch_fwd_m(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                const FwdParams& p, int grid, cudaStream_t st) {
    using C = FwdCfg<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(jfa_fwd_kernel<D, OT, GDPA, WIN, DENSE, SPLIT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    jfa_fwd_kernel<D, OT, GDPA, WIN, DENSE, SPLIT><<<grid, C::kThreads, C::kSmemBytes, st>>>(tmQ, tmK, tmV, p);
    return cudaGetLastError();
}

template <int D, typename OT>
static cudaError_t launch_fwd_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                const FwdParams& p, int grid, bool split_list, cudaStream_t st) {
    const bool sm = p.mode == JFA_SOFTMAX;
    if (p.dense)  // dense bias: the window, if any, is taken at run time
        return sm ? launch_fwd_m<D, OT, false, true, true, false>(tmQ, tmK, tmV, p, grid, st)
                  : launch_fwd_m<D, OT, true, true, true, false>(tmQ, tmK, tmV, p, grid, st);
    if (p.window >= 0)
        return sm ? launch_fwd_m<D, OT, false, true, false, false>(tmQ, tmK, tmV, p, grid, st)
                  : launch_fwd_m<D, OT, true, true, false, false>(tmQ, tmK, tmV, p, grid, st);
    if (split_list)
        return sm ? launch_fwd_m<D, OT, false, false, false, true>(tmQ, tmK, tmV, p, grid, st)
                  : launch_fwd_m<D, OT, true, false, false, true>(tmQ, tmK, tmV, p, grid, st);
    return sm ? launch_fwd_m<D, OT, false, false, false, false>(tmQ, tmK, tmV, p, grid, st)
              : launch_fwd_m<D, OT, true, false, false, false>(tmQ, tmK, tmV, p, grid, st);
}

cudaError_t launch_fwd(int dtype, int o_dtype, int D, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const FwdParams& p, int grid, bool split_list, cudaStream_t st) {
    using bf16 = __nv_bfloat16;
    if (dtype != JFA_BF16) return cudaErrorInvalidValue;
    if (D == 128 && o_dtype == JFA_BF16) return launch_fwd_t<128, bf16>(tmQ, tmK, tmV, p, grid, split_list, st);
    if (D == 128 && o_dtype == JFA_F32) return launch_fwd_t<128, float>(tmQ, tmK, tmV, p, grid, split_list, st);
    if (D == 64 && o_dtype == JFA_BF16) return launch_fwd_t<64, bf16>(tmQ, tmK, tmV, p, grid, split_list, st);
    if (D == 64 && o_dtype == JFA_F32) return launch_fwd_t<64, float>(tmQ, tmK, tmV, p, grid, split_list, st);
    return cudaErrorInvalidValue;
}

bool supported(int dtype, int D) {
    return (dtype == JFA_BF16 && (D == 64 || D == 128)) || (dtype == JFA_F32 && (D == 32 || D == 64));
}

}  // namespace jfa
