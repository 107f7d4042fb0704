// Short-query softmax forward with two key tiles per score tile (bf16 inputs, head_dim 64,
// query sets of at most 64 rows, no bias, no causal mask or window).
//
// In the cross-attention shapes of the GEM articles a query set has at most 64 rows
// against a long key/value history (aihot.vn GEM article, "Generalized Dot-Product
// Attention (GDPA)": short or asymmetric K/V).  A 128-row query tile then leaves half of
// the tensor core's 128 accumulator lanes or more on padding rows.  Here each score tile
// holds the query set twice, once per lane half, against two different key tiles:
//   S = [Q 0; 0 Q] [K_a | K_b]^T     one M = 128, N = 128 product with K = 2 D:
//                                    lanes 0-63 score key tile a, lanes 64-127 key tile b
//   P' = [P_a 0; 0 P_b]              bf16 in TMEM: lanes 0-63 hold P over tile a's keys and
//                                    zeros over b's, lanes 64-127 the other way round
//   O += P' [V_a; V_b]               one product with K = 256 keys
// Each lane keeps its own online softmax (running max m and sum l, in log2 units of the
// scaled score) over the key tiles of its half, so a query row has two partial results,
// one per lane half, merged at the end of the item:
//   m = max(m_a, m_b),  l = l_a 2^(m_a - m) + l_b 2^(m_b - m),
//   o = (o_a 2^(m_a - m) + o_b 2^(m_b - m)) / l,  lse = (m + log2 l) ln 2.
// A row rescales O only when its maximum has grown by more than 8 (a factor 256) since
// the last rescale; until then P is formed against the older maximum and stays below 2^8.
// Item = (sequence, head) with all of its key tiles; Q stays in shared memory.
// TMEM: S double-buffered [0, 128) and [128, 256), P' [256, 384), O [384, 448); 512 columns.
//
// CTA = 6 warps: 0-3 softmax (thread = TMEM lane; lane r is query row r mod 64 of lane half
// r / 64), 4 TMA producer, 5 MMA issuer.
#include <cuda_bf16.h>

#include "bwd_common.cuh"
#include "jfa_internal.h"
#include "ptx.cuh"
#include "tilemath.cuh"

namespace jfa {

namespace {

struct FpCfg {
    static constexpr int D = 64, BQ = 64, BN = kFwdBN;
    static constexpr int kKVTile = BN * D * 2;     // one key tile, 16 KB
    static constexpr int kQ2 = 2 * 128 * 128;      // [Q 0; 0 Q]: two 128-row x 128-byte blocks
    static constexpr int kPair = 2 * kKVTile;      // two key (or value) tiles
    static constexpr int kOffQ2 = 0;
    static constexpr int kOffK = kOffQ2 + kQ2;     // two stages of key-tile pairs
    static constexpr int kOffV = kOffK + 2 * kPair;  // two stages of value-tile pairs
    // merge: lane half 1's O row (64 floats), m and l for each of the 64 query rows
    static constexpr int kOffX = kOffV + 2 * kPair;
    static constexpr int kXBytes = BQ * (D + 2) * 4;
    static constexpr int kOffBar = kOffX + kXBytes;
    static constexpr int kNumBars = 20;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
    static_assert(kSmemBytes <= 227 * 1024 && kSmemBytes > 114 * 1024, "one CTA per SM, within the budget");
    static constexpr uint32_t kTmS = 0, kTmP = 256, kTmO = 384, kTmCols = 512;
    static constexpr uint32_t kIdescS = make_idesc(kFmtBF16, 128, BN, false, false);
    static constexpr uint32_t kIdescPV = make_idesc(kFmtBF16, 128, D, false, true);
    static constexpr int kSoftWarps = 4, kProdWarp = 4, kMmaWarp = 5, kThreads = 6 * 32;
    static constexpr float kRescale = 8.f;  // log2 of the growth that forces a rescale of O
};

enum {
    FP_K_FULL = 0,   // +stage
    FP_K_EMPTY = 2,  // +stage
    FP_V_FULL = 4,   // +stage
    FP_V_EMPTY = 6,  // +stage
    FP_Q_FULL = 8,
    FP_Q_EMPTY = 9,
    FP_S_FULL = 10,  // +buffer
    FP_S_FREE = 12,  // +buffer: every softmax warp has read the S buffer
    FP_P_FULL = 14,  // every softmax warp has written P' (and any rescale of O)
    FP_P_FREE = 15,  // the P' V product is done: P' may be rewritten, O is stable
    FP_O_FULL = 16,  // the item's last product is done
    FP_O_EMPTY = 17, // every softmax warp has read O
    FP_X_FULL = 18,  // lane half 1 has written its partial results for the merge
    FP_DRAIN = 19,
};

template <typename OT>
__global__ void __launch_bounds__(FpCfg::kThreads, 1)
    jfa_fwd_pack_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using C = FpCfg;
    constexpr int D = C::D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ2 = sbase + C::kOffQ2, sK = sbase + C::kOffK, sV = sbase + C::kOffV;
    float* xbuf = reinterpret_cast<float*>(smem + C::kOffX);
    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * uint32_t(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The zero quarters of [Q 0; 0 Q] (block 0 rows 64-127 and block 1 rows 0-63: bytes
    // [8 KB, 24 KB) of the operand) are written once; the loads only ever fill the other two.
    for (int i = threadIdx.x; i < 16384 / 16; i += blockDim.x) st_shared_v4(sQ2 + 8192u + uint32_t(16 * i), 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(FP_K_FULL + s), 1);
            mbar_init(bar(FP_K_EMPTY + s), 1);
            mbar_init(bar(FP_V_FULL + s), 1);
            mbar_init(bar(FP_V_EMPTY + s), 1);
            mbar_init(bar(FP_S_FULL + s), 1);
            mbar_init(bar(FP_S_FREE + s), C::kSoftWarps);
        }
        mbar_init(bar(FP_Q_FULL), 1);
        mbar_init(bar(FP_Q_EMPTY), 1);
        mbar_init(bar(FP_P_FULL), C::kSoftWarps);
        mbar_init(bar(FP_P_FREE), 1);
        mbar_init(bar(FP_O_FULL), 1);
        mbar_init(bar(FP_O_EMPTY), C::kSoftWarps);
        mbar_init(bar(FP_X_FULL), 2);
        mbar_init(bar(FP_DRAIN), 1);
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
            uint32_t g = 0, item_it = 0;  // pairs loaded, items whose Q was loaded
            uint32_t k_extra = 0;         // 1: the last K pair went out but its V pair did not
            bool ok = true;
            // key and value tiles 2u and 2u+1 of the item (the second may lie past the
            // sequence: those keys are masked, and the rows read are finite)
            auto load_pair = [&](int h, int row) -> bool {
                const uint32_t st = g & 1, ph = ((g >> 1) & 1) ^ 1;
                if (!mbar_wait_bounded(bar(FP_K_EMPTY + st), ph, abort_flag)) return false;
                mbar_arrive_expect_tx(bar(FP_K_FULL + st), C::kPair);
                for (int t = 0; t < 2; ++t)
                    tma_load_2d(sK + st * C::kPair + t * C::kKVTile, &tmK, bar(FP_K_FULL + st), h * D,
                                row + t * C::BN);
                if (!mbar_wait_bounded(bar(FP_V_EMPTY + st), ph, abort_flag)) {
                    k_extra = 1;
                    return false;
                }
                mbar_arrive_expect_tx(bar(FP_V_FULL + st), C::kPair);
                for (int t = 0; t < 2; ++t)
                    tma_load_2d(sV + st * C::kPair + t * C::kKVTile, &tmV, bar(FP_V_FULL + st), h * D,
                                row + t * C::BN);
                ++g;
                return true;
            };
            for (int it = it_begin; it < it_end && ok; ++it) {
                const int4 w = p.items[it];
                if (!short_fwd_item_ok(w, p, C::BQ)) {  // not an item of this plan: skipped by every role
                    atomicOr(p.status, kStatusBounds);
                    continue;
                }
                const int b = w.x, h = w.y, n = w.w;
                const int q0 = p.q_off[b], q_len = p.q_off[b + 1] - q0, kv0 = p.kv_off[b];
                if (q_len == 0 || n == 0) continue;
                const int steps = (n + 1) / 2;
                if (!load_pair(h, kv0)) { ok = false; break; }
                if (!mbar_wait_bounded(bar(FP_Q_EMPTY), (item_it & 1) ^ 1, abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(FP_Q_FULL), 2 * C::BQ * 128);
                tma_load_2d(sQ2, &tmQ, bar(FP_Q_FULL), h * D, q0);                          // block 0, rows 0-63
                tma_load_2d(sQ2 + 128 * 128 + 64 * 128, &tmQ, bar(FP_Q_FULL), h * D, q0);  // block 1, rows 64-127
                ++item_it;
                for (int u = 1; u < steps; ++u)
                    if (!load_pair(h, kv0 + 2 * u * C::BN)) { ok = false; break; }
            }
            if (!ok) fail();
            drain_ring(bar(FP_Q_FULL), item_it, 1);
            drain_ring(bar(FP_K_FULL), g + k_extra, 2);
            drain_ring(bar(FP_V_FULL), g, 2);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        uint32_t g0 = 0, item_it = 0;
        bool ok = true;
        const SDesc dQ2 = sdesc_sw128(sQ2, 16, 1024);
        auto koff = [](int s) -> uint32_t { return uint32_t(((s * 32) >> 7) * 128 * 128 + ((s * 32) & 127)); };
        // S(g) = [Q 0; 0 Q] [K_a | K_b]^T into buffer g & 1, once its previous scores are read
        auto issue_s = [&](uint32_t g, bool last_of_item) -> bool {
            const uint32_t st = g & 1;
            if (!warp_wait(FP_K_FULL + st, (g >> 1) & 1)) return false;
            if (g >= 2 && !warp_wait(FP_S_FREE + st, ((g >> 1) - 1) & 1)) return false;
            tc_fence_after();
            if (elect_one()) {
                const SDesc kb = sdesc_sw128(sK + st * C::kPair, 16, 1024);
#pragma unroll
                for (int s = 0; s < 2 * D / 16; ++s)
                    mma_ss(tmem + C::kTmS + st * 128u, dQ2, koff(s), kb, koff(s), C::kIdescS, s > 0);
                tc_commit(bar(FP_S_FULL + st));
                tc_commit(bar(FP_K_EMPTY + st));
                if (last_of_item) tc_commit(bar(FP_Q_EMPTY));
            }
            __syncwarp();
            return true;
        };
        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 w = p.items[it];
            if (!short_fwd_item_ok(w, p, C::BQ)) continue;
            const int b = w.x, n = w.w;
            const int q_len = p.q_off[b + 1] - p.q_off[b];
            if (q_len == 0 || n == 0) continue;
            const int steps = (n + 1) / 2;
            if (!warp_wait(FP_Q_FULL, item_it & 1)) { ok = false; break; }
            if (!issue_s(g0, steps == 1)) { ok = false; break; }
            for (int u = 0; u < steps && ok; ++u) {
                const uint32_t g = g0 + uint32_t(u), st = g & 1;
                if (u + 1 < steps && !issue_s(g + 1, u + 2 == steps)) { ok = false; break; }
                // O += P' [V_a; V_b] once P' is written (the item's first product also waits for
                // the previous item's O to have been read out)
                if (!warp_wait(FP_P_FULL, g & 1) || !warp_wait(FP_V_FULL + st, (g >> 1) & 1)) { ok = false; break; }
                if (u == 0 && item_it > 0 && !warp_wait(FP_O_EMPTY, (item_it - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                if (elect_one()) {
                    const SDesc vb = sdesc_sw128(sV + st * C::kPair, 128 * 128, 1024);
#pragma unroll
                    for (int s = 0; s < 2 * C::BN / 16; ++s)
                        mma_ts(tmem + C::kTmO, tmem + C::kTmP + 8u * uint32_t(s), vb, uint32_t(s) * 2048u, C::kIdescPV,
                               u > 0 || s > 0);
                    tc_commit(bar(FP_P_FREE));
                    tc_commit(bar(FP_V_EMPTY + st));
                    if (u + 1 == steps) tc_commit(bar(FP_O_FULL));
                }
                __syncwarp();
            }
            if (!ok) break;
            g0 += uint32_t(steps);
            ++item_it;
        }
        if (!ok) fail();
        if (elect_one()) tc_commit(bar(FP_DRAIN));
        __syncwarp();
        mbar_wait_bounded(bar(FP_DRAIN), 0, nullptr);
    } else {
        // ------------------------------------------------------------ softmax, merge, epilogue
        const int r = warp * 32 + lane;  // TMEM lane
        const int half = r >> 6, qi = r & 63;
        const uint32_t lane_base = uint32_t(warp * 32) << 16;
        const uint32_t tP = tmem + lane_base + C::kTmP, tO = tmem + lane_base + C::kTmO;
        const float xs = p.scale_log2;
        uint32_t g = 0, item_it = 0;
        bool ok = true;
        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 w = p.items[it];
            if (!short_fwd_item_ok(w, p, C::BQ)) continue;
            const int b = w.x, h = w.y, n = w.w;
            const int q0 = p.q_off[b], q_len = p.q_off[b + 1] - q0;
            const int kv_len = p.kv_off[b + 1] - p.kv_off[b];
            if (q_len == 0) continue;
            OT* o_row = reinterpret_cast<OT*>(p.O) + (size_t(q0 + qi) * size_t(p.H) + size_t(h)) * D;
            float* lse_row = p.lse + size_t(q0 + qi) * size_t(p.H) + size_t(h);
            if (n == 0) {  // no key: O = 0, lse = -inf
                if (half == 0 && qi < q_len) {
#pragma unroll
                    for (int i = 0; i < D; ++i) o_row[i] = OT(0.f);
                    *lse_row = -INFINITY;
                }
                continue;
            }
            const int steps = (n + 1) / 2;
            const bool row_ok = qi < q_len;
            float m_use = -INFINITY, l = 0.f;  // running maximum (as used for P) and sum
            for (int u = 0; u < steps; ++u, ++g) {
                const uint32_t st = g & 1;
                const uint32_t tS = tmem + lane_base + C::kTmS + st * 128u;
                // valid keys of this lane's tile 2u + half: [0, hi)
                const int hi = row_ok ? min(C::BN, max(0, kv_len - (2 * u + half) * C::BN)) : 0;
                // Masking is per lane where each lane's tile is wholly valid or wholly masked
                // (a query row past the set's end, a tile past the sequence's end): such a lane
                // gets m = -inf and an exponent argument of -inf, so P = 0 with no per-element
                // select.  Only a sequence's last, partial key tile is masked per element, and a
                // warp with no valid key at all only writes zeros.
                const bool partial = __any_sync(0xffffffffu, hi > 0 && hi < C::BN);
                const bool none = __all_sync(0xffffffffu, hi == 0);
                if (!warp_wait(FP_S_FULL + st, (g >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                // pass 1: the tile's row maximum
                float mx = -INFINITY;
                if (!none) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t v[32];
                        tmem_ld32(tS + 32u * k, v);
                        tmem_ld_wait(v);
                        if (partial) {
#pragma unroll
                            for (int c = 0; c < 32; c += 2) {
                                const int cc = 32 * k + c;
                                const float a = cc < hi ? __uint_as_float(v[c]) : -INFINITY;
                                const float a1 = cc + 1 < hi ? __uint_as_float(v[c + 1]) : -INFINITY;
                                mx = fmax3(mx, a, a1);
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < 32; c += 2) mx = fmax3(mx, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
                        }
                    }
                }
                const float m_tile = hi > 0 ? mx * xs : -INFINITY;
                // P' may be rewritten, and O is stable, once the previous product is done
                if (g > 0 && !warp_wait(FP_P_FREE, (g - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                // A new maximum more than 2^8 above the one in use: rescale this row's O and sum
                // to it (O and l are still 0 before the row's first valid key).  TMEM loads
                // and stores are warp-wide, so the warp rescales when any of its rows must
                // (alpha = 1 for the others).
                const bool grow = m_tile > m_use + C::kRescale;
                const float alpha = (grow && m_use != -INFINITY) ? ex2_approx(m_use - m_tile) : 1.f;
                if (__any_sync(0xffffffffu, grow && m_use != -INFINITY)) {
                    l *= alpha;
                    uint32_t o[32];
#pragma unroll
                    for (int k = 0; k < D / 32; ++k) {
                        tmem_ld32(tO + 32u * k, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                        tmem_st32(tO + 32u * k, o);
                    }
                }
                if (grow) m_use = m_tile;
                // pass 2: P = 2^(x s - m) over the lane's key tile, into its half of P'; zeros
                // into the other half (and into both for a warp with no valid key)
                const float nmv = hi > 0 ? -m_use : -INFINITY;
                const float2 nm = make_float2(nmv, nmv), xs2 = make_float2(xs, xs);
                float2 sum2 = make_float2(0.f, 0.f);
                uint32_t z[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) z[c] = 0u;
                if (!none) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t v[32];
                        tmem_ld32(tS + 32u * k, v);
                        tmem_ld_wait(v);
                        uint32_t pk[16];
#pragma unroll
                        for (int c = 0; c < 32; c += 2) {
                            const float2 e =
                                fma2(make_float2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), xs2, nm);
                            float p0 = ex2_approx(e.x), p1 = ex2_approx(e.y);
                            if (partial) {
                                const int cc = 32 * k + c;
                                p0 = cc < hi ? p0 : 0.f;
                                p1 = cc + 1 < hi ? p1 : 0.f;
                            }
                            sum2 = add2(sum2, make_float2(p0, p1));
                            pk[c >> 1] = pack_bf16x2(p0, p1);
                        }
                        tmem_st16(tP + uint32_t(64 * half + 16 * k), pk);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) tmem_st16(tP + uint32_t(64 * half + 16 * k), z);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) tmem_st16(tP + uint32_t(64 * (1 - half) + 16 * k), z);
                l += sum2.x + sum2.y;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(FP_S_FREE + st));
                    mbar_arrive(bar(FP_P_FULL));
                }
            }
            if (!ok) break;
            // merge the two lane halves' partial results for each query row, then write O
            // and lse (lane half 0)
            if (!warp_wait(FP_O_FULL, item_it & 1)) { ok = false; break; }
            tc_fence_after();
            uint32_t o[D];
            {
                uint32_t (&o0)[32] = *reinterpret_cast<uint32_t(*)[32]>(o);
                uint32_t (&o1)[32] = *reinterpret_cast<uint32_t(*)[32]>(o + 32);
                tmem_ld32(tO, o0);
                tmem_ld32(tO + 32u, o1);
                tmem_ld_wait(o0);
                tmem_ld_wait(o1);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(FP_O_EMPTY));
            float* xr = xbuf + qi * (D + 2);
            if (half == 1) {
#pragma unroll
                for (int c = 0; c < D; ++c) xr[c] = __uint_as_float(o[c]);
                xr[D] = m_use;
                xr[D + 1] = l;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(FP_X_FULL));
            } else {
                if (!warp_wait(FP_X_FULL, item_it & 1)) { ok = false; break; }
                if (row_ok) {
                    const float mb = xr[D], lb = xr[D + 1];
                    const float m = fmaxf(m_use, mb);
                    const float aa = m_use == -INFINITY ? 0.f : ex2_approx(m_use - m);
                    const float ab = mb == -INFINITY ? 0.f : ex2_approx(mb - m);
                    const float lt = l * aa + lb * ab;
                    const float inv = lt > 0.f ? 1.f / lt : 0.f;
                    float out[D];
#pragma unroll
                    for (int c = 0; c < D; ++c) out[c] = (__uint_as_float(o[c]) * aa + xr[c] * ab) * inv;
                    if constexpr (sizeof(OT) == 2) {
                        store_bf16_row(reinterpret_cast<__nv_bfloat16*>(o_row), out, D, 1.f);
                    } else {
#pragma unroll
                        for (int c = 0; c < D; c += 4)
                            *reinterpret_cast<float4*>(reinterpret_cast<float*>(o_row) + c) =
                                make_float4(out[c], out[c + 1], out[c + 2], out[c + 3]);
                    }
                    *lse_row = lt > 0.f ? (m + __log2f(lt)) * 0.6931471805599453f : -INFINITY;
                }
            }
            ++item_it;
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kMmaWarp) tmem_dealloc(tmem, C::kTmCols);
}

template <typename OT>
cudaError_t launch_fp_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const FwdParams& p,
                        int grid, cudaStream_t st) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(jfa_fwd_pack_kernel<OT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             FpCfg::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    jfa_fwd_pack_kernel<OT><<<grid, FpCfg::kThreads, FpCfg::kSmemBytes, st>>>(tmQ, tmK, tmV, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_pack(int o_dtype, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const FwdParams& p, int grid, cudaStream_t st) {
    if (p.mode != JFA_SOFTMAX) return cudaErrorInvalidValue;
    if (o_dtype == JFA_BF16) return launch_fp_t<__nv_bfloat16>(tmQ, tmK, tmV, p, grid, st);
    if (o_dtype == JFA_F32) return launch_fp_t<float>(tmQ, tmK, tmV, p, grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace jfa
