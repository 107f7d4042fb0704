// Backward kernels: jagged flash attention / GDPA gradients on sm_103a.
//
// The backward is parallelised over key/value tiles, as the kerneldigest.dev
// summary of the GEM work describes for JFA ("paralelización de backward pass",
// section "Arquitectura del Sistema"), and dQ is accumulated without any padded
// tensor -- the "backward accumulation" the vibekk.com article lists among the
// bottlenecks that remain once padding is gone (section 第一轮瓶颈迁移).
//
//   preprocess  Delta_i = sum_d dO_id O_id (softmax only), dQ accumulator := 0
//   main        persistent over (sequence, head, 128-row key tile); K and V stay in
//               shared memory while 64-row query tiles stream through:
//                 S^T  = K Q_i^T           (TMEM, lanes = key rows)
//                 dP^T = V dO_i^T          (TMEM)
//                 P^T  = exp(S^T - lse) or act(S^T);  dS^T = P^T (dP^T - Delta) or
//                        act'(S^T) dP^T     (registers -> shared memory, bf16/fp32)
//                 dV  += P^T dO_i,  dK += dS^T Q_i      (TMEM accumulators)
//                 dQ_i^T = K^T dS^T         (TMEM, lanes = head-dim) -> fp32
//                        atomics into the jagged dQ accumulator, coalesced along D
//   post        dQ = scale * accumulator, converted to the element type
//
// CTA = 10 warps: 0-3 compute P/dS (thread = key row), 4-7 dQ reduction and the
// dK/dV epilogue, 8 TMA producer, 9 MMA issuer.  TMEM (512 columns): dV [0,128),
// dK [128,256), S^T double buffer [256,320) [320,384), dP^T [384,448),
// dQ^T [448,512).
#include "jfa_internal.h"
#include "ptx.cuh"
#include "tilemath.cuh"

#include <algorithm>

namespace jfa {

namespace {

template <typename T>
struct BElem;
template <>
struct BElem<__nv_bfloat16> {
    static constexpr int kBytes = 2;
    static constexpr uint32_t kFmt = kFmtBF16;
    static constexpr int kUmmaK = 16;
};
template <>
struct BElem<float> {
    static constexpr int kBytes = 4;
    static constexpr uint32_t kFmt = kFmtTF32;
    static constexpr int kUmmaK = 8;
};

template <typename T, int D>
struct BwdCfg {
    static constexpr int BN = kBwdBN;  // key rows (TMEM lanes)
    static constexpr int BM = kBwdBM;  // query rows per step
    static constexpr int E = BElem<T>::kBytes;
    static constexpr int kRowBytes = D * E;
    static_assert(kRowBytes % 128 == 0 && kRowBytes <= 256, "head row must be 128 or 256 bytes");
    static constexpr int kCB = kRowBytes / 128;
    static constexpr int kBoxCols = 128 / E;
    static constexpr int kKVTile = BN * kRowBytes;  // one of K, V
    static constexpr int kQTile = BM * kRowBytes;   // one of Q_i, dO_i
    static constexpr int kPRowBytes = BM * E;       // P^T / dS^T row (one key row)
    static constexpr int kPTile = BN * kPRowBytes;
    static constexpr int kStages = 2;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kKVTile;
    static constexpr int kOffQ = kOffV + kKVTile;               // + stage * kQTile
    static constexpr int kOffDO = kOffQ + kStages * kQTile;     // + stage * kQTile
    static constexpr int kOffPt = kOffDO + kStages * kQTile;
    static constexpr int kOffDSt = kOffPt + kPTile;
    static constexpr int kOffBar = kOffDSt + kPTile;
    static constexpr int kNumBars = 24;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    // Warp roles: kCompWarps compute warps (two warpgroups, each owning 32 of the 64
    // query columns of a step), 4 dQ/epilogue warps, 1 TMA producer, 1 MMA issuer.
    static constexpr int kCompWarps = 8;
    static constexpr int kDqWarp0 = kCompWarps;
    static constexpr int kProdWarp = kCompWarps + 4;
    static constexpr int kMmaWarp = kCompWarps + 5;
    static constexpr int kColsPerWarp = BM * 4 / kCompWarps;  // query columns per compute thread
    // tmem slot + abort flag (16 B), per compute warp: lse, delta (one per column), bias[32]
    static constexpr int kMiscBytes = 16 + kCompWarps * (2 * kColsPerWarp + 32) * 4;
    static constexpr int kSmemNeed = kOffMisc + kMiscBytes + 1024;
    // At least 120 KB so that exactly one CTA fits on an SM: the CTA allocates all
    // 512 TMEM columns.
    static constexpr int kSmemBytes = kSmemNeed > 120 * 1024 ? kSmemNeed : 120 * 1024;
    static constexpr int kUmmaK = BElem<T>::kUmmaK;
    static constexpr int kDSteps = D / kUmmaK;    // contraction over head_dim
    static constexpr int kQSteps = BM / kUmmaK;   // contraction over query rows
    static constexpr int kKVSteps = BN / kUmmaK;  // contraction over key rows
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTmDV = 0, kTmDK = 128, kTmS = 256, kTmDP = 384, kTmDQ = 448;
    static constexpr uint32_t kIdescST = make_idesc(BElem<T>::kFmt, BN, BM, false, false);
    static constexpr uint32_t kIdescAcc = make_idesc(BElem<T>::kFmt, BN, D, false, true);
    static constexpr uint32_t kIdescDQ = make_idesc(BElem<T>::kFmt, 128, BM, true, true);
    static constexpr int kThreads = (kCompWarps + 6) * 32;
};

enum {
    C_KV_FULL = 0,
    C_KV_EMPTY = 1,
    C_Q_FULL = 2,    // +stage
    C_Q_EMPTY = 4,   // +stage
    C_S_FULL = 6,    // +buffer
    C_S_EMPTY = 8,   // +buffer
    C_DP_FULL = 10,
    C_DP_EMPTY = 11,
    C_PT_FULL = 12,
    C_PT_EMPTY = 13,
    C_DS_FULL = 14,
    C_DS_EMPTY = 15,
    C_DQ_FULL = 16,
    C_DQ_EMPTY = 17,
    C_ACC_FULL = 18,
    C_ACC_EMPTY = 19,
    C_DRAIN = 20,
};

template <typename T>
__device__ __forceinline__ void store_vec(T* dst, const float* v, int n, float mul);

template <>
__device__ __forceinline__ void store_vec<__nv_bfloat16>(__nv_bfloat16* dst, const float* v, int n, float mul) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (int i = 0; i < n / 8; ++i) {
        uint4 u;
        u.x = pack_bf16x2(v[8 * i + 0] * mul, v[8 * i + 1] * mul);
        u.y = pack_bf16x2(v[8 * i + 2] * mul, v[8 * i + 3] * mul);
        u.z = pack_bf16x2(v[8 * i + 4] * mul, v[8 * i + 5] * mul);
        u.w = pack_bf16x2(v[8 * i + 6] * mul, v[8 * i + 7] * mul);
        d4[i] = u;
    }
}

template <>
__device__ __forceinline__ void store_vec<float>(float* dst, const float* v, int n, float mul) {
    float4* d4 = reinterpret_cast<float4*>(dst);
    for (int i = 0; i < n / 4; ++i)
        d4[i] = make_float4(v[4 * i] * mul, v[4 * i + 1] * mul, v[4 * i + 2] * mul, v[4 * i + 3] * mul);
}

// Write 32 values (query columns [32*half, 32*half+32)) of key row `r` of P^T or
// dS^T into the 128-byte swizzled K-major bf16 tile at `base` (a row is 64 columns =
// 128 bytes = 8 chunks of 16 bytes).
template <typename T>
__device__ __forceinline__ void write_ptile_half(uint32_t base, int r, int half, const float* v) {
    static_assert(sizeof(T) == 2, "bf16 tiles only");
#pragma unroll
    for (int k = 0; k < 4; ++k)
        st_shared_v4(base + sw128_offset(r, half * 4 + k), pack_bf16x2(v[8 * k], v[8 * k + 1]),
                     pack_bf16x2(v[8 * k + 2], v[8 * k + 3]), pack_bf16x2(v[8 * k + 4], v[8 * k + 5]),
                     pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
}

template <typename T, int D>
__global__ void __launch_bounds__(448, 1)
    jfa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                   const BwdParams p) {
    using C = BwdCfg<T, D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sK = sbase + C::kOffK, sV = sbase + C::kOffV, sQ = sbase + C::kOffQ,
                   sDO = sbase + C::kOffDO, sPt = sbase + C::kOffPt, sDSt = sbase + C::kOffDSt;
    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * uint32_t(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    float* misc_f = reinterpret_cast<float*>(smem + C::kOffMisc + 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(bar(C_KV_FULL), 1);
        mbar_init(bar(C_KV_EMPTY), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(C_Q_FULL + s), 1);
            mbar_init(bar(C_Q_EMPTY + s), 1);
            mbar_init(bar(C_S_FULL + s), 1);
            mbar_init(bar(C_S_EMPTY + s), C::kCompWarps);
        }
        mbar_init(bar(C_DP_FULL), 1);
        mbar_init(bar(C_DP_EMPTY), C::kCompWarps);
        mbar_init(bar(C_PT_FULL), C::kCompWarps);
        mbar_init(bar(C_PT_EMPTY), 1);
        mbar_init(bar(C_DS_FULL), C::kCompWarps);
        mbar_init(bar(C_DS_EMPTY), 1);
        mbar_init(bar(C_DQ_FULL), 1);
        mbar_init(bar(C_DQ_EMPTY), 4);
        mbar_init(bar(C_ACC_FULL), 1);
        mbar_init(bar(C_ACC_EMPTY), 4);
        mbar_init(bar(C_DRAIN), 1);
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
            bool ok = true;
            for (int it = it_begin; it < it_end && ok; ++it) {
                const int4 w = p.items[it];
                const int n = w.w;
                if (n == 0) continue;
                const int b = w.x, h = w.y, nt = w.z;
                const int q0 = p.q_off[b], q_len = p.q_off[b + 1] - q0, kv0 = p.kv_off[b];
                const int first_qt = (q_len + C::BM - 1) / C::BM - n;
                if (!mbar_wait_bounded(bar(C_KV_EMPTY), (item_it & 1) ^ 1, abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(C_KV_FULL), 2 * C::kKVTile);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb) {
                    tma_load_2d(sK + cb * C::BN * 128, &tmK, bar(C_KV_FULL), h * D + cb * C::kBoxCols, kv0 + nt * C::BN);
                    tma_load_2d(sV + cb * C::BN * 128, &tmV, bar(C_KV_FULL), h * D + cb * C::kBoxCols, kv0 + nt * C::BN);
                }
                ++item_it;
                for (int i = 0; i < n; ++i, ++step_it) {
                    const uint32_t st = step_it & 1, ph = (step_it >> 1) & 1;
                    const int y = q0 + (first_qt + i) * C::BM;
                    if (!mbar_wait_bounded(bar(C_Q_EMPTY + st), ph ^ 1, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(bar(C_Q_FULL + st), 2 * C::kQTile);
#pragma unroll
                    for (int cb = 0; cb < C::kCB; ++cb) {
                        tma_load_2d(sQ + st * C::kQTile + cb * C::BM * 128, &tmQ, bar(C_Q_FULL + st),
                                    h * D + cb * C::kBoxCols, y);
                        tma_load_2d(sDO + st * C::kQTile + cb * C::BM * 128, &tmdO, bar(C_Q_FULL + st),
                                    h * D + cb * C::kBoxCols, y);
                    }
                }
            }
            if (!ok) fail();
            if (item_it > 0) mbar_wait_bounded(bar(C_KV_FULL), (item_it - 1) & 1, nullptr);
            for (uint32_t s = 0; s < 2; ++s)
                if (step_it > s) {
                    const uint32_t last = ((step_it - 1 - s) / 2) * 2 + s;
                    mbar_wait_bounded(bar(C_Q_FULL + s), (last >> 1) & 1, nullptr);
                }
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t step_it = 0, item_it = 0;
            bool ok = true;
            // Descriptors built once; each MMA adds a compile-time byte offset.
            const SDesc dK = sdesc_sw128(sK, 16, 1024), dV = sdesc_sw128(sV, 16, 1024);
            const SDesc dQk[2] = {sdesc_sw128(sQ, 16, 1024), sdesc_sw128(sQ + C::kQTile, 16, 1024)};
            const SDesc dOk[2] = {sdesc_sw128(sDO, 16, 1024), sdesc_sw128(sDO + C::kQTile, 16, 1024)};
            const SDesc dQm[2] = {sdesc_sw128(sQ, C::BM * 128, 1024), sdesc_sw128(sQ + C::kQTile, C::BM * 128, 1024)};
            const SDesc dOm[2] = {sdesc_sw128(sDO, C::BM * 128, 1024),
                                  sdesc_sw128(sDO + C::kQTile, C::BM * 128, 1024)};
            const SDesc dPt = sdesc_sw128(sPt, 16, 1024), dDSt = sdesc_sw128(sDSt, 16, 1024);
            const SDesc dKm = sdesc_sw128(sK, C::BN * 128, 1024), dDSm = sdesc_sw128(sDSt, C::BN * 128, 1024);
            for (int it = it_begin; it < it_end && ok; ++it) {
                const int n = p.items[it].w;
                if (n == 0) continue;
                if (!mbar_wait_bounded(bar(C_KV_FULL), item_it & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                for (int i = 0; i <= n && ok; ++i) {
                    if (i < n) {
                        const uint32_t g = step_it + i, st = g & 1, ph = (g >> 1) & 1;
                        if (!mbar_wait_bounded(bar(C_Q_FULL + st), ph, abort_flag) ||
                            !mbar_wait_bounded(bar(C_S_EMPTY + st), ph ^ 1, abort_flag)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int s = 0; s < C::kDSteps; ++s)  // S^T = K Q^T
                            mma_ss(tmem + C::kTmS + st * 64u, dK, ((s * 32) >> 7) * C::BN * 128 + ((s * 32) & 127),
                                   dQk[st], ((s * 32) >> 7) * C::BM * 128 + ((s * 32) & 127), C::kIdescST, s > 0);
                        tc_commit(bar(C_S_FULL + st));
                        if (!mbar_wait_bounded(bar(C_DP_EMPTY), (g & 1) ^ 1, abort_flag)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int s = 0; s < C::kDSteps; ++s)  // dP^T = V dO^T
                            mma_ss(tmem + C::kTmDP, dV, ((s * 32) >> 7) * C::BN * 128 + ((s * 32) & 127), dOk[st],
                                   ((s * 32) >> 7) * C::BM * 128 + ((s * 32) & 127), C::kIdescST, s > 0);
                        tc_commit(bar(C_DP_FULL));
                    }
                    if (i > 0) {
                        const int ii = i - 1;
                        const uint32_t g = step_it + ii, st = g & 1;
                        if (!mbar_wait_bounded(bar(C_PT_FULL), g & 1, abort_flag)) { ok = false; break; }
                        if (ii == 0 && !mbar_wait_bounded(bar(C_ACC_EMPTY), (item_it & 1) ^ 1, abort_flag)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int s = 0; s < C::kQSteps; ++s)  // dV += P^T dO
                            mma_ss(tmem + C::kTmDV, dPt, ((s * 32) >> 7) * C::BN * 128 + ((s * 32) & 127), dOm[st],
                                   s * C::kUmmaK * 128, C::kIdescAcc, (ii > 0 || s > 0));
                        tc_commit(bar(C_PT_EMPTY));
                        if (!mbar_wait_bounded(bar(C_DS_FULL), g & 1, abort_flag)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int s = 0; s < C::kQSteps; ++s)  // dK += dS^T Q
                            mma_ss(tmem + C::kTmDK, dDSt, ((s * 32) >> 7) * C::BN * 128 + ((s * 32) & 127), dQm[st],
                                   s * C::kUmmaK * 128, C::kIdescAcc, (ii > 0 || s > 0));
                        if (!mbar_wait_bounded(bar(C_DQ_EMPTY), (g & 1) ^ 1, abort_flag)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int s = 0; s < C::kKVSteps; ++s)  // dQ^T = K^T dS^T
                            mma_ss(tmem + C::kTmDQ, dKm, s * C::kUmmaK * 128, dDSm, s * C::kUmmaK * 128, C::kIdescDQ,
                                   s > 0);
                        tc_commit(bar(C_DQ_FULL));
                        tc_commit(bar(C_DS_EMPTY));
                        tc_commit(bar(C_Q_EMPTY + st));
                    }
                }
                if (!ok) break;
                tc_commit(bar(C_ACC_FULL));
                tc_commit(bar(C_KV_EMPTY));
                step_it += n;
                ++item_it;
            }
            if (!ok) fail();
            tc_commit(bar(C_DRAIN));
            mbar_wait_bounded(bar(C_DRAIN), 0, nullptr);
        }
    } else if (warp < C::kCompWarps) {
        // ------------------------------------------------------------ P^T and dS^T
        // Thread = key row r (TMEM lane); warpgroup cw owns query columns
        // [cw*32, cw*32+32) of each 64-row step.
        constexpr int NC = C::kColsPerWarp;
        const int r = (warp & 3) * 32 + lane;
        const int cw = warp >> 2;
        const int c0 = cw * NC;
        const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
        float* lse_s = misc_f + warp * (2 * NC + 32);
        float* del_s = lse_s + NC;
        float* bias_w = del_s + NC;
        const bool softmax = p.mode == JFA_SOFTMAX;
        const bool gelu = p.mode == JFA_GDPA_GELU_TANH;
        uint32_t step_it = 0;
        bool ok = true;
        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 w = p.items[it];
            const int n = w.w;
            if (n == 0) continue;
            const int b = w.x, h = w.y, nt = w.z;
            const int q0 = p.q_off[b], q_len = p.q_off[b + 1] - q0;
            const int kv_len = p.kv_off[b + 1] - p.kv_off[b];
            const int diag = kv_len - q_len;
            const int first_qt = (q_len + C::BM - 1) / C::BM - n;
            const int j = nt * C::BN + r;  // key row within the sequence
            const bool key_valid = j < kv_len;
            if (p.bias) bias_w[lane] = p.bias[h * 32 + lane] * (softmax ? 1.4426950408889634f : 1.0f);
            // Row terms (lse in log2 units, Delta) of this warp's query columns: lane l
            // holds column c0 + l, fetched one step ahead so the latency hides.
            float nl = 0.f, nd = 0.f;
            auto fetch = [&](int qrow0) {
                const int c = c0 + lane;
                const bool v = softmax && qrow0 + c < q_len;
                const size_t ridx = (size_t(q0) + size_t(v ? qrow0 + c : 0)) * size_t(p.H) + size_t(h);
                nl = v ? p.lse[ridx] * 1.4426950408889634f : 0.f;
                nd = v ? p.delta[ridx] : 0.f;
            };
            fetch(first_qt * C::BM);
            for (int i = 0; i < n; ++i) {
                const uint32_t g = step_it + i, sb = g & 1, ph = (g >> 1) & 1;
                const int qrow0 = (first_qt + i) * C::BM;  // first query row of the step
                lse_s[lane] = nl;
                del_s[lane] = nd;
                __syncwarp();
                if (i + 1 < n) fetch(qrow0 + C::BM);
                // subtraction scheme: valid local columns are [lo, hi)
                const int hi = key_valid ? min(NC, q_len - qrow0 - c0) : 0;
                const int lo = p.causal ? max(0, j - diag - qrow0 - c0) : 0;
                const bool full = __all_sync(0xffffffffu, lo == 0 && hi == NC);
                const int rbase = qrow0 + c0 + diag - j;  // relative position of local column 0
                const float xs = softmax ? p.scale_log2 : p.scale;
                int bk = 0;
                bool cconst = true;
                if (p.bias) cconst = chunk_bucket_const(rbase + NC - 1, bk);
                const float cbias = p.bias ? bias_w[bk] : 0.f;
                cconst = __all_sync(0xffffffffu, cconst);

                if (!warp_wait(C_S_FULL + sb, ph)) { ok = false; break; }
                tc_fence_after();
                float pv[NC];
                {
                    uint32_t (&rr)[NC] = *reinterpret_cast<uint32_t(*)[NC]>(pv);
                    tmem_ld32(tmem + lane_base + C::kTmS + sb * 64u + uint32_t(c0), rr);
                    tmem_ld_wait(rr);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C_S_EMPTY + sb));

                // P^T = exp2(xs * s + bias - lse) (softmax) or act(scale * s + bias):
                // packed FMA with the per-column addend (bias - lse) precomputed.
                if (!warp_wait(C_PT_EMPTY, (g & 1) ^ 1)) { ok = false; break; }
                if (softmax) {
                    float lv[NC];
#pragma unroll
                    for (int c = 0; c < NC; c += 4) {
                        const float4 q4 = *reinterpret_cast<const float4*>(lse_s + c);
                        lv[c] = q4.x;
                        lv[c + 1] = q4.y;
                        lv[c + 2] = q4.z;
                        lv[c + 3] = q4.w;
                    }
                    const float2 xs2 = make_float2(xs, xs);
                    if (cconst) {
#pragma unroll
                        for (int c = 0; c < NC; c += 2) {
                            const float2 e = fma2(make_float2(pv[c], pv[c + 1]), xs2,
                                                  make_float2(cbias - lv[c], cbias - lv[c + 1]));
                            pv[c] = ex2_approx(e.x);
                            pv[c + 1] = ex2_approx(e.y);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < NC; ++c)
                            pv[c] = ex2_approx(fmaf(pv[c], xs, bias_w[relpos_bucket(rbase + c)] - lv[c]));
                    }
                    if (!full) {
#pragma unroll
                        for (int c = 0; c < NC; ++c) pv[c] = (c >= lo && c < hi) ? pv[c] : 0.f;
                    }
                    write_ptile_half<T>(sPt, r, cw, pv);
                } else {
                    if (cconst) {
#pragma unroll
                        for (int c = 0; c < NC; ++c) pv[c] = fmaf(pv[c], xs, cbias);
                    } else {
#pragma unroll
                        for (int c = 0; c < NC; ++c) pv[c] = fmaf(pv[c], xs, bias_w[relpos_bucket(rbase + c)]);
                    }
                    float pa[NC];
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        const float a = gdpa_act(gelu, pv[c]);
                        pa[c] = (full || (c >= lo && c < hi)) ? a : 0.f;
                    }
                    write_ptile_half<T>(sPt, r, cw, pa);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C_PT_FULL));

                if (!warp_wait(C_DP_FULL, g & 1)) { ok = false; break; }
                tc_fence_after();
                float dp[NC];
                {
                    uint32_t (&rr)[NC] = *reinterpret_cast<uint32_t(*)[NC]>(dp);
                    tmem_ld32(tmem + lane_base + C::kTmDP + uint32_t(c0), rr);
                    tmem_ld_wait(rr);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C_DP_EMPTY));
                if (softmax) {
                    // dS^T = P^T (dP^T - Delta), packed
#pragma unroll
                    for (int c = 0; c < NC; c += 4) {
                        const float4 d4 = *reinterpret_cast<const float4*>(del_s + c);
                        const float2 a = mul2(make_float2(pv[c], pv[c + 1]),
                                              add2(make_float2(dp[c], dp[c + 1]), make_float2(-d4.x, -d4.y)));
                        const float2 b2 = mul2(make_float2(pv[c + 2], pv[c + 3]),
                                               add2(make_float2(dp[c + 2], dp[c + 3]), make_float2(-d4.z, -d4.w)));
                        dp[c] = a.x;
                        dp[c + 1] = a.y;
                        dp[c + 2] = b2.x;
                        dp[c + 3] = b2.y;
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        float a, da;
                        gdpa_act_grad(gelu, pv[c], a, da);
                        dp[c] = (full || (c >= lo && c < hi)) ? da * dp[c] : 0.f;
                    }
                }
                if (!warp_wait(C_DS_EMPTY, (g & 1) ^ 1)) { ok = false; break; }
                write_ptile_half<T>(sDSt, r, cw, dp);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C_DS_FULL));
            }
            step_it += n;
        }
        if (!ok) fail();
    } else {
        // ------------------------------------------------------------ dQ reduction, dK/dV epilogue
        const int wq = warp - C::kDqWarp0;
        const int r = wq * 32 + lane;  // TMEM lane: head-dim index for dQ^T, key row for dK/dV
        const uint32_t lane_base = uint32_t(wq * 32) << 16;
        uint32_t step_it = 0, item_it = 0;
        bool ok = true;
        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 w = p.items[it];
            const int n = w.w, b = w.x, h = w.y, nt = w.z;
            const int q0 = p.q_off[b], q_len = p.q_off[b + 1] - q0;
            const int kv0 = p.kv_off[b], kv_len = p.kv_off[b + 1] - kv0;
            const int first_qt = (q_len + C::BM - 1) / C::BM - n;
            const int j = nt * C::BN + r;
            const size_t krow = (size_t(kv0) + size_t(j)) * size_t(p.H) + size_t(h);
            if (n == 0) {
                if (j < kv_len) {
                    float z[D];
#pragma unroll
                    for (int d = 0; d < D; ++d) z[d] = 0.f;
                    store_vec<T>(reinterpret_cast<T*>(p.dK) + krow * D, z, D, 1.f);
                    store_vec<T>(reinterpret_cast<T*>(p.dV) + krow * D, z, D, 1.f);
                }
                continue;
            }
            for (int i = 0; i < n; ++i) {
                const uint32_t g = step_it + i;
                const int qrow0 = (first_qt + i) * C::BM;
                if (!warp_wait(C_DQ_FULL, g & 1)) { ok = false; break; }
                tc_fence_after();
                float acc[C::BM];
                {
                    uint32_t rr[C::BM / 32][32];
#pragma unroll
                    for (int c = 0; c < C::BM / 32; ++c) tmem_ld32(tmem + lane_base + C::kTmDQ + c * 32u, rr[c]);
#pragma unroll
                    for (int c = 0; c < C::BM / 32; ++c) tmem_ld_wait(rr[c]);
#pragma unroll
                    for (int c = 0; c < C::BM / 32; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e) acc[c * 32 + e] = __uint_as_float(rr[c][e]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C_DQ_EMPTY));
                if (r < D) {
                    const int nrows = min(C::BM, q_len - qrow0);
                    float* dst = p.dq_acc + ((size_t(q0) + size_t(qrow0)) * size_t(p.H) + size_t(h)) * D + r;
                    const size_t stride = size_t(p.H) * D;
#pragma unroll
                    for (int c = 0; c < C::BM; ++c)
                        if (c < nrows) atomicAdd(dst + size_t(c) * stride, acc[c]);
                }
            }
            if (!ok) break;
            if (!warp_wait(C_ACC_FULL, item_it & 1)) { ok = false; break; }
            tc_fence_after();
            {
                const bool kv_ok = j < kv_len;
                T* dv_row = reinterpret_cast<T*>(p.dV) + krow * D;
                T* dk_row = reinterpret_cast<T*>(p.dK) + krow * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t rr[32];
                    float v[32];
                    tmem_ld32(tmem + lane_base + C::kTmDV + c * 32u, rr);
                    tmem_ld_wait(rr);
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(rr[e]);
                    if (kv_ok) store_vec<T>(dv_row + c * 32, v, 32, 1.f);
                    tmem_ld32(tmem + lane_base + C::kTmDK + c * 32u, rr);
                    tmem_ld_wait(rr);
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(rr[e]);
                    if (kv_ok) store_vec<T>(dk_row + c * 32, v, 32, p.scale);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C_ACC_EMPTY));
            step_it += n;
            ++item_it;
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kMmaWarp) tmem_dealloc(tmem, C::kTmemCols);
}

// Delta_i = sum_d dO_id * O_id for each (row, head); one 8-lane group per row.
template <typename TO, typename T, int D>
__global__ void jfa_bwd_pre_kernel(const TO* __restrict__ O, const T* __restrict__ dO, float* __restrict__ delta,
                                   int64_t rows) {
    constexpr int kLanes = 8;
    constexpr int kPer = D / kLanes;
    const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t row = gid / kLanes;
    const int sub = int(gid % kLanes);
    float acc = 0.f;
    if (row < rows) {
        const TO* o = O + row * D + sub * kPer;
        const T* g = dO + row * D + sub * kPer;
#pragma unroll
        for (int k = 0; k < kPer; ++k) acc += float(o[k]) * float(g[k]);
    }
#pragma unroll
    for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && sub == 0) delta[row] = acc;
}

// dQ = scale * accumulator, converted.
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

template <typename T, int D>
cudaError_t launch_main_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const CUtensorMap& tmdO, const BwdParams& p, int grid, cudaStream_t st) {
    using C = BwdCfg<T, D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(jfa_bwd_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    jfa_bwd_kernel<T, D><<<grid, C::kThreads, C::kSmemBytes, st>>>(tmQ, tmK, tmV, tmdO, p);
    return cudaGetLastError();
}

template <typename TO, typename T, int D>
cudaError_t launch_pre_t(const void* O, const void* dO, float* delta, int64_t rows, cudaStream_t st) {
    const int64_t threads = rows * 8;
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
    cudaError_t e = cudaMemsetAsync(dq_acc, 0, size_t(rows) * size_t(D) * 4, st);
    if (e != cudaSuccess || mode != JFA_SOFTMAX) return e;
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
    if (dtype == JFA_BF16 && D == 128) return launch_main_t<__nv_bfloat16, 128>(tmQ, tmK, tmV, tmdO, p, grid, st);
    if (dtype == JFA_BF16 && D == 64) return launch_main_t<__nv_bfloat16, 64>(tmQ, tmK, tmV, tmdO, p, grid, st);
    return cudaErrorInvalidValue;
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
