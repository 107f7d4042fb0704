// Forward kernel: jagged flash attention / GDPA on sm_103a.
//
// Computes, per (sequence, head, 128-row query tile) work item, the attention of
// the GEM articles' "Jagged Sequence Flash Attention" (aihot.vn, that section):
// directly on packed values plus offsets, never materialising a padded tensor.
// Masking follows the "subtraction scheme" the kerneldigest.dev summary names
// (section "Arquitectura del Sistema"): for a key tile starting at column c0 the
// kernel subtracts c0 from the sequence's key length (and from the row's causal
// limit) and masks columns at or beyond what remains -- no mask tensor, no padding.
// The GDPA mode (aihot.vn, "Generalized Dot-Product Attention (GDPA)") swaps the
// online softmax for an elementwise GELU/SiLU with no normalisation.
//
// CTA = 6 warps, persistent, one CTA per SM, work list from the LPT planner:
//   warps 0-3  softmax/activation + correction + epilogue; thread t owns query row t
//              of the tile and TMEM lane t;
//   warp 4     TMA producer (Q once per item; K_j, V_j through 2-stage rings);
//   warp 5     tcgen05.mma issuer and TMEM owner.
// TMEM (512 columns): S double buffer at columns [0,128) and [128,256), O at
// [256, 256+D).  The MMA warp computes S_{j+1} = Q K_{j+1}^T while the softmax
// warps turn S_j into P_j; P_j goes to shared memory (bf16, or fp32 read as TF32)
// in the 128-byte-swizzled K-major layout, and O += P_j V_j runs with V as an
// MN-major operand.
#include "jfa_internal.h"
#include "ptx.cuh"
#include "tilemath.cuh"

namespace jfa {

template <typename T>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kBytes = 2;
    static constexpr uint32_t kFmt = kFmtBF16;
    static constexpr int kUmmaK = 16;  // K elements per tcgen05.mma (32 bytes)
    static constexpr CUtensorMapDataType kTmaType = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
};
template <>
struct Elem<float> {
    static constexpr int kBytes = 4;
    static constexpr uint32_t kFmt = kFmtTF32;
    static constexpr int kUmmaK = 8;
    static constexpr CUtensorMapDataType kTmaType = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
};

template <typename T, int D>
struct FwdCfg {
    static constexpr int BM = kFwdBM, BN = kFwdBN;
    static constexpr int E = Elem<T>::kBytes;
    static constexpr int kRowBytes = D * E;
    static_assert(kRowBytes % 128 == 0 && kRowBytes <= 256, "head row must be 128 or 256 bytes");
    static constexpr int kCB = kRowBytes / 128;  // 128-byte column blocks of a tile
    static constexpr int kBoxCols = 128 / E;     // elements per 128-byte box row
    static constexpr int kQBytes = BM * kRowBytes;
    static constexpr int kKVBytes = BN * kRowBytes;
    static constexpr int kPRowBytes = BN * E;
    static constexpr int kPBytes = BM * kPRowBytes;
    static constexpr int kStages = 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + kStages * kKVBytes;
    static constexpr int kOffP = kOffV + kStages * kKVBytes;
    static constexpr int kOffP2 = kOffP + kPBytes;  // GDPA: P - bf16(P), second PV product
    static constexpr int kOffBar = kOffP2 + kPBytes;
    static constexpr int kNumBars = 20;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kMiscBytes = 16 + 2 * 4 * 32 * 4;  // tmem slot, abort flag, bias tables
    static constexpr int kSmemNeed = kOffMisc + kMiscBytes + 1024;
    // At least 120 KB so that exactly one CTA fits on an SM: the CTA allocates all
    // 512 TMEM columns.
    static constexpr int kSmemBytes = kSmemNeed > 120 * 1024 ? kSmemNeed : 120 * 1024;
    static constexpr int kUmmaK = Elem<T>::kUmmaK;
    static constexpr int kQKSteps = D / kUmmaK;
    static constexpr int kPVSteps = BN / kUmmaK;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTmemO = 256;
    static constexpr uint32_t kIdescQK = make_idesc(Elem<T>::kFmt, BM, BN, false, false);
    static constexpr uint32_t kIdescPV = make_idesc(Elem<T>::kFmt, BM, D, false, true);
    static constexpr int kThreads = 192;
};

// Barrier slots.
enum {
    B_Q_FULL = 0,
    B_Q_EMPTY = 1,
    B_K_FULL = 2,   // +stage
    B_K_EMPTY = 4,  // +stage
    B_V_FULL = 6,
    B_V_EMPTY = 8,
    B_S_FULL = 10,   // +buffer
    B_S_EMPTY = 12,  // +buffer
    B_P_FULL = 14,
    B_O_FULL = 15,
    B_O_EMPTY = 16,
    B_DRAIN = 17,
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

template <typename T, int D, typename OT>
__global__ void __launch_bounds__(192, 1)
    jfa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using C = FwdCfg<T, D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::kOffQ, sK = sbase + C::kOffK, sV = sbase + C::kOffV,
                   sP = sbase + C::kOffP, sP2 = sbase + C::kOffP2;
    const bool gdpa = p.mode != JFA_SOFTMAX;
    auto bar = [&](int i) -> uint32_t { return sbase + C::kOffBar + 8u * uint32_t(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
    float* bias_s = reinterpret_cast<float*>(smem + C::kOffMisc + 16);

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
            mbar_init(bar(B_S_EMPTY + s), 4);
        }
        mbar_init(bar(B_P_FULL), 4);
        mbar_init(bar(B_O_FULL), 1);
        mbar_init(bar(B_O_EMPTY), 4);
        mbar_init(bar(B_DRAIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
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

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t kv_it = 0, item_it = 0;
            bool ok = true;
            for (int it = it_begin; it < it_end && ok; ++it) {
                const int4 w = p.items[it];
                const int n = w.w;
                if (n == 0) continue;
                const int b = w.x, h = w.y, mt = w.z;
                const int q0 = p.q_off[b], kv0 = p.kv_off[b];
                if (!mbar_wait_bounded(bar(B_Q_EMPTY), (item_it & 1) ^ 1, abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(bar(B_Q_FULL), C::kQBytes);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb)
                    tma_load_2d(sQ + cb * C::BM * 128, &tmQ, bar(B_Q_FULL), h * D + cb * C::kBoxCols,
                                q0 + mt * C::BM);
                ++item_it;
                for (int j = 0; j < n; ++j, ++kv_it) {
                    const uint32_t st = kv_it & 1, ph = (kv_it >> 1) & 1;
                    const int y = kv0 + j * C::BN;
                    if (!mbar_wait_bounded(bar(B_K_EMPTY + st), ph ^ 1, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(bar(B_K_FULL + st), C::kKVBytes);
#pragma unroll
                    for (int cb = 0; cb < C::kCB; ++cb)
                        tma_load_2d(sK + st * C::kKVBytes + cb * C::BN * 128, &tmK, bar(B_K_FULL + st),
                                    h * D + cb * C::kBoxCols, y);
                    if (!mbar_wait_bounded(bar(B_V_EMPTY + st), ph ^ 1, abort_flag)) { ok = false; break; }
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
            for (uint32_t s = 0; s < 2; ++s) {
                if (kv_it > s) {
                    const uint32_t last = ((kv_it - 1 - s) / 2) * 2 + s;  // last index with stage s
                    mbar_wait_bounded(bar(B_K_FULL + s), (last >> 1) & 1, nullptr);
                    mbar_wait_bounded(bar(B_V_FULL + s), (last >> 1) & 1, nullptr);
                }
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t kv_it = 0, item_it = 0, pv_it = 0;
            bool ok = true;
            for (int it = it_begin; it < it_end && ok; ++it) {
                const int n = p.items[it].w;
                if (n == 0) continue;
                if (!mbar_wait_bounded(bar(B_Q_FULL), item_it & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                for (int j = 0; j <= n && ok; ++j) {
                    if (j < n) {
                        const uint32_t g = kv_it + j, st = g & 1, ph = (g >> 1) & 1;
                        if (!mbar_wait_bounded(bar(B_K_FULL + st), ph, abort_flag) ||
                            !mbar_wait_bounded(bar(B_S_EMPTY + st), ph ^ 1, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t d_tmem = tmem + st * 128u;
                        const uint32_t kbase = sK + st * C::kKVBytes;
#pragma unroll
                        for (int s = 0; s < C::kQKSteps; ++s) {
                            const uint32_t koff = (s * 32) & 127;  // bytes into the 128-byte row
                            const uint32_t cb = (s * 32) >> 7;     // 128-byte column block
                            const uint64_t a = make_sdesc_sw128(sQ + cb * C::BM * 128 + koff, 16, 1024);
                            const uint64_t bd = make_sdesc_sw128(kbase + cb * C::BN * 128 + koff, 16, 1024);
                            mma_f16_ss(d_tmem, a, bd, C::kIdescQK, s > 0);
                        }
                        tc_commit(bar(B_S_FULL + st));
                        tc_commit(bar(B_K_EMPTY + st));
                        if (j == n - 1) tc_commit(bar(B_Q_EMPTY));
                    }
                    if (j > 0) {
                        const int jj = j - 1;
                        const uint32_t g = kv_it + jj, st = g & 1, ph = (g >> 1) & 1;
                        if (!mbar_wait_bounded(bar(B_P_FULL), pv_it & 1, abort_flag) ||
                            !mbar_wait_bounded(bar(B_V_FULL + st), ph, abort_flag)) { ok = false; break; }
                        if (jj == 0 && !mbar_wait_bounded(bar(B_O_EMPTY), (item_it & 1) ^ 1, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t vbase = sV + st * C::kKVBytes;
#pragma unroll
                        for (int s = 0; s < C::kPVSteps; ++s) {
                            const uint32_t koff = (s * 32) & 127;
                            const uint32_t cb = (s * 32) >> 7;
                            const uint64_t a = make_sdesc_sw128(sP + cb * C::BM * 128 + koff, 16, 1024);
                            const uint64_t bd = make_sdesc_sw128(vbase + s * C::kUmmaK * 128, C::BN * 128, 1024);
                            mma_f16_ss(tmem + C::kTmemO, a, bd, C::kIdescPV, (jj > 0 || s > 0));
                        }
                        if (gdpa) {  // O += (P - bf16(P)) V: P to ~16 significant bits
#pragma unroll
                            for (int s = 0; s < C::kPVSteps; ++s) {
                                const uint32_t koff = (s * 32) & 127;
                                const uint32_t cb = (s * 32) >> 7;
                                const uint64_t a = make_sdesc_sw128(sP2 + cb * C::BM * 128 + koff, 16, 1024);
                                const uint64_t bd = make_sdesc_sw128(vbase + s * C::kUmmaK * 128, C::BN * 128, 1024);
                                mma_f16_ss(tmem + C::kTmemO, a, bd, C::kIdescPV, 1u);
                            }
                        }
                        tc_commit(bar(B_O_FULL));
                        tc_commit(bar(B_V_EMPTY + st));
                        ++pv_it;
                    }
                }
                kv_it += n;
                ++item_it;
            }
            if (!ok) fail();
            // Drain all issued MMAs before TMEM is released.
            tc_commit(bar(B_DRAIN));
            mbar_wait_bounded(bar(B_DRAIN), 0, nullptr);
        }
    } else {
        // ------------------------------------------------------------ softmax / epilogue
        const int t = threadIdx.x;  // query row in the tile == TMEM lane
        const uint32_t lane_base = uint32_t(warp * 32) << 16;
        const bool softmax = p.mode == JFA_SOFTMAX;
        uint32_t kv_it = 0, item_it = 0, pv_wait = 0;
        bool ok = true;
        for (int it = it_begin; it < it_end && ok; ++it) {
            const int4 w = p.items[it];
            const int n = w.w, b = w.x, h = w.y, mt = w.z;
            const int q0 = p.q_off[b], q_len = p.q_off[b + 1] - q0;
            const int kv_len = p.kv_off[b + 1] - p.kv_off[b];
            const int row = mt * C::BM + t;
            const bool row_valid = row < q_len;
            const int diag = kv_len - q_len;
            // Each warp keeps its own copy of the head's bias row (log2 units for
            // softmax), double-buffered by item parity, so no cross-warp barrier.
            float* btab = bias_s + ((item_it & 1) * 4 + warp) * 32;
            if (p.bias) {
                btab[lane] = p.bias[h * 32 + lane] * (softmax ? 1.4426950408889634f : 1.0f);
                __syncwarp();
            }
            const size_t orow = (size_t(q0) + size_t(row)) * size_t(p.H) + size_t(h);
            if (n == 0) {
                if (row_valid) {
                    float z[D];
#pragma unroll
                    for (int d = 0; d < D; ++d) z[d] = 0.f;
                    store_row<OT>(reinterpret_cast<OT*>(p.O) + orow * D, z, D);
                    if (p.lse) p.lse[orow] = -INFINITY;
                }
                ++item_it;
                continue;
            }
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < n; ++j) {
                const uint32_t g = kv_it + j, sb = g & 1, ph = (g >> 1) & 1;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar(B_S_FULL + sb), ph, abort_flag))) { ok = false; break; }
                tc_fence_after();
                float x[C::BN];
                {
                    uint32_t r[C::BN / 32][32];
#pragma unroll
                    for (int c = 0; c < C::BN / 32; ++c) tmem_ld32(tmem + lane_base + sb * 128u + c * 32u, r[c]);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < C::BN / 32; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(r[c][i]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_S_EMPTY + sb));

                const int col0 = j * C::BN;
                int lim = kv_len - col0;  // subtraction scheme: columns >= lim are masked
                if (p.causal) lim = min(lim, row + diag + 1 - col0);
                const int rbase = row + diag - col0;  // relative position of column 0
                const bool full = __all_sync(0xffffffffu, lim >= C::BN);
                const float xs = softmax ? p.scale_log2 : p.scale;
                // x = scale * s + bias: one constant per 32-column chunk when the whole
                // chunk sits in one bucket (warp-uniform), else per element.
                bool cconst = true;
                float cb[C::BN / 32];
#pragma unroll
                for (int k = 0; k < C::BN / 32; ++k) {
                    int bk = 0;
                    if (p.bias) cconst &= chunk_bucket_const(rbase - 32 * k, bk);
                    cb[k] = p.bias ? btab[bk] : 0.f;
                }
                if (__all_sync(0xffffffffu, cconst)) {
#pragma unroll
                    for (int c = 0; c < C::BN; ++c) x[c] = fmaf(x[c], xs, cb[c >> 5]);
                } else {
#pragma unroll
                    for (int c = 0; c < C::BN; ++c) x[c] = fmaf(x[c], xs, btab[relpos_bucket(rbase - c)]);
                }
                bool need_rescale = false;
                float alpha = 1.f;
                if (softmax) {
                    if (!full) {
#pragma unroll
                        for (int c = 0; c < C::BN; ++c) x[c] = (c < lim) ? x[c] : -INFINITY;
                    }
                    float mx8[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) mx8[k] = x[k];
#pragma unroll
                    for (int c = 8; c < C::BN; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], x[c]);
                    const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                           fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                    // Lazy rescaling: keep the running max unless it grows by more
                    // than 2^8; both O and l use the same stale max, so the final
                    // O / l is unchanged.
                    float m_new = m;
                    if (mx > m + 8.f) m_new = mx;
                    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                    alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_use);
                    if (m_new != m) need_rescale = (j > 0);
                    m = m_new;
                    float rs8[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) rs8[k] = 0.f;
#pragma unroll
                    for (int c = 0; c < C::BN; ++c) {
                        x[c] = ex2_approx(x[c] - m_use);
                        rs8[c & 7] += x[c];
                    }
                    l = l * alpha + (((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7])));
                } else {
                    const bool gelu = p.mode == JFA_GDPA_GELU_TANH;
#pragma unroll
                    for (int c = 0; c < C::BN; ++c) {
                        const float a = gdpa_act(gelu, x[c]);
                        x[c] = (full || c < lim) ? a : 0.f;
                    }
                }
                // P buffer and O are free once the previous P V product is done.
                if (j > 0) {
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar(B_O_FULL), pv_wait & 1, abort_flag))) { ok = false; break; }
                    ++pv_wait;
                    tc_fence_after();
                }
                if (__any_sync(0xffffffffu, need_rescale)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        const uint32_t ta = tmem + lane_base + C::kTmemO + c * 32u;
                        tmem_ld32(ta, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st32(ta, r);
                    }
                    tmem_st_wait();
                }
                // P row -> shared memory, 128-byte swizzled K-major (bf16).  GDPA also
                // writes the rounding remainder P - bf16(P) for a second P V product.
#pragma unroll
                for (int k = 0; k < C::BN / 8; ++k) {
                    const uint32_t off = (k >> 3) * (C::BM * 128) + sw128_offset(t, k & 7);
                    uint32_t u[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) u[e] = pack_bf16x2(x[8 * k + 2 * e], x[8 * k + 2 * e + 1]);
                    st_shared_v4(sP + off, u[0], u[1], u[2], u[3]);
                    if (gdpa) {
                        uint32_t v[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float lo0 = x[8 * k + 2 * e] - __uint_as_float(u[e] << 16);
                            const float lo1 = x[8 * k + 2 * e + 1] - __uint_as_float(u[e] & 0xffff0000u);
                            v[e] = pack_bf16x2(lo0, lo1);
                        }
                        st_shared_v4(sP2 + off, v[0], v[1], v[2], v[3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_P_FULL));
            }
            if (!ok) break;
            // Epilogue: wait for the last P V product, read O, release it.
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar(B_O_FULL), pv_wait & 1, abort_flag))) { ok = false; break; }
            ++pv_wait;
            tc_fence_after();
            {
                const float inv = (softmax && l > 0.f) ? 1.f / l : (softmax ? 0.f : 1.f);
                OT* orow_p = reinterpret_cast<OT*>(p.O) + orow * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    float v[32];
                    tmem_ld32(tmem + lane_base + C::kTmemO + c * 32u, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * inv;
                    if (row_valid) store_row<OT>(orow_p + c * 32, v, 32);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_O_EMPTY));
            if (row_valid && softmax && p.lse)
                p.lse[orow] = l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
            kv_it += n;
            ++item_it;
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, C::kTmemCols);
}

template <typename T, int D, typename OT>
static cudaError_t launch_fwd_t(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                const FwdParams& p, int grid, cudaStream_t st) {
    using C = FwdCfg<T, D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(jfa_fwd_kernel<T, D, OT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    jfa_fwd_kernel<T, D, OT><<<grid, C::kThreads, C::kSmemBytes, st>>>(tmQ, tmK, tmV, p);
    return cudaGetLastError();
}

cudaError_t launch_fwd(int dtype, int o_dtype, int D, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const FwdParams& p, int grid, cudaStream_t st) {
    using bf16 = __nv_bfloat16;
    if (dtype != JFA_BF16) return cudaErrorInvalidValue;
    if (D == 128 && o_dtype == JFA_BF16) return launch_fwd_t<bf16, 128, bf16>(tmQ, tmK, tmV, p, grid, st);
    if (D == 128 && o_dtype == JFA_F32) return launch_fwd_t<bf16, 128, float>(tmQ, tmK, tmV, p, grid, st);
    if (D == 64 && o_dtype == JFA_BF16) return launch_fwd_t<bf16, 64, bf16>(tmQ, tmK, tmV, p, grid, st);
    if (D == 64 && o_dtype == JFA_F32) return launch_fwd_t<bf16, 64, float>(tmQ, tmK, tmV, p, grid, st);
    return cudaErrorInvalidValue;
}

bool supported(int dtype, int D) {
    return (dtype == JFA_BF16 && (D == 64 || D == 128)) || (dtype == JFA_F32 && (D == 32 || D == 64));
}

}  // namespace jfa
