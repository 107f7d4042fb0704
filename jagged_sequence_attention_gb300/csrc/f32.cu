// fp32 path: jagged attention forward and backward on the CUDA cores in fp32.
//
// Same operation, work items and conventions as the bf16 tensor-core kernels (the
// GEM articles' jagged flash attention and GDPA), for float inputs.  The tensor
// cores' fp32-input format (TF32) drops 13 mantissa bits and tcgen05 takes TF32
// operands only K-major, while V, dO and Q enter the products MN-major; for the
// float element type the kernels therefore use plain fp32 FMA, one thread per
// row, with K/V (forward) or Q/dO (backward) tiles staged in shared memory.
#include "jfa_internal.h"

#include <math.h>

namespace jfa {

namespace {

constexpr int kF32Rows = 128;   // threads per CTA = rows of the outer tile
constexpr int kF32Inner = 64;   // rows of the staged inner tile (forward)
constexpr int kF32InnerB = 32;  // rows of the staged inner tile (backward)

__device__ __forceinline__ int bucket_f32(int r) {
    r = r < 0 ? -r : r;
    if (r >= 46340) return 31;
    const uint32_t v = uint32_t(r + 1) * uint32_t(r + 1);
    return 31 - __clz(v);
}

__device__ __forceinline__ float act_f32(int mode, float x) {
    if (mode == JFA_GDPA_GELU_TANH) {
        const float c = 0.7978845608028654f;
        return 0.5f * x * (1.f + tanhf(c * (x + 0.044715f * x * x * x)));
    }
    return x / (1.f + expf(-x));
}

__device__ __forceinline__ float act_grad_f32(int mode, float x) {
    if (mode == JFA_GDPA_GELU_TANH) {
        const float c = 0.7978845608028654f;
        const float t = tanhf(c * (x + 0.044715f * x * x * x));
        return 0.5f * (1.f + t) + 0.5f * x * (1.f - t * t) * c * (1.f + 3.f * 0.044715f * x * x);
    }
    const float sg = 1.f / (1.f + expf(-x));
    return sg * (1.f + x * (1.f - sg));
}

// Two CTAs per forward work item (a pair of 128-row query tiles); thread = query row.
template <int D>
__global__ void __launch_bounds__(kF32Rows) jfa_fwd_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                                                                const float* __restrict__ V, const FwdParams p) {
    __shared__ float sK[kF32Inner][D];
    __shared__ float sV[kF32Inner][D];
    __shared__ float sB[32];
    const int4 w = p.items[blockIdx.x >> 1];
    if (!fwd_item_ok(w, p, p.window)) {  // not an item of this plan (the whole CTA returns)
        if (threadIdx.x == 0 && (blockIdx.x & 1) == 0) atomicOr(p.status, kStatusBounds);
        return;
    }
    const int b = w.x, h = w.y, mt = 2 * w.z + int(blockIdx.x & 1);
    const int q0 = p.q_off[b], q_len = p.q_off[b + 1] - q0;
    const int kb = p.kv_map ? p.kv_map[b] : b;  // key/value sequence (shared: the user)
    const int k0 = p.kv_off[kb], kv_len = p.kv_off[kb + 1] - k0;
    if (mt * kF32Rows >= q_len) return;  // second tile of a short last pair (uniform exit)
    int kf, n_tiles;  // key tiles [kf, kf + n_tiles)
    key_tile_range(q_len, kv_len, mt, p.causal, p.window, kf, n_tiles);
    const int t = threadIdx.x, row = mt * kF32Rows + t;
    const bool valid = row < q_len;
    const int diag = kv_len - q_len;
    const bool softmax = p.mode == JFA_SOFTMAX;
    if (t < 32) sB[t] = p.bias ? p.bias[h * 32 + t] : 0.f;
    float q[D], o[D];
    const size_t rq = (size_t(q0) + size_t(valid ? row : 0)) * p.H + h;
#pragma unroll
    for (int d = 0; d < D; ++d) {
        q[d] = valid ? Q[rq * D + d] : 0.f;
        o[d] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    // keys of the tile's range (causal limit of its last row, window start of its first
    // row, in 128-key units), staged 64 at a time
    const int kv_end = min(kv_len, (kf + n_tiles) * kFwdBN);
    const int lim = p.causal ? min(kv_len, row + diag + 1) : kv_len;  // keys [lo, lim) allowed
    const int lo = p.window >= 0 ? row + diag - p.window : 0;
    // dense per-pair bias of this row (read only at allowed keys)
    const float* drow = p.dense ? p.dense + size_t(h) * size_t(p.n_pairs) + size_t(p.pair_off[b]) +
                                      size_t(valid ? row : 0) * size_t(kv_len)
                                : nullptr;
    for (int c0 = kf * kFwdBN; c0 < kv_end; c0 += kF32Inner) {
        __syncthreads();
        for (int e = t; e < kF32Inner * D; e += kF32Rows) {
            const int r = e / D, d = e % D;
            const bool in = c0 + r < kv_len;
            const size_t rk = (size_t(k0) + size_t(in ? c0 + r : 0)) * p.H + h;
            sK[r][d] = in ? K[rk * D + d] : 0.f;
            sV[r][d] = in ? V[rk * D + d] : 0.f;
        }
        __syncthreads();
        float s[kF32Inner];
        float mx = -INFINITY;
#pragma unroll 4
        for (int j = 0; j < kF32Inner; ++j) {
            float acc = 0.f;
#pragma unroll
            for (int d = 0; d < D; ++d) acc = fmaf(q[d], sK[j][d], acc);
            float x = acc * p.scale;
            if (p.bias) x += sB[bucket_f32(row + diag - (c0 + j))];
            const bool ok = valid && (c0 + j) < lim && (c0 + j) >= lo;
            if (drow && ok) x += __ldg(drow + c0 + j);
            s[j] = ok ? x : -INFINITY;
            mx = fmaxf(mx, s[j]);
        }
        if (softmax) {
            const float m_new = fmaxf(m, mx);
            if (m_new == -INFINITY) continue;
            const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
            l *= alpha;
#pragma unroll
            for (int d = 0; d < D; ++d) o[d] *= alpha;
            for (int j = 0; j < kF32Inner; ++j) {
                const float pj = expf(s[j] - m_new);
                l += pj;
#pragma unroll
                for (int d = 0; d < D; ++d) o[d] = fmaf(pj, sV[j][d], o[d]);
            }
            m = m_new;
        } else {
            for (int j = 0; j < kF32Inner; ++j) {
                if (s[j] == -INFINITY) continue;
                const float a = act_f32(p.mode, s[j]);
#pragma unroll
                for (int d = 0; d < D; ++d) o[d] = fmaf(a, sV[j][d], o[d]);
            }
        }
    }
    if (!valid) return;
    float* O = static_cast<float*>(p.O) + rq * D;
    const float inv = softmax ? (l > 0.f ? 1.f / l : 0.f) : 1.f;
#pragma unroll
    for (int d = 0; d < D; ++d) O[d] = o[d] * inv;
    if (softmax && p.lse) p.lse[rq] = l > 0.f ? m + logf(l) : -INFINITY;
}

// One CTA per backward work item (key tile of 128 rows); thread = key row.  Query
// rows stream through shared memory kF32InnerB at a time; dS for the chunk is kept in
// shared memory so that dQ is reduced over the CTA's keys before one atomic add per
// (query row, d).  With p.dbias_part set, the chunk's dS is also summed along its
// diagonals (one relative position each) and the diagonals by bucket, in a fixed
// order, into the item's partial table gradient p.dbias_part[item][32].
template <int D>
__global__ void __launch_bounds__(kF32Rows) jfa_bwd_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                                                                const float* __restrict__ V, const float* __restrict__ dO,
                                                                const BwdParams p) {
    __shared__ float sQ[kF32InnerB][D];
    __shared__ float sdO[kF32InnerB][D];
    __shared__ float sDS[kF32InnerB][kF32Rows + 1];
    __shared__ float sL[kF32InnerB], sDel[kF32InnerB];
    __shared__ float sB[32];
    constexpr int kDiags = kF32InnerB + kF32Rows - 1;  // diagonals i - t of a chunk
    __shared__ float sDiag[kDiags];
    __shared__ float sDB[32];  // the item's table gradient, bucket t owned by thread t
    const int4 w = p.items[blockIdx.x];
    if (!kv_item_ok(w, p, p.steps != nullptr)) {  // not an item of this plan (the whole CTA returns)
        if (threadIdx.x == 0) atomicOr(p.status, kStatusBounds);
        return;
    }
    // b: the key/value sequence of the item (shared key/value: the user)
    const int b = w.x, h = w.y, nt = w.z, n = w.w;
    const int k0 = p.kv_off[b], kv_len = p.kv_off[b + 1] - k0;
    const int t = threadIdx.x, j = nt * kBwdBN + t;
    const bool kvalid = j < kv_len;
    const bool softmax = p.mode == JFA_SOFTMAX;
    if (t < 32) sB[t] = p.bias ? p.bias[h * 32 + t] : 0.f;
    if (t < 32) sDB[t] = 0.f;
    const size_t rk = (size_t(k0) + size_t(kvalid ? j : 0)) * p.H + h;
    float k[D], v[D], dk[D], dv[D];
#pragma unroll
    for (int d = 0; d < D; ++d) {
        k[d] = kvalid ? K[rk * D + d] : 0.f;
        v[d] = kvalid ? V[rk * D + d] : 0.f;
        dk[d] = 0.f;
        dv[d] = 0.f;
    }
    const int n_keys = min(kBwdBN, kv_len - nt * kBwdBN);
    // Query rows that see this key tile, as segments of one query sequence each: the
    // sequence's own tile range, or (shared key/value) one 128-row query tile per step
    // of every query set of the user.
    const int n_seg = p.steps ? n : 1;
    const int s0 = p.steps ? p.step_off[p.ktile_off[b] + nt] : 0;
    for (int sg = 0; sg < n_seg; ++sg) {
        int qb, row_begin, row_end;
        if (p.steps) {
            const int2 st = p.steps[s0 + sg];
            qb = st.x;
            row_begin = st.y * kBwdBM;
            row_end = min(p.q_off[qb + 1] - p.q_off[qb], row_begin + kBwdBM);
        } else {
            int first_qt, nq;  // query tiles [first_qt, first_qt + n) see this key tile
            qb = b;
            query_tile_range(p.q_off[b + 1] - p.q_off[b], kv_len, nt, p.causal, p.window, first_qt, nq);
            row_begin = first_qt * kBwdBM;
            row_end = min(p.q_off[b + 1] - p.q_off[b], (first_qt + n) * kBwdBM);
        }
        const int q0 = p.q_off[qb], q_len = p.q_off[qb + 1] - q0;
        const int diag = kv_len - q_len;
        // dense per-pair bias and its gradient of key j: element (query row i) at [i * kv_len]
        const size_t dcol = size_t(h) * size_t(p.n_pairs) + size_t(p.pair_off ? p.pair_off[qb] : 0) + size_t(kvalid ? j : 0);
        for (int r0 = row_begin; r0 < row_end; r0 += kF32InnerB) {
            __syncthreads();
            for (int e = t; e < kF32InnerB * D; e += kF32Rows) {
                const int r = e / D, d = e % D;
                const bool in = r0 + r < q_len;
                const size_t rq = (size_t(q0) + size_t(in ? r0 + r : 0)) * p.H + h;
                sQ[r][d] = in ? Q[rq * D + d] : 0.f;
                sdO[r][d] = in ? dO[rq * D + d] : 0.f;
            }
            if (t < kF32InnerB) {
                const bool in = r0 + t < q_len;
                const size_t rq = (size_t(q0) + size_t(in ? r0 + t : 0)) * p.H + h;
                sL[t] = (in && softmax) ? p.lse[rq] : 0.f;
                sDel[t] = (in && softmax) ? p.delta[rq] : 0.f;
            }
            __syncthreads();
            for (int i = 0; i < kF32InnerB; ++i) {
                const int row = r0 + i;
                const bool ok = kvalid && row < q_len && (!p.causal || j <= row + diag) &&
                                (p.window < 0 || j >= row + diag - p.window);
                float ds = 0.f;
                if (ok) {
                    float acc = 0.f, dp = 0.f;
    #pragma unroll
                    for (int d = 0; d < D; ++d) {
                        acc = fmaf(sQ[i][d], k[d], acc);
                        dp = fmaf(sdO[i][d], v[d], dp);
                    }
                    float x = acc * p.scale;
                    if (p.bias) x += sB[bucket_f32(row + diag - j)];
                    if (p.dense) x += __ldg(p.dense + dcol + size_t(row) * size_t(kv_len));
                    float pij;
                    if (softmax) {
                        pij = expf(x - sL[i]);
                        ds = pij * (dp - sDel[i]);
                    } else {
                        pij = act_f32(p.mode, x);
                        ds = act_grad_f32(p.mode, x) * dp;
                    }
                    if (p.ddense) p.ddense[dcol + size_t(row) * size_t(kv_len)] = ds;
    #pragma unroll
                    for (int d = 0; d < D; ++d) {
                        dv[d] = fmaf(pij, sdO[i][d], dv[d]);
                        dk[d] = fmaf(ds, sQ[i][d], dk[d]);
                    }
                }
                sDS[i][t] = ds;
            }
            __syncthreads();
            // dQ rows of this chunk: sum over the CTA's keys (K rows re-read through the
            // cache), then one atomic per element
            for (int e = t; e < kF32InnerB * D; e += kF32Rows) {
                const int i = e / D, d = e % D;
                if (r0 + i >= q_len) continue;
                float acc = 0.f;
                for (int jj = 0; jj < n_keys; ++jj)
                    acc = fmaf(sDS[i][jj], __ldg(K + ((size_t(k0) + size_t(nt * kBwdBN + jj)) * p.H + h) * D + d), acc);
                const size_t rq = (size_t(q0) + size_t(r0 + i)) * p.H + h;
                atomicAdd(p.dq_acc + rq * D + d, acc);
            }
            if (p.dbias_part) {
                // diagonal dd holds the elements with i - t = dd - (kF32Rows - 1), i ascending
                for (int dd = t; dd < kDiags; dd += kF32Rows) {
                    const int off = dd - (kF32Rows - 1);
                    const int i0 = max(0, off), i1 = min(kF32InnerB - 1, kF32Rows - 1 + off);
                    float acc = 0.f;
                    for (int i = i0; i <= i1; ++i) acc += sDS[i][i - off];
                    sDiag[dd] = acc;
                }
                __syncthreads();
                if (t < 32) {
                    // element (i, t') has relative position r0 + i + diag - (nt * 128 + t')
                    const int rel0 = r0 + diag - nt * kBwdBN - (kF32Rows - 1);
                    float acc = 0.f;
                    for (int dd = 0; dd < kDiags; ++dd)
                        if (bucket_f32(rel0 + dd) == t) acc += sDiag[dd];
                    sDB[t] += acc;
                }
            }
        }
    }
    if (p.dbias_part && t < 32) p.dbias_part[size_t(blockIdx.x) * 32 + t] = sDB[t];
    if (!kvalid) return;
    float* dK = static_cast<float*>(p.dK) + rk * D;
    float* dV = static_cast<float*>(p.dV) + rk * D;
#pragma unroll
    for (int d = 0; d < D; ++d) {
        dK[d] = dk[d] * p.scale;
        dV[d] = dv[d];
    }
}

}  // namespace

cudaError_t launch_fwd_f32(int D, const void* Q, const void* K, const void* V, const FwdParams& p, int64_t n_items,
                           cudaStream_t st) {
    if (n_items <= 0) return cudaSuccess;
    const unsigned g = unsigned(2 * n_items);
    if (D == 32)
        jfa_fwd_f32_kernel<32><<<g, kF32Rows, 0, st>>>(static_cast<const float*>(Q), static_cast<const float*>(K),
                                                       static_cast<const float*>(V), p);
    else if (D == 64)
        jfa_fwd_f32_kernel<64><<<g, kF32Rows, 0, st>>>(static_cast<const float*>(Q), static_cast<const float*>(K),
                                                       static_cast<const float*>(V), p);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_bwd_f32(int D, const void* Q, const void* K, const void* V, const void* dO, const BwdParams& p,
                           int64_t n_items, cudaStream_t st) {
    if (n_items <= 0) return cudaSuccess;
    const unsigned g = unsigned(n_items);
    if (D == 32)
        jfa_bwd_f32_kernel<32><<<g, kF32Rows, 0, st>>>(static_cast<const float*>(Q), static_cast<const float*>(K),
                                                       static_cast<const float*>(V), static_cast<const float*>(dO), p);
    else if (D == 64)
        jfa_bwd_f32_kernel<64><<<g, kF32Rows, 0, st>>>(static_cast<const float*>(Q), static_cast<const float*>(K),
                                                       static_cast<const float*>(V), static_cast<const float*>(dO), p);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace jfa
