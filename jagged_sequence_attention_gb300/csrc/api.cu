// C-ABI of libjfa: argument validation, plans, tensor maps and kernel launches.
// Semantics of every entry point are documented in include/jfa.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "jfa_internal.h"

using namespace jfa;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t elem_bytes(int dtype) { return dtype == JFA_F32 ? 4 : 2; }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// 2-D view [rows, H*D] of a token-major [T, H, D] tensor, box = box_bytes (128 or 64) x
// box_rows, swizzled over the box row (128- or 64-byte swizzle), zero fill beyond the last row.
jfa_status make_map(CUtensorMap* map, int dtype, const void* base, int64_t rows, int H, int D,
                    const void* dummy, int box_rows = 128, int box_bytes = 128) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return JFA_ERR_CUDA;
    const size_t E = elem_bytes(dtype);
    if (rows <= 0) {  // never read; keep the descriptor well-formed
        rows = 1;
        base = dummy;
    }
    cuuint64_t dims[2] = {cuuint64_t(H) * cuuint64_t(D), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(H) * cuuint64_t(D) * E};
    cuuint32_t box[2] = {cuuint32_t(box_bytes / int(E)), cuuint32_t(box_rows)};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(map, dtype == JFA_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? JFA_OK : JFA_ERR_CUDA;
}

cudaEvent_t take_event(jfa_plan plan) {
    if (!plan->ev_pool.empty()) {
        cudaEvent_t e = plan->ev_pool.back();
        plan->ev_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Records a start event before a kernel launch when timing is enabled.
struct KernelTimer {
    jfa_plan plan;
    int kind;
    cudaStream_t st;
    cudaEvent_t a = nullptr, b = nullptr;
    KernelTimer(jfa_plan p, int k, cudaStream_t s) : plan(p), kind(k), st(s) {
        if (!plan->timing) return;
        a = take_event(plan);
        b = take_event(plan);
        if (a && b) cudaEventRecord(a, st);
    }
    void done() {
        if (!plan->timing || !a || !b) return;
        cudaEventRecord(b, st);
        plan->ev_pending.push_back({kind, {a, b}});
        a = b = nullptr;
    }
};

jfa_status check_plan_call(jfa_plan plan, int dtype, int bias_kind, const float* bias_table) {
    if (!plan) return JFA_ERR_INVALID_ARG;
    if (dtype != JFA_BF16 && dtype != JFA_F32) return JFA_ERR_INVALID_ARG;
    if (!supported(dtype, plan->D)) return JFA_ERR_UNSUPPORTED;
    if (bias_kind != JFA_BIAS_NONE && bias_kind != JFA_BIAS_RELPOS32 && bias_kind != JFA_BIAS_DENSE)
        return JFA_ERR_INVALID_ARG;
    if (bias_kind == JFA_BIAS_RELPOS32 && !bias_table) return JFA_ERR_INVALID_ARG;
    if (bias_kind == JFA_BIAS_DENSE && !bias_table && plan->n_pairs > 0) return JFA_ERR_INVALID_ARG;
    return JFA_OK;
}

// The work lists a call runs on.  A shared key/value plan without causal masking or
// a window also holds a merged view: consecutive query sets of one user form one query
// sequence, so their rows fill whole 128-row tiles.  A row's result does not depend on
// which query set it belongs to unless the relative-position table is used (its
// positions are per query set), so every call but those with JFA_BIAS_RELPOS32 runs on
// the merged view.  A dense bias keeps its layout: the query sets' consecutive
// [q_len, kv_len] blocks are the merged sequence's block.
const jfa_plan_t* work_view(const jfa_plan_t* plan, int32_t bias_kind) {
    return (plan->merged && bias_kind != JFA_BIAS_RELPOS32) ? plan->merged : plan;
}

}  // namespace

extern "C" {

const char* jfa_status_string(int32_t s) {
    switch (s) {
        case JFA_OK: return "ok";
        case JFA_ERR_INVALID_ARG: return "invalid argument";
        case JFA_ERR_UNSUPPORTED: return "unsupported head_dim/dtype/mode";
        case JFA_ERR_CUDA: return "CUDA error";
        case JFA_ERR_TIMEOUT: return "kernel pipeline wait timed out";
        case JFA_ERR_DEVICE_BOUNDS: return "kernel bounds check fired";
        case JFA_ERR_PLAN_MISMATCH: return "call does not match the plan";
        case JFA_ERR_NO_DEVICE: return "no usable sm_100-family GPU";
        case JFA_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the static array holds (JFA_STATIC_SCRATCH_BYTES)";
        default: return "unknown status";
    }
}

jfa_status jfa_worklist_size(const int32_t* q_offsets, const int32_t* kv_offsets, int32_t B, int32_t H,
                             int32_t causal, int32_t window, int32_t pass, int64_t* n_items) {
    if (!n_items || H < 1 || pass < kPassFwd || pass > kPassBwdShort) return JFA_ERR_INVALID_ARG;
    if (window < -1 || (window >= 0 && causal != 1)) return JFA_ERR_INVALID_ARG;
    if (pass == kPassBwdShort && (causal != 0 || window >= 0)) return JFA_ERR_INVALID_ARG;
    jfa_status s = validate_offsets(q_offsets, kv_offsets, B);
    if (s != JFA_OK) return s;
    *n_items = count_items(q_offsets, kv_offsets, B, H, causal, pass);
    return JFA_OK;
}

jfa_status jfa_worklist_build(const int32_t* q_offsets, const int32_t* kv_offsets, int32_t B, int32_t H,
                              int32_t causal, int32_t window, int32_t pass, int32_t n_ctas, int32_t* items,
                              int32_t* cta_offsets, int64_t* cta_cost) {
    if (H < 1 || n_ctas < 1 || !cta_offsets || pass < kPassFwd || pass > kPassBwdShort) return JFA_ERR_INVALID_ARG;
    if (window < -1 || (window >= 0 && causal != 1)) return JFA_ERR_INVALID_ARG;
    if (pass == kPassBwdShort && (causal != 0 || window >= 0)) return JFA_ERR_INVALID_ARG;
    jfa_status s = validate_offsets(q_offsets, kv_offsets, B);
    if (s != JFA_OK) return s;
    const int64_t n = count_items(q_offsets, kv_offsets, B, H, causal, pass);
    if (n > 0 && !items) return JFA_ERR_INVALID_ARG;
    build_worklist(q_offsets, kv_offsets, B, H, causal, window, pass, n_ctas, reinterpret_cast<WorkItem*>(items),
                   cta_offsets, cta_cost);
    return JFA_OK;
}

jfa_status jfa_partition_sequences(const int32_t* q_offsets, const int32_t* kv_offsets, int32_t B, int32_t H,
                                   int32_t causal, int32_t window, int32_t n_parts, int32_t* part_of_seq,
                                   int64_t* part_cost) {
    if (H < 1 || n_parts < 1 || (causal != 0 && causal != 1) || (B > 0 && !part_of_seq)) return JFA_ERR_INVALID_ARG;
    if (window < -1 || (window >= 0 && causal != 1)) return JFA_ERR_INVALID_ARG;
    jfa_status s = validate_offsets(q_offsets, kv_offsets, B);
    if (s != JFA_OK) return s;
    partition_sequences(q_offsets, kv_offsets, B, H, causal, window, n_parts, part_of_seq, part_cost);
    return JFA_OK;
}

jfa_status jfa_partition_users(const int32_t* q_offsets, int32_t B, const int32_t* kv_offsets, int32_t U,
                               const int32_t* kv_index, int32_t H, int32_t causal, int32_t window, int32_t n_parts,
                               int32_t* part_of_user, int64_t* part_cost) {
    if (!q_offsets || !kv_offsets || (B > 0 && !kv_index) || B < 0 || U < 0 || H < 1 || n_parts < 1 ||
        (causal != 0 && causal != 1) || (U > 0 && !part_of_user))
        return JFA_ERR_INVALID_ARG;
    if (window < -1 || (window >= 0 && causal != 1)) return JFA_ERR_INVALID_ARG;
    if (q_offsets[0] != 0 || kv_offsets[0] != 0) return JFA_ERR_INVALID_ARG;
    for (int32_t b = 0; b < B; ++b)
        if (q_offsets[b + 1] < q_offsets[b] || kv_index[b] < 0 || kv_index[b] >= U) return JFA_ERR_INVALID_ARG;
    for (int32_t u = 0; u < U; ++u)
        if (kv_offsets[u + 1] < kv_offsets[u]) return JFA_ERR_INVALID_ARG;
    partition_users(q_offsets, kv_offsets, kv_index, B, U, H, causal, window, n_parts, part_of_user, part_cost);
    return JFA_OK;
}

jfa_status jfa_plan_create(const int32_t* q_offsets, const int32_t* kv_offsets, int32_t B, int32_t H, int32_t D,
                           int32_t mode, int32_t causal, int32_t offsets_on_device, void* stream, jfa_plan* out) {
    return jfa_plan_create_ex(q_offsets, kv_offsets, B, H, D, mode, causal, -1, offsets_on_device, stream, out);
}

// Builds a plan from host offsets.  kv_map (length B) is the query-set-to-user map of
// shared key/value attention, with U users in kv_off; without it U == B and sequence b
// attends to its own rows.
static jfa_status plan_create_impl(const std::vector<int32_t>& qo, const std::vector<int32_t>& ko,
                                   const std::vector<int32_t>* kv_map, int32_t B, int32_t U, int32_t H, int32_t D,
                                   int32_t mode, int32_t causal, int32_t window, cudaStream_t st, jfa_plan* out,
                                   bool allow_merge = true) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return JFA_ERR_NO_DEVICE;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return JFA_ERR_NO_DEVICE;
    if (prop.major != 10) return JFA_ERR_NO_DEVICE;

    // Per query set, the offsets of its key/value rows as if each had its own copy: the
    // forward and dQ passes (and a dense bias's pair offsets) only need the lengths.
    std::vector<int32_t> kvv(size_t(B) + 1, 0);
    for (int32_t b = 0; b < B; ++b) {
        const int32_t u = kv_map ? (*kv_map)[size_t(b)] : b;
        kvv[size_t(b) + 1] = kvv[size_t(b)] + (ko[size_t(u) + 1] - ko[size_t(u)]);
    }

    jfa_plan_t* p = new (std::nothrow) jfa_plan_t();
    if (!p) return JFA_ERR_CUDA;
    p->B = B;
    p->U = U;
    p->shared_kv = kv_map != nullptr;
    p->H = H;
    p->D = D;
    p->mode = mode;
    p->causal = causal;
    p->window = window;
    p->Tq = qo[size_t(B)];
    p->Tkv = ko[size_t(U)];
    p->device = dev;
    p->num_sms = prop.multiProcessorCount;
    p->q_off = qo;
    p->kv_off = ko;
    p->timing = false;

    std::vector<int2> steps;
    std::vector<int32_t> step_off, ktile_off;
    p->n_fwd_items = count_items(qo.data(), kvv.data(), B, H, causal, kPassFwd);
    p->n_bwd_items = kv_map ? count_shared_kv_dkdv_items(ko.data(), U, H)
                            : count_items(qo.data(), ko.data(), B, H, causal, kPassBwdKV);
    p->n_dq_items = count_items(qo.data(), kvv.data(), B, H, causal, kPassBwdQ);
    p->fwd_grid = int(std::max<int64_t>(1, std::min<int64_t>(p->num_sms, p->n_fwd_items)));
    p->fwd_split = prefer_split_forward(qo.data(), kvv.data(), B, causal, window);
    p->bwd_grid = int(std::max<int64_t>(1, std::min<int64_t>(p->num_sms, p->n_bwd_items)));
    p->dq_grid = int(std::max<int64_t>(1, std::min<int64_t>(p->num_sms, p->n_dq_items)));
    std::vector<WorkItem> fi(size_t(std::max<int64_t>(1, p->n_fwd_items)));
    std::vector<WorkItem> bi(size_t(std::max<int64_t>(1, p->n_bwd_items)));
    std::vector<WorkItem> qi(size_t(std::max<int64_t>(1, p->n_dq_items)));
    std::vector<int32_t> fo(size_t(p->fwd_grid) + 1), bo(size_t(p->bwd_grid) + 1), qio(size_t(p->dq_grid) + 1);
    build_worklist(qo.data(), kvv.data(), B, H, causal, window, kPassFwd, p->fwd_grid, fi.data(), fo.data(), nullptr);
    if (kv_map)
        build_shared_kv_dkdv(qo.data(), ko.data(), kv_map->data(), B, U, H, causal, window, p->bwd_grid, bi.data(),
                             bo.data(), &steps, &step_off, &ktile_off);
    else
        build_worklist(qo.data(), ko.data(), B, H, causal, window, kPassBwdKV, p->bwd_grid, bi.data(), bo.data(),
                       nullptr);
    build_worklist(qo.data(), kvv.data(), B, H, causal, window, kPassBwdQ, p->dq_grid, qi.data(), qio.data(), nullptr);
    {
        // Backward form: the fused kernel saves the whole dQ pass but pays more per step
        // (dQ's reduce-adds and their drain), so it wins while key tiles visit few query
        // tiles (short sequences) and loses on long ones.
        int64_t total_steps = 0;
        if (!kv_map)
            for (int64_t i = 0; i < p->n_bwd_items; ++i) total_steps += bi[size_t(i)].n_inner;
        p->fused_pref = !kv_map && p->n_bwd_items > 0 && total_steps <= kFusedMaxMeanSteps * p->n_bwd_items;
    }
    // Short-query backward: one (sequence, head) item per query set, when each fits one tile.
    p->short_bq = short_query_rows(qo.data(), B, D, causal, window, kv_map != nullptr);
    // The forward's kernel holds a different number of CTAs per SM (one for the softmax
    // kernel with two key tiles per score tile), so it has its own grouping of the items.
    std::vector<WorkItem> si(1), sfi(1);
    std::vector<int32_t> sio(2, 0), sfo(2, 0);
    if (p->short_bq > 0) {
        p->n_short_items = count_items(qo.data(), ko.data(), B, H, 0, kPassBwdShort);
        auto grid_of = [&](int per_sm) {
            return int(std::max<int64_t>(1, std::min<int64_t>(int64_t(p->num_sms) * per_sm, p->n_short_items)));
        };
        p->short_grid = grid_of(short_ctas_per_sm(D, p->short_bq));
        const bool pack = mode == JFA_SOFTMAX;  // (applies at D = 64 with 64-row tiles only)
        p->short_fwd_grid = grid_of(pack ? 1 : short_fwd_ctas_per_sm(D, p->short_bq));
        si.resize(size_t(std::max<int64_t>(1, p->n_short_items)));
        sfi.resize(si.size());
        sio.resize(size_t(p->short_grid) + 1);
        sfo.resize(size_t(p->short_fwd_grid) + 1);
        build_worklist(qo.data(), ko.data(), B, H, 0, -1, kPassBwdShort, p->short_grid, si.data(), sio.data(), nullptr);
        build_worklist(qo.data(), ko.data(), B, H, 0, -1, kPassBwdShort, p->short_fwd_grid, sfi.data(), sfo.data(),
                       nullptr);
    }
    std::vector<int64_t> po(size_t(B) + 1, 0);  // pair offsets of a dense bias
    for (int32_t b = 0; b < B; ++b)
        po[size_t(b) + 1] = po[size_t(b)] + int64_t(qo[size_t(b) + 1] - qo[size_t(b)]) * int64_t(kvv[size_t(b) + 1] - kvv[size_t(b)]);
    p->n_pairs = po[size_t(B)];
    p->n_steps = int64_t(steps.size());
    if (steps.empty()) steps.push_back(make_int2(0, 0));
    if (step_off.empty()) step_off.push_back(0);
    if (ktile_off.empty()) ktile_off.push_back(0);
    std::vector<int32_t> map_h = kv_map ? *kv_map : std::vector<int32_t>(1, 0);

    // One device block: offsets, status word, work lists (16-byte aligned pieces).
    size_t cur = 0;
    const size_t o_q = cur; cur += round_up((size_t(B) + 1) * 4, 256);
    const size_t o_kv = cur; cur += round_up((size_t(U) + 1) * 4, 256);
    const size_t o_st = cur; cur += 256;
    const size_t o_fi = cur; cur += round_up(fi.size() * 16, 256);
    const size_t o_fo = cur; cur += round_up(fo.size() * 4, 256);
    const size_t o_bi = cur; cur += round_up(bi.size() * 16, 256);
    const size_t o_bo = cur; cur += round_up(bo.size() * 4, 256);
    const size_t o_qi = cur; cur += round_up(qi.size() * 16, 256);
    const size_t o_qo = cur; cur += round_up(qio.size() * 4, 256);
    const size_t o_po = cur; cur += round_up(po.size() * 8, 256);
    const size_t o_map = cur; cur += round_up(map_h.size() * 4, 256);
    const size_t o_sp = cur; cur += round_up(steps.size() * 8, 256);
    const size_t o_so = cur; cur += round_up(step_off.size() * 4, 256);
    const size_t o_ko = cur; cur += round_up(ktile_off.size() * 4, 256);
    const size_t o_si = cur; cur += round_up(si.size() * 16, 256);
    const size_t o_sio = cur; cur += round_up(sio.size() * 4, 256);
    const size_t o_sfi = cur; cur += round_up(sfi.size() * 16, 256);
    const size_t o_sfo = cur; cur += round_up(sfo.size() * 4, 256);
    if (cudaMalloc(&p->dev_block, cur) != cudaSuccess) {
        delete p;
        return JFA_ERR_CUDA;
    }
    char* base = static_cast<char*>(p->dev_block);
    p->d_q_off = reinterpret_cast<int32_t*>(base + o_q);
    p->d_kv_off = reinterpret_cast<int32_t*>(base + o_kv);
    p->d_status = reinterpret_cast<int*>(base + o_st);
    p->d_fwd_items = reinterpret_cast<int4*>(base + o_fi);
    p->d_fwd_cta_off = reinterpret_cast<int32_t*>(base + o_fo);
    p->d_bwd_items = reinterpret_cast<int4*>(base + o_bi);
    p->d_bwd_cta_off = reinterpret_cast<int32_t*>(base + o_bo);
    p->d_dq_items = reinterpret_cast<int4*>(base + o_qi);
    p->d_dq_cta_off = reinterpret_cast<int32_t*>(base + o_qo);
    p->d_pair_off = reinterpret_cast<int64_t*>(base + o_po);
    p->d_kv_map = kv_map ? reinterpret_cast<int32_t*>(base + o_map) : nullptr;
    p->d_steps = kv_map ? reinterpret_cast<int2*>(base + o_sp) : nullptr;
    p->d_step_off = kv_map ? reinterpret_cast<int32_t*>(base + o_so) : nullptr;
    p->d_ktile_off = kv_map ? reinterpret_cast<int32_t*>(base + o_ko) : nullptr;
    p->d_short_items = reinterpret_cast<int4*>(base + o_si);
    p->d_short_cta_off = reinterpret_cast<int32_t*>(base + o_sio);
    p->d_sfwd_items = reinterpret_cast<int4*>(base + o_sfi);
    p->d_sfwd_cta_off = reinterpret_cast<int32_t*>(base + o_sfo);
    auto up = [&](void* dst, const void* src, size_t bytes) {
        return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, st) == cudaSuccess;
    };
    bool ok = up(p->d_q_off, qo.data(), qo.size() * 4) && up(p->d_kv_off, ko.data(), ko.size() * 4) &&
              cudaMemsetAsync(p->d_status, 0, 256, st) == cudaSuccess &&
              up(p->d_fwd_items, fi.data(), fi.size() * 16) && up(p->d_fwd_cta_off, fo.data(), fo.size() * 4) &&
              up(p->d_bwd_items, bi.data(), bi.size() * 16) && up(p->d_bwd_cta_off, bo.data(), bo.size() * 4) &&
              up(p->d_dq_items, qi.data(), qi.size() * 16) && up(p->d_dq_cta_off, qio.data(), qio.size() * 4) &&
              up(p->d_pair_off, po.data(), po.size() * 8) && up(base + o_map, map_h.data(), map_h.size() * 4) &&
              up(base + o_sp, steps.data(), steps.size() * 8) && up(base + o_so, step_off.data(), step_off.size() * 4) &&
              up(base + o_ko, ktile_off.data(), ktile_off.size() * 4) &&
              up(base + o_si, si.data(), si.size() * 16) && up(base + o_sio, sio.data(), sio.size() * 4) &&
              up(base + o_sfi, sfi.data(), sfi.size() * 16) && up(base + o_sfo, sfo.data(), sfo.size() * 4);
    // The host vectors are pageable: the copies above are staged before returning,
    // but keep the stream ordered before the vectors go out of scope.
    if (!ok || cudaStreamSynchronize(st) != cudaSuccess) {
        cudaFree(p->dev_block);
        delete p;
        return JFA_ERR_CUDA;
    }
    // Shared key/value without causal masking or a window: also plan the merged view,
    // runs of consecutive query sets of one user as one query sequence (see work_view).
    if (allow_merge && kv_map && !causal && window < 0) {
        std::vector<int32_t> mqo(1, 0), mmap;
        for (int32_t b = 0; b < B; ++b) {
            const int32_t u = (*kv_map)[size_t(b)];
            if (mmap.empty() || mmap.back() != u) {
                mmap.push_back(u);
                mqo.push_back(qo[size_t(b) + 1]);
            } else {
                mqo.back() = qo[size_t(b) + 1];
            }
        }
        const int32_t M = int32_t(mmap.size());
        if (M < B) {
            jfa_plan child = nullptr;
            const jfa_status s = plan_create_impl(mqo, ko, &mmap, M, U, H, D, mode, causal, window, st, &child, false);
            if (s != JFA_OK) {
                cudaFree(p->dev_block);
                delete p;
                return s;
            }
            p->merged = child;
        }
    }
    *out = p;
    return JFA_OK;
}

// Host copies of offsets (or of a map) given on the host or, with on_device, on the
// device (copied on `st`, which this synchronises).
static bool host_copy(const int32_t* src, size_t n, int32_t on_device, cudaStream_t st, std::vector<int32_t>* dst) {
    dst->resize(n);
    if (n == 0) return true;
    if (on_device)
        return cudaMemcpyAsync(dst->data(), src, n * 4, cudaMemcpyDeviceToHost, st) == cudaSuccess &&
               cudaStreamSynchronize(st) == cudaSuccess;
    std::memcpy(dst->data(), src, n * 4);
    return true;
}

jfa_status jfa_plan_create_ex(const int32_t* q_offsets, const int32_t* kv_offsets, int32_t B, int32_t H, int32_t D,
                              int32_t mode, int32_t causal, int32_t window, int32_t offsets_on_device, void* stream,
                              jfa_plan* out) {
    if (!out) return JFA_ERR_INVALID_ARG;
    *out = nullptr;
    if (!q_offsets || !kv_offsets || B < 0 || H < 1 || H > 65535) return JFA_ERR_INVALID_ARG;
    if (mode != JFA_SOFTMAX && mode != JFA_GDPA_GELU_TANH && mode != JFA_GDPA_SILU) return JFA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return JFA_ERR_INVALID_ARG;
    if (window < -1 || (window >= 0 && causal != 1)) return JFA_ERR_INVALID_ARG;
    if (D != 32 && D != 64 && D != 128) return JFA_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::vector<int32_t> qo, ko;
    if (!host_copy(q_offsets, size_t(B) + 1, offsets_on_device, st, &qo) ||
        !host_copy(kv_offsets, size_t(B) + 1, offsets_on_device, st, &ko))
        return JFA_ERR_CUDA;
    jfa_status s = validate_offsets(qo.data(), ko.data(), B);
    if (s != JFA_OK) return s;
    return plan_create_impl(qo, ko, nullptr, B, B, H, D, mode, causal, window, st, out);
}

jfa_status jfa_plan_create_shared_kv(const int32_t* q_offsets, int32_t B, const int32_t* kv_offsets, int32_t U,
                                     const int32_t* kv_index, int32_t H, int32_t D, int32_t mode, int32_t causal,
                                     int32_t window, int32_t offsets_on_device, void* stream, jfa_plan* out) {
    if (!out) return JFA_ERR_INVALID_ARG;
    *out = nullptr;
    if (!q_offsets || !kv_offsets || (B > 0 && !kv_index) || B < 0 || U < 0 || H < 1 || H > 65535)
        return JFA_ERR_INVALID_ARG;
    if (mode != JFA_SOFTMAX && mode != JFA_GDPA_GELU_TANH && mode != JFA_GDPA_SILU) return JFA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return JFA_ERR_INVALID_ARG;
    if (window < -1 || (window >= 0 && causal != 1)) return JFA_ERR_INVALID_ARG;
    if (D != 32 && D != 64 && D != 128) return JFA_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::vector<int32_t> qo, ko, map;
    if (!host_copy(q_offsets, size_t(B) + 1, offsets_on_device, st, &qo) ||
        !host_copy(kv_offsets, size_t(U) + 1, offsets_on_device, st, &ko) ||
        !host_copy(kv_index, size_t(B), offsets_on_device, st, &map))
        return JFA_ERR_CUDA;
    if (qo[0] != 0 || ko[0] != 0) return JFA_ERR_INVALID_ARG;
    for (int32_t b = 0; b < B; ++b)
        if (qo[size_t(b) + 1] < qo[size_t(b)] || map[size_t(b)] < 0 || map[size_t(b)] >= U) return JFA_ERR_INVALID_ARG;
    for (int32_t u = 0; u < U; ++u)
        if (ko[size_t(u) + 1] < ko[size_t(u)]) return JFA_ERR_INVALID_ARG;
    return plan_create_impl(qo, ko, &map, B, U, H, D, mode, causal, window, st, out);
}

jfa_status jfa_plan_destroy(jfa_plan plan) {
    if (!plan) return JFA_OK;
    if (plan->merged) jfa_plan_destroy(plan->merged);
    for (auto& pr : plan->ev_pending) {
        cudaEventDestroy(pr.second.first);
        cudaEventDestroy(pr.second.second);
    }
    for (cudaEvent_t e : plan->ev_pool) cudaEventDestroy(e);
    cudaError_t e = cudaFree(plan->dev_block);
    delete plan;
    return e == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

jfa_status jfa_plan_info(jfa_plan plan, int64_t* info, int32_t n) {
    if (!plan || !info || n < 0) return JFA_ERR_INVALID_ARG;
    const int64_t v[22] = {plan->Tq,       plan->Tkv,     plan->B,           plan->H,        plan->D,
                           plan->mode,     plan->causal,  plan->n_fwd_items, plan->fwd_grid, plan->n_bwd_items,
                           plan->bwd_grid, plan->num_sms, plan->n_dq_items,  plan->dq_grid,  plan->window,
                           plan->n_pairs,  plan->shared_kv ? plan->U : -1,
                           plan->merged ? int64_t(plan->merged->B) : -1,
                           plan->fwd_split ? 1 : 0,
                           fused_backward(plan) ? 1 : 0,
                           short_backward(plan, JFA_BIAS_NONE, false) ? plan->short_bq : 0,
                           short_forward(plan, JFA_BIAS_NONE) ? plan->short_bq : 0};
    for (int32_t i = 0; i < n && i < 22; ++i) info[i] = v[i];
    return JFA_OK;
}

jfa_status jfa_plan_set_work_item(jfa_plan plan, int32_t pass, int64_t index, const int32_t* item) {
    // pass 4: the short-query forward's list (pass 3's items, grouped for its grid)
    if (!plan || !item || pass < kPassFwd || pass > kPassBwdShort + 1 || index < 0) return JFA_ERR_INVALID_ARG;
    const int64_t n = pass == kPassFwd     ? plan->n_fwd_items
                      : pass == kPassBwdKV ? plan->n_bwd_items
                      : pass == kPassBwdQ  ? plan->n_dq_items
                                           : plan->n_short_items;
    if (index >= n) return JFA_ERR_INVALID_ARG;
    int4* list = pass == kPassFwd         ? plan->d_fwd_items
                 : pass == kPassBwdKV     ? plan->d_bwd_items
                 : pass == kPassBwdQ      ? plan->d_dq_items
                 : pass == kPassBwdShort  ? plan->d_short_items
                                          : plan->d_sfwd_items;
    const int4 w = make_int4(item[0], item[1], item[2], item[3]);
    return cudaMemcpy(list + index, &w, sizeof(w), cudaMemcpyHostToDevice) == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

jfa_status jfa_plan_set_deterministic(jfa_plan plan, int32_t enable) {
    if (!plan || (enable != 0 && enable != 1)) return JFA_ERR_INVALID_ARG;
    plan->deterministic = enable != 0;
    return JFA_OK;
}

jfa_status jfa_plan_set_timing(jfa_plan plan, int32_t enable) {
    if (!plan) return JFA_ERR_INVALID_ARG;
    plan->timing = enable != 0;
    return JFA_OK;
}

jfa_status jfa_plan_kernel_times(jfa_plan plan, double* total_ms, int64_t* launches) {
    if (!plan) return JFA_ERR_INVALID_ARG;
    double t[kNumKernelKinds] = {};
    int64_t n[kNumKernelKinds] = {};
    jfa_status st = JFA_OK;
    for (auto& pr : plan->ev_pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(pr.second.second) != cudaSuccess ||
            cudaEventElapsedTime(&ms, pr.second.first, pr.second.second) != cudaSuccess)
            st = JFA_ERR_CUDA;
        t[pr.first] += ms;
        n[pr.first] += 1;
        plan->ev_pool.push_back(pr.second.first);
        plan->ev_pool.push_back(pr.second.second);
    }
    plan->ev_pending.clear();
    for (int i = 0; i < kNumKernelKinds; ++i) {
        if (total_ms) total_ms[i] = t[i];
        if (launches) launches[i] = n[i];
    }
    return st;
}

jfa_status jfa_plan_device_status(jfa_plan plan, void* stream) {
    if (!plan) return JFA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int h = 0;
    if (cudaMemcpyAsync(&h, plan->d_status, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemsetAsync(plan->d_status, 0, 4, st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
        return JFA_ERR_CUDA;
    if (h & kStatusTimeout) return JFA_ERR_TIMEOUT;
    if (h & kStatusBounds) return JFA_ERR_DEVICE_BOUNDS;
    return JFA_OK;
}

jfa_status jfa_fwd(jfa_plan plan, int32_t dtype, const void* Q, const void* K, const void* V, int32_t bias_kind,
                   const float* bias_table, float scale, void* O, int32_t o_dtype, float* lse, void* stream) {
    jfa_status s = check_plan_call(plan, dtype, bias_kind, bias_table);
    if (s != JFA_OK) return s;
    const jfa_plan_t* v = work_view(plan, bias_kind);  // work lists and offsets
    if (o_dtype != JFA_BF16 && o_dtype != JFA_F32) return JFA_ERR_INVALID_ARG;
    if (dtype == JFA_F32 && o_dtype != JFA_F32) return JFA_ERR_UNSUPPORTED;
    const bool softmax = plan->mode == JFA_SOFTMAX;
    if (plan->Tq > 0 && (!Q || !O || (softmax && !lse))) return JFA_ERR_INVALID_ARG;
    if (plan->Tkv > 0 && (!K || !V)) return JFA_ERR_INVALID_ARG;
    // softmax: each row's maximum is bounded by scale times its largest raw score
    if (softmax && !(scale > 0.f && scale < INFINITY)) return JFA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(bias_table) & 3u))
        return JFA_ERR_INVALID_ARG;
    if (plan->Tq == 0 || v->n_fwd_items == 0) return JFA_OK;
    // bf16 GDPA without a bias, every query set in one tile: the transposed short-query
    // forward over (sequence, head) items (fwd_short.cu)
    const bool short_q = dtype == JFA_BF16 && short_forward(v, bias_kind);
    CUtensorMap mq, mk, mv;
    if (dtype == JFA_BF16 &&
        ((s = make_map(&mq, dtype, Q, plan->Tq, plan->H, plan->D, plan->dev_block, short_q ? v->short_bq : 128)) !=
             JFA_OK ||
         (s = make_map(&mk, dtype, K, plan->Tkv, plan->H, plan->D, plan->dev_block)) != JFA_OK ||
         (s = make_map(&mv, dtype, V, plan->Tkv, plan->H, plan->D, plan->dev_block)) != JFA_OK))
        return s;
    FwdParams p;
    p.items = v->d_fwd_items;
    p.cta_off = v->d_fwd_cta_off;
    p.q_off = v->d_q_off;
    p.kv_off = v->d_kv_off;
    p.H = plan->H;
    p.mode = plan->mode;
    p.causal = plan->causal;
    p.window = plan->window;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.bias = bias_kind == JFA_BIAS_RELPOS32 ? bias_table : nullptr;
    p.O = O;
    p.lse = softmax ? lse : nullptr;
    p.status = plan->d_status;
    if (bias_kind == JFA_BIAS_DENSE) {
        p.dense = bias_table;
        p.pair_off = v->d_pair_off;
        p.n_pairs = plan->n_pairs;
    }
    p.kv_map = v->d_kv_map;
    p.n_seq = v->B;
    p.n_kv = v->U;
    KernelTimer tm(plan, 0, static_cast<cudaStream_t>(stream));
    cudaError_t e;
    if (short_q) {
        p.items = v->d_sfwd_items;
        p.cta_off = v->d_sfwd_cta_off;
        e = softmax ? launch_fwd_pack(o_dtype, mq, mk, mv, p, v->short_fwd_grid, static_cast<cudaStream_t>(stream))
                    : launch_fwd_short(o_dtype, plan->D, v->short_bq, mq, mk, mv, p, v->short_fwd_grid,
                                       static_cast<cudaStream_t>(stream));
    } else {
        e = dtype == JFA_BF16 ? launch_fwd(dtype, o_dtype, plan->D, mq, mk, mv, p, v->fwd_grid, v->fwd_split,
                                           static_cast<cudaStream_t>(stream))
                              : launch_fwd_f32(plan->D, Q, K, V, p, v->n_fwd_items, static_cast<cudaStream_t>(stream));
    }
    tm.done();
    return e == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

size_t jfa_bwd_workspace_size(jfa_plan plan, int32_t dtype) {
    if (!plan || (dtype != JFA_BF16 && dtype != JFA_F32)) return 0;
    const size_t rows = size_t(plan->Tq) * size_t(plan->H);
    // row terms; fp32 inputs, and bf16 inputs on the fused backward, also accumulate dQ in
    // fp32 before converting it
    const bool acc = dtype == JFA_F32 || fused_backward(plan);
    return round_up(rows * 4, 256) + (acc ? round_up(rows * size_t(plan->D) * 4, 256) : 0);
}

// Bytes of the partial table gradients: one [H][32] table per (CTA, compute warp) of
// the dK/dV grid (bf16), or one [32] row per work item (fp32).
static size_t dbias_part_bytes(jfa_plan plan, int32_t dtype) {
    const size_t n = dtype == JFA_BF16 ? size_t(plan->bwd_grid) * kDkdvCompWarps * size_t(plan->H) * 32
                                       : size_t(plan->n_bwd_items) * 32;
    return round_up(n * 4, 256);
}

size_t jfa_bwd_ex_workspace_size(jfa_plan plan, int32_t dtype, int32_t bias_kind) {
    const size_t base = jfa_bwd_workspace_size(plan, dtype);
    if (base == 0 && !plan) return 0;
    return base + (bias_kind == JFA_BIAS_RELPOS32 ? dbias_part_bytes(plan, dtype) : 0);
}

static jfa_status bwd_impl(jfa_plan plan, int32_t dtype, const void* Q, const void* K, const void* V, const void* O,
                           int32_t o_dtype, const void* dO, const float* lse, int32_t bias_kind,
                           const float* bias_table, float scale, void* dQ, void* dK, void* dV, float* dbias,
                           void* workspace, size_t workspace_bytes, void* stream);

jfa_status jfa_bwd(jfa_plan plan, int32_t dtype, const void* Q, const void* K, const void* V, const void* O,
                   int32_t o_dtype, const void* dO, const float* lse, int32_t bias_kind, const float* bias_table,
                   float scale, void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                   void* stream) {
    return bwd_impl(plan, dtype, Q, K, V, O, o_dtype, dO, lse, bias_kind, bias_table, scale, dQ, dK, dV, nullptr,
                    workspace, workspace_bytes, stream);
}

jfa_status jfa_bwd_ex(jfa_plan plan, int32_t dtype, const void* Q, const void* K, const void* V, const void* O,
                      int32_t o_dtype, const void* dO, const float* lse, int32_t bias_kind, const float* bias_table,
                      float scale, void* dQ, void* dK, void* dV, float* dbias, void* workspace,
                      size_t workspace_bytes, void* stream) {
    if (dbias && ((bias_kind != JFA_BIAS_RELPOS32 && bias_kind != JFA_BIAS_DENSE) ||
                  (reinterpret_cast<uintptr_t>(dbias) & 3u)))
        return JFA_ERR_INVALID_ARG;
    return bwd_impl(plan, dtype, Q, K, V, O, o_dtype, dO, lse, bias_kind, bias_table, scale, dQ, dK, dV, dbias,
                    workspace, workspace_bytes, stream);
}

static jfa_status bwd_impl(jfa_plan plan, int32_t dtype, const void* Q, const void* K, const void* V, const void* O,
                           int32_t o_dtype, const void* dO, const float* lse, int32_t bias_kind,
                           const float* bias_table, float scale, void* dQ, void* dK, void* dV, float* dbias,
                           void* workspace, size_t workspace_bytes, void* stream) {
    jfa_status s = check_plan_call(plan, dtype, bias_kind, bias_table);
    if (s != JFA_OK) return s;
    const jfa_plan_t* v = work_view(plan, bias_kind);  // work lists and offsets
    if (o_dtype != JFA_BF16 && o_dtype != JFA_F32) return JFA_ERR_INVALID_ARG;
    if (dtype == JFA_F32 && o_dtype != JFA_F32) return JFA_ERR_UNSUPPORTED;
    const bool softmax = plan->mode == JFA_SOFTMAX;
    if (plan->Tq > 0 && (!Q || !O || !dO || !dQ || (softmax && !lse))) return JFA_ERR_INVALID_ARG;
    if (plan->Tkv > 0 && (!K || !V || !dK || !dV)) return JFA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) || !aligned16(dQ) ||
        !aligned16(dK) || !aligned16(dV) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
        (reinterpret_cast<uintptr_t>(bias_table) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return JFA_ERR_INVALID_ARG;
    const size_t base = jfa_bwd_workspace_size(plan, dtype);
    const size_t need = dbias ? jfa_bwd_ex_workspace_size(plan, dtype, bias_kind) : base;
    if (workspace_bytes < need || (need > 0 && !workspace)) return JFA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool dense = bias_kind == JFA_BIAS_DENSE;
    if (dbias && (v->n_bwd_items == 0 || (dense && (plan->causal || plan->window >= 0)))) {
        // The kernels write the gradient of allowed pairs only: zero it first where some
        // pair is masked (dense), or everywhere when no key tile sees a query.
        const size_t n = dense ? size_t(plan->H) * size_t(plan->n_pairs) : size_t(plan->H) * 32;
        if (n > 0 && cudaMemsetAsync(dbias, 0, n * 4, st) != cudaSuccess) return JFA_ERR_CUDA;
        if (v->n_bwd_items == 0) dbias = nullptr;
    }
    if (plan->Tkv == 0 && plan->Tq == 0) return JFA_OK;
    const size_t rows = size_t(plan->Tq) * size_t(plan->H);
    // bf16 inputs without a bias or a bias gradient, every query set in one tile: dQ, dK and
    // dV in one kernel over (sequence, head) items, dQ held in TMEM (bwd_short.cu)
    const bool short_q = dtype == JFA_BF16 && short_backward(v, bias_kind, dbias != nullptr);
    // bf16 inputs without a dense bias or a bias gradient: dK, dV and dQ in one kernel that
    // adds dQ into an fp32 accumulator (bwd_fused.cu)
    const bool fused = dtype == JFA_BF16 && !short_q && !plan->deterministic && v->fused_pref && !dense && !dbias;
    float* delta = static_cast<float*>(workspace);
    float* dq_acc = (dtype == JFA_F32 || fused)
                        ? reinterpret_cast<float*>(static_cast<char*>(workspace) + round_up(rows * 4, 256))
                        : nullptr;
    float* dbias_part = (dbias && !dense) ? reinterpret_cast<float*>(static_cast<char*>(workspace) + base) : nullptr;

    cudaError_t e = cudaSuccess;
    if (plan->Tq > 0) {
        KernelTimer tm(plan, 1, st);
        e = launch_bwd_pre(dtype, o_dtype, plan->D, O, dO, delta, dq_acc, plan->Tq, plan->H, plan->mode, st);
        tm.done();
        if (e != cudaSuccess) return JFA_ERR_CUDA;
    }
    CUtensorMap mq, mk, mv, mdo, mdq, mdk, mdv;
    BwdParams p;
    if (v->n_bwd_items > 0 || (dtype == JFA_BF16 && v->n_dq_items > 0)) {
        const int q_box = short_q ? v->short_bq : kBwdBM;  // Q and dO rows per load
        if (dtype == JFA_BF16 &&
            ((s = make_map(&mq, dtype, Q, plan->Tq, plan->H, plan->D, plan->dev_block, q_box)) != JFA_OK ||
             (s = make_map(&mk, dtype, K, plan->Tkv, plan->H, plan->D, plan->dev_block, kBwdBN)) != JFA_OK ||
             (s = make_map(&mv, dtype, V, plan->Tkv, plan->H, plan->D, plan->dev_block, kBwdBN)) != JFA_OK ||
             (s = make_map(&mdo, dtype, dO, plan->Tq, plan->H, plan->D, plan->dev_block, q_box)) != JFA_OK))
            return s;
        // the fused backward's dQ accumulator, [T_q, H*D] fp32 in 32 x 32 boxes (reduce-adds)
        if (fused && (s = make_map(&mdq, JFA_F32, dq_acc, plan->Tq, plan->H, plan->D, plan->dev_block, 32)) != JFA_OK)
            return s;
        // and its dK, dV outputs, [T_kv, H*D] bf16 in 32-row boxes (stores of whole warps' rows)
        if (fused && ((s = make_map(&mdk, JFA_BF16, dK, plan->Tkv, plan->H, plan->D, plan->dev_block, 32)) != JFA_OK ||
                      (s = make_map(&mdv, JFA_BF16, dV, plan->Tkv, plan->H, plan->D, plan->dev_block, 32)) != JFA_OK))
            return s;
        p.items = v->d_bwd_items;
        p.cta_off = v->d_bwd_cta_off;
        p.q_off = v->d_q_off;
        p.kv_off = v->d_kv_off;
        p.H = plan->H;
        p.mode = plan->mode;
        p.causal = plan->causal;
        p.window = plan->window;
        p.scale = scale;
        p.scale_log2 = scale * 1.4426950408889634f;
        p.bias = bias_kind == JFA_BIAS_RELPOS32 ? bias_table : nullptr;
        p.lse = softmax ? lse : nullptr;
        p.delta = delta;
        p.dq_acc = dq_acc;
        p.dQ = dQ;
        p.dK = dK;
        p.dV = dV;
        p.status = plan->d_status;
        p.dbias_part = dbias_part;
        if (dense) {
            p.bias = nullptr;
            p.dense = bias_table;
            p.ddense = dbias;
            p.pair_off = v->d_pair_off;
            p.n_pairs = plan->n_pairs;
        }
        // shared key/value: the dK/dV pass walks the user's step lists, the dQ pass maps
        p.steps = v->d_steps;
        p.step_off = v->d_step_off;
        p.ktile_off = v->d_ktile_off;
        p.kv_map = v->d_kv_map;
        p.n_seq = v->B;
        p.n_kv = v->U;
    }
    if (short_q) {
        // one kernel writes dQ, dK and dV (also the zero rows of sequences without a query
        // or a key); dK and dV of whole warps' rows by TMA stores of 32 x 32 boxes
        if (v->n_short_items > 0 &&
            ((s = make_map(&mdk, dtype, dK, plan->Tkv, plan->H, plan->D, plan->dev_block, 32, 64)) != JFA_OK ||
             (s = make_map(&mdv, dtype, dV, plan->Tkv, plan->H, plan->D, plan->dev_block, 32, 64)) != JFA_OK))
            return s;
        p.items = v->d_short_items;
        p.cta_off = v->d_short_cta_off;
        KernelTimer tm(plan, 2, st);
        e = v->n_short_items > 0
                ? launch_bwd_short(plan->D, v->short_bq, mq, mk, mv, mdo, mdk, mdv, p, v->short_grid, st)
                : cudaSuccess;
        tm.done();
        return e == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
    }
    if (v->n_bwd_items > 0) {
        KernelTimer tm(plan, 2, st);
        e = dtype == JFA_BF16 ? (fused ? launch_bwd_fused(plan->D, mq, mk, mv, mdo, mdq, mdk, mdv, p, v->bwd_grid, st)
                                       : launch_bwd_main(dtype, plan->D, mq, mk, mv, mdo, p, v->bwd_grid, st))
                              : launch_bwd_f32(plan->D, Q, K, V, dO, p, v->n_bwd_items, st);
        tm.done();
        if (e != cudaSuccess) return JFA_ERR_CUDA;
        if (dbias_part) {
            e = dtype == JFA_BF16
                    ? launch_dbias_reduce(dbias_part, int64_t(v->bwd_grid) * kDkdvCompWarps, plan->H, dbias, st)
                    : launch_dbias_reduce_items(dbias_part, v->d_bwd_items, v->n_bwd_items, plan->H, dbias, st);
            if (e != cudaSuccess) return JFA_ERR_CUDA;
        }
        p.dbias_part = nullptr;  // the dQ pass does not take part
    }
    if (dtype == JFA_BF16 && !fused && v->n_dq_items > 0) {
        // dQ per query tile, written directly (also the zero rows of tiles that see no key)
        p.items = v->d_dq_items;
        p.cta_off = v->d_dq_cta_off;
        p.kv_map = v->d_kv_map;
        p.steps = nullptr;
        KernelTimer tm(plan, 4, st);
        e = launch_bwd_dq(dtype, plan->D, mq, mk, mv, mdo, p, v->dq_grid, st);
        tm.done();
        if (e != cudaSuccess) return JFA_ERR_CUDA;
    }
    if ((dtype == JFA_F32 || fused) && plan->Tq > 0) {
        KernelTimer tm(plan, 3, st);
        e = launch_bwd_post(dtype, plan->D, dq_acc, dQ, plan->Tq, plan->H, scale, st);
        tm.done();
        if (e != cudaSuccess) return JFA_ERR_CUDA;
    }
    return JFA_OK;
}

}  // extern "C"
