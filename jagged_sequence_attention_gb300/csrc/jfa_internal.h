// Internal declarations shared by the C-ABI layer, the planner and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>
#include <vector>

#include "jfa.h"

namespace jfa {

// Forward tiles: 128 query rows x 128 key rows, and a forward work item is a pair of
// query tiles (256 rows) sharing its key/value tiles.  Backward dK/dV tiles: 128 key
// rows (resident) x 128 query rows (streamed); backward dQ tiles: 128 query rows
// (resident) x 128 key rows (streamed), the forward's single-tile geometry.
constexpr int kFwdBM = 128;
constexpr int kFwdBN = 128;
constexpr int kFwdPairRows = 2 * kFwdBM;
constexpr int kBwdBN = 128;
constexpr int kBwdBM = 128;

// Work-list passes: forward query-tile pairs, backward key tiles (dK/dV), backward
// query tiles (dQ), and the short-query backward's (sequence, head) items.
enum : int { kPassFwd = 0, kPassBwdKV = 1, kPassBwdQ = 2, kPassBwdShort = 3 };

// Kernel kinds of the timing hook: forward, backward preprocess, backward dK/dV (or
// the fp32 main kernel), fp32 dQ conversion, bf16 dQ.
constexpr int kNumKernelKinds = 5;
// Compute warps of the bf16 dK/dV kernel (each keeps its own partial table gradient).
constexpr int kDkdvCompWarps = 8;

// One unit of persistent-grid work: sequence, head, tile index (query tile for the
// forward, key/value tile for the backward) and the number of inner tiles visited.
struct WorkItem {
    int32_t b, h, tile, n_inner;
};
static_assert(sizeof(WorkItem) == 16, "WorkItem must match int4");

// Key tiles a 128-row query tile visits: [first, first + count).  All of them, or
// (causal, bottom-right) up to the one holding its last row's diagonal; with a sliding
// window W >= 0 (row i sees keys i' - W .. i', i' = i + kv_len - q_len) they start at
// the tile holding its first row's lowest key.  count is 0 for a tile past the
// sequence end or one that sees no key.
__host__ __device__ inline void key_tile_range(int64_t q_len, int64_t kv_len, int64_t tile, int causal,
                                               int window, int& first, int& count) {
    first = 0;
    count = 0;
    const int64_t rows0 = tile * kFwdBM;
    if (rows0 >= q_len) return;
    int64_t end = (kv_len + kFwdBN - 1) / kFwdBN;
    const int64_t diag = kv_len - q_len;
    if (causal) {
        const int64_t last_row = (q_len < rows0 + kFwdBM ? q_len : rows0 + kFwdBM) - 1;
        const int64_t max_col = last_row + diag;
        end = max_col < 0 ? 0 : (end < max_col / kFwdBN + 1 ? end : max_col / kFwdBN + 1);
    }
    int64_t beg = 0;
    if (window >= 0) {
        const int64_t min_col = rows0 + diag - window;
        beg = min_col > 0 ? min_col / kFwdBN : 0;
    }
    if (end > beg) {
        first = int(beg);
        count = int(end - beg);
    }
}

__host__ __device__ inline int fwd_tiles_of(int64_t q_len, int64_t kv_len, int64_t tile, int causal, int window = -1) {
    int first, count;
    key_tile_range(q_len, kv_len, tile, causal, window, first, count);
    return count;
}

// Key tiles streamed by a forward pair item (query tiles 2t and 2t+1): the union of the
// two tiles' ranges, [first, first + count).
__host__ __device__ inline void pair_stream(int64_t q_len, int64_t kv_len, int64_t t, int causal, int window, int& first, int& count,
                        int& na, int& nb) {
    int fa, fb;
    key_tile_range(q_len, kv_len, 2 * t, causal, window, fa, na);
    key_tile_range(q_len, kv_len, 2 * t + 1, causal, window, fb, nb);
    if (na == 0 && nb == 0) {
        first = 0;
        count = 0;
    } else if (na == 0) {
        first = fb;
        count = nb;
    } else if (nb == 0) {
        first = fa;
        count = na;
    } else {
        first = fa < fb ? fa : fb;
        const int ea = fa + na, eb = fb + nb;
        count = (ea > eb ? ea : eb) - first;
    }
}

// A forward pair item (query tiles 2t and 2t+1) whose pair holds a single tile (2t + 1 is past
// the sequence end) that visits na >= 2 key tiles can be split: its key range is cut in two
// halves run as the pair's two tiles over the same query rows and merged at the end.  The
// split kernel splits such an item when the sequence is one tile, and for the last, odd tile
// of a longer sequence when its key range has at least kSplitMinTiles tiles: halving a long
// chain pays for the merge, a short one does not.
constexpr int kSplitMinTiles = 16;
__host__ __device__ inline bool fwd_split_item(int64_t q_len, int64_t t, int na) {
    return (2 * t + 1) * kFwdBM >= q_len && na >= 2 && (q_len <= kFwdBM || na >= kSplitMinTiles);
}

// Query tiles (kBwdBM rows) that see key tile nt (kBwdBN keys): [first, first + count).
// Row i sees key j when j <= i' (causal) and j >= i' - W (window), i' = i + kv_len - q_len.
__host__ __device__ inline void query_tile_range(int64_t q_len, int64_t kv_len, int64_t nt, int causal, int window,
                                                 int& first, int& count) {
    first = 0;
    count = 0;
    const int64_t diag = kv_len - q_len;
    const int64_t j0 = nt * kBwdBN;
    const int64_t j1 = (kv_len < j0 + kBwdBN ? kv_len : j0 + kBwdBN) - 1;  // last key of the tile
    if (j1 < j0 || q_len <= 0) return;
    int64_t first_row = causal ? j0 - diag : 0;
    if (first_row < 0) first_row = 0;
    int64_t last_row = q_len - 1;
    if (window >= 0 && j1 + window - diag < last_row) last_row = j1 + window - diag;
    if (first_row > last_row) return;
    first = int(first_row / kBwdBM);
    count = int(last_row / kBwdBM - first_row / kBwdBM + 1);
}

// Status bits the kernels OR into the plan's device status word.
enum : int { kStatusTimeout = 1, kStatusBounds = 2 };

struct FwdParams {
    const int4* items;
    const int32_t* cta_off;
    const int32_t* q_off;
    const int32_t* kv_off;
    int H;
    int mode;       // jfa_mode
    int causal;
    int window;     // sliding window W (>= 0), or -1
    float scale;        // multiplies <q,k>
    float scale_log2;   // scale * log2(e)
    const float* bias;  // [H,32] fp32 or nullptr
    void* O;
    float* lse;         // [T_q,H] or nullptr (GDPA)
    int* status;
    // Dense per-pair bias [H, n_pairs] (sequence b's block row-major [q_len, kv_len] from
    // pair_off[b]), or nullptr.
    const float* dense = nullptr;
    const int64_t* pair_off = nullptr;
    int64_t n_pairs = 0;
    // Shared key/value: kv_map[b] is query set b's key/value sequence (its user), whose
    // rows are kv_off[u] .. kv_off[u+1]; nullptr: sequence b's own.
    const int32_t* kv_map = nullptr;
    int n_seq = 0;  // query sequences (entries of q_off minus one)
    int n_kv = 0;   // key/value sequences (entries of kv_off minus one)
};

struct BwdParams {
    const int4* items;
    const int32_t* cta_off;
    const int32_t* q_off;
    const int32_t* kv_off;
    int H;
    int mode;
    int causal;
    int window;  // sliding window W (>= 0), or -1
    float scale;
    float scale_log2;
    const float* bias;
    const float* lse;    // [T_q,H] (softmax)
    const float* delta;  // [T_q,H] rowsum(dO*O) (softmax)
    float* dq_acc;       // [T_q,H,D] fp32, zeroed first (fp32 inputs; bf16 inputs on the fused backward)
    void* dQ;            // [T_q,H,D] (bf16 inputs: written by the dQ kernel)
    void* dK;
    void* dV;
    int* status;
    // Partial gradients of the relative-position bias table, or nullptr: bf16 inputs
    // [grid][compute warps][H][32], fp32 inputs [work item][32].
    float* dbias_part = nullptr;
    // Dense per-pair bias and its gradient [H, n_pairs] (either may be nullptr), as in
    // FwdParams.
    const float* dense = nullptr;
    float* ddense = nullptr;
    const int64_t* pair_off = nullptr;
    int64_t n_pairs = 0;
    // Shared key/value, as in FwdParams.  The dK/dV pass then works per user key tile:
    // item (u, h, tile, n) visits steps[step_off[g] .. + n), g = ktile_off[u] + tile, each
    // a (query set, query tile) pair.
    const int32_t* kv_map = nullptr;
    const int2* steps = nullptr;
    const int32_t* step_off = nullptr;
    const int32_t* ktile_off = nullptr;
    int n_seq = 0;  // query sequences (entries of q_off minus one)
    int n_kv = 0;   // key/value sequences (entries of kv_off minus one)
};

// Work-item checks.  Every kernel checks each item it reads against the plan before it
// touches anything the item indexes: the sequence, head and tile must lie inside the
// batch and the inner count must be the one the tile ranges give.  The planner never
// writes an item that fails; a kernel that meets one skips it (every role of the CTA
// takes the same decision from the same item) and sets kStatusBounds, which
// jfa_plan_device_status reports as JFA_ERR_DEVICE_BOUNDS.
__device__ inline bool fwd_item_ok(const int4 w, const FwdParams& p, int window) {
    if (w.x < 0 || w.x >= p.n_seq || w.y < 0 || w.y >= p.H || w.z < 0 || w.w < 0) return false;
    const int kb = p.kv_map ? p.kv_map[w.x] : w.x;
    if (kb < 0 || kb >= p.n_kv) return false;
    const int q_len = p.q_off[w.x + 1] - p.q_off[w.x], kv_len = p.kv_off[kb + 1] - p.kv_off[kb];
    if (int64_t(w.z) * kFwdPairRows >= int64_t(q_len)) return false;
    int f0, ns, na, nb;
    pair_stream(q_len, kv_len, w.z, p.causal, window, f0, ns, na, nb);
    return w.w == ns;
}

// dQ pass: query tile w.z of sequence w.x, visiting the forward's key-tile range.
__device__ inline bool dq_item_ok(const int4 w, const BwdParams& p) {
    if (w.x < 0 || w.x >= p.n_seq || w.y < 0 || w.y >= p.H || w.z < 0 || w.w < 0) return false;
    const int kb = p.kv_map ? p.kv_map[w.x] : w.x;
    if (kb < 0 || kb >= p.n_kv) return false;
    const int q_len = p.q_off[w.x + 1] - p.q_off[w.x], kv_len = p.kv_off[kb + 1] - p.kv_off[kb];
    if (int64_t(w.z) * kFwdBM >= int64_t(q_len)) return false;
    return w.w == fwd_tiles_of(q_len, kv_len, w.z, p.causal, p.window);
}

// dK/dV pass: key tile w.z of sequence w.x (shared key/value: of user w.x, visiting the
// steps the planner listed for it).
__device__ inline bool kv_item_ok(const int4 w, const BwdParams& p, bool shared) {
    if (w.x < 0 || w.x >= p.n_kv || w.y < 0 || w.y >= p.H || w.z < 0 || w.w < 0) return false;
    if (shared) {
        if (w.z >= p.ktile_off[w.x + 1] - p.ktile_off[w.x]) return false;
        const int g = p.ktile_off[w.x] + w.z;
        return w.w == p.step_off[g + 1] - p.step_off[g];
    }
    if (w.x >= p.n_seq) return false;
    const int q_len = p.q_off[w.x + 1] - p.q_off[w.x], kv_len = p.kv_off[w.x + 1] - p.kv_off[w.x];
    if (int64_t(w.z) * kBwdBN >= int64_t(kv_len)) return false;
    int first, n;
    query_tile_range(q_len, kv_len, w.z, p.causal, p.window, first, n);
    return w.w == n;
}

// Short-query backward: item (sequence w.x, head w.y, 0, key tiles of the sequence) of a
// sequence with at most bq query rows (no shared key/value, no causal mask or window).
__device__ inline bool short_item_ok(const int4 w, const BwdParams& p, int bq) {
    if (w.x < 0 || w.x >= p.n_seq || w.x >= p.n_kv || w.y < 0 || w.y >= p.H || w.z != 0 || w.w < 0) return false;
    const int q_len = p.q_off[w.x + 1] - p.q_off[w.x], kv_len = p.kv_off[w.x + 1] - p.kv_off[w.x];
    if (q_len > bq) return false;
    return w.w == (kv_len + kBwdBN - 1) / kBwdBN;
}

// Short-query GDPA forward: the same items, checked against the forward's parameters.
__device__ inline bool short_fwd_item_ok(const int4 w, const FwdParams& p, int bq) {
    if (w.x < 0 || w.x >= p.n_seq || w.x >= p.n_kv || w.y < 0 || w.y >= p.H || w.z != 0 || w.w < 0) return false;
    const int q_len = p.q_off[w.x + 1] - p.q_off[w.x], kv_len = p.kv_off[w.x + 1] - p.kv_off[w.x];
    if (q_len > bq) return false;
    return w.w == (kv_len + kFwdBN - 1) / kFwdBN;
}

// Host planner (plan.cpp).  Returns JFA_OK or an error for bad offsets.
jfa_status validate_offsets(const int32_t* q_off, const int32_t* kv_off, int32_t B);
int64_t count_items(const int32_t* q_off, const int32_t* kv_off, int32_t B, int32_t H,
                    int32_t causal, int32_t pass);
void build_worklist(const int32_t* q_off, const int32_t* kv_off, int32_t B, int32_t H,
                    int32_t causal, int32_t window, int32_t pass, int32_t n_ctas, WorkItem* items,
                    int32_t* cta_off, int64_t* cta_cost);

void build_shared_kv_dkdv(const int32_t* q_off, const int32_t* u_off, const int32_t* kv_index, int32_t B,
                          int32_t U, int32_t H, int32_t causal, int32_t window, int32_t n_ctas, WorkItem* items,
                          int32_t* cta_off, std::vector<int2>* steps, std::vector<int32_t>* step_off,
                          std::vector<int32_t>* ktile_off);
int64_t count_shared_kv_dkdv_items(const int32_t* u_off, int32_t U, int32_t H);
bool prefer_split_forward(const int32_t* q_off, const int32_t* kv_off, int32_t B, int32_t causal, int32_t window);

int64_t sequence_cost(int64_t q_len, int64_t kv_len, int32_t H, int32_t causal, int32_t window);
void partition_users(const int32_t* q_off, const int32_t* u_off, const int32_t* kv_index, int32_t B, int32_t U,
                     int32_t H, int32_t causal, int32_t window, int32_t n_parts, int32_t* part_of_user,
                     int64_t* part_cost);
void partition_sequences(const int32_t* q_off, const int32_t* kv_off, int32_t B, int32_t H, int32_t causal,
                         int32_t window, int32_t n_parts, int32_t* part_of_seq, int64_t* part_cost);

// Kernel launchers (fwd.cu, bwd.cu, bwd_dq.cu).  Return cudaSuccess or the launch error.
cudaError_t launch_fwd(int dtype, int o_dtype, int D, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const FwdParams& p, int grid, bool split_list, cudaStream_t st);
cudaError_t launch_bwd_pre(int dtype, int o_dtype, int D, const void* O, const void* dO, float* delta,
                           float* dq_acc, int64_t Tq, int H, int mode, cudaStream_t st);
cudaError_t launch_bwd_main(int dtype, int D, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const CUtensorMap& tmdO, const BwdParams& p,
                            int grid, cudaStream_t st);
cudaError_t launch_bwd_dq(int dtype, int D, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, const CUtensorMap& tmdO, const BwdParams& p,
                          int grid, cudaStream_t st);
cudaError_t launch_bwd_post(int dtype, int D, const float* dq_acc, void* dQ, int64_t Tq, int H,
                            float scale, cudaStream_t st);
// bf16 inputs, fused backward (bwd_fused.cu): dK, dV and the key tile's part of dQ, added
// into the fp32 accumulator (zeroed first; tmDQ: its [T_q, H*D] view in 32 x 32 boxes,
// 128-byte swizzle) for launch_bwd_post to scale and convert.  tmDK, tmDV: the [T_kv, H*D]
// bf16 outputs in 32-row x 64-column boxes, 128-byte swizzle (stores of whole boxes).
cudaError_t launch_bwd_fused(int D, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const CUtensorMap& tmdO, const CUtensorMap& tmDQ, const CUtensorMap& tmDK,
                             const CUtensorMap& tmDV, const BwdParams& p, int grid, cudaStream_t st);
// bf16 inputs, short-query backward (bwd_short.cu): dQ, dK and dV in one kernel over
// (sequence, head) items of plans whose query sets have at most bq (64 or 128) rows.
// tmDK, tmDV: the [T_kv, H*D] bf16 outputs in 32 x 32 boxes, 64-byte swizzle (stores).
cudaError_t launch_bwd_short(int D, int bq, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const CUtensorMap& tmdO, const CUtensorMap& tmDK, const CUtensorMap& tmDV,
                             const BwdParams& p, int grid, cudaStream_t st);
// CTAs of that kernel an SM holds (2 at D = 64 with 64-row query tiles), 0 if unsupported.
int short_ctas_per_sm(int D, int bq);
// bf16 inputs, GDPA modes, short-query forward (fwd_short.cu): O over the same (sequence,
// head) items and grid as launch_bwd_short, scores formed transposed (keys on the lanes).
cudaError_t launch_fwd_short(int o_dtype, int D, int bq, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                             const CUtensorMap& tmV, const FwdParams& p, int grid, cudaStream_t st);
int short_fwd_ctas_per_sm(int D, int bq);
// bf16 inputs, softmax, head_dim 64, query sets of at most 64 rows (fwd_pack.cu): the
// short-query forward with two key tiles per score tile, one CTA per SM.
cudaError_t launch_fwd_pack(int o_dtype, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const FwdParams& p, int grid, cudaStream_t st);
// Query-tile rows of the short-query backward for a plan (0: the form does not apply):
// every query set fits one tile, no shared key/value, no causal mask, no window.
int short_query_rows(const int32_t* q_off, int32_t B, int32_t D, int32_t causal, int32_t window, bool shared_kv);
// Whether jfa_bwd on bf16 inputs runs the fused backward for this plan (without a dense
// bias or a bias gradient): plans whose dK/dV items visit at most kFusedMaxMeanSteps
// query tiles on average (not shared key/value plans), unless the caller asked for the
// deterministic two-pass backward.  On GB300 the fused kernel measured faster on the
// short-sequence workloads (1 to 4 query tiles per key tile) and 1.2x slower on 32K-token
// causal sequences (about 90).
constexpr int64_t kFusedMaxMeanSteps = 6;
inline bool fused_backward(const jfa_plan_t* plan);

// fp32 element type: CUDA-core kernels, one CTA per work item (f32.cu).
cudaError_t launch_fwd_f32(int D, const void* Q, const void* K, const void* V, const FwdParams& p, int64_t n_items,
                           cudaStream_t st);
// Sums the partial table gradients in a fixed order into dbias [H][32]: slots of
// [n_slots][H][32] (bf16 path), or items' [n_items][32] partials by their head (fp32).
cudaError_t launch_dbias_reduce(const float* part, int64_t n_slots, int H, float* dbias, cudaStream_t st);
cudaError_t launch_dbias_reduce_items(const float* part, const int4* items, int64_t n_items, int H, float* dbias,
                                      cudaStream_t st);
cudaError_t launch_bwd_f32(int D, const void* Q, const void* K, const void* V, const void* dO, const BwdParams& p,
                           int64_t n_items, cudaStream_t st);

bool supported(int dtype, int D);

}  // namespace jfa

struct jfa_plan_t {
    int32_t B, H, D, mode, causal, window;
    int32_t U;        // key/value sequences (users with shared key/value; else B)
    bool shared_kv;   // query set b attends to user d_kv_map[b]
    int64_t Tq, Tkv;
    int device, num_sms;
    std::vector<int32_t> q_off, kv_off;   // host copies
    // one device allocation holding everything below
    void* dev_block;
    int32_t* d_q_off;
    int32_t* d_kv_off;
    int* d_status;
    int4* d_fwd_items;
    int32_t* d_fwd_cta_off;
    int4* d_bwd_items;
    int32_t* d_bwd_cta_off;
    int4* d_dq_items;
    int32_t* d_dq_cta_off;
    int64_t* d_pair_off;  // [B+1] first (query, key) pair of each sequence, for a dense bias
    int64_t n_pairs;      // sum over sequences of q_len * kv_len
    // shared key/value (nullptr otherwise): map [B], dK/dV steps and their offsets
    int32_t* d_kv_map;
    int2* d_steps;
    int32_t* d_step_off;
    int32_t* d_ktile_off;
    int64_t n_steps;
    // shared key/value without causal masking or a window: the merged view (runs of
    // consecutive query sets of one user as one query sequence), owned by this plan
    jfa_plan_t* merged = nullptr;
    int64_t n_fwd_items, n_bwd_items, n_dq_items;
    int fwd_grid, bwd_grid, dq_grid;
    bool fwd_split;  // forward kernel with split items (prefer_split_forward)
    bool deterministic = false;  // jfa_plan_set_deterministic: the two-pass bf16 backward
    bool fused_pref = false;     // the planner's choice of the fused bf16 backward
    // short-query backward: query-tile rows (0: not applicable) and its work list
    int short_bq = 0;
    int64_t n_short_items = 0;
    int short_grid = 1;
    int4* d_short_items = nullptr;
    int32_t* d_short_cta_off = nullptr;
    // the short-query forward's list: the same items, grouped for its own grid
    int short_fwd_grid = 1;
    int4* d_sfwd_items = nullptr;
    int32_t* d_sfwd_cta_off = nullptr;
    // optional per-kernel timing (jfa_plan_set_timing)
    bool timing;
    std::vector<cudaEvent_t> ev_pool;                 // reusable events
    std::vector<std::pair<int, std::pair<cudaEvent_t, cudaEvent_t>>> ev_pending;  // kind, (start, stop)
};

namespace jfa {
// Whether jfa_fwd on bf16 inputs with this bias runs a short-query forward: the transposed
// GDPA kernel, or for softmax at head_dim 64 with query sets of at most 64 rows the kernel
// with two key tiles per score tile.
inline bool short_forward(const jfa_plan_t* plan, int32_t bias_kind) {
    return plan->short_bq > 0 && bias_kind == JFA_BIAS_NONE &&
           (plan->mode != JFA_SOFTMAX || (plan->D == 64 && plan->short_bq == 64));
}
// Whether jfa_bwd on bf16 inputs with this bias (and no bias gradient) runs the
// short-query backward.
inline bool short_backward(const jfa_plan_t* plan, int32_t bias_kind, bool dbias) {
    return !plan->deterministic && plan->short_bq > 0 && bias_kind == JFA_BIAS_NONE && !dbias;
}
}  // namespace jfa

inline bool jfa::fused_backward(const jfa_plan_t* plan) {
    return !plan->deterministic && (plan->fused_pref || (plan->merged && plan->merged->fused_pref));
}
