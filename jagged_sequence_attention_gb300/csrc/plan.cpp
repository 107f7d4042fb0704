// Host planner: turns jagged offsets into LPT-balanced work lists for the
// persistent kernels.
//
// Once padding is gone, the GEM articles note that tile scheduling and load balance
// become the bottleneck (vibekk.com GEM article, section 第一轮瓶颈迁移: short sequences
// finish early, long ones keep computing; aihot.vn article, "Jagged Sequence Flash
// Attention": padding-free kernels otherwise leave SMs idle).  Each (sequence, head,
// tile) is costed by the tensor-core products it issues.  Items are listed group by group --
// a group is one (sequence, head), the largest groups first and, inside a group, the
// costliest tiles first -- and each item goes to the CTA with the least accumulated
// cost (greedy list scheduling).  Greedy assignment keeps every CTA within one item
// of the least loaded one, and because CTAs then run their items in list order, the
// tiles in flight at any moment belong to a few groups: their K/V (forward, dQ) or
// Q and dO rows (dK/dV) stay in L2 instead of being re-read from HBM.
#include <algorithm>
#include <cstring>
#include <numeric>
#include <queue>
#include <utility>
#include <vector>

#include "jfa_internal.h"

namespace jfa {

jfa_status validate_offsets(const int32_t* q_off, const int32_t* kv_off, int32_t B) {
    if (B < 0 || !q_off || !kv_off) return JFA_ERR_INVALID_ARG;
    if (q_off[0] != 0 || kv_off[0] != 0) return JFA_ERR_INVALID_ARG;
    for (int32_t b = 0; b < B; ++b) {
        if (q_off[b + 1] < q_off[b] || kv_off[b + 1] < kv_off[b]) return JFA_ERR_INVALID_ARG;
    }
    return JFA_OK;
}

namespace {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Costed {
    WorkItem w;
    int64_t cost;
};

void build_items(const int32_t* q_off, const int32_t* kv_off, int32_t B, int32_t H,
                 int32_t causal, int32_t window, int32_t pass, std::vector<Costed>* out) {
    for (int32_t b = 0; b < B; ++b) {
        const int64_t q_len = q_off[b + 1] - q_off[b];
        const int64_t kv_len = kv_off[b + 1] - kv_off[b];
        if (pass == 0) {
            // Forward: one item per pair of 128-row query tiles; each tile visits its
            // key-tile range (causal: up to the diagonal of its last row; window: from
            // its first row's lowest key), and the item streams the union of the two.
            const int64_t np = ceil_div(q_len, kFwdPairRows);
            for (int32_t h = 0; h < H; ++h)
                for (int64_t t = 0; t < np; ++t) {
                    int first, n, na, nb;
                    pair_stream(q_len, kv_len, t, causal, window, first, n, na, nb);
                    out->push_back({{b, h, int32_t(t), int32_t(n)}, 2 * (int64_t(na) + nb) + 2});
                }
        } else if (pass == kPassBwdKV) {
            // Backward dK/dV: one item per key tile (also when it sees no query, so
            // that its dK/dV rows are written); it visits its query-tile range, four
            // products each.
            const int64_t nt = ceil_div(kv_len, kBwdBN);
            for (int32_t h = 0; h < H; ++h)
                for (int64_t t = 0; t < nt; ++t) {
                    int first, n;
                    query_tile_range(q_len, kv_len, t, causal, window, first, n);
                    out->push_back({{b, h, int32_t(t), int32_t(n)}, 4 * int64_t(n) + 2});
                }
        } else if (pass == kPassBwdShort) {
            // Short-query backward: one item per (sequence, head) with a query or a key,
            // visiting all of the sequence's key tiles, five products each (a sequence
            // without queries only has its dK/dV rows zeroed).
            if (q_len == 0 && kv_len == 0) continue;
            const int64_t n = ceil_div(kv_len, kBwdBN);
            for (int32_t h = 0; h < H; ++h)
                out->push_back({{b, h, 0, int32_t(n)}, (q_len > 0 ? 5 * n : n) + 2});
        } else {
            // Backward dQ: one item per 128-row query tile (also when it sees no key, so
            // that its dQ rows are written); it visits the forward's key-tile range, three
            // products each.
            const int64_t nt = ceil_div(q_len, kFwdBM);
            for (int32_t h = 0; h < H; ++h)
                for (int64_t t = 0; t < nt; ++t) {
                    const int64_t n = fwd_tiles_of(q_len, kv_len, t, causal, window);
                    out->push_back({{b, h, int32_t(t), int32_t(n)}, 3 * n + 2});
                }
        }
    }
}

}  // namespace

int64_t count_items(const int32_t* q_off, const int32_t* kv_off, int32_t B, int32_t H,
                    int32_t causal, int32_t pass) {
    (void)causal;
    int64_t n = 0;
    if (pass == kPassBwdShort) {
        for (int32_t b = 0; b < B; ++b)
            if (q_off[b + 1] > q_off[b] || kv_off[b + 1] > kv_off[b]) n += H;
        return n;
    }
    for (int32_t b = 0; b < B; ++b) {
        const int64_t len = pass == kPassBwdKV ? kv_off[b + 1] - kv_off[b] : q_off[b + 1] - q_off[b];
        const int64_t tile = pass == kPassFwd ? kFwdPairRows : pass == kPassBwdKV ? kBwdBN : kFwdBM;
        n += ceil_div(len, tile) * H;
    }
    return n;
}

namespace {

// Group-major LPT assignment of costed items (groups: (item.b, item.h), n_groups_b
// values of item.b) to n_ctas CTAs; writes the items in CTA order.
void assign_lpt(std::vector<Costed>& all, int32_t n_groups_b, int32_t H, int32_t n_ctas, WorkItem* items,
                int32_t* cta_off, int64_t* cta_cost) {
    const int32_t B = n_groups_b;
    // Group-major order: groups by total cost (largest first, ties by sequence and
    // head), then items by cost inside the group; the sort is stable so equal keys
    // keep (sequence, head, tile) order and the plan is deterministic.
    std::vector<int64_t> group_cost(size_t(B) * size_t(H), 0);
    for (const Costed& c : all) group_cost[size_t(c.w.b) * size_t(H) + size_t(c.w.h)] += c.cost;
    auto gkey = [&](const Costed& c) { return size_t(c.w.b) * size_t(H) + size_t(c.w.h); };
    std::stable_sort(all.begin(), all.end(), [&](const Costed& a, const Costed& b) {
        const size_t ga = gkey(a), gb = gkey(b);
        if (ga != gb) {
            if (group_cost[ga] != group_cost[gb]) return group_cost[ga] > group_cost[gb];
            return ga < gb;
        }
        return a.cost > b.cost;
    });

    // Greedy: each item goes to the currently least-loaded CTA (ties: lowest index).
    using Slot = std::pair<int64_t, int32_t>;
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int32_t c = 0; c < n_ctas; ++c) heap.push({0, c});
    std::vector<int32_t> owner(all.size());
    std::vector<int64_t> load(size_t(n_ctas), 0);
    std::vector<int32_t> count(size_t(n_ctas), 0);
    for (size_t i = 0; i < all.size(); ++i) {
        Slot s = heap.top();
        heap.pop();
        owner[i] = s.second;
        s.first += all[i].cost;
        load[size_t(s.second)] = s.first;
        count[size_t(s.second)]++;
        heap.push(s);
    }
    cta_off[0] = 0;
    for (int32_t c = 0; c < n_ctas; ++c) cta_off[c + 1] = cta_off[c] + count[size_t(c)];
    std::vector<int32_t> cursor(cta_off, cta_off + n_ctas);
    for (size_t i = 0; i < all.size(); ++i) items[cursor[size_t(owner[i])]++] = all[i].w;
    if (cta_cost)
        for (int32_t c = 0; c < n_ctas; ++c) cta_cost[c] = load[size_t(c)];
}

}  // namespace

void build_worklist(const int32_t* q_off, const int32_t* kv_off, int32_t B, int32_t H,
                    int32_t causal, int32_t window, int32_t pass, int32_t n_ctas, WorkItem* items,
                    int32_t* cta_off, int64_t* cta_cost) {
    std::vector<Costed> all;
    all.reserve(size_t(count_items(q_off, kv_off, B, H, causal, pass)));
    build_items(q_off, kv_off, B, H, causal, window, pass, &all);
    assign_lpt(all, B, H, n_ctas, items, cta_off, cta_cost);
}

// Shared key/value (in-kernel broadcast): query set b attends to user kv_index[b]'s
// rows.  The dK/dV pass works per user key tile; its steps are the (query set, query
// tile) pairs of all the user's query sets that see the tile, listed per (user, key
// tile) in steps[step_off[g]..step_off[g+1]), g = ktile_off[u] + tile (shared by the
// heads).  Items are (u, h, tile, step count), costed and assigned as above.
void build_shared_kv_dkdv(const int32_t* q_off, const int32_t* u_off, const int32_t* kv_index, int32_t B,
                          int32_t U, int32_t H, int32_t causal, int32_t window, int32_t n_ctas, WorkItem* items,
                          int32_t* cta_off, std::vector<int2>* steps, std::vector<int32_t>* step_off,
                          std::vector<int32_t>* ktile_off) {
    std::vector<std::vector<int32_t>> cands(size_t(U > 0 ? U : 0));
    for (int32_t b = 0; b < B; ++b) cands[size_t(kv_index[b])].push_back(b);
    ktile_off->assign(size_t(U) + 1, 0);
    for (int32_t u = 0; u < U; ++u)
        (*ktile_off)[size_t(u) + 1] = (*ktile_off)[size_t(u)] + int32_t(ceil_div(u_off[u + 1] - u_off[u], kBwdBN));
    step_off->assign(size_t((*ktile_off)[size_t(U)]) + 1, 0);
    steps->clear();
    std::vector<Costed> all;
    for (int32_t u = 0; u < U; ++u) {
        const int64_t kv_len = u_off[u + 1] - u_off[u];
        const int64_t nt = ceil_div(kv_len, kBwdBN);
        for (int64_t t = 0; t < nt; ++t) {
            const size_t g = size_t((*ktile_off)[size_t(u)] + t);
            for (int32_t b : cands[size_t(u)]) {
                int first, n;
                query_tile_range(q_off[b + 1] - q_off[b], kv_len, t, causal, window, first, n);
                for (int k = 0; k < n; ++k) steps->push_back(make_int2(b, first + k));
            }
            (*step_off)[g + 1] = int32_t(steps->size());
            const int32_t n = (*step_off)[g + 1] - (*step_off)[g];
            for (int32_t h = 0; h < H; ++h) all.push_back({{u, h, int32_t(t), n}, 4 * int64_t(n) + 2});
        }
    }
    assign_lpt(all, U, H, n_ctas, items, cta_off, nullptr);
}

// The forward's split items (fwd_split_item): a pair holding a single query tile that
// visits two key tiles or more has no second tile to overlap its softmax with, so the
// kernel splits its key range into two halves run as if they were the two tiles of a
// pair and merges the halves' (max, sum, O) at the end.  The plan picks the kernel with
// split items when one-tile sequences' split items carry at least half the forward's
// products, or when a longer sequence's last tile has a long key range to split (on the
// long causal workload that kernel ran its forward 47.1 -> 46.7 ms).  The sliding-window
// forward has no split form.
bool prefer_split_forward(const int32_t* q_off, const int32_t* kv_off, int32_t B, int32_t causal, int32_t window) {
    if (window >= 0) return false;
    int64_t split = 0, total = 0;  // products of one-tile sequences' split items, of all items
    bool long_split = false;        // a longer sequence's last tile is split
    for (int32_t b = 0; b < B; ++b) {
        const int64_t q_len = q_off[b + 1] - q_off[b];
        const int64_t kv_len = kv_off[b + 1] - kv_off[b];
        const int64_t np = ceil_div(q_len, kFwdPairRows);
        for (int64_t t = 0; t < np; ++t) {
            int first, n, na, nb;
            pair_stream(q_len, kv_len, t, causal, window, first, n, na, nb);
            const int64_t c = 2 * (int64_t(na) + nb) + 2;
            total += c;
            if (fwd_split_item(q_len, t, na)) {
                if (q_len <= kFwdBM)
                    split += c;
                else
                    long_split = true;
            }
        }
    }
    return (split > 0 && 2 * split >= total) || long_split;
}

// The short-query backward keeps a whole query set in one tile of 64 or 128 rows and its
// dQ in TMEM across the key tiles.  Its TMEM budget (S^T, dP^T/dV, dK and dQ columns)
// fits a 64-row tile at head_dim 64 in 256 columns, so two CTAs share an SM; other
// tiles take all 512.
int short_query_rows(const int32_t* q_off, int32_t B, int32_t D, int32_t causal, int32_t window, bool shared_kv) {
    if (shared_kv || causal || window >= 0 || (D != 64 && D != 128)) return 0;
    int32_t max_q = 0;
    for (int32_t b = 0; b < B; ++b) max_q = std::max(max_q, q_off[b + 1] - q_off[b]);
    if (max_q == 0) return 0;
    if (D == 64 && max_q <= 64) return 64;
    return max_q <= 128 ? 128 : 0;
}

int64_t count_shared_kv_dkdv_items(const int32_t* u_off, int32_t U, int32_t H) {
    int64_t n = 0;
    for (int32_t u = 0; u < U; ++u) n += ceil_div(u_off[u + 1] - u_off[u], kBwdBN) * H;
    return n;
}

// Data-parallel split of a batch: sequences are independent problems, so a batch
// shards across GPUs with no exchange.  Each sequence is costed by the tensor-core
// products its forward and backward issue over all heads (two forward, four dK/dV and
// three dQ products per visited 128x128 score tile, plus a per-tile constant), and the
// sequences go longest-first to the least loaded part (greedy LPT, ties to the lower
// part and the lower sequence index, so the result is deterministic).
int64_t sequence_cost(int64_t q_len, int64_t kv_len, int32_t H, int32_t causal, int32_t window) {
    const int64_t nq = ceil_div(q_len, kFwdBM), nk = ceil_div(kv_len, kBwdBN);
    int64_t tiles = 0;
    for (int64_t t = 0; t < nq; ++t) tiles += fwd_tiles_of(q_len, kv_len, t, causal, window);
    return int64_t(H) * (9 * tiles + 2 * (nq + nk));
}

void partition_sequences(const int32_t* q_off, const int32_t* kv_off, int32_t B, int32_t H, int32_t causal,
                         int32_t window, int32_t n_parts, int32_t* part_of_seq, int64_t* part_cost) {
    std::vector<std::pair<int64_t, int32_t>> order(size_t(B > 0 ? B : 0));
    for (int32_t b = 0; b < B; ++b)
        order[size_t(b)] = {sequence_cost(q_off[b + 1] - q_off[b], kv_off[b + 1] - kv_off[b], H, causal, window), b};
    std::stable_sort(order.begin(), order.end(),
                     [](const std::pair<int64_t, int32_t>& a, const std::pair<int64_t, int32_t>& b) {
                         return a.first > b.first;
                     });
    using Slot = std::pair<int64_t, int32_t>;
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int32_t c = 0; c < n_parts; ++c) heap.push({0, c});
    std::vector<int64_t> load(size_t(n_parts), 0);
    for (const auto& o : order) {
        Slot sl = heap.top();
        heap.pop();
        part_of_seq[o.second] = sl.second;
        sl.first += o.first;
        load[size_t(sl.second)] = sl.first;
        heap.push(sl);
    }
    if (part_cost)
        for (int32_t c = 0; c < n_parts; ++c) part_cost[c] = load[size_t(c)];
}

// Shared key/value batches split by user: a user's query sets all go with it, so each
// user's dK and dV are summed on one GPU and no exchange is needed.  A user's cost is
// that of its query sets (as above, with the user's key/value length) plus the zero
// rows of its key tiles; greedy LPT as above.
void partition_users(const int32_t* q_off, const int32_t* u_off, const int32_t* kv_index, int32_t B, int32_t U,
                     int32_t H, int32_t causal, int32_t window, int32_t n_parts, int32_t* part_of_user,
                     int64_t* part_cost) {
    std::vector<int64_t> cost(size_t(U > 0 ? U : 0), 0);
    for (int32_t u = 0; u < U; ++u) cost[size_t(u)] = int64_t(H) * 2 * ceil_div(u_off[u + 1] - u_off[u], kBwdBN);
    for (int32_t b = 0; b < B; ++b) {
        const int32_t u = kv_index[b];
        const int64_t q_len = q_off[b + 1] - q_off[b], kv_len = u_off[u + 1] - u_off[u];
        const int64_t nq = ceil_div(q_len, kFwdBM);
        int64_t tiles = 0;
        for (int64_t t = 0; t < nq; ++t) tiles += fwd_tiles_of(q_len, kv_len, t, causal, window);
        cost[size_t(u)] += int64_t(H) * (9 * tiles + 2 * nq);
    }
    std::vector<std::pair<int64_t, int32_t>> order(size_t(U > 0 ? U : 0));
    for (int32_t u = 0; u < U; ++u) order[size_t(u)] = {cost[size_t(u)], u};
    std::stable_sort(order.begin(), order.end(),
                     [](const std::pair<int64_t, int32_t>& a, const std::pair<int64_t, int32_t>& b) {
                         return a.first > b.first;
                     });
    using Slot = std::pair<int64_t, int32_t>;
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int32_t c = 0; c < n_parts; ++c) heap.push({0, c});
    std::vector<int64_t> load(size_t(n_parts), 0);
    for (const auto& o : order) {
        Slot sl = heap.top();
        heap.pop();
        part_of_user[o.second] = sl.second;
        sl.first += o.first;
        load[size_t(sl.second)] = sl.first;
        heap.push(sl);
    }
    if (part_cost)
        for (int32_t c = 0; c < n_parts; ++c) part_cost[c] = load[size_t(c)];
}

}  // namespace jfa
