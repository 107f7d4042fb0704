/*
 * libjfa -- Jagged Flash Attention and GDPA for GB300 (sm_103a).
 *
 * The operation (GEM training-efficiency article, aihot.vn, section "Jagged
 * Sequence Flash Attention"; vibekk.com GEM article, FAQ "Jagged tensor 是什么"):
 * attention computed directly on jagged tensors -- packed values plus offsets --
 * with no padding, where every sequence b attends only within itself.  Query and
 * key/value lengths may differ per sequence ("asymmetric query/key-value
 * lengths"), an additive per-head bias may apply ("custom attention bias"), and the
 * backward pass is provided.  The GDPA mode (same article, section "Generalized
 * Dot-Product Attention (GDPA)") replaces softmax by an elementwise GELU or SiLU
 * with no row normalisation.
 *
 * For sequence b, head h, query row i (0-based within the sequence), key row j:
 *   s_ij   = scale * <q_i, k_j> + bias[h, bucket(|i + (kv_len - q_len) - j|)]
 *   allowed(i, j) = (!causal || j <= i') && (W < 0 || j >= i' - W),  i' = i + (kv_len - q_len)
 *                   (bottom-right causal; optional sliding window of W keys before i')
 *   SOFTMAX: o_i = sum_j softmax_j(s_ij) v_j over allowed j;  lse_i = log sum exp s_ij
 *   GDPA:    o_i = sum_j act(s_ij) v_j over allowed j, act = tanh-GELU or SiLU
 *   bucket(r) = min(31, floor(log2((1 + r)^2)))   (exact integer arithmetic)
 * A row with no allowed key gets o = 0 (and lse = -inf); its gradients are 0.
 *
 * Layout and conventions (all calls):
 *  - Q, O, dO, dQ are [T_q, H, D] row-major (token-major), T_q = q_offsets[B];
 *    K, V, dK, dV are [T_kv, H, D], T_kv = kv_offsets[B].  Contiguous, 16-byte
 *    aligned DEVICE pointers owned by the caller.  lse is fp32 [T_q, H].
 *  - Element type: JFA_BF16 (bfloat16, head_dim 64 or 128; tensor-core products)
 *    or JFA_F32 (float, head_dim 32 or 64; plain fp32 arithmetic on the CUDA cores,
 *    no TF32 rounding).  Accumulation is fp32.
 *  - Values must be finite: a key/value row of a neighbouring sequence is read
 *    (and multiplied by an exact zero weight) at jagged tile edges.
 *  - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy default
 *    stream).  jfa_plan_create (which uploads the work lists), jfa_plan_destroy,
 *    jfa_plan_device_status and jfa_plan_kernel_times synchronise; jfa_fwd and
 *    jfa_bwd never do.
 *  - Every call returns a jfa_status; argument errors are detected on the host
 *    before anything is launched.  No call aborts the process.
 *  - A plan is not thread-safe: do not use one plan from two host threads at once.
 */
#ifndef JFA_H
#define JFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    JFA_OK = 0,
    JFA_ERR_INVALID_ARG = 1,    /* null pointer, bad offsets, misaligned pointer, bad size */
    JFA_ERR_UNSUPPORTED = 2,    /* head_dim / dtype / mode combination not built */
    JFA_ERR_CUDA = 3,           /* a CUDA runtime or driver call failed */
    JFA_ERR_TIMEOUT = 4,        /* a kernel pipeline wait exceeded its limit (device status) */
    JFA_ERR_DEVICE_BOUNDS = 5,  /* a kernel's own bounds check fired (device status) */
    JFA_ERR_PLAN_MISMATCH = 6,  /* the call does not match the plan (mode, head_dim) */
    JFA_ERR_NO_DEVICE = 7,      /* no usable sm_100-family GPU */
    JFA_ERR_SCRATCH_LIMIT = 8   /* the problem needs more scratch than JFA_STATIC_SCRATCH_BYTES */
} jfa_status;

typedef enum { JFA_SOFTMAX = 0, JFA_GDPA_GELU_TANH = 1, JFA_GDPA_SILU = 2 } jfa_mode;
typedef enum { JFA_BF16 = 0, JFA_F32 = 1 } jfa_dtype;
/* JFA_BIAS_RELPOS32: a per-head table [H, 32] indexed by bucket(relative position).
 * JFA_BIAS_DENSE: one fp32 value per (head, sequence, query row, key row), the most
 *   general form of the article's "custom attention bias": [H, P] head-major, with
 *   P = sum_b q_len_b * kv_len_b (jfa_plan_info fact 15).  Sequence b's block starts at
 *   pair_off[b] = sum_{b' < b} q_len_b' * kv_len_b' within each head's row and is
 *   row-major [q_len_b, kv_len_b]: the pair (i, j) is at h * P + pair_off[b] + i * kv_len_b
 *   + j.  Values of masked pairs are never read.  Meant for short sequences: it moves
 *   4 bytes per pair (and 4 more for its gradient), where the table moves none. */
typedef enum { JFA_BIAS_NONE = 0, JFA_BIAS_RELPOS32 = 1, JFA_BIAS_DENSE = 2 } jfa_bias_kind;

typedef struct jfa_plan_t* jfa_plan;

/*
 * Builds the work lists for one batch shape (the planner): validates offsets,
 * splits every (sequence, head) into query tiles (forward, backward dQ) and
 * key/value tiles (backward dK/dV), costs each tile by the tensor-core products it
 * issues (causal tiles stop at the diagonal), and assigns them longest-first to the least loaded
 * CTA of a persistent grid, so that short sequences never leave SMs idle while a
 * long one finishes (the article's point that padding-free kernels otherwise idle
 * SMs when short sequences end early).
 *   q_offsets, kv_offsets: int32[B+1], non-decreasing, offsets[0] == 0; host
 *     pointers, or device pointers when offsets_on_device != 0 (then copied to the
 *     host on `stream`).  Copied; the caller keeps ownership.
 *   The plan's device memory (offsets, work lists, status word) is allocated here
 *   and uploaded on `stream`, which this call synchronises.
 *   B >= 0 sequences, H >= 1 heads, D head_dim, mode a jfa_mode, causal 0/1.
 *   out: receives a library-owned plan; free with jfa_plan_destroy.
 * Errors: INVALID_ARG (bad offsets or sizes), UNSUPPORTED (D not 32/64/128),
 * NO_DEVICE, CUDA.
 */
jfa_status jfa_plan_create(const int32_t* q_offsets, const int32_t* kv_offsets, int32_t B,
                           int32_t H, int32_t D, int32_t mode, int32_t causal,
                           int32_t offsets_on_device, void* stream, jfa_plan* out);

/*
 * jfa_plan_create with a sliding window (aihot.vn GEM article, section
 * "BlockAttention": each token limited to its neighbouring events, O(L * window)
 * work): with window W >= 0, query i attends only to keys i' - W <= j <= i', where
 * i' = i + (kv_len - q_len) is its aligned causal position; the kernels skip every
 * tile outside the band.  window = -1 is jfa_plan_create.  A window requires causal
 * = 1.  Errors: those of jfa_plan_create; INVALID_ARG for window < -1 or a window
 * without causal.
 */
jfa_status jfa_plan_create_ex(const int32_t* q_offsets, const int32_t* kv_offsets, int32_t B,
                              int32_t H, int32_t D, int32_t mode, int32_t causal, int32_t window,
                              int32_t offsets_on_device, void* stream, jfa_plan* out);

/*
 * Shared key/value attention: the in-kernel broadcast (IKBO) of the PyTorch blog
 * "In-Kernel Broadcast Optimization: Co-Designing Kernels for RecSys Inference",
 * section 3 "IKBO Flash Attention" and figure 1.  Many candidate query sets of a
 * request attend to the same user history, and the kernels read each user's keys and
 * values once per use instead of from a copy made per query set.
 *   Query set b (rows q_offsets[b] .. q_offsets[b+1] of Q, O, dO, dQ) attends to the
 *   rows of user u = kv_index[b], kv_offsets[u] .. kv_offsets[u+1] of K and V.  The
 *   results are those of jfa_fwd / jfa_bwd on the broadcast batch, with each query set
 *   holding its own copy of its user's rows.  dK and dV of a user's rows sum over all
 *   of its query sets, and are zero for a user that no query set uses.
 *   kv_offsets: int32[U+1] over the users (T_kv = kv_offsets[U]); kv_index: int32[B],
 *   each in [0, U).  Host arrays, or device arrays with offsets_on_device (copied to the
 *   host on `stream`, which this call synchronises).
 *   Causal alignment, the sliding window and the bias use each query set's q_len and
 *   its user's kv_len, as in jfa_plan_create_ex.  A dense bias (JFA_BIAS_DENSE) has one
 *   block per query set, q_len_b x kv_len_{kv_index[b]}.
 *   Planning: the forward and dQ passes work per query set, reading its user's rows.
 *   The dK/dV pass works per user key tile over the query tiles of all of that user's
 *   query sets, so dK and dV accumulate on chip and each user row is written once.
 *   Without causal masking or a window, a row's result does not depend on which query
 *   set it belongs to, except through the relative-position table.  The plan then
 *   also holds a merged view: each run of consecutive query sets of one user is one
 *   query sequence, so short query sets fill whole 128-row tiles.  Calls use it unless
 *   they pass JFA_BIAS_RELPOS32.  Query sets of a user placed next to each other in Q
 *   thus share tiles.
 *   jfa_plan_info fact 16 is U.
 *   The other calls take the plan as usual.  jfa_worklist_* and
 *   jfa_partition_sequences describe plain batches only; jfa_partition_users splits a
 *   shared key/value batch.
 * Errors: INVALID_ARG for bad offsets or an index outside [0, U); otherwise those of
 * jfa_plan_create_ex.
 */
jfa_status jfa_plan_create_shared_kv(const int32_t* q_offsets, int32_t B, const int32_t* kv_offsets,
                                     int32_t U, const int32_t* kv_index, int32_t H, int32_t D,
                                     int32_t mode, int32_t causal, int32_t window,
                                     int32_t offsets_on_device, void* stream, jfa_plan* out);

/* Frees a plan and its device memory (cudaFree synchronises the device, so launches
 * still using the plan finish first).  NULL is accepted. */
jfa_status jfa_plan_destroy(jfa_plan plan);

/*
 * Plan facts for callers and tests, written to info[0..n): T_q, T_kv, B, H, D,
 * mode, causal, forward work items, forward grid, backward dK/dV work items, its
 * grid, SM count, backward dQ work items, its grid, window (-1: none), P, the number
 * of (query, key) pairs sum_b q_len_b * kv_len_b, the number of users U of a
 * shared key/value plan (-1 for other plans), and the number of merged query sequences
 * of a shared key/value plan's merged view (-1 when it has none; see
 * jfa_plan_create_shared_kv), and 1 when the forward runs the kernel with split items
 * (sequences of one query tile whose key range is split in two halves that are merged
 * at the end; chosen when such items carry at least half the forward's tensor-core
 * products and the plan has no window), else 0, and 1 when jfa_bwd on JFA_BF16 inputs
 * (without a dense bias or a bias gradient) may run the fused backward, in which every
 * key tile also adds its part of dQ into an fp32 accumulator held in the workspace, else
 * 0.  The planner chooses the fused form when the backward's key tiles visit few query
 * tiles on average (short sequences), unless jfa_plan_set_deterministic chose the
 * two-pass form; see jfa_plan_set_deterministic.  Fact 20 is the query-tile rows (64 or
 * 128) of the short-query backward when jfa_bwd on JFA_BF16 inputs without a bias runs
 * it for this plan, else 0: one kernel per (sequence, head) for batches whose query sets
 * all fit one tile, with no causal mask, window or shared key/value (it then takes the
 * place of the fused form for calls without a bias).  Fact 21 is the same query-tile rows
 * when jfa_fwd on JFA_BF16 inputs without a bias runs a short-query forward for this plan,
 * else 0: in GDPA modes the scores formed transposed, with the keys on the tensor-core
 * accumulator's lanes; in SOFTMAX mode (head_dim 64, query sets of at most 64 rows) two key
 * tiles per score tile, one per half of the lanes.  Either way short query sets leave no
 * lane on padding rows.  n may be smaller than 22.
 */
jfa_status jfa_plan_info(jfa_plan plan, int64_t* info, int32_t n);

/*
 * Forward pass.
 *   Q [T_q,H,D], K, V [T_kv,H,D] (dtype); bias_table fp32 [H,32] when bias_kind is
 *   JFA_BIAS_RELPOS32, the dense bias fp32 [H,P] when it is JFA_BIAS_DENSE (see
 *   jfa_bias_kind), else ignored; scale multiplies <q,k> (typically 1/sqrt(D)); in
 *   SOFTMAX mode it must be finite and positive (the kernels bound each row's maximum by
 *   scale times the row's largest raw score), else INVALID_ARG.
 *   O [T_q,H,D] is written for every row covered by the offsets, in o_dtype:
 *   JFA_F32 (the fp32 accumulator, no output rounding) or JFA_BF16 (rounded to
 *   nearest even); with dtype JFA_F32, o_dtype must be JFA_F32.
 *   lse fp32 [T_q,H]: written in SOFTMAX mode (natural log, -inf for a row with
 *   no allowed key) and required there; ignored and may be NULL in GDPA modes.
 * Errors: INVALID_ARG, UNSUPPORTED, PLAN_MISMATCH, CUDA (launch failure).
 */
jfa_status jfa_fwd(jfa_plan plan, int32_t dtype, const void* Q, const void* K, const void* V,
                   int32_t bias_kind, const float* bias_table, float scale, void* O, int32_t o_dtype,
                   float* lse, void* stream);

/* Bytes of device workspace jfa_bwd needs for this plan and dtype: fp32 row terms
 * [T_q,H], and an fp32 dQ accumulator [T_q,H,D] for JFA_F32 and for plans whose bf16
 * backward may be fused (jfa_plan_info fact 19); 0 on a bad plan. */
size_t jfa_bwd_workspace_size(jfa_plan plan, int32_t dtype);

/*
 * Backward pass of L = sum(O * dO) for the forward with the same arguments.
 *   O (in o_dtype) and lse are the forward's outputs (both ignored in GDPA modes);
 *   dO is the upstream gradient [T_q,H,D] (dtype).  Writes dQ [T_q,H,D], dK, dV
 *   [T_kv,H,D] (dtype).
 *   workspace: caller-owned device memory of at least jfa_bwd_workspace_size bytes,
 *   256-byte aligned; its contents need not be initialised and are clobbered.
 * Errors: INVALID_ARG (incl. too small a workspace), UNSUPPORTED, PLAN_MISMATCH,
 * CUDA.
 */
jfa_status jfa_bwd(jfa_plan plan, int32_t dtype, const void* Q, const void* K, const void* V,
                   const void* O, int32_t o_dtype, const void* dO, const float* lse,
                   int32_t bias_kind, const float* bias_table, float scale, void* dQ, void* dK,
                   void* dV, void* workspace, size_t workspace_bytes, void* stream);

/*
 * jfa_bwd that also returns the gradient of the bias (the article's "custom attention
 * bias", aihot.vn GEM article, section "Jagged Sequence Flash Attention", made
 * trainable): a bias adds to the score, so its gradient is dS,
 *   ds_ij = p_ij (dp_ij - sum_l p_il dp_il) (softmax) or act'(s_ij) dp_ij (GDPA).
 * For the table of JFA_BIAS_RELPOS32, entry (h, k) receives the sum of ds_ij over the
 * allowed pairs (i, j) of head h, in every sequence, whose relative position falls in
 * bucket k:
 *   dbias[h, k] = sum_{b, i, j allowed, bucket(|i + kv_len - q_len - j|) = k} ds_ij.
 * For JFA_BIAS_DENSE, dbias has the dense bias's layout [H, P] and receives ds_ij at
 * every allowed pair and 0 at every masked one.
 *   dbias: fp32 device pointer, [H, 32] or [H, P] by bias_kind, 4-byte aligned,
 *     caller-owned; overwritten (not accumulated into).  NULL makes the call exactly
 *     jfa_bwd.  Requires bias_kind JFA_BIAS_RELPOS32 or JFA_BIAS_DENSE (the gradient
 *     is taken at the given bias).
 *   workspace: at least jfa_bwd_ex_workspace_size(plan, dtype, bias_kind) bytes when
 *     dbias is set (jfa_bwd_workspace_size otherwise), 256-byte aligned.
 *   The result is the same on every run: each CTA and warp sums its part in a fixed
 *   order, and a last kernel adds the parts in a fixed order.
 * Errors: those of jfa_bwd; INVALID_ARG for a dbias with bias_kind JFA_BIAS_NONE, a
 * misaligned dbias or too small a workspace.
 */
size_t jfa_bwd_ex_workspace_size(jfa_plan plan, int32_t dtype, int32_t bias_kind);
jfa_status jfa_bwd_ex(jfa_plan plan, int32_t dtype, const void* Q, const void* K, const void* V,
                      const void* O, int32_t o_dtype, const void* dO, const float* lse,
                      int32_t bias_kind, const float* bias_table, float scale, void* dQ, void* dK,
                      void* dV, float* dbias, void* workspace, size_t workspace_bytes, void* stream);

/* Size of the library-held scratch array that jfa_bwd_static_scratch uses on each
 * GPU (64 MiB).  A plan fits when jfa_bwd_workspace_size(plan, dtype) is at most
 * this.  With an fp32 dQ accumulator in the scratch (JFA_F32, and JFA_BF16 on a fused
 * backward) that is T_q * H up to about 130,000 (token, head) rows at head_dim 128 and
 * 258,000 at head_dim 64; with row terms alone (shared key/value plans on JFA_BF16),
 * about 16.7 million. */
#define JFA_STATIC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * jfa_bwd without a caller-supplied workspace, for callers that cannot allocate
 * device memory at all.  Examples are a host program whose device buffers are all
 * handed to it by another runtime, or one whose device memory is entirely reserved
 * by a pool at start-up, where one more cudaMalloc fails or defeats the pool.  The
 * paper has no counterpart to this call; it exists only for such callers.
 *   Arguments, layout, results and asynchrony are those of jfa_bwd.  The scratch is
 *   the library's own JFA_STATIC_SCRATCH_BYTES device array, which every GPU that
 *   loads the library holds until the process exits.  This call allocates nothing:
 *   no cudaMalloc, no cudaFree, no allocating library routine.  The plan's timing
 *   hook, when a caller has switched it on, creates CUDA events as it does for
 *   jfa_bwd; it is off by default.
 *   Set-up: the first call in a CUDA context (normally the device's primary
 *   context, made current by cudaSetDevice) looks up the array's device address
 *   and keeps it, keyed by the context's unique id, for later calls in that
 *   context.  A new context -- the primary context re-created after
 *   cudaDeviceReset, or a caller's own driver-API context -- gets a fresh look-up,
 *   and the array's contents do not survive a reset.  The look-up can load the
 *   library's module on the device, so make the first call in each context before
 *   any stream capture.
 *   Every call on a device uses the same array.  A call rewrites the row terms
 *   held there before reading them.  Where the scratch holds a dQ accumulator
 *   (JFA_F32, and JFA_BF16 on a fused backward) it also clears that on its stream
 *   before adding anything in.  So no call depends on
 *   what an earlier call left there.  Calls that may overlap on the GPU race on the
 *   array and corrupt each other's gradients: order them on one stream, or by
 *   events.
 *   The current device must be the plan's device.
 * Errors: SCRATCH_LIMIT when jfa_bwd_workspace_size(plan, dtype) exceeds
 * JFA_STATIC_SCRATCH_BYTES (checked before anything is launched); PLAN_MISMATCH
 * when another device is current; CUDA if the address look-up fails; otherwise
 * those of jfa_bwd.
 */
jfa_status jfa_bwd_static_scratch(jfa_plan plan, int32_t dtype, const void* Q, const void* K,
                                  const void* V, const void* O, int32_t o_dtype, const void* dO,
                                  const float* lse, int32_t bias_kind, const float* bias_table,
                                  float scale, void* dQ, void* dK, void* dV, void* stream);

/*
 * The bf16 backward has three forms (the articles leave the backward's accumulation open;
 * see jfa_bwd):
 *   fused: one kernel over key tiles forms dK, dV and each key tile's part of dQ, adding
 *     the parts into an fp32 accumulator in the workspace with reduce-adds at L2, and a
 *     conversion pass writes dQ.  The order of the additions varies from run to run, so
 *     dQ can differ in its last bit between runs; dK and dV do not.
 *   two-pass: a second kernel over query tiles recomputes S and dP and accumulates dQ
 *     on chip, with no atomics: every result is the same bit for bit on every run, at
 *     1.4x the tensor-core work of the backward.
 *   short-query: when every query set fits one tile of 64 or 128 rows (64 at head_dim
 *     64) and the plan has no causal mask, window or shared key/value, and the call has no
 *     bias: one kernel per (sequence, head) keeps the query set on chip while the key
 *     tiles stream past, and sums dQ in TMEM.  No atomics: the same bits on every run.
 * By default (enable = 0) the planner picks the faster form for the batch: short-query
 * where it applies; else fused when the key tiles visit few query tiles on average (short
 * sequences, where it saves the second pass); two-pass otherwise (long sequences, where
 * the reduce-adds cost more than the recomputation).  enable = 1 always runs the two-pass
 * form.  Shared key/value plans
 * (unless their merged view is used), a dense bias and bias gradients always run the
 * two-pass form.  The choice changes jfa_bwd_workspace_size (the fused backward needs the
 * fp32 accumulator); query it after this call.  jfa_plan_info facts 19 and 20 report the
 * form.
 * fp32 inputs are unaffected.
 * Errors: INVALID_ARG for a null plan or enable not 0 or 1.
 */
jfa_status jfa_plan_set_deterministic(jfa_plan plan, int32_t enable);

/*
 * Test hook for the kernels' own checks (not a counterpart of anything in the articles).
 * Every kernel checks each work item it reads against the plan -- sequence, head and
 * tile inside the batch, inner count equal to the one the tile ranges give -- before it
 * touches anything the item indexes.  It skips an item that fails and sets the status
 * that jfa_plan_device_status reports as JFA_ERR_DEVICE_BOUNDS.  The planner never writes
 * such an item; this call overwrites work item `index` of a pass (0 forward, 1 backward
 * dK/dV, 2 backward dQ, 3 the short-query backward, 4 the short-query forward; numbering as
 * jfa_plan_info facts 7, 9, 12, and for passes 3 and 4 as jfa_worklist_build's pass 3 on the
 * plan's offsets, grouped for each kernel's own grid) in the plan's device
 * memory so that a test can plant one.  The lists are the plan's own (a shared key/value
 * plan's merged view keeps its lists).  Synchronises.  A plan holding a changed item gives
 * wrong results for that item's rows until it is destroyed.
 *   item: int32[4] (sequence, head, tile, inner count), host memory.
 * Errors: INVALID_ARG for a bad pass, an index outside the list or a null pointer; CUDA.
 */
jfa_status jfa_plan_set_work_item(jfa_plan plan, int32_t pass, int64_t index, const int32_t* item);

/* Synchronises `stream`, then reads and clears the plan's device status word, which
 * the kernels set when a pipeline wait times out (TIMEOUT) or a bounds check fires
 * (DEVICE_BOUNDS).  Returns JFA_OK when no kernel reported anything. */
jfa_status jfa_plan_device_status(jfa_plan plan, void* stream);

/* Host-only planner, usable without a GPU (the same code jfa_plan_create runs).
 * pass 0 = forward (pairs of 128-row query tiles), 1 = backward dK/dV (key/value
 * tiles of 128 rows, visiting 128-row query tiles), 2 = backward dQ (128-row query
 * tiles), 3 = the short-query backward (one item (sequence, head, 0, key tiles) per
 * sequence with a query or a key; causal must be 0 and window -1).  jfa_worklist_size
 * gives the number of work items; jfa_worklist_build writes items as int32 quadruples
 * (sequence, head, tile index, inner tiles visited) grouped by CTA, cta_offsets[n_ctas+1]
 * delimiting each CTA's items, and optionally each CTA's total cost in units of
 * tensor-core products.  window as in jfa_plan_create_ex (-1: none).  With a window the
 * inner tiles are a band: a forward pair streams the union of its two query tiles' key
 * ranges.  Errors: INVALID_ARG for bad offsets, H < 1, n_ctas < 1, an unknown pass, or
 * pass 3 with a causal mask or a window. */
jfa_status jfa_worklist_size(const int32_t* q_offsets, const int32_t* kv_offsets, int32_t B,
                             int32_t H, int32_t causal, int32_t window, int32_t pass, int64_t* n_items);
jfa_status jfa_worklist_build(const int32_t* q_offsets, const int32_t* kv_offsets, int32_t B,
                              int32_t H, int32_t causal, int32_t window, int32_t pass, int32_t n_ctas,
                              int32_t* items, int32_t* cta_offsets, int64_t* cta_cost);

/* Data-parallel split, host only (no GPU needed).  Sequences are independent, so a
 * batch shards across GPUs with no exchange (GEM articles: jagged batches with long
 * and short sequences, where balance decides throughput).  Each sequence is costed by
 * the tensor-core products its forward and backward issue over all heads, and the
 * sequences are assigned longest-first to the least loaded of n_parts parts
 * (deterministic: ties go to the lower part and the lower sequence index).
 *   part_of_seq[B] receives each sequence's part; part_cost[n_parts] (may be NULL)
 *   each part's total cost.  The greedy bound holds: the most loaded part exceeds
 *   the least loaded by at most one sequence's cost.
 * window as in jfa_plan_create_ex (-1: none).
 * Errors: INVALID_ARG (bad offsets, H < 1, n_parts < 1, causal not 0/1, a window
 * without causal). */
jfa_status jfa_partition_sequences(const int32_t* q_offsets, const int32_t* kv_offsets, int32_t B,
                                   int32_t H, int32_t causal, int32_t window, int32_t n_parts,
                                   int32_t* part_of_seq, int64_t* part_cost);

/*
 * jfa_partition_sequences for a shared key/value batch (jfa_plan_create_shared_kv):
 * users, each with all of its query sets, split over n_parts GPUs by greedy LPT on
 * their cost, the cost of their query sets plus their key tiles.  A user's dK and dV sum
 * over its query sets, so keeping them together means no GPU exchanges anything.
 *   Host arrays: q_offsets int32[B+1], kv_offsets int32[U+1], kv_index int32[B].
 *   part_of_user: int32[U] out, each in [0, n_parts); part_cost: int64[n_parts] out
 *   (may be NULL).  Deterministic.
 * Errors: INVALID_ARG for bad offsets or sizes, or an index outside [0, U).
 */
jfa_status jfa_partition_users(const int32_t* q_offsets, int32_t B, const int32_t* kv_offsets,
                               int32_t U, const int32_t* kv_index, int32_t H, int32_t causal,
                               int32_t window, int32_t n_parts, int32_t* part_of_user,
                               int64_t* part_cost);

/* Kernel timing for measurement.  With timing enabled, every kernel launch made for
 * this plan is bracketed by a pair of CUDA events recorded on the launch stream.
 * jfa_plan_kernel_times synchronises those events and returns, per kernel kind
 * (0 forward, 1 backward preprocess, 2 backward dK/dV (fp32 inputs: backward main),
 * 3 fp32 dQ conversion, 4 bf16 backward dQ), the summed milliseconds and the number
 * of launches since the previous query, then forgets them.  Timing is off by
 * default; enabling it adds one event record before and after each launch.
 * total_ms and launches point to arrays of 5 (either may be NULL). */
jfa_status jfa_plan_set_timing(jfa_plan plan, int32_t enable);
jfa_status jfa_plan_kernel_times(jfa_plan plan, double* total_ms, int64_t* launches);

/* Static description of a status code. */
const char* jfa_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* JFA_H */
