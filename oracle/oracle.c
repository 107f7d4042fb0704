/*
 * Oracle for jagged attention: the plain, slow, fp64 CPU definition.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the test-suite, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant with the CUDA
 * library: it is written from the definition of the operation, one
 * (sequence, head) row at a time, with no tiling, no online softmax and no
 * reordering beyond what the definition states.
 *
 * What it computes (sources: the GEM training-efficiency articles):
 *  - "Jagged Sequence Flash Attention" (aihot.vn GEM article, that section;
 *    vibekk.com GEM article, section 第一轮瓶颈迁移 and FAQ "Jagged tensor 是什么"):
 *    a jagged tensor is packed values plus offsets; jagged attention is, for every
 *    sequence b and head h, ordinary attention over that sequence's own query and
 *    key/value rows only.  Query and key/value lengths may differ, and a custom
 *    additive bias applies to the scores.
 *  - "Generalized Dot-Product Attention (GDPA)" (aihot.vn GEM article, that
 *    section): two matrix products with an elementwise activation (GELU or SiLU)
 *    between them in place of softmax; no row normalisation.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - causal alignment is bottom-right: key j is allowed for query i iff
 *    j <= i + (kv_len - q_len);
 *  - the bias is a per-head table of 32 relative-position buckets,
 *    r = |i + (kv_len - q_len) - j|, bucket(r) = min(31, floor(log2((1+r)^2)));
 *  - sliding window (aihot.vn GEM article, section "BlockAttention": each token
 *    limited to its neighbouring events, O(L * window) work): with window W >= 0,
 *    key j is allowed for query i only if j >= i + (kv_len - q_len) - W, i.e. the
 *    aligned position itself and the W keys before it (together with the causal
 *    bound); W < 0 means no window;
 *  - a query row with no allowed key gives o = 0 and lse = -inf, and all
 *    gradients through it are 0;
 *  - besides the bucket table, a dense per-pair bias may be given (the "custom
 *    attention bias" of the aihot.vn GEM article, section "Jagged Sequence Flash
 *    Attention", in its most general form): one value per (head, sequence, query
 *    row, key row), stored head-major as [H, P] with P = sum_b q_len_b * kv_len_b,
 *    sequence b's block starting at pair_off[b] = sum_{b' < b} q_len_b' * kv_len_b'
 *    and laid out row-major [q_len_b, kv_len_b] inside it.  Both biases add to the
 *    score; the dense value of a masked pair is never read;
 *  - the gradient of a bias is that of the score it adds to: d bias_dense[h, (i, j)]
 *    = ds_ij at allowed pairs (0 at masked ones), and d table[h, k] = sum of ds_ij
 *    over the allowed pairs whose relative position falls in bucket k;
 *  - GDPA masked entries contribute exactly 0 (the activation is never evaluated
 *    on them); GELU is the tanh form of Hendrycks and Gimpel (2016), SiLU is
 *    x * sigmoid(x).
 *
 * Layout: values are [T, H, D] row-major fp64 (token-major), offsets int32[B+1].
 * Parallelism: OpenMP over independent (sequence, head) pairs only.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_SOFTMAX = 0, ORACLE_GELU_TANH = 1, ORACLE_SILU = 2 };

/* floor(log2((1+r)^2)), capped at 31: count how many times the square can be
 * halved (integer division) before it drops below 2. */
int oracle_relpos_bucket(int64_t r)
{
    if (r < 0) r = -r;
    uint64_t v = (uint64_t)(1 + r) * (uint64_t)(1 + r);
    int k = 0;
    while (v >= 2) {
        v /= 2;
        k++;
    }
    return k < 31 ? k : 31;
}

/* GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))). */
static double gelu_tanh(double x)
{
    const double c = sqrt(2.0 / M_PI);
    return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
}

/* d/dx of the tanh-form GELU, by the product and chain rules. */
static double gelu_tanh_grad(double x)
{
    const double c = sqrt(2.0 / M_PI);
    double u = c * (x + 0.044715 * x * x * x);
    double t = tanh(u);
    double du = c * (1.0 + 3.0 * 0.044715 * x * x);
    return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * du;
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static double silu(double x) { return x * sigmoid(x); }

/* d/dx x*sigmoid(x) = sigmoid(x) + x*sigmoid(x)*(1-sigmoid(x)). */
static double silu_grad(double x)
{
    double sg = sigmoid(x);
    return sg + x * sg * (1.0 - sg);
}

double oracle_act(int mode, double x)
{
    if (mode == ORACLE_GELU_TANH) return gelu_tanh(x);
    if (mode == ORACLE_SILU) return silu(x);
    return NAN;
}

double oracle_act_grad(int mode, double x)
{
    if (mode == ORACLE_GELU_TANH) return gelu_tanh_grad(x);
    if (mode == ORACLE_SILU) return silu_grad(x);
    return NAN;
}

/* Score s_ij = scale * <q_i, k_j> + bias[h, bucket(|i + kv_len - q_len - j|)]
 *              + dense_h_b[i * kv_len + j]. */
static double score(const double *qi, const double *kj, int D, double scale,
                    const double *bias_h, const double *dense_hb, int64_t i, int64_t j,
                    int64_t q_len, int64_t kv_len)
{
    double dot = 0.0;
    for (int d = 0; d < D; d++) dot += qi[d] * kj[d];
    double s = scale * dot;
    if (bias_h) s += bias_h[oracle_relpos_bucket(i + (kv_len - q_len) - j)];
    if (dense_hb) s += dense_hb[i * kv_len + j];
    return s;
}

/* First pair of sequence b in a dense per-pair array: sum of q_len * kv_len before b. */
static int64_t pair_offset(const int32_t *q_off, const int32_t *kv_off, int b)
{
    int64_t acc = 0;
    for (int c = 0; c < b; c++)
        acc += ((int64_t)q_off[c + 1] - q_off[c]) * ((int64_t)kv_off[c + 1] - kv_off[c]);
    return acc;
}

/* P = sum_b q_len_b * kv_len_b: the number of (query, key) pairs of the batch. */
int64_t oracle_num_pairs(int B, const int32_t *q_off, const int32_t *kv_off)
{
    return pair_offset(q_off, kv_off, B);
}

static int allowed(int causal, int window, int64_t i, int64_t j, int64_t q_len, int64_t kv_len)
{
    const int64_t ip = i + (kv_len - q_len);  /* the query's aligned key position */
    if (causal && j > ip) return 0;
    if (window >= 0 && j < ip - window) return 0;
    return 1;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Forward.  O[T_q, H, D]; LSE[T_q, H] (softmax: log of the row's partition
 * function, -inf for a row with no allowed key; GDPA: 0).
 * bias: [H, 32] or NULL; dense: [H, P] per-pair bias or NULL.
 * Returns 0, or -1 on an allocation failure.
 */
int oracle_fwd(int B, int H, int D, const int32_t *q_off, const int32_t *kv_off,
               const double *Q, const double *K, const double *V, int mode, int causal,
               int window, const double *bias, const double *dense, double scale, double *O,
               double *LSE, int nthreads)
{
    int failed = 0;
    const int64_t P = oracle_num_pairs(B, q_off, kv_off);
    set_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; b++) {
        for (int h = 0; h < H; h++) {
            const int64_t q0 = q_off[b], q_len = (int64_t)q_off[b + 1] - q_off[b];
            const int64_t k0 = kv_off[b], kv_len = (int64_t)kv_off[b + 1] - kv_off[b];
            const double *bias_h = bias ? bias + (int64_t)h * 32 : NULL;
            const double *dense_hb = dense ? dense + (int64_t)h * P + pair_offset(q_off, kv_off, b) : NULL;
            double *s = (double *)malloc(sizeof(double) * (size_t)(kv_len > 0 ? kv_len : 1));
            if (!s) {
#pragma omp atomic write
                failed = 1;
                continue;
            }
            for (int64_t i = 0; i < q_len; i++) {
                const double *qi = Q + ((q0 + i) * H + h) * D;
                double *oi = O + ((q0 + i) * H + h) * D;
                double *lse = LSE + (q0 + i) * H + h;
                for (int d = 0; d < D; d++) oi[d] = 0.0;

                double m = -INFINITY;
                int64_t n_allowed = 0;
                for (int64_t j = 0; j < kv_len; j++) {
                    if (!allowed(causal, window, i, j, q_len, kv_len)) continue;
                    s[j] = score(qi, K + ((k0 + j) * H + h) * D, D, scale, bias_h, dense_hb, i, j, q_len, kv_len);
                    if (s[j] > m) m = s[j];
                    n_allowed++;
                }
                if (mode == ORACLE_SOFTMAX) {
                    if (n_allowed == 0) {
                        *lse = -INFINITY;
                        continue;
                    }
                    double l = 0.0;
                    for (int64_t j = 0; j < kv_len; j++)
                        if (allowed(causal, window, i, j, q_len, kv_len)) l += exp(s[j] - m);
                    for (int64_t j = 0; j < kv_len; j++) {
                        if (!allowed(causal, window, i, j, q_len, kv_len)) continue;
                        double p = exp(s[j] - m) / l;
                        const double *vj = V + ((k0 + j) * H + h) * D;
                        for (int d = 0; d < D; d++) oi[d] += p * vj[d];
                    }
                    *lse = m + log(l);
                } else {
                    for (int64_t j = 0; j < kv_len; j++) {
                        if (!allowed(causal, window, i, j, q_len, kv_len)) continue;
                        double a = oracle_act(mode, s[j]);
                        const double *vj = V + ((k0 + j) * H + h) * D;
                        for (int d = 0; d < D; d++) oi[d] += a * vj[d];
                    }
                    *lse = 0.0;
                }
            }
            free(s);
        }
    }
    return failed ? -1 : 0;
}

/*
 * Backward of L = sum(O * dO) through the forward above.
 *   dv_j  = sum_i p_ij do_i
 *   dp_ij = <do_i, v_j>
 *   ds_ij = p_ij (dp_ij - sum_k p_ik dp_ik)   (softmax)
 *   ds_ij = act'(s_ij) dp_ij                  (GDPA, p_ij = act(s_ij))
 *   dq_i  = scale sum_j ds_ij k_j,   dk_j = scale sum_i ds_ij q_i
 *   d_dense[h, (i, j)] = ds_ij,       dbias[h, k] = sum of ds_ij with bucket(r_ij) = k
 * Each (sequence, head) pair owns its rows of dQ, dK and dV and its block of d_dense.
 * dbias [H, 32] and d_dense [H, P] are optional outputs (NULL: not computed); the
 * table's gradient is summed over sequences in sequence order after the parallel
 * loop, from one partial table per (sequence, head).
 */
int oracle_bwd(int B, int H, int D, const int32_t *q_off, const int32_t *kv_off,
               const double *Q, const double *K, const double *V, const double *dO, int mode,
               int causal, int window, const double *bias, const double *dense, double scale,
               double *dQ, double *dK, double *dV, double *dbias, double *d_dense, int nthreads)
{
    int failed = 0;
    const int64_t P = oracle_num_pairs(B, q_off, kv_off);
    double *dbias_part = NULL;
    if (dbias) {
        dbias_part = (double *)calloc((size_t)(B > 0 ? B : 1) * (size_t)H * 32, sizeof(double));
        if (!dbias_part) return -1;
    }
    set_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; b++) {
        for (int h = 0; h < H; h++) {
            const int64_t q0 = q_off[b], q_len = (int64_t)q_off[b + 1] - q_off[b];
            const int64_t k0 = kv_off[b], kv_len = (int64_t)kv_off[b + 1] - kv_off[b];
            const double *bias_h = bias ? bias + (int64_t)h * 32 : NULL;
            const int64_t pb = pair_offset(q_off, kv_off, b);
            const double *dense_hb = dense ? dense + (int64_t)h * P + pb : NULL;
            double *d_dense_hb = d_dense ? d_dense + (int64_t)h * P + pb : NULL;
            double *dbias_bh = dbias_part ? dbias_part + ((int64_t)b * H + h) * 32 : NULL;
            if (d_dense_hb)
                for (int64_t e = 0; e < q_len * kv_len; e++) d_dense_hb[e] = 0.0;
            size_t n = (size_t)(kv_len > 0 ? kv_len : 1);
            double *s = (double *)malloc(sizeof(double) * n);
            double *p = (double *)malloc(sizeof(double) * n);
            double *dp = (double *)malloc(sizeof(double) * n);
            if (!s || !p || !dp) {
                free(s);
                free(p);
                free(dp);
#pragma omp atomic write
                failed = 1;
                continue;
            }
            for (int64_t j = 0; j < kv_len; j++) {
                double *dkj = dK + ((k0 + j) * H + h) * D;
                double *dvj = dV + ((k0 + j) * H + h) * D;
                for (int d = 0; d < D; d++) dkj[d] = dvj[d] = 0.0;
            }
            for (int64_t i = 0; i < q_len; i++) {
                const double *qi = Q + ((q0 + i) * H + h) * D;
                const double *doi = dO + ((q0 + i) * H + h) * D;
                double *dqi = dQ + ((q0 + i) * H + h) * D;
                for (int d = 0; d < D; d++) dqi[d] = 0.0;

                double m = -INFINITY;
                int64_t n_allowed = 0;
                for (int64_t j = 0; j < kv_len; j++) {
                    if (!allowed(causal, window, i, j, q_len, kv_len)) continue;
                    s[j] = score(qi, K + ((k0 + j) * H + h) * D, D, scale, bias_h, dense_hb, i, j, q_len, kv_len);
                    if (s[j] > m) m = s[j];
                    n_allowed++;
                }
                if (n_allowed == 0) continue;
                if (mode == ORACLE_SOFTMAX) {
                    double l = 0.0;
                    for (int64_t j = 0; j < kv_len; j++)
                        if (allowed(causal, window, i, j, q_len, kv_len)) l += exp(s[j] - m);
                    for (int64_t j = 0; j < kv_len; j++)
                        p[j] = allowed(causal, window, i, j, q_len, kv_len) ? exp(s[j] - m) / l : 0.0;
                } else {
                    for (int64_t j = 0; j < kv_len; j++)
                        p[j] = allowed(causal, window, i, j, q_len, kv_len) ? oracle_act(mode, s[j]) : 0.0;
                }
                double delta = 0.0;
                for (int64_t j = 0; j < kv_len; j++) {
                    if (!allowed(causal, window, i, j, q_len, kv_len)) {
                        dp[j] = 0.0;
                        continue;
                    }
                    const double *vj = V + ((k0 + j) * H + h) * D;
                    double acc = 0.0;
                    for (int d = 0; d < D; d++) acc += doi[d] * vj[d];
                    dp[j] = acc;
                    delta += p[j] * dp[j];
                }
                for (int64_t j = 0; j < kv_len; j++) {
                    if (!allowed(causal, window, i, j, q_len, kv_len)) continue;
                    double ds;
                    if (mode == ORACLE_SOFTMAX)
                        ds = p[j] * (dp[j] - delta);
                    else
                        ds = oracle_act_grad(mode, s[j]) * dp[j];
                    if (d_dense_hb) d_dense_hb[i * kv_len + j] = ds;
                    if (dbias_bh) dbias_bh[oracle_relpos_bucket(i + (kv_len - q_len) - j)] += ds;
                    const double *kj = K + ((k0 + j) * H + h) * D;
                    double *dkj = dK + ((k0 + j) * H + h) * D;
                    double *dvj = dV + ((k0 + j) * H + h) * D;
                    for (int d = 0; d < D; d++) {
                        dqi[d] += scale * ds * kj[d];
                        dkj[d] += scale * ds * qi[d];
                        dvj[d] += p[j] * doi[d];
                    }
                }
            }
            free(s);
            free(p);
            free(dp);
        }
    }
    if (dbias) {
        for (int64_t e = 0; e < (int64_t)H * 32; e++) dbias[e] = 0.0;
        for (int b = 0; b < B; b++)
            for (int64_t e = 0; e < (int64_t)H * 32; e++) dbias[e] += dbias_part[(int64_t)b * H * 32 + e];
        free(dbias_part);
    }
    return failed ? -1 : 0;
}
