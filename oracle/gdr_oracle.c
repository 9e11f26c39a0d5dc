/*
 * Oracle for the gated delta rule forward pass -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, double-precision CPU statement of what the GPU path computes.
 * Only the test-suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library.  It shares no code, header, table or helper with the
 * CUDA path (gated_delta_rule_37_gb300/csrc) and includes nothing from it.
 *
 * The recurrence (Gated DeltaNet, one value-head h, state S in R^{V x K},
 * stored V-major S[v][k]):
 *
 *   decay       S~   = exp(g_t) * S_{t-1}        (KDA: S_{t-1} diag(exp(gk_t)))
 *   prediction  kS   = S~ k_t
 *   delta       n_t  = beta_t * (v_t - kS)
 *   update      S_t  = S~ + n_t k_t^T
 *   read        o_t  = scale * S_t q_t           (post-update read)
 *
 * Sources: FlashQLA PR #1 "Fused recurrent GDN decode + SGLang DFlash verify
 * kernel", the "core single-role decode kernel" commit (order decay -> kS ->
 * v_new -> rank-1 -> o, post-update read, raw g without a cumsum) and the
 * design commit (exact single-token recurrence); the paged verify commit of
 * the same page (state_indices gather, slot < 0 skipped, per-token
 * intermediate states, no-commit mode, V-major [num_slots, H, V, K] pool).
 * The value-head -> key-head map h // (Hv/Hk) is the one that page's review
 * commit checks against the h % Hk negative control.
 *
 * Every function runs in fp64 on fp64 copies of the exact input values.
 * Loops are parallel over independent (sequence, value-head) units only.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Negative-control switches (plant a known mistake; tests check it FAILS). */
#define ORACLE_READ_PRE_UPDATE 1 /* o_t = scale * S~ q_t (before the rank-1)   */
#define ORACLE_HEAD_MOD        2 /* key-head = h % Hk instead of h / (Hv/Hk)   */
#define ORACLE_TRANSPOSED      4 /* state read/written K-major instead of V-major */

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int key_head(int h, int Hk, int Hv, int variant) {
    if (variant & ORACLE_HEAD_MOD) return h % Hk;
    return h / (Hv / Hk);
}

/* Load S[v][k] for one (sequence, head) from a [.., V, K] block (or zeros). */
static void load_state(double* S, const double* src, int K, int V, int variant) {
    if (!src) {
        memset(S, 0, sizeof(double) * (size_t)V * K);
        return;
    }
    for (int v = 0; v < V; ++v)
        for (int c = 0; c < K; ++c)
            S[(size_t)v * K + c] = (variant & ORACLE_TRANSPOSED) ? src[(size_t)c * V + v]
                                                                 : src[(size_t)v * K + c];
}

static void store_state(double* dst, const double* S, int K, int V, int variant) {
    for (int v = 0; v < V; ++v)
        for (int c = 0; c < K; ++c) {
            if (variant & ORACLE_TRANSPOSED) dst[(size_t)c * V + v] = S[(size_t)v * K + c];
            else dst[(size_t)v * K + c] = S[(size_t)v * K + c];
        }
}

/*
 * One token of the recurrence on S (in place).  dec[c] = exp(gate) per key
 * channel (all equal for the scalar gate).  Writes o_row[V] (scaled read).
 */
static void token_step(double* S, const double* dec, const double* q, const double* k,
                       const double* vv, double beta, double scale, int K, int V,
                       int variant, double* o_row) {
    for (int v = 0; v < V; ++v) {
        double* row = S + (size_t)v * K;
        double kS = 0.0;
        for (int c = 0; c < K; ++c) {
            row[c] *= dec[c];
            kS += row[c] * k[c];
        }
        double pre = 0.0;
        if (variant & ORACLE_READ_PRE_UPDATE)
            for (int c = 0; c < K; ++c) pre += row[c] * q[c];
        double n = beta * (vv[v] - kS);
        double post = 0.0;
        for (int c = 0; c < K; ++c) {
            row[c] += n * k[c];
            post += row[c] * q[c];
        }
        if (o_row) o_row[v] = scale * ((variant & ORACLE_READ_PRE_UPDATE) ? pre : post);
    }
}

/*
 * Tokenwise prefill over packed variable-length sequences.
 *   q, k   [T, Hk, K]      v, o [T, Hv, V]
 *   g      [T, Hv]  (scalar gate)  or  gk [T, Hv, K] (per-key-channel gate);
 *          exactly one is non-NULL.
 *   beta   [T, Hv]
 *   s0     [N, Hv, V, K] or NULL (zeros);  s_final [N, Hv, V, K] or NULL.
 *   cu     [N+1] sequence boundaries into the packed token axis.
 * Returns 0, or -1 on a malformed argument.
 */
int oracle_tokenwise(const double* q, const double* k, const double* v, const double* g,
                     const double* gk, const double* beta, const double* s0,
                     const int64_t* cu, int N, int Hk, int Hv, int K, int V, double scale,
                     int variant, double* o, double* s_final, int nthreads) {
    if ((g == NULL) == (gk == NULL) || Hk <= 0 || Hv % Hk != 0 || K <= 0 || V <= 0) return -1;
    set_threads(nthreads);
    const int units = N * Hv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int u = 0; u < units; ++u) {
        const int b = u / Hv, h = u % Hv;
        const int kh = key_head(h, Hk, Hv, variant);
        double* S = (double*)malloc(sizeof(double) * (size_t)V * K);
        double* dec = (double*)malloc(sizeof(double) * (size_t)K);
        load_state(S, s0 ? s0 + ((size_t)b * Hv + h) * V * K : NULL, K, V, variant);
        for (int64_t t = cu[b]; t < cu[b + 1]; ++t) {
            for (int c = 0; c < K; ++c)
                dec[c] = exp(gk ? gk[((size_t)t * Hv + h) * K + c] : g[(size_t)t * Hv + h]);
            token_step(S, dec, q + ((size_t)t * Hk + kh) * K, k + ((size_t)t * Hk + kh) * K,
                       v + ((size_t)t * Hv + h) * V, beta[(size_t)t * Hv + h], scale, K, V,
                       variant, o + ((size_t)t * Hv + h) * V);
        }
        if (s_final) store_state(s_final + ((size_t)b * Hv + h) * V * K, S, K, V, variant);
        free(dec);
        free(S);
    }
    return 0;
}

/*
 * Chunked (WY) form of the same recurrence, chunk size C, restarting chunks at
 * every sequence start (the last chunk of a sequence may be partial).  This is
 * the independent second statement used to cross-check the tokenwise form.
 * Within a chunk (local i = 0..L-1, state S0 at chunk start):
 *   gam_i      = sum_{s<=i} g_s                   (per channel for gk)
 *   A_ij       = beta_i sum_c k_i[c] exp(gam_i[c]-gam_j[c]) k_j[c],  j < i
 *   Tm         = (I + A)^{-1}  (unit lower triangular; forward substitution)
 *   W          = Tm diag(beta) (K o exp(Gam))      U = Tm diag(beta) V
 *   Nn         = U - W S0^T                        (rows are the deltas n_i)
 *   O_i        = scale [ S0 (q_i o exp(gam_i)) + sum_{j<=i} (sum_c q_i[c] exp(gam_i[c]-gam_j[c]) k_j[c]) n_j ]
 *   S_L        = S0 diag(exp(gam_L)) + sum_j n_j (k_j o exp(gam_L - gam_j))^T
 * Every exponent is of gam_i - gam_j with i >= j (or of gam_i = gam_i - gam_{-1}),
 * never of a negated prefix.  Sources: the chunked-prefill pieces named on the
 * FlashQLA page (cumsum, A, kkt solve) and the attention-gym PR #344 inter-chunk
 * state kernel (per-chunk state h, v_new, 64-token chunks).
 */
int oracle_chunked(const double* q, const double* k, const double* v, const double* g,
                   const double* gk, const double* beta, const double* s0, const int64_t* cu,
                   int N, int Hk, int Hv, int K, int V, double scale, int C, double* o,
                   double* s_final, int nthreads) {
    if ((g == NULL) == (gk == NULL) || Hk <= 0 || Hv % Hk != 0 || C <= 0) return -1;
    set_threads(nthreads);
    const int units = N * Hv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int u = 0; u < units; ++u) {
        const int b = u / Hv, h = u % Hv;
        const int kh = key_head(h, Hk, Hv, 0);
        double* S = (double*)malloc(sizeof(double) * (size_t)V * K);
        double* gam = (double*)malloc(sizeof(double) * (size_t)C * K);
        double* A = (double*)calloc((size_t)C * C, sizeof(double));
        double* Tm = (double*)calloc((size_t)C * C, sizeof(double));
        double* W = (double*)malloc(sizeof(double) * (size_t)C * K);
        double* U = (double*)malloc(sizeof(double) * (size_t)C * V);
        double* Nn = (double*)malloc(sizeof(double) * (size_t)C * V);
        double* P = (double*)calloc((size_t)C * C, sizeof(double));
        load_state(S, s0 ? s0 + ((size_t)b * Hv + h) * V * K : NULL, K, V, 0);
        for (int64_t cs = cu[b]; cs < cu[b + 1]; cs += C) {
            const int L = (int)((cu[b + 1] - cs) < C ? (cu[b + 1] - cs) : C);
#define QP(i) (q + ((size_t)(cs + (i)) * Hk + kh) * K)
#define KP(i) (k + ((size_t)(cs + (i)) * Hk + kh) * K)
#define VP(i) (v + ((size_t)(cs + (i)) * Hv + h) * V)
#define BT(i) (beta[(size_t)(cs + (i)) * Hv + h])
            /* in-chunk inclusive prefix sum of the gate */
            for (int c = 0; c < K; ++c) {
                double acc = 0.0;
                for (int i = 0; i < L; ++i) {
                    acc += gk ? gk[((size_t)(cs + i) * Hv + h) * K + c] : g[(size_t)(cs + i) * Hv + h];
                    gam[(size_t)i * K + c] = acc;
                }
            }
            /* strictly lower A and the attention-like P (j <= i) */
            for (int i = 0; i < L; ++i)
                for (int j = 0; j < L; ++j) {
                    double a = 0.0, p = 0.0;
                    if (j <= i)
                        for (int c = 0; c < K; ++c) {
                            const double e = exp(gam[(size_t)i * K + c] - gam[(size_t)j * K + c]);
                            a += KP(i)[c] * e * KP(j)[c];
                            p += QP(i)[c] * e * KP(j)[c];
                        }
                    A[(size_t)i * C + j] = (j < i) ? BT(i) * a : 0.0;
                    P[(size_t)i * C + j] = (j <= i) ? p : 0.0;
                }
            /* Tm = (I + A)^{-1} by forward substitution, column by column */
            for (int j = 0; j < L; ++j)
                for (int i = 0; i < L; ++i) {
                    double x = (i == j) ? 1.0 : 0.0;
                    for (int m = 0; m < i; ++m) x -= A[(size_t)i * C + m] * Tm[(size_t)m * C + j];
                    Tm[(size_t)i * C + j] = x;
                }
            /* WY factors */
            for (int i = 0; i < L; ++i) {
                for (int c = 0; c < K; ++c) {
                    double w = 0.0;
                    for (int j = 0; j < L; ++j)
                        w += Tm[(size_t)i * C + j] * BT(j) * exp(gam[(size_t)j * K + c]) * KP(j)[c];
                    W[(size_t)i * K + c] = w;
                }
                for (int e = 0; e < V; ++e) {
                    double uu = 0.0;
                    for (int j = 0; j < L; ++j) uu += Tm[(size_t)i * C + j] * BT(j) * VP(j)[e];
                    U[(size_t)i * V + e] = uu;
                }
            }
            /* deltas n_i = u_i - S0 w_i */
            for (int i = 0; i < L; ++i)
                for (int e = 0; e < V; ++e) {
                    double ws = 0.0;
                    for (int c = 0; c < K; ++c) ws += W[(size_t)i * K + c] * S[(size_t)e * K + c];
                    Nn[(size_t)i * V + e] = U[(size_t)i * V + e] - ws;
                }
            /* output: inter-chunk (from S0) + intra-chunk (from the deltas) */
            for (int i = 0; i < L; ++i) {
                double* orow = o + ((size_t)(cs + i) * Hv + h) * V;
                for (int e = 0; e < V; ++e) {
                    double inter = 0.0, intra = 0.0;
                    for (int c = 0; c < K; ++c)
                        inter += S[(size_t)e * K + c] * QP(i)[c] * exp(gam[(size_t)i * K + c]);
                    for (int j = 0; j <= i; ++j) intra += P[(size_t)i * C + j] * Nn[(size_t)j * V + e];
                    orow[e] = scale * (inter + intra);
                }
            }
            /* state carried to the next chunk */
            for (int e = 0; e < V; ++e)
                for (int c = 0; c < K; ++c) {
                    const double gl = gam[(size_t)(L - 1) * K + c];
                    double s = exp(gl) * S[(size_t)e * K + c];
                    for (int j = 0; j < L; ++j)
                        s += Nn[(size_t)j * V + e] * KP(j)[c] * exp(gl - gam[(size_t)j * K + c]);
                    S[(size_t)e * K + c] = s;
                }
#undef QP
#undef KP
#undef VP
#undef BT
        }
        if (s_final) store_state(s_final + ((size_t)b * Hv + h) * V * K, S, K, V, 0);
        free(S); free(gam); free(A); free(Tm); free(W); free(U); free(Nn); free(P);
    }
    return 0;
}

/*
 * Slot-indexed decode / multi-step verify over a state pool.
 *   g        [T, Hv] scalar log-decay, used when gk is NULL
 *   gk       [T, Hv, K] per-key-channel log-decay, or NULL (the per-channel
 *            decode of tokenspeed PR #834: column c of the state is scaled
 *            by e^{gk[c]} before the delta-rule update, as in the tokenwise
 *            definition above)
 *   pool_in  [num_slots, Hv, V, K]   fp64 copy of the pool as the GPU sees it
 *   pool_out same shape; on entry a copy of pool_in; slot state_idx[b] is
 *            overwritten with the final state when commit != 0
 *   state_idx[N]  pool slot of sequence b; < 0 means padding: nothing of row
 *            b is computed or written (o rows, pool slot, ibuf row untouched)
 *   cu       [N+1]  token range of sequence b (decode: arange)
 *   ibuf     [rows, steps, Hv, V, K] or NULL; ibuf[b, t] = state after token t
 *            of sequence b (t < L_b), written only for non-padding rows
 * Returns 0, or -1 on a malformed argument (e.g. L_b > steps with ibuf).
 */
int oracle_pool(const double* q, const double* k, const double* v, const double* g,
                const double* gk, const double* beta, const double* pool_in, double* pool_out,
                const int32_t* state_idx, const int64_t* cu, int N, int num_slots, int Hk,
                int Hv, int K, int V, double scale, int commit, double* o, double* ibuf,
                int steps, int nthreads) {
    if (Hk <= 0 || Hv % Hk != 0) return -1;
    for (int b = 0; b < N; ++b) {
        if (state_idx[b] >= num_slots) return -1;
        if (ibuf && state_idx[b] >= 0 && cu[b + 1] - cu[b] > steps) return -1;
    }
    set_threads(nthreads);
    const int units = N * Hv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int u = 0; u < units; ++u) {
        const int b = u / Hv, h = u % Hv;
        const int slot = state_idx[b];
        if (slot < 0) continue;
        const int kh = key_head(h, Hk, Hv, 0);
        double* S = (double*)malloc(sizeof(double) * (size_t)V * K);
        double* dec = (double*)malloc(sizeof(double) * (size_t)K);
        load_state(S, pool_in + ((size_t)slot * Hv + h) * V * K, K, V, 0);
        for (int64_t t = cu[b]; t < cu[b + 1]; ++t) {
            if (gk) {  /* per-key-channel decay: column c of S scaled by e^{gk[c]} */
                for (int c = 0; c < K; ++c) dec[c] = exp(gk[((size_t)t * Hv + h) * K + c]);
            } else {
                const double a = exp(g[(size_t)t * Hv + h]);
                for (int c = 0; c < K; ++c) dec[c] = a;
            }
            token_step(S, dec, q + ((size_t)t * Hk + kh) * K, k + ((size_t)t * Hk + kh) * K,
                       v + ((size_t)t * Hv + h) * V, beta[(size_t)t * Hv + h], scale, K, V, 0,
                       o + ((size_t)t * Hv + h) * V);
            if (ibuf) {
                const int64_t step = t - cu[b];
                store_state(ibuf + (((size_t)b * steps + step) * Hv + h) * V * K, S, K, V, 0);
            }
        }
        if (commit) store_state(pool_out + ((size_t)slot * Hv + h) * V * K, S, K, V, 0);
        free(dec);
        free(S);
    }
    return 0;
}

/*
 * Gate preparation from raw projections (FlashQLA PR #1, host-gating and
 * in-kernel-gating commits):
 *   g    = -exp(A_log[h]) * softplus(a[t,h] + dt_bias[h])    softplus with
 *          beta 1 and threshold 20 (x > 20 -> x, else log(1 + exp(x)))
 *   beta = sigmoid(b[t,h]), doubled when neg_eigval != 0.
 */
void oracle_gating(const double* a, const double* dt_bias, const double* A_log, const double* b,
                   int64_t T, int Hv, int neg_eigval, double* g, double* beta) {
    for (int64_t t = 0; t < T; ++t)
        for (int h = 0; h < Hv; ++h) {
            const double x = a[(size_t)t * Hv + h] + dt_bias[h];
            const double sp = (x > 20.0) ? x : log1p(exp(x));
            g[(size_t)t * Hv + h] = -exp(A_log[h]) * sp;
            const double s = 1.0 / (1.0 + exp(-b[(size_t)t * Hv + h]));
            beta[(size_t)t * Hv + h] = neg_eigval ? 2.0 * s : s;
        }
}

/* Row-wise l2 normalisation y = x / sqrt(sum x^2 + eps) over rows of length D. */
void oracle_l2norm(const double* x, int64_t rows, int D, double eps, double* y) {
    for (int64_t r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int d = 0; d < D; ++d) ss += x[(size_t)r * D + d] * x[(size_t)r * D + d];
        const double inv = 1.0 / sqrt(ss + eps);
        for (int d = 0; d < D; ++d) y[(size_t)r * D + d] = x[(size_t)r * D + d] * inv;
    }
}
