/*
 * kda_oracle.c -- plain, slow, fp64 CPU oracle for the Kimi Delta Attention
 * (KDA) forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file: only the test-suite, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it computes
 * ----------------
 * "Flashkda Delta Attention", section "Core Kernel API", gives the call
 *   fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
 *       initial_state=None, final_state=None, cu_seqlens=None)
 * and says the kernel performs the recurrent state updates of delta attention.
 * "MoonshotAI/FlashKDA" (trend summary), section "Kernel API and Constraints",
 * fixes K = V = 128, allows cu_seqlens only with B = 1 and lets each state be
 * bf16, fp32 or absent.  The pages print no formula, so this oracle takes the
 * plain reading of a gated delta rule with a per-channel (per key-dimension)
 * decay, run independently for every sequence n and head h:
 *
 *   x_t      = g_t + dt_bias[h]                       (vector over K channels)
 *   la_t     = max(-exp(A_log[h]) * softplus(x_t), lower_bound)   (log decay)
 *   S        <- Diag(exp(la_t)) S                     (S is K x V, S[c][j])
 *   S        <- S + beta_t k_t (v_t - S^T k_t)^T      (delta-rule write)
 *   o_t      = scale * S^T q_t
 *
 * which is S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T.
 * The gate form (softplus of g + dt_bias, scaled by -exp(A_log), clamped
 * below at lower_bound) is a reading: the pages only name A_log, dt_bias and
 * lower_bound in the argument list.  softplus is evaluated exactly as
 * max(x,0) + log1p(exp(-|x|)) (no threshold shortcut).
 *
 * Two forms are provided:
 *   kda_oracle_fwd_*   the token-by-token recurrence above (the definition);
 *   kda_oracle_chunk   one chunk of the chunkwise form (cumsum G, strictly
 *                      lower A, T = (I + A)^-1 by forward substitution, WY
 *                      factors W and U, the query/key score matrix and the
 *                      chunk-end decay), with every exponential taken
 *                      elementwise on a difference of cumulative sums, and
 *   kda_oracle_fwd_chunked, which chains kda_oracle_chunk over a sequence.
 * The chunked form exists so that the test-suite can check it against the
 * recurrence and expose per-chunk intermediates; it is not used to define
 * anything.
 *
 * Optional query/key normalisation (kda_oracle_l2norm): each row x (one token
 * of one head, K channels) becomes x / sqrt(sum_c x_c^2 + eps), applied to q
 * and k before the recurrence.  The pages describe no normalisation inside the
 * call (the fwd signature has no flag); this is the reading of the separate
 * normalised entry point, with eps = 1e-6 keeping an all-zero row at zero.
 *
 * Layouts (all row-major, contiguous):
 *   q, k, g      [NT, H, K]      NT = total tokens (B*T, or the packed length)
 *   v, out       [NT, H, V]
 *   beta         [NT, H]
 *   A_log        [H]             dt_bias [H, K]
 *   h0, hT       [N, H, K, V]    state S[c][j] = S[(n*H + h)*K*V + c*V + j]
 *   cu           [N + 1]         token offsets of the N sequences
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2

int kda_oracle_abi_version(void) { return 1; }

/* x[r][c] <- x[r][c] / sqrt(sum_c x[r][c]^2 + eps) for every row r of D
 * channels (rows = tokens x heads). */
void kda_oracle_l2norm(double* x, int64_t rows, int64_t D, double eps) {
    for (int64_t r = 0; r < rows; ++r) {
        double* row = x + r * D;
        double ss = 0.0;
        for (int64_t c = 0; c < D; ++c) ss += row[c] * row[c];
        const double inv = 1.0 / sqrt(ss + eps);
        for (int64_t c = 0; c < D; ++c) row[c] *= inv;
    }
}

/* bf16 bit pattern -> exact double (bf16 is the top half of an IEEE fp32). */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double softplus(double x) {
    double pos = x > 0.0 ? x : 0.0;
    return pos + log1p(exp(-fabs(x)));
}

/* Log-decay of one channel (see header). */
double kda_oracle_log_decay(double g, double A_log, double dt_bias, double lower_bound) {
    double la = -exp(A_log) * softplus(g + dt_bias);
    return la < lower_bound ? lower_bound : la;
}

/* Element accessors: the fp64 entry point reads doubles, the "typed" entry
 * point reads bf16 activations and fp32 / bf16 states and upcasts exactly. */
typedef struct {
    int kind; /* 0 = double, 1 = bf16 bits, 2 = float */
    const void* p;
} src_t;

static double src_get(src_t s, int64_t i) {
    switch (s.kind) {
        case 0: return ((const double*)s.p)[i];
        case 1: return bf16_bits_to_double(((const uint16_t*)s.p)[i]);
        default: return (double)((const float*)s.p)[i];
    }
}

typedef struct {
    src_t q, k, v, g, beta, A_log, dt_bias, h0;
    double scale, lower_bound, erase;
    double* out;
    double* hT;
    const int64_t* cu;
    int64_t N, H, K, V;
} problem_t;

static int validate(const problem_t* P) {
    if (P->N < 0 || P->H <= 0 || P->K <= 0 || P->V <= 0) return ORACLE_EINVAL;
    if (!P->cu || P->cu[0] != 0) return ORACLE_EINVAL;
    for (int64_t n = 0; n < P->N; ++n)
        if (P->cu[n + 1] < P->cu[n]) return ORACLE_EINVAL;
    return ORACLE_OK;
}

/* The token-by-token recurrence for one (sequence, head).  S, r and a are
 * caller-provided scratch of K*V, V and K doubles. */
static void recur_one(const problem_t* P, int64_t n, int64_t h, double* S, double* r, double* a) {
    const int64_t K = P->K, V = P->V, H = P->H;
    const int64_t sbase = (n * H + h) * K * V;
    for (int64_t i = 0; i < K * V; ++i) S[i] = P->h0.p ? src_get(P->h0, sbase + i) : 0.0;
    const double A_log = src_get(P->A_log, h);
    for (int64_t t = P->cu[n]; t < P->cu[n + 1]; ++t) {
        const int64_t qk_row = (t * H + h) * K;
        const int64_t v_row = (t * H + h) * V;
        /* decay */
        for (int64_t c = 0; c < K; ++c) {
            double la = kda_oracle_log_decay(src_get(P->g, qk_row + c), A_log,
                                             src_get(P->dt_bias, h * K + c), P->lower_bound);
            a[c] = exp(la);
        }
        for (int64_t c = 0; c < K; ++c)
            for (int64_t j = 0; j < V; ++j) S[c * V + j] *= a[c];
        /* r = S^T k */
        for (int64_t j = 0; j < V; ++j) r[j] = 0.0;
        for (int64_t c = 0; c < K; ++c) {
            const double kc = src_get(P->k, qk_row + c);
            for (int64_t j = 0; j < V; ++j) r[j] += S[c * V + j] * kc;
        }
        /* S += beta k (v - erase * r)^T */
        const double b = src_get(P->beta, t * H + h);
        for (int64_t j = 0; j < V; ++j) r[j] = b * (src_get(P->v, v_row + j) - P->erase * r[j]);
        for (int64_t c = 0; c < K; ++c) {
            const double kc = src_get(P->k, qk_row + c);
            for (int64_t j = 0; j < V; ++j) S[c * V + j] += kc * r[j];
        }
        /* o = scale S^T q */
        double* o = P->out + v_row;
        for (int64_t j = 0; j < V; ++j) o[j] = 0.0;
        for (int64_t c = 0; c < K; ++c) {
            const double qc = src_get(P->q, qk_row + c);
            for (int64_t j = 0; j < V; ++j) o[j] += S[c * V + j] * qc;
        }
        for (int64_t j = 0; j < V; ++j) o[j] *= P->scale;
    }
    if (P->hT)
        for (int64_t i = 0; i < K * V; ++i) P->hT[sbase + i] = S[i];
}

static int run_recurrent(const problem_t* P, int nthreads) {
    int rc = validate(P);
    if (rc) return rc;
    const int64_t pairs = P->N * P->H;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (int64_t p = 0; p < pairs; ++p) {
        double* S = (double*)malloc(sizeof(double) * (size_t)(P->K * P->V + P->V + P->K));
        if (!S) {
            failed = 1;
            continue;
        }
        recur_one(P, p / P->H, p % P->H, S, S + P->K * P->V, S + P->K * P->V + P->V);
        free(S);
    }
    return failed ? ORACLE_ENOMEM : ORACLE_OK;
}

/*
 * All-fp64 entry point.  erase scales the S^T k term of the delta-rule write
 * (1 for KDA; 0 gives a plain gated linear-attention write, used only by the
 * test-suite).  h0 / hT may be NULL.  Returns 0 on success.
 */
int kda_oracle_fwd_f64(const double* q, const double* k, const double* v, const double* g,
                       const double* beta, double scale, const double* A_log,
                       const double* dt_bias, double lower_bound, const double* h0,
                       double* out, double* hT, const int64_t* cu, int64_t N, int64_t H,
                       int64_t K, int64_t V, double erase, int nthreads) {
    problem_t P = {{0, q}, {0, k}, {0, v}, {0, g}, {0, beta}, {0, A_log}, {0, dt_bias}, {0, h0},
                   scale, lower_bound, erase, out, hT, cu, N, H, K, V};
    return run_recurrent(&P, nthreads);
}

/*
 * Typed entry point: q, k, v, g, beta are bf16 bit patterns; A_log and
 * dt_bias are fp32; h0 is fp32 (h0_kind = 2), bf16 (h0_kind = 1) or absent
 * (h0 = NULL).  Every value is upcast exactly to fp64 before use.
 */
int kda_oracle_fwd_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const uint16_t* g, const uint16_t* beta, double scale,
                        const float* A_log, const float* dt_bias, double lower_bound,
                        const void* h0, int h0_kind, double* out, double* hT,
                        const int64_t* cu, int64_t N, int64_t H, int64_t K, int64_t V,
                        int nthreads) {
    if (h0 && h0_kind != 1 && h0_kind != 2) return ORACLE_EINVAL;
    problem_t P = {{1, q}, {1, k}, {1, v}, {1, g}, {1, beta}, {2, A_log}, {2, dt_bias},
                   {h0 ? h0_kind : 2, h0}, scale, lower_bound, 1.0, out, hT, cu, N, H, K, V};
    return run_recurrent(&P, nthreads);
}

/*
 * One chunk of the chunkwise form, for one head, in fp64.
 *
 * Inputs are the chunk's c token rows: q, k (row stride ldk), v (row stride
 * ldv), per-channel log decays la (c x K, contiguous) and beta (stride ldb).
 * Outputs (contiguous, any may be NULL):
 *   G     c x K   G_t = sum_{s<=t} la_s                    (in-chunk cumsum)
 *   A     c x c   A[i][j] = beta_i sum_ch k_i k_j exp(G_i - G_j), j < i, else 0
 *   Aqk   c x c   Aqk[i][j] = sum_ch q_i k_j exp(G_i - G_j),      j <= i, else 0
 *   T     c x c   (I + A)^-1, unit lower triangular, by forward substitution
 *   W     c x K   T diag(beta) (K o exp(G))
 *   U     c x V   T diag(beta) V
 *   gam   K       exp(G_{c-1})                              (chunk-end decay)
 * With these, for the state S0 entering the chunk,
 *   Delta = U - W S0,
 *   o_i   = scale (S0^T (q_i o exp(G_i)) + sum_{j<=i} Aqk[i][j] Delta_j),
 *   S_end = Diag(gam) S0 + sum_j (k_j o exp(G_{c-1} - G_j)) Delta_j^T,
 * which follows from unrolling the recurrence across the chunk.
 */
int kda_oracle_chunk(const double* q, int64_t ldq, const double* k, int64_t ldk,
                     const double* v, int64_t ldv, const double* la, const double* beta,
                     int64_t ldb, int64_t c, int64_t K, int64_t V, double* G, double* A,
                     double* Aqk, double* T, double* W, double* U, double* gam) {
    if (c <= 0 || K <= 0 || V <= 0) return ORACLE_EINVAL;
    double* Gl = (double*)malloc(sizeof(double) * (size_t)(c * K + 3 * c * c));
    if (!Gl) return ORACLE_ENOMEM;
    double* Al = Gl + c * K;
    double* Ql = Al + c * c;
    double* Tl = Ql + c * c;
    for (int64_t ch = 0; ch < K; ++ch) {
        double run = 0.0;
        for (int64_t t = 0; t < c; ++t) {
            run += la[t * K + ch];
            Gl[t * K + ch] = run;
        }
    }
    for (int64_t i = 0; i < c; ++i)
        for (int64_t j = 0; j < c; ++j) {
            double skk = 0.0, sqk = 0.0;
            if (j <= i)
                for (int64_t ch = 0; ch < K; ++ch) {
                    const double d = exp(Gl[i * K + ch] - Gl[j * K + ch]);
                    skk += k[i * ldk + ch] * k[j * ldk + ch] * d;
                    sqk += q[i * ldq + ch] * k[j * ldk + ch] * d;
                }
            Al[i * c + j] = (j < i) ? beta[i * ldb] * skk : 0.0;
            Ql[i * c + j] = (j <= i) ? sqk : 0.0;
        }
    /* forward substitution: row i of T solves (I + A) T = I */
    for (int64_t i = 0; i < c; ++i)
        for (int64_t j = 0; j < c; ++j) {
            double s = (i == j) ? 1.0 : 0.0;
            for (int64_t l = 0; l < i; ++l) s -= Al[i * c + l] * Tl[l * c + j];
            Tl[i * c + j] = s;
        }
    if (G) memcpy(G, Gl, sizeof(double) * (size_t)(c * K));
    if (A) memcpy(A, Al, sizeof(double) * (size_t)(c * c));
    if (Aqk) memcpy(Aqk, Ql, sizeof(double) * (size_t)(c * c));
    if (T) memcpy(T, Tl, sizeof(double) * (size_t)(c * c));
    if (W)
        for (int64_t i = 0; i < c; ++i)
            for (int64_t ch = 0; ch < K; ++ch) {
                double s = 0.0;
                for (int64_t l = 0; l < c; ++l)
                    s += Tl[i * c + l] * beta[l * ldb] * k[l * ldk + ch] * exp(Gl[l * K + ch]);
                W[i * K + ch] = s;
            }
    if (U)
        for (int64_t i = 0; i < c; ++i)
            for (int64_t j = 0; j < V; ++j) {
                double s = 0.0;
                for (int64_t l = 0; l < c; ++l) s += Tl[i * c + l] * beta[l * ldb] * v[l * ldv + j];
                U[i * V + j] = s;
            }
    if (gam)
        for (int64_t ch = 0; ch < K; ++ch) gam[ch] = exp(Gl[(c - 1) * K + ch]);
    free(Gl);
    return ORACLE_OK;
}

/*
 * The chunkwise form chained over every sequence and head, chunk size C
 * (chunks start at each sequence start; the last one may be shorter).
 * Same arguments and layouts as kda_oracle_fwd_f64 (erase is fixed to 1).
 */
int kda_oracle_fwd_chunked(const double* q, const double* k, const double* v,
                           const double* g, const double* beta, double scale,
                           const double* A_log, const double* dt_bias, double lower_bound,
                           const double* h0, double* out, double* hT, const int64_t* cu,
                           int64_t N, int64_t H, int64_t K, int64_t V, int64_t C) {
    if (C <= 0 || N < 0 || H <= 0 || K <= 0 || V <= 0 || !cu || cu[0] != 0) return ORACLE_EINVAL;
    for (int64_t n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return ORACLE_EINVAL;
    const size_t need = (size_t)(K * V + C * K * 3 + C * C * 3 + C * V * 2 + K);
    double* buf = (double*)malloc(sizeof(double) * need);
    if (!buf) return ORACLE_ENOMEM;
    double* S = buf;
    double* la = S + K * V;
    double* G = la + C * K;
    double* W = G + C * K;
    double* A = W + C * K;
    double* Aqk = A + C * C;
    double* T = Aqk + C * C;
    double* U = T + C * C;
    double* D = U + C * V;
    double* gam = D + C * V;
    int rc = ORACLE_OK;
    for (int64_t n = 0; n < N && rc == ORACLE_OK; ++n)
        for (int64_t h = 0; h < H && rc == ORACLE_OK; ++h) {
            const int64_t sbase = (n * H + h) * K * V;
            for (int64_t i = 0; i < K * V; ++i) S[i] = h0 ? h0[sbase + i] : 0.0;
            for (int64_t t0 = cu[n]; t0 < cu[n + 1]; t0 += C) {
                const int64_t c = (cu[n + 1] - t0 < C) ? cu[n + 1] - t0 : C;
                for (int64_t t = 0; t < c; ++t)
                    for (int64_t ch = 0; ch < K; ++ch)
                        la[t * K + ch] = kda_oracle_log_decay(g[((t0 + t) * H + h) * K + ch],
                                                              A_log[h], dt_bias[h * K + ch],
                                                              lower_bound);
                const double* qc = q + (t0 * H + h) * K;
                const double* kc = k + (t0 * H + h) * K;
                const double* vc = v + (t0 * H + h) * V;
                const double* bc = beta + t0 * H + h;
                rc = kda_oracle_chunk(qc, H * K, kc, H * K, vc, H * V, la, bc, H, c, K, V, G, A,
                                      Aqk, T, W, U, gam);
                if (rc) break;
                /* Delta = U - W S0 */
                for (int64_t i = 0; i < c; ++i)
                    for (int64_t j = 0; j < V; ++j) {
                        double s = U[i * V + j];
                        for (int64_t ch = 0; ch < K; ++ch) s -= W[i * K + ch] * S[ch * V + j];
                        D[i * V + j] = s;
                    }
                /* outputs */
                for (int64_t i = 0; i < c; ++i)
                    for (int64_t j = 0; j < V; ++j) {
                        double s = 0.0;
                        for (int64_t ch = 0; ch < K; ++ch)
                            s += qc[i * H * K + ch] * exp(G[i * K + ch]) * S[ch * V + j];
                        for (int64_t l = 0; l <= i; ++l) s += Aqk[i * c + l] * D[l * V + j];
                        out[((t0 + i) * H + h) * V + j] = scale * s;
                    }
                /* state to the end of the chunk */
                for (int64_t ch = 0; ch < K; ++ch)
                    for (int64_t j = 0; j < V; ++j) {
                        double s = gam[ch] * S[ch * V + j];
                        for (int64_t l = 0; l < c; ++l)
                            s += kc[l * H * K + ch] * exp(G[(c - 1) * K + ch] - G[l * K + ch]) *
                                 D[l * V + j];
                        S[ch * V + j] = s;
                    }
            }
            if (hT)
                for (int64_t i = 0; i < K * V; ++i) hT[sbase + i] = S[i];
        }
    free(buf);
    return rc;
}

/* Log-decays for a block of tokens: la[t][h][c] for g laid out [n_tok, H, K]. */
int kda_oracle_gate(const double* g, int64_t n_tok, int64_t H, int64_t K, const double* A_log,
                    const double* dt_bias, double lower_bound, double* la) {
    if (n_tok < 0 || H <= 0 || K <= 0) return ORACLE_EINVAL;
    for (int64_t t = 0; t < n_tok; ++t)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t c = 0; c < K; ++c) {
                const int64_t i = (t * H + h) * K + c;
                la[i] = kda_oracle_log_decay(g[i], A_log[h], dt_bias[h * K + c], lower_bound);
            }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------------
 * Reverse mode of the token-by-token recurrence (the backward pass).
 *
 * The pages describe the forward call only (and recommend running it under
 * torch.inference_mode, "MoonshotAI/FlashKDA", "Automatic Branching for
 * Installation and Usage"); the gradients below are those of the recurrence
 * defined at the top of this file, taken by the chain rule step by step in
 * reverse token order.  For one (sequence, head), with the scalar loss
 * L = sum_t <dout_t, o_t> + <dhT, S_final>, per token t (forward quantities as
 * in recur_one: x, sp = softplus(x), pre = -exp(A_log) sp, la = max(pre, lb),
 * alpha = exp(la), St = Diag(alpha) S_{t-1}, r = St^T k, u = beta (v - r),
 * S_t = St + k u^T, o_t = scale S_t^T q):
 *
 *   dS  += scale q dout_t^T            dq   = scale S_t dout_t
 *   dk  += dS u                         du   = dS^T k          (dSt = dS)
 *   dbeta = <du, v - r>                dv   = beta du          dr = -beta du
 *   dSt += k dr^T                       dk  += St dr
 *   dalpha_c = sum_j dSt[c][j] S_{t-1}[c][j]                   dS_{t-1} = Diag(alpha) dSt
 *   dla = dalpha alpha;  dpre = dla where pre >= lb, else 0   (the max passes its
 *                        gradient to the argument it returns; at a tie, to pre)
 *   dA_log += sum_c pre_c dpre_c        dsp = -exp(A_log) dpre
 *   dx  = dsp sigmoid(x)                dg = dx, ddt_bias += dx
 *
 * and dh0 = dS after the first token.  The forward states S_0 .. S_L of the
 * sequence are kept (L + 1 matrices of K x V doubles), so this is meant for the
 * small problems of the test-suite.
 * ------------------------------------------------------------------------------ */

static double sigmoid(double x) {
    if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
    const double e = exp(x);
    return e / (1.0 + e);
}

typedef struct {
    const double *q, *k, *v, *g, *beta, *A_log, *dt_bias, *h0, *dout, *dhT;
    double scale, lower_bound;
    double *dq, *dk, *dv, *dg, *dbeta, *dA_log, *ddt_bias, *dh0;
    const int64_t* cu;
    int64_t N, H, K, V;
} grad_problem_t;

/* One (sequence, head).  dA_log_h and ddt_bias_h are this pair's private
 * accumulators (the caller sums them over sequences). */
static int grad_one(const grad_problem_t* P, int64_t n, int64_t h, double* dA_log_h,
                    double* ddt_bias_h) {
    const int64_t K = P->K, V = P->V, H = P->H, KV = K * V;
    const int64_t t0 = P->cu[n], L = P->cu[n + 1] - P->cu[n];
    const double a = exp(P->A_log[h]);
    double* Ss = (double*)malloc(sizeof(double) * (size_t)((L + 1) * KV));
    double* work = (double*)malloc(sizeof(double) * (size_t)(2 * KV + 6 * V + 4 * K));
    if (!Ss || !work) {
        free(Ss);
        free(work);
        return ORACLE_ENOMEM;
    }
    double* dS = work;
    double* St = dS + KV;
    double* r = St + KV;
    double* u = r + V;
    double* du = u + V;
    double* dr = du + V;
    double* tmp = dr + V;
    double* spare = tmp + V;
    double* alpha = spare + V;
    double* pre = alpha + K;
    double* xg = pre + K;
    double* dal = xg + K;
    (void)spare;

    /* forward: S_0 = h0, S_{t+1} after token t */
    for (int64_t i = 0; i < KV; ++i) Ss[i] = P->h0 ? P->h0[(n * H + h) * KV + i] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
        const int64_t row = (t0 + t) * H + h;
        const double* S0 = Ss + t * KV;
        double* S1 = Ss + (t + 1) * KV;
        for (int64_t c = 0; c < K; ++c) {
            const double x = P->g[row * K + c] + P->dt_bias[h * K + c];
            double la = -a * softplus(x);
            if (la < P->lower_bound) la = P->lower_bound;
            for (int64_t j = 0; j < V; ++j) S1[c * V + j] = exp(la) * S0[c * V + j];
        }
        for (int64_t j = 0; j < V; ++j) r[j] = 0.0;
        for (int64_t c = 0; c < K; ++c)
            for (int64_t j = 0; j < V; ++j) r[j] += S1[c * V + j] * P->k[row * K + c];
        const double b = P->beta[row];
        for (int64_t j = 0; j < V; ++j) u[j] = b * (P->v[row * V + j] - r[j]);
        for (int64_t c = 0; c < K; ++c)
            for (int64_t j = 0; j < V; ++j) S1[c * V + j] += P->k[row * K + c] * u[j];
    }

    /* backward */
    for (int64_t i = 0; i < KV; ++i) dS[i] = P->dhT ? P->dhT[(n * H + h) * KV + i] : 0.0;
    for (int64_t t = L - 1; t >= 0; --t) {
        const int64_t row = (t0 + t) * H + h;
        const double* Sprev = Ss + t * KV;
        const double* Scur = Ss + (t + 1) * KV;
        const double* qv = P->q + row * K;
        const double* kv = P->k + row * K;
        const double* vv = P->v + row * V;
        const double* dov = P->dout + row * V;
        const double b = P->beta[row];
        /* recompute the token's forward quantities */
        for (int64_t c = 0; c < K; ++c) {
            xg[c] = P->g[row * K + c] + P->dt_bias[h * K + c];
            pre[c] = -a * softplus(xg[c]);
            const double la = pre[c] < P->lower_bound ? P->lower_bound : pre[c];
            alpha[c] = exp(la);
            for (int64_t j = 0; j < V; ++j) St[c * V + j] = alpha[c] * Sprev[c * V + j];
        }
        for (int64_t j = 0; j < V; ++j) r[j] = 0.0;
        for (int64_t c = 0; c < K; ++c)
            for (int64_t j = 0; j < V; ++j) r[j] += St[c * V + j] * kv[c];
        for (int64_t j = 0; j < V; ++j) u[j] = b * (vv[j] - r[j]);
        /* o_t = scale S_t^T q */
        for (int64_t c = 0; c < K; ++c) {
            double s = 0.0;
            for (int64_t j = 0; j < V; ++j) {
                dS[c * V + j] += P->scale * qv[c] * dov[j];
                s += Scur[c * V + j] * dov[j];
            }
            P->dq[row * K + c] = P->scale * s;
        }
        /* S_t = St + k u^T */
        for (int64_t j = 0; j < V; ++j) du[j] = 0.0;
        for (int64_t c = 0; c < K; ++c) {
            double s = 0.0;
            for (int64_t j = 0; j < V; ++j) {
                s += dS[c * V + j] * u[j];
                du[j] += dS[c * V + j] * kv[c];
            }
            P->dk[row * K + c] = s;
        }
        /* u = beta (v - r) */
        double db = 0.0;
        for (int64_t j = 0; j < V; ++j) {
            db += du[j] * (vv[j] - r[j]);
            P->dv[row * V + j] = b * du[j];
            dr[j] = -b * du[j];
        }
        P->dbeta[row] = db;
        /* r = St^T k: dSt = dS + k dr^T, dk += St dr */
        for (int64_t c = 0; c < K; ++c) {
            double s = 0.0;
            for (int64_t j = 0; j < V; ++j) {
                s += St[c * V + j] * dr[j];
                dS[c * V + j] += kv[c] * dr[j];
            }
            P->dk[row * K + c] += s;
        }
        /* St = Diag(alpha) S_{t-1} */
        for (int64_t c = 0; c < K; ++c) {
            double s = 0.0;
            for (int64_t j = 0; j < V; ++j) {
                s += dS[c * V + j] * Sprev[c * V + j];
                dS[c * V + j] *= alpha[c];
            }
            dal[c] = s;
        }
        /* gate */
        for (int64_t c = 0; c < K; ++c) {
            const double dla = dal[c] * alpha[c];
            const double dpre = pre[c] >= P->lower_bound ? dla : 0.0;
            *dA_log_h += pre[c] * dpre;
            const double dx = -a * dpre * sigmoid(xg[c]);
            P->dg[row * K + c] = dx;
            ddt_bias_h[c] += dx;
        }
    }
    if (P->dh0)
        for (int64_t i = 0; i < KV; ++i) P->dh0[(n * H + h) * KV + i] = dS[i];
    free(Ss);
    free(work);
    return ORACLE_OK;
}

/*
 * Gradients of L = sum <dout, out> + <dhT, final_state> with respect to every
 * input of kda_oracle_fwd_f64 (erase = 1).  Layouts as for the forward; dhT,
 * h0 and dh0 may be NULL (no final-state gradient / zero initial state / not
 * wanted).  dA_log [H] and ddt_bias [H, K] are sums over all tokens.
 */
int kda_oracle_bwd_f64(const double* q, const double* k, const double* v, const double* g,
                       const double* beta, double scale, const double* A_log,
                       const double* dt_bias, double lower_bound, const double* h0,
                       const double* dout, const double* dhT, const int64_t* cu, int64_t N,
                       int64_t H, int64_t K, int64_t V, double* dq, double* dk, double* dv,
                       double* dg, double* dbeta, double* dA_log, double* ddt_bias, double* dh0,
                       int nthreads) {
    if (N < 0 || H <= 0 || K <= 0 || V <= 0 || !cu || cu[0] != 0) return ORACLE_EINVAL;
    for (int64_t n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return ORACLE_EINVAL;
    grad_problem_t P = {q, k, v, g, beta, A_log, dt_bias, h0, dout, dhT, scale, lower_bound,
                        dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dh0, cu, N, H, K, V};
    const int64_t pairs = N * H;
    double* acc = (double*)calloc((size_t)(pairs * (K + 1)), sizeof(double));
    if (!acc) return ORACLE_ENOMEM;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (int64_t p = 0; p < pairs; ++p)
        failed |= grad_one(&P, p / H, p % H, acc + p * (K + 1), acc + p * (K + 1) + 1);
    /* per-head sums over the sequences, in a fixed order */
    for (int64_t h = 0; h < H; ++h) {
        dA_log[h] = 0.0;
        for (int64_t c = 0; c < K; ++c) ddt_bias[h * K + c] = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            const double* ac = acc + (n * H + h) * (K + 1);
            dA_log[h] += ac[0];
            for (int64_t c = 0; c < K; ++c) ddt_bias[h * K + c] += ac[1 + c];
        }
    }
    free(acc);
    return failed ? ORACLE_ENOMEM : ORACLE_OK;
}
