/*
 * KDA oracle: a plain, slow, fp64, token-by-token CPU evaluation of the Kimi
 * Delta Attention recurrent prefill forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header or constant with the CUDA path.
 *
 * What it computes (per (sequence, head) unit, per token t, in this order):
 *   lambda_d = gate(g[t,d], A_log[h], dt_bias[h,d], lower_bound)      natural log-decay
 *   qh = q / sqrt(sum q^2 + eps),  kh = k / sqrt(sum k^2 + eps)        L2 normalisation
 *   S[:,d] *= exp(lambda_d)                                             diagonal decay
 *   S += beta_t * (v_t - S kh) kh^T                                     delta-rule correction
 *   out[t] = scale * S qh                                               read-out after the write
 * with S the V x K state, starting from initial_state (or zero) at every sequence
 * start and written to final_state after the sequence's last token.
 *
 * Sources (web pages the method is described on):
 *  - "FlashInfer PR #4262: Core Optimization Summary", section 3 (equations for
 *    L, Mqk, INV, Q_d, K_d, K_r, a, S_d, O_0, P, R, U and the final update): the
 *    chunk form whose token-level meaning is the recurrence above (decay first,
 *    inclusive prefix, read-out after the write, beta on the token's update).
 *  - same page, section 2: the gate lives in [lower_bound, 0] per key channel.
 *  - "How FlashKDA Manages Recurrent State Across Sequences and Batch Modes":
 *    batched mode ([B,H,V,K] state, one chain per batch element) and packed
 *    variable-length mode (cu_seqlens, B == 1, [N,H,V,K] state, no state flows
 *    across a sequence boundary).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - gate(): lower_bound * sigmoid(exp(A_log) * (g + dt_bias)).  The pages name
 *    the inputs and the range [lower_bound, 0] but never print the formula.
 *    PARITY UNPINNED for the exact functional form; only its range, its
 *    lower_bound == 0 case and its monotonicity are pinned by tests.
 *  - eps = 1e-6 inside the square root of the L2 norm (not stated on the pages).
 *  - packed mode: sequence n starts from initial_state[n] when one is given,
 *    else from zero; tokens at or beyond cu_seqlens[N] are not written.
 *  - beta is used as given (no sigmoid).
 * Interface variants (kda_oracle_fwd_ex flags; the pages name both, neither is the default):
 *  - KDA_ORACLE_BETA_LOGIT: beta is a logit, the step uses sigmoid(beta) ("logit beta" is
 *    an eligibility condition of the FlashInfer page, section 12).
 *  - KDA_ORACLE_GATE_SOFTPLUS: the gate max(-exp(A_log) softplus(g + dt_bias), lower_bound),
 *    the other public lower-bounded form of the KDA gate; it also lies in [lower_bound, 0].
 *    PARITY UNPINNED for its functional form, like the default gate; its special values
 *    (g + dt_bias = 0, large |g + dt_bias|) and range are pinned by tests.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KDA_ORACLE_EPS 1e-6
#define KDA_ORACLE_BETA_LOGIT 0x1u
#define KDA_ORACLE_GATE_SOFTPLUS 0x2u

/* Gate: natural-log decay of one key channel (reading stated in the header). */
double kda_oracle_gate(double g, double A_log, double dt_bias, double lower_bound)
{
    double x = exp(A_log) * (g + dt_bias);
    double sig = 1.0 / (1.0 + exp(-x));
    return lower_bound * sig;
}

/* The alternative gate: max(-exp(A_log) softplus(g + dt_bias), lower_bound), with
 * softplus(z) = log(1 + exp(z)) evaluated without overflow. */
double kda_oracle_gate_softplus(double g, double A_log, double dt_bias, double lower_bound)
{
    double z = g + dt_bias;
    double sp = z > 0.0 ? z + log1p(exp(-z)) : log1p(exp(z));
    double lam = -exp(A_log) * sp;
    return lam > lower_bound ? lam : lower_bound;
}

/* One (sequence, head) unit over tokens [bos, eos) of the flattened token axis. */
static void oracle_unit(int64_t H, int64_t K, int64_t V, int64_t h, int64_t bos, int64_t eos,
                        const double* q, const double* k, const double* v, const double* g,
                        const double* beta, double scale, const double* A_log,
                        const double* dt_bias, double lower_bound, const double* S0,
                        double* out, double* S_final, double* S, double* work, unsigned flags)
{
    double* decay = work;        /* [K] exp(lambda)     */
    double* qh = work + K;       /* [K] normalised q    */
    double* kh = work + 2 * K;   /* [K] normalised k    */

    if (S0) {
        memcpy(S, S0, (size_t)(V * K) * sizeof(double));
    } else {
        memset(S, 0, (size_t)(V * K) * sizeof(double));
    }

    for (int64_t t = bos; t < eos; ++t) {
        const double* qt = q + (t * H + h) * K;
        const double* kt = k + (t * H + h) * K;
        const double* gt = g + (t * H + h) * K;
        const double* vt = v + (t * H + h) * V;
        const double braw = beta[t * H + h];
        const double bt = (flags & KDA_ORACLE_BETA_LOGIT) ? 1.0 / (1.0 + exp(-braw)) : braw;

        double sq = 0.0, sk = 0.0;
        for (int64_t d = 0; d < K; ++d) {
            decay[d] = exp((flags & KDA_ORACLE_GATE_SOFTPLUS)
                               ? kda_oracle_gate_softplus(gt[d], A_log[h], dt_bias[h * K + d], lower_bound)
                               : kda_oracle_gate(gt[d], A_log[h], dt_bias[h * K + d], lower_bound));
            sq += qt[d] * qt[d];
            sk += kt[d] * kt[d];
        }
        const double rq = 1.0 / sqrt(sq + KDA_ORACLE_EPS);
        const double rk = 1.0 / sqrt(sk + KDA_ORACLE_EPS);
        for (int64_t d = 0; d < K; ++d) {
            qh[d] = qt[d] * rq;
            kh[d] = kt[d] * rk;
        }

        for (int64_t i = 0; i < V; ++i) {
            double* Si = S + i * K;
            /* decay */
            for (int64_t d = 0; d < K; ++d) Si[d] *= decay[d];
            /* delta-rule correction: S_i += beta (v_i - S_i . kh) kh */
            double pred = 0.0;
            for (int64_t d = 0; d < K; ++d) pred += Si[d] * kh[d];
            const double r = bt * (vt[i] - pred);
            for (int64_t d = 0; d < K; ++d) Si[d] += r * kh[d];
            /* read-out after the write */
            double o = 0.0;
            for (int64_t d = 0; d < K; ++d) o += Si[d] * qh[d];
            out[(t * H + h) * V + i] = scale * o;
        }
    }
    if (S_final) memcpy(S_final, S, (size_t)(V * K) * sizeof(double));
}

/*
 * Whole forward.  Layouts (all contiguous, row-major):
 *   q, k, g [B,T,H,K];  v, out [B,T,H,V];  beta [B,T,H];  A_log [H];  dt_bias [H,K]
 *   initial_state / final_state [Nseq,H,V,K]  (either may be NULL)
 *   cu_seqlens [N+1] int64 or NULL.  With cu_seqlens, B must be 1 and Nseq = N;
 *   without, Nseq = B and sequence b covers flattened tokens [b*T, (b+1)*T).
 * Rows of out that belong to no sequence are left untouched.
 * Returns 0 on success, a negative code on invalid arguments.
 */
int kda_oracle_fwd_ex(int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                      const double* q, const double* k, const double* v, const double* g,
                      const double* beta, double scale, const double* A_log, const double* dt_bias,
                      double lower_bound, const double* initial_state, const int64_t* cu_seqlens,
                      int64_t N, double* out, double* final_state, int nthreads, unsigned flags)
{
    if (B < 1 || T < 0 || H < 1 || K < 1 || V < 1) return -1;
    int64_t nseq = B;
    if (cu_seqlens) {
        if (B != 1 || N < 0) return -2;
        if (cu_seqlens[0] != 0) return -3;
        for (int64_t n = 0; n < N; ++n)
            if (cu_seqlens[n + 1] < cu_seqlens[n]) return -3;
        if (cu_seqlens[N] > T) return -3;
        nseq = N;
    }
    const int64_t units = nseq * H;
    const size_t state_elems = (size_t)(V * K);
    int rc = 0;

#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

#pragma omp parallel
    {
        double* S = (double*)malloc(state_elems * sizeof(double));
        double* work = (double*)malloc((size_t)(3 * K) * sizeof(double));
        if (!S || !work) {
#pragma omp atomic write
            rc = -4;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t u = 0; u < units; ++u) {
                const int64_t n = u / H, h = u % H;
                int64_t bos, eos;
                if (cu_seqlens) {
                    bos = cu_seqlens[n];
                    eos = cu_seqlens[n + 1];
                } else {
                    bos = n * T;
                    eos = bos + T;
                }
                const double* S0 = initial_state ? initial_state + (size_t)u * state_elems : NULL;
                double* Sf = final_state ? final_state + (size_t)u * state_elems : NULL;
                oracle_unit(H, K, V, h, bos, eos, q, k, v, g, beta, scale, A_log, dt_bias,
                            lower_bound, S0, out, Sf, S, work, flags);
            }
        }
        free(S);
        free(work);
    }
    return rc;
}

/* The forward with neither interface variant (beta as given, the sigmoid gate). */
int kda_oracle_fwd(int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                   const double* q, const double* k, const double* v, const double* g,
                   const double* beta, double scale, const double* A_log, const double* dt_bias,
                   double lower_bound, const double* initial_state, const int64_t* cu_seqlens,
                   int64_t N, double* out, double* final_state, int nthreads)
{
    return kda_oracle_fwd_ex(B, T, H, K, V, q, k, v, g, beta, scale, A_log, dt_bias, lower_bound,
                             initial_state, cu_seqlens, N, out, final_state, nthreads, 0u);
}

/* Number of OpenMP threads a parallel region of this library would use. */
int kda_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
