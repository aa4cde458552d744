/*
 * Plain float64 CTC loss and gradient over sequence-packed log probabilities.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA path is
 * checked against.  Only the tests, the package's smoke check and the CPU
 * baseline of the benchmark may load it; the library never does.
 *
 * What it computes (page "feat(asr): native CTC loss kernel over
 * sequence-packed log probabilities", NVIDIA-NeMo/Speech PR #16437, file
 * nemo/collections/asr/parts/triton/ctc_loss.py, module docstring and the two
 * kernels):
 *
 *   The log probabilities of a batch are one token-flat (T_total, D) buffer;
 *   utterance b owns rows [cu[b], cu[b] + len[b]).  For its target
 *   l_1..l_U the extended label sequence is l' = (blank, l_1, blank, ...,
 *   l_U, blank), S = 2U + 1 states.
 *
 *   alpha_0(s) = lp[0, l'_s] for s < min(2, S), -inf elsewhere;
 *   alpha_t(s) = log( e^alpha_{t-1}(s) + e^alpha_{t-1}(s-1)
 *                     + [skip(s)] e^alpha_{t-1}(s-2) ) + lp[t, l'_s],
 *   with skip(s) = (s odd, s >= 2, l'_s != l'_{s-2}): a target id equal to
 *   the blank is a label like any other.
 *   nll = -log( e^alpha_{T-1}(S-1) + e^alpha_{T-1}(S-2) ); with T = 0 the
 *   loss is 0 when U = 0 and +inf otherwise.
 *
 *   beta_{T-1}(s) = lp[T-1, l'_s] for s >= S-2, -inf elsewhere;
 *   beta_t(s) = log( e^beta_{t+1}(s) + e^beta_{t+1}(s+1)
 *                    + [skip'(s)] e^beta_{t+1}(s+2) ) + lp[t, l'_s],
 *   skip'(s) = (s odd, s + 2 < S, l'_s != l'_{s+2}); beta includes lp[t].
 *
 *   posterior gamma_t(s) = exp(alpha_t(s) + beta_t(s) - lp[t, l'_s] + nll),
 *   P_t(c) = sum of gamma_t(s) over the states with l'_s = c, and the
 *   gradient row (for unit upstream gradient) is exp(lp[t, c]) - P_t(c),
 *   the gradient with respect to the logits when lp is a log_softmax output.
 *   Rows that belong to no utterance get a zero gradient.
 *
 * Everything is a direct transcription of these definitions: full alpha and
 * beta tables, a natural-order sum per class.  No blocking, no rescaling.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* log(e^a + e^b), exact for -inf operands. */
static double log_add(double a, double b) {
    if (a == -INFINITY) return b;
    if (b == -INFINITY) return a;
    double m = a > b ? a : b;
    return m + log(exp(a - m) + exp(b - m));
}

/* Extended label of state s: blank at even s, l_{(s-1)/2} at odd s. */
static int64_t ext_label(const int64_t* labels, int64_t s, int64_t blank) {
    return (s % 2 == 0) ? blank : labels[(s - 1) / 2];
}

/*
 * One utterance.  lp points at its first row (T rows of D), labels at its U
 * target ids.  Writes *nll and, when grad is not NULL, the T x D unit-scale
 * gradient rows.  Returns 0, or -1 when memory runs out.
 */
int ctc_oracle_utterance(const double* lp, int64_t T, int64_t D, const int64_t* labels, int64_t U,
                         int64_t blank, double* nll, double* grad) {
    const int64_t S = 2 * U + 1;
    if (T == 0) {
        *nll = (U == 0) ? 0.0 : INFINITY;
        return 0;
    }
    double* alpha = (double*)malloc(sizeof(double) * (size_t)(T * S));
    double* beta = (double*)malloc(sizeof(double) * (size_t)(T * S));
    if (!alpha || !beta) {
        free(alpha);
        free(beta);
        return -1;
    }
#define LP(t, c) lp[(t) * D + (c)]
#define ALPHA(t, s) alpha[(t) * S + (s)]
#define BETA(t, s) beta[(t) * S + (s)]
    /* forward */
    for (int64_t s = 0; s < S; ++s) ALPHA(0, s) = -INFINITY;
    ALPHA(0, 0) = LP(0, blank);
    if (S > 1) ALPHA(0, 1) = LP(0, ext_label(labels, 1, blank));
    for (int64_t t = 1; t < T; ++t) {
        for (int64_t s = 0; s < S; ++s) {
            double a = ALPHA(t - 1, s);
            if (s >= 1) a = log_add(a, ALPHA(t - 1, s - 1));
            if (s >= 2 && s % 2 == 1 && ext_label(labels, s, blank) != ext_label(labels, s - 2, blank))
                a = log_add(a, ALPHA(t - 1, s - 2));
            ALPHA(t, s) = a + LP(t, ext_label(labels, s, blank));
        }
    }
    double total = ALPHA(T - 1, S - 1);
    if (S > 1) total = log_add(total, ALPHA(T - 1, S - 2));
    *nll = -total;

    if (grad) {
        /* backward */
        for (int64_t s = 0; s < S; ++s) BETA(T - 1, s) = -INFINITY;
        BETA(T - 1, S - 1) = LP(T - 1, ext_label(labels, S - 1, blank));
        if (S > 1) BETA(T - 1, S - 2) = LP(T - 1, ext_label(labels, S - 2, blank));
        for (int64_t t = T - 2; t >= 0; --t) {
            for (int64_t s = 0; s < S; ++s) {
                double b = BETA(t + 1, s);
                if (s + 1 < S) b = log_add(b, BETA(t + 1, s + 1));
                if (s % 2 == 1 && s + 2 < S && ext_label(labels, s, blank) != ext_label(labels, s + 2, blank))
                    b = log_add(b, BETA(t + 1, s + 2));
                BETA(t, s) = b + LP(t, ext_label(labels, s, blank));
            }
        }
        /* gradient rows: exp(lp) minus the class posteriors */
        for (int64_t t = 0; t < T; ++t) {
            double* g = grad + t * D;
            for (int64_t c = 0; c < D; ++c) g[c] = exp(LP(t, c));
            for (int64_t s = 0; s < S; ++s) {
                int64_t c = ext_label(labels, s, blank);
                g[c] -= exp(ALPHA(t, s) + BETA(t, s) - LP(t, c) + *nll);
            }
        }
    }
#undef LP
#undef ALPHA
#undef BETA
    free(alpha);
    free(beta);
    return 0;
}

/*
 * A packed batch.  lp is T_total x D, targets are concatenated (utterance b's
 * ids start at sum_{j<b} tlen[j]).  nll gets B values; grad, when not NULL,
 * gets T_total x D unit-scale rows, zero outside every utterance.  Utterances
 * run in parallel over nthreads OpenMP threads (0 keeps the runtime default).
 * Returns 0, or -1 when memory runs out.
 */
int ctc_oracle_batch(const double* lp, int64_t T_total, int64_t D, const int64_t* cu, const int64_t* len,
                     const int64_t* targets, const int64_t* tlen, int64_t B, int64_t blank, double* nll,
                     double* grad, int nthreads) {
    int64_t* toff = (int64_t*)malloc(sizeof(int64_t) * (size_t)(B + 1));
    if (!toff) return -1;
    toff[0] = 0;
    for (int64_t b = 0; b < B; ++b) toff[b + 1] = toff[b] + tlen[b];
    if (grad) memset(grad, 0, sizeof(double) * (size_t)(T_total * D));
    int failed = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (int64_t b = 0; b < B; ++b) {
        const double* lpb = lp + cu[b] * D;
        double* gb = grad ? grad + cu[b] * D : NULL;
        if (ctc_oracle_utterance(lpb, len[b], D, targets + toff[b], tlen[b], blank, &nll[b], gb) != 0) failed = 1;
    }
    (void)nthreads;
    free(toff);
    return failed ? -1 : 0;
}

int ctc_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
