/*
 * GatedDeltaNet oracle: a plain, slow, FP64 CPU evaluation of the gated delta
 * rule, its compact state-update capsules, prefix replay and the packed causal
 * convolution that precedes it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the tests, the smoke check of the package entry point and the
 * CPU-baseline leg of the benchmark use it.  It shares no code, header, table
 * or helper with the CUDA library.
 *
 * Sources (page title, then section):
 *  - "Add GatedDeltaNet evaluation export for Qwen hybrid models", Summary /
 *    What changed: packed THD Q/K/V with cumulative sequence lengths, FP32
 *    V-major recurrent state, the gated_delta update rule, precomputed
 *    effective decay and beta gates with activation "none".
 *  - "[CUDA] Add compact GatedDeltaNet operator", Description: fused Qwen gate
 *    normalisation, native gate arithmetic from raw A_log, and the three
 *    outputs [output, final_state, state_update]; the FP32 capsule packs the
 *    decay, the shared key and the delta of each token.
 *  - "Replay compact fixed state for hybrid decoding", Summary / Key changes:
 *    an accepted prefix of capsules is replayed into an inactive state bank.
 *  - "[CUDA] Add compact GatedDeltaNet operator", embedded commit "Add compact
 *    VarlenCausalConv state updates": packed token-major depthwise causal conv
 *    with SiLU, a carried [channels, kernel_size-1] state and a compact capture
 *    of the appended values shaped [batch, capacity, channels].
 *
 * The pages name the update rule but do not print its equations.  The
 * per-token recurrence evaluated here is the gated delta rule, for sequence b,
 * value head h, key head kh = h / (Hv/Hk):
 *     qn = q / max(|q|, eps),  kn = k / max(|k|, eps)            (eps = 1e-6)
 *     raw gates: g = exp(-exp(A_log[h]) * softplus(a + dt_bias[h])),
 *                beta = 1 / (1 + exp(-b))
 *     S <- g S ;  u = beta (v - S kn) ;  S <- S + u kn^T ;  o = scale S qn
 * with S the dv x dk state (V-major: row i is value channel i).
 *
 * Everything is FP64.  Chains (sequence, value head) are independent and are
 * spread over OpenMP threads; within a chain the tokens run in order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_EPS 1e-6

static double oracle_softplus(double x) {
    /* log(1 + e^x), written so that neither branch overflows */
    return fmax(x, 0.0) + log1p(exp(-fabs(x)));
}

static double oracle_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static void oracle_unit(const double *x, int n, double *out) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double nrm = sqrt(ss);
    if (nrm < ORACLE_EPS) nrm = ORACLE_EPS;
    for (int i = 0; i < n; ++i) out[i] = x[i] / nrm;
}

int gdn_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Checks the packing: cu[0] = 0, non-decreasing, cu[B] = T.  Returns 0 if valid. */
static int oracle_check_cu(const int32_t *cu, int B, int T) {
    if (cu[0] != 0 || cu[B] != T) return 1;
    for (int b = 0; b < B; ++b)
        if (cu[b + 1] < cu[b]) return 1;
    return 0;
}

/*
 * Forward pass.  Layouts (all contiguous, FP64):
 *   q, k [T, Hk, dk]; v [T, Hv, dv]; a, b [T, Hv]; A_log, dt_bias [Hv]
 *   gate_mode 0: a, b are the raw inputs of the gate arithmetic above.
 *   gate_mode 1: a holds the effective decay g, b holds beta ("precomputed").
 *   initial [num_slots, Hv, dv, dk] or NULL (zero state); final: same shape.
 *   slots [B] or NULL (sequence b uses slot b).
 *   out [T, Hv, dv].
 *   caps [B, cap, W] with W = Hv + Hk*dk + Hv*dv, or NULL / cap = 0: per
 *   captured token (the first min(len_b, cap) tokens of sequence b) the row is
 *   [g for each value head][kn for each key head][u for each value head].
 *   Rows past a sequence's length are not written.
 * Returns 0, or 1 for a bad packing, 2 for a bad slot, 3 for bad geometry.
 */
int gdn_oracle_forward(int B, int T, int Hk, int Hv, int dk, int dv, int num_slots,
                       const double *q, const double *k, const double *v,
                       const double *a, const double *b,
                       const double *A_log, const double *dt_bias, int gate_mode,
                       double scale, const int32_t *cu, const int32_t *slots,
                       const double *initial, double *final_state, double *out,
                       double *caps, int cap) {
    if (Hk <= 0 || Hv <= 0 || Hv % Hk != 0 || dk <= 0 || dv <= 0) return 3;
    if (oracle_check_cu(cu, B, T)) return 1;
    for (int s = 0; s < B; ++s) {
        int slot = slots ? slots[s] : s;
        if (slot < 0 || slot >= num_slots) return 2;
    }
    const int r = Hv / Hk;
    const long W = (long)Hv + (long)Hk * dk + (long)Hv * dv;
    const long state_sz = (long)dv * dk;

    /* All chains read their initial state before any chain writes (the final
     * state may alias the initial one). */
    double *result = (double *)malloc(sizeof(double) * (size_t)B * Hv * state_sz + 1);
    int nchains = B * Hv;

#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * state_sz);
        double *qn = (double *)malloc(sizeof(double) * dk);
        double *kn = (double *)malloc(sizeof(double) * dk);
        double *u = (double *)malloc(sizeof(double) * dv);
#pragma omp for schedule(dynamic, 1)
        for (int c = 0; c < nchains; ++c) {
            const int s = c / Hv, h = c % Hv, kh = h / r;
            const int slot = slots ? slots[s] : s;
            if (initial)
                memcpy(S, initial + ((long)slot * Hv + h) * state_sz, sizeof(double) * state_sz);
            else
                memset(S, 0, sizeof(double) * state_sz);
            for (int t = cu[s]; t < cu[s + 1]; ++t) {
                oracle_unit(q + ((long)t * Hk + kh) * dk, dk, qn);
                oracle_unit(k + ((long)t * Hk + kh) * dk, dk, kn);
                double g, beta;
                if (gate_mode == 0) {
                    g = exp(-exp(A_log[h]) * oracle_softplus(a[(long)t * Hv + h] + dt_bias[h]));
                    beta = oracle_sigmoid(b[(long)t * Hv + h]);
                } else {
                    g = a[(long)t * Hv + h];
                    beta = b[(long)t * Hv + h];
                }
                /* decay */
                for (long e = 0; e < state_sz; ++e) S[e] *= g;
                /* delta against the decayed state */
                const double *vt = v + ((long)t * Hv + h) * dv;
                for (int i = 0; i < dv; ++i) {
                    double p = 0.0;
                    for (int j = 0; j < dk; ++j) p += S[(long)i * dk + j] * kn[j];
                    u[i] = beta * (vt[i] - p);
                }
                /* rank-1 write */
                for (int i = 0; i < dv; ++i)
                    for (int j = 0; j < dk; ++j) S[(long)i * dk + j] += u[i] * kn[j];
                /* read-out with the updated state */
                double *ot = out + ((long)t * Hv + h) * dv;
                for (int i = 0; i < dv; ++i) {
                    double acc = 0.0;
                    for (int j = 0; j < dk; ++j) acc += S[(long)i * dk + j] * qn[j];
                    ot[i] = scale * acc;
                }
                const int tl = t - cu[s];
                if (caps && tl < cap) {
                    double *row = caps + ((long)s * cap + tl) * W;
                    row[h] = g;
                    if (h % r == 0)
                        for (int j = 0; j < dk; ++j) row[Hv + (long)kh * dk + j] = kn[j];
                    for (int i = 0; i < dv; ++i) row[Hv + (long)Hk * dk + (long)h * dv + i] = u[i];
                }
            }
            memcpy(result + (long)c * state_sz, S, sizeof(double) * state_sz);
        }
        free(S);
        free(qn);
        free(kn);
        free(u);
    }
    for (int c = 0; c < nchains; ++c) {
        const int s = c / Hv, h = c % Hv;
        const int slot = slots ? slots[s] : s;
        memcpy(final_state + ((long)slot * Hv + h) * state_sz, result + (long)c * state_sz,
               sizeof(double) * state_sz);
    }
    free(result);
    return 0;
}

/*
 * Prefix replay.  banks [num_slots, Hv, dv, dk]; caps [R, cap, W] in the
 * capsule layout above; n [R] accepted counts in [0, cap].  For request j:
 *   S = banks[src[j]];  for i < n[j]: S <- g_i S + u_i kn_i^T;  banks[dst[j]] = S
 * (n[j] = 0 copies the source bank into the destination).  All sources are read
 * before any destination is written.
 * Returns 0, or 2 for a bad slot, 4 for a bad accepted count.
 */
int gdn_oracle_replay(double *banks, int num_slots, int R, int Hk, int Hv, int dk, int dv,
                      const int32_t *src, const int32_t *dst, const double *caps, int cap,
                      const int32_t *n) {
    if (Hk <= 0 || Hv <= 0 || Hv % Hk != 0) return 3;
    for (int j = 0; j < R; ++j) {
        if (src[j] < 0 || src[j] >= num_slots || dst[j] < 0 || dst[j] >= num_slots) return 2;
        if (n[j] < 0 || n[j] > cap) return 4;
    }
    const int r = Hv / Hk;
    const long W = (long)Hv + (long)Hk * dk + (long)Hv * dv;
    const long state_sz = (long)dv * dk;
    double *result = (double *)malloc(sizeof(double) * (size_t)R * Hv * state_sz + 1);
#pragma omp parallel for schedule(dynamic, 1)
    for (int c = 0; c < R * Hv; ++c) {
        const int j = c / Hv, h = c % Hv, kh = h / r;
        double *S = result + (long)c * state_sz;
        memcpy(S, banks + ((long)src[j] * Hv + h) * state_sz, sizeof(double) * state_sz);
        for (int i = 0; i < n[j]; ++i) {
            const double *row = caps + ((long)j * cap + i) * W;
            const double g = row[h];
            const double *kn = row + Hv + (long)kh * dk;
            const double *u = row + Hv + (long)Hk * dk + (long)h * dv;
            for (int a = 0; a < dv; ++a)
                for (int bb = 0; bb < dk; ++bb)
                    S[(long)a * dk + bb] = g * S[(long)a * dk + bb] + u[a] * kn[bb];
        }
    }
    for (int c = 0; c < R * Hv; ++c) {
        const int j = c / Hv, h = c % Hv;
        memcpy(banks + ((long)dst[j] * Hv + h) * state_sz, result + (long)c * state_sz,
               sizeof(double) * state_sz);
    }
    free(result);
    return 0;
}

/*
 * Packed depthwise causal convolution with a carried state, followed by SiLU.
 *   x [T, C] token-major; w [C, K]; bias [C] or NULL;
 *   conv_state [num_slots, C, K-1]: the K-1 inputs that precede the first
 *   token of the sequence, oldest first; updated in place to the last K-1
 *   inputs of the extended history.
 *   out [T, C]:  y[t, c] = silu(bias[c] + sum_{j<K} w[c, j] * x_ext[t - (K-1) + j, c])
 *   where x_ext is the history (state) followed by the sequence's tokens.
 *   values [B, cap, C] or NULL: the first n_b appended inputs of sequence b
 *   (the compact capture), n_b = min(len_b, cap, capture_count[b]) -- the
 *   per-request capture_count being optional (NULL: no third bound).
 * Returns 0, 1 for a bad packing, 2 for a bad slot, 5 for a capture count
 * outside [0, cap].
 */
int conv_oracle_forward(int B, int T, int C, int K, int num_slots, const double *x,
                        const double *w, const double *bias, const int32_t *cu,
                        const int32_t *slots, double *conv_state, double *out,
                        double *values, int cap, const int32_t *capture_count) {
    if (oracle_check_cu(cu, B, T)) return 1;
    for (int s = 0; s < B; ++s) {
        int slot = slots ? slots[s] : s;
        if (slot < 0 || slot >= num_slots) return 2;
        if (capture_count && (capture_count[s] < 0 || capture_count[s] > cap)) return 5;
    }
    const int Km1 = K - 1;
#pragma omp parallel for schedule(static)
    for (int c = 0; c < C; ++c) {
        double *hist = (double *)malloc(sizeof(double) * (Km1 + 1));
        for (int s = 0; s < B; ++s) {
            const int slot = slots ? slots[s] : s;
            double *st = conv_state + ((long)slot * C + c) * Km1;
            for (int j = 0; j < Km1; ++j) hist[j] = st[j];
            for (int t = cu[s]; t < cu[s + 1]; ++t) {
                double acc = bias ? bias[c] : 0.0;
                const double xt = x[(long)t * C + c];
                for (int j = 0; j < Km1; ++j) acc += w[(long)c * K + j] * hist[j];
                acc += w[(long)c * K + Km1] * xt;
                out[(long)t * C + c] = acc / (1.0 + exp(-acc));
                for (int j = 0; j + 1 < Km1; ++j) hist[j] = hist[j + 1];
                if (Km1 > 0) hist[Km1 - 1] = xt;
                const int tl = t - cu[s];
                const int ncap = capture_count ? capture_count[s] : cap;
                if (values && tl < cap && tl < ncap) values[((long)s * cap + tl) * C + c] = xt;
            }
            for (int j = 0; j < Km1; ++j) st[j] = hist[j];
        }
        free(hist);
    }
    return 0;
}
