/*
 * ssd_oracle.c -- plain fp64 CPU oracle of the Mamba2 SSD selective scan over
 * packed variable-length sequences.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker of the CUDA path: only
 * the tests, the package smoke check and the benchmark's CPU-baseline leg may
 * build, load or call it.  It shares no code with the CUDA library.
 *
 * What it computes (the definition the CUDA path must reproduce):
 *   The SSD scan that the pages run as a chunked kernel ("cumsum, chunk
 *   state, state passing, bmm, chunk scan", vLLM PR #61501 "Details") is,
 *   without the chunking, the token-by-token recurrence of Mamba2, kept in
 *   fp32 or better ("The FP32 recurrence and final-state writeback arithmetic
 *   remain unchanged", vLLM PR #62922 "Details").  For sequence s (tokens
 *   cu[s] .. cu[s+1]-1) and head h, with group g = h / (H/G):
 *
 *     dt'_t  = softplus(dt[t,h] + dt_bias[h])     (dt_softplus = 1)
 *            = dt[t,h] + dt_bias[h]               (dt_softplus = 0)
 *     h_0    = h_init[s,h]  (or 0)
 *     h_t[p,n] = exp(dt'_t * A[h]) * h_{t-1}[p,n] + dt'_t * x[t,h,p] * B[t,g,n]
 *     y[t,h,p] = sum_n C[t,g,n] * h_t[p,n] + D[h] * x[t,h,p]
 *
 *   y uses the state after token t's update.  The chunked form is an exact
 *   regrouping of this recurrence, so the oracle does no chunking at all.
 *
 *   Checkpoint (per-chunk) states: prefills that store Mamba checkpoints need
 *   the state at every chunk boundary ("Prefills that store Mamba checkpoints
 *   need every chunk state", vLLM PR #61501 "Details").  Read plainly: with
 *   chunk size L, row cu_chunks[s] + c of h_chunk is the state after token
 *   min((c + 1) L, len_s) - 1 of sequence s, for c = 0 .. ceil(len_s / L) - 1;
 *   the last row of a sequence is its final state.
 *
 * Everything is fp64 and walks the tokens in order; independent (sequence,
 * head) chains may run on different threads, which does not change any
 * arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(z) = log(1 + exp(z)), written in the overflow-safe form
 * max(z, 0) + log1p(exp(-|z|)). */
static double softplus(double z) {
    return (z > 0.0 ? z : 0.0) + log1p(exp(-fabs(z)));
}

int ssd_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Arguments (all arrays dense, row-major, fp64 unless noted):
 *   x [T,H,P], dt [T,H], dt_bias [H] or NULL, A [H], B/C [T,G,N], D [H] or NULL,
 *   cu_seqlens int64 [S+1], h_init [S,H,P,N] or NULL (zero initial state),
 *   y [T,H,P] (written for heads in [head_begin, head_end)),
 *   h_final [S,H,P,N] or NULL, h_inter [T,H,P,N] or NULL,
 *   chunk_size L, cu_chunks int64 [S+1] and h_chunk [cu_chunks[S],H,P,N], or
 *   h_chunk NULL (then L and cu_chunks are not read).
 * Returns 0, or -1 for inconsistent sizes.
 */
int ssd_oracle_scan(int64_t total_tokens, int32_t num_seqs, int32_t nheads,
                    int32_t headdim, int32_t dstate, int32_t ngroups,
                    int32_t head_begin, int32_t head_end,
                    const double *x, const double *dt, const double *dt_bias,
                    int32_t dt_softplus, const double *A, const double *B,
                    const double *C, const double *D, const int64_t *cu_seqlens,
                    const double *h_init, double *y, double *h_final,
                    double *h_inter, int32_t num_threads, int32_t chunk_size,
                    const int64_t *cu_chunks, double *h_chunk) {
    const int64_t T = total_tokens;
    const int S = num_seqs, H = nheads, P = headdim, N = dstate, G = ngroups;
    if (S < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0) return -1;
    if (head_begin < 0 || head_end > H || head_begin > head_end) return -1;
    if (S > 0 && (cu_seqlens[0] != 0 || cu_seqlens[S] != T)) return -1;
    for (int s = 0; s < S; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;
    if (h_chunk) {
        if (chunk_size <= 0 || cu_chunks[0] != 0) return -1;
        for (int s = 0; s < S; ++s) {
            const int64_t len = cu_seqlens[s + 1] - cu_seqlens[s];
            if (cu_chunks[s + 1] - cu_chunks[s] != (len + chunk_size - 1) / chunk_size) return -1;
        }
    }
    const int heads_per_group = H / G;
    const int nh = head_end - head_begin;
    const int64_t pairs = (int64_t)S * nh;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t job = 0; job < pairs; ++job) {
        const int s = (int)(job / nh);
        const int h = head_begin + (int)(job % nh);
        const int g = h / heads_per_group;
        double *state = (double *)malloc(sizeof(double) * (size_t)P * N);
        /* initial state */
        for (int64_t i = 0; i < (int64_t)P * N; ++i)
            state[i] = h_init ? h_init[((int64_t)s * H + h) * P * N + i] : 0.0;
        for (int64_t t = cu_seqlens[s]; t < cu_seqlens[s + 1]; ++t) {
            double z = dt[t * H + h] + (dt_bias ? dt_bias[h] : 0.0);
            double d = dt_softplus ? softplus(z) : z;
            double a = exp(d * (double)A[h]);
            const double *xt = x + (t * H + h) * P;
            const double *Bt = B + (t * G + g) * N;
            const double *Ct = C + (t * G + g) * N;
            for (int p = 0; p < P; ++p)
                for (int n = 0; n < N; ++n)
                    state[p * N + n] = a * state[p * N + n] + d * xt[p] * Bt[n];
            for (int p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int n = 0; n < N; ++n) acc += Ct[n] * state[p * N + n];
                y[(t * H + h) * P + p] = acc + (D ? D[h] : 0.0) * xt[p];
            }
            if (h_inter)
                memcpy(h_inter + (t * H + h) * (int64_t)P * N, state,
                       sizeof(double) * (size_t)P * N);
            const int64_t pos = t - cu_seqlens[s];          /* token index within the sequence */
            if (h_chunk && ((pos + 1) % chunk_size == 0 || t == cu_seqlens[s + 1] - 1)) {
                const int64_t row = cu_chunks[s] + pos / chunk_size;
                memcpy(h_chunk + (row * H + h) * (int64_t)P * N, state,
                       sizeof(double) * (size_t)P * N);
            }
        }
        if (h_final)
            memcpy(h_final + ((int64_t)s * H + h) * P * N, state,
                   sizeof(double) * (size_t)P * N);
        free(state);
    }
    return 0;
}
