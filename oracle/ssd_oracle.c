/*
 * ssd_oracle.c -- TEST INFRASTRUCTURE ONLY (never linked into the product).
 *
 * Plain, slow, fp64 CPU oracle for the Mamba2 SSD varlen prefill scan.  Only
 * tests/, the smoke check and the bench's CPU-baseline leg may load it.  It
 * shares no code, header or table with the CUDA library.
 *
 * What it computes (token by token, no chunking, no blocking):
 *   for every request i (tokens cu[i] .. cu[i+1]-1 of the packed batch) and
 *   every head h, with group g = h / (H/G):
 *     state <- initial state of (i, h)         (zeros when none is given)
 *     for each token t of request i, in order:
 *       dt'   = softplus(dt[t,h] + dt_bias[h])   softplus(v) = log1p(exp(v)),
 *                                               v itself when v > 20
 *       state = exp(dt' * A[h]) * state + dt' * x[t,h,:] (outer) B[t,g,:]
 *       y[t,h,p] = sum_n state[p,n] * C[t,g,n] + D[h] * x[t,h,p]
 *       y[t,h,p] *= silu(z[t,h,p])             (only when z is given)
 *
 * Sources: the recurrence and the y readout are the SSD scan named on the
 * "[Model] Mamba2 varlen and metadata refactor" page (Purpose, item 1: packed
 * (seqlen, hidden) tensors with cu_seqlens marking each request, so the state
 * restarts at every request boundary); the initial state that seeds each
 * request is the "prev_states or initstates" of the "[Bugfix] Mamba2 SSD
 * varlen bug fix initstates decay" page (instinctive explanation, items 1-4);
 * recording the state after chosen token counts serves the per-chunk state
 * export and the block-aligned checkpoint scatter of the "Automatic prefix
 * caching for GDN hybrid models" page (Purpose; Kernels/layers).
 * The softplus threshold, the group map h/(H/G) and the gate order
 * (scan + D skip, then silu(z)) are readings where the pages are silent.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double oracle_softplus(double v) { return v > 20.0 ? v : log1p(exp(v)); }

static double oracle_silu(double v) { return v / (1.0 + exp(-v)); }

/* Returns 0 on success, a negative code on a bad argument. */
int ssd_oracle_varlen(
    int64_t T, int32_t R, int32_t H, int32_t P, int32_t N, int32_t G,
    const int64_t *cu_seqlens, /* (R+1), cu[0] = 0, non-decreasing, cu[R] = T */
    const double *x,           /* (T,H,P) */
    const double *dt,          /* (T,H)   */
    const double *dt_bias,     /* (H)     */
    const double *A,           /* (H)     */
    const double *B,           /* (T,G,N) */
    const double *C,           /* (T,G,N) */
    const double *D,           /* (H) or NULL */
    const double *z,           /* (T,H,P) or NULL */
    const double *h0,          /* (R,H,P,N) initial states, or NULL for zeros */
    const int64_t *rec_off,    /* (R+1) offsets into rec_k, or NULL */
    const int64_t *rec_k,      /* per request, ascending token counts 0..L_i after which to record */
    int64_t n_tasks,           /* number of (request, head) pairs in tasks, when tasks != NULL */
    const int32_t *tasks,      /* (n_tasks, 2) pairs, or NULL for every pair */
    double *y,                 /* (T,H,P) out: rows of the computed pairs are written */
    double *h_final,           /* (R,H,P,N) out, or NULL */
    double *rec_states,        /* (rec_off[R], H, P, N) out, or NULL */
    int n_threads)
{
    if (T < 0 || R < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0)
        return -1;
    if (!cu_seqlens || !x || !dt || !dt_bias || !A || !B || !C || !y)
        return -2;
    if (cu_seqlens[0] != 0 || cu_seqlens[R] != T)
        return -3;
    for (int32_t i = 0; i < R; ++i)
        if (cu_seqlens[i + 1] < cu_seqlens[i])
            return -3;
    if (rec_off && (!rec_k || !rec_states))
        return -4;
    const int32_t heads_per_group = H / G;
    const int64_t total = tasks ? n_tasks : (int64_t)R * H;
    const size_t state_elems = (size_t)P * (size_t)N;
    int bad = 0;
#ifdef _OPENMP
    if (n_threads <= 0)
        n_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads) reduction(| : bad)
#endif
    for (int64_t w = 0; w < total; ++w) {
        const int32_t i = tasks ? tasks[2 * w] : (int32_t)(w / H);
        const int32_t h = tasks ? tasks[2 * w + 1] : (int32_t)(w % H);
        if (i < 0 || i >= R || h < 0 || h >= H) {
            bad = 1;
            continue;
        }
        const int32_t g = h / heads_per_group;
        double *st = (double *)malloc(state_elems * sizeof(double));
        if (!st) {
            bad = 1;
            continue;
        }
        if (h0)
            memcpy(st, h0 + ((size_t)i * H + h) * state_elems, state_elems * sizeof(double));
        else
            memset(st, 0, state_elems * sizeof(double));
        int64_t r = rec_off ? rec_off[i] : 0;
        const int64_t r_end = rec_off ? rec_off[i + 1] : 0;
        while (r < r_end && rec_k[r] == 0) {
            memcpy(rec_states + ((size_t)r * H + h) * state_elems, st, state_elems * sizeof(double));
            ++r;
        }
        for (int64_t t = cu_seqlens[i]; t < cu_seqlens[i + 1]; ++t) {
            const double dtp = oracle_softplus(dt[t * H + h] + dt_bias[h]);
            const double decay = exp(dtp * A[h]);
            const double *xt = x + ((size_t)t * H + h) * P;
            const double *Bt = B + ((size_t)t * G + g) * N;
            const double *Ct = C + ((size_t)t * G + g) * N;
            for (int32_t p = 0; p < P; ++p) {
                const double u = dtp * xt[p];
                double *row = st + (size_t)p * N;
                for (int32_t n = 0; n < N; ++n)
                    row[n] = decay * row[n] + u * Bt[n];
            }
            double *yt = y + ((size_t)t * H + h) * P;
            for (int32_t p = 0; p < P; ++p) {
                const double *row = st + (size_t)p * N;
                double acc = 0.0;
                for (int32_t n = 0; n < N; ++n)
                    acc += row[n] * Ct[n];
                if (D)
                    acc += D[h] * xt[p];
                if (z)
                    acc *= oracle_silu(z[((size_t)t * H + h) * P + p]);
                yt[p] = acc;
            }
            const int64_t k = t - cu_seqlens[i] + 1;
            while (r < r_end && rec_k[r] == k) {
                memcpy(rec_states + ((size_t)r * H + h) * state_elems, st, state_elems * sizeof(double));
                ++r;
            }
        }
        if (r != r_end)
            bad = 1; /* a requested record lies beyond the request or is out of order */
        if (h_final)
            memcpy(h_final + ((size_t)i * H + h) * state_elems, st, state_elems * sizeof(double));
        free(st);
    }
    return bad ? -5 : 0;
}
