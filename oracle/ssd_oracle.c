/*
 * ssd_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 CPU oracle for the forward Mamba-2 SSD (structured
 * state-space duality) scan.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library; the product path
 * (libssd) never does.  It shares no code, header or constant with the CUDA
 * path.
 *
 * What it computes is the definition of the method: the sequential
 * recurrence, one time step after another, in double precision.
 *
 *   dt_t   = softplus(dt_raw[b,t,h] + dt_bias[h])
 *   A_h    = -exp(A_log[h])                  (A_log stores log(-A))
 *   dA_t   = exp(dt_t * A_h)
 *   h_t    = dA_t * h_{t-1} + dt_t * B_t x_t^T   (state N x P per head)
 *   y_t    = C_t^T h_t + D_h * x_t
 *
 * Sources followed:
 *   - @seanhogg/builderforce-memory-engine 2026.6.18, package/dist/kernels/
 *     ssd.js (and ssd.d.ts), header comment of the SSD module: scalar decay
 *     per head, MIMO state per head, D skip per head, buffer layouts
 *     x[B,L,H*P], B/C[B,L,G,N], dt[B,L,H], A_log/dt_bias/D[H]; A_log is
 *     documented there as "log(-A)".
 *   - same page, WGSL entry point ssd_chunk_forward: order of a time step
 *     (decay the carried state, add the input term, read the output from the
 *     updated state, add the D skip), head -> group map
 *     group = head * G / H, dt = softplus(dt_raw + dt_bias), carry-in state
 *     feeding the first step.
 *   - where that page disagrees with itself (its A is -softplus(A_log) in
 *     the kernel, -exp via "log(-A)" in the layout note; its input term
 *     omits dt; its readout sums over the head dimension), the readings
 *     taken are: A = -exp(A_log), input term dt * B x^T, readout per
 *     channel p.  These are the discretised Mamba-2 SSD recurrence that the
 *     project's statement of the method fixes.
 *
 * Layouts (row-major, contiguous):
 *   x, y        [B, L, H, P]
 *   dt_raw      [B, L, H]
 *   B, C        [B, L, G, N]
 *   dt_bias, A_log, D  [H]
 *   init_state, final_state  [B, H, P, N]   (state stored P-major, N-minor)
 *
 * Work is split over (batch, head) pairs with OpenMP; each pair runs the
 * plain time loop.  No blocking, fusion or reordering of the arithmetic.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(z) = log(1 + e^z), written in the overflow-free form
 * max(z, 0) + log1p(exp(-|z|)). */
static double oracle_softplus(double z)
{
    return (z > 0.0 ? z : 0.0) + log1p(exp(-fabs(z)));
}

double ssd_oracle_softplus(double z) { return oracle_softplus(z); }

/* Returns 0 on success, -1 on bad sizes, -2 on allocation failure. */
int ssd_oracle_fwd(const double *x, const double *dt_raw, const double *dt_bias,
                   const double *A_log, const double *Bm, const double *Cm,
                   const double *D, const double *init_state, double *y,
                   double *final_state, long batch, long seqlen, long nheads,
                   long headdim, long dstate, long ngroups, int nthreads)
{
    if (batch < 0 || seqlen < 0 || nheads <= 0 || headdim <= 0 || dstate <= 0 ||
        ngroups <= 0 || nheads % ngroups != 0)
        return -1;
    const long H = nheads, P = headdim, N = dstate, G = ngroups, L = seqlen;
    const long pairs = batch * H;
    int status = 0;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long bh = 0; bh < pairs; ++bh) {
        const long b = bh / H, h = bh % H;
        const long g = h * G / H; /* head -> group */
        double *hs = (double *)malloc(sizeof(double) * (size_t)(N * P)); /* hs[n][p] */
        if (!hs) {
            status = -2;
            continue;
        }
        for (long n = 0; n < N; ++n)
            for (long p = 0; p < P; ++p)
                hs[n * P + p] = init_state ? init_state[((b * H + h) * P + p) * N + n] : 0.0;
        const double A = -exp(A_log[h]);
        for (long t = 0; t < L; ++t) {
            const double dt = oracle_softplus(dt_raw[(b * L + t) * H + h] + dt_bias[h]);
            const double dA = exp(dt * A);
            const double *xv = x + ((b * L + t) * H + h) * P;
            const double *Bv = Bm + ((b * L + t) * G + g) * N;
            const double *Cv = Cm + ((b * L + t) * G + g) * N;
            double *yv = y + ((b * L + t) * H + h) * P;
            /* h_t = dA_t h_{t-1} + dt_t B_t x_t^T */
            for (long n = 0; n < N; ++n)
                for (long p = 0; p < P; ++p)
                    hs[n * P + p] = dA * hs[n * P + p] + dt * Bv[n] * xv[p];
            /* y_t = C_t^T h_t + D_h x_t */
            for (long p = 0; p < P; ++p) {
                double acc = 0.0;
                for (long n = 0; n < N; ++n)
                    acc += Cv[n] * hs[n * P + p];
                yv[p] = acc + D[h] * xv[p];
            }
        }
        if (final_state)
            for (long n = 0; n < N; ++n)
                for (long p = 0; p < P; ++p)
                    final_state[((b * H + h) * P + p) * N + n] = hs[n * P + p];
        free(hs);
    }
    return status;
}

int ssd_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
