/*
 * ss_oracle.c -- plain float64 CPU reference of the Mamba selective scan (S6).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do. It shares no code with the CUDA library.
 *
 * What it computes, for every batch row b and channel d, one time step after
 * another ("Mamba and selective state spaces", box "Selective state-space
 * model (S6)" and section "The discretization the code actually uses"):
 *
 *   v       = dt[b,d,t] + dt_bias[d]                 (bias 0 when absent)
 *   delta   = softplus(v) if the flag is set, else v
 *   h[n]    = exp(delta * A[d,n]) * h[n] + delta * B[b,n,t] * x[b,d,t]
 *   y       = sum_n C[b,n,t] * h[n] + D[d] * x[b,d,t]  (state read after the
 *                                                        write of token t)
 *   y      *= z * sigmoid(z)                         (gate, when z is given;
 *                                                     "The Mamba block")
 *
 * starting from h = 0 (or from h0 when given: the decode step of "Decoding
 * with a constant-size cache" continues from a cached state). The input weight
 * is delta*B (exponential-Euler), not the zero-order-hold weight.
 *
 * Layouts (row-major, contiguous): x, dt, z, y: (batch, d_inner, L);
 * B, C: (batch, N, L); A: (d_inner, N); D, dt_bias: (d_inner);
 * h0, final_state: (batch, d_inner, N). A row is r = b * d_inner + d.
 *
 * Every quantity is double; there is no blocking, reordering or fusion beyond
 * the loop order above.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

/* log(1 + e^v), in the form max(v, 0) + log1p(e^-|v|), finite for any finite v. */
double oracle_softplus(double v)
{
    if (v > 0.0)
        return v + log1p(exp(-v));
    return log1p(exp(v));
}

static double sigmoid(double v)
{
    return 1.0 / (1.0 + exp(-v));
}

/*
 * Runs rows [row_begin, row_end). Returns 0 on success, -1 on bad arguments,
 * -2 when the state buffer cannot be allocated. D, z, dt_bias, h0 and
 * final_state may be NULL.
 */
int oracle_scan_rows(const double *x, const double *dt, const double *A,
                     const double *B, const double *C, const double *D,
                     const double *z, const double *dt_bias, int delta_softplus,
                     const double *h0, double *y, double *final_state,
                     int64_t batch, int64_t d_inner, int64_t L, int64_t N,
                     int64_t row_begin, int64_t row_end)
{
    if (!x || !dt || !A || !B || !C || !y)
        return -1;
    if (batch < 0 || d_inner < 0 || L < 0 || N <= 0)
        return -1;
    if (row_begin < 0 || row_end > batch * d_inner || row_begin > row_end)
        return -1;

    double *h = (double *)malloc((size_t)N * sizeof(double));
    if (!h)
        return -2;

    for (int64_t r = row_begin; r < row_end; ++r) {
        const int64_t b = r / d_inner;
        const int64_t d = r % d_inner;
        const double *xr = x + r * L;
        const double *dtr = dt + r * L;
        const double *zr = z ? z + r * L : NULL;
        double *yr = y + r * L;

        for (int64_t n = 0; n < N; ++n)
            h[n] = h0 ? h0[r * N + n] : 0.0;

        for (int64_t t = 0; t < L; ++t) {
            double v = dtr[t] + (dt_bias ? dt_bias[d] : 0.0);
            double delta = delta_softplus ? oracle_softplus(v) : v;

            for (int64_t n = 0; n < N; ++n) {
                double a_bar = exp(delta * A[d * N + n]);
                double write = delta * B[(b * N + n) * L + t] * xr[t];
                h[n] = a_bar * h[n] + write;
            }

            double out = 0.0;
            for (int64_t n = 0; n < N; ++n)
                out += C[(b * N + n) * L + t] * h[n];
            out += (D ? D[d] : 0.0) * xr[t];

            if (zr)
                out *= zr[t] * sigmoid(zr[t]);
            yr[t] = out;
        }

        if (final_state)
            for (int64_t n = 0; n < N; ++n)
                final_state[r * N + n] = h[n];
    }
    free(h);
    return 0;
}

/*
 * Causal depthwise convolution of "The Mamba block" (box "The Mamba block"):
 *
 *   out[b,d,t] = act( sum_{i=0}^{k-1} w[d,i] * xin[b,d,t-i] + bias[d] )
 *
 * with act = SiLU (v * sigmoid(v)) when `silu` is set, identity otherwise. The
 * inputs before t = 0 are the k-1 values in `state` (batch, k-1, d_inner),
 * oldest first, or zero when `state` is NULL (the block's zero history). When
 * `state_out` is given, the last k-1 inputs (oldest first, reaching into
 * `state` for short sequences) are written there: the decode cache that
 * prefill hands to the single-token steps ("Decoding with a constant-size
 * cache"). Layouts: xin, out (batch, d_inner, L); w (d_inner, k); bias
 * (d_inner). Runs rows r = b * d_inner + d in [row_begin, row_end).
 */
int oracle_causal_conv1d_rows(const double *xin, const double *w, const double *bias,
                              int silu, const double *state, double *out, double *state_out,
                              int64_t batch, int64_t d_inner, int64_t L, int64_t k,
                              int64_t row_begin, int64_t row_end)
{
    if (!xin || !w || !out || k < 1 || L < 0 || batch < 0 || d_inner < 0)
        return -1;
    if (row_begin < 0 || row_end > batch * d_inner || row_begin > row_end)
        return -1;
    for (int64_t r = row_begin; r < row_end; ++r) {
        const int64_t b = r / d_inner;
        const int64_t d = r % d_inner;
        const double *xr = xin + r * L;
        for (int64_t t = 0; t < L; ++t) {
            double acc = bias ? bias[d] : 0.0;
            for (int64_t i = 0; i < k; ++i) {
                const int64_t s = t - i;   /* input i steps back */
                double v;
                if (s >= 0)
                    v = xr[s];
                else if (state)
                    v = state[(b * (k - 1) + (k - 1 + s)) * d_inner + d];
                else
                    v = 0.0;
                acc += w[d * k + i] * v;
            }
            out[r * L + t] = silu ? acc * sigmoid(acc) : acc;
        }
        if (state_out) {
            for (int64_t j = 0; j < k - 1; ++j) {
                const int64_t s = L - (k - 1) + j;   /* input index held in slot j */
                double v;
                if (s >= 0)
                    v = xr[s];
                else if (state)
                    v = state[(b * (k - 1) + (k - 1 + s)) * d_inner + d];
                else
                    v = 0.0;
                state_out[(b * (k - 1) + j) * d_inner + d] = v;
            }
        }
    }
    return 0;
}

/*
 * Gradient of the selective scan (oracle_scan_rows) by the chain rule, run as
 * the pages describe the backward pass ("Mamba and selective state spaces",
 * section "Why the scan must be fused": the states are recomputed from the
 * inputs, and the backward of a linear recurrence is a linear recurrence run
 * in reverse). The formulas are derived here; the pages do not print them.
 *
 * With g(z) = z sigmoid(z) and, per row (b, d) and state n,
 *   a_t = exp(delta_t A_n),  h_t = a_t h_{t-1} + delta_t B_t x_t,
 *   y_t = sum_n C_t h_t + D x_t,  out_t = y_t g(z_t),
 * and the incoming gradients dout_t (of out) and dh_L (of the final state):
 *   gy_t     = dout_t g(z_t)                       (dout_t without the gate)
 *   dz_t     = dout_t y_t g'(z_t),  g'(z) = s (1 + z (1 - s)), s = sigmoid(z)
 *   lam_{L-1} = dh_L + C_{L-1} gy_{L-1},  lam_t = a_{t+1} lam_{t+1} + C_t gy_t
 *   dx_t     = D gy_t + sum_n lam_t delta_t B_t
 *   ddelta_t = sum_n lam_t (A_n a_t h_{t-1} + B_t x_t)
 *   dA_n    += sum_t lam_t delta_t a_t h_{t-1}
 *   dB_t[n] += lam_t delta_t x_t          (summed over the channels d)
 *   dC_t[n] += gy_t h_t                   (summed over the channels d)
 *   dD      += sum_t gy_t x_t
 *   ddt_t    = ddelta_t sigmoid(v_t) with softplus, ddelta_t without
 *   ddt_bias += sum_t ddt_t
 *   dh0[n]   = a_0 lam_0                  (gradient of the initial state)
 *
 * Per-row outputs dx, ddt, dz (batch, d_inner, L) and dh0 (batch, d_inner, N)
 * are written; dA (d_inner, N), dB, dC (batch, N, L), dD and ddt_bias
 * (d_inner) are ADDED to (the caller zeroes them). dz, dD, ddt_bias, dh0,
 * dfinal and h0 may be NULL. All states of a row are kept (L x N doubles):
 * this is the plain reference, not the recomputing kernel.
 */
int oracle_scan_bwd_rows(const double *x, const double *dt, const double *A,
                         const double *B, const double *C, const double *D,
                         const double *z, const double *dt_bias, int delta_softplus,
                         const double *h0, const double *dout, const double *dfinal,
                         double *dx, double *ddt, double *dz, double *dA, double *dB,
                         double *dC, double *dD, double *ddt_bias, double *dh0,
                         int64_t batch, int64_t d_inner, int64_t L, int64_t N,
                         int64_t row_begin, int64_t row_end)
{
    if (!x || !dt || !A || !B || !C || !dout || !dx || !ddt || !dA || !dB || !dC)
        return -1;
    if (batch < 0 || d_inner < 0 || L < 1 || N <= 0)
        return -1;
    if (row_begin < 0 || row_end > batch * d_inner || row_begin > row_end)
        return -1;

    double *hs = (double *)malloc((size_t)(L + 1) * N * sizeof(double)); /* hs[t+1] = h_t, hs[0] = h_{-1} */
    double *as = (double *)malloc((size_t)L * N * sizeof(double));
    double *del = (double *)malloc((size_t)L * sizeof(double));
    double *lam = (double *)malloc((size_t)N * sizeof(double));
    if (!hs || !as || !del || !lam) {
        free(hs); free(as); free(del); free(lam);
        return -2;
    }

    for (int64_t r = row_begin; r < row_end; ++r) {
        const int64_t b = r / d_inner;
        const int64_t d = r % d_inner;
        const double *xr = x + r * L;
        const double *dtr = dt + r * L;
        const double *zr = z ? z + r * L : NULL;
        const double *gr = dout + r * L;
        const double Dd = D ? D[d] : 0.0;

        /* forward, keeping every state */
        for (int64_t n = 0; n < N; ++n)
            hs[n] = h0 ? h0[r * N + n] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            const double v = dtr[t] + (dt_bias ? dt_bias[d] : 0.0);
            del[t] = delta_softplus ? oracle_softplus(v) : v;
            for (int64_t n = 0; n < N; ++n) {
                const double a = exp(del[t] * A[d * N + n]);
                as[t * N + n] = a;
                hs[(t + 1) * N + n] = a * hs[t * N + n] + del[t] * B[(b * N + n) * L + t] * xr[t];
            }
        }

        /* reverse */
        for (int64_t n = 0; n < N; ++n)
            lam[n] = dfinal ? dfinal[r * N + n] : 0.0;
        for (int64_t t = L - 1; t >= 0; --t) {
            double y = Dd * xr[t];
            for (int64_t n = 0; n < N; ++n)
                y += C[(b * N + n) * L + t] * hs[(t + 1) * N + n];
            double gy = gr[t];
            if (zr) {
                const double s = sigmoid(zr[t]);
                gy = gr[t] * zr[t] * s;
                if (dz)
                    dz[r * L + t] = gr[t] * y * s * (1.0 + zr[t] * (1.0 - s));
            }
            double dxt = Dd * gy;
            double ddel = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const double Bn = B[(b * N + n) * L + t];
                const double Cn = C[(b * N + n) * L + t];
                if (t < L - 1)
                    lam[n] *= as[(t + 1) * N + n];
                lam[n] += Cn * gy;
                const double ah = as[t * N + n] * hs[t * N + n];  /* a_t h_{t-1} */
                dxt += lam[n] * del[t] * Bn;
                ddel += lam[n] * (A[d * N + n] * ah + Bn * xr[t]);
                dA[d * N + n] += lam[n] * del[t] * ah;
                dB[(b * N + n) * L + t] += lam[n] * del[t] * xr[t];
                dC[(b * N + n) * L + t] += gy * hs[(t + 1) * N + n];
            }
            dx[r * L + t] = dxt;
            const double v = dtr[t] + (dt_bias ? dt_bias[d] : 0.0);
            const double dv = delta_softplus ? ddel * sigmoid(v) : ddel;
            ddt[r * L + t] = dv;
            if (ddt_bias)
                ddt_bias[d] += dv;
            if (dD)
                dD[d] += gy * xr[t];
        }
        if (dh0)
            for (int64_t n = 0; n < N; ++n)
                dh0[r * N + n] = as[n] * lam[n];
    }
    free(hs); free(as); free(del); free(lam);
    return 0;
}

/*
 * Gradient of oracle_scan_ex_rows (the scan with sequence starts and/or the
 * reverse direction). Walking order i = 0 .. L-1 visits t(i) = i, or L-1-i
 * when `reverse` is set. The scan it differentiates is, in that order,
 *   h_in(i)  = (i == 0 ? h0 : out(i-1) * (1 - e(i-1))) * (1 - c(i))
 *   out(i)   = a_t h_in(i) + delta_t B_t x_t,   y_t = C_t out(i) + D x_t (gated)
 *   final    = out(L-1) * (1 - e(L-1))
 * where the cut c(i) ("zero before the step") is seq_start[t(i)] walking
 * forward and e(i) ("zero after the step") is seq_start[t(i)] walking
 * backward (the other one is 0). Its adjoint, lam(i) = dLoss / d out(i):
 *   lam(L-1) = C gy + (1 - e(L-1)) dfinal
 *   lam(i)   = C_t gy_t + (1 - e(i)) (1 - c(i+1)) a_{t(i+1)} lam(i+1)
 *   dh0      = (1 - c(0)) a_{t(0)} lam(0)
 * and every term that the plain backward forms with a_t h_{t-1} uses
 * a_t h_in(i). The per-step formulas are those of oracle_scan_bwd_rows.
 */
int oracle_scan_bwd_ex_rows(const double *x, const double *dt, const double *A,
                            const double *B, const double *C, const double *D,
                            const double *z, const double *dt_bias, int delta_softplus,
                            const double *h0, const unsigned char *seq_start, int reverse,
                            const double *dout, const double *dfinal,
                            double *dx, double *ddt, double *dz, double *dA, double *dB,
                            double *dC, double *dD, double *ddt_bias, double *dh0,
                            int64_t batch, int64_t d_inner, int64_t L, int64_t N,
                            int64_t row_begin, int64_t row_end)
{
    if (!x || !dt || !A || !B || !C || !dout || !dx || !ddt || !dA || !dB || !dC)
        return -1;
    if (batch < 0 || d_inner < 0 || L < 1 || N <= 0)
        return -1;
    if (row_begin < 0 || row_end > batch * d_inner || row_begin > row_end)
        return -1;

    double *hin = (double *)malloc((size_t)L * N * sizeof(double));   /* h_in(i), by walking index */
    double *out = (double *)malloc((size_t)L * N * sizeof(double));   /* out(i) */
    double *as = (double *)malloc((size_t)L * N * sizeof(double));    /* a_{t(i)} */
    double *del = (double *)malloc((size_t)L * sizeof(double));       /* delta_{t(i)} */
    double *lam = (double *)malloc((size_t)N * sizeof(double));
    double *h = (double *)malloc((size_t)N * sizeof(double));
    if (!hin || !out || !as || !del || !lam || !h) {
        free(hin); free(out); free(as); free(del); free(lam); free(h);
        return -2;
    }

    for (int64_t r = row_begin; r < row_end; ++r) {
        const int64_t b = r / d_inner;
        const int64_t d = r % d_inner;
        const double *xr = x + r * L;
        const double *dtr = dt + r * L;
        const double *zr = z ? z + r * L : NULL;
        const double *gr = dout + r * L;
        const double Dd = D ? D[d] : 0.0;
#define TW(i) (reverse ? L - 1 - (i) : (i))
#define CUT_BEFORE(i) (!reverse && seq_start && seq_start[b * L + TW(i)])
#define CUT_AFTER(i) (reverse && seq_start && seq_start[b * L + TW(i)])

        /* forward in walking order, keeping h_in and out of every step */
        for (int64_t n = 0; n < N; ++n)
            h[n] = h0 ? h0[r * N + n] : 0.0;
        for (int64_t i = 0; i < L; ++i) {
            const int64_t t = TW(i);
            if (CUT_BEFORE(i))
                for (int64_t n = 0; n < N; ++n)
                    h[n] = 0.0;
            const double v = dtr[t] + (dt_bias ? dt_bias[d] : 0.0);
            del[i] = delta_softplus ? oracle_softplus(v) : v;
            for (int64_t n = 0; n < N; ++n) {
                const double a = exp(del[i] * A[d * N + n]);
                as[i * N + n] = a;
                hin[i * N + n] = h[n];
                h[n] = a * h[n] + del[i] * B[(b * N + n) * L + t] * xr[t];
                out[i * N + n] = h[n];
            }
            if (CUT_AFTER(i))
                for (int64_t n = 0; n < N; ++n)
                    h[n] = 0.0;
        }

        /* adjoint, walking order reversed */
        for (int64_t n = 0; n < N; ++n)
            lam[n] = dfinal ? dfinal[r * N + n] : 0.0;
        for (int64_t i = L - 1; i >= 0; --i) {
            const int64_t t = TW(i);
            if (i < L - 1) {
                const int cut = CUT_BEFORE(i + 1);
                for (int64_t n = 0; n < N; ++n)
                    lam[n] = cut ? 0.0 : lam[n] * as[(i + 1) * N + n];
            }
            if (CUT_AFTER(i))
                for (int64_t n = 0; n < N; ++n)
                    lam[n] = 0.0;
            double y = Dd * xr[t];
            for (int64_t n = 0; n < N; ++n)
                y += C[(b * N + n) * L + t] * out[i * N + n];
            double gy = gr[t];
            if (zr) {
                const double s = sigmoid(zr[t]);
                gy = gr[t] * zr[t] * s;
                if (dz)
                    dz[r * L + t] = gr[t] * y * s * (1.0 + zr[t] * (1.0 - s));
            }
            double dxt = Dd * gy;
            double ddel = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const double Bn = B[(b * N + n) * L + t];
                const double Cn = C[(b * N + n) * L + t];
                lam[n] += Cn * gy;
                const double ah = as[i * N + n] * hin[i * N + n];   /* a_t h_in(i) */
                dxt += lam[n] * del[i] * Bn;
                ddel += lam[n] * (A[d * N + n] * ah + Bn * xr[t]);
                dA[d * N + n] += lam[n] * del[i] * ah;
                dB[(b * N + n) * L + t] += lam[n] * del[i] * xr[t];
                dC[(b * N + n) * L + t] += gy * out[i * N + n];
            }
            dx[r * L + t] = dxt;
            const double v = dtr[t] + (dt_bias ? dt_bias[d] : 0.0);
            const double dv = delta_softplus ? ddel * sigmoid(v) : ddel;
            ddt[r * L + t] = dv;
            if (ddt_bias)
                ddt_bias[d] += dv;
            if (dD)
                dD[d] += gy * xr[t];
        }
        if (dh0) {
            const int cut = CUT_BEFORE(0);
            for (int64_t n = 0; n < N; ++n)
                dh0[r * N + n] = cut ? 0.0 : as[n] * lam[n];
        }
#undef TW
#undef CUT_BEFORE
#undef CUT_AFTER
    }
    free(hin); free(out); free(as); free(del); free(lam); free(h);
    return 0;
}

/*
 * The scan with the options of the extended entry point, written as its
 * definition: the same step as oracle_scan_rows, walked over t = 0 .. L-1 or,
 * when `reverse` is set, over t = L-1 .. 0 (h_t = a_t h_{t+1} + delta_t B_t x_t,
 * one direction of a bidirectional layer). `seq_start` (batch, L), when given,
 * marks the first step of each sequence packed into a row ("What each parameter
 * does": the state should forget everything at a document break): nothing is
 * carried across the boundary between t-1 and t, so the state is set to zero
 * before step t when walking forward and after step t when walking backward.
 * The walk starts from h0 (or zero).
 */
int oracle_scan_ex_rows(const double *x, const double *dt, const double *A,
                        const double *B, const double *C, const double *D,
                        const double *z, const double *dt_bias, int delta_softplus,
                        const double *h0, const unsigned char *seq_start, int reverse,
                        double *y, double *final_state,
                        int64_t batch, int64_t d_inner, int64_t L, int64_t N,
                        int64_t row_begin, int64_t row_end)
{
    if (!x || !dt || !A || !B || !C || !y)
        return -1;
    if (batch < 0 || d_inner < 0 || L < 0 || N <= 0)
        return -1;
    if (row_begin < 0 || row_end > batch * d_inner || row_begin > row_end)
        return -1;
    double *h = (double *)malloc((size_t)N * sizeof(double));
    if (!h)
        return -2;
    for (int64_t r = row_begin; r < row_end; ++r) {
        const int64_t b = r / d_inner;
        const int64_t d = r % d_inner;
        for (int64_t n = 0; n < N; ++n)
            h[n] = h0 ? h0[r * N + n] : 0.0;
        for (int64_t i = 0; i < L; ++i) {
            const int64_t t = reverse ? L - 1 - i : i;
            const int starts = seq_start && seq_start[b * L + t];
            if (starts && !reverse)
                for (int64_t n = 0; n < N; ++n)
                    h[n] = 0.0;
            const double v = dt[r * L + t] + (dt_bias ? dt_bias[d] : 0.0);
            const double delta = delta_softplus ? oracle_softplus(v) : v;
            double out = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                h[n] = exp(delta * A[d * N + n]) * h[n] + delta * B[(b * N + n) * L + t] * x[r * L + t];
                out += C[(b * N + n) * L + t] * h[n];
            }
            out += (D ? D[d] : 0.0) * x[r * L + t];
            if (z)
                out *= z[r * L + t] * sigmoid(z[r * L + t]);
            y[r * L + t] = out;
            if (starts && reverse)
                for (int64_t n = 0; n < N; ++n)
                    h[n] = 0.0;
        }
        if (final_state)
            for (int64_t n = 0; n < N; ++n)
                final_state[r * N + n] = h[n];
    }
    free(h);
    return 0;
}

/*
 * Mamba-2's scalar-decay scan (SSD), written as its recurrence ("Mamba and
 * selective state spaces": each head, a group of P channels, has one scalar
 * decay; "Mamba in practice": h_t = alpha_t h_{t-1} + Bbar_t x_t with the
 * decay a scalar). Per batch b, head h (group g = h / (H / G)):
 *
 *   delta_t = softplus(dt[b,t,h] + dt_bias[h])   (or dt + dt_bias)
 *   alpha_t = exp(delta_t * A[h])
 *   S_t[p][n] = alpha_t * S_{t-1}[p][n] + delta_t * x[b,t,h,p] * B[b,t,g,n]
 *   y[b,t,h,p] = sum_n C[b,t,g,n] * S_t[p][n] + D[h] * x[b,t,h,p]
 *   y *= z * sigmoid(z)                          (when z is given)
 *
 * from S_{-1} = h0[b,h] (or 0). Layouts (time-major, as a projection writes
 * them): x, z, y (batch, L, H, P); dt (batch, L, H); B, C (batch, L, G, N);
 * A, D, dt_bias (H); h0, final_state (batch, H, P, N). Runs heads
 * (b, h) = r / H, r % H for r in [row_begin, row_end).
 */
int oracle_ssd_rows(const double *x, const double *dt, const double *A, const double *B,
                    const double *C, const double *D, const double *z, const double *dt_bias,
                    int delta_softplus, const double *h0, double *y, double *final_state,
                    int64_t batch, int64_t L, int64_t H, int64_t P, int64_t G, int64_t N,
                    int64_t row_begin, int64_t row_end)
{
    if (!x || !dt || !A || !B || !C || !y || G <= 0 || H % G != 0)
        return -1;
    if (batch < 0 || L < 0 || H <= 0 || P <= 0 || N <= 0)
        return -1;
    if (row_begin < 0 || row_end > batch * H || row_begin > row_end)
        return -1;
    double *S = (double *)malloc((size_t)(P * N) * sizeof(double));
    if (!S)
        return -2;
    for (int64_t r = row_begin; r < row_end; ++r) {
        const int64_t b = r / H;
        const int64_t h = r % H;
        const int64_t g = h / (H / G);
        for (int64_t i = 0; i < P * N; ++i)
            S[i] = h0 ? h0[r * P * N + i] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            const double v = dt[(b * L + t) * H + h] + (dt_bias ? dt_bias[h] : 0.0);
            const double delta = delta_softplus ? oracle_softplus(v) : v;
            const double alpha = exp(delta * A[h]);
            const double *Bt = B + ((b * L + t) * G + g) * N;
            const double *Ct = C + ((b * L + t) * G + g) * N;
            for (int64_t p = 0; p < P; ++p) {
                const double xv = x[((b * L + t) * H + h) * P + p];
                double out = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    S[p * N + n] = alpha * S[p * N + n] + delta * xv * Bt[n];
                    out += Ct[n] * S[p * N + n];
                }
                out += (D ? D[h] : 0.0) * xv;
                const int64_t o = ((b * L + t) * H + h) * P + p;
                if (z)
                    out *= z[o] * sigmoid(z[o]);
                y[o] = out;
            }
        }
        if (final_state)
            for (int64_t i = 0; i < P * N; ++i)
                final_state[r * P * N + i] = S[i];
    }
    free(S);
    return 0;
}
