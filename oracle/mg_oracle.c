/*
 * Float64 CPU oracle for the minGRU scan family.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the test suite, the smoke check and the bench's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA
 * library: it is the plain sequential definition of each operation, written
 * out in double precision so that a reader can check it against the source
 * page ("minGRU - Triton kernels" API reference, mingru.triton_scans) by eye.
 *
 * Layout (the plain reading of the shapes on that page): row-major C order,
 * last dimension fastest.
 *   (B,T,D)      element (b,t,d)        at (b*T + t)*D + d
 *   (B,T,n,k,k)  element (b,t,n,i,j)    at (((b*T + t)*n + n_)*k + i)*k + j
 *   (B,T,n,k,v)  element (b,t,n,i,j)    at (((b*T + t)*n + n_)*k + i)*v + j
 * Time index t runs 1..T in the formulas and is stored at 0..T-1.
 *
 * Build: gcc -O2 -ffp-contract=off -shared -fPIC (no fast-math, no FMA
 * contraction), so both x86-64 and aarch64 evaluate the same IEEE sequence.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/*
 * linear_scan_fwd -- "Channel-tiled k=1 affine prefix scan (Kernel 1)".
 * Page: mingru.triton_scans.linear_scan_fwd.
 *   A_t  = a_t * A_{t-1},           A_0 = 1   (running product, inclusive)
 *   Bc_t = a_t * Bc_{t-1} + b_t,    Bc_0 = 0  (the h_0 = 0 solution)
 */
void orc_linear_scan_fwd(const double *a, const double *b, double *A, double *Bc,
                         int64_t B, int64_t T, int64_t D)
{
    double *Ap = (double *)malloc((size_t)(D > 0 ? D : 1) * sizeof(double));
    double *h = (double *)malloc((size_t)(D > 0 ? D : 1) * sizeof(double));
    for (int64_t bi = 0; bi < B; ++bi) {
        for (int64_t d = 0; d < D; ++d) {
            Ap[d] = 1.0;
            h[d] = 0.0;
        }
        for (int64_t t = 0; t < T; ++t) {
            const int64_t row = (bi * T + t) * D;
            for (int64_t d = 0; d < D; ++d) {
                const double at = a[row + d];
                Ap[d] = at * Ap[d];
                h[d] = at * h[d] + b[row + d];
                A[row + d] = Ap[d];
                Bc[row + d] = h[d];
            }
        }
    }
    free(Ap);
    free(h);
}

/*
 * linear_scan_bwd -- "Channel-tiled k=1 affine-scan adjoint".
 * Page: mingru.triton_scans.linear_scan_bwd.  Inputs are the forward input a,
 * the forward outputs A and Bc (taken as given) and the upstream gradients
 * gA, gBc of a loss L = sum(gA*A) + sum(gBc*Bc).  Outputs da = dL/da, db = dL/db.
 *
 * Reverse-mode adjoint of the forward recurrences:
 *   mu_t  = gA_t  + a_{t+1} * mu_{t+1}     (mu_T  = gA_T)
 *   lam_t = gBc_t + a_{t+1} * lam_{t+1}    (lam_T = gBc_T)
 *   db_t  = lam_t
 *   da_t  = mu_t * A_{t-1} + lam_t * Bc_{t-1},   A_0 = 1, Bc_0 = 0
 */
void orc_linear_scan_bwd(const double *a, const double *A, const double *Bc,
                         const double *gA, const double *gBc, double *da, double *db,
                         int64_t B, int64_t T, int64_t D)
{
    double *mu = (double *)malloc((size_t)(D > 0 ? D : 1) * sizeof(double));
    double *lam = (double *)malloc((size_t)(D > 0 ? D : 1) * sizeof(double));
    for (int64_t bi = 0; bi < B; ++bi) {
        for (int64_t d = 0; d < D; ++d) {
            mu[d] = 0.0;
            lam[d] = 0.0;
        }
        for (int64_t t = T - 1; t >= 0; --t) {
            const int64_t row = (bi * T + t) * D;
            for (int64_t d = 0; d < D; ++d) {
                const double a_next = (t + 1 < T) ? a[row + D + d] : 0.0;
                mu[d] = gA[row + d] + a_next * mu[d];
                lam[d] = gBc[row + d] + a_next * lam[d];
                const double A_prev = (t > 0) ? A[row - D + d] : 1.0;
                const double Bc_prev = (t > 0) ? Bc[row - D + d] : 0.0;
                da[row + d] = mu[d] * A_prev + lam[d] * Bc_prev;
                db[row + d] = lam[d];
            }
        }
    }
    free(mu);
    free(lam);
}

/*
 * parallel_scan_log_fwd -- "Fused log-space forward scan (Kernel 2)".
 * Page: mingru.triton_scans.parallel_scan_log_fwd.  log_coeffs is (B,T,D),
 * log_values is (B,T+1,D) with slot 0 = log h_0 and slots 1..T = log b_t.
 * Returns h_1..h_T as (B,T,D), in linear space.
 *
 * The log-space scan reaches exactly the linear recurrence it encodes:
 *   h_0 = exp(log_values[0])
 *   h_t = exp(log_coeffs[t]) * h_{t-1} + exp(log_values[t]),   t = 1..T
 * with log_coeffs[t] the t-th (1-based) step, i.e. storage index t-1.  Every
 * term is non-negative, so the double-precision linear form has no
 * cancellation; -inf inputs give exp(-inf) = 0 exactly.  Its range limit:
 * inputs above about 709 overflow double.
 */
void orc_log_scan_fwd(const double *log_coeffs, const double *log_values, double *h_out,
                      int64_t B, int64_t T, int64_t D)
{
    double *h = (double *)malloc((size_t)(D > 0 ? D : 1) * sizeof(double));
    for (int64_t bi = 0; bi < B; ++bi) {
        const int64_t v0 = (bi * (T + 1)) * D;
        for (int64_t d = 0; d < D; ++d)
            h[d] = exp(log_values[v0 + d]);
        for (int64_t t = 1; t <= T; ++t) {
            const int64_t crow = (bi * T + (t - 1)) * D;   /* log_coeffs / output row */
            const int64_t vrow = (bi * (T + 1) + t) * D;   /* log_values row */
            for (int64_t d = 0; d < D; ++d) {
                h[d] = exp(log_coeffs[crow + d]) * h[d] + exp(log_values[vrow + d]);
                h_out[crow + d] = h[d];
            }
        }
    }
    free(h);
}

/*
 * Log-space scan adjoint (the backward of parallel_scan_log_fwd, for
 * training; the page lists only the forward op, the gradient is derived).
 * For a loss L = sum_t gh_t * h_t with h_t = a_t h_{t-1} + b_t,
 * a_t = exp(log_coeffs_t), b_t = exp(log_values_t), h_0 = exp(log_values_0):
 *   mu_t        = gh_t + a_{t+1} * mu_{t+1}          (mu_T = gh_T)
 *   dlog_coeffs_t = mu_t * a_t * h_{t-1}             t = 1..T
 *   dlog_values_t = mu_t * b_t                        t = 1..T
 *   dlog_values_0 = a_1 * mu_1 * h_0                  (dL/dh_0 times h_0)
 * h is recomputed here in double from the inputs.  dlog_values has the shape
 * of log_values, (B,T+1,D).
 */
void orc_log_scan_bwd(const double *log_coeffs, const double *log_values, const double *gh,
                      double *dlog_coeffs, double *dlog_values, int64_t B, int64_t T, int64_t D)
{
    double *h = (double *)malloc((size_t)(T + 1) * sizeof(double));
    for (int64_t bi = 0; bi < B; ++bi) {
        for (int64_t d = 0; d < D; ++d) {
            h[0] = exp(log_values[(bi * (T + 1)) * D + d]);
            for (int64_t t = 1; t <= T; ++t)
                h[t] = exp(log_coeffs[(bi * T + (t - 1)) * D + d]) * h[t - 1] +
                       exp(log_values[(bi * (T + 1) + t) * D + d]);
            double mu = 0.0;
            for (int64_t t = T; t >= 1; --t) {
                const int64_t crow = (bi * T + (t - 1)) * D + d;
                const int64_t vrow = (bi * (T + 1) + t) * D + d;
                const double a_next = t < T ? exp(log_coeffs[crow + D]) : 0.0;
                mu = gh[crow] + a_next * mu;
                dlog_coeffs[crow] = mu * exp(log_coeffs[crow]) * h[t - 1];
                dlog_values[vrow] = mu * exp(log_values[vrow]);
            }
            /* after the loop mu = mu_1 */
            const int64_t v0 = (bi * (T + 1)) * D + d;
            dlog_values[v0] = T >= 1 ? exp(log_coeffs[(bi * T) * D + d]) * mu * h[0] : 0.0;
        }
    }
    free(h);
}

/* C = X @ Y for row-major X (r x m), Y (m x c). */
static void mat_mul(const double *X, const double *Y, double *C, int r, int m, int c)
{
    for (int i = 0; i < r; ++i)
        for (int j = 0; j < c; ++j) {
            double s = 0.0;
            for (int l = 0; l < m; ++l)
                s += X[i * m + l] * Y[l * c + j];
            C[i * c + j] = s;
        }
}

/* C = X^T @ Y for row-major X (m x r), Y (m x c). */
static void mat_tmul(const double *X, const double *Y, double *C, int r, int m, int c)
{
    for (int i = 0; i < r; ++i)
        for (int j = 0; j < c; ++j) {
            double s = 0.0;
            for (int l = 0; l < m; ++l)
                s += X[l * r + i] * Y[l * c + j];
            C[i * c + j] = s;
        }
}

/* C += X @ Y^T for row-major X (r x m), Y (c x m). */
static void mat_mul_tadd(const double *X, const double *Y, double *C, int r, int m, int c)
{
    for (int i = 0; i < r; ++i)
        for (int j = 0; j < c; ++j) {
            double s = 0.0;
            for (int l = 0; l < m; ++l)
                s += X[i * m + l] * Y[j * m + l];
            C[i * c + j] += s;
        }
}

/*
 * affine_scan_fwd -- "Generic k x k affine prefix scan (Kernel 1)".
 * Page: mingru.triton_scans.affine_scan_fwd.  A is (B,T,n,k,k), Bm is
 * (B,T,n,k,v).  For each (b, n_) independently:
 *   Abar_t = A_t @ Abar_{t-1},          Abar_0 = I   (composition A_current @ A_earlier)
 *   Bbar_t = A_t @ Bbar_{t-1} + B_t,    Bbar_0 = 0   (the H_0 = 0 solution)
 */
void orc_affine_scan_fwd(const double *A, const double *Bm, double *Abar, double *Bbar,
                         int64_t B, int64_t T, int64_t n, int k, int v)
{
    const int64_t kk = (int64_t)k * k, kv = (int64_t)k * v;
    double *P = (double *)malloc((size_t)kk * sizeof(double));
    double *H = (double *)malloc((size_t)kv * sizeof(double));
    double *tmp = (double *)malloc((size_t)(kk > kv ? kk : kv) * sizeof(double));
    for (int64_t bi = 0; bi < B; ++bi)
        for (int64_t ni = 0; ni < n; ++ni) {
            for (int i = 0; i < k; ++i)
                for (int j = 0; j < k; ++j)
                    P[i * k + j] = (i == j) ? 1.0 : 0.0;
            memset(H, 0, (size_t)kv * sizeof(double));
            for (int64_t t = 0; t < T; ++t) {
                const int64_t s = (bi * T + t) * n + ni;
                const double *At = A + s * kk;
                mat_mul(At, P, tmp, k, k, k);
                memcpy(P, tmp, (size_t)kk * sizeof(double));
                mat_mul(At, H, tmp, k, k, v);
                for (int64_t e = 0; e < kv; ++e)
                    H[e] = tmp[e] + Bm[s * kv + e];
                memcpy(Abar + s * kk, P, (size_t)kk * sizeof(double));
                memcpy(Bbar + s * kv, H, (size_t)kv * sizeof(double));
            }
        }
    free(P);
    free(H);
    free(tmp);
}

/*
 * affine_scan_bwd -- "Generic k x k affine-scan adjoint (Kernel 3)".
 * Page: mingru.triton_scans.affine_scan_bwd.  Inputs: forward input A, forward
 * outputs Abar, Bbar (taken as given), upstream gradients gAbar, gBbar of
 * L = <gAbar, Abar> + <gBbar, Bbar>.  Outputs dA (shape of A), dB (shape of Bbar).
 *
 * Reverse-mode adjoint of the forward recurrences:
 *   M_t   = gAbar_t + A_{t+1}^T @ M_{t+1}     (k x k, M_T = gAbar_T)
 *   Lam_t = gBbar_t + A_{t+1}^T @ Lam_{t+1}   (k x v, Lam_T = gBbar_T)
 *   dB_t  = Lam_t
 *   dA_t  = M_t @ Abar_{t-1}^T + Lam_t @ Bbar_{t-1}^T,   Abar_0 = I, Bbar_0 = 0
 */
void orc_affine_scan_bwd(const double *A, const double *Abar, const double *Bbar,
                         const double *gAbar, const double *gBbar, double *dA, double *dB,
                         int64_t B, int64_t T, int64_t n, int k, int v)
{
    const int64_t kk = (int64_t)k * k, kv = (int64_t)k * v;
    double *M = (double *)malloc((size_t)kk * sizeof(double));
    double *L = (double *)malloc((size_t)kv * sizeof(double));
    double *tmp = (double *)malloc((size_t)(kk > kv ? kk : kv) * sizeof(double));
    double *eye = (double *)malloc((size_t)kk * sizeof(double));
    double *zero = (double *)calloc((size_t)kv, sizeof(double));
    for (int i = 0; i < k; ++i)
        for (int j = 0; j < k; ++j)
            eye[i * k + j] = (i == j) ? 1.0 : 0.0;
    for (int64_t bi = 0; bi < B; ++bi)
        for (int64_t ni = 0; ni < n; ++ni) {
            memset(M, 0, (size_t)kk * sizeof(double));
            memset(L, 0, (size_t)kv * sizeof(double));
            for (int64_t t = T - 1; t >= 0; --t) {
                const int64_t s = (bi * T + t) * n + ni;
                if (t + 1 < T) {
                    const double *Anext = A + (s + n) * kk;
                    mat_tmul(Anext, M, tmp, k, k, k);
                    for (int64_t e = 0; e < kk; ++e)
                        M[e] = tmp[e] + gAbar[s * kk + e];
                    mat_tmul(Anext, L, tmp, k, k, v);
                    for (int64_t e = 0; e < kv; ++e)
                        L[e] = tmp[e] + gBbar[s * kv + e];
                } else {
                    memcpy(M, gAbar + s * kk, (size_t)kk * sizeof(double));
                    memcpy(L, gBbar + s * kv, (size_t)kv * sizeof(double));
                }
                const double *Aprev = (t > 0) ? Abar + (s - n) * kk : eye;
                const double *Bprev = (t > 0) ? Bbar + (s - n) * kv : zero;
                double *dAt = dA + s * kk;
                memset(dAt, 0, (size_t)kk * sizeof(double));
                mat_mul_tadd(M, Aprev, dAt, k, k, k);
                mat_mul_tadd(L, Bprev, dAt, k, v, k);
                memcpy(dB + s * kv, L, (size_t)kv * sizeof(double));
            }
        }
    free(M);
    free(L);
    free(tmp);
    free(eye);
    free(zero);
}

/*
 * ---------------------------------------------------------------------------
 * The minGRU gate fused with the linear scan.
 *
 * A minGRU layer (the module whose scans the page "minGRU - Triton kernels"
 * serves; its dispatch section names linear_scan_fwd and
 * parallel_scan_log_fwd as the ops it calls) computes from two projections
 * x1, x2 of its input the gate z = sigmoid(x1), the coefficient a = 1 - z
 * and the value b = z * g(x2), with g(x) = x + 0.5 for x >= 0 and sigmoid(x)
 * otherwise, then scans h_t = a_t h_{t-1} + b_t.  The gate is written here as
 * that definition; 1 - sigmoid(x) is evaluated as sigmoid(-x), the same
 * number without the cancellation of 1 - z near z = 1.
 */
static double orc_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static double orc_g(double x) { return x >= 0.0 ? x + 0.5 : orc_sigmoid(x); }

/* dg/dx; at x = 0 the derivative of the branch that defines g there (x + 0.5). */
static double orc_g_grad(double x)
{
    if (x >= 0.0) return 1.0;
    const double s = orc_sigmoid(x);
    return s * (1.0 - s);
}

/* a = 1 - sigmoid(x1), b = sigmoid(x1) g(x2), elementwise over n values. */
void orc_mingru_gate(const double *x1, const double *x2, double *a, double *b, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        a[i] = orc_sigmoid(-x1[i]);
        b[i] = orc_sigmoid(x1[i]) * orc_g(x2[i]);
    }
}

/* The gate, then linear_scan_fwd: A and Bc of the scan on (a, b). */
void orc_mingru_scan_fwd(const double *x1, const double *x2, double *A, double *Bc,
                         int64_t B, int64_t T, int64_t D)
{
    const int64_t n = B * T * D;
    double *a = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    double *b = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    orc_mingru_gate(x1, x2, a, b, n);
    orc_linear_scan_fwd(a, b, A, Bc, B, T, D);
    free(a);
    free(b);
}

/*
 * Gradients dx1, dx2 of L = sum(gA*A) + sum(gBc*Bc) for the fused op, A and
 * Bc taken as given: linear_scan_bwd on the gate's (a, b) gives da, db, and
 * the chain rule through the gate gives, with z = sigmoid(x1),
 *   da/dx1 = -z (1 - z),   db/dx1 = z (1 - z) g(x2),   db/dx2 = z g'(x2)
 *   dx1 = (db g(x2) - da) z (1 - z),   dx2 = db z g'(x2),
 * with 1 - z taken as sigmoid(-x1) here too.
 */
void orc_mingru_scan_bwd(const double *x1, const double *x2, const double *A, const double *Bc,
                         const double *gA, const double *gBc, double *dx1, double *dx2,
                         int64_t B, int64_t T, int64_t D)
{
    const int64_t n = B * T * D;
    const size_t bytes = (size_t)(n > 0 ? n : 1) * sizeof(double);
    double *a = (double *)malloc(bytes), *b = (double *)malloc(bytes);
    double *da = (double *)malloc(bytes), *db = (double *)malloc(bytes);
    orc_mingru_gate(x1, x2, a, b, n);
    orc_linear_scan_bwd(a, A, Bc, gA, gBc, da, db, B, T, D);
    for (int64_t i = 0; i < n; ++i) {
        /* z (1 - z) as sigmoid(x1) sigmoid(-x1): the same number without the
         * cancellation of 1 - z near z = 1 (for x1 above ~37, 1 - z is 0 in
         * double while z (1 - z) is still representable) */
        const double z = orc_sigmoid(x1[i]), zc = orc_sigmoid(-x1[i]);
        dx1[i] = (db[i] * orc_g(x2[i]) - da[i]) * z * zc;
        dx2[i] = db[i] * z * orc_g_grad(x2[i]);
    }
    free(a);
    free(b);
    free(da);
    free(db);
}

/*
 * ---------------------------------------------------------------------------
 * Nonzero initial state and packed variable-length batches.
 *
 * The page's log-space op takes log h_0 in slot 0 of log_values; the linear
 * and affine ops start from h_0 = 0.  These give the linear recurrence a
 * caller-chosen start state and let one packed (Ttot, D) tensor hold several
 * sequences of different lengths, sequence s occupying rows cu[s] ..
 * cu[s+1]-1 (cu[0] = 0, cu[nseq] = Ttot, non-decreasing).  For each sequence
 * and channel d, with h0 the sequence's start state (0 when h0 is NULL):
 *   A_t = a_t A_{t-1},          A before the first row = 1
 *   H_t = a_t H_{t-1} + b_t,    H before the first row = h0[s, d]
 */
void orc_linear_scan_varlen_fwd(const double *a, const double *b, const int64_t *cu, int64_t nseq,
                                const double *h0, double *A, double *H, int64_t D)
{
    for (int64_t s = 0; s < nseq; ++s)
        for (int64_t d = 0; d < D; ++d) {
            double Ap = 1.0, h = h0 ? h0[s * D + d] : 0.0;
            for (int64_t r = cu[s]; r < cu[s + 1]; ++r) {
                const double at = a[r * D + d];
                Ap = at * Ap;
                h = at * h + b[r * D + d];
                A[r * D + d] = Ap;
                H[r * D + d] = h;
            }
        }
}

/*
 * Gradients of L = sum(gA*A) + sum(gH*H) for the varlen forward, A and H
 * taken as given.  Within each sequence (rows r0 .. r1-1):
 *   mu_r  = gA_r + a_{r+1} mu_{r+1},   lam_r = gH_r + a_{r+1} lam_{r+1}   (zero past r1-1)
 *   da_r  = mu_r A_{r-1} + lam_r H_{r-1},  db_r = lam_r
 * with A_{r0-1} = 1 and H_{r0-1} = h0[s, d]; and dL/dh0[s, d] = a_{r0} lam_{r0}
 * (0 for an empty sequence).  dh0 is written only when h0 is not NULL.
 */
void orc_linear_scan_varlen_bwd(const double *a, const int64_t *cu, int64_t nseq,
                                const double *h0, const double *A, const double *H,
                                const double *gA, const double *gH, double *da, double *db,
                                double *dh0, int64_t D)
{
    for (int64_t s = 0; s < nseq; ++s)
        for (int64_t d = 0; d < D; ++d) {
            double mu = 0.0, lam = 0.0;
            const int64_t r0 = cu[s], r1 = cu[s + 1];
            for (int64_t r = r1 - 1; r >= r0; --r) {
                const double a_next = (r + 1 < r1) ? a[(r + 1) * D + d] : 0.0;
                mu = gA[r * D + d] + a_next * mu;
                lam = gH[r * D + d] + a_next * lam;
                const double A_prev = (r > r0) ? A[(r - 1) * D + d] : 1.0;
                const double H_prev = (r > r0) ? H[(r - 1) * D + d] : (h0 ? h0[s * D + d] : 0.0);
                da[r * D + d] = mu * A_prev + lam * H_prev;
                db[r * D + d] = lam;
            }
            /* after the loop lam is lam_{r0} (or 0 for an empty sequence) */
            if (h0 && dh0) dh0[s * D + d] = r1 > r0 ? a[r0 * D + d] * lam : 0.0;
        }
}

/*
 * affine_scan_fwd with a caller-chosen start state H0 (B,n,k,v):
 *   Abar_t = A_t @ Abar_{t-1},  Abar_0 = I
 *   Bbar_t = A_t @ Bbar_{t-1} + B_t,  Bbar_0 = H0[b, n]
 */
void orc_affine_scan_h0_fwd(const double *A, const double *Bm, const double *H0, double *Abar,
                            double *Bbar, int64_t B, int64_t T, int64_t n, int k, int v)
{
    const int64_t kk = (int64_t)k * k, kv = (int64_t)k * v;
    double *P = (double *)malloc((size_t)kk * sizeof(double));
    double *Hs = (double *)malloc((size_t)kv * sizeof(double));
    double *tmp = (double *)malloc((size_t)(kk > kv ? kk : kv) * sizeof(double));
    for (int64_t bi = 0; bi < B; ++bi)
        for (int64_t ni = 0; ni < n; ++ni) {
            for (int i = 0; i < k; ++i)
                for (int j = 0; j < k; ++j)
                    P[i * k + j] = (i == j) ? 1.0 : 0.0;
            memcpy(Hs, H0 + (bi * n + ni) * kv, (size_t)kv * sizeof(double));
            for (int64_t t = 0; t < T; ++t) {
                const int64_t s = (bi * T + t) * n + ni;
                const double *At = A + s * kk;
                mat_mul(At, P, tmp, k, k, k);
                memcpy(P, tmp, (size_t)kk * sizeof(double));
                mat_mul(At, Hs, tmp, k, k, v);
                for (int64_t e = 0; e < kv; ++e)
                    Hs[e] = tmp[e] + Bm[s * kv + e];
                memcpy(Abar + s * kk, P, (size_t)kk * sizeof(double));
                memcpy(Bbar + s * kv, Hs, (size_t)kv * sizeof(double));
            }
        }
    free(P);
    free(Hs);
    free(tmp);
}

/*
 * Gradients of L = <gAbar, Abar> + <gBbar, Bbar> for the forward with H0:
 * the affine adjoint recurrences, with Bbar_0 = H0 in dA_1, and
 *   dH0 = A_1^T @ Lam_1   (k x v; zero when T = 0).
 */
void orc_affine_scan_h0_bwd(const double *A, const double *H0, const double *Abar,
                            const double *Bbar, const double *gAbar, const double *gBbar,
                            double *dA, double *dB, double *dH0, int64_t B, int64_t T, int64_t n,
                            int k, int v)
{
    const int64_t kk = (int64_t)k * k, kv = (int64_t)k * v;
    double *M = (double *)malloc((size_t)kk * sizeof(double));
    double *L = (double *)malloc((size_t)kv * sizeof(double));
    double *tmp = (double *)malloc((size_t)(kk > kv ? kk : kv) * sizeof(double));
    double *eye = (double *)malloc((size_t)kk * sizeof(double));
    for (int i = 0; i < k; ++i)
        for (int j = 0; j < k; ++j)
            eye[i * k + j] = (i == j) ? 1.0 : 0.0;
    for (int64_t bi = 0; bi < B; ++bi)
        for (int64_t ni = 0; ni < n; ++ni) {
            const double *h0 = H0 + (bi * n + ni) * kv;
            memset(M, 0, (size_t)kk * sizeof(double));
            memset(L, 0, (size_t)kv * sizeof(double));
            for (int64_t t = T - 1; t >= 0; --t) {
                const int64_t s = (bi * T + t) * n + ni;
                if (t + 1 < T) {
                    const double *Anext = A + (s + n) * kk;
                    mat_tmul(Anext, M, tmp, k, k, k);
                    for (int64_t e = 0; e < kk; ++e)
                        M[e] = tmp[e] + gAbar[s * kk + e];
                    mat_tmul(Anext, L, tmp, k, k, v);
                    for (int64_t e = 0; e < kv; ++e)
                        L[e] = tmp[e] + gBbar[s * kv + e];
                } else {
                    memcpy(M, gAbar + s * kk, (size_t)kk * sizeof(double));
                    memcpy(L, gBbar + s * kv, (size_t)kv * sizeof(double));
                }
                const double *Aprev = (t > 0) ? Abar + (s - n) * kk : eye;
                const double *Bprev = (t > 0) ? Bbar + (s - n) * kv : h0;
                double *dAt = dA + s * kk;
                memset(dAt, 0, (size_t)kk * sizeof(double));
                mat_mul_tadd(M, Aprev, dAt, k, k, k);
                mat_mul_tadd(L, Bprev, dAt, k, v, k);
                memcpy(dB + s * kv, L, (size_t)kv * sizeof(double));
            }
            /* after the loop L = Lam_1 */
            double *dh = dH0 + (bi * n + ni) * kv;
            if (T > 0)
                mat_tmul(A + ((bi * T) * n + ni) * kk, L, dh, k, k, v);
            else
                memset(dh, 0, (size_t)kv * sizeof(double));
        }
    free(M);
    free(L);
    free(tmp);
    free(eye);
}

/*
 * ---------------------------------------------------------------------------
 * The angle-fused scan (Kernel 4: page sections "angle_scan_fwd",
 * "angle_scan_bwd", "angle_scan_impl").  The page gives the shapes --
 * theta (B,T,n,R,half), scale and gamma (B,T,n), b (B,T,n,k), h0 (B,n,k),
 * perm/sgn/p2p (R,k), half = k/2 -- the returned state h (B,T,n,k), the
 * backward's outputs (dtheta, dscale, dgamma, db, dh0), and that scale and
 * gamma are a tanh and an exp(-lambda dt) of the module's parameters, used
 * only under has_scale / has_decay.  It does not define how theta, perm,
 * sgn and p2p form the transition.  The reading taken here (the plainest
 * one those shapes support): the transition of step t is
 *   A_t = s_t g_t Q_t,   s_t = scale_t (has_scale) or 1,  g_t = gamma_t (has_decay) or 1,
 *   Q_t = L_{R-1} ... L_1 L_0,   L_r x: for i = 0 .. half-1, with p = perm[r][2i],
 *         q = perm[r][2i+1] and c, s = cos, sin theta_{t,r,i}:
 *           (x_p, x_q) <- (c x_p - s x_q,  s x_p + c x_q)
 *         then x_j <- sgn[r][j] x_j for every j,
 * and the state runs h_t = A_t h_{t-1} + b_t from h_0 = h0 (the affine
 * recurrence of affine_scan_fwd with a vector state).  perm[r] is a
 * permutation of 0..k-1; p2p[r] is its inverse (the position of each
 * coordinate in perm[r]), which the oracle does not need.
 * The arithmetic of this reading is pinned (a hand-derived case, the dense
 * affine recurrence it equals, finite differences of its adjoint); the
 * reading itself is not fixed by the page, so against the page the angle
 * scan is "parity unpinned".
 */

/* x <- Q_t x for one step: R layers of paired rotations and signs. */
static void orc_angle_apply(double *x, const double *th, const int32_t *perm, const double *sgn,
                            int R, int k)
{
    const int half = k / 2;
    for (int r = 0; r < R; ++r) {
        for (int i = 0; i < half; ++i) {
            const int p = perm[r * k + 2 * i], q = perm[r * k + 2 * i + 1];
            const double c = cos(th[r * half + i]), s = sin(th[r * half + i]);
            const double xp = x[p], xq = x[q];
            x[p] = c * xp - s * xq;
            x[q] = s * xp + c * xq;
        }
        for (int j = 0; j < k; ++j)
            x[j] *= sgn[r * k + j];
    }
}

void orc_angle_scan_fwd(const double *theta, const double *scale, const double *gamma,
                        const double *b, const double *h0, const int32_t *perm, const double *sgn,
                        int has_scale, int has_decay, double *h_out, int64_t B, int64_t T,
                        int64_t n, int R, int k)
{
    const int half = k / 2;
    double *x = (double *)malloc((size_t)k * sizeof(double));
    for (int64_t bi = 0; bi < B; ++bi)
        for (int64_t ni = 0; ni < n; ++ni) {
            memcpy(x, h0 + (bi * n + ni) * k, (size_t)k * sizeof(double));
            for (int64_t t = 0; t < T; ++t) {
                const int64_t s = (bi * T + t) * n + ni;   /* step index (b, t, n) */
                orc_angle_apply(x, theta + s * R * half, perm, sgn, R, k);
                const double f = (has_scale ? scale[s] : 1.0) * (has_decay ? gamma[s] : 1.0);
                for (int j = 0; j < k; ++j) {
                    x[j] = f * x[j] + b[s * k + j];
                    h_out[s * k + j] = x[j];
                }
            }
        }
    free(x);
}

/*
 * Gradients of L = sum(grad_out * h) for the forward above, with the stored
 * states h (out) used as given for every h_{t-1} (h_0 = h0):
 *   lam_t = grad_out_t + A_{t+1}^T lam_{t+1}   (zero past T),   db_t = lam_t
 *   y_t = Q_t h_{t-1}:  dscale_t = g_t lam_t . y_t (has_scale),  dgamma_t = s_t lam_t . y_t (has_decay)
 *   dtheta_{t,r,i}: u = s_t g_t lam_t carried back through the layers
 *     (through the signs, then the transposed rotations), with x the input of
 *     layer r recomputed forward from h_{t-1}; for the pair (p, q) of angle i
 *     and u' the gradient after the signs:
 *       dtheta = u'_p (-s x_p - c x_q) + u'_q (c x_p - s x_q)
 *   A_t^T lam_t is that u after layer 0;  dh0 = A_1^T lam_1.
 * dscale (dgamma) is zero when has_scale (has_decay) is 0.
 */
void orc_angle_scan_bwd(const double *theta, const double *scale, const double *gamma,
                        const double *h0, const double *out, const double *grad_out,
                        const int32_t *perm, const double *sgn, int has_scale, int has_decay,
                        double *dtheta, double *dscale, double *dgamma, double *db, double *dh0,
                        int64_t B, int64_t T, int64_t n, int R, int k)
{
    const int half = k / 2;
    double *xs = (double *)malloc((size_t)(R + 1) * k * sizeof(double));   /* layer inputs */
    double *u = (double *)malloc((size_t)k * sizeof(double));
    double *lam = (double *)malloc((size_t)k * sizeof(double));
    double *carry = (double *)malloc((size_t)k * sizeof(double));
    for (int64_t bi = 0; bi < B; ++bi)
        for (int64_t ni = 0; ni < n; ++ni) {
            for (int j = 0; j < k; ++j) carry[j] = 0.0;
            for (int64_t t = T - 1; t >= 0; --t) {
                const int64_t s = (bi * T + t) * n + ni;
                const double *hp = t > 0 ? out + (s - n) * k : h0 + (bi * n + ni) * k;
                const double *th = theta + s * R * half;
                const double sc = has_scale ? scale[s] : 1.0, ga = has_decay ? gamma[s] : 1.0;
                for (int j = 0; j < k; ++j) {
                    lam[j] = grad_out[s * k + j] + carry[j];
                    db[s * k + j] = lam[j];
                }
                /* forward through the layers from h_{t-1}, keeping each layer's input */
                memcpy(xs, hp, (size_t)k * sizeof(double));
                for (int r = 0; r < R; ++r) {
                    memcpy(xs + (r + 1) * k, xs + r * k, (size_t)k * sizeof(double));
                    orc_angle_apply(xs + (r + 1) * k, th + r * half, perm + r * k, sgn + r * k, 1, k);
                }
                double dot = 0.0;   /* lam_t . y_t */
                for (int j = 0; j < k; ++j) dot += lam[j] * xs[R * k + j];
                dscale[s] = has_scale ? ga * dot : 0.0;
                dgamma[s] = has_decay ? sc * dot : 0.0;
                for (int j = 0; j < k; ++j) u[j] = sc * ga * lam[j];
                for (int r = R - 1; r >= 0; --r) {
                    const double *x = xs + r * k;
                    for (int j = 0; j < k; ++j) u[j] *= sgn[r * k + j];
                    for (int i = 0; i < half; ++i) {
                        const int p = perm[r * k + 2 * i], q = perm[r * k + 2 * i + 1];
                        const double c = cos(th[r * half + i]), sn = sin(th[r * half + i]);
                        dtheta[s * R * half + r * half + i] =
                            u[p] * (-sn * x[p] - c * x[q]) + u[q] * (c * x[p] - sn * x[q]);
                        const double up = u[p], uq = u[q];
                        u[p] = c * up + sn * uq;
                        u[q] = -sn * up + c * uq;
                    }
                }
                memcpy(carry, u, (size_t)k * sizeof(double));   /* A_t^T lam_t */
            }
            memcpy(dh0 + (bi * n + ni) * k, carry, (size_t)k * sizeof(double));
            if (T == 0)
                for (int j = 0; j < k; ++j) dh0[(bi * n + ni) * k + j] = 0.0;
        }
    free(xs);
    free(u);
    free(lam);
    free(carry);
}
