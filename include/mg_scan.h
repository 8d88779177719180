/*
 * mg_scan.h -- C ABI of the GB300 (sm_103a) minGRU scan library.
 *
 * The operations are those of the page "minGRU - Triton kernels"
 * (mingru.triton_scans API reference, section "Kernel entry points"):
 *
 *   mg_linear_scan_fwd   <- linear_scan_fwd        ("Channel-tiled k=1 affine prefix scan")
 *   mg_linear_scan_bwd   <- linear_scan_bwd        ("Channel-tiled k=1 affine-scan adjoint")
 *   mg_log_scan_fwd      <- parallel_scan_log_fwd  ("Fused log-space forward scan")
 *   mg_log_scan_bwd      <- its adjoint (derived; the page lists the forward only)
 *   mg_affine_scan_fwd   <- affine_scan_fwd        ("Generic k x k affine prefix scan")
 *   mg_affine_scan_bwd   <- affine_scan_bwd        ("Generic k x k affine-scan adjoint")
 *   mg_mingru_scan_fwd/bwd, mg_linear_scan_bwd_bf16_grads <- the minGRU layer's
 *                           gate fused into linear_scan_fwd/bwd, and the
 *                           backward with bf16 gradients
 *   mg_linear_scan_h0_fwd/bwd, mg_linear_scan_varlen_fwd/bwd <- linear_scan_fwd/bwd
 *                           from start states, over (B,T,D) or packed
 *                           variable-length sequences
 *   mg_affine_scan_h0_fwd/bwd <- affine_scan_fwd/bwd from start states
 *   mg_angle_scan_fwd/bwd   <- angle_scan_fwd/bwd   ("Angle-fused forward", Kernel 4)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout.  Every tensor is dense, row-major (C order), last dimension
 *   fastest: (B,T,D) element (b,t,d) sits at (b*T + t)*D + d; (B,T,n,k,k)
 *   element (b,t,n,i,j) is row i, column j of the step-t matrix.  Time index
 *   t = 1..T in the formulas is stored at 0..T-1.
 * Pointers.  All tensor pointers are DEVICE pointers of the current device,
 *   16-byte aligned.  Inputs are read-only; outputs are written in full and
 *   must not overlap any input or each other.
 * Ownership.  The caller allocates every input, output and workspace buffer.
 *   The library allocates nothing, frees nothing and keeps no state between
 *   calls apart from what it leaves in the caller's workspace.
 * Workspace.  Each call needs a device workspace of at least the size the
 *   matching *_workspace_size function returns, 256-byte aligned, zero-filled
 *   before its FIRST use (mg_workspace_init does that, or any memset to 0).
 *   After that a workspace may be reused by any later call of any op and any
 *   size up to the one it was sized for, without clearing: each launch resets
 *   its own control words.  One workspace serves one call at a time: calls
 *   that overlap on the GPU (two streams, or two threads) must use separate
 *   workspaces or they race.
 * Streams.  Calls are asynchronous on `stream` (0 = the legacy default
 *   stream).  Argument errors are reported synchronously, before any launch,
 *   by the return value.  The device-side chunk look-back waits are bounded;
 *   if one gives up (a predecessor chunk never published), the kernel still
 *   finishes, the outputs OF THAT LAUNCH are unspecified, and the next
 *   mg_workspace_status on that workspace returns MG_ERR_TIMEOUT.  The error
 *   record is tagged with the launch it belongs to: later launches on the
 *   same workspace run normally (their waits do not give up early because of
 *   it) whether or not the caller has read the record yet.
 * Errors.  Every entry point returns an mg_status.  On failure
 *   mg_last_error_detail() gives a human-readable reason (thread-local, valid
 *   until the next call on the same thread).  An out-of-envelope request
 *   (unsupported dtype, k or v) returns MG_ERR_UNSUPPORTED: there is never a
 *   silent downgrade to another implementation.
 * Degenerate sizes.  B, T, D, n equal to 0 return MG_OK without a launch
 *   (for mg_log_scan_fwd, T = 0 still needs log_values of shape (B,1,D), which
 *   is not read).  Negative sizes return MG_ERR_INVALID_ARG.  The channel-wise
 *   ops (linear, log) index channels with 32-bit integers: D above
 *   2^31 - 2^16 returns MG_ERR_UNSUPPORTED.
 * Precision.  Arithmetic and outputs are float32.  bf16 inputs (MG_BF16)
 *   are widened to float32 on load.
 */
#ifndef MG_SCAN_H
#define MG_SCAN_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MG_SCAN_ABI_VERSION 1

typedef enum mg_status {
    MG_OK = 0,
    MG_ERR_INVALID_ARG = 1,  /* bad pointer, alignment, size, overlap or workspace */
    MG_ERR_UNSUPPORTED = 2,  /* outside the kernels' envelope (dtype, k, v)        */
    MG_ERR_LAUNCH = 3,       /* the CUDA runtime refused the launch                */
    MG_ERR_TIMEOUT = 4       /* a bounded device-side look-back wait gave up       */
} mg_status;

typedef enum mg_dtype {
    MG_F32 = 0,
    MG_BF16 = 1
} mg_dtype;

/* ABI version of the loaded library (MG_SCAN_ABI_VERSION at build time). */
int mg_abi_version(void);

/* Short fixed text for a status code. */
const char *mg_strerror(mg_status status);

/* Detail of the last failure on this thread ("" if none). */
const char *mg_last_error_detail(void);

/* Workspace bytes for mg_linear_scan_fwd and mg_linear_scan_bwd on (B,T,D),
 * for either input dtype.  Returns 0 for invalid (negative) sizes. */
size_t mg_linear_scan_workspace_size(int64_t B, int64_t T, int64_t D);

/* Workspace bytes for mg_log_scan_fwd and mg_log_scan_bwd on log_coeffs of
 * shape (B,T,D). */
size_t mg_log_scan_workspace_size(int64_t B, int64_t T, int64_t D);

/* Workspace bytes for mg_affine_scan_fwd and mg_affine_scan_bwd on
 * A (B,T,n,k,k), Bm (B,T,n,k,v).  Returns 0 for an unsupported k or v. */
size_t mg_affine_scan_workspace_size(int64_t B, int64_t T, int64_t n, int k, int v);

/* Zero-fill a workspace before its first use (cudaMemsetAsync on `stream`). */
mg_status mg_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream);

/* Synchronise `stream`, then report whether any launch since the last check
 * on this workspace gave up a look-back wait (MG_ERR_TIMEOUT), and clear the
 * record.  MG_OK otherwise. */
mg_status mg_workspace_status(void *ws, cudaStream_t stream);

/*
 * linear_scan_fwd (page section "linear_scan_fwd"): a, b of shape (B,T,D)
 * with dtype in_dt (MG_F32 or MG_BF16, the same for both).  Writes float32
 *   A[b,t,d]  = a_t * A_{t-1},          A_0 = 1  (running product, inclusive)
 *   Bc[b,t,d] = a_t * Bc_{t-1} + b_t,   Bc_0 = 0 (the h_0 = 0 solution)
 * for every channel (b,d) independently.  A and Bc are (B,T,D) float32.
 */
mg_status mg_linear_scan_fwd(const void *a, const void *b, mg_dtype in_dt,
                             float *A, float *Bc,
                             int64_t B, int64_t T, int64_t D,
                             void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * linear_scan_bwd (page section "linear_scan_bwd"): reads the forward input
 * a (dtype a_dt), the forward outputs A, Bc and the upstream gradients gA,
 * gBc (all (B,T,D), float32 except a), and writes da = dL/da, db = dL/db of
 * L = sum(gA*A) + sum(gBc*Bc) (float32, (B,T,D)):
 *   mu_t  = gA_t  + a_{t+1} mu_{t+1},   lam_t = gBc_t + a_{t+1} lam_{t+1}  (zero past T)
 *   db_t  = lam_t,   da_t = mu_t A_{t-1} + lam_t Bc_{t-1}   (A_0 = 1, Bc_0 = 0)
 * The operator b is not needed.  A and Bc are used as given.
 */
mg_status mg_linear_scan_bwd(const void *a, mg_dtype a_dt,
                             const float *A, const float *Bc,
                             const float *gA, const float *gBc,
                             float *da, float *db,
                             int64_t B, int64_t T, int64_t D,
                             void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * linear_scan_bwd with the gradients rounded to bf16 (round to nearest
 * even) instead of float32: the same arguments as mg_linear_scan_bwd except
 * that da and db are (B,T,D) bf16 buffers, as autograd returns gradients in
 * the dtype of a bf16 input.  Arithmetic stays float32; only the stores
 * round.  Workspace: mg_linear_scan_workspace_size.
 */
mg_status mg_linear_scan_bwd_bf16_grads(const void *a, mg_dtype a_dt,
                                        const float *A, const float *Bc,
                                        const float *gA, const float *gBc,
                                        void *da, void *db,
                                        int64_t B, int64_t T, int64_t D,
                                        void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * linear_scan_fwd from a start state.  The page's linear and affine ops start
 * from h_0 = 0; its log-space op (section "parallel_scan_log_fwd") takes
 * log h_0 in slot 0 of log_values.  These give the linear op the same start
 * state: h0 is (B, D) float32 and, per channel,
 *   A_t = a_t A_{t-1}  (A_0 = 1),   H_t = a_t H_{t-1} + b_t  (H_0 = h0[b, d])
 * A and H are (B,T,D) float32 (H = Bc + A h0 of mg_linear_scan_fwd).
 * Workspace: mg_linear_scan_workspace_size.
 */
mg_status mg_linear_scan_h0_fwd(const void *a, const void *b, mg_dtype in_dt, const float *h0,
                                float *A, float *H,
                                int64_t B, int64_t T, int64_t D,
                                void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Gradients of L = sum(gA*A) + sum(gH*H) for mg_linear_scan_h0_fwd (A, H
 * used as given): da, db as mg_linear_scan_bwd with H_0 = h0 in da_1, and
 * dh0 = dL/dh0 = a_1 lam_1, (B, D) float32 (zero-filled for T = 0).
 */
mg_status mg_linear_scan_h0_bwd(const void *a, mg_dtype a_dt, const float *h0,
                                const float *A, const float *H,
                                const float *gA, const float *gH,
                                float *da, float *db, float *dh0,
                                int64_t B, int64_t T, int64_t D,
                                void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * The linear scan over a packed batch of variable-length sequences (the
 * ragged batch layout that the page on causal_conv1d lists among its
 * unsupported features, applied to this op).  a, b are (Ttot, D) with
 * sequence s in rows cu_seqlens[s] .. cu_seqlens[s+1]-1; cu_seqlens is a
 * DEVICE array of nseq + 1 int64 offsets (8-byte aligned), non-decreasing
 * from 0 to Ttot (empty sequences allowed).  Each sequence is an independent
 * linear scan started from h0[s] ((nseq, D) float32; NULL means 0):
 *   A_r = a_r A_{r-1},  H_r = a_r H_{r-1} + b_r,  (A, H) before the sequence = (1, h0[s])
 * A, H are (Ttot, D) float32.  A cu_seqlens that breaks the rules above is
 * detected on the device: the outputs are unspecified and the next
 * mg_workspace_status returns MG_ERR_INVALID_ARG; no memory outside the
 * buffers is touched.  Workspace: mg_linear_scan_varlen_workspace_size.
 */
size_t mg_linear_scan_varlen_workspace_size(int64_t Ttot, int64_t D);

mg_status mg_linear_scan_varlen_fwd(const void *a, const void *b, mg_dtype in_dt,
                                    const int64_t *cu_seqlens, int64_t nseq, const float *h0,
                                    float *A, float *H, int64_t Ttot, int64_t D,
                                    void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Gradients of L = sum(gA*A) + sum(gH*H) for mg_linear_scan_varlen_fwd (A, H
 * used as given): per sequence, the adjoint of mg_linear_scan_bwd with
 * (A, H) before the sequence = (1, h0[s]); dh0[s] = a_first lam_first, and 0
 * for an empty sequence.  h0 and dh0 are given together or both NULL.
 */
mg_status mg_linear_scan_varlen_bwd(const void *a, mg_dtype a_dt,
                                    const int64_t *cu_seqlens, int64_t nseq, const float *h0,
                                    const float *A, const float *H,
                                    const float *gA, const float *gH,
                                    float *da, float *db, float *dh0,
                                    int64_t Ttot, int64_t D,
                                    void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * The minGRU gate fused into linear_scan_fwd.  A minGRU layer feeds the
 * scan (page section "linear_scan_fwd", the op the layer's scan dispatch
 * min_gru._dispatch_scan calls) with, for two projections x1, x2 of its
 * input,
 *   z = sigmoid(x1),  a = 1 - z,  b = z g(x2),  g(x) = x + 0.5 (x >= 0), sigmoid(x) (x < 0)
 * This op computes a and b in registers from x1, x2 ((B,T,D), dtype x_dt,
 * MG_F32 or MG_BF16) and writes the scan of (a, b) exactly as
 * mg_linear_scan_fwd would: A (running product; may be NULL, then it is not
 * written) and Bc (the h_0 = 0 solution), float32 (B,T,D).  a and b never
 * reach memory.  Workspace: mg_mingru_scan_workspace_size.
 */
size_t mg_mingru_scan_workspace_size(int64_t B, int64_t T, int64_t D);

mg_status mg_mingru_scan_fwd(const void *x1, const void *x2, mg_dtype x_dt,
                             float *A, float *Bc,
                             int64_t B, int64_t T, int64_t D,
                             void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Gradients of the fused op: for L = sum(gA*A) + sum(gBc*Bc), with A and Bc
 * the forward outputs (used as given), writes
 *   dx1 = (db g(x2) - da) z (1 - z),   dx2 = db z g'(x2)
 * where da, db are the linear-scan adjoints (mg_linear_scan_bwd) at the
 * gate's (a, b), and g'(0) = 1 (the branch x + 0.5 defines g at 0).  gA and
 * A are optional together: NULL for both means gA = 0 (a minGRU layer's loss
 * depends on Bc = h only), and then A is not read.  dx1, dx2 are (B,T,D) of
 * dtype grad_dt (MG_F32, or MG_BF16 rounded to nearest even).  Workspace:
 * mg_mingru_scan_workspace_size.
 */
mg_status mg_mingru_scan_bwd(const void *x1, const void *x2, mg_dtype x_dt,
                             const float *A, const float *Bc,
                             const float *gA, const float *gBc,
                             void *dx1, void *dx2, mg_dtype grad_dt,
                             int64_t B, int64_t T, int64_t D,
                             void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * parallel_scan_log_fwd (page section "parallel_scan_log_fwd"):
 * log_coeffs (B,T,D) and log_values (B,T+1,D) float32, slot 0 of log_values
 * = log h_0 and slots 1..T = log b_t.  Writes the linear-space states
 *   h[b,t-1,d] = h_t = exp(log_coeffs[b,t-1,d]) h_{t-1} + exp(log_values[b,t,d])
 * for t = 1..T, computed as a log-space scan (log-sum-exp combine), so the
 * running products may leave float32 range without loss.  -inf inputs mean
 * zero coefficients or values and give h = 0 where every term is zero, never
 * NaN.  h is (B,T,D) float32.
 */
mg_status mg_log_scan_fwd(const float *log_coeffs, const float *log_values, float *h,
                          int64_t B, int64_t T, int64_t D,
                          void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Log-space scan adjoint (the backward of mg_log_scan_fwd for training; the
 * page lists only the forward op, section "parallel_scan_log_fwd", and this
 * is the gradient of its recurrence).  Inputs: log_coeffs (B,T,D),
 * log_values (B,T+1,D), the forward output h (B,T,D) and the upstream
 * gradient gh (B,T,D), all float32.  For L = sum_t gh_t h_t with
 * a_t = exp(log_coeffs_t), b_t = exp(log_values_t), h_0 = exp(log_values_0):
 *   mu_t = gh_t + a_{t+1} mu_{t+1}                    (mu_T = gh_T)
 *   dlog_coeffs_t = mu_t a_t h_{t-1}                    t = 1..T
 *   dlog_values_t = mu_t b_t (t = 1..T),   dlog_values_0 = a_1 mu_1 h_0
 * dlog_coeffs is (B,T,D), dlog_values (B,T+1,D), both written in full (for
 * T = 0, dlog_values is zero-filled).  The mu recurrence runs in linear
 * space: coefficients a_t <= 1 (log_coeffs <= 0, as in minGRU) keep it in
 * range.  Workspace: mg_log_scan_workspace_size covers this call too.
 */
mg_status mg_log_scan_bwd(const float *log_coeffs, const float *log_values, const float *h,
                          const float *gh, float *dlog_coeffs, float *dlog_values,
                          int64_t B, int64_t T, int64_t D,
                          void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * affine_scan_fwd (page section "affine_scan_fwd"): A (B,T,n,k,k) and
 * Bm (B,T,n,k,v) float32.  For every (b,n) independently writes
 *   Abar_t = A_t @ Abar_{t-1},          Abar_0 = I   (composition A_current @ A_earlier)
 *   Bbar_t = A_t @ Bbar_{t-1} + B_t,    Bbar_0 = 0
 * Abar has the shape of A, Bbar that of Bm.  k, v in {1, 2, 4, 8, 16}.
 */
mg_status mg_affine_scan_fwd(const float *A, const float *Bm, float *Abar, float *Bbar,
                             int64_t B, int64_t T, int64_t n, int k, int v,
                             void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * affine_scan_bwd (page section "affine_scan_bwd"): reads the forward input
 * A, the forward outputs Abar, Bbar and the upstream gradients gAbar, gBbar
 * (shapes of Abar, Bbar) and writes dA (shape of A) and dB (shape of Bbar),
 * the gradients of L = <gAbar, Abar> + <gBbar, Bbar>:
 *   M_t = gAbar_t + A_{t+1}^T M_{t+1},   Lam_t = gBbar_t + A_{t+1}^T Lam_{t+1}  (zero past T)
 *   dB_t = Lam_t,   dA_t = M_t Abar_{t-1}^T + Lam_t Bbar_{t-1}^T   (Abar_0 = I, Bbar_0 = 0)
 * k, v in {1, 2, 4, 8, 16}.
 */
mg_status mg_affine_scan_bwd(const float *A, const float *Abar, const float *Bbar,
                             const float *gAbar, const float *gBbar,
                             float *dA, float *dB,
                             int64_t B, int64_t T, int64_t n, int k, int v,
                             void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * affine_scan_fwd (page section "affine_scan_fwd") from a start state: H0 is
 * (B, n, k, v) float32 and, per (b, n),
 *   Abar_t = A_t @ Abar_{t-1}  (Abar_0 = I),   Bbar_t = A_t @ Bbar_{t-1} + B_t  (Bbar_0 = H0[b, n])
 * (Bbar = Bbar(H0 = 0) + Abar H0).  Workspace: mg_affine_scan_workspace_size.
 */
mg_status mg_affine_scan_h0_fwd(const float *A, const float *Bm, const float *H0,
                                float *Abar, float *Bbar,
                                int64_t B, int64_t T, int64_t n, int k, int v,
                                void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Gradients of L = <gAbar, Abar> + <gBbar, Bbar> for mg_affine_scan_h0_fwd
 * (Abar, Bbar used as given): dA, dB as mg_affine_scan_bwd with Bbar_0 = H0
 * in dA_1, and dH0 = A_1^T Lam_1 ((B, n, k, v) float32; zero-filled for
 * T = 0).  Runs the backward and then one small kernel for the first step.
 */
mg_status mg_affine_scan_h0_bwd(const float *A, const float *H0,
                                const float *Abar, const float *Bbar,
                                const float *gAbar, const float *gBbar,
                                float *dA, float *dB, float *dH0,
                                int64_t B, int64_t T, int64_t n, int k, int v,
                                void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * The angle-fused scan (page sections "angle_scan_fwd", "angle_scan_impl";
 * Kernel 4).  theta (B,T,n,R,half), scale and gamma (B,T,n), b (B,T,n,k),
 * h0 (B,n,k) are float32 device arrays, half = k/2; h (B,T,n,k) is written.
 * perm, p2p (int32) and sgn (float32) are (R,k) HOST arrays (module
 * constants; validated before launch: every perm[r] a permutation of
 * 0..k-1, p2p[r] its inverse).  The page does not define the transition;
 * this library reads it as
 *   h_t = s_t g_t Q_t h_{t-1} + b_t,  h_0 = h0,   s_t = scale_t if has_scale else 1,
 *   g_t = gamma_t if has_decay else 1,   Q_t = L_{R-1} ... L_0, where L_r
 *   rotates each pair (x_p, x_q), p = perm[r][2i], q = perm[r][2i+1], to
 *   (c x_p - s x_q, s x_p + c x_q) with c, s = cos, sin theta_{t,r,i},
 *   then multiplies each x_j by sgn[r][j].
 * scale (gamma) may be NULL when has_scale (has_decay) is 0.  k in
 * {2, 4, 8, 16, 32}, 1 <= R <= 8; T and n*R*k below 2^31
 * (MG_ERR_UNSUPPORTED otherwise).  No workspace.
 */
mg_status mg_angle_scan_fwd(const float *theta, const float *scale, const float *gamma,
                            const float *b, const float *h0,
                            const int32_t *perm, const float *sgn, const int32_t *p2p,
                            int has_scale, int has_decay, float *h,
                            int64_t B, int64_t T, int64_t n, int R, int k, cudaStream_t stream);

/*
 * Exact backward of mg_angle_scan_fwd from the stored states (page section
 * "angle_scan_bwd"): out is the forward's h (the source of every h_{t-1}),
 * grad_out = dL/dh.  Writes dtheta (shape of theta), dscale and dgamma
 * (B,T,n; zero when the flag is 0, as the page's zeros_like outputs), db
 * (shape of b) and dh0 (shape of h0).  b itself is not needed.
 */
mg_status mg_angle_scan_bwd(const float *theta, const float *scale, const float *gamma,
                            const float *h0, const float *out, const float *grad_out,
                            const int32_t *perm, const float *sgn, const int32_t *p2p,
                            int has_scale, int has_decay,
                            float *dtheta, float *dscale, float *dgamma, float *db, float *dh0,
                            int64_t B, int64_t T, int64_t n, int R, int k, cudaStream_t stream);

/*
 * mg_linear_scan_fwd without a workspace argument (the page has no
 * counterpart: this entry point exists for callers, not for the method).
 * Some callers cannot allocate device memory when they call the scan: a
 * plugin that its host framework gives no allocator, or code that must not
 * allocate once it has started (real-time loops, fixed memory budgets).  This
 * variant allocates nothing and frees nothing: its look-back workspace is a
 * static device array of mg_linear_scan_fwd_noalloc_max_scratch() bytes
 * (32 MiB) inside the library, which every GPU that loads the library holds
 * until the process exits.  The caller still passes inputs and outputs,
 * exactly as for mg_linear_scan_fwd.
 *
 * The first call on a device looks up that device's address of the array
 * (with the device current) and keeps it for the life of the process; make
 * that first call before any stream capture.  The address belongs to the
 * device's primary context: after cudaDeviceReset, or from another context
 * on the same device, the kept address is not valid and this entry point
 * must not be used.
 * Each call clears the array's two launch counters (an asynchronous memset
 * of 8 bytes on `stream`; everything else the kernel needs is tagged with
 * the launch, so the previous call's contents do no harm) and then launches
 * the same kernel as mg_linear_scan_fwd, so both give bitwise the same
 * outputs.  All calls share the one array: calls whose work overlaps on the
 * GPU (other streams, other host threads) race and must be serialised by the
 * caller.  Sizes whose forward workspace would exceed the array return
 * MG_ERR_INVALID_ARG before any launch.  That workspace depends on the
 * input dtype and on how B, T and D fall into tiles; every (B,T,D) with
 * mg_linear_scan_workspace_size(B,T,D) <= mg_linear_scan_fwd_noalloc_max_scratch()
 * is accepted.  Use mg_linear_scan_fwd with a caller workspace beyond it.  A
 * device-side wait that gave up is reported by
 * mg_linear_scan_fwd_noalloc_status.
 */
mg_status mg_linear_scan_fwd_noalloc(const void *a, const void *b, mg_dtype in_dt,
                                     float *A, float *Bc,
                                     int64_t B, int64_t T, int64_t D, cudaStream_t stream);

/* Bytes of the static scratch behind mg_linear_scan_fwd_noalloc. */
size_t mg_linear_scan_fwd_noalloc_max_scratch(void);

/* mg_workspace_status for the static scratch of mg_linear_scan_fwd_noalloc on
 * the current device: synchronises `stream`, then returns MG_ERR_TIMEOUT if a
 * look-back wait of any mg_linear_scan_fwd_noalloc call since the last query
 * gave up (MG_ERR_INVALID_ARG if calls overlapped and took bad tickets), and
 * clears the record; MG_OK otherwise.  Allocates nothing. */
mg_status mg_linear_scan_fwd_noalloc_status(cudaStream_t stream);

/*
 * Testing hook for the look-back's failure path (no counterpart on the page).
 * Runs mg_linear_scan_fwd (float32 inputs) with the look-back record of tile
 * `stall_tile` never published and every look-back wait bounded by
 * `wait_limit_ns` nanoseconds.  A successor of that tile must give up its
 * wait; the launch still completes, its outputs are unspecified, and the next
 * mg_workspace_status on `ws` returns MG_ERR_TIMEOUT.  The workspace and the
 * CUDA context stay usable.  stall_tile < 0 stalls nothing.
 */
mg_status mg_testing_linear_scan_fwd_stall(const float *a, const float *b, float *A, float *Bc,
                                           int64_t B, int64_t T, int64_t D,
                                           void *ws, size_t ws_bytes,
                                           int64_t stall_tile, uint64_t wait_limit_ns,
                                           cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MG_SCAN_H */
