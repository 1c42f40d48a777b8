/*
 * ss_scan.h -- C ABI of the B300 (sm_103a) selective-scan library (libssscan.so).
 *
 * Besides the scan and its decode update, the library carries the causal
 * depthwise convolution that feeds the scan in a Mamba block, with its
 * decode cache.
 *
 * The library computes the Mamba selective state-space layer (S6) forward
 * pass and its single-token state update, as defined in "Mamba and selective
 * state spaces" (box "Selective state-space model (S6)", section "The
 * discretization the code actually uses"):
 *
 *   delta_t   = softplus(dt_t + dt_bias_d)             (or dt_t + dt_bias_d)
 *   h_t[n]    = exp(delta_t * A[d,n]) * h_{t-1}[n] + delta_t * B_t[n] * x_t
 *   y_t       = sum_n C_t[n] * h_t[n] + D[d] * x_t
 *   out_t     = y_t * z_t * sigmoid(z_t)                (gate, "The Mamba block")
 *
 * with the exponential-Euler input weight delta*B (not zero-order hold), the
 * state read after the write of token t, and h_0 = 0.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor pointer is DEVICE memory of the current CUDA device,
 *   contiguous and row-major, owned by the caller. The library allocates
 *   nothing and keeps no state between calls, apart from a thread-local
 *   message for the last error (ss_last_error) and the built-in scratch of
 *   ss_scan_bwd_noalloc_* (see there).
 * - A is the negative real state eigenvalue lambda itself (not its log).
 *   A, D, dt_bias and every state buffer are fp32 whatever the io dtype.
 * - "bf16" arguments are raw bfloat16 bit patterns (ss_bf16).
 * - Work is enqueued on `stream` (0 = legacy default stream) and the call
 *   returns without synchronising: a fault during execution surfaces at the
 *   caller's next synchronisation, like any CUDA launch.
 * - Arguments are validated on the host before anything is enqueued; a
 *   non-zero ss_status means nothing was launched. There is no CPU fallback.
 * - Outputs must not overlap any input.
 */
#ifndef SS_SCAN_H
#define SS_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *cudaStream_t;
typedef uint16_t ss_bf16; /* raw bfloat16 bits */

typedef enum ss_status {
    SS_OK = 0,
    SS_ERR_NULL = -1,        /* a required pointer is NULL */
    SS_ERR_DIM = -2,         /* a size is <= 0 or the element count overflows */
    SS_ERR_N = -3,           /* N outside [1, SS_MAX_N] */
    SS_ERR_DEVICE_PTR = -4,  /* a pointer is not device memory of the current device */
    SS_ERR_LAUNCH = -5,      /* the kernel launch itself failed */
    SS_ERR_INTERNAL = -6     /* a CUDA runtime query failed */
} ss_status;

#define SS_MAX_N 64
#define SS_ABI_VERSION 2

/*
 * ss_scan_fwd_bf16 / ss_scan_fwd_f32 -- selective scan over a whole sequence.
 *
 * Defines: "Mamba and selective state spaces", box "Selective state-space
 * model (S6)" (the recurrence and readout), section "The discretization the
 * code actually uses" (input weight delta*B), section "The Mamba block" (the
 * silu(z) gate); the fused one-pass design of section "Why the scan must be
 * fused" (only x, delta, z, B, C, A are read, only y and the final state are
 * written; the (batch, L, d_inner, N) states are never stored).
 *
 *   x, delta, z : (batch, d_inner, L) io dtype. `delta` is the raw step dt.
 *   A           : (d_inner, N) fp32, the eigenvalues lambda (normally < 0).
 *   B, C        : (batch, N, L) io dtype, shared by all channels.
 *   D           : (d_inner) fp32 skip weight, or NULL for none.
 *   z           : or NULL for no gate.
 *   dt_bias     : (d_inner) fp32, or NULL for a bias of 0.
 *   delta_softplus : non-zero: step = softplus(delta + dt_bias);
 *                    zero:     step = delta + dt_bias.
 *                    The bias is added exactly once in either case.
 *   y           : (batch, d_inner, L) io dtype output (gated when z != NULL).
 *   final_state : (batch, d_inner, N) fp32 output h_L, or NULL to skip.
 *   batch, d_inner, L >= 1; 1 <= N <= SS_MAX_N.
 *
 * Errors: SS_ERR_NULL (x, delta, A, B, C or y NULL), SS_ERR_DIM, SS_ERR_N,
 * SS_ERR_DEVICE_PTR, SS_ERR_LAUNCH, SS_ERR_INTERNAL.
 * Alignment: 16-byte aligned io pointers and L a multiple of 16 select the
 * vectorised path; any other layout takes a scalar-load path (not an error).
 */
ss_status ss_scan_fwd_bf16(const ss_bf16 *x, const ss_bf16 *delta, const float *A,
                           const ss_bf16 *B, const ss_bf16 *C, const float *D,
                           const ss_bf16 *z, const float *dt_bias, int delta_softplus,
                           ss_bf16 *y, float *final_state, int64_t batch,
                           int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream);

ss_status ss_scan_fwd_f32(const float *x, const float *delta, const float *A,
                          const float *B, const float *C, const float *D,
                          const float *z, const float *dt_bias, int delta_softplus,
                          float *y, float *final_state, int64_t batch,
                          int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream);

/*
 * ss_scan_fwd_ex_bf16 / ss_scan_fwd_ex_f32 -- ss_scan_fwd_* with three
 * extensions, each off when its argument is NULL / 0:
 *
 *   h0        : (batch, d_inner, N) fp32 state before the first step walked
 *               (chunked prefill continues from a cached state, "Decoding with
 *               a constant-size cache"); NULL = zero.
 *   seq_start : (batch, L) bytes; non-zero at t means a new sequence starts
 *               there (documents packed into one row, "What each parameter
 *               does": the state should forget everything at a document
 *               break). Nothing carries across the boundary between t-1 and
 *               t: the state entering step t is zero (forward), or the state
 *               leaving step t towards t-1 is zero (reverse). h0 reaches only
 *               the first sequence walked.
 *   reverse   : non-zero runs the recurrence from t = L-1 down to 0,
 *               h_t = exp(delta_t A) h_{t+1} + delta_t B_t x_t, y_t read from h_t
 *               (one direction of a bidirectional layer, "Mamba and selective
 *               state spaces", section on later uses: Vision Mamba scans
 *               patches both ways); final_state is then the state after t = 0.
 *
 * Other arguments as ss_scan_fwd_*. With any extension on, 1 <= N <= 32
 * (SS_ERR_N otherwise).
 */
ss_status ss_scan_fwd_ex_bf16(const ss_bf16 *x, const ss_bf16 *delta, const float *A,
                              const ss_bf16 *B, const ss_bf16 *C, const float *D,
                              const ss_bf16 *z, const float *dt_bias, int delta_softplus,
                              const float *h0, const uint8_t *seq_start, int reverse, ss_bf16 *y,
                              float *final_state, int64_t batch, int64_t d_inner, int64_t L,
                              int64_t N, cudaStream_t stream);

ss_status ss_scan_fwd_ex_f32(const float *x, const float *delta, const float *A, const float *B,
                             const float *C, const float *D, const float *z, const float *dt_bias,
                             int delta_softplus, const float *h0, const uint8_t *seq_start,
                             int reverse, float *y, float *final_state, int64_t batch,
                             int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream);

/*
 * ss_state_update_bf16 / ss_state_update_f32 -- one decode step on a cached
 * state, "Mamba and selective state spaces", section "Decoding with a
 * constant-size cache": the state update of the definition applied once,
 * O(d_inner * N) work whatever the context length.
 *
 *   state  : (batch, d_inner, N) fp32, read and updated in place
 *            (h <- exp(delta*A) * h + delta * B * x).
 *   x, delta, z, y : (batch, d_inner) io dtype; `delta` is the final positive
 *            step (no bias, no softplus is applied here).
 *   A      : (d_inner, N) fp32.  D : (d_inner) fp32 or NULL.  z : or NULL.
 *   B, C   : (batch, N) io dtype.
 *   y      : output, sum_n C[n] * h[n] + D * x, gated by silu(z).
 *
 * Errors: as ss_scan_fwd_*; state, x, delta, A, B, C and y are required.
 */
ss_status ss_state_update_bf16(float *state, const ss_bf16 *x, const ss_bf16 *delta,
                               const float *A, const ss_bf16 *B, const ss_bf16 *C,
                               const float *D, const ss_bf16 *z, ss_bf16 *y,
                               int64_t batch, int64_t d_inner, int64_t N,
                               cudaStream_t stream);

ss_status ss_state_update_f32(float *state, const float *x, const float *delta,
                              const float *A, const float *B, const float *C,
                              const float *D, const float *z, float *y,
                              int64_t batch, int64_t d_inner, int64_t N,
                              cudaStream_t stream);

#define SS_MAX_CONV_K 8

/*
 * ss_causal_conv1d_bf16 / ss_causal_conv1d_f32 -- the causal depthwise
 * convolution that precedes the scan in a Mamba block ("Mamba and selective
 * state spaces", box "The Mamba block"):
 *
 *   out[b,d,t] = act( sum_{i=0}^{k-1} w[d,i] * x[b,d,t-i] + bias[d] ),
 *   act = SiLU(v) = v * sigmoid(v) when `silu` is non-zero, identity otherwise,
 *
 * where w[d,i] weighs the input i steps back and the inputs before t = 0 are
 * zero ("x~_s = 0 for s <= 0"), or, when `state_in` is given, the k-1 inputs
 * that preceded this call.
 *
 *   x, out         : (batch, d_inner, L) io dtype.
 *   w              : (d_inner, k) fp32.   bias : (d_inner) fp32 or NULL.
 *   state_in       : (batch, k-1, d_inner) io dtype, oldest first, or NULL.
 *   state_out      : (batch, k-1, d_inner) io dtype or NULL: receives the last
 *                    k-1 inputs, oldest first -- the decode cache that prefill
 *                    hands to ss_conv_state_update ("Decoding with a
 *                    constant-size cache"). It must not overlap state_in.
 *   1 <= k <= SS_MAX_CONV_K.
 * Errors: as ss_scan_fwd_* (SS_ERR_DIM also for k out of range).
 */
ss_status ss_causal_conv1d_bf16(const ss_bf16 *x, const float *w, const float *bias,
                                const ss_bf16 *state_in, int silu, ss_bf16 *out,
                                ss_bf16 *state_out, int64_t batch, int64_t d_inner,
                                int64_t L, int64_t k, cudaStream_t stream);

ss_status ss_causal_conv1d_f32(const float *x, const float *w, const float *bias,
                               const float *state_in, int silu, float *out, float *state_out,
                               int64_t batch, int64_t d_inner, int64_t L, int64_t k,
                               cudaStream_t stream);

/*
 * ss_conv_state_update_bf16 / ss_conv_state_update_f32 -- one decode step of
 * the convolution ("Decoding with a constant-size cache"): with the cached
 * k-1 previous inputs and the new input x, out = act(sum_i w[d,i] x_{t-i} +
 * bias[d]); then the cache drops its oldest entry and appends x (the cache
 * holds the convolution's inputs, not its outputs).
 *
 *   conv_state : (batch, k-1, d_inner) io dtype, oldest first, updated in
 *                place (may be NULL when k = 1).
 *   x, out     : (batch, d_inner) io dtype.  w : (d_inner, k).  bias : or NULL.
 */
ss_status ss_conv_state_update_bf16(ss_bf16 *conv_state, const ss_bf16 *x, const float *w,
                                    const float *bias, int silu, ss_bf16 *out, int64_t batch,
                                    int64_t d_inner, int64_t k, cudaStream_t stream);

ss_status ss_conv_state_update_f32(float *conv_state, const float *x, const float *w,
                                   const float *bias, int silu, float *out, int64_t batch,
                                   int64_t d_inner, int64_t k, cudaStream_t stream);

/*
 * ss_scan_bwd_bf16 / ss_scan_bwd_f32 -- gradient of ss_scan_fwd_* (training).
 *
 * Defines: the backward pass of section "Why the scan must be fused"
 * ("Mamba and selective state spaces"): the states are not stored by the
 * forward pass; this call reloads the forward inputs and recomputes them, and
 * runs the adjoint of the recurrence (itself a linear recurrence) in reverse.
 * With g(z) = z sigmoid(z), s = sigmoid(z), per channel d and state n:
 *   gy_t   = dout_t g(z_t)                  (dout_t when z == NULL)
 *   lam_t  = exp(delta_{t+1} A) lam_{t+1} + C_t gy_t,  lam_{L-1} = dfinal + C_{L-1} gy_{L-1}
 *   dx_t   = D gy_t + delta_t sum_n lam_t B_t
 *   ddelta = (sum_n lam_t (A a_t h_{t-1} + B_t x_t)) * (sigmoid(delta_t + dt_bias) with softplus)
 *   dA    += sum_t lam_t delta_t a_t h_{t-1}     dB_t += lam_t delta_t x_t
 *   dC_t  += gy_t h_t                            dD   += sum_t gy_t x_t
 *   dz_t   = dout_t y_t s (1 + z (1 - s)),  y_t the output before the gate
 *   ddt_bias = sum_t ddelta_t,  dh0 = exp(delta_0 A) lam_0
 * (a_t = exp(delta_t A); delta_t here is the step after bias and softplus.)
 *
 *   Inputs x .. delta_softplus : exactly as given to ss_scan_fwd_*.
 *   h0          : (batch, d_inner, N) fp32 initial state, or NULL for zero.
 *   dout        : (batch, d_inner, L) io dtype, gradient of y.
 *   dfinal_state: (batch, d_inner, N) fp32 gradient of final_state, or NULL.
 *   dx, ddelta  : (batch, d_inner, L) io dtype outputs; ddelta is the
 *                 gradient of the raw `delta` input (and of delta + dt_bias).
 *   dz          : (batch, d_inner, L) io dtype, or NULL (ignored if z NULL).
 *   dA          : (d_inner, N) fp32.   dB, dC : (batch, N, L) fp32.
 *   dD, ddt_bias: (d_inner) fp32, or NULL to skip (dD ignored if D NULL).
 *   dh0         : (batch, d_inner, N) fp32, or NULL to skip.
 *   workspace   : device scratch of at least ss_scan_bwd_workspace_bytes(...)
 *                 bytes, 16-byte aligned, owned by the caller; it holds the
 *                 state at every 16th step between the forward and reverse
 *                 walks and may be reused after the call's work completes.
 *   states_from_forward : non-zero when ss_scan_fwd_train_* has already
 *                 filled the workspace from these inputs (the backward's own
 *                 forward walk is then skipped).
 *   1 <= N <= 32.
 * dA, dB, dC, dD and ddt_bias are cleared on `stream` and accumulated with
 * fp32 atomic adds, so their last bits may differ between runs.
 * Errors: as ss_scan_fwd_* (SS_ERR_N for N > 32; SS_ERR_DIM also for a
 * workspace that is too small or misaligned).
 */
size_t ss_scan_bwd_workspace_bytes(int64_t batch, int64_t d_inner, int64_t L, int64_t N);

ss_status ss_scan_bwd_bf16(const ss_bf16 *x, const ss_bf16 *delta, const float *A, const ss_bf16 *B,
                           const ss_bf16 *C, const float *D, const ss_bf16 *z, const float *dt_bias,
                           int delta_softplus, const float *h0, const ss_bf16 *dout,
                           const float *dfinal_state, ss_bf16 *dx, ss_bf16 *ddelta, float *dA, float *dB,
                           float *dC, float *dD, ss_bf16 *dz, float *ddt_bias, float *dh0,
                           void *workspace, size_t workspace_bytes, int states_from_forward,
                           int64_t batch, int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream);

ss_status ss_scan_bwd_f32(const float *x, const float *delta, const float *A, const float *B,
                          const float *C, const float *D, const float *z, const float *dt_bias,
                          int delta_softplus, const float *h0, const float *dout,
                          const float *dfinal_state, float *dx, float *ddelta, float *dA, float *dB,
                          float *dC, float *dD, float *dz, float *ddt_bias, float *dh0, void *workspace,
                          size_t workspace_bytes, int states_from_forward, int64_t batch,
                          int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream);

/*
 * ss_scan_bwd_ex_bf16 / ss_scan_bwd_ex_f32 -- gradient of ss_scan_fwd_ex_*:
 * the backward pass above for the scan with sequence starts and/or the
 * reverse direction ("What each parameter does": the state forgets everything
 * at a document break; one direction of a bidirectional layer).
 *   seq_start : (batch, L) bytes, non-zero at the first step of each packed
 *               sequence, or NULL. As in the forward, nothing crosses the
 *               boundary before a marked step: no state into it and no
 *               gradient back across it.
 *   reverse   : non-zero for the reverse-direction scan
 *               h_t = exp(delta_t A) h_{t+1} + delta_t B_t x_t.
 * Every other argument as ss_scan_bwd_* (the workspace holds the backward's
 * own stored states; there is no states_from_forward). dh0 is the gradient of
 * the state that enters the walk (at t = 0, or t = L-1 when reversed).
 * Errors: as ss_scan_bwd_*.
 */
ss_status ss_scan_bwd_ex_bf16(const ss_bf16 *x, const ss_bf16 *delta, const float *A, const ss_bf16 *B,
                              const ss_bf16 *C, const float *D, const ss_bf16 *z, const float *dt_bias,
                              int delta_softplus, const float *h0, const uint8_t *seq_start, int reverse,
                              const ss_bf16 *dout, const float *dfinal_state, ss_bf16 *dx, ss_bf16 *ddelta,
                              float *dA, float *dB, float *dC, float *dD, ss_bf16 *dz, float *ddt_bias,
                              float *dh0, void *workspace, size_t workspace_bytes, int64_t batch,
                              int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream);

ss_status ss_scan_bwd_ex_f32(const float *x, const float *delta, const float *A, const float *B,
                             const float *C, const float *D, const float *z, const float *dt_bias,
                             int delta_softplus, const float *h0, const uint8_t *seq_start, int reverse,
                             const float *dout, const float *dfinal_state, float *dx, float *ddelta,
                             float *dA, float *dB, float *dC, float *dD, float *dz, float *ddt_bias,
                             float *dh0, void *workspace, size_t workspace_bytes, int64_t batch,
                             int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream);

/*
 * ss_scan_fwd_train_bf16 / ss_scan_fwd_train_f32 -- ss_scan_fwd_* for training:
 * the same outputs (with an optional initial state h0, as ss_scan_fwd_ex_*),
 * and in `workspace` (at least ss_scan_bwd_workspace_bytes(...) bytes, 16-byte
 * aligned, caller-owned) the state at every 16th step, which the backward pass
 * would otherwise recompute with a forward walk of its own. Pass the same
 * workspace, untouched, and the same inputs to ss_scan_bwd_* with
 * states_from_forward = 1. 1 <= N <= 32.
 */
ss_status ss_scan_fwd_train_bf16(const ss_bf16 *x, const ss_bf16 *delta, const float *A,
                                 const ss_bf16 *B, const ss_bf16 *C, const float *D,
                                 const ss_bf16 *z, const float *dt_bias, int delta_softplus,
                                 const float *h0, ss_bf16 *y, float *final_state, void *workspace,
                                 size_t workspace_bytes, int64_t batch, int64_t d_inner, int64_t L,
                                 int64_t N, cudaStream_t stream);

ss_status ss_scan_fwd_train_f32(const float *x, const float *delta, const float *A, const float *B,
                                const float *C, const float *D, const float *z, const float *dt_bias,
                                int delta_softplus, const float *h0, float *y, float *final_state,
                                void *workspace, size_t workspace_bytes, int64_t batch,
                                int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream);

/*
 * ss_scan_bwd_noalloc_bf16 / ss_scan_bwd_noalloc_f32 -- ss_scan_bwd_* without
 * a caller workspace, for callers that cannot call cudaMalloc (code that runs
 * under a framework which owns all device memory through its own pool, or a
 * library that may not allocate on its caller's behalf). The stored states live
 * in a device array built into the library (SS_BWD_NOALLOC_MAX_BYTES bytes),
 * so the call needs no memory beyond its inputs and outputs and allocates
 * nothing. The pages have no counterpart: this is a packaging of the backward
 * pass. Arguments and results are those of ss_scan_bwd_* minus workspace /
 * workspace_bytes.
 *
 * Limits: a problem whose ss_scan_bwd_workspace_bytes(...) exceeds
 * SS_BWD_NOALLOC_MAX_BYTES is rejected with SS_ERR_DIM (use ss_scan_bwd_*);
 * sizes are validated before any size product is formed. Every CUDA context
 * that loads the library holds one copy of the array (SS_BWD_NOALLOC_MAX_BYTES
 * of device memory, until the context is destroyed), whether or not it calls
 * this entry point. The copy is shared by every call in that context: calls
 * whose work overlaps on the GPU (unordered streams, several host threads)
 * race on it and must be ordered by the caller. Nothing in the array needs
 * clearing between calls. The first call in a context resolves the array's
 * address (which can load the module) and should come before any stream
 * capture; the address is cached with the context's unique id, so a call after
 * cudaDeviceReset (or in another context) resolves it again.
 */
#define SS_BWD_NOALLOC_MAX_BYTES (64u << 20)

ss_status ss_scan_bwd_noalloc_bf16(const ss_bf16 *x, const ss_bf16 *delta, const float *A,
                                   const ss_bf16 *B, const ss_bf16 *C, const float *D,
                                   const ss_bf16 *z, const float *dt_bias, int delta_softplus,
                                   const float *h0, const ss_bf16 *dout, const float *dfinal_state,
                                   ss_bf16 *dx, ss_bf16 *ddelta, float *dA, float *dB, float *dC,
                                   float *dD, ss_bf16 *dz, float *ddt_bias, float *dh0,
                                   int64_t batch, int64_t d_inner, int64_t L, int64_t N,
                                   cudaStream_t stream);

ss_status ss_scan_bwd_noalloc_f32(const float *x, const float *delta, const float *A,
                                  const float *B, const float *C, const float *D, const float *z,
                                  const float *dt_bias, int delta_softplus, const float *h0,
                                  const float *dout, const float *dfinal_state, float *dx,
                                  float *ddelta, float *dA, float *dB, float *dC, float *dD,
                                  float *dz, float *ddt_bias, float *dh0, int64_t batch,
                                  int64_t d_inner, int64_t L, int64_t N, cudaStream_t stream);

/*
 * ss_ssd_fwd_bf16 -- Mamba-2's scalar-decay scan (SSD): one decay per head of
 * P channels, B and C shared by the heads of a group ("Mamba and selective
 * state spaces": Mamba-2 gives each head a single scalar decay, which turns
 * most of the work into matrix products and allows N = 64 to 256; "Mamba in
 * practice": h_t = alpha_t h_{t-1} + Bbar_t x_t, Y = M o (C B^T) X with a
 * 1-semiseparable mask M). Per batch b, head h, group g = h / (nheads / ngroups):
 *
 *   delta_t = softplus(dt[b,t,h] + dt_bias[h])   (or dt + dt_bias)
 *   S_t[p][n] = exp(delta_t A[h]) S_{t-1}[p][n] + delta_t x[b,t,h,p] B[b,t,g,n]
 *   y[b,t,h,p] = (sum_n C[b,t,g,n] S_t[p][n] + D[h] x[b,t,h,p]) * silu(z[b,t,h,p])
 *
 * computed chunk by chunk (64 steps) with the products on the tensor cores
 * (bf16 operands, fp32 accumulation; the decays, masks and the carried state
 * are fp32).
 *
 *   x, z, y     : (batch, L, nheads, headdim) bf16, time-major; z may be NULL.
 *   dt          : (batch, L, nheads) bf16 raw step.
 *   A, D, dt_bias : (nheads) fp32 (A the negative decay rate); D, dt_bias may be NULL.
 *   B, C        : (batch, L, ngroups, N) bf16.
 *   h0          : (batch, nheads, headdim, N) fp32 initial state, or NULL.
 *   final_state : (batch, nheads, headdim, N) fp32 output, or NULL.
 *   workspace   : >= ss_ssd_workspace_bytes(batch, L, nheads, ngroups, N) bytes
 *                 of device scratch, caller-owned: C_c B_c^T of every chunk, the
 *                 counters of the chunk walk's work items, and the states handed
 *                 from one chunk segment of a (batch, head) row to the next (the
 *                 walk may cut each row into 2 or 4 segments, run in order, so that
 *                 rows x segments spread evenly over the resident CTAs). Calls that
 *                 share a workspace must not overlap on the GPU.
 *   headdim = 64, N = 64, 128 or 256, nheads a multiple of ngroups; x, B, C,
 *   y, z and the workspace 16-byte aligned. N = 256 runs as two passes over the
 *   128-state halves (the first stores its partial y, rounded to bf16, in y;
 *   the second adds it and applies the gate), on the tensor-core kernels only.
 * Errors: SS_ERR_NULL, SS_ERR_DIM (sizes, alignment, workspace), SS_ERR_N,
 * SS_ERR_DEVICE_PTR, SS_ERR_LAUNCH, SS_ERR_INTERNAL.
 */
size_t ss_ssd_workspace_bytes(int64_t batch, int64_t L, int64_t nheads, int64_t ngroups, int64_t N);

ss_status ss_ssd_fwd_bf16(const ss_bf16 *x, const ss_bf16 *dt, const float *A, const ss_bf16 *B,
                          const ss_bf16 *C, const float *D, const ss_bf16 *z, const float *dt_bias,
                          int delta_softplus, const float *h0, ss_bf16 *y, float *final_state,
                          void *workspace, size_t workspace_bytes, int64_t batch, int64_t L,
                          int64_t nheads, int64_t headdim, int64_t ngroups, int64_t N,
                          cudaStream_t stream);

/* Device-side faults recorded by the kernels since the last clear, as a bit
 * set: SS_FAULT_WAIT_TIMEOUT = a bounded wait in a kernel (for a tensor copy
 * into shared memory -- the tiles of "Why the scan must be fused": inputs are
 * staged once on chip -- or for the hand-over of a buffer between the warps
 * of a CTA) ran out of its one-second limit; the thread then stops waiting,
 * the call's outputs are not valid, and the copies already issued are let
 * land before the kernel exits. Synchronises the device (reads a device word).
 *   flags  host pointer, receives the bit set
 *   clear  non-zero: reset the recorded faults to none
 * Errors: SS_ERR_NULL (flags NULL), SS_ERR_INTERNAL (the read failed). */
#define SS_FAULT_WAIT_TIMEOUT 1u
/* SS_FAULT_SMEM_ALIGN: a kernel that stages its tiles by tensor copies into
 * dynamic shared memory without aligning the base itself (the forward scan,
 * the backward pass, the decode update and the SSD chunk kernel that runs
 * without the tensor cores' operand layouts) found that
 * memory off the boundary the copies need and returned without writing its
 * outputs. */
#define SS_FAULT_SMEM_ALIGN 2u
ss_status ss_device_faults(unsigned int *flags, int clear);

/* Exercises the fault word: one GPU thread waits on a barrier that nothing
 * completes, with the same one-second bound every kernel's waits have; the
 * wait gives up, records SS_FAULT_WAIT_TIMEOUT and the kernel returns, so the
 * context stays usable. No counterpart in the pages: a check of the bounded
 * waits themselves, for tests. Asynchronous on `stream` (about one second of
 * GPU time); read the result with ss_device_faults after synchronising.
 * Errors: SS_ERR_LAUNCH. */
ss_status ss_fault_probe(cudaStream_t stream);

/* The architecture the library's kernels were compiled for, as the CUDA
 * runtime reports it for the loaded module on the current device
 * (cudaFuncGetAttributes(...).binaryVersion of the forward scan kernel:
 * major * 10 + minor, 103 for sm_103a). A build check with no counterpart in
 * the pages; it needs a GPU (it loads the module in the current context).
 *   binary_version  host pointer, receives the value
 * Errors: SS_ERR_NULL (binary_version NULL), SS_ERR_INTERNAL (the query
 * failed, e.g. no GPU or no image for this GPU in the library). */
ss_status ss_kernel_binary_version(int *binary_version);

/* Message describing the last non-OK status returned on this host thread
 * ("" if none). The string is owned by the library. */
const char *ss_last_error(void);

/* SS_ABI_VERSION of the loaded library. */
int ss_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SS_SCAN_H */
