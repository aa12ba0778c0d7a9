/*
 * m2rnn.h -- C ABI of libm2rnn.so, the GB300 (sm_103a) M2RNN recurrence.
 *
 * The operation (paper "M2RNN: Non-Linear RNNs with Matrix-Valued States for
 * Scalable Language Modeling", arXiv 2603.14360v2; discussion deck frame
 * "Write, transform, retain, and read a matrix state", Eqs. (10)-(12)), per
 * batch item b and value head n, for t = 1..T:
 *
 *     Z_t = tanh(H_{t-1} W + k_t v_t^T)          H_t, Z_t in R^{K x V}
 *     H_t = f_t H_{t-1} + (1 - f_t) Z_t          W in R^{V x V}
 *     y_t = H_t^T q_t + w_r (.) v_t              q_t, k_t in R^K; v_t, w_r in R^V
 *
 * with H_0 = 0 unless an initial state is passed.  q and k are shared by the
 * N value heads (frame "Shared queries and keys buy more recurrent
 * capacity": N_q = N_k = 1, N_v = N_f = N_w = N), or by groups of them:
 * with Nq = N_q = N_k > 1 query/key groups (frame "Tensor parallelism
 * trades topology dependence for sync", one group per block of heads),
 * value head n reads group n / (N / Nq).  The backward pass is the
 * chain rule of the backup frame "the recurrent gradient needs both paths"
 * (R_t = C_t + q_t u_t^T, D_t = ((1-f_t) R_t) (.) (1 - Z_t (.) Z_t),
 * C_{t-1} = f_t R_t + D_t W^T, df_t = <R_t, H_{t-1} - Z_t>, dW = sum H_{t-1}^T D_t)
 * plus the value-residual and q/k/v terms that follow from Eqs. (10)-(12).
 *
 * Layouts (all row-major and contiguous; element type in brackets):
 *   q, k          [B,T,Nq,K]  (in_dtype); [B,T,K] when Nq = 1
 *   v             [B,T,N,V]   (in_dtype)
 *   f             [B,T,N]     (in_dtype), values in [0,1]
 *   W             [N,V,V]     (in_dtype); (H W)_{ij} = sum_l H_{il} W[n][l][j]
 *   w_r           [N,V]       (in_dtype)
 *   H0, H_T       [B,N,K,V]   (float32)
 *   y, dy         [B,T,N,V]   (in_dtype)
 *   ckpt          [B,N,nck,K,V] (float32), nck = ceil(T / ckpt_every);
 *                 ckpt[b][n][c] is the state after c*ckpt_every steps
 *                 (ckpt[b][n][0] = H0, or 0)
 *   dq, dk        [B,T,Nq,K]  (float32), summed over the heads of each group
 *   dv            [B,T,N,V]   (float32)
 *   df            [B,T,N]     (float32)
 *   dW            [N,V,V]     (float32), summed over b and t
 *   dw_r          [N,V]       (float32), summed over b and t
 *   dH_T, dH0     [B,N,K,V]   (float32)
 *
 * Supported shapes: K in {16, 32, 64, 128}, V in {16, 32}, B, N >= 1,
 * T >= 0, Nq >= 1 dividing N, B*T*N*V < 2^40.  T = 0 launches no recurrence and writes
 * H_T = H0 (or 0).
 *
 * Ownership and execution: every tensor pointer is device memory (cudaMalloc
 * or managed) owned by the caller, on the current device, 16-byte aligned.
 * The library keeps no pointer after a call returns and allocates no device
 * memory per call; scratch for the backward pass is a caller-provided
 * workspace whose size m2rnn_bwd_workspace_size() reports.  Work is enqueued
 * asynchronously on `stream` (a cudaStream_t; NULL = legacy default stream);
 * the caller synchronises.  Outputs are overwritten, never accumulated into.
 *
 * Errors: every entry point returns an m2rnn_status.  Argument errors are
 * detected on the host before anything is launched.  A kernel whose internal
 * wait exceeds its time limit stops early, leaves its outputs unspecified and
 * records M2RNN_ERR_TIMEOUT in a device status word that
 * m2rnn_device_status() reads.  Nothing crosses the ABI as an exception.
 */
#ifndef M2RNN_H_
#define M2RNN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    M2RNN_OK = 0,
    M2RNN_ERR_INVALID_ARG = -1,       /* null required pointer, negative size, bad dtype */
    M2RNN_ERR_UNSUPPORTED_SHAPE = -2, /* K, V or sizes outside the supported set */
    M2RNN_ERR_MISALIGNED = -3,        /* a tensor pointer is not 16-byte aligned */
    M2RNN_ERR_POINTER = -4,           /* a pointer is not device memory of the current device */
    M2RNN_ERR_WORKSPACE = -5,         /* workspace missing or smaller than required */
    M2RNN_ERR_CUDA = -6,              /* a CUDA runtime call or launch failed */
    M2RNN_ERR_TIMEOUT = -7,           /* a kernel wait exceeded its limit (device status) */
    M2RNN_ERR_BOUNDS = -8             /* checked build only: a kernel computed an index outside
                                         its array and skipped the access (device status) */
} m2rnn_status;

typedef enum {
    M2RNN_F32 = 0,  /* q, k, v, f, W, w_r, y, dy are float32 */
    M2RNN_BF16 = 1  /* q, k, v, f, W, w_r, y, dy are bfloat16 */
} m2rnn_dtype;

typedef struct {
    int B, T, N, K, V;
    int in_dtype;    /* m2rnn_dtype */
    int ckpt_every;  /* checkpoint interval C in steps; 0 = no checkpoints */
    int Nq;          /* query/key groups N_q = N_k; 0 is read as 1 (shared by
                        all heads); must divide N.  Zero-initialise the struct. */
} m2rnn_shape;

/* Library version (major*10000 + minor*100 + patch). */
int m2rnn_version(void);  /* 200 and later: m2rnn_shape carries Nq; 201: M2RNN_ERR_BOUNDS */

/* 1 for the checked build (libm2rnn_check.so), 0 for the normal one.  The
 * checked build compiles the same kernels with an index check in front of
 * every global-memory access whose index a kernel computes: an index outside
 * the extent that the call's shape gives its array records M2RNN_ERR_BOUNDS
 * and the location code of the access in the device status word, and the
 * access is skipped (no trap).  The normal build has no such checks. */
int m2rnn_checked(void);

/* Human-readable text for a status code; never NULL. */
const char *m2rnn_status_string(int status);

/* Number of checkpoints per (b, n) for `s`: ceil(T / ckpt_every), 0 when
 * ckpt_every == 0 or T == 0. */
size_t m2rnn_num_checkpoints(const m2rnn_shape *s);

/* Forward pass, Eqs. (10)-(12).
 *   q, k, v, f, W, w_r : inputs (required), layouts above.
 *   H0   : initial state, or NULL for H_0 = 0.
 *   y    : output (required).
 *   H_T  : final state output, or NULL.
 *   ckpt : checkpoint output, or NULL; written only when s->ckpt_every > 0. */
int m2rnn_fwd(const m2rnn_shape *s, const void *q, const void *k, const void *v,
              const void *f, const void *W, const void *w_r, const float *H0,
              void *y, float *H_T, float *ckpt, void *stream);

/* Bytes of workspace m2rnn_bwd needs for shape `s`; ckpt_given = 1 when the
 * caller will pass checkpoints from the forward pass, 0 when the backward
 * must recompute them into the workspace. */
size_t m2rnn_bwd_workspace_size(const m2rnn_shape *s, int ckpt_given);

/* Backward pass (BPTT) for the loss L with dL/dy = dy and dL/dH_T = dH_T.
 *   q, k, v, f, W, w_r, H0 : the forward inputs (H0 may be NULL = 0).
 *   ckpt : checkpoints written by m2rnn_fwd with the same s->ckpt_every,
 *          or NULL to have them recomputed into the workspace.
 *          s->ckpt_every must be > 0 (it is the recomputation interval).
 *   dy   : upstream gradient of y (required); dH_T may be NULL (= 0).
 *   dq, dk, dv, df, dW, dw_r : gradient outputs (required, float32).
 *   dH0  : gradient of H0, or NULL.
 *   dckpt: gradient of every checkpoint state, dL/dH_{c*ckpt_every}, laid
 *          out like ckpt ([B,N,nck,K,V] float32; dckpt[..][0] = dH0), or
 *          NULL.  It lets a caller split a sequence at checkpoints.
 *   workspace, ws_bytes : at least m2rnn_bwd_workspace_size(s, ckpt != NULL)
 *          bytes of device memory; its contents on entry are ignored. */
int m2rnn_bwd(const m2rnn_shape *s, const void *q, const void *k, const void *v,
              const void *f, const void *W, const void *w_r, const float *H0,
              const float *ckpt, const void *dy, const float *dH_T,
              float *dq, float *dk, float *dv, float *df, float *dW, float *dw_r,
              float *dH0, float *dckpt, void *workspace, size_t ws_bytes, void *stream);

/* Forward pass with the fused input gate of the frame "The gate preserves a
 * direct path through time" (Eq. 13):
 *     f_{t,n} = exp(-alpha_n softplus(a_{t,n} + beta_n)),   alpha_n >= 0,
 * evaluated in fp32 inside the kernel instead of reading f.
 *   a     : [B,T,N] (in_dtype), the gate's pre-activation (required)
 *   alpha : [N] (in_dtype), beta : [N] (in_dtype) (required)
 * Everything else is as for m2rnn_fwd.  alpha < 0 is not rejected (the
 * formula is evaluated as given); f then exceeds 1. */
int m2rnn_fwd_gated(const m2rnn_shape *s, const void *q, const void *k, const void *v,
                    const void *a, const void *alpha, const void *beta, const void *W,
                    const void *w_r, const float *H0, void *y, float *H_T, float *ckpt,
                    void *stream);

/* Backward pass through the fused input gate: as m2rnn_bwd, with f computed
 * from (a, alpha, beta) as in m2rnn_fwd_gated, and the chain rule
 *     df/da = df/dbeta = -alpha f sigmoid(a + beta),  df/dalpha = -softplus(a + beta) f
 * applied inside the kernel:
 *   da     : [B,T,N] float32, dL/da (in place of df)
 *   dalpha : [N] float32, dL/dalpha summed over b and t (overwritten)
 *   dbeta  : [N] float32, dL/dbeta summed over b and t (overwritten)
 * ckpt (if given) must come from m2rnn_fwd_gated with the same inputs.
 * The workspace rule is that of m2rnn_bwd (m2rnn_bwd_workspace_size). */
int m2rnn_bwd_gated(const m2rnn_shape *s, const void *q, const void *k, const void *v,
                    const void *a, const void *alpha, const void *beta, const void *W,
                    const void *w_r, const float *H0, const float *ckpt, const void *dy,
                    const float *dH_T, float *dq, float *dk, float *dv, float *da,
                    float *dalpha, float *dbeta, float *dW, float *dw_r, float *dH0,
                    float *dckpt, void *workspace, size_t ws_bytes, void *stream);

/* Forward pass with the readout epilogue of the frame "Most of the block can
 * be computed before recurrence" (after readout: multiply by the output gate
 * g_t, apply RMSNorm) in the form of the backup frame "RMSNormTP synchronizes
 * per-token statistics", over a token's d = N*V features:
 *     o = y (.) g,   rstd = (sum_d o^2 / d + eps)^(-1/2),   out = w_norm (.) o rstd.
 * The forward kernel's epilogue adds each CTA's share of sum_d o^2 per token
 * as it stores y; a second kernel scales.
 *   f, or the gate (a, alpha, beta): exactly one of the two forms (the other
 *        pointers NULL), as for m2rnn_fwd / m2rnn_fwd_gated.
 *   g      : [B,T,N,V] (in_dtype), the output gate (required)
 *   w_norm : [N,V] (in_dtype), the norm's weight (required)
 *   eps    : >= 0 (the pages omit it: 0 is their form; then a token whose
 *            o is all zero gets rstd = inf)
 *   y      : [B,T,N,V] (in_dtype), the readout of Eq. (12) (required: the
 *            backward pass needs it)
 *   out    : [B,T,N,V] (in_dtype), the normalised output (required)
 *   rstd   : [B,T] float32, rstd per token (required; the backward needs it)
 *   H_T, ckpt : as for m2rnn_fwd. */
int m2rnn_fwd_norm(const m2rnn_shape *s, const void *q, const void *k, const void *v,
                   const void *f, const void *a, const void *alpha, const void *beta,
                   const void *W, const void *w_r, const float *H0, const void *g,
                   const void *w_norm, float eps, void *y, void *out, float *rstd, float *H_T,
                   float *ckpt, void *stream);

/* Bytes of workspace m2rnn_bwd_norm needs: dL/dy ([B,T,N,V] in_dtype, 256-byte
 * aligned) plus m2rnn_bwd_workspace_size(s, ckpt_given). */
size_t m2rnn_bwd_norm_workspace_size(const m2rnn_shape *s, int ckpt_given);

/* Backward pass through the readout epilogue and the recurrence, for
 * dL/dout = dout ([B,T,N,V] in_dtype) and dL/dH_T = dH_T:
 *     p = w_norm (.) dout,  r = sum_d p o,  do = rstd p - r rstd^3 o / d,
 *     dL/dy = do (.) g,  dg = do (.) y,  dw_norm = sum over (b, t) of dout (.) o rstd,
 * then the recurrence's backward pass with that dL/dy (rounded to in_dtype,
 * the dtype m2rnn_bwd takes dy in).
 *   y, rstd : from m2rnn_fwd_norm with the same inputs.
 *   f or (a, alpha, beta) : as for m2rnn_fwd_norm; df receives dL/df, or
 *            dL/da with dalpha, dbeta ([N] float32, required then, NULL
 *            otherwise) as for m2rnn_bwd_gated.
 *   dg      : [B,T,N,V] float32 (required);  dw_norm : [N,V] float32 (required)
 *   everything else as for m2rnn_bwd; workspace: at least
 *   m2rnn_bwd_norm_workspace_size(s, ckpt != NULL) bytes. */
int m2rnn_bwd_norm(const m2rnn_shape *s, const void *q, const void *k, const void *v,
                   const void *f, const void *a, const void *alpha, const void *beta,
                   const void *W, const void *w_r, const float *H0, const float *ckpt,
                   const void *g, const void *w_norm, const void *y, const float *rstd,
                   const void *dout, const float *dH_T, float *dq, float *dk, float *dv,
                   float *df, float *dalpha, float *dbeta, float *dW, float *dw_r, float *dg,
                   float *dw_norm, float *dH0, float *dckpt, void *workspace, size_t ws_bytes,
                   void *stream);

/* Reads (after synchronising `stream`) and optionally clears the device
 * status word of the current device.  *status receives M2RNN_OK or the
 * first code a kernel recorded (M2RNN_ERR_TIMEOUT, or in the checked build
 * M2RNN_ERR_BOUNDS); *detail receives the location code of the wait that
 * gave up or of the access that was skipped (may be NULL).  Returns
 * M2RNN_OK or M2RNN_ERR_CUDA. */
int m2rnn_device_status(int *status, int *detail, int clear, void *stream);

/* Sets the time limit, in nanoseconds, of every internal wait of kernels
 * launched afterwards from this process (default 2e9 = 2 s; values <= 0
 * restore the default).  Exposed so that the time-out path can be tested
 * with a wait that cannot complete in time.  Returns M2RNN_OK. */
int m2rnn_set_wait_limit_ns(long long limit_ns);

/* Size of the checkpoint buffer built into the library for
 * m2rnn_bwd_noalloc (bytes, per GPU). */
#define M2RNN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/* Backward pass for callers that cannot allocate device memory.
 *
 * The paper has no counterpart to this entry point; it exists for callers
 * that must not call cudaMalloc (or any allocating routine) at the point
 * where they run the backward pass -- for example code running while a
 * memory pool is frozen or exhausted, code inside a framework whose
 * allocator must not be re-entered, or a runtime that only hands out
 * pre-registered buffers.  It computes the same gradients as m2rnn_bwd
 * with ckpt = NULL and dckpt = NULL, but recomputes the checkpoints into a
 * buffer compiled into the library instead of a caller workspace, and
 * allocates nothing.  The caller still passes every input and output.
 *
 *   - The buffer holds M2RNN_NOALLOC_SCRATCH_BYTES (64 MiB); problems whose
 *     checkpoints need more (m2rnn_bwd_workspace_size(s, 0) bytes) are
 *     refused with M2RNN_ERR_WORKSPACE before any device work.
 *   - Every GPU that loads this part of the library holds the buffer until
 *     the process exits.
 *   - Shape and argument errors are refused on the host before any CUDA
 *     call.
 *   - The first call on a device looks up the buffer's device address on
 *     that device (which must be current); make that first call before any
 *     stream capture.  The address is kept for the life of the process; do
 *     not use the library on a device again after a cudaDeviceReset of it.
 *   - All calls share the buffer and it keeps the last call's contents;
 *     nothing in it needs to start at zero (the forward recomputation writes
 *     every checkpoint the backward reads).  Calls that overlap on the GPU
 *     (different streams, or threads sharing a device) race on it: the
 *     caller must serialise them. */
int m2rnn_bwd_noalloc(const m2rnn_shape *s, const void *q, const void *k, const void *v,
                      const void *f, const void *W, const void *w_r, const float *H0,
                      const void *dy, const float *dH_T, float *dq, float *dk, float *dv,
                      float *df, float *dW, float *dw_r, float *dH0, void *stream);

/* Single-step decode: the inference path, one new token for each of B
 * sequences with the state carried between calls.  One step of Eqs.
 * (10)-(12) per (b, n):
 *     H_out = f H_in + (1 - f) tanh(H_in W + k v^T),  y = H_out^T q + w_r (.) v.
 * The paper's pages give the recurrence, not a decoding kernel; this is the
 * forward pass at T = 1 with the state in and out, kept apart because it is
 * bound by the state's HBM traffic rather than by the serial chain.
 *   s->T must be 1; s->ckpt_every is ignored.
 *   q, k  : [B,Nq,K]   (in_dtype)      v : [B,N,V] (in_dtype)
 *   f     : [B,N]      (in_dtype)      W, w_r : as for m2rnn_fwd
 *   H_in  : [B,N,K,V]  (float32), the state before the step (required)
 *   H_out : [B,N,K,V]  (float32), the state after it (required); it may be
 *           H_in itself (in-place update), otherwise the two must not overlap
 *   y     : [B,N,V]    (in_dtype), output
 * The state update performs the forward kernel's operations in the same
 * order, so T calls reproduce m2rnn_fwd's H_T for the same inputs. */
int m2rnn_decode(const m2rnn_shape *s, const void *q, const void *k, const void *v,
                 const void *f, const void *W, const void *w_r, const float *H_in,
                 float *H_out, void *y, void *stream);

/* Single-step decode with the fused input gate of Eq. (13): as m2rnn_decode,
 * with f = exp(-alpha softplus(a + beta)) computed in the kernel from
 * a [B,N] (in_dtype) and alpha, beta [N] (in_dtype) instead of f.  T such
 * calls reproduce m2rnn_fwd_gated's H_T for the same inputs bit for bit. */
int m2rnn_decode_gated(const m2rnn_shape *s, const void *q, const void *k, const void *v,
                       const void *a, const void *alpha, const void *beta, const void *W,
                       const void *w_r, const float *H_in, float *H_out, void *y,
                       void *stream);

/* Test hook for the time-out path.  mode 1: kernels launched afterwards
 * from this process start no input transfers, so every internal wait runs
 * into the wait limit, the kernel stops early (outputs unspecified) and
 * M2RNN_ERR_TIMEOUT is recorded in the device status word.  mode 0 (the
 * default) turns it off.  Returns M2RNN_OK, or M2RNN_ERR_INVALID_ARG for an
 * unknown mode. */
int m2rnn_set_fault_injection(int mode);

#ifdef __cplusplus
}
#endif
#endif /* M2RNN_H_ */
