/*
 * ssm_scan.h -- C ABI of the B300 selective state-space scan library (libssm_b300.so).
 *
 * The library computes the Mamba-1 selective scan, per batch row b, channel d and state n:
 *
 *   v_t   = u_t, or SiLU(conv_b[d] + sum_k conv_w[d,k] x_{t-W+1+k}) with the fused causal conv
 *   dt_t  = softplus(delta_t + delta_bias[d])          (or delta_t + bias when softplus is off)
 *   Abar  = exp(dt_t A[d,n])
 *   Bbar  = (exp(dt_t A[d,n]) - 1) / A[d,n] * B_t[n]   zero-order hold (limit dt_t B_t[n] at A = 0)
 *         = dt_t B_t[n]                                 simplified form
 *   h_t[n] = Abar h_{t-1}[n] + Bbar v_t,  h_{-1} = h0 (or 0)
 *   y_t   = (sum_n C_t[n] h_t[n] + Dskip[d] v_t) * SiLU(z_t)
 *
 * Sources (page address, section; two of the pages carry an unrelated site title):
 *   zero-order hold and the recurrence: dpshk.com/news/3333417 sections 2.2, 2.3;
 *     lshu.cn/news/79586 section 2.2;
 *   diagonal (S4D) A, element-wise update: dpshk.com/news/3333417 section 3.2;
 *   selection dt = softplus(.), input-dependent B and C: dpshk.com/news/3333417 section 4.1;
 *     lshu.cn/news/79586 section 3.1 (B, C of shape (batch, seq_len, d_state));
 *   simplified Bbar = dt B and the D skip: dpshk.com/news/3333417 section 5.1 (SelectiveSSM);
 *   causal conv1d (padding W-1, cropped to L) + SiLU ahead of the SSM, gate y * SiLU(z):
 *     dpshk.com/news/3333417 section 5.2 (MambaBlock); lshu.cn/news/79586 section 3.3;
 *   carrying the final state of one segment into the next: pwwt.cn/news/5168881 section 3.1;
 *   single-token step from a constant-size state cache: datadaily.news "State space models vs
 *     Transformer: a practical guide", section on how state space models work; cache shape
 *     (batch, d_inner, d_state): lshu.cn/news/79586 section 6.5.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers into memory the caller owns.  Every tensor is
 *     dense row-major in the layout given below.  The library keeps no state between calls.
 *     It allocates no memory: a call that needs scratch space takes a caller-provided workspace.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default stream).
 *   - Errors: the return value is a status code.  Arguments are validated on the host before
 *     anything is launched: no kernel runs on an invalid call.  ssm_last_error() returns a
 *     thread-local message describing the most recent failure on the calling thread.  A launch
 *     error reported by the CUDA runtime is returned as SSM_ERR_CUDA.  Faults inside a kernel
 *     surface later, on the caller's next synchronisation, as with any CUDA launch.
 *   - Any sequence length L >= 1 is accepted.  Unaligned base pointers or row lengths whose byte
 *     size is not a multiple of 16 select a slower element-wise load path; they are not errors.
 *   - Supported state sizes: 1 <= dstate <= 16 for every dtype; 32 and 64 for bf16 inputs and
 *     output with 16-byte-aligned rows and seqlen % 8 == 0 (ssm_scan_fwd); any of 1..16, 32, 64
 *     for ssm_state_update.
 */
#ifndef SSM_SCAN_H
#define SSM_SCAN_H

#include <stddef.h>

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so the header needs no CUDA include. */
typedef struct CUstream_st *ssm_stream_t;

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = 1,   /* null required pointer, non-positive size, bad enum value     */
    SSM_ERR_UNSUPPORTED = 2,   /* well-formed request outside what the kernels implement       */
    SSM_ERR_CUDA = 3           /* the CUDA runtime reported an error at launch                 */
} ssm_status;

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

/*
 * Parameters of one selective scan.  Shapes: B = batch, D = dim (d_inner), N = dstate, L = seqlen.
 *
 *   u           (B, D, L) in_dtype   input v; the conv input x when conv_w != NULL      required
 *   delta       (B, D, L) in_dtype   raw step before bias/softplus                       required
 *   A           (D, N)    float32    diagonal state matrix (any finite value; 0 allowed)  required
 *   Bm, Cm      (B, N, L) in_dtype   input-dependent B and C, shared by all D channels    required
 *   Dskip       (D)       float32    skip weight, or NULL for none
 *   delta_bias  (D)       float32    added to delta before softplus, or NULL for none
 *   z           (B, D, L) in_dtype   gate input, or NULL for no gate
 *   conv_w      (D, conv_width) f32  causal depthwise conv taps, or NULL for no conv;
 *                                    tap conv_width-1 multiplies x_t
 *   conv_b      (D)       float32    conv bias, or NULL for zero (ignored without conv_w)
 *   conv_width  int                  1..4 when conv_w != NULL
 *   h0          (B, D, N) float32    initial state, or NULL for zeros; may alias h_out
 *   h_out       (B, D, N) float32    final state, or NULL if not wanted
 *   y           (B, D, L) out_dtype  output; must not overlap any input
 *   delta_softplus  1: dt = softplus(delta + bias); 0: dt = delta + bias
 *   zoh             1: zero-order-hold Bbar;        0: simplified Bbar = dt B
 *   workspace, workspace_bytes
 *                   optional device scratch that lets the scan split L across thread blocks when
 *                   B * D alone cannot fill the GPU.  NULL / too small is not an error: the call
 *                   then runs without the split.  Size it with ssm_scan_workspace_size().  The
 *                   workspace must not be shared by calls that may run concurrently.
 *   conv_init   (B, D, conv_width-1) in_dtype   the conv inputs x_{-W+1} .. x_{-1} (oldest first)
 *                   that precede this call's x, or NULL for zeros: the history a chunked prefill
 *                   carries from one call to the next.  Ignored without conv_w.
 *   conv_final  (B, D, conv_width-1) in_dtype   receives the last conv_width-1 inputs of the
 *                   sequence (reaching back into conv_init when seqlen < conv_width-1), ready to be
 *                   the next call's conv_init or the decode conv state; NULL if not wanted.  May be
 *                   the same buffer as conv_init; must not overlap any other tensor.  Ignored
 *                   without conv_w.
 *   state_indices (B) int32, or NULL.  Per-request state slots (pwwt.cn/news/5168881 section 3.4:
 *                   a state cache indexed by request): h0, h_out, conv_init and conv_final are then
 *                   caches with a leading slot dimension, (S, D, N) and (S, D, W-1), and batch row b
 *                   reads and writes slot state_indices[b].  A negative index marks a padding row:
 *                   nothing of any slot is read or written for it and its y is written as zeros.  The
 *                   caller guarantees indices < S and no index used twice.  Takes the element-wise
 *                   kernel: dstate <= 16, no L split.
 *   h_all       (B, L, D, N) float32, or NULL: receives the state after every step, the state
 *                   sequence a multi-token verification pass keeps so that the caller can commit the
 *                   state at the accepted length (pwwt.cn/news/5168881 section 3.4: speculative
 *                   decoding).  Takes the element-wise kernel (dstate <= 16); must not overlap any
 *                   other tensor; padding rows leave theirs untouched.
 *   h_ckpt      (B, ceil(L / SSM_CKPT_STEPS), D, N) float32, or NULL: receives one state every
 *                   SSM_CKPT_STEPS steps, entry c being the state after step min(8c + 7, L - 1): the
 *                   checkpoints from which ssm_scan_bwd recomputes the states it needs, instead of
 *                   keeping every state (the states saved for the backward pass of
 *                   dpshk.com/news/3333417 section 5.3, with the gradient checkpointing of
 *                   pwwt.cn/news/5168881 section 3.2).  Not together with h_all or state_indices;
 *                   dstate <= 16; must not overlap any other tensor.
 */
typedef struct ssm_scan_params {
    int batch, dim, dstate, seqlen;
    ssm_dtype in_dtype, out_dtype;
    const void *u;
    const void *delta;
    const float *A;
    const void *Bm;
    const void *Cm;
    const float *Dskip;
    const float *delta_bias;
    const void *z;
    const float *conv_w;
    const float *conv_b;
    int conv_width;
    const float *h0;
    float *h_out;
    void *y;
    int delta_softplus;
    int zoh;
    void *workspace;
    size_t workspace_bytes;
    const void *conv_init;
    void *conv_final;
    const int *state_indices;
    float *h_all;
    float *h_ckpt;
} ssm_scan_params;

/* Steps between the forward's state checkpoints (h_ckpt) that the backward pass recomputes from. */
#define SSM_CKPT_STEPS 8

/* Selective scan forward (with the optional fused conv front end, D skip and gate).
   Errors: SSM_ERR_INVALID_ARG (null p, null required pointer, size <= 0, bad dtype/flag value,
   conv_width outside 1..4), SSM_ERR_UNSUPPORTED (dstate not supported), SSM_ERR_CUDA. */
SSM_API ssm_status ssm_scan_fwd(const ssm_scan_params *p, ssm_stream_t stream);

/*
 * ssm_scan_fwd without any allocation.  (No counterpart on the pages: this is an interface for
 * callers of this library.)  Some callers cannot call cudaMalloc: a serving runtime that plans all
 * device memory at start-up and forbids allocation afterwards, code running in a stream callback or
 * host function (where CUDA calls are not allowed), or latency-critical paths where an allocation
 * may synchronise the device and stall other streams.  This entry point computes exactly what
 * ssm_scan_fwd computes with a large enough workspace, but takes the scratch for the L split from a
 * fixed 4 MiB buffer inside the library (p->workspace and p->workspace_bytes are ignored).  The
 * caller still provides every input and output.
 *   - The buffer lives in each device's memory from the first use until the process exits.
 *   - The first call on a device looks up the buffer's device address (once per device, with that
 *     device current); make that first call before any stream capture.  The address is looked up
 *     again when the device's current context is no longer the one it was taken in (for example after
 *     cudaDeviceReset); such a call, too, should come before any stream capture.
 *   - Every call shares the one buffer per device: calls whose kernels may overlap on the GPU
 *     (different streams, or several host threads) race on it and must be serialised by the caller.
 *   - A problem whose split needs more than 4 MiB of scratch is rejected with SSM_ERR_UNSUPPORTED
 *     and a message; nothing is launched.  Problems that need no split use no scratch at all.
 * Errors: as ssm_scan_fwd, plus SSM_ERR_UNSUPPORTED for a problem beyond the buffer and SSM_ERR_CUDA
 * if the device address cannot be obtained.
 */
SSM_API ssm_status ssm_scan_fwd_static(const ssm_scan_params *p, ssm_stream_t stream);

/* Bytes of workspace that let ssm_scan_fwd split L for this problem on the current device
   (0 when no split would be used).  Returns 0 for an invalid p. */
SSM_API size_t ssm_scan_workspace_size(const ssm_scan_params *p);

/*
 * Standalone causal depthwise conv1d (+ optional SiLU), the scan's front end on its own:
 *   y[b,d,t] = act(b[d] + sum_{k<width} w[d,k] x[b,d,t-width+1+k]),  x before t = 0 is zero.
 *   x, y (B, D, L) of `dtype`; w (D, width) float32; b (D) float32 or NULL.  width in 1..4.
 *   y must not overlap x.
 * Errors: SSM_ERR_INVALID_ARG, SSM_ERR_CUDA.
 */
SSM_API ssm_status causal_conv1d_fwd(const void *x, const float *w, const float *b, void *y, int batch, int dim,
                             int seqlen, int width, int silu, ssm_dtype dtype, ssm_stream_t stream);

/*
 * Single-token decode step from a constant-size state cache (the scan body with L = 1):
 *   state (B, D, N) float32, read and written in place
 *   u, delta, z, y (B, D) of `dtype` (z may be NULL); Bm, Cm (B, N) of `dtype`
 *   A (D, N) float32; Dskip, delta_bias (D) float32 or NULL
 *   y must not overlap any input.
 * Errors: SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED (dstate), SSM_ERR_CUDA.
 */
SSM_API ssm_status ssm_state_update(float *state, const void *u, const void *delta, const float *A, const void *Bm,
                            const void *Cm, const float *Dskip, const float *delta_bias, const void *z, void *y,
                            int batch, int dim, int dstate, int delta_softplus, int zoh, ssm_dtype dtype,
                            ssm_stream_t stream);

/*
 * Backward pass of the selective scan (training; pwwt.cn/news/5168881 section 3.2): the gradients of
 * sum(y * dy) + sum(h_L * dh_out) with respect to every input of the forward call.
 *
 * Forward inputs (batch, dim, dstate, seqlen, in_dtype, u, delta, A, Bm, Cm, Dskip, delta_bias, z,
 * conv_w, conv_b, conv_width, conv_init, h0, delta_softplus, zoh) are exactly those of the forward
 * call, and
 *   h_ckpt   (B, ceil(L/8), D, N) float32  the forward's state checkpoints (ssm_scan_fwd with h_ckpt)  required;
 *            the pass reloads the checkpoint before each group of 8 steps and recomputes the group's
 *            states from it (with the inputs, dt, Abar and the zero-order-hold factor), so the forward
 *            never stores every state
 *   dy       (B, D, L) in_dtype    gradient of y                                                  required
 *   dh_out   (B, D, N) float32     gradient of the final state, or NULL for zero
 * Outputs (element-wise ones in in_dtype, the rest float32; each may be NULL only where its input was):
 *   du, ddelta (B, D, L)           required (du is the gradient of x when the conv is fused)
 *   dz (B, D, L)                   required with z
 *   dA (D, N); dB, dC (B, N, L)    required
 *   dDskip, ddelta_bias (D); dconv_w (D, W); dconv_b (D); dconv_init (B, D, W-1); dh0 (B, D, N)
 * dA, dB, dC, dDskip, ddelta_bias, dconv_w and dconv_b are sums over rows and steps: the call zeroes
 * them on `stream` and accumulates.  The outputs must not overlap each other or any input.
 *   workspace, workspace_bytes: optional device scratch that lets the pass split L across thread
 *       blocks (the adjoint recurrence is linear: per segment a short summary pass, then every segment
 *       starts from its exact incoming adjoint), sized by ssm_scan_bwd_workspace_size(); NULL or too
 *       small runs without the split.  Not to be shared by calls that may run concurrently.
 * dstate 1..16.  Errors: SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED, SSM_ERR_CUDA.
 */
typedef struct ssm_scan_bwd_params {
    int batch, dim, dstate, seqlen;
    ssm_dtype in_dtype;
    const void *u;
    const void *delta;
    const float *A;
    const void *Bm;
    const void *Cm;
    const float *Dskip;
    const float *delta_bias;
    const void *z;
    const float *conv_w;
    const float *conv_b;
    int conv_width;
    const void *conv_init;
    const float *h0;
    int delta_softplus;
    int zoh;
    const float *h_ckpt;
    const void *dy;
    const float *dh_out;
    void *du;
    void *ddelta;
    void *dz;
    float *dA;
    float *dB;
    float *dC;
    float *dDskip;
    float *ddelta_bias;
    float *dconv_w;
    float *dconv_b;
    void *dconv_init;
    float *dh0;
    void *workspace;
    size_t workspace_bytes;
} ssm_scan_bwd_params;

SSM_API ssm_status ssm_scan_bwd(const ssm_scan_bwd_params *p, ssm_stream_t stream);

/* Bytes of workspace that let ssm_scan_bwd split L for this problem on the current device (0 when no
   split would be used, or for an invalid p). */
SSM_API size_t ssm_scan_bwd_workspace_size(const ssm_scan_bwd_params *p);

/*
 * Device-side failures that a kernel could only record, not return.  (No counterpart on the pages.)
 * The streamed decode kernel and the packed scan kernel bound every wait for their own bulk copies to
 * about one second; on a timeout they set a bit in a per-device flag, let their copies still in flight
 * land (again bounded) and return, leaving the outputs of the affected tiles unwritten and the context
 * usable.  This call
 * synchronises the current device, stores the flags in *flags (0: nothing recorded; bit 0: a decode
 * wait timed out; bit 1: a scan block stopped waiting for its staged chunk, likewise bounded; bit 2: an
 * SSD block stopped waiting for its copies or its tensor-core products) and clears them.
 * Errors: SSM_ERR_INVALID_ARG (flags NULL), SSM_ERR_CUDA (the synchronisation or the read failed).
 */
SSM_API ssm_status ssm_device_error(unsigned *flags);

/*
 * Test hook, not for production use.  (No counterpart on the pages.)  With on != 0, later calls of the
 * packed scan's single-pass launch (block (0, 0)), the streamed decode kernel (block 0) and the SSD
 * kernel (every block) leave out their first staged copy, so that their bounded waits for it run out
 * after about a second and ssm_device_error reports bits 1, 0 and 2; the outputs of those blocks are
 * then not written.  on == 0 (the state at load) restores normal operation.  A process-wide flag read at
 * each launch; setting it while another thread launches is allowed (the launch sees the old or the new
 * value).  No errors.
 */
SSM_API void ssm_test_withhold_first_copy(int on);

/*
 * Single-token decode step with the conv front end fused: the decode cache holds a conv state and
 * the SSM state (dpshk.com/news/5205047 section 1.3; lshu.cn/news/79586 section 6.5).  Per (b, d):
 *   v   = SiLU(conv_b[d] + sum_{k<W-1} conv_w[d,k] conv_state[b,d,k] + conv_w[d,W-1] x[b,d])
 *   conv_state[b,d,:] <- (conv_state[b,d,1:], x[b,d])        (the last W-1 inputs, oldest first)
 * then the step of ssm_state_update with v as its input.  With conv_w == NULL this is exactly
 * ssm_state_update (x is u; conv_state is ignored).
 *
 *   x           (B, D)    dtype      conv input (u when conv_w is NULL)            required
 *   delta, z, y, Bm, Cm, A, Dskip, delta_bias, state: as in ssm_state_update
 *   conv_w      (D, conv_width) f32  taps, tap conv_width-1 multiplies x; or NULL
 *   conv_b      (D)       float32    conv bias or NULL (zero)
 *   conv_width  int                  1..4 when conv_w != NULL
 *   conv_state  (B, D, conv_width-1) dtype, read and written in place; required when
 *                                    conv_width > 1; must not overlap any other tensor
 *   state_indices (B) int32 or NULL: state and conv_state are then slot caches (S, D, N) and
 *                                    (S, D, W-1) and batch row b uses slot state_indices[b]; a
 *                                    negative index marks a padding row (no slot touched, y = 0).
 *                                    Indices < S, none used twice (pwwt.cn/news/5168881 section 3.4)
 * Errors: SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED (dstate), SSM_ERR_CUDA.
 */
typedef struct ssm_step_params {
    int batch, dim, dstate;
    ssm_dtype dtype;
    float *state;
    const void *x;
    const void *delta;
    const float *A;
    const void *Bm;
    const void *Cm;
    const float *Dskip;
    const float *delta_bias;
    const void *z;
    const float *conv_w;
    const float *conv_b;
    int conv_width;
    void *conv_state;
    void *y;
    int delta_softplus;
    int zoh;
    const int *state_indices;
} ssm_step_params;

SSM_API ssm_status ssm_state_update_conv(const ssm_step_params *p, ssm_stream_t stream);

/*
 * Mamba-2 (SSD) scan: the selective recurrence with ONE scalar A per head, run by every channel of the
 * head, with B and C shared by the heads of a group (dpshk.com/news/3333417 sections 6.1 and 6.2;
 * pwwt.cn/news/5168881 section 2.3).  Per batch row b, head h, channel p of the head and state n, with
 * g = h / (H / G) the head's group and d = h * P + p its channel:
 *
 *   dt_t     = softplus(dt[b,h,t] + dt_bias[h])          (or dt + dt_bias when delta_softplus = 0)
 *   h_t[p,n] = exp(dt_t A[h]) h_{t-1}[p,n] + w_t B[b,g,t,n] x[b,d,t]
 *   w_t      = dt_t                       (zoh = 0, the simplified input scale)
 *            = expm1(dt_t A[h]) / A[h]    (zoh = 1; dt_t at A[h] = 0)
 *   y[b,d,t] = (sum_n C[b,g,t,n] h_t[p,n] + Dskip[h] x[b,d,t]) * SiLU(z[b,d,t])
 *
 * The library evaluates it in its chunked matrix ("dual") form on the tensor cores: per chunk of 128
 * steps the decayed causal matrix (C B^T masked and scaled) times X, plus the carried state's
 * contribution, and the chunk's state increment, as bf16 products with fp32 accumulation.
 *
 *   x, z, y   (B, H*P, L) bf16    channel d = h*P + p, contiguous in L; z may be NULL (no gate)
 *   dt        (B, H, L)   bf16    raw step of each head                                   required
 *   A         (H)         float32 one scalar per head (any finite value)                  required
 *   Bm, Cm    (B, G, L, N) bf16   contiguous in N                                         required
 *   Dskip, dt_bias (H)    float32 or NULL
 *   h0, h_out (B, H, P, N) float32 initial state (NULL: zeros) and final state (NULL: not wanted);
 *                                 h0 may be the same buffer as h_out
 * Supported: headdim P = 64, dstate N = 64 or 128, ngroups dividing nheads, seqlen % 8 == 0 (the rows of x,
 * dt and y are moved by TMA bulk copies, whose rows are whole multiples of 16 bytes), x, dt, Bm, Cm
 * and y 16-byte aligned.  y must not overlap any input; h_out must not overlap y or any input but h0.
 * Errors: SSM_ERR_INVALID_ARG (null params or required pointer, size <= 0, bad flag, overlap),
 * SSM_ERR_UNSUPPORTED (shape or alignment outside the above), SSM_ERR_CUDA.  A wait for a copy or an
 * MMA that runs out (about one second) is recorded for ssm_device_error (bit 2).
 */
typedef struct ssd_scan_params {
    int batch, nheads, headdim, ngroups, dstate, seqlen;
    const void *x;
    const void *dt;
    const float *A;
    const void *Bm;
    const void *Cm;
    const float *Dskip;
    const float *dt_bias;
    const void *z;
    const float *h0;
    float *h_out;
    void *y;
    int delta_softplus;
    int zoh;
} ssd_scan_params;

SSM_API ssm_status ssd_scan_fwd(const ssd_scan_params *p, ssm_stream_t stream);

/* Thread-local description of the most recent failed call on this thread ("" if none). */
SSM_API const char *ssm_last_error(void);

/* Library version string. */
SSM_API const char *ssm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H */
