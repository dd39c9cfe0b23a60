/*
 * s5.h -- C ABI of libs5.so, the GB300 (sm_103a) S5 layer library.
 *
 * The S5 layer is one diagonal multi-input multi-output state-space model
 * applied to batched sequences.  Sources (page title, then section):
 *  - "S5: Simplified State Space Layers for Sequence Modeling" (abhik.ai review
 *    of paper v3), sections "Discretization controls both retention and input
 *    gain", "Associative scans preserve the recurrence", and "Paper equations
 *    beside executable Python" rows 1-4;
 *  - "SIMPLIFIED STATE SPACE LAYERS FOR SEQUENCE MODELING" (papercache.org
 *    summary), section 2.2, section 3.2 eq. 4-6, section 3.3, App. A, App. H;
 *  - "Simplified State Space Layers for Sequence Modeling" (wikillm.com
 *    2208.04933), "Method" and "Paper vs code".
 *
 * Conventions for every entry point:
 *  - All array pointers are DEVICE pointers, owned by the caller, 16-byte
 *    aligned and row-major.  The library allocates no memory in any call.
 *  - A complex array is stored as interleaved (re, im) float32 pairs; its
 *    documented shape counts complex elements.
 *  - P is the number of STORED complex modes: one member of each conjugate
 *    pair.  The readout therefore doubles the real part of C~x.
 *  - Work is queued on `stream` (NULL = legacy default stream) and the call
 *    returns without waiting.  The return value reports argument checks and
 *    launch errors.  Conditions only the GPU can see (a non-finite or
 *    negative interval, a carry wait that gave up) are latched in the
 *    workspace and reported by s5_sync_status().
 *  - Stream order is kept.  Some kernels (the weight images and scans of
 *    s5_forward and s5_forward_bidirectional on the tensor-core shapes, and
 *    s5_step) are launched with programmatic dependent launch: they may be
 *    scheduled while the kernel queued before them is still running, but
 *    each waits for that kernel to complete before it reads or writes any
 *    memory.
 *  - No CPU fallback exists: a shape the kernels do not cover returns
 *    S5_ERR_UNSUPPORTED.
 */
#ifndef S5_H
#define S5_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that callers need no CUDA header. */
typedef struct CUstream_st *s5_stream_t;

typedef enum {
    S5_OK = 0,
    S5_ERR_INVALID_ARGUMENT = 1, /* null/misaligned pointer, bad size or dtype, workspace too small */
    S5_ERR_UNSUPPORTED = 2,      /* valid arguments outside what the kernels cover */
    S5_ERR_CUDA = 3,             /* a CUDA runtime call or launch failed; see s5_last_cuda_error() */
    S5_ERR_TIMEOUT = 4,          /* a cross-tile carry wait gave up (output is not valid) */
    S5_ERR_NONFINITE = 5         /* a non-finite or negative interval reached the kernel */
} s5_status;

typedef enum { S5_F32 = 0, S5_BF16 = 1 } s5_dtype;

typedef enum { S5_ZOH = 0, S5_BILINEAR = 1 } s5_discretization;

/*
 * Zero-order-hold discretisation ("SIMPLIFIED STATE SPACE LAYERS ...",
 * section 3.2 eq. 6; review row 2):
 *   Delta_n      = exp(log_dt[n])
 *   lambda_bar_n = exp(lambda_n * Delta_n)
 *   b_bar[n,:]   = (lambda_bar_n - 1) / lambda_n * b_tilde[n,:]
 * with the removable singularity lambda_n*Delta_n -> 0 taken as the limit
 * Delta_n * b_tilde[n,:].  Computed on the device in float-float arithmetic
 * (pairs of floats, ~48 significant bits, from FP32 instructions) and rounded
 * once to float.  Launched with programmatic stream serialisation: it may
 * start while the kernel before it runs, reads only its inputs until that
 * kernel has completed, and writes lambda_bar and b_bar after.
 *   lambda     [P]    complex   in
 *   log_dt     [P]    float32   in
 *   b_tilde    [P,H]  complex   in
 *   lambda_bar [P]    complex   out
 *   b_bar      [P,H]  complex   out
 * Errors: S5_ERR_INVALID_ARGUMENT for null/misaligned pointers or P, H < 1.
 */
s5_status s5_discretize(const float *lambda, const float *log_dt, const float *b_tilde,
                        int P, int H, float *lambda_bar, float *b_bar, s5_stream_t stream);

/*
 * Discretisation with the options of the official implementation.
 *   method  S5_ZOH as s5_discretize, or S5_BILINEAR (review "Discretization
 *           controls both retention and input gain": the official code offers
 *           the bilinear transform beside ZOH; the S4 page, "Discretize",
 *           prints it): per mode
 *             lambda_bar_n = (1 + Delta_n lambda_n / 2) / (1 - Delta_n lambda_n / 2)
 *             b_bar[n,:]   = Delta_n / (1 - Delta_n lambda_n / 2) * b_tilde[n,:]
 *   clip_re clip_eigs ("Simplified State Space Layers ...", "Paper vs code":
 *           the real part of lambda clipped to at most -1e-4): when non-zero,
 *           Re(lambda_n) is replaced by min(Re(lambda_n), clip_re) before
 *           discretising.  0 disables clipping; a positive value is rejected.
 *   dt_scale sampling-rate rescaling (review "Sampling intervals carry
 *           physical meaning"; summary section 6.2):
 *           Delta_n = dt_scale * exp(log_dt[n]) with dt_scale = old sampling
 *           rate / new sampling rate (16 kHz -> 8 kHz gives 2).  Must be > 0.
 * Computed in float-float arithmetic and rounded once, as s5_discretize.
 * Arrays as in s5_discretize.  Errors: S5_ERR_INVALID_ARGUMENT for null/misaligned
 * pointers, P, H < 1, an unknown method, dt_scale <= 0 or clip_re > 0.
 */
s5_status s5_discretize_ex(const float *lambda, const float *log_dt, const float *b_tilde, int P, int H,
                           s5_discretization method, float clip_re, float dt_scale, float *lambda_bar,
                           float *b_bar, s5_stream_t stream);

/*
 * Forward pass of the time-invariant layer over B sequences of length L
 * (review rows 1, 3, 4; summary App. A and App. H):
 *   Bu_k = b_bar u_k                          (input projection)
 *   x_k  = lambda_bar * x_{k-1} + Bu_k         (diagonal recurrence, k = 1..L,
 *                                              x_0 = x0 or 0; evaluated as an
 *                                              associative scan over time)
 *   y_k  = 2 Re(c_tilde x_k) + d * u_k        (readout, d not doubled)
 *   lambda_bar [P] complex; b_bar [P,H] complex; c_tilde [H,P] complex; d [H] float32
 *   u [B,L,H] of u_dtype; y [B,L,H] of y_dtype (float32 or bfloat16)
 *   proj_dtype: S5_F32 computes both projections in float32; S5_BF16 lets the
 *     kernel round b_bar, c_tilde, u and x to bfloat16 as tensor-core inputs
 *     (float32 accumulation; the recurrence always runs in complex float32).
 *   x0 [B,P] complex or NULL (zero initial state); x_last [B,P] complex or NULL
 *     (receives x_L, so a long sequence can be fed in consecutive calls).
 *   workspace: device scratch of at least s5_workspace_size(B,L,H,P) bytes,
 *     zero-filled before its first use; each call leaves it ready for the
 *     next.  One workspace serves one call at a time.
 * B = 0 or L = 0 is a no-op (x_last then receives x0, or zeros).
 */
s5_status s5_forward(const float *lambda_bar, const float *b_bar, const float *c_tilde,
                     const float *d, const void *u, s5_dtype u_dtype, void *y, s5_dtype y_dtype,
                     s5_dtype proj_dtype, int B, int L, int H, int P, const float *x0,
                     float *x_last, void *workspace, size_t workspace_bytes, s5_stream_t stream);

/*
 * Forward pass with a different interval at every step (irregular sampling;
 * summary sections 3.3 and 6.3, review "Sampling intervals carry physical
 * meaning").  Step k of sequence b and mode n uses
 *   Delta_{b,k,n} = dt_scale[b,k] * exp(log_dt[n])
 *   a_{b,k,n}     = exp(lambda_n Delta_{b,k,n})
 *   x_k           = a_k * x_{k-1} + ((a_k - 1)/lambda) * (b_tilde u_k)
 *   y_k           = 2 Re(c_tilde x_k) + d * u_k
 * The discretised matrices are never formed.  dt_scale [B,L] float32 holds the
 * gaps g_k >= 0; a negative or non-finite gap latches S5_ERR_NONFINITE.
 * Other arguments as in s5_forward, with the continuous parameters lambda [P],
 * log_dt [P], b_tilde [P,H] in place of lambda_bar and b_bar.
 */
s5_status s5_forward_varying_dt(const float *lambda, const float *log_dt, const float *b_tilde,
                                const float *c_tilde, const float *d, const float *dt_scale,
                                const void *u, s5_dtype u_dtype, void *y, s5_dtype y_dtype,
                                s5_dtype proj_dtype, int B, int L, int H, int P,
                                const float *x0, float *x_last, void *workspace,
                                size_t workspace_bytes, s5_stream_t stream);

/*
 * One streaming step of B independent sequences (review "Associative scans
 * preserve the recurrence": streaming inference keeps just the current state;
 * summary App. C.1, online generation at O(PH) per step):
 *   x_b <- lambda_bar * x_b + b_bar u_b
 *   y_b  = 2 Re(c_tilde x_b) + d * u_b
 *   lambda_bar [P], b_bar [P,H], c_tilde [H,P] complex; d [H] float32
 *   x [B,P] complex, updated in place (the state of s5_forward's x0 / x_last)
 *   u [B,H] float32 in; y [B,H] float32 out
 * Float32 throughout.  Errors: S5_ERR_INVALID_ARGUMENT for null/misaligned
 * pointers or B < 0, H < 1, P < 1; B = 0 is a no-op (x, u, y may then be
 * null); S5_ERR_UNSUPPORTED when the 8 * (8 * (P + ceil(P/8)) + 4H) bytes of
 * staged states and inputs exceed 200 KiB (about P, H > 2000).
 */
s5_status s5_step(const float *lambda_bar, const float *b_bar, const float *c_tilde, const float *d,
                  float *x, const float *u, float *y, int B, int H, int P, s5_stream_t stream);

/*
 * Bidirectional layer ("Simplified State Space Layers ...", "Paper vs code":
 * the code runs a forward and a backward scan and concatenates them, so C~
 * has 2P columns; review "Published results": the backward scan sees future
 * inputs, so this is for offline use).  Both scans use lambda_bar and b_bar:
 *   xf_k = lambda_bar * xf_{k-1} + b_bar u_k,   xf_0 = 0
 *   xb_k = lambda_bar * xb_{k+1} + b_bar u_k,   xb_{L+1} = 0
 *   y_k  = 2 Re(c_tilde2[:, 0:P] xf_k + c_tilde2[:, P:2P] xb_k) + d * u_k
 *   c_tilde2 [H,2P] complex; other arrays, dtypes and proj_dtype as in
 *   s5_forward (the same kernel path is chosen for both scans).
 *   workspace: at least s5_bidirectional_workspace_size(B,L,H,P,u_dtype,y_dtype)
 *   bytes, zero-filled before its first use.
 * Runs as (all on `stream`): the two halves of c_tilde2 split into [H,P]
 * arrays; then
 *  - tensor-core shapes (H = P = 128, bf16 u, y and projections): s5_forward
 *    on u with the first half and d, then one more launch of the same kernel
 *    that scans every sequence from its end with the second half and adds its
 *    readout into y in place;
 *  - other shapes: u reversed in time, s5_forward on u (with d) and on the
 *    reversed u (with d = 0), and the second result reversed and added into y.
 * Errors: those of s5_forward; S5_ERR_UNSUPPORTED when B*L*H >= 2^31.
 */
s5_status s5_forward_bidirectional(const float *lambda_bar, const float *b_bar, const float *c_tilde2,
                                   const float *d, const void *u, s5_dtype u_dtype, void *y,
                                   s5_dtype y_dtype, s5_dtype proj_dtype, int B, int L, int H, int P,
                                   void *workspace, size_t workspace_bytes, s5_stream_t stream);

/* Bytes of workspace s5_forward_bidirectional needs; 0 for invalid sizes. */
size_t s5_bidirectional_workspace_size(int B, int L, int H, int P, s5_dtype u_dtype, s5_dtype y_dtype);

/* Bytes of workspace that s5_forward / s5_forward_varying_dt need for these
 * sizes (carry flags and per-tile aggregates of the chunked scan, plus a
 * small header).  Returns 0 for invalid sizes. */
size_t s5_workspace_size(int B, int L, int H, int P);

/*
 * s5_forward without a workspace, for callers that cannot allocate device
 * memory (a plugin in a host application that owns all device memory, a
 * latency-critical loop that must not enter the allocator, an embedded
 * deployment with a fixed memory budget).  The paper has no counterpart.
 * Arguments, layouts, dtypes, results and errors are those of s5_forward,
 * including its choice of kernel: bf16 u, y and projections at H = P = 128
 * run the tensor-core kernel, everything else the CUDA-core kernel.  The
 * caller still passes every input and output.  The workspace is a fixed
 * device array of S5_NOALLOC_SCRATCH_BYTES inside the library (zeroed when
 * the library loads), held on every GPU that loads it until the process
 * exits.
 *  - Sizes whose s5_workspace_size(B,L,H,P) exceeds S5_NOALLOC_SCRATCH_BYTES
 *    are rejected with S5_ERR_INVALID_ARGUMENT before anything is queued.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any
 *    stream capture.
 *  - The call allocates nothing (no cudaMalloc, no cudaFree, no allocating
 *    library routine) and clears nothing: like any workspace, the array needs
 *    no clearing between calls.  It queues the same kernels as s5_forward.
 *  - A failed CUDA call returns S5_ERR_CUDA, its text in s5_last_cuda_error().
 *  - Every call shares the one array: calls that overlap on the GPU (other
 *    streams, other host threads) race and give wrong results.  Serialize them.
 *  - Device-side conditions (a carry wait that gave up) are not reported.
 */
#define S5_NOALLOC_SCRATCH_BYTES (16u << 20)
s5_status s5_forward_noalloc(const float *lambda_bar, const float *b_bar, const float *c_tilde,
                             const float *d, const void *u, s5_dtype u_dtype, void *y,
                             s5_dtype y_dtype, s5_dtype proj_dtype, int B, int L, int H, int P,
                             const float *x0, float *x_last, s5_stream_t stream);

/* ========================================================================
 * Layer stack (pre-LayerNorm -> S5 layer -> gated activation -> residual)
 * and its backward, for general shapes (the deep-stack workload: H = 512,
 * P = 256, bf16 GEMM operands, complex fp32 scans).  Sources: "SIMPLIFIED
 * STATE SPACE LAYERS FOR SEQUENCE MODELING" section 6 (pre-norm layers); the
 * wiki "Method" step 4 and pseudocode (hidden = GELU(y), out = hidden *
 * sigmoid(W hidden), no bias per its "Paper vs code"); the review's row 4
 * (residual in the wrapper).  The backward is not on the pages: it is the
 * chain rule of the forward, with grad(z) = dL/dRe z + i dL/dIm z.
 *
 * Shared conventions: device pointers owned by the caller, 16-byte aligned;
 * T = N = B*L tokens, row-major [T][H] activations; complex arrays are
 * interleaved (re, im) float pairs.  Dense contractions are bf16 GEMMs with
 * fp32 accumulation on the tensor cores (s5_gemm_bf16 below); every step
 * runs in this library's kernels.  Calls are asynchronous on `stream`; the return value reports
 * argument and launch errors (S5_ERR_CUDA: text in s5_stack_last_error()).
 * ======================================================================== */

/* Bytes of `workspace` that s5_ssm_forward_states and s5_ssm_backward need;
 * it also covers s5_gate_residual and s5_gate_backward.  Contents need no
 * initialisation and are scratch between calls. */
size_t s5_stack_workspace_size(int B, int L, int H, int P);

/* Text of the last CUDA error of the stack entry points. */
const char *s5_stack_last_error(void);

/* The stack's dense contraction (wiki "Method" step 4 and its pseudocode:
 * B_bar z, the readout 2 Re(C~ x) over X, the gate's W h; review rows 1 and
 * 4; and the adjoint products of the backward):
 *   C[M][N] = op(A) op(B),  bf16 operands, fp32 accumulation and output.
 * A is row-major [M][K] (lda >= K), or with ta != 0 [K][M] (lda >= M);
 * B is row-major [K][N] (ldb >= N), or with tb != 0 [N][K] (ldb >= K);
 * C is row-major [M][N], ldc >= N.  Pitches are in elements.  C is
 * overwritten (no accumulation into it).  When the operand bases are
 * 16-byte aligned and lda, ldb are multiples of 8 the product runs on the
 * tensor cores (tcgen05, TMA-fed, K split over the SMs when the output is
 * small and K long); other shapes run on a CUDA-core kernel.  M, N = 0 is a
 * no-op; K = 0 writes zeros.  Asynchronous on `stream`.  Errors:
 * S5_ERR_INVALID_ARGUMENT (negative sizes, null pointers, pitches too small),
 * S5_ERR_CUDA (launch; text in s5_stack_last_error()). */
s5_status s5_gemm_bf16(int ta, int tb, int M, int N, int K, const void *A, long long lda, const void *B,
                       long long ldb, float *C, long long ldc, s5_stream_t stream);

/* 1 if a wait inside the tensor-core GEMM ran out since the last call (the
 * products of that launch are then not valid), 0 if none; the flag is
 * cleared.  Synchronises the device. */
int s5_gemm_fault(void);

/* LayerNorm over the last axis without affine parameters, biased variance,
 * eps = 1e-5:  z = (x - mean(x)) / sqrt(var(x) + eps) per row.
 * x [N][H] f32 -> z [N][H] f32 and, if z_bf16 is not NULL, its bf16 copy.
 * H <= 1024 (S5_ERR_UNSUPPORTED otherwise).  N = 0 is a no-op. */
s5_status s5_layernorm(const float *x, float *z, void *z_bf16, long long N, int H,
                       s5_stream_t stream);

/* bf16 GEMM operands of one layer's weights:
 *   bs [2P][H]: rows 0..P-1 = Re B_bar, rows P..2P-1 = Im B_bar
 *   cp [H][2P]: (2 Re C~, -2 Im C~) interleaved per mode (readout, K = 2P)
 *   cx [H][2P]: [2 Re C~ | -2 Im C~] as two halves (adjoint readout)
 *   w16 [H][H]: the gate's W
 * from b_bar [P][H] complex, c_tilde [H][P] complex, W [H][H] f32. */
s5_status s5_stack_weights(const float *b_bar, const float *c_tilde, const float *W, int H, int P,
                           void *bs, void *cp, void *cx, void *w16, s5_stream_t stream);

/* S5 layer with its states kept for the backward (review rows 3 and 4; paper
 * section 3.2 eq. 6, App. H):
 *   Bu_k = B_bar z_k (bf16 GEMM of z_bf16 and bs),  x_k = lambda_bar x_{k-1} + Bu_k
 *   (complex fp32, per sequence, from x0 or zero),  y_k = 2 Re(C~ x_k)
 *   (bf16 GEMM of X and cp).
 * The feed-through D z_k is NOT included in y: s5_gate_residual adds it.
 * z [B][L][H] f32 and its bf16 copy -> y [B][L][H] f32, x [B][L][P] complex
 * f32 (all states), X [B][L][2P] bf16 (states, interleaved Re, Im).
 * x0 [B][P] complex or NULL.  d is unused here (kept for symmetry). */
s5_status s5_ssm_forward_states(const float *lambda_bar, const void *bs, const void *cp,
                                const float *d, const float *z, const void *z_bf16, int B, int L,
                                int H, int P, const float *x0, float *y, float *x, void *X,
                                void *workspace, size_t workspace_bytes, s5_stream_t stream);

/* Gated activation and residual (wiki "Method" step 4; review row 4):
 *   y = y_ssm + d * z,  h = GELU(y) (exact erf form),  a = W h (bf16 GEMM),
 *   u_next = u + h * sigmoid(a).
 * y_ssm, z, u [N][H] f32; d [H]; w16 from s5_stack_weights -> y, a, u_next
 * [N][H] f32 (y and a are kept for the backward).  workspace >= 2*N*H bytes. */
s5_status s5_gate_residual(const float *y_ssm, const float *z, const float *d, const void *w16,
                           const float *u, long long N, int H, float *y, float *a, float *u_next,
                           void *workspace, size_t workspace_bytes, s5_stream_t stream);

/* Backward of the gate: given ubar = dL/du_next [N][H] and the kept y, a:
 *   act = ubar * h * s (1 - s) with s = sigmoid(a), h = GELU(y),
 *   ybar = (ubar * s + W^T act) * GELU'(y),  dW = act^T h  (bf16 GEMMs).
 * -> ybar [N][H] f32 and bf16, dW [H][H] f32.  workspace >= 12*N*H + 768 bytes. */
s5_status s5_gate_backward(const float *ubar, const float *y, const float *a, const void *w16,
                           long long N, int H, float *ybar, void *ybar_bf16, float *dW,
                           void *workspace, size_t workspace_bytes, s5_stream_t stream);

/* Backward of the S5 layer, the LayerNorm and the residual, given ybar =
 * dL/dy [B][L][H] (f32 and bf16) and ubar_in = dL/du_next:
 *   x_hat_k = 2 C~^H ybar_k (bf16 GEMM with cx),
 *   s_k = x_hat_k + conj(lambda_bar) s_{k+1}, s past the end = 0 (reverse scan),
 *   zbar_k = Re(B_bar^H s_k) + D ybar_k (bf16 GEMM with bs),
 *   ubar_out = ubar_in + LayerNorm'(u)^T zbar   (u = the layer input),
 *   dD = sum_k ybar_k z_k,  dC~ = 2 sum_k ybar_k x_k^H,  dB_bar = sum_k s_k z_k^T,
 *   dlambda_bar = sum_k conj(x_{k-1}) s_k (x_{-1} = x0),
 * then through the zero-order hold (float64): dB~ = conj(gain) dB_bar,
 *   dlambda = conj(dt e^z) dlambda_bar + conj(d gain/d lambda) sum_h dB_bar conj(B~),
 *   dlog_dt = dt (Re(conj(dlambda_bar) lambda e^z) + Re(conj(gphi) e^z)),
 * gain = (e^z - 1)/lambda, z = lambda dt (series below |z| = 1e-4).
 * lambda [P], log_dt [P], b_tilde [P][H] are the layer's parameters;
 * lambda_bar, bs, cx its discretised operands; z, z_bf16, x, X from the
 * forward.  Outputs: ubar_out [B][L][H] (may alias ubar_in), dlambda [P]
 * complex, dlog_dt [P], db_tilde [P][H] complex, dc_tilde [H][P] complex,
 * dd [H].  H <= 1024. */
s5_status s5_ssm_backward(const float *lambda, const float *log_dt, const float *b_tilde,
                          const float *lambda_bar, const void *bs, const void *cx, const float *d,
                          const float *u, const float *z, const void *z_bf16, const float *x,
                          const void *X, const float *x0, const float *ybar, const void *ybar_bf16,
                          const float *ubar_in, int B, int L, int H, int P, float *ubar_out,
                          float *dlambda, float *dlog_dt, float *db_tilde, float *dc_tilde,
                          float *dd, void *workspace, size_t workspace_bytes, s5_stream_t stream);

/* Waits for `stream`, returns the first device-side condition latched in
 * `workspace` since the last call (S5_OK if none) and clears it. */
s5_status s5_sync_status(void *workspace, s5_stream_t stream);

/* Static description of a status code. */
const char *s5_status_string(s5_status status);

/* Text of the last CUDA error seen by this thread ("" if none). */
const char *s5_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* S5_H */
