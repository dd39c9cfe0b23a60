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

/*
 * Zero-order-hold discretisation ("SIMPLIFIED STATE SPACE LAYERS ...",
 * section 3.2 eq. 6; review row 2):
 *   Delta_n      = exp(log_dt[n])
 *   lambda_bar_n = exp(lambda_n * Delta_n)
 *   b_bar[n,:]   = (lambda_bar_n - 1) / lambda_n * b_tilde[n,:]
 * with the removable singularity lambda_n*Delta_n -> 0 taken as the limit
 * Delta_n * b_tilde[n,:].  Computed in float64 on the device and rounded once.
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

/* Bytes of workspace that s5_forward / s5_forward_varying_dt need for these
 * sizes (carry flags and per-tile aggregates of the chunked scan, plus a
 * small header).  Returns 0 for invalid sizes. */
size_t s5_workspace_size(int B, int L, int H, int P);

/*
 * s5_forward without a workspace, for callers that cannot allocate device
 * memory (a plugin in a host application that owns all device memory, a
 * latency-critical loop that must not enter the allocator, an embedded
 * deployment with a fixed memory budget).  The paper has no counterpart.
 * Arguments, layouts and results are those of s5_forward; the caller still
 * passes every input and output.  The carry scratch is a fixed device array
 * of S5_NOALLOC_SCRATCH_BYTES inside the library, held on every GPU that loads
 * it until the process exits.
 *  - Sizes whose s5_workspace_size(B,L,H,P) exceeds S5_NOALLOC_SCRATCH_BYTES
 *    are rejected with S5_ERR_INVALID_ARGUMENT before anything is queued.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any
 *    stream capture.
 *  - The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 *    library routine.  It clears the scratch's header and flags on `stream`
 *    (cudaMemsetAsync) and launches the CUDA-core forward kernel.
 *  - Every call shares the one array: calls that overlap on the GPU (other
 *    streams, other host threads) race and give wrong results.  Serialize them.
 *  - Device-side conditions (a carry wait that gave up) are not reported.
 */
#define S5_NOALLOC_SCRATCH_BYTES (8u << 20)
s5_status s5_forward_noalloc(const float *lambda_bar, const float *b_bar, const float *c_tilde,
                             const float *d, const void *u, s5_dtype u_dtype, void *y,
                             s5_dtype y_dtype, s5_dtype proj_dtype, int B, int L, int H, int P,
                             const float *x0, float *x_last, s5_stream_t stream);

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
