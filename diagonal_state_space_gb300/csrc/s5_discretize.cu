// s5_discretize.cu -- zero-order-hold discretisation of the diagonal modes.
//
// "SIMPLIFIED STATE SPACE LAYERS FOR SEQUENCE MODELING", section 3.2 eq. 6, and
// the abhik.ai review "S5: Simplified State Space Layers for Sequence Modeling",
// "Paper equations beside executable Python" row 2:
//   lambda_bar = exp(lambda*Delta),  B_bar = (lambda_bar - 1)/lambda * B_tilde,
// where (lambda_bar - 1)/lambda = Delta*phi1(lambda*Delta), phi1(z) = (e^z-1)/z,
// has a removable singularity at z = 0 (limit Delta).
//
// The per-mode factors are computed in float64 (only P values per call) with
// a complex expm1, e^z - 1 = expm1(x)cos(y) - 2 sin^2(y/2) + i e^x sin(y), so
// that small |z| loses no digits; below |z| = 1e-4 a Taylor series of phi1 is
// used instead, as the review's reference does.
#include "s5_internal.cuh"

namespace s5 {

struct dcplx { double re, im; };

__device__ inline dcplx dmul(dcplx a, dcplx b) {
    return {a.re * b.re - a.im * b.im, a.re * b.im + a.im * b.re};
}
__device__ inline dcplx ddiv(dcplx a, dcplx b) {
    double den = b.re * b.re + b.im * b.im;
    return {(a.re * b.re + a.im * b.im) / den, (a.im * b.re - a.re * b.im) / den};
}

// One block per mode (float64 throughput per SM is small, so the work is
// spread over P SMs).  The float64 functions of the mode's factors run side by
// side on the first lane of four different warps (lanes of one warp taking
// different branches would run them one after another):
//   every thread  dt = exp(log_dt)
//   warp 0  sin(Im z), cos(Im z)      warp 1  exp(Re z)
//   warp 2  expm1(Re z)               warp 3  sin(Im z / 2)
//   warp 4  1 / lambda
// then lambda_bar = e^Re z (cos, sin) and, for |z| >= 1e-4,
// (e^z - 1)/lambda = (expm1(Re z) cos(Im z) - 2 sin^2(Im z/2) + i e^Re z sin(Im z)) * (1/lambda);
// below |z| = 1e-4, Delta * phi1(z) from its Taylor series.  Every thread of
// the block then scales a slice of the B_tilde row.  Blocks have >= 160 threads.
//
// Options (all in float64, applied before the factors above):
//   clip_re != 0   clip_eigs: Re(lambda) <- min(Re(lambda), clip_re)
//                  (wikillm "Paper vs code": the official value is -1e-4);
//   dt_scale       sampling-rate rescaling, Delta <- Delta * dt_scale with
//                  dt_scale = old rate / new rate (review "Sampling intervals
//                  carry physical meaning"; summary section 6.2);
//   method 1       bilinear transform instead of the zero-order hold (review
//                  "Discretization controls both retention and input gain";
//                  the S4 page, "Discretize"): for a diagonal mode
//                  lambda_bar = (1 + Delta lambda/2) / (1 - Delta lambda/2) and
//                  gain = Delta / (1 - Delta lambda/2).
__global__ void discretize_kernel(const float2 *__restrict__ lambda, const float *__restrict__ log_dt,
                                  const float2 *__restrict__ b_tilde, int P, int H,
                                  float2 *__restrict__ lambda_bar, float2 *__restrict__ b_bar, int method,
                                  double clip_re, double dt_scale) {
    const int p = blockIdx.x;
    // the kernel that consumes Lambda_bar and B_bar may be scheduled now; it
    // waits for this one to complete before reading them
    griddep_launch_dependents();
    __shared__ double s_f[7];      // sin Im z, cos Im z, exp Re z, expm1 Re z, sin(Im z / 2), 1/lambda
    __shared__ double s_gain[2];
    // Only the first lane of each of the first five warps needs Delta and z:
    // float64 work on the other lanes would still occupy the SM's few float64
    // units, so they skip it.
    const bool leader = (threadIdx.x & 31) == 0 && threadIdx.x < 160;
    // this thread's first B_tilde element, fetched now so that its latency
    // overlaps the float64 work below
    const float2 *src = b_tilde + (size_t)p * H;
    const float2 bt0 = (int)threadIdx.x < H ? src[threadIdx.x] : make_float2(0.f, 0.f);
    dcplx lam = {0.0, 0.0}, z = {0.0, 0.0};
    double dt = 0.0;
    if (leader) {
        const float2 l = lambda[p];
        lam = {(double)l.x, (double)l.y};
        if (clip_re != 0.0 && lam.re > clip_re) lam.re = clip_re;
        dt = exp((double)log_dt[p]) * dt_scale;
        z = {lam.re * dt, lam.im * dt};
    }
    if (method == 1) {
        if (threadIdx.x == 0) {
            const dcplx den = {1.0 - 0.5 * z.re, -0.5 * z.im};
            const dcplx lb = ddiv(dcplx{1.0 + 0.5 * z.re, 0.5 * z.im}, den);
            const dcplx gain = ddiv(dcplx{dt, 0.0}, den);
            lambda_bar[p] = make_float2((float)lb.re, (float)lb.im);
            s_gain[0] = gain.re;
            s_gain[1] = gain.im;
        }
    } else if (leader) {
        const int w = threadIdx.x >> 5;
        if (w == 0) sincos(z.im, &s_f[0], &s_f[1]);
        else if (w == 1) s_f[2] = exp(z.re);
        else if (w == 2) s_f[3] = expm1(z.re);
        else if (w == 3) s_f[4] = sin(0.5 * z.im);
        else if (w == 4) {
            // 1/lambda, off the path of the functions above
            const double den = lam.re * lam.re + lam.im * lam.im;
            s_f[5] = lam.re / den;
            s_f[6] = -lam.im / den;
        }
    }
    __syncthreads();
    if (method != 1 && threadIdx.x == 0) {
        const double s = s_f[0], c = s_f[1], mag = s_f[2], em1r = s_f[3], sh = s_f[4];
        dcplx gain;
        const double zabs = sqrt(z.re * z.re + z.im * z.im);
        if (zabs < 1e-4) {
            // dt * (1 + z/2 + z^2/6 + z^3/24 + z^4/120); the next term is below 1e-22.
            dcplx term = {1.0, 0.0}, phi = {1.0, 0.0};
            for (int n = 1; n <= 4; ++n) {
                term = dmul(term, z);
                const double f = 1.0 / (double)(n + 1);
                term.re *= f;
                term.im *= f;
                phi.re += term.re;
                phi.im += term.im;
            }
            gain = {dt * phi.re, dt * phi.im};
        } else {
            const dcplx em1 = {em1r * c - 2.0 * sh * sh, mag * s};
            gain = dmul(em1, dcplx{s_f[5], s_f[6]});
        }
        lambda_bar[p] = make_float2((float)(mag * c), (float)(mag * s));
        s_gain[0] = gain.re;
        s_gain[1] = gain.im;
    }
    __syncthreads();
    const dcplx g = {s_gain[0], s_gain[1]};
    float2 *dst = b_bar + (size_t)p * H;
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        const float2 bt = h == (int)threadIdx.x ? bt0 : src[h];
        const dcplx v = dmul(g, dcplx{(double)bt.x, (double)bt.y});
        dst[h] = make_float2((float)v.re, (float)v.im);
    }
}

// Per-mode constants of the irregular-sampling path (see ModeConst).
__global__ void mode_consts_kernel(const float2 *__restrict__ lambda, const float *__restrict__ log_dt,
                                   int P, ModeConst *__restrict__ out) {
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= P) return;
    float2 l = lambda[p];
    double lr = l.x, li = l.y;
    double dt = exp((double)log_dt[p]);
    double om = li * dt;
    ModeConst m;
    m.om_hi = (float)om;
    m.om_lo = (float)(om - (double)m.om_hi);
    m.rho = (float)(lr * dt);
    m.dt = (float)dt;
    double den = lr * lr + li * li;
    m.inv_re = den > 0 ? (float)(lr / den) : 0.f;
    m.inv_im = den > 0 ? (float)(-li / den) : 0.f;
    m.zabs = (float)(sqrt(den) * dt);
    m.pad = 0.f;
    out[p] = m;
}

cudaError_t launch_discretize(const float2 *lambda, const float *log_dt, const float2 *b_tilde,
                              int P, int H, float2 *lambda_bar, float2 *b_bar, cudaStream_t st, int method,
                              double clip_re, double dt_scale) {
    const int threads = H >= 256 ? 256 : 160;   // at least five warps (see discretize_kernel)
    discretize_kernel<<<P, threads, 0, st>>>(lambda, log_dt, b_tilde, P, H, lambda_bar, b_bar, method, clip_re,
                                             dt_scale);
    return cudaGetLastError();
}

cudaError_t launch_mode_consts(const float2 *lambda, const float *log_dt, int P, ModeConst *out,
                               cudaStream_t st) {
    // a few modes per block so that the float64 work spreads over many SMs
    const int threads = 32;
    mode_consts_kernel<<<(P + threads - 1) / threads, threads, 0, st>>>(lambda, log_dt, P, out);
    return cudaGetLastError();
}

}  // namespace s5
