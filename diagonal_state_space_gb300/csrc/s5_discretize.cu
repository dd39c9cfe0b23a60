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
// spread over P SMs).  The float64 functions of the mode's factors are spread
// over the first four threads, so that each evaluates at most two of them in
// sequence:
//   every thread  dt = exp(log_dt)
//   thread 0      sin(Im z), cos(Im z)      thread 1  exp(Re z)
//   thread 2      expm1(Re z)               thread 3  sin(Im z / 2)
// then lambda_bar = e^Re z (cos, sin) and, for |z| >= 1e-4,
// (e^z - 1)/lambda = (expm1(Re z) cos(Im z) - 2 sin^2(Im z/2) + i e^Re z sin(Im z))/lambda;
// below |z| = 1e-4, Delta * phi1(z) from its Taylor series.  Every thread of
// the block then scales a slice of the B_tilde row.
__global__ void discretize_kernel(const float2 *__restrict__ lambda, const float *__restrict__ log_dt,
                                  const float2 *__restrict__ b_tilde, int P, int H,
                                  float2 *__restrict__ lambda_bar, float2 *__restrict__ b_bar) {
    const int p = blockIdx.x;
    __shared__ double s_gain[2];
    if (threadIdx.x < 32) {
        const int q = threadIdx.x & 3;
        const float2 l = lambda[p];
        const dcplx lam = {(double)l.x, (double)l.y};
        const double dt = exp((double)log_dt[p]);
        const dcplx z = {lam.re * dt, lam.im * dt};
        double f0 = 0.0, f1 = 0.0;
        if (threadIdx.x < 4) {
            if (q == 0) sincos(z.im, &f0, &f1);
            else if (q == 1) f0 = exp(z.re);
            else if (q == 2) f0 = expm1(z.re);
            else f0 = sin(0.5 * z.im);
        }
        const unsigned full = 0xffffffffu;
        const double s = __shfl_sync(full, f0, 0), c = __shfl_sync(full, f1, 0);
        const double mag = __shfl_sync(full, f0, 1);
        const double em1r = __shfl_sync(full, f0, 2);
        const double sh = __shfl_sync(full, f0, 3);
        if (threadIdx.x == 0) {
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
                gain = ddiv(em1, lam);
            }
            lambda_bar[p] = make_float2((float)(mag * c), (float)(mag * s));
            s_gain[0] = gain.re;
            s_gain[1] = gain.im;
        }
    }
    __syncthreads();
    const dcplx g = {s_gain[0], s_gain[1]};
    const float2 *src = b_tilde + (size_t)p * H;
    float2 *dst = b_bar + (size_t)p * H;
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        const float2 bt = src[h];
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
                              int P, int H, float2 *lambda_bar, float2 *b_bar, cudaStream_t st) {
    const int threads = H >= 256 ? 256 : (H >= 128 ? 128 : 64);
    discretize_kernel<<<P, threads, 0, st>>>(lambda, log_dt, b_tilde, P, H, lambda_bar, b_bar);
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
